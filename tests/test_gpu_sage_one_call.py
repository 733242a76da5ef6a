"""sage_attention, the one-call Sage op (CUDA through the C ABI), equals the
two-call sequence sage_prepare (+ smoothing) + sage_attn_fwd / sage_attn_fwd_pv16
bit for bit: its prepare writes the Q/K codes as FP16 straight into the
workspace the forward reads and V's as sage_prepare does, and the forward's
arithmetic from the codes on is the same.  With q_on_load the forward codes Q
itself as it loads it (RMSNorm and RoPE first when asked); equal outputs then
pin those in-kernel Q codes and scales to the prepare's, which
test_gpu_prepare.py pins to the oracle bit for bit; with k_on_load the forward
codes every K tile as well (block scales in shared memory), with the same result.  Every output with Q coded
on load is also compared with the oracle directly, on the same shapes: with
the format gate against the exact value of its format (oracle.sage_attention
for e4m3 P V, oracle.sage_attention_v16 for the 16-bit P V) and with the
acceptance gates against the FP64 attention of the BF16 inputs (after the
oracle's RMSNorm + RoPE), as test_gpu_sage.py and test_gpu_sage_pv16.py do for
the two-call path."""
import dataclasses

import pytest
import torch

import oracle
import sage_attention_forward_gb300 as sa
from parity import (BF16_A, BF16_B, SAGE_A, SAGE_B, assert_bf16_gate, assert_sage_exact_gate,
                    assert_sage_format_gate, gather_rows, metrics)
from workloads import make_inputs, sample_rows, small_case, to_device, wide_bf16

pytestmark = pytest.mark.gpu


def kwargs(g, wl):
    kw = {}
    if g.q_norm_w is not None:
        kw.update(q_norm_w=g.q_norm_w, k_norm_w=g.k_norm_w, rms_eps=wl.rms_eps)
    if g.rope_cos is not None:
        kw.update(rope_cos=g.rope_cos, rope_sin=g.rope_sin, rope_dim=wl.rope_dim)
    return kw


def two_calls(g, wl, smooth_k, pv):
    prep = sa.sage_prepare(g.q, g.k, g.v, softmax_scale=wl.softmax_scale, smooth_k=smooth_k, **kwargs(g, wl))
    if pv == "bf16":
        return sa.sage_attn_fwd_pv16(prep, g.v)
    return sa.sage_attn_fwd(prep)


def oracle_check(o, cpu, pv, smooth_k=False, rows=None, exact_gate=True):
    """The output against the oracle: the format gate against its format's exact value
    and the acceptance gates against FP64 attention of the (normed, roped) BF16 inputs
    (exact_gate False: within 0.002 of the format's own cosine there instead; None: the
    format gate alone)."""
    wl = cpu.wl
    if rows is None:
        rows = oracle.all_rows(wl.B, wl.S, wl.H)
    prep = oracle.prepare(cpu.q, cpu.k, cpu.v, wl.softmax_scale, q_norm_w=cpu.q_norm_w, k_norm_w=cpu.k_norm_w,
                          rms_eps=wl.rms_eps, rope_cos=cpu.rope_cos, rope_sin=cpu.rope_sin, rope_dim=wl.rope_dim,
                          smooth_k=smooth_k)
    got = gather_rows(o, rows)
    if pv == "bf16":
        fmt = oracle.sage_attention_v16(prep, cpu.v, rows)
        m_fmt = metrics(got, fmt, oracle.sage_attention_v16(prep, cpu.v, rows, abs_v=True), BF16_A, BF16_B)
        assert_bf16_gate(m_fmt, "q_on_load, 16-bit P V, vs format")
    else:
        fmt = oracle.sage_attention(prep, wl.S, rows, wl.H)
        m_fmt = metrics(got, fmt, oracle.sage_attention(prep, wl.S, rows, wl.H, abs_v=True), SAGE_A, SAGE_B)
        assert_sage_format_gate(m_fmt, "q_on_load, e4m3 P V, vs format")
    if exact_gate is None:
        return
    exact = oracle.attention(prep["q_pre"], prep["k_pre"], cpu.v, wl.softmax_scale, rows=rows)
    m_exact = metrics(got, exact)
    print("q_on_load", pv, "vs format:", m_fmt, "\n   vs exact:", m_exact)
    if exact_gate:
        assert_sage_exact_gate(m_exact, f"q_on_load {pv} vs exact")
    else:
        m_floor = metrics(fmt, exact)
        assert m_exact["cos"] >= m_floor["cos"] - 0.002, f"{m_exact} vs format floor {m_floor}"


# on-load levels: 0 the prepare codes Q and K, 1 the forward codes Q, 2 the forward codes Q and K
LOAD = {0: dict(), 1: dict(q_on_load=True), 2: dict(q_on_load=True, k_on_load=True)}


@pytest.mark.parametrize("load", [0, 1, 2])
@pytest.mark.parametrize("pv", ["e4m3", "bf16"])
@pytest.mark.parametrize("smooth_k", [False, True])
@pytest.mark.parametrize("B,H,S,kw", [(1, 2, 31, {}), (2, 3, 300, dict(k_channel_offset_std=1.0)),
                                      (1, 2, 500, dict(rms_norm=True, rope_dim=64)), (1, 1, 1, {}),
                                      (1, 2, 900, dict(rms_norm=True, rope_dim=128))])
def test_one_call_equals_two_calls(cuda_dev, B, H, S, kw, smooth_k, pv, load):
    inp = make_inputs(small_case(B, H, S, 1500 + S, **kw))
    g = to_device(inp, cuda_dev)
    if smooth_k and load == 2:
        # K's sequence mean needs a pass of its own, which coding K tile by tile does not have
        with pytest.raises(sa.AttnError) as e:
            sa.sage_attention(g.q, g.k, g.v, smooth_k=True, pv=pv, **LOAD[load])
        assert e.value.status == 3
        return
    o1 = sa.sage_attention(g.q, g.k, g.v, softmax_scale=inp.wl.softmax_scale, smooth_k=smooth_k, pv=pv,
                           **LOAD[load], **kwargs(g, inp.wl))
    o2 = two_calls(g, inp.wl, smooth_k, pv)
    torch.cuda.synchronize()
    sa.attn_get_device_status()
    assert torch.equal(o1, o2)
    if load:
        oracle_check(o1, inp, pv, smooth_k)


@pytest.mark.parametrize("pv", ["e4m3", "bf16"])
def test_one_call_equals_two_calls_flux1024(cuda_dev, workload_inputs, pv):
    cpu, g = workload_inputs("flux1024")
    o1 = sa.sage_attention(g.q, g.k, g.v, softmax_scale=cpu.wl.softmax_scale, pv=pv)
    o2 = two_calls(g, cpu.wl, False, pv)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)


def test_non_default_stream_and_permuted_output(cuda_dev):
    inp = make_inputs(small_case(1, 3, 777, 1551))
    g = to_device(inp, cuda_dev)
    o1 = sa.sage_attention(g.q, g.k, g.v)
    B, S, H, D = g.q.shape
    store = torch.empty((B, H, S, D), dtype=torch.bfloat16, device=cuda_dev)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        sa.sage_attention(g.q, g.k, g.v, out=store.permute(0, 2, 1, 3), stream=s)
    s.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(store.permute(0, 2, 1, 3), o1)


@pytest.mark.parametrize("load", [1, 2])
@pytest.mark.parametrize("pv", ["e4m3", "bf16"])
@pytest.mark.parametrize("rope_dim,norm", [(32, True), (96, True), (128, True), (128, False), (0, True)])
def test_q_coded_on_load_with_norm_and_rope(cuda_dev, rope_dim, norm, pv, load):
    inp = make_inputs(small_case(1, 3, 400, 1600 + rope_dim, rms_norm=norm, rope_dim=rope_dim))
    g = to_device(inp, cuda_dev)
    o1 = sa.sage_attention(g.q, g.k, g.v, pv=pv, **LOAD[load], **kwargs(g, inp.wl))
    o2 = two_calls(g, inp.wl, False, pv)
    torch.cuda.synchronize()
    sa.attn_get_device_status()
    assert torch.equal(o1, o2)
    oracle_check(o1, inp, pv)


@pytest.mark.parametrize("load", [1, 2])
@pytest.mark.parametrize("S", [129, 300, 513])
def test_q_coded_on_load_zero_eps_ragged(cuda_dev, S, load):
    """rms_eps = 0: the rows past S, zeros whose RMSNorm factor is infinite, code to 0
    in the forward as in the prepare (also the rows past the padded length), for Q and,
    coded on load too, for K."""
    wl = dataclasses.replace(small_case(1, 2, S, 1700 + S, rms_norm=True, rope_dim=64), rms_eps=0.0)
    inp = make_inputs(wl)
    g = to_device(inp, cuda_dev)
    o1 = sa.sage_attention(g.q, g.k, g.v, **LOAD[load], **kwargs(g, wl))
    o2 = two_calls(g, wl, False, "e4m3")
    torch.cuda.synchronize()
    sa.attn_get_device_status()
    assert torch.equal(o1, o2)
    oracle_check(o1, inp, "e4m3")


def test_q_coded_on_load_extreme_blocks(cuda_dev):
    """Q blocks at the low end of the BF16 range, among them blocks whose 127 / max
    overflows (every code +-127: the forward's clamped branch) and subnormal ones,
    next to blocks spanning many binades."""
    S, H = 256, 2
    # scores stay below 2^20 (beyond 2^24 they are outside the kernels' range)
    ranges = [(-130, -123), (-20, 13), (5, 13), (-133, -126), (-3, 3), (-126, -100), (0, 1), (-60, 13)]
    q = torch.cat([wide_bf16(1800 + i, (1, 32, H, 128), lo, hi) for i, (lo, hi) in enumerate(ranges)], dim=1)
    inp = make_inputs(small_case(1, H, S, 1810))
    inp.q = q
    g = to_device(inp, cuda_dev)
    for pv, load in (("e4m3", 1), ("bf16", 1), ("e4m3", 2), ("bf16", 2)):
        o1 = sa.sage_attention(g.q, g.k, g.v, pv=pv, **LOAD[load])
        o2 = two_calls(g, inp.wl, False, pv)
        torch.cuda.synchronize()
        sa.attn_get_device_status()
        assert torch.equal(o1, o2), (pv, load)
        # one-hot softmaxes next to blocks whose scores are ~1e-38: the format gate, as the
        # two-call path's saturated-softmax test asks
        oracle_check(o1, inp, pv, exact_gate=None)


def test_k_coded_on_load_extreme_blocks(cuda_dev):
    """K blocks at the low end of the BF16 range (127 / max overflowing: every code +-127)
    and spanning many binades, coded tile by tile in the forward exactly as the prepare
    codes them."""
    S, H = 256, 2
    ranges = [(-130, -123), (-20, 3), (5, 10), (-133, -126), (-3, 3), (-126, -100), (0, 1), (-60, 5)]
    k = torch.cat([wide_bf16(1850 + i, (1, 32, H, 128), lo, hi) for i, (lo, hi) in enumerate(ranges)], dim=1)
    inp = make_inputs(small_case(1, H, S, 1860))
    inp.k = k
    g = to_device(inp, cuda_dev)
    for pv in ("e4m3", "bf16"):
        o1 = sa.sage_attention(g.q, g.k, g.v, pv=pv, q_on_load=True, k_on_load=True)
        o2 = two_calls(g, inp.wl, False, pv)
        torch.cuda.synchronize()
        sa.attn_get_device_status()
        assert torch.equal(o1, o2), pv
        oracle_check(o1, inp, pv, exact_gate=None)


@pytest.mark.parametrize("load", [1, 2])
@pytest.mark.parametrize("name", ["flux2048", "hunyuan720p"])
def test_q_coded_on_load_workloads(cuda_dev, workload_inputs, name, load):
    """FLUX-2048 (RMSNorm + RoPE 64 on Q and K) and HunyuanVideo-720p (head-major Q/K
    strides) at full size."""
    cpu, g = workload_inputs(name)
    o1 = sa.sage_attention(g.q, g.k, g.v, softmax_scale=cpu.wl.softmax_scale, **LOAD[load], **kwargs(g, cpu.wl))
    o2 = two_calls(g, cpu.wl, False, "e4m3")
    torch.cuda.synchronize()
    sa.attn_get_device_status()
    assert torch.equal(o1, o2)
    oracle_check(o1, cpu, "e4m3", rows=sample_rows(cpu.wl, 384, outlier_tokens=cpu.outlier_tokens))
