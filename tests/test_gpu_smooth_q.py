"""Q smoothing on the GPU (sage_prepare_smoothed, sage_attn_fwd_smooth_q,
sage_attn_fwd_pv16_smooth_q and sage_attention(smooth_q=1), CUDA through the C
ABI).

The prepare is bit-exact against the oracle: the INT8 codes of Q minus its
32-row block means, the scales, the block means in step units (binary16) --
also with K smoothing, RMSNorm + RoPE, ragged lengths and blocks at the ends
of the BF16 range -- with K and V unchanged.  The attention passes the Sage
gates against the oracle's exact value of the smoothed format (its Q operand
f16(code + mean) carries the correction term) and against FP64 attention of
the BF16 inputs; on Q with per-channel offsets it is closer to FP64 than the
unsmoothed format.  The one-call op equals the two-call sequence bit for bit.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import sage_attention_forward_gb300 as sa
from parity import (BF16_A, BF16_B, SAGE_A, SAGE_B, assert_bf16_gate, assert_sage_exact_gate,
                    assert_sage_format_gate, gather_rows, metrics)
from workloads import make_inputs, sample_rows, small_case, to_device, wide_bf16

pytestmark = pytest.mark.gpu

NAMES = ("q_i8", "k_i8", "v_fp8", "q_scale", "k_scale", "v_scale")


def kwargs(g, wl):
    kw = {}
    if g.q_norm_w is not None:
        kw.update(q_norm_w=g.q_norm_w, k_norm_w=g.k_norm_w, rms_eps=wl.rms_eps)
    if g.rope_cos is not None:
        kw.update(rope_cos=g.rope_cos, rope_sin=g.rope_sin, rope_dim=wl.rope_dim)
    return kw


def oracle_prepare(cpu, S_pad, smooth_k=False):
    wl = cpu.wl
    return oracle.prepare(cpu.q, cpu.k, cpu.v, wl.softmax_scale, S_pad=S_pad, q_norm_w=cpu.q_norm_w,
                          k_norm_w=cpu.k_norm_w, rms_eps=wl.rms_eps, rope_cos=cpu.rope_cos, rope_sin=cpu.rope_sin,
                          rope_dim=wl.rope_dim, smooth_k=smooth_k, smooth_q=True)


def assert_bit_exact(prep, exp, what, smooth_k=False):
    pairs = [(getattr(prep, n), exp[n]) for n in NAMES] + [(prep.q_mean.view(torch.int16), exp["q_mean16"])]
    if smooth_k:
        pairs.append((prep.k_mean, exp["k_mean"]))
    for i, (got, ref) in enumerate(pairs):
        got = got.cpu()
        same = torch.equal(got.view(torch.int32), ref.view(torch.int32)) if got.dtype == torch.float32 \
            else torch.equal(got, ref)
        if not same:
            diff = (got != ref)
            raise AssertionError(f"{what}: output {i} differs at {int(diff.sum())} places, first "
                                 f"{diff.nonzero()[:5].tolist()}")


@pytest.mark.parametrize("smooth_k", [False, True])
@pytest.mark.parametrize("B,H,S,kw", [
    (1, 1, 1, {}), (1, 3, 31, {}), (2, 2, 200, dict(q_channel_offset_std=3.0)), (1, 2, 1000, {}),
    (1, 3, 300, dict(rms_norm=True, rope_dim=64, q_channel_offset_std=1.0)), (2, 1, 129, dict(rope_dim=128)),
    (1, 2, 161, dict(q_channel_offset_std=50.0)),
])
def test_prepare_smooth_q_bit_exact(cuda_dev, B, H, S, kw, smooth_k):
    inp = make_inputs(small_case(B, H, S, 2400 + S, **kw))
    g = to_device(inp, cuda_dev)
    prep = sa.sage_prepare(g.q, g.k, g.v, softmax_scale=inp.wl.softmax_scale, smooth_q=True, smooth_k=smooth_k,
                           **kwargs(g, inp.wl))
    torch.cuda.synchronize()
    sa.attn_get_device_status()
    assert_bit_exact(prep, oracle_prepare(inp, prep.S_pad, smooth_k), f"B{B} H{H} S{S} {kw}", smooth_k)


@pytest.mark.parametrize("name", ["flux2048", "wan720p", "hunyuan720p"])
def test_workload_prepare_smooth_q_bit_exact(cuda_dev, workload_inputs, name):
    cpu, g = workload_inputs(name)
    prep = sa.sage_prepare(g.q, g.k, g.v, softmax_scale=cpu.wl.softmax_scale, smooth_q=True, **kwargs(g, cpu.wl))
    torch.cuda.synchronize()
    assert_bit_exact(prep, oracle_prepare(cpu, prep.S_pad), name)


def test_prepare_smooth_q_extreme_blocks(cuda_dev):
    """Blocks at both ends of the BF16 range (127 / a_eff overflowing: stored as zeros),
    constant blocks (deviations 0: the floor max|mean|/256 sets the step), a block with a
    huge common offset and tiny deviations, and ordinary ones."""
    S, H = 224, 2
    ranges = [(-130, -123), (-20, 13), (5, 13), (-133, -126), (-3, 3), (0, 1), (-60, 13)]
    q = torch.cat([wide_bf16(2500 + i, (1, 32, H, 128), lo, hi) for i, (lo, hi) in enumerate(ranges)], dim=1)
    q[:, 160:192] = q[:, 160:161]                                   # a constant block
    q[:, 192:224] = (1000.0 + 8.0 * torch.randn((1, 32, H, 128), generator=torch.Generator().manual_seed(2511))).to(torch.bfloat16)
    inp = make_inputs(small_case(1, H, S, 2510))
    inp.q = q
    g = to_device(inp, cuda_dev)
    prep = sa.sage_prepare(g.q, g.k, g.v, smooth_q=True)
    torch.cuda.synchronize()
    assert_bit_exact(prep, oracle_prepare(inp, prep.S_pad), "extreme blocks")


def check_attention(o, cpu, rows, pv, what, exact_gate=True, smooth_k=False):
    wl = cpu.wl
    prep = oracle_prepare(cpu, sa.sage_padded_len(wl.S), smooth_k)
    got = gather_rows(o, rows)
    if pv == "bf16":
        fmt = oracle.sage_attention_v16(prep, cpu.v, rows)
        m_fmt = metrics(got, fmt, oracle.sage_attention_v16(prep, cpu.v, rows, abs_v=True), BF16_A, BF16_B)
        assert_bf16_gate(m_fmt, what + " vs format")
    else:
        fmt = oracle.sage_attention(prep, wl.S, rows, wl.H)
        m_fmt = metrics(got, fmt, oracle.sage_attention(prep, wl.S, rows, wl.H, abs_v=True), SAGE_A, SAGE_B)
        assert_sage_format_gate(m_fmt, what + " vs format")
    exact = oracle.attention(prep["q_pre"], prep["k_pre"], cpu.v, wl.softmax_scale, rows=rows)
    m_exact = metrics(got, exact)
    m_floor = metrics(fmt, exact)
    print(what, "vs format:", m_fmt, "\n   vs exact:", m_exact, "\n   format vs exact:", m_floor)
    if exact_gate:
        assert_sage_exact_gate(m_exact, what + " vs exact")
    else:
        assert m_exact["cos"] >= m_floor["cos"] - 0.002, f"{what}: {m_exact} vs format floor {m_floor}"
    return m_exact


@pytest.mark.parametrize("pv", ["e4m3", "bf16"])
@pytest.mark.parametrize("B,H,S,kw", [
    (1, 1, 1, {}), (1, 2, 31, {}), (2, 3, 300, dict(q_channel_offset_std=3.0)),
    (1, 2, 513, dict(rms_norm=True, rope_dim=64, q_channel_offset_std=2.0)),
])
def test_attention_smooth_q(cuda_dev, B, H, S, kw, pv):
    inp = make_inputs(small_case(B, H, S, 2600 + S, **kw))
    g = to_device(inp, cuda_dev)
    o1 = sa.sage_attention(g.q, g.k, g.v, softmax_scale=inp.wl.softmax_scale, smooth_q=True, pv=pv,
                           **kwargs(g, inp.wl))
    prep = sa.sage_prepare(g.q, g.k, g.v, softmax_scale=inp.wl.softmax_scale, smooth_q=True, **kwargs(g, inp.wl))
    o2 = sa.sage_attn_fwd_pv16(prep, g.v) if pv == "bf16" else sa.sage_attn_fwd(prep)
    torch.cuda.synchronize()
    sa.attn_get_device_status()
    assert torch.equal(o1, o2)
    # Q with channel offsets sharpens the softmax until e4m3 P alone passes the 0.1 max-abs:
    # there the kernel is held to the format gate and the format's own cosine floor
    check_attention(o1, inp, oracle.all_rows(B, S, H), pv, f"smooth_q {pv} B{B} H{H} S{S}",
                    exact_gate=not (pv == "e4m3" and kw.get("q_channel_offset_std")))


def test_attention_smooth_q_and_k(cuda_dev):
    inp = make_inputs(small_case(1, 3, 700, 2700, q_channel_offset_std=2.0, k_channel_offset_std=2.0))
    g = to_device(inp, cuda_dev)
    o1 = sa.sage_attention(g.q, g.k, g.v, smooth_q=True, smooth_k=True)
    prep = sa.sage_prepare(g.q, g.k, g.v, smooth_q=True, smooth_k=True)
    o2 = sa.sage_attn_fwd(prep)
    torch.cuda.synchronize()
    sa.attn_get_device_status()
    assert torch.equal(o1, o2)
    check_attention(o1, inp, oracle.all_rows(1, 700, 3), "e4m3", "smooth_q + smooth_k", exact_gate=False,
                    smooth_k=True)


def test_smoothing_q_helps_offset_queries(cuda_dev):
    """Q with large per-channel offsets: the smoothed kernel output is clearly closer to the
    FP64 attention than the plain one (both through the 16-bit P V).  The gain is bounded:
    K's own INT8 error, which Q's (large) mean multiplies, remains."""
    inp = make_inputs(small_case(1, 4, 1024, 2800, q_channel_offset_std=4.0))
    g = to_device(inp, cuda_dev)
    plain = sa.sage_attention(g.q, g.k, g.v, pv="bf16")
    smooth = sa.sage_attention(g.q, g.k, g.v, pv="bf16", smooth_q=True)
    torch.cuda.synchronize()
    rows = oracle.all_rows(1, 1024, 4)
    exact = oracle.attention(inp.q, inp.k, inp.v, inp.wl.softmax_scale, rows=rows)
    e_plain = metrics(gather_rows(plain, rows), exact)["rel_l2"]
    e_smooth = metrics(gather_rows(smooth, rows), exact)["rel_l2"]
    print("rel-L2 plain", e_plain, "smoothed", e_smooth)
    assert e_smooth < 0.8 * e_plain


@pytest.mark.parametrize("name,n_rows", [("flux2048", 512), ("hunyuan720p", 384)])
def test_workload_attention_smooth_q(cuda_dev, workload_inputs, name, n_rows):
    cpu, g = workload_inputs(name)
    o = sa.sage_attention(g.q, g.k, g.v, softmax_scale=cpu.wl.softmax_scale, smooth_q=True, **kwargs(g, cpu.wl))
    torch.cuda.synchronize()
    sa.attn_get_device_status()
    rows = sample_rows(cpu.wl, n_rows, outlier_tokens=cpu.outlier_tokens)
    check_attention(o, cpu, rows, "e4m3", name)


def test_smooth_q_with_q_on_load_is_refused(cuda_dev):
    inp = make_inputs(small_case(1, 2, 64, 2900))
    g = to_device(inp, cuda_dev)
    with pytest.raises(sa.AttnError) as e:
        sa.sage_attention(g.q, g.k, g.v, smooth_q=True, q_on_load=True)
    assert e.value.status == 3
