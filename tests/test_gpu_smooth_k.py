"""K smoothing on the GPU (sage_prepare_smooth_k through the C ABI).

The prepare is bit-exact against the oracle: k_mean (binary32, in the
documented summation order), the INT8 codes and scales of K - k_mean, and Q/V
unchanged.  The attention of the smoothed prepare passes the same gates as the
plain Sage path: against the oracle's exact value of the smoothed format, and
against FP64 attention of the BF16 inputs.
"""
import math

import pytest
import torch

import oracle
import sage_attention_forward_gb300 as sa
from parity import assert_sage_exact_gate, assert_sage_format_gate, gather_rows, metrics, SAGE_A, SAGE_B
from workloads import make_inputs, sample_rows, small_case, to_device

pytestmark = pytest.mark.gpu

NAMES = ("q_i8", "k_i8", "v_fp8", "q_scale", "k_scale", "v_scale", "k_mean")


def kwargs(g, wl):
    kw = {}
    if g.q_norm_w is not None:
        kw.update(q_norm_w=g.q_norm_w, k_norm_w=g.k_norm_w, rms_eps=wl.rms_eps)
    if g.rope_cos is not None:
        kw.update(rope_cos=g.rope_cos, rope_sin=g.rope_sin, rope_dim=wl.rope_dim)
    return kw


def oracle_prepare(cpu, S_pad):
    wl = cpu.wl
    return oracle.prepare(cpu.q, cpu.k, cpu.v, wl.softmax_scale, S_pad=S_pad, q_norm_w=cpu.q_norm_w,
                          k_norm_w=cpu.k_norm_w, rms_eps=wl.rms_eps, rope_cos=cpu.rope_cos, rope_sin=cpu.rope_sin,
                          rope_dim=wl.rope_dim, smooth_k=True)


def assert_bit_exact(prep, exp, what):
    for name in NAMES:
        got = getattr(prep, name).cpu()
        ref = exp[name]
        same = torch.equal(got.view(torch.int32), ref.view(torch.int32)) if got.dtype == torch.float32 \
            else torch.equal(got, ref)
        if not same:
            diff = (got != ref)
            raise AssertionError(f"{what}: {name} differs at {int(diff.sum())} places, first "
                                 f"{diff.nonzero()[:5].tolist()}")


@pytest.mark.parametrize("B,H,S,kw", [
    (1, 1, 1, {}), (1, 3, 31, {}), (2, 2, 200, dict(k_channel_offset_std=2.0)), (1, 2, 1000, {}),
    (1, 3, 300, dict(rms_norm=True, rope_dim=64)), (2, 1, 129, dict(rope_dim=128)),
])
def test_prepare_smooth_k_bit_exact(cuda_dev, B, H, S, kw):
    inp = make_inputs(small_case(B, H, S, 500 + S, **kw))
    g = to_device(inp, cuda_dev)
    prep = sa.sage_prepare(g.q, g.k, g.v, softmax_scale=inp.wl.softmax_scale, smooth_k=True, **kwargs(g, inp.wl))
    torch.cuda.synchronize()
    assert_bit_exact(prep, oracle_prepare(inp, prep.S_pad), f"B{B} H{H} S{S} {kw}")


@pytest.mark.parametrize("name", ["flux1024", "wan720p"])
def test_workload_prepare_smooth_k_bit_exact(cuda_dev, workload_inputs, name):
    cpu, g = workload_inputs(name)
    prep = sa.sage_prepare(g.q, g.k, g.v, softmax_scale=cpu.wl.softmax_scale, smooth_k=True, **kwargs(g, cpu.wl))
    torch.cuda.synchronize()
    assert_bit_exact(prep, oracle_prepare(cpu, prep.S_pad), name)


def test_smoothing_leaves_q_and_v_alone(cuda_dev):
    inp = make_inputs(small_case(1, 2, 333, 77, k_channel_offset_std=1.0))
    g = to_device(inp, cuda_dev)
    a = sa.sage_prepare(g.q, g.k, g.v)
    b = sa.sage_prepare(g.q, g.k, g.v, smooth_k=True)
    torch.cuda.synchronize()
    for name in ("q_i8", "q_scale", "v_fp8", "v_scale"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    assert a.k_mean is None


def check_attention(o, cpu, rows, what, exact_gate=True):
    wl = cpu.wl
    prep = oracle_prepare(cpu, oracle.padded_len(wl.S))
    fmt = oracle.sage_attention(prep, wl.S, rows, wl.H)
    fmt_abs = oracle.sage_attention(prep, wl.S, rows, wl.H, abs_v=True)
    q, k = cpu.q, cpu.k
    if cpu.q_norm_w is not None or wl.rope_dim:
        q = oracle.norm_rope(q, cpu.q_norm_w, wl.rms_eps, cpu.rope_cos, cpu.rope_sin, wl.rope_dim)
        k = oracle.norm_rope(k, cpu.k_norm_w, wl.rms_eps, cpu.rope_cos, cpu.rope_sin, wl.rope_dim)
    exact = oracle.attention(q, k, cpu.v, wl.softmax_scale, rows=rows)
    got = gather_rows(o, rows)
    m_fmt = metrics(got, fmt, fmt_abs, SAGE_A, SAGE_B)
    m_exact = metrics(got, exact)
    print(what, "vs smoothed format:", m_fmt, "\n   vs exact:", m_exact)
    assert_sage_format_gate(m_fmt, what)
    if exact_gate:
        assert_sage_exact_gate(m_exact, what)
    return m_exact


@pytest.mark.parametrize("B,H,S", [(1, 2, 31), (2, 2, 300), (1, 3, 1000)])
def test_attention_smooth_k_small(cuda_dev, B, H, S):
    inp = make_inputs(small_case(B, H, S, 600 + S, k_channel_offset_std=1.0))
    g = to_device(inp, cuda_dev)
    o = sa.sage_attention(g.q, g.k, g.v, smooth_k=True)
    torch.cuda.synchronize()
    sa.attn_get_device_status()
    check_attention(o, inp, oracle.all_rows(B, S, H), f"smooth B{B} H{H} S{S}")


def test_attention_smooth_k_flux1024(cuda_dev, workload_inputs):
    """The FLUX 1024 workload (per-channel K offsets), sampled rows; smoothing
    does not lose accuracy against the plain Sage path there."""
    cpu, g = workload_inputs("flux1024")
    o_s = sa.sage_attention(g.q, g.k, g.v, softmax_scale=cpu.wl.softmax_scale, smooth_k=True)
    o_p = sa.sage_attention(g.q, g.k, g.v, softmax_scale=cpu.wl.softmax_scale)
    torch.cuda.synchronize()
    sa.attn_get_device_status()
    rows = sample_rows(cpu.wl, 1024)
    m_s = check_attention(o_s, cpu, rows, "flux1024 smooth_k")
    exact = oracle.attention(cpu.q, cpu.k, cpu.v, cpu.wl.softmax_scale, rows=rows)
    m_p = metrics(gather_rows(o_p, rows), exact)
    assert m_s["rel_l2"] <= m_p["rel_l2"] * 1.02, (m_s, m_p)
