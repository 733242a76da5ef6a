"""Parity of the Sage forward with a 16-bit P V product (sage_attn_fwd_pv16,
CUDA through the C ABI).

Two references from the oracle:
  * the exact value of its own format -- FP64 attention of the INT8 Q/K codes
    with V taken from the BF16 input (oracle.sage_attention_v16).  The kernel's
    arithmetic after the exact INT8 score product is that of the BF16 path
    (probabilities rounded to BF16, FP32 accumulation, BF16 output), so it
    takes the BF16 path's gate: cosine >= 0.99999 and
    |O - O_fmt| <= 2e-2 + 2^-7 A|V| (tests/parity.py);
  * FP64 attention of the BF16 inputs: the Sage gates (cosine >= 0.995, max-abs
    <= 0.1 and the Sage op's band), on the Wan-720p workload the format's own
    floor (x8 outlier tokens) as in the FP8 mode's tests.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import sage_attention_forward_gb300 as sa
from parity import (BF16_A, BF16_B, assert_bf16_gate, assert_sage_exact_gate, gather_rows, metrics)
from workloads import make_inputs, sample_rows, small_case, to_device

pytestmark = pytest.mark.gpu


def run(g, wl, smooth_k=False):
    kw = {}
    if g.q_norm_w is not None:
        kw.update(q_norm_w=g.q_norm_w, k_norm_w=g.k_norm_w, rms_eps=wl.rms_eps)
    if g.rope_cos is not None:
        kw.update(rope_cos=g.rope_cos, rope_sin=g.rope_sin, rope_dim=wl.rope_dim)
    return sa.sage_attention(g.q, g.k, g.v, softmax_scale=wl.softmax_scale, pv="bf16", smooth_k=smooth_k, **kw)


def check(o, cpu, rows, what, exact_gate=True, smooth_k=False):
    wl = cpu.wl
    prep = oracle.prepare(cpu.q, cpu.k, cpu.v, wl.softmax_scale, q_norm_w=cpu.q_norm_w, k_norm_w=cpu.k_norm_w,
                          rms_eps=wl.rms_eps, rope_cos=cpu.rope_cos, rope_sin=cpu.rope_sin, rope_dim=wl.rope_dim,
                          smooth_k=smooth_k)
    fmt = oracle.sage_attention_v16(prep, cpu.v, rows)
    fmt_abs = oracle.sage_attention_v16(prep, cpu.v, rows, abs_v=True)
    q, k = prep["q_pre"], prep["k_pre"]
    exact = oracle.attention(q, k, cpu.v, wl.softmax_scale, rows=rows)
    got = gather_rows(o, rows)
    m_fmt = metrics(got, fmt, fmt_abs, BF16_A, BF16_B)
    m_exact = metrics(got, exact)
    m_floor = metrics(fmt, exact)
    print(what, "vs format:", m_fmt, "\n   vs exact:", m_exact, "\n   format vs exact:", m_floor)
    assert_bf16_gate(m_fmt, what)
    if exact_gate:
        assert_sage_exact_gate(m_exact, what)
    else:
        assert m_exact["cos"] >= m_floor["cos"] - 0.001, f"{what}: {m_exact} vs format floor {m_floor}"
    return m_exact


@pytest.mark.parametrize("B,H,S", [(1, 1, 1), (1, 2, 31), (2, 3, 129), (1, 2, 300), (1, 3, 1000)])
def test_small_and_ragged_shapes_full(cuda_dev, B, H, S):
    inp = make_inputs(small_case(B, H, S, 700 + S))
    g = to_device(inp, cuda_dev)
    o = run(g, inp.wl)
    torch.cuda.synchronize()
    sa.attn_get_device_status()
    check(o, inp, oracle.all_rows(B, S, H), f"pv16 B{B} H{H} S{S}")


def test_single_key_returns_value(cuda_dev):
    # one key: every probability is 1 (exactly representable), so O = V exactly
    inp = make_inputs(small_case(2, 3, 1, 6))
    g = to_device(inp, cuda_dev)
    o = run(g, inp.wl)
    torch.cuda.synchronize()
    assert torch.equal(o.cpu(), inp.v)


def test_norm_rope_and_smoothing(cuda_dev):
    inp = make_inputs(small_case(1, 2, 500, 741, rms_norm=True, rope_dim=64, k_channel_offset_std=1.0))
    g = to_device(inp, cuda_dev)
    o = run(g, inp.wl, smooth_k=True)
    torch.cuda.synchronize()
    check(o, inp, oracle.all_rows(1, 500, 2), "pv16 norm+rope64 smooth_k", smooth_k=True)


@pytest.mark.parametrize("name,n_rows", [("flux1024", 1024), ("wan720p", 512), ("hunyuan720p", 384)])
def test_dit_workloads_sampled_rows(cuda_dev, workload_inputs, name, n_rows):
    cpu, g = workload_inputs(name)
    o = run(g, cpu.wl)
    torch.cuda.synchronize()
    sa.attn_get_device_status()
    rows = sample_rows(cpu.wl, n_rows, outlier_tokens=cpu.outlier_tokens)
    check(o, cpu, rows, name, exact_gate=(name != "wan720p"))


def test_more_accurate_than_the_fp8_mode(cuda_dev):
    inp = make_inputs(small_case(1, 2, 2000, 751))
    g = to_device(inp, cuda_dev)
    o16 = run(g, inp.wl)
    o8 = sa.sage_attention(g.q, g.k, g.v)
    torch.cuda.synchronize()
    rows = oracle.all_rows(1, 2000, 2)[::7]
    exact = oracle.attention(inp.q, inp.k, inp.v, inp.wl.softmax_scale, rows=rows)
    e16 = metrics(gather_rows(o16, rows), exact)["rel_l2"]
    e8 = metrics(gather_rows(o8, rows), exact)["rel_l2"]
    assert e16 < 0.8 * e8, (e16, e8)


def test_deterministic_and_non_default_stream(cuda_dev):
    inp = make_inputs(small_case(1, 4, 1500, 761))
    g = to_device(inp, cuda_dev)
    prep = sa.sage_prepare(g.q, g.k, g.v)
    o1 = sa.sage_attn_fwd_pv16(prep, g.v)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o2 = sa.sage_attn_fwd_pv16(prep, g.v, stream=s)
    s.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)
