"""Parity of the Sage path (sage_prepare + sage_attn_fwd, CUDA through the C ABI)
with the FP64 oracle attention.  Gate: cosine >= 0.995 and
max |O - O_ref| / max(1, |O_ref|) <= 0.1, plus the secondary band of the Sage
op's test plan (see tests/parity.py).  The reference is the exact attention of
the BF16 inputs (after the oracle's RMSNorm + RoPE where the workload fuses
them)."""
import math

import numpy as np
import pytest
import torch

import oracle
import sage_attention_forward_gb300 as sa
from parity import assert_sage_gate, gather_rows, metrics
from workloads import make_inputs, sample_rows, small_case, to_device

pytestmark = pytest.mark.gpu


def sage(g, wl):
    kw = {}
    if g.q_norm_w is not None:
        kw.update(q_norm_w=g.q_norm_w, k_norm_w=g.k_norm_w, rms_eps=wl.rms_eps)
    if g.rope_cos is not None:
        kw.update(rope_cos=g.rope_cos, rope_sin=g.rope_sin, rope_dim=wl.rope_dim)
    return sa.sage_attention(g.q, g.k, g.v, softmax_scale=wl.softmax_scale, **kw)


def reference_inputs(cpu):
    q, k = cpu.q, cpu.k
    if cpu.q_norm_w is not None or cpu.wl.rope_dim:
        q = oracle.norm_rope(q, cpu.q_norm_w, cpu.wl.rms_eps, cpu.rope_cos, cpu.rope_sin, cpu.wl.rope_dim)
        k = oracle.norm_rope(k, cpu.k_norm_w, cpu.wl.rms_eps, cpu.rope_cos, cpu.rope_sin, cpu.wl.rope_dim)
    return q, k, cpu.v


@pytest.mark.parametrize("B,H,S", [(1, 1, 1), (1, 2, 31), (2, 3, 129), (1, 2, 200), (2, 2, 300), (1, 3, 513),
                                   (1, 2, 1000)])
def test_small_and_ragged_shapes_full(cuda_dev, B, H, S):
    inp = make_inputs(small_case(B, H, S, 400 + S))
    g = to_device(inp, cuda_dev)
    o = sage(g, inp.wl)
    torch.cuda.synchronize()
    sa.attn_get_device_status()
    ref = oracle.attention(inp.q, inp.k, inp.v, 1 / math.sqrt(128))
    m = metrics(o, ref)
    print((B, H, S), m)
    assert_sage_gate(m, f"B{B} H{H} S{S}")


def test_tiny_workload_full(cuda_dev, workload_inputs):
    cpu, g = workload_inputs("tiny")
    o = sage(g, cpu.wl)
    ref = oracle.attention(cpu.q, cpu.k, cpu.v, cpu.wl.softmax_scale)
    m = metrics(o, ref)
    print("tiny", m)
    assert_sage_gate(m, "tiny")


@pytest.mark.parametrize("name,n_rows", [("flux1024", 2048), ("flux2048", 768), ("wan720p", 768), ("hunyuan720p", 512)])
def test_dit_workloads_sampled_rows(cuda_dev, workload_inputs, name, n_rows):
    cpu, g = workload_inputs(name)
    o = sage(g, cpu.wl)
    torch.cuda.synchronize()
    sa.attn_get_device_status()
    rows = sample_rows(cpu.wl, n_rows, outlier_tokens=cpu.outlier_tokens)
    q, k, v = reference_inputs(cpu)
    ref = oracle.attention(q, k, v, cpu.wl.softmax_scale, rows=rows)
    m = metrics(gather_rows(o, rows), ref)
    print(name, m)
    assert_sage_gate(m, name)


def test_deterministic_and_non_default_stream(cuda_dev):
    inp = make_inputs(small_case(1, 4, 2000, 19))
    g = to_device(inp, cuda_dev)
    o1 = sa.sage_attention(g.q, g.k, g.v)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o2 = sa.sage_attention(g.q, g.k, g.v, stream=s)
    s.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)


def test_forward_on_oracle_prepared_tensors(cuda_dev):
    """sage_attn_fwd alone, fed the oracle's prepared tensors, matches the exact attention."""
    inp = make_inputs(small_case(2, 2, 400, 23))
    exp = oracle.prepare(inp.q, inp.k, inp.v, 1 / math.sqrt(128))
    prep = sa.Prepared(exp["q_i8"].to(cuda_dev), exp["k_i8"].to(cuda_dev), exp["v_fp8"].to(cuda_dev),
                       exp["q_scale"].to(cuda_dev), exp["k_scale"].to(cuda_dev), exp["v_scale"].to(cuda_dev),
                       400, exp["S_pad"])
    o = sa.sage_attn_fwd(prep)
    ref = oracle.attention(inp.q, inp.k, inp.v, 1 / math.sqrt(128))
    assert_sage_gate(metrics(o, ref), "oracle-prepared")


def test_device_status_is_clean(cuda_dev):
    sa.attn_get_device_status()
