"""Parity of attn_fwd_bf16 (CUDA, through the C ABI) with the FP64 oracle.

Small and ragged shapes are compared on every element; the DiT-shaped
workloads on sampled rows (every row of the ragged last tile, outlier tokens
where the workload has them, the rest uniform), run in the launch
configuration the benchmark times.  Gate: cosine >= 0.99999 and
|O - O_ref| <= 2e-2 + 2^-7 A|V| elementwise (derivation in tests/parity.py);
on inputs without x8 outlier tokens also the stated max-abs <= 2e-2 itself.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import sage_attention_forward_gb300 as sa
from parity import BF16_A, BF16_B, assert_bf16_gate, assert_bf16_raw, gather_rows, metrics
from workloads import make_inputs, sample_rows, small_case, to_device, wide_bf16, WORKLOADS

pytestmark = pytest.mark.gpu


def reference(q, k, v, scale, rows=None):
    """FP64 attention and the attention-weighted mean |V| (the rounding bound's scale)."""
    return (oracle.attention(q, k, v, scale, rows=rows), oracle.attention(q, k, v.abs(), scale, rows=rows))


def check(o, q, k, v, scale, what, rows=None, raw=True):
    """raw: also assert max-abs <= 2e-2 (inputs without outlier-dominated rows)."""
    ref, av = reference(q, k, v, scale, rows)
    m = metrics(o if rows is None else gather_rows(o, rows), ref, av, BF16_A, BF16_B)
    print(what, m)
    assert_bf16_gate(m, what)
    if raw:
        assert_bf16_raw(m, what)
    return m


@pytest.mark.parametrize("B,H,S", [(1, 1, 1), (1, 2, 31), (1, 1, 128), (2, 3, 129), (1, 2, 200), (1, 1, 256),
                                   (2, 2, 300), (1, 3, 513), (1, 2, 1000)])
def test_small_and_ragged_shapes_full(cuda_dev, B, H, S):
    inp = make_inputs(small_case(B, H, S, 100 + S))
    g = to_device(inp, cuda_dev)
    o = sa.attn_fwd_bf16(g.q, g.k, g.v)
    torch.cuda.synchronize()
    sa.attn_get_device_status()
    check(o, inp.q, inp.k, inp.v, 1 / math.sqrt(128), f"B{B} H{H} S{S}")


def test_single_key_returns_value(cuda_dev):
    inp = make_inputs(small_case(2, 3, 1, 5))
    g = to_device(inp, cuda_dev)
    o = sa.attn_fwd_bf16(g.q, g.k, g.v)
    assert torch.equal(o.cpu(), inp.v)


def test_tiny_workload_full(cuda_dev, workload_inputs):
    cpu, g = workload_inputs("tiny")
    o = sa.attn_fwd_bf16(g.q, g.k, g.v)
    check(o, cpu.q, cpu.k, cpu.v, cpu.wl.softmax_scale, "tiny")


@pytest.mark.parametrize("name,n_rows", [("flux1024", 2048), ("flux2048", 768), ("wan720p", 768), ("hunyuan720p", 512)])
def test_dit_workloads_sampled_rows(cuda_dev, workload_inputs, name, n_rows):
    cpu, g = workload_inputs(name)
    o = sa.attn_fwd_bf16(g.q, g.k, g.v)
    torch.cuda.synchronize()
    sa.attn_get_device_status()
    rows = sample_rows(cpu.wl, n_rows, outlier_tokens=cpu.outlier_tokens)
    # the Wan-720p workload's x8 outlier rows put the stated 2e-2 out of reach of any
    # kernel that rounds P to BF16 (tests/parity.py): there the derived bound alone
    check(o, cpu.q, cpu.k, cpu.v, cpu.wl.softmax_scale, name, rows=rows, raw=not cpu.wl.outlier_frac)


def test_permuted_output_layout(cuda_dev, workload_inputs):
    """Head-major storage for the output as well as the inputs (the [B, H, S, D] buffer seen as [B, S, H, D])."""
    cpu, g = workload_inputs("hunyuan720p")
    B, S, H, D = g.q.shape
    o_contig = sa.attn_fwd_bf16(g.q, g.k, g.v)
    o_store = torch.empty((B, H, S, D), dtype=torch.bfloat16, device=cuda_dev)
    o_perm = o_store.permute(0, 2, 1, 3)
    sa.attn_fwd_bf16(g.q, g.k, g.v, out=o_perm)
    torch.cuda.synchronize()
    assert torch.equal(o_perm, o_contig)


def test_deterministic_and_non_default_stream(cuda_dev):
    inp = make_inputs(small_case(1, 4, 3000, 9))
    g = to_device(inp, cuda_dev)
    o1 = sa.attn_fwd_bf16(g.q, g.k, g.v)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o2 = torch.empty_like(o1)
        sa.attn_fwd_bf16(g.q, g.k, g.v, out=o2, stream=s)
    s.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)


def test_key_value_permutation_changes_only_rounding(cuda_dev):
    """Reordering the K/V tokens leaves attention unchanged in exact arithmetic (aiter pull
    request, Test Result: the K/V-reversal noise floor); the kernel's result moves only by
    summation-order rounding, and both orders pass the gate."""
    inp = make_inputs(small_case(1, 2, 700, 11))
    g = to_device(inp, cuda_dev)
    o1 = sa.attn_fwd_bf16(g.q, g.k, g.v)
    rev = torch.arange(699, -1, -1)
    o2 = sa.attn_fwd_bf16(g.q, g.k[:, rev.to(cuda_dev)].contiguous(), g.v[:, rev.to(cuda_dev)].contiguous())
    check(o1, inp.q, inp.k, inp.v, 1 / math.sqrt(128), "forward order")
    check(o2, inp.q, inp.k, inp.v, 1 / math.sqrt(128), "reversed order")
    assert (o1.float() - o2.float()).abs().max().item() <= 2e-2


def test_other_softmax_scale(cuda_dev):
    inp = make_inputs(small_case(1, 2, 333, 12))
    g = to_device(inp, cuda_dev)
    for scale in (0.02, 0.3):
        o = sa.attn_fwd_bf16(g.q, g.k, g.v, softmax_scale=scale)
        # at scale 0.3 a row's weight sits on a few keys, |O| approaches max |V| and the
        # BF16 spacing of the output alone is up to 2^-6: the derived bound there
        check(o, inp.q, inp.k, inp.v, scale, f"scale {scale}", raw=scale < 0.1)


def test_device_status_is_clean(cuda_dev):
    sa.attn_get_device_status()


def test_saturated_softmax_large_logits(cuda_dev):
    """Query rows scaled by 2^4 to 2^10 next to ordinary ones: logits up to ~2000 (log2
    units), a softmax that is one-hot to BF16 precision, where the row maximum and the
    lazily moved reference decide everything.  Within the BF16 gate.  (Logits of 2^24 and
    beyond are outside the kernel's range: see the fused exponent argument.)"""
    S, H = 300, 2
    inp = make_inputs(small_case(1, H, S, 71))
    gain = torch.pow(2.0, torch.tensor([0.0, 4.0, 7.0, 10.0]).repeat_interleave(75)).view(1, S, 1, 1)
    inp.q = (inp.q.double() * gain).to(torch.bfloat16)
    g = to_device(inp, cuda_dev)
    o = sa.attn_fwd_bf16(g.q, g.k, g.v)
    torch.cuda.synchronize()
    sa.attn_get_device_status()
    check(o, inp.q, inp.k, inp.v, 1 / math.sqrt(128), "logits up to ~2000", raw=False)
