"""Edge sizes through the C ABI on the GPU: an empty batch, and the largest grid.

* B = 0 or H = 0 has no query rows: every entry point returns at once with empty
  outputs (S = 0, attention over no keys, is an error: tests/test_abi.py).
* B * H = 65535 fills one grid column of heads; beyond it the attention kernels
  put heads on grid.z as well and the prepare runs one launch per group of whole
  batch entries.  Both sizes run all three attention modes and the prepare,
  checked against the oracle (the prepare on every head, the attention on rows
  of sampled heads, among them the first and last of each launch or grid slice).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import sage_attention_forward_gb300 as sa
from parity import (BF16_A, BF16_B, SAGE_A, SAGE_B, assert_bf16_gate, assert_sage_format_gate, gather_rows,
                    metrics)
from workloads import make_inputs, small_case, to_device

pytestmark = pytest.mark.gpu


def test_empty_batch(cuda_dev):
    q = torch.empty((0, 300, 2, 128), dtype=torch.bfloat16, device=cuda_dev)
    assert sa.attn_fwd_bf16(q, q, q).shape == (0, 300, 2, 128)
    prep = sa.sage_prepare(q, q, q)
    assert prep.q_i8.shape == (0, 2, 384, 128) and prep.v_scale.shape == (0, 2, 128)
    assert sa.sage_attn_fwd(prep).shape == (0, 300, 2, 128)
    assert sa.sage_attn_fwd_pv16(prep, q).shape == (0, 300, 2, 128)
    assert sa.sage_prepare(q, q, q, smooth_k=True).k_mean.shape == (0, 2, 128)
    h0 = torch.empty((1, 50, 0, 128), dtype=torch.bfloat16, device=cuda_dev)
    assert sa.attn_fwd_bf16(h0, h0, h0).shape == (1, 50, 0, 128)
    torch.cuda.synchronize()
    sa.attn_get_device_status()


@pytest.mark.parametrize("B,H,S,heads", [
    (1, 65535, 40, [0, 1, 12345, 40000, 65533, 65534]),
    # 75000 heads: grid.z slices of 65535 heads; prepare launches of batches {0, 1} and {2}
    (3, 25000, 8, [0, 24999, 25000, 49999, 50000, 65534, 65535, 65536, 74999]),
])
def test_largest_grid(cuda_dev, B, H, S, heads):
    inp = make_inputs(small_case(B, H, S, 1401))
    g = to_device(inp, cuda_dev)
    sm = 1 / math.sqrt(128)
    o = sa.attn_fwd_bf16(g.q, g.k, g.v)
    prep = sa.sage_prepare(g.q, g.k, g.v)
    o8 = sa.sage_attn_fwd(prep)
    o16 = sa.sage_attn_fwd_pv16(prep, g.v)
    o1 = sa.sage_attention(g.q, g.k, g.v)        # its prepare writes FP16 codes, also per launch group
    torch.cuda.synchronize()
    sa.attn_get_device_status()
    assert torch.equal(o1, o8)
    # prepare: bit-exact on every head
    exp = oracle.prepare(inp.q, inp.k, inp.v, sm)
    for name in ("q_i8", "k_i8", "v_fp8", "q_scale", "k_scale", "v_scale"):
        assert torch.equal(getattr(prep, name).cpu(), exp[name]), name
    # attention: every row of the sampled heads (flattened b * H + h)
    bh = torch.tensor(heads)
    rows = torch.stack([torch.stack([bh // H, torch.full_like(bh, s), bh % H], dim=1) for s in range(S)]).reshape(-1, 3)
    ref = oracle.attention(inp.q, inp.k, inp.v, sm, rows=rows)
    ref_abs = oracle.attention(inp.q, inp.k, inp.v.abs(), sm, rows=rows)
    assert_bf16_gate(metrics(gather_rows(o, rows), ref, ref_abs, BF16_A, BF16_B), f"BF16, {B * H} heads")
    fmt = oracle.sage_attention(exp, S, rows, H)
    fmt_abs = oracle.sage_attention(exp, S, rows, H, abs_v=True)
    assert_sage_format_gate(metrics(gather_rows(o8, rows), fmt, fmt_abs, SAGE_A, SAGE_B), f"Sage FP8, {B * H} heads")
    fmt16 = oracle.sage_attention_v16(exp, inp.v, rows)
    fmt16_abs = oracle.sage_attention_v16(exp, inp.v, rows, abs_v=True)
    assert_bf16_gate(metrics(gather_rows(o16, rows), fmt16, fmt16_abs, BF16_A, BF16_B), f"Sage 16-bit PV, {B * H} heads")
