"""The failure path on the GPU: a kernel whose wait runs out returns with the
timeout recorded, and the context stays usable (CUDA through the C ABI).

attn_selftest_wait_timeout launches the BF16 attention kernel with its loads
withheld, so nothing ever completes the barrier its MMA warp waits on; the wait
gives up after the 2 s limit, the kernel tears down and returns, and the host
reads ATTN_ERR_DEVICE_TIMEOUT.  No fault, trap or hang is involved.
"""
import math

import pytest
import torch

import oracle
import sage_attention_forward_gb300 as sa
from parity import BF16_A, BF16_B, assert_bf16_gate, metrics
from workloads import make_inputs, small_case, to_device

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_the_context_survives(cuda_dev):
    assert sa.attn_selftest_wait_timeout(cuda_dev) == "ATTN_ERR_DEVICE_TIMEOUT"
    # the error word was cleared by the read: the next status is clean
    sa.attn_get_device_status()
    # and the same context still computes correctly
    inp = make_inputs(small_case(1, 2, 300, 1301))
    g = to_device(inp, cuda_dev)
    o = sa.attn_fwd_bf16(g.q, g.k, g.v)
    torch.cuda.synchronize()
    sa.attn_get_device_status()
    rows = oracle.all_rows(1, 300, 2)
    ref = oracle.attention(inp.q, inp.k, inp.v, 1 / math.sqrt(128), rows=rows)
    ref_abs = oracle.attention(inp.q, inp.k, inp.v.abs(), 1 / math.sqrt(128), rows=rows)
    m = metrics(o.reshape(-1, 128), ref, ref_abs, BF16_A, BF16_B)
    assert_bf16_gate(m, "after the self-test")
    # a second self-test behaves the same
    assert sa.attn_selftest_wait_timeout(cuda_dev) == "ATTN_ERR_DEVICE_TIMEOUT"
