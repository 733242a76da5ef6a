"""sage_attention, the one-call Sage op (CUDA through the C ABI), equals the
two-call sequence sage_prepare (+ smoothing) + sage_attn_fwd / sage_attn_fwd_pv16
bit for bit: its prepare writes the same codes, as FP16, straight into the
workspace the forward reads, and the forward kernel is the same.  (The two-call
path is checked against the oracle in test_gpu_prepare.py, test_gpu_sage.py,
test_gpu_sage_pv16.py and test_gpu_smooth_k.py.)"""
import pytest
import torch

import sage_attention_forward_gb300 as sa
from workloads import make_inputs, small_case, to_device

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


@pytest.mark.parametrize("pv", ["e4m3", "bf16"])
@pytest.mark.parametrize("smooth_k", [False, True])
@pytest.mark.parametrize("B,H,S,kw", [(1, 2, 31, {}), (2, 3, 300, dict(k_channel_offset_std=1.0)),
                                      (1, 2, 500, dict(rms_norm=True, rope_dim=64))])
def test_one_call_equals_two_calls(cuda_dev, B, H, S, kw, smooth_k, pv):
    inp = make_inputs(small_case(B, H, S, 1500 + S, **kw))
    g = to_device(inp, cuda_dev)
    o1 = sa.sage_attention(g.q, g.k, g.v, softmax_scale=inp.wl.softmax_scale, smooth_k=smooth_k, pv=pv,
                           **kwargs(g, inp.wl))
    o2 = two_calls(g, inp.wl, smooth_k, pv)
    torch.cuda.synchronize()
    sa.attn_get_device_status()
    assert torch.equal(o1, o2)


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
