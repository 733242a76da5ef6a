"""sage_prepare_noalloc: the prepare stage for callers that cannot allocate.

Some callers cannot call cudaMalloc when they run us -- their device memory is
owned and budgeted by a host framework or engine, they must not risk an
out-of-memory error or the device-wide synchronisation an allocation can cause
mid-step, or they are plug-ins handed only their input and output buffers.
This entry point takes no workspace: its scratch is a fixed array inside the
library.  These tests check, through the C ABI, that it writes exactly what
sage_prepare (which takes a caller-allocated workspace) writes, on two calls in
a row with different shapes, at its full capacity (2048 heads, the last slot
of the fixed array in use) followed by a small call, and that calls beyond its
fixed capacity, or with output buffers that do not match the inputs, are
refused before anything is launched.  This file is collected last on purpose.
"""
import ctypes
import math

import pytest
import torch

import sage_attention_forward_gb300 as sa
from workloads import make_inputs, small_case, to_device

I64x3 = ctypes.c_int64 * 3
FIELDS = ("q_i8", "k_i8", "v_fp8", "q_scale", "k_scale", "v_scale")


def _both(inp, dev):
    g = to_device(inp, dev)
    kw = {}
    if g.q_norm_w is not None:
        kw.update(q_norm_w=g.q_norm_w, k_norm_w=g.k_norm_w, rms_eps=inp.wl.rms_eps)
    if g.rope_cos is not None:
        kw.update(rope_cos=g.rope_cos, rope_sin=g.rope_sin, rope_dim=inp.wl.rope_dim)
    ref = sa.sage_prepare(g.q, g.k, g.v, softmax_scale=inp.wl.softmax_scale, **kw)
    out = sa.Prepared.empty(inp.wl.B, inp.wl.H, inp.wl.S, ref.S_pad, dev)
    for t in (out.q_i8, out.k_i8, out.v_fp8):
        t.fill_(0x55)                      # garbage in the outputs must not survive
    sa.sage_prepare_noalloc(g.q, g.k, g.v, out, softmax_scale=inp.wl.softmax_scale, **kw)
    torch.cuda.synchronize()
    sa.attn_get_device_status()
    return ref, out


@pytest.mark.gpu
def test_matches_sage_prepare_on_two_calls_in_a_row(cuda_dev):
    # first call: fused RMSNorm + RoPE, several heads; second call: a different,
    # ragged shape -- the shared scratch must not carry anything over
    first = make_inputs(small_case(2, 3, 300, 901, rms_norm=True, rope_dim=64))
    second = make_inputs(small_case(1, 5, 129, 902))
    for inp in (first, second):
        ref, out = _both(inp, cuda_dev)
        for name in FIELDS:
            a, b = getattr(ref, name), getattr(out, name)
            if a.dtype == torch.float32:
                assert torch.equal(a.view(torch.int32), b.view(torch.int32)), name
            else:
                assert torch.equal(a, b), name


@pytest.mark.gpu
def test_matches_sage_prepare_at_capacity(cuda_dev):
    # B * H = 2048 heads fill the fixed scratch to its last slot; the ragged small call
    # after it must see none of those channel maxima
    for inp in (make_inputs(small_case(2, 1024, 40, 903)), make_inputs(small_case(1, 3, 77, 904))):
        ref, out = _both(inp, cuda_dev)
        for name in FIELDS:
            a, b = getattr(ref, name), getattr(out, name)
            if a.dtype == torch.float32:
                assert torch.equal(a.view(torch.int32), b.view(torch.int32)), name
            else:
                assert torch.equal(a, b), name


@pytest.mark.gpu
def test_refuses_outputs_made_for_other_shapes(cuda_dev):
    # a Prepared made at set-up time for fewer heads or a shorter sequence would be written
    # past its ends: the binding refuses it before the library is called
    inp = make_inputs(small_case(1, 4, 300, 905))
    g = to_device(inp, cuda_dev)
    S_pad = sa.sage_padded_len(300)
    for B, H, S, Sp in ((1, 3, 300, S_pad), (1, 4, 200, sa.sage_padded_len(200)), (1, 4, 299, S_pad)):
        small = sa.Prepared.empty(B, H, S, Sp, cuda_dev)
        with pytest.raises(sa.AttnError):
            sa.sage_prepare_noalloc(g.q, g.k, g.v, small)
    ok = sa.Prepared.empty(1, 4, 300, S_pad, cuda_dev)
    ok.v_scale = ok.v_scale.to(torch.float64)
    with pytest.raises(sa.AttnError):
        sa.sage_prepare_noalloc(g.q, g.k, g.v, ok)


def test_refuses_more_heads_than_its_scratch_holds():
    # validation runs on the host before any CUDA call, so this needs no GPU;
    # the pointers are never dereferenced
    L = sa.lib()
    fake = 0x10000
    B, H, S = 1, 2049, 64
    st = I64x3(S * H * 128, H * 128, 128)
    status = L.sage_prepare_noalloc(fake, fake, fake, B, S, H, 128, st, st, st, 1 / math.sqrt(128), None, None,
                                    1e-6, None, None, 0, 128, fake, fake, fake, fake, fake, fake, None)
    assert status == 1
    assert "2048" in L.attn_last_error().decode()
