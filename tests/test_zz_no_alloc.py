"""sage_prepare_noalloc: the prepare stage for callers that cannot allocate.

Some callers cannot call cudaMalloc when they run us -- their device memory is
owned and budgeted by a host framework or engine, they must not risk an
out-of-memory error or the device-wide synchronisation an allocation can cause
mid-step, or they are plug-ins handed only their input and output buffers.
This entry point takes no workspace: its scratch is a fixed array inside the
library.  These tests check, through the C ABI, that it writes exactly what
sage_prepare (which takes a caller-allocated workspace) writes, on two calls in
a row with different shapes, at its full capacity (2048 heads, the last slot
of the fixed array in use) followed by a small call, in a second CUDA context of
the same device (the array's address belongs to the library as loaded in one
context, so each context looks its own up), and that calls beyond its fixed
capacity, or with output buffers that do not match the inputs, are refused
before anything is launched.  This file is collected last on purpose.
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


SECOND_CONTEXT = r"""
import ctypes, math, sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
import sage_attention_forward_gb300 as sa
from workloads import make_inputs, small_case

inp = make_inputs(small_case(2, 3, 200, 906))
B, S, H = 2, 200, 3
S_pad = sa.sage_padded_len(S)
dev = torch.device("cuda:0")
q, k, v = (t.to(dev) for t in (inp.q, inp.k, inp.v))
ref = sa.Prepared.empty(B, H, S, S_pad, dev)
sa.sage_prepare_noalloc(q, k, v, ref)          # the primary context: its own address lookup
torch.cuda.synchronize()

cu = ctypes.CDLL("libcuda.so.1")
def ok(r, what):
    assert r == 0, f"{what}: CUresult {r}"
ctx = ctypes.c_void_p()
ok(cu.cuCtxCreate_v2(ctypes.byref(ctx), 0, 0), "cuCtxCreate")      # a second context on device 0
ok(cu.cuCtxPushCurrent_v2(ctx), "cuCtxPushCurrent")
bufs = []
def alloc(nbytes):
    p = ctypes.c_uint64()
    ok(cu.cuMemAlloc_v2(ctypes.byref(p), ctypes.c_size_t(nbytes)), "cuMemAlloc")
    bufs.append(p.value)
    return p.value
def upload(t):
    a = np.ascontiguousarray(t.contiguous().view(torch.int16).numpy())
    p = alloc(a.nbytes)
    ok(cu.cuMemcpyHtoD_v2(ctypes.c_uint64(p), a.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(a.nbytes)), "HtoD")
    return p
dq, dk, dv = upload(inp.q), upload(inp.k), upload(inp.v)
shapes = {"q_i8": (B * H * S_pad * 128, np.int8), "k_i8": (B * H * S_pad * 128, np.int8),
          "v_fp8": (B * H * 128 * S_pad, np.uint8), "q_scale": (B * H * S_pad // 32, np.float32),
          "k_scale": (B * H * S_pad // 32, np.float32), "v_scale": (B * H * 128, np.float32)}
outs = {n: alloc(c * np.dtype(t).itemsize) for n, (c, t) in shapes.items()}
st = (ctypes.c_int64 * 3)(S * H * 128, H * 128, 128)
L = sa.lib()
r = L.sage_prepare_noalloc(dq, dk, dv, B, S, H, 128, st, st, st, 1 / math.sqrt(128), None, None, 1e-6, None, None,
                           0, S_pad, outs["q_i8"], outs["k_i8"], outs["v_fp8"], outs["q_scale"], outs["k_scale"],
                           outs["v_scale"], None)
assert r == 0, L.attn_last_error()
ok(cu.cuCtxSynchronize(), "cuCtxSynchronize")
for n, (c, t) in shapes.items():
    host = np.empty(c, dtype=t)
    ok(cu.cuMemcpyDtoH_v2(host.ctypes.data_as(ctypes.c_void_p), ctypes.c_uint64(outs[n]), ctypes.c_size_t(host.nbytes)),
       "DtoH")
    want = getattr(ref, n).cpu().numpy().reshape(-1)
    assert np.array_equal(host.view(np.uint8), want.view(np.uint8)), n
for p in bufs:
    cu.cuMemFree_v2(ctypes.c_uint64(p))
ok(cu.cuCtxPopCurrent_v2(ctypes.byref(ctypes.c_void_p())), "cuCtxPopCurrent")
ok(cu.cuCtxDestroy_v2(ctx), "cuCtxDestroy")
# back in the primary context, where the address looked up first still serves
again = sa.Prepared.empty(B, H, S, S_pad, dev)
sa.sage_prepare_noalloc(q, k, v, again)
torch.cuda.synchronize()
assert all(torch.equal(getattr(ref, n), getattr(again, n)) for n in shapes)
print("second context ok")
"""


@pytest.mark.gpu
def test_second_context_on_the_same_device(cuda_dev, tmp_path):
    # run in a process of its own: it creates and destroys a driver context
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    script = tmp_path / "second_context.py"
    script.write_text(SECOND_CONTEXT)
    r = subprocess.run([sys.executable, str(script), root], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "second context ok" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]


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
