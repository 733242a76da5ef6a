"""GB300 (sm_103a) attention forward: BF16 flash attention and the Sage
INT8/FP8 variant, behind the C ABI declared in include/sageattn.h.

This module only marshals torch tensors into the C calls of
_build/libsageattn.so (pointers, shapes, strides, the current CUDA stream);
every step of the computation runs in the library's CUDA kernels.  Output and
scratch buffers the caller does not pass are allocated with torch.  If the
library has not been built, every call raises.

    attn_fwd_bf16(q, k, v)            -> O                 (BF16 [B, S, H, 128])
    sage_prepare(q, k, v, ...)        -> Prepared           (INT8 Q/K, e4m3 V, scales)
    sage_attn_fwd(prepared, S)        -> O
    sage_attention(q, k, v, ...)      -> O                 (prepare + fwd)
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass

import torch

from .build import LIB as _LIB_PATH

__all__ = ["AttnError", "attn_fwd_bf16", "sage_prepare", "sage_prepare_noalloc", "sage_attn_fwd", "sage_attention",
           "Prepared", "e4m3_encode",
           "sage_padded_len", "attn_get_device_status", "lib", "STATUS"]

STATUS = {0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_ALIGNMENT", 3: "ATTN_ERR_UNSUPPORTED",
          4: "ATTN_ERR_CUDA", 5: "ATTN_ERR_DEVICE_TIMEOUT"}


class AttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status
        self.name = STATUS.get(status, str(status))


_lib = None
_I64x3 = ctypes.c_int64 * 3
_vp = ctypes.c_void_p


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"CUDA library not built ({_LIB_PATH} missing): run `python -c 'import "
                               f"__graft_entry__ as g; g.build()'` first")
        L = ctypes.CDLL(_LIB_PATH)
        i = ctypes.c_int
        L.attn_fwd_bf16.argtypes = [_vp, _vp, _vp, _vp, i, i, i, i, _I64x3, _I64x3, _I64x3, _I64x3, ctypes.c_float, _vp]
        L.attn_fwd_bf16.restype = i
        L.sage_padded_len.argtypes = [ctypes.c_int64]
        L.sage_padded_len.restype = ctypes.c_int64
        L.sage_prepare_workspace_size.argtypes = [i, i]
        L.sage_prepare_workspace_size.restype = ctypes.c_size_t
        L.sage_prepare.argtypes = [_vp, _vp, _vp, i, i, i, i, _I64x3, _I64x3, _I64x3, ctypes.c_float, _vp, _vp,
                                   ctypes.c_float, _vp, _vp, i, ctypes.c_int64, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                   ctypes.c_size_t, _vp]
        L.sage_prepare.restype = i
        L.sage_prepare_smooth_k_workspace_size.argtypes = [i, i, ctypes.c_int64]
        L.sage_prepare_smooth_k_workspace_size.restype = ctypes.c_size_t
        L.sage_prepare_smooth_k.argtypes = [_vp, _vp, _vp, i, i, i, i, _I64x3, _I64x3, _I64x3, ctypes.c_float, _vp,
                                            _vp, ctypes.c_float, _vp, _vp, i, ctypes.c_int64, _vp, _vp, _vp, _vp,
                                            _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
        L.sage_prepare_smooth_k.restype = i
        L.sage_prepare_noalloc.argtypes = [_vp, _vp, _vp, i, i, i, i, _I64x3, _I64x3, _I64x3, ctypes.c_float, _vp,
                                           _vp, ctypes.c_float, _vp, _vp, i, ctypes.c_int64, _vp, _vp, _vp, _vp, _vp,
                                           _vp, _vp]
        L.sage_prepare_noalloc.restype = i
        L.sage_attn_workspace_size.argtypes = [i, i, ctypes.c_int64]
        L.sage_attn_workspace_size.restype = ctypes.c_size_t
        L.sage_attn_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _I64x3, i, i, i, i, ctypes.c_int64, _vp,
                                    ctypes.c_size_t, _vp]
        L.sage_attn_fwd.restype = i
        L.sage_attn_fwd_pv16.argtypes = [_vp, _vp, _vp, _vp, _vp, _I64x3, _vp, _I64x3, i, i, i, i, ctypes.c_int64,
                                         _vp, ctypes.c_size_t, _vp]
        L.sage_attn_fwd_pv16.restype = i
        L.sage_attention_workspace_size.argtypes = [i, i, ctypes.c_int64, i, i, i]
        L.sage_attention_workspace_size.restype = ctypes.c_size_t
        L.sage_attention.argtypes = [_vp, _vp, _vp, i, i, i, i, _I64x3, _I64x3, _I64x3, ctypes.c_float, _vp, _vp,
                                     ctypes.c_float, _vp, _vp, i, i, i, i, i, _vp, _I64x3, _vp, ctypes.c_size_t, _vp]
        L.sage_prepare_smoothed.argtypes = [_vp, _vp, _vp, i, i, i, i, _I64x3, _I64x3, _I64x3, ctypes.c_float, _vp,
                                            _vp, ctypes.c_float, _vp, _vp, i, ctypes.c_int64, i, i, _vp, _vp, _vp,
                                            _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
        L.sage_prepare_smoothed.restype = i
        L.sage_attn_fwd_smooth_q.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _I64x3, i, i, i, i,
                                             ctypes.c_int64, _vp, ctypes.c_size_t, _vp]
        L.sage_attn_fwd_smooth_q.restype = i
        L.sage_attn_fwd_pv16_smooth_q.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _I64x3, _vp, _I64x3, i, i, i, i,
                                                  ctypes.c_int64, _vp, ctypes.c_size_t, _vp]
        L.sage_attn_fwd_pv16_smooth_q.restype = i
        L.sage_attention.restype = i
        L.attn_selftest_wait_timeout.argtypes = [_vp, _vp, _vp, _vp, _vp]
        L.attn_selftest_wait_timeout.restype = i
        L.attn_sm_clock_sample.argtypes = [_vp, i, _vp]
        L.attn_sm_clock_sample.restype = i
        L.sage_e4m3_encode.argtypes = [_vp, _vp, ctypes.c_int64, _vp]
        L.sage_e4m3_encode.restype = i
        L.attn_get_device_status.argtypes = [_vp]
        L.attn_get_device_status.restype = i
        L.attn_last_error.argtypes = []
        L.attn_last_error.restype = ctypes.c_char_p
        L.attn_status_name.argtypes = [i]
        L.attn_status_name.restype = ctypes.c_char_p
        _lib = L
    return _lib


def _check(status: int):
    if status != 0:
        raise AttnError(status, lib().attn_last_error().decode(errors="replace"))


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _bshd(name: str, t: torch.Tensor):
    if t.dim() != 4:
        raise ValueError(f"{name} must be [B, S, H, D], got {tuple(t.shape)}")
    if t.dtype != torch.bfloat16:
        raise ValueError(f"{name} must be bfloat16, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.stride(3) != 1:
        raise ValueError(f"{name} must have unit channel stride")
    sb, ss, sh, _ = t.stride()
    return _I64x3(sb, ss, sh)


def sage_padded_len(S: int) -> int:
    return int(lib().sage_padded_len(S))


def attn_fwd_bf16(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor | None = None,
                  softmax_scale: float | None = None, stream=None) -> torch.Tensor:
    """O = softmax(softmax_scale * Q K^T) V for BF16 [B, S, H, 128] (any 16-byte-multiple strides)."""
    B, S, H, D = q.shape
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, S, H, D), dtype=torch.bfloat16, device=q.device)
    qs, ks, vs, os_ = _bshd("q", q), _bshd("k", k), _bshd("v", v), _bshd("out", out)
    _check(lib().attn_fwd_bf16(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, S, H, D, qs, ks, vs,
                               os_, float(softmax_scale), _stream_ptr(stream)))
    return out


@dataclass
class Prepared:
    """Outputs of sage_prepare (device tensors, layouts of include/sageattn.h)."""
    q_i8: torch.Tensor      # int8  [B, H, S_pad, 128]
    k_i8: torch.Tensor      # int8  [B, H, S_pad, 128]
    v_fp8: torch.Tensor     # uint8 [B, H, 128, S_pad] (e4m3 bit patterns)
    q_scale: torch.Tensor   # fp32  [B, H, S_pad / 32]
    k_scale: torch.Tensor   # fp32  [B, H, S_pad / 32]
    v_scale: torch.Tensor   # fp32  [B, H, 128]
    S: int
    S_pad: int
    k_mean: torch.Tensor | None = None   # fp32 [B, H, 128], set when K was smoothed
    q_mean: torch.Tensor | None = None   # fp16 [B, H, S_pad / 32, 128], set when Q was smoothed: each
                                         # block's mean in units of its step

    @staticmethod
    def empty(B: int, H: int, S: int, S_pad: int, device) -> "Prepared":
        return Prepared(torch.empty((B, H, S_pad, 128), dtype=torch.int8, device=device),
                        torch.empty((B, H, S_pad, 128), dtype=torch.int8, device=device),
                        torch.empty((B, H, 128, S_pad), dtype=torch.uint8, device=device),
                        torch.empty((B, H, S_pad // 32), dtype=torch.float32, device=device),
                        torch.empty((B, H, S_pad // 32), dtype=torch.float32, device=device),
                        torch.empty((B, H, 128), dtype=torch.float32, device=device), S, S_pad)


def _check_prepared(out: Prepared, q: torch.Tensor, S_pad: int | None = None) -> None:
    """A caller-supplied Prepared must match q's batch, heads and length: the kernels write
    through its pointers with the sizes these imply."""
    B, S, H, _ = q.shape
    S_pad = out.S_pad if S_pad is None else S_pad
    if out.S != S or out.S_pad != S_pad:
        raise AttnError(1, f"out was made for S={out.S}, S_pad={out.S_pad}; this call has S={S}, S_pad={S_pad}")
    want = {"q_i8": ((B, H, S_pad, 128), torch.int8), "k_i8": ((B, H, S_pad, 128), torch.int8),
            "v_fp8": ((B, H, 128, S_pad), torch.uint8), "q_scale": ((B, H, S_pad // 32), torch.float32),
            "k_scale": ((B, H, S_pad // 32), torch.float32), "v_scale": ((B, H, 128), torch.float32)}
    if out.k_mean is not None:
        want["k_mean"] = ((B, H, 128), torch.float32)
    if out.q_mean is not None:
        want["q_mean"] = ((B, H, S_pad // 32, 128), torch.float16)
    for name, (shape, dtype) in want.items():
        t = getattr(out, name)
        if tuple(t.shape) != shape or t.dtype != dtype:
            raise AttnError(1, f"out.{name} is {tuple(t.shape)} {t.dtype}, expected {shape} {dtype}")
        if t.device != q.device:
            raise AttnError(1, f"out.{name} is on {t.device}, q on {q.device}")
        if not t.is_contiguous():
            raise AttnError(1, f"out.{name} must be contiguous")


def prepare_workspace(B: int, H: int, device, S_pad: int | None = None, smooth_k: bool = False) -> torch.Tensor:
    if smooth_k:
        n = int(lib().sage_prepare_smooth_k_workspace_size(B, H, int(S_pad)))
    else:
        n = int(lib().sage_prepare_workspace_size(B, H))
    return torch.empty(n, dtype=torch.uint8, device=device)


def attn_workspace(B: int, H: int, S_pad: int, device) -> torch.Tensor:
    return torch.empty(int(lib().sage_attn_workspace_size(B, H, S_pad)), dtype=torch.uint8, device=device)


def sage_prepare(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, softmax_scale: float | None = None,
                 S_pad: int | None = None, q_norm_w: torch.Tensor | None = None,
                 k_norm_w: torch.Tensor | None = None, rms_eps: float = 1e-6, rope_cos: torch.Tensor | None = None,
                 rope_sin: torch.Tensor | None = None, rope_dim: int = 0, out: Prepared | None = None,
                 workspace: torch.Tensor | None = None, stream=None, smooth_k: bool = False,
                 smooth_q: bool = False) -> Prepared:
    """Quantise Q/K to INT8 and V to e4m3 (optionally RMSNorm + RoPE on Q/K first;
    with smooth_k, K's per-channel token mean is subtracted before quantising K
    and returned in out.k_mean; with smooth_q, each 32-row block's mean is
    subtracted from Q and returned, in step units, in out.q_mean)."""
    B, S, H, D = q.shape
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if S_pad is None:
        S_pad = sage_padded_len(S)
    if out is None:
        out = Prepared.empty(B, H, S, S_pad, q.device)
    if smooth_k and out.k_mean is None:
        out.k_mean = torch.empty((B, H, 128), dtype=torch.float32, device=q.device)
    if smooth_q and out.q_mean is None:
        out.q_mean = torch.empty((B, H, S_pad // 32, 128), dtype=torch.float16, device=q.device)
    if not smooth_q:
        out.q_mean = None
    _check_prepared(out, q, S_pad)
    if workspace is None:
        workspace = prepare_workspace(B, H, q.device, S_pad, smooth_k)
    qs, ks, vs = _bshd("q", q), _bshd("k", k), _bshd("v", v)

    def ptr(t):
        return None if t is None else t.data_ptr()

    if smooth_q:
        _check(lib().sage_prepare_smoothed(q.data_ptr(), k.data_ptr(), v.data_ptr(), B, S, H, D, qs, ks, vs,
                                           float(softmax_scale), ptr(q_norm_w), ptr(k_norm_w), float(rms_eps),
                                           ptr(rope_cos), ptr(rope_sin), int(rope_dim), int(S_pad), 1, int(smooth_k),
                                           out.q_i8.data_ptr(), out.k_i8.data_ptr(), out.v_fp8.data_ptr(),
                                           out.q_scale.data_ptr(), out.k_scale.data_ptr(), out.v_scale.data_ptr(),
                                           out.q_mean.data_ptr(), ptr(out.k_mean) if smooth_k else None,
                                           workspace.data_ptr(), workspace.numel(), _stream_ptr(stream)))
        return out
    if smooth_k:
        _check(lib().sage_prepare_smooth_k(q.data_ptr(), k.data_ptr(), v.data_ptr(), B, S, H, D, qs, ks, vs,
                                           float(softmax_scale), ptr(q_norm_w), ptr(k_norm_w), float(rms_eps),
                                           ptr(rope_cos), ptr(rope_sin), int(rope_dim), int(S_pad),
                                           out.q_i8.data_ptr(), out.k_i8.data_ptr(), out.v_fp8.data_ptr(),
                                           out.q_scale.data_ptr(), out.k_scale.data_ptr(), out.v_scale.data_ptr(),
                                           out.k_mean.data_ptr(), workspace.data_ptr(), workspace.numel(),
                                           _stream_ptr(stream)))
        return out
    _check(lib().sage_prepare(q.data_ptr(), k.data_ptr(), v.data_ptr(), B, S, H, D, qs, ks, vs,
                              float(softmax_scale), ptr(q_norm_w), ptr(k_norm_w), float(rms_eps), ptr(rope_cos),
                              ptr(rope_sin), int(rope_dim), int(S_pad), out.q_i8.data_ptr(), out.k_i8.data_ptr(),
                              out.v_fp8.data_ptr(), out.q_scale.data_ptr(), out.k_scale.data_ptr(),
                              out.v_scale.data_ptr(), workspace.data_ptr(), workspace.numel(), _stream_ptr(stream)))
    return out


def sage_prepare_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: Prepared,
                         softmax_scale: float | None = None, q_norm_w: torch.Tensor | None = None,
                         k_norm_w: torch.Tensor | None = None, rms_eps: float = 1e-6,
                         rope_cos: torch.Tensor | None = None, rope_sin: torch.Tensor | None = None,
                         rope_dim: int = 0, stream=None) -> Prepared:
    """sage_prepare for callers that cannot allocate device memory at call time.

    The library call allocates nothing: the caller passes every output buffer
    (`out`, e.g. from Prepared.empty at set-up time) and the scratch comes from a
    fixed 1 MiB array inside the library, so B * H is limited to 2048 heads.
    Calls on one device share that array: order calls that could overlap on the
    GPU, and make the first call on a device before capturing a stream.
    """
    B, S, H, D = q.shape
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    qs, ks, vs = _bshd("q", q), _bshd("k", k), _bshd("v", v)
    _check_prepared(out, q)

    def ptr(t):
        return None if t is None else t.data_ptr()

    _check(lib().sage_prepare_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), B, S, H, D, qs, ks, vs,
                                      float(softmax_scale), ptr(q_norm_w), ptr(k_norm_w), float(rms_eps),
                                      ptr(rope_cos), ptr(rope_sin), int(rope_dim), int(out.S_pad),
                                      out.q_i8.data_ptr(), out.k_i8.data_ptr(), out.v_fp8.data_ptr(),
                                      out.q_scale.data_ptr(), out.k_scale.data_ptr(), out.v_scale.data_ptr(),
                                      _stream_ptr(stream)))
    return out


def sage_attn_fwd(prep: Prepared, out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                  stream=None) -> torch.Tensor:
    """Attention on prepared tensors -> BF16 [B, S, H, 128]."""
    B, H, S_pad, D = prep.q_i8.shape
    S = prep.S
    if out is None:
        out = torch.empty((B, S, H, D), dtype=torch.bfloat16, device=prep.q_i8.device)
    if workspace is None:
        workspace = attn_workspace(B, H, S_pad, prep.q_i8.device)
    os_ = _bshd("out", out)
    if prep.q_mean is not None:
        _check(lib().sage_attn_fwd_smooth_q(prep.q_i8.data_ptr(), prep.q_mean.data_ptr(), prep.k_i8.data_ptr(),
                                            prep.v_fp8.data_ptr(), prep.q_scale.data_ptr(), prep.k_scale.data_ptr(),
                                            prep.v_scale.data_ptr(), out.data_ptr(), os_, B, S, H, D, int(S_pad),
                                            workspace.data_ptr(), workspace.numel(), _stream_ptr(stream)))
        return out
    _check(lib().sage_attn_fwd(prep.q_i8.data_ptr(), prep.k_i8.data_ptr(), prep.v_fp8.data_ptr(),
                               prep.q_scale.data_ptr(), prep.k_scale.data_ptr(), prep.v_scale.data_ptr(),
                               out.data_ptr(), os_, B, S, H, D, int(S_pad), workspace.data_ptr(), workspace.numel(),
                               _stream_ptr(stream)))
    return out


def sage_attn_fwd_pv16(prep: Prepared, v: torch.Tensor, out: torch.Tensor | None = None,
                       workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Attention on prepared INT8 Q/K with a 16-bit P V product: P in BF16 times
    the BF16 input v [B, S, H, 128] (not quantised) -> BF16 [B, S, H, 128]."""
    B, H, S_pad, D = prep.q_i8.shape
    S = prep.S
    if out is None:
        out = torch.empty((B, S, H, D), dtype=torch.bfloat16, device=prep.q_i8.device)
    if workspace is None:
        workspace = attn_workspace(B, H, S_pad, prep.q_i8.device)
    vs, os_ = _bshd("v", v), _bshd("out", out)
    if prep.q_mean is not None:
        _check(lib().sage_attn_fwd_pv16_smooth_q(prep.q_i8.data_ptr(), prep.q_mean.data_ptr(), prep.k_i8.data_ptr(),
                                                 prep.q_scale.data_ptr(), prep.k_scale.data_ptr(), v.data_ptr(), vs,
                                                 out.data_ptr(), os_, B, S, H, D, int(S_pad), workspace.data_ptr(),
                                                 workspace.numel(), _stream_ptr(stream)))
        return out
    _check(lib().sage_attn_fwd_pv16(prep.q_i8.data_ptr(), prep.k_i8.data_ptr(), prep.q_scale.data_ptr(),
                                    prep.k_scale.data_ptr(), v.data_ptr(), vs, out.data_ptr(), os_, B, S, H, D,
                                    int(S_pad), workspace.data_ptr(), workspace.numel(), _stream_ptr(stream)))
    return out


def _on_load_level(q_on_load: bool, k_on_load: bool) -> int:
    """0: the prepare codes Q and K; 1: the forward codes Q; 2: the forward codes Q and K."""
    return 2 if k_on_load else int(bool(q_on_load))


def sage_attention_workspace(B: int, H: int, S: int, device, smooth_k: bool = False, pv: str = "e4m3",
                             q_on_load: bool = False, k_on_load: bool = False) -> torch.Tensor:
    n = int(lib().sage_attention_workspace_size(B, H, sage_padded_len(S), int(smooth_k), int(pv == "bf16"),
                                                _on_load_level(q_on_load, k_on_load)))
    return torch.empty(n, dtype=torch.uint8, device=device)


def sage_attention(q, k, v, softmax_scale=None, q_norm_w=None, k_norm_w=None, rms_eps=1e-6, rope_cos=None,
                   rope_sin=None, rope_dim=0, out=None, stream=None, smooth_k=False, pv="e4m3",
                   workspace=None, q_on_load=False, smooth_q=False, k_on_load=False) -> torch.Tensor:
    """Prepare + attention in one library call: the SageAttention-style forward of BF16 Q/K/V.

    pv="e4m3": P and V in FP8; pv="bf16": P in BF16 times the unquantised V.  The
    prepared tensors stay in `workspace` (allocated here unless given).  q_on_load:
    Q is coded by the forward as it loads it instead of by the prepare (the same
    output; slower on a GB300).  k_on_load: the forward codes K (and Q) too, per tile,
    so neither reaches memory as codes (with pv="bf16" nothing is prepared at all);
    every CTA of a head then codes all its K tiles, which is slower at every size.
    smooth_q / smooth_k: block-mean smoothing of Q (with its correction term) /
    sequence-mean smoothing of K before INT8."""
    if pv not in ("e4m3", "bf16"):
        raise ValueError(f"pv must be 'e4m3' or 'bf16', not {pv!r}")
    B, S, H, D = q.shape
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, S, H, D), dtype=torch.bfloat16, device=q.device)
    if workspace is None:
        workspace = sage_attention_workspace(B, H, S, q.device, smooth_k, pv, q_on_load, k_on_load)
    qs, ks, vs, os_ = _bshd("q", q), _bshd("k", k), _bshd("v", v), _bshd("out", out)

    def ptr(t):
        return None if t is None else t.data_ptr()

    _check(lib().sage_attention(q.data_ptr(), k.data_ptr(), v.data_ptr(), B, S, H, D, qs, ks, vs,
                                float(softmax_scale), ptr(q_norm_w), ptr(k_norm_w), float(rms_eps), ptr(rope_cos),
                                ptr(rope_sin), int(rope_dim), int(bool(smooth_q)), int(bool(smooth_k)), int(pv == "bf16"),
                                _on_load_level(q_on_load, k_on_load), out.data_ptr(), os_, workspace.data_ptr(),
                                workspace.numel(), _stream_ptr(stream)))
    return out


def attn_selftest_wait_timeout(device=None, stream=None) -> str:
    """Run the library's failure-path self-test on `device` (about 2 s): a kernel
    whose loads are withheld must give up on its bounded wait and report it.
    Returns the status name; "ATTN_ERR_DEVICE_TIMEOUT" means the path works."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    bufs = [torch.zeros((1, 128, 1, 128), dtype=torch.bfloat16, device=dev) for _ in range(4)]
    code = lib().attn_selftest_wait_timeout(*(b.data_ptr() for b in bufs), _stream_ptr(stream))
    return STATUS.get(code, str(code))


def e4m3_encode(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """e4m3 codes (uint8, x's shape) of a float32 CUDA tensor: nearest even, saturating
    at +-448, through the conversion the prepare's V pass and the FP8 P V use."""
    if x.dtype != torch.float32 or not x.is_cuda:
        raise ValueError("x must be a float32 CUDA tensor")
    x = x.contiguous()
    if out is None:
        out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    elif out.dtype != torch.uint8 or out.shape != x.shape or not out.is_contiguous() or out.device != x.device:
        raise ValueError("out must be a contiguous uint8 tensor of x's shape on x's device")
    _check(lib().sage_e4m3_encode(x.data_ptr(), out.data_ptr(), x.numel(), _stream_ptr(stream)))
    return out


def sm_clock_sample(out: torch.Tensor, stream=None) -> torch.Tensor:
    """Enqueue a sample of every SM's cycle counter and the GPU's nanosecond timer into
    out (int64 [n_slots, 2] on the device, n_slots >= the SM count): timing
    instrumentation, see attn_sm_clock_sample in include/sageattn.h."""
    if out.dtype != torch.int64 or out.dim() != 2 or out.shape[1] != 2 or not out.is_contiguous() or not out.is_cuda:
        raise ValueError("out must be a contiguous CUDA int64 tensor [n_slots, 2]")
    _check(lib().attn_sm_clock_sample(out.data_ptr(), out.shape[0], _stream_ptr(stream)))
    return out


def sm_clock_mhz(a, b) -> float | None:
    """Median over SMs of the average SM clock (MHz) between two host copies of
    sm_clock_sample outputs; None if no SM appears in both."""
    import numpy as np
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    ok = (a[:, 0] > 0) & (b[:, 0] > 0) & (b[:, 1] > a[:, 1])
    if not ok.any():
        return None
    return float(np.median((b[ok, 0] - a[ok, 0]) / (b[ok, 1] - a[ok, 1]) * 1e3))


def attn_get_device_status(stream=None) -> None:
    """Synchronise the stream and raise AttnError if a kernel gave up on a bounded wait."""
    _check(lib().attn_get_device_status(_stream_ptr(stream)))
