"""CPU oracle for the attention forward and the Sage prepare.

TEST INFRASTRUCTURE ONLY: tests/, the smoke check and the benchmark's CPU
baseline call it; the product library never does.  It shares no code with
the CUDA path.  The arithmetic lives in oracle.c (plain C, FP64 attention,
binary32 quantisation written step by step); this module only marshals
torch/numpy arrays into it.

Functions and the passages they follow:
  attention      -- O = softmax(scale Q K^T) V in FP64, the `naive` form of the
                    ai-infra handbook chapter "Kernel acceleration: attention,
                    compilation and fusion" (section "Attention: from O(N^2)
                    memory to blocks").
  norm_rope      -- RMSNorm then rotate-half RoPE of a Q or K row, with the
                    BF16 rounding points of PyTorch's eager ops (aiter pull request
                    "gfx1201_sage_prepare / gfx1201_sage_attention",
                    gfx1201_sage_prepare commit message).
  quant_qk       -- INT8 codes for Q or K, each 32-row block of a (batch,
                    head) with its own FP32 scale; Q's scales also hold
                    softmax_scale*log2(e) (same pull request, Technical Details).
  k_mean         -- K smoothing: the per-(batch, head, channel) mean of K over
                    its tokens, subtracted before quantising K (ai-infra
                    handbook chapter above, section "SageAttention:
                    quantizing attention too").
  quant_q_smooth -- Q smoothing (same section): each 32-row block's mean is
                    subtracted before quantising Q and kept, in units of the
                    block's step, as binary16 values that the score product
                    adds back (the correction term qbar . k).
  quant_v        -- e4m3 codes for V, stored channel-major [B, H, 128, S_pad],
                    each channel with its own FP32 scale (same pull request,
                    Technical Details).
  prepare        -- the three above in order, as the prepare stage runs them.
  sage_attention -- FP64 attention evaluated on prepared tensors: the exact
                    value of the INT8/e4m3 format the Sage forward consumes
                    (same pull request, commit message of
                    gfx1201_sage_attention), with no further rounding.
  sage_attention_v16 -- the same with V taken from the BF16 input (the Sage
                    mode whose P V product is 16-bit: "P and V ... in FP8
                    or FP16", ai-infra handbook chapter above, section
                    "SageAttention: quantizing attention too").
  e4m3_encode / e4m3_decode / f32_to_bf16 -- the scalar encoders.
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np
import torch

from . import build as _build

_lib = None

LOG2E = 1.4426950408889634  # log2(e) as a binary64 constant


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        c_p = ctypes.c_void_p
        L.oracle_attention.argtypes = [c_p, c_p, c_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_double, c_p, ctypes.c_int64, c_p, ctypes.c_int]
        L.oracle_norm_rope.argtypes = [c_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, c_p, ctypes.c_float,
                                       c_p, c_p, ctypes.c_int, c_p]
        L.oracle_quant_qk.argtypes = [c_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                      ctypes.c_float, c_p, c_p, c_p]
        L.oracle_k_mean.argtypes = [c_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64, c_p]
        L.oracle_quant_v.argtypes = [c_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64, c_p, c_p]
        L.oracle_quant_q_smooth.argtypes = [c_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                            ctypes.c_float, c_p, c_p, c_p]
        L.oracle_f16_encode_array.argtypes = [c_p, c_p, ctypes.c_int64]
        L.oracle_f16_decode.argtypes = [ctypes.c_uint16]
        L.oracle_f16_decode.restype = ctypes.c_double
        L.oracle_e4m3_encode_array.argtypes = [c_p, c_p, ctypes.c_int64]
        L.oracle_e4m3_decode_array.argtypes = [c_p, c_p, ctypes.c_int64]
        L.oracle_f32_to_bf16_array.argtypes = [c_p, c_p, ctypes.c_int64]
        L.oracle_sage_attention.argtypes = [c_p, c_p, c_p, c_p, c_p, c_p, c_p, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int64, c_p, ctypes.c_int64, ctypes.c_int,
                                            ctypes.c_int, c_p, ctypes.c_int]
        L.oracle_sage_attention_v16.argtypes = [c_p, c_p, c_p, c_p, c_p, c_p, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_int, ctypes.c_int64, c_p, ctypes.c_int64, ctypes.c_int, c_p,
                                                ctypes.c_int]
        L.oracle_num_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def _bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Contiguous [.., 128]-ordered BF16 tensor -> numpy uint16 bit patterns."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def softmax_log2_factor(softmax_scale: float) -> float:
    """fl32(softmax_scale * log2 e), the factor Q's INT8 scale carries."""
    return float(np.float32(float(np.float32(softmax_scale)) * LOG2E))


def attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, softmax_scale: float,
              rows: torch.Tensor | None = None, nthreads: int = 0) -> np.ndarray:
    """FP64 attention of BF16 [B, S, H, D] tensors (any strides).

    rows: optional int64 [n, 3] of (b, s, h) query rows; returns [n, D] float64.
    Without rows returns [B, S, H, D] float64.
    """
    B, S, H, D = q.shape
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    if rows is not None:
        r = rows.to(torch.int64)
        flat = ((r[:, 0] * S + r[:, 1]) * H + r[:, 2]).contiguous().numpy()
        out = np.empty((len(flat), D), dtype=np.float64)
        lib().oracle_attention(_ptr(qb), _ptr(kb), _ptr(vb), B, S, H, D, float(softmax_scale),
                               _ptr(flat), len(flat), _ptr(out), int(nthreads))
        return out
    out = np.empty((B, S, H, D), dtype=np.float64)
    lib().oracle_attention(_ptr(qb), _ptr(kb), _ptr(vb), B, S, H, D, float(softmax_scale),
                           None, 0, _ptr(out), int(nthreads))
    return out


def norm_rope(x: torch.Tensor, norm_w: torch.Tensor | None, eps: float,
              rope_cos: torch.Tensor | None, rope_sin: torch.Tensor | None, rope_dim: int) -> torch.Tensor:
    """RMSNorm (if norm_w) then rotate-half RoPE (if rope_dim) -> BF16 [B, S, H, 128]."""
    B, S, H, D = x.shape
    assert D == 128
    xb = _bf16_bits(x)
    out = np.empty_like(xb)
    wb = _bf16_bits(norm_w) if norm_w is not None else None
    cb = _bf16_bits(rope_cos) if rope_dim else None
    sb = _bf16_bits(rope_sin) if rope_dim else None
    lib().oracle_norm_rope(_ptr(xb), B, S, H, _ptr(wb) if wb is not None else None, float(eps),
                           _ptr(cb) if cb is not None else None, _ptr(sb) if sb is not None else None,
                           int(rope_dim), _ptr(out))
    return torch.from_numpy(out.view(np.int16)).view(torch.bfloat16).reshape(B, S, H, D)


def quant_qk(x: torch.Tensor, S_pad: int, scale_mult: float = 1.0, mean: torch.Tensor | None = None):
    """INT8 codes [B, H, S_pad, 128] and FP32 scales [B, H, S_pad/32]; with
    `mean` ([B, H, 128] float32) the value quantised is fl32(x - mean)."""
    B, S, H, D = x.shape
    xb = _bf16_bits(x)
    codes = np.empty((B, H, S_pad, 128), dtype=np.int8)
    scales = np.empty((B, H, S_pad // 32), dtype=np.float32)
    mb = None
    if mean is not None:
        mb = np.ascontiguousarray(mean.to(torch.float32).numpy())
        assert mb.shape == (B, H, 128)
    lib().oracle_quant_qk(_ptr(xb), B, S, H, int(S_pad), float(np.float32(scale_mult)),
                          _ptr(mb) if mb is not None else None, _ptr(codes), _ptr(scales))
    return torch.from_numpy(codes), torch.from_numpy(scales)


def k_mean(x: torch.Tensor, S_pad: int) -> torch.Tensor:
    """Per-(batch, head, channel) mean of K over its S tokens, float32 [B, H, 128],
    summed in the order oracle.c documents (K smoothing)."""
    B, S, H, D = x.shape
    xb = _bf16_bits(x)
    out = np.empty((B, H, 128), dtype=np.float32)
    lib().oracle_k_mean(_ptr(xb), B, S, H, int(S_pad), _ptr(out))
    return torch.from_numpy(out)


def quant_q_smooth(x: torch.Tensor, S_pad: int, scale_mult: float):
    """Q smoothing: INT8 codes of fl32(x - block mean) [B, H, S_pad, 128], FP32 scales
    [B, H, S_pad/32] (carrying scale_mult) and the block means in units of the block's
    step as binary16 bit patterns (int16 tensor) [B, H, S_pad/32, 128]."""
    B, S, H, D = x.shape
    xb = _bf16_bits(x)
    codes = np.empty((B, H, S_pad, 128), dtype=np.int8)
    scales = np.empty((B, H, S_pad // 32), dtype=np.float32)
    mean16 = np.empty((B, H, S_pad // 32, 128), dtype=np.uint16)
    lib().oracle_quant_q_smooth(_ptr(xb), B, S, H, int(S_pad), float(np.float32(scale_mult)), _ptr(codes),
                                _ptr(scales), _ptr(mean16))
    return torch.from_numpy(codes), torch.from_numpy(scales), torch.from_numpy(mean16.view(np.int16))


def f16_encode(x: np.ndarray) -> np.ndarray:
    """binary64 -> binary16 bit patterns (uint16), nearest-even."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().oracle_f16_encode_array(_ptr(x), _ptr(out), x.size)
    return out


def f16_decode(h) -> float:
    return float(lib().oracle_f16_decode(int(h) & 0xFFFF))


def quant_v(x: torch.Tensor, S_pad: int):
    """e4m3 codes (uint8) [B, H, 128, S_pad] and FP32 scales [B, H, 128]."""
    B, S, H, D = x.shape
    xb = _bf16_bits(x)
    codes = np.empty((B, H, 128, S_pad), dtype=np.uint8)
    scales = np.empty((B, H, 128), dtype=np.float32)
    lib().oracle_quant_v(_ptr(xb), B, S, H, int(S_pad), _ptr(codes), _ptr(scales))
    return torch.from_numpy(codes), torch.from_numpy(scales)


def padded_len(S: int) -> int:
    """Smallest multiple of 128 that is >= S (the sequence length of the prepared tensors)."""
    return ((S + 127) // 128) * 128


def prepare(q, k, v, softmax_scale, S_pad=None, q_norm_w=None, k_norm_w=None, rms_eps=1e-6,
            rope_cos=None, rope_sin=None, rope_dim=0, smooth_k=False, smooth_q=False):
    """The Sage prepare stage: optional norm/RoPE of Q and K, optional K
    smoothing (subtract k_mean before quantising K), optional Q smoothing
    (subtract each block's mean, kept as q_mean16), then the quantisers.

    Returns a dict with q_i8, k_i8, v_fp8 (uint8), q_scale, k_scale, v_scale,
    the BF16 Q/K that were quantised (q_pre, k_pre), k_mean (None unless
    smooth_k) and q_mean16 (None unless smooth_q).
    """
    B, S, H, D = q.shape
    if S_pad is None:
        S_pad = padded_len(S)
    q_pre, k_pre = q, k
    if q_norm_w is not None or rope_dim:
        q_pre = norm_rope(q, q_norm_w, rms_eps, rope_cos, rope_sin, rope_dim)
        k_pre = norm_rope(k, k_norm_w, rms_eps, rope_cos, rope_sin, rope_dim)
    c = softmax_log2_factor(softmax_scale)
    qm = None
    if smooth_q:
        q_i8, q_scale, qm = quant_q_smooth(q_pre, S_pad, c)
    else:
        q_i8, q_scale = quant_qk(q_pre, S_pad, c)
    km = k_mean(k_pre, S_pad) if smooth_k else None
    k_i8, k_scale = quant_qk(k_pre, S_pad, 1.0, km)
    v_fp8, v_scale = quant_v(v, S_pad)
    return dict(q_i8=q_i8, k_i8=k_i8, v_fp8=v_fp8, q_scale=q_scale, k_scale=k_scale, v_scale=v_scale,
                q_pre=q_pre.contiguous(), k_pre=k_pre.contiguous(), S_pad=S_pad, log2_factor=c, k_mean=km,
                q_mean16=qm)


def _q_mean_arg(prep):
    qm = prep.get("q_mean16")
    return None if qm is None else np.ascontiguousarray(qm.numpy().view(np.uint16))


def sage_attention(prep: dict, S: int, rows: torch.Tensor, H: int, abs_v: bool = False, p_e4m3: bool = False,
                   nthreads: int = 0) -> np.ndarray:
    """FP64 attention of the prepared codes (dict as returned by prepare(), CPU
    tensors) for query rows (b, s, h) -> [n, 128] float64.  p_e4m3 also rounds
    the probabilities to e4m3 (448 * w) in the numerator, as the FP8 P V product
    of the Sage forward needs; abs_v weights |V| instead of V.  With Q smoothing
    (prep["q_mean16"]) Q's operand is f16(code + mean16), see oracle.c."""
    q8 = np.ascontiguousarray(prep["q_i8"].numpy())
    k8 = np.ascontiguousarray(prep["k_i8"].numpy())
    v8 = np.ascontiguousarray(prep["v_fp8"].numpy())
    qs = np.ascontiguousarray(prep["q_scale"].numpy())
    ks = np.ascontiguousarray(prep["k_scale"].numpy())
    vs = np.ascontiguousarray(prep["v_scale"].numpy())
    B, _, S_pad, _ = q8.shape
    r = rows.to(torch.int64)
    flat = ((r[:, 0] * S + r[:, 1]) * H + r[:, 2]).contiguous().numpy()
    out = np.empty((len(flat), 128), dtype=np.float64)
    qm = _q_mean_arg(prep)
    lib().oracle_sage_attention(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(qs), _ptr(ks), _ptr(vs),
                                _ptr(qm) if qm is not None else None, B, S, H, int(S_pad),
                                _ptr(flat), len(flat), int(abs_v), int(p_e4m3), _ptr(out), int(nthreads))
    return out


def sage_attention_v16(prep: dict, v: torch.Tensor, rows: torch.Tensor, abs_v: bool = False,
                       nthreads: int = 0) -> np.ndarray:
    """FP64 attention of the prepared INT8 Q/K codes with V taken from the BF16
    input v [B, S, H, 128] (the Sage mode with a 16-bit P V product), for query
    rows (b, s, h) -> [n, 128] float64."""
    q8 = np.ascontiguousarray(prep["q_i8"].numpy())
    k8 = np.ascontiguousarray(prep["k_i8"].numpy())
    qs = np.ascontiguousarray(prep["q_scale"].numpy())
    ks = np.ascontiguousarray(prep["k_scale"].numpy())
    B, S, H, D = v.shape
    vb = _bf16_bits(v)
    S_pad = q8.shape[2]
    r = rows.to(torch.int64)
    flat = ((r[:, 0] * S + r[:, 1]) * H + r[:, 2]).contiguous().numpy()
    out = np.empty((len(flat), 128), dtype=np.float64)
    qm = _q_mean_arg(prep)
    lib().oracle_sage_attention_v16(_ptr(q8), _ptr(k8), _ptr(qs), _ptr(ks), _ptr(qm) if qm is not None else None,
                                    _ptr(vb), B, S, H, int(S_pad), _ptr(flat), len(flat), int(abs_v), _ptr(out),
                                    int(nthreads))
    return out


def all_rows(B: int, S: int, H: int) -> torch.Tensor:
    """Every (b, s, h) query row, in [B, S, H] order."""
    b, s, h = torch.meshgrid(torch.arange(B), torch.arange(S), torch.arange(H), indexing="ij")
    return torch.stack([b.flatten(), s.flatten(), h.flatten()], dim=1)


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().oracle_e4m3_encode_array(_ptr(x), _ptr(out), x.size)
    return out


def e4m3_decode(c: np.ndarray) -> np.ndarray:
    c = np.ascontiguousarray(c, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    lib().oracle_e4m3_decode_array(_ptr(c), _ptr(out), c.size)
    return out


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """binary32 -> BF16 bit patterns (uint16), nearest-even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().oracle_f32_to_bf16_array(_ptr(x), _ptr(out), x.size)
    return out


def dequantized(prep: dict, S: int):
    """FP64 tensors the prepared codes stand for, in [B, S, H, 128] order.

    Q's scale carries softmax_scale*log2(e); dividing it back out gives the
    quantised Q in the units of the input.  Used only for diagnostics (the
    error floor the format itself sets).
    """
    c = prep["log2_factor"]
    q8 = prep["q_i8"].double()
    k8 = prep["k_i8"].double()
    B, H, S_pad, D = q8.shape
    qs = prep["q_scale"].double().repeat_interleave(32, dim=2)[..., None] / c
    ks = prep["k_scale"].double().repeat_interleave(32, dim=2)[..., None]
    qd = (q8 * qs)[:, :, :S].permute(0, 2, 1, 3)
    kd = (k8 * ks)[:, :, :S].permute(0, 2, 1, 3)
    vv = torch.from_numpy(e4m3_decode(prep["v_fp8"].numpy()))  # [B, H, 128, S_pad]
    vd = (vv * prep["v_scale"].double()[..., None])[..., :S].permute(0, 3, 1, 2)
    return qd, kd, vd
