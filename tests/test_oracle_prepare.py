"""Pins for the oracle's Sage prepare arithmetic (CPU only).

The scalar encoders are checked against torch's own casts (an independent
implementation) and against closed-form properties; the quantisers against
the invariants their definitions imply; RMSNorm and RoPE against FP64
evaluations within their rounding bounds and against the eager torch BF16
sequence the aiter pull request "gfx1201_sage_prepare /
gfx1201_sage_attention" names as the rounding model (gfx1201_sage_prepare
commit message).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from sage_attention_forward_gb300 import roofline
from workloads import make_inputs, rope_tables, small_case, WORKLOADS


# ------------------------------------------------------------------ BF16 rounding

def test_bf16_rounding_matches_torch_cast():
    g = np.random.default_rng(0)
    bits = g.integers(0, 2**32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x) & (np.abs(x) < 3.0e38)]
    mine = oracle.f32_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)


def test_bf16_rounding_ties_go_to_even():
    # exact midpoints between consecutive BF16 values: bf16 pattern p, plus half a step
    pats = np.arange(0x3f80, 0x3f90, dtype=np.uint32)
    mids = ((pats << 16) | 0x8000).view(np.float32)
    got = oracle.f32_to_bf16(mids)
    expect = np.where(pats % 2 == 0, pats, pats + 1).astype(np.uint16)
    assert np.array_equal(got, expect)


# ------------------------------------------------------------------ e4m3

def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert nan.sum() == 2                                   # S.1111.111
    assert np.array_equal(mine[~nan], ref[~nan])
    assert np.nanmax(mine) == 448.0 and mine[1] == 2.0 ** -9


def test_e4m3_encode_matches_torch_in_range():
    g = np.random.default_rng(1)
    # every BF16-representable value in (-448, 448), plus random binary32 patterns in range
    b = np.arange(0, 2**16, dtype=np.uint32)
    xb = (b << 16).view(np.float32)
    xr = g.uniform(-448, 448, size=500_000).astype(np.float32)
    xs = (g.standard_normal(500_000) * np.exp2(g.integers(-12, 8, 500_000))).astype(np.float32)
    x = np.concatenate([xb, xr, xs])
    x = x[np.isfinite(x) & (np.abs(x) < 448)]
    mine = oracle.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(mine, ref)


def test_e4m3_encode_matches_torch_on_every_binary32_below_448():
    """Every binary32 bit pattern of magnitude below 448, with both signs (2.27e9
    values, denormals and signed zeros included): the oracle's encoder against
    torch's float8_e4m3fn cast, nearest-even in that range (above it torch's cast
    does not saturate, so saturation is pinned separately)."""
    top = 0x43E00000                        # the bit pattern of 448.0
    chunk = 1 << 26
    for sign in (0, 0x80000000):
        for start in range(0, top, chunk):
            bits = np.arange(start, min(start + chunk, top), dtype=np.uint32) | np.uint32(sign)
            x = bits.view(np.float32)
            mine = oracle.e4m3_encode(x)
            ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            bad = np.flatnonzero(mine != ref)
            assert bad.size == 0, f"{bad.size} mismatches, the first at bits {int(bits[bad[0]]):#010x}"


def test_e4m3_midpoints_round_to_even_code():
    mags = oracle.e4m3_decode(np.arange(126, dtype=np.uint8))
    nxt = oracle.e4m3_decode(np.arange(1, 127, dtype=np.uint8))
    mids = ((mags + nxt) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (mags + nxt) / 2)   # midpoints are exact in binary32
    got = oracle.e4m3_encode(mids)
    lo = np.arange(126)
    expect = np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint8)
    assert np.array_equal(got, expect)
    assert np.array_equal(oracle.e4m3_encode(-mids), expect | 0x80)


def test_e4m3_saturates_above_range():
    x = np.array([448.0, 449.0, 464.0, 500.0, 1e6, 3e38, -450.0, -1e9], dtype=np.float32)
    got = oracle.e4m3_encode(x)
    assert np.array_equal(got, np.array([126, 126, 126, 126, 126, 126, 126 | 0x80, 126 | 0x80], dtype=np.uint8))


# ------------------------------------------------------------------ Q/K INT8

def test_qk_quant_block_invariants():
    inp = make_inputs(small_case(2, 3, 200, 21))
    S_pad = 256
    codes, scales = oracle.quant_qk(inp.k, S_pad, 1.0)
    x = inp.k.float().permute(0, 2, 1, 3)                  # [B, H, S, D]
    c = codes.float()
    for b in range(2):
        for h in range(3):
            for j in range(S_pad // 32):
                r0, r1 = 32 * j, min(32 * j + 32, 200)
                sc = scales[b, h, j].item()
                if r0 >= 200:
                    assert sc == 0.0 and (codes[b, h, r0:r0 + 32] == 0).all()
                    continue
                blk = x[b, h, r0:r1]
                a = blk.abs().max().item()
                assert sc == float(np.float32(np.float32(a) / np.float32(127)))
                # the element of largest magnitude maps to +-127
                idx = blk.abs().argmax()
                assert abs(c[b, h, r0:r1].flatten()[idx].item()) == 127
                # reconstruction error within half a step (plus binary32 rounding of the step)
                err = (blk - c[b, h, r0:r1] * sc).abs().max().item()
                assert err <= 0.5 * sc * (1 + 1e-5)
                assert (codes[b, h, r1:r0 + 32] == 0).all()      # padding rows
    assert codes.abs().max() <= 127


def test_qk_quant_ties_to_even_and_zero_block():
    # a block whose maximum is 127 has inv = 1 exactly, so x.5 values are exact ties
    x = torch.zeros(1, 64, 1, 128)
    x[0, 0, 0, 0] = 127
    x[0, 1, 0, :6] = torch.tensor([2.5, 3.5, -2.5, -3.5, 0.5, 1.5])
    xb = x.to(torch.bfloat16)
    codes, scales = oracle.quant_qk(xb, 128, 1.0)
    assert codes[0, 0, 1, :6].tolist() == [2, 4, -2, -4, 0, 2]
    assert scales[0, 0, 0].item() == 1.0
    assert scales[0, 0, 1].item() == 0.0 and (codes[0, 0, 32:] == 0).all()   # all-zero block


def test_q_scale_carries_log2e_softmax_factor():
    inp = make_inputs(small_case(1, 2, 64, 22))
    sm = 1 / math.sqrt(128)
    c = oracle.softmax_log2_factor(sm)
    assert c == float(np.float32(np.float32(sm) * math.log2(math.e)))
    q1, s1 = oracle.quant_qk(inp.q, 128, c)
    q0, s0 = oracle.quant_qk(inp.q, 128, 1.0)
    assert torch.equal(q1, q0)                               # codes do not depend on the factor
    assert torch.equal(s1, (s0 * torch.tensor(c, dtype=torch.float32)))


# ------------------------------------------------------------------ V e4m3

def test_v_quant_channel_invariants():
    inp = make_inputs(small_case(1, 2, 150, 23))
    S_pad = 256
    codes, scales = oracle.quant_v(inp.v, S_pad)
    assert codes.shape == (1, 2, 128, S_pad)
    x = inp.v.double().permute(0, 2, 3, 1)                   # [B, H, D, S]
    dec = torch.from_numpy(oracle.e4m3_decode(codes.numpy()))
    for h in range(2):
        a = x[0, h].abs().max(dim=1).values                   # per channel
        sc = scales[0, h].double()
        assert torch.equal(scales[0, h], (a.float() / 448.0))
        recon = dec[0, h, :, :150] * sc[:, None]
        rel = (recon - x[0, h]).abs() / torch.clamp(x[0, h].abs(), min=1e-30)
        normal = x[0, h].abs() >= 2.0 ** -6 * sc[:, None] * (1 + 1e-6)
        assert (rel[normal] <= 2.0 ** -4 * (1 + 1e-5)).all()  # half an e4m3 step, relative
        # the channel maximum encodes to +-448
        idx = x[0, h].abs().argmax(dim=1)
        top = codes[0, h, torch.arange(128), idx]
        assert ((top & 0x7f) == 126).all()
    assert (codes[..., 150:] == 0).all()


def test_v_quant_is_transposed():
    v = torch.zeros(1, 40, 2, 128)
    v[0, 17, 1, 93] = 3.0
    v[0, 5, 0, 2] = -1.0
    codes, scales = oracle.quant_v(v.to(torch.bfloat16), 128)
    assert codes[0, 1, 93, 17].item() == 126 and codes[0, 0, 2, 5].item() == 126 | 0x80
    assert int((codes != 0).sum()) == 2
    assert scales[0, 1, 93].item() == np.float32(3.0) / np.float32(448.0)
    assert scales[0, 0, 0].item() == 0.0


# ------------------------------------------------------------------ RMSNorm / RoPE

def _bf16_ulp(x):
    x = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(x, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def test_rmsnorm_within_rounding_bound_of_fp64():
    inp = make_inputs(WORKLOADS["flux2048"].__class__("n", 1, 3, 64, 31, rms_norm=True))
    x = inp.q
    w = inp.q_norm_w
    out = oracle.norm_rope(x, w, 1e-6, None, None, 0).double().numpy()
    xd = x.double().numpy()
    exact = xd / np.sqrt((xd ** 2).mean(-1, keepdims=True) + 1e-6) * w.double().numpy()
    # two BF16 roundings: half a step of y (scaled by |w| <= 1.5) plus half a step
    # of the output -- at most 1.5 output steps
    assert (np.abs(out - exact) <= 1.5 * _bf16_ulp(exact) * 1.0001).all()


def test_rmsnorm_agrees_with_eager_torch_sequence():
    inp = make_inputs(small_case(1, 4, 256, 32, rms_norm=True))
    x, w = inp.q, inp.q_norm_w
    out = oracle.norm_rope(x, w, 1e-6, None, None, 0)
    xf = x.float()
    y = (xf * torch.rsqrt(xf.pow(2).mean(-1, keepdim=True) + 1e-6)).to(torch.bfloat16)
    eager = y * w
    same = (out.view(torch.int16) == eager.view(torch.int16)).double().mean().item()
    # the summation order and rsqrt of torch's kernels are not specified; the
    # two BF16 roundings dominate, so nearly every element agrees bit for bit
    assert same > 0.995
    assert ((out.float() - eager.float()).abs() <= torch.from_numpy(_bf16_ulp(eager.double().numpy())).float()).all()


@pytest.mark.parametrize("rope_dim", [32, 64, 96, 128])
def test_rope_matches_eager_torch_bitwise(rope_dim):
    B, S, H = 1, 48, 3
    inp = make_inputs(small_case(B, H, S, 33 + rope_dim))
    cos, sin = rope_tables(S, rope_dim)
    out = oracle.norm_rope(inp.k, None, 0.0, cos, sin, rope_dim)
    x = inp.k
    xr, xp = x[..., :rope_dim], x[..., rope_dim:]
    h = rope_dim // 2
    rot = torch.cat([-xr[..., h:], xr[..., :h]], dim=-1)
    c, s = cos[None, :, None, :], sin[None, :, None, :]
    eager = torch.cat([(xr * c) + (rot * s), xp], dim=-1)
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))


def test_rope_identity_at_position_zero_and_rotation_norms():
    S, rope_dim = 64, 128
    inp = make_inputs(small_case(1, 2, S, 34))
    cos, sin = rope_tables(S, rope_dim)
    out = oracle.norm_rope(inp.q, None, 0.0, cos, sin, rope_dim)
    assert torch.equal(out[:, 0].view(torch.int16), inp.q[:, 0].view(torch.int16))
    # rotation of channel pairs (c, c + 64) keeps their norm up to BF16 rounding
    x = inp.q.double()
    o = out.double()
    n_in = x[..., :64] ** 2 + x[..., 64:] ** 2
    n_out = o[..., :64] ** 2 + o[..., 64:] ** 2
    assert ((n_out.sqrt() - n_in.sqrt()).abs() <= 4 * 2.0 ** -8 * n_in.sqrt() + 1e-30).all()


def test_fused_norm_rope_equals_the_two_steps():
    inp = make_inputs(small_case(1, 2, 64, 35, rms_norm=True, rope_dim=64))
    fused = oracle.norm_rope(inp.q, inp.q_norm_w, 1e-6, inp.rope_cos, inp.rope_sin, 64)
    step1 = oracle.norm_rope(inp.q, inp.q_norm_w, 1e-6, None, None, 0)
    step2 = oracle.norm_rope(step1, None, 0.0, inp.rope_cos, inp.rope_sin, 64)
    assert torch.equal(fused.view(torch.int16), step2.view(torch.int16))


# ------------------------------------------------------------------ accounting pins

def _table(name):
    rows = []
    import os
    for line in open(os.path.join(os.path.dirname(__file__), "golden", name)):
        line = line.split("#")[0].split()
        if line:
            rows.append(line)
    return rows


def test_byte_model_reproduces_handbook_table():
    GB = 1024 ** 3
    for name, n, h, scores, naive, flash in _table("handbook_attention_bytes.txt"):
        n, h = int(n), int(h)
        assert f"{roofline.score_matrix_bytes(n, h) / GB:.1f}" == scores
        assert f"{roofline.naive_bytes(1, h, n) / GB:.1f}" == naive
        assert f"{roofline.flash_bytes(1, h, n) / GB:.2f}" == flash


def test_flop_model_reproduces_handbook_block_profile():
    g = dict(_table("handbook_dit_block_attention.txt"))
    n, d = int(g["n"]), int(g["d"])
    flops = roofline.attention_flops(1, d // 128, n, 128)
    byts = roofline.flash_bytes(1, d // 128, n, 128)
    assert f"{flops / 1e9:.1f}" == g["gflop"]
    assert f"{byts / 2 ** 20:.0f}" == g["mbytes"]
    assert f"{flops / byts:.0f}" == g["intensity"]


@pytest.mark.parametrize("name,gb", [("flux2048", 1.14), ("wan720p", 4.29), ("hunyuan720p", 4.03)])
def test_prepare_byte_model_matches_the_scope_figures(name, gb):
    """The prepare's algorithmic bytes (the benchmark's HBM-fraction numerator): read Q, K, V
    and V again, write the INT8 Q/K and e4m3 V codes and the scales (plus the RoPE tables and
    RMSNorm weights where fused) -- 1.14, 4.29 and 4.03 GB at the FLUX-2048, Wan-720p and
    HunyuanVideo-720p shapes, and K smoothing adds one more pass over K and its block sums."""
    from workloads import WORKLOADS
    w = WORKLOADS[name]
    S_pad = oracle.padded_len(w.S)
    got = roofline.prepare_bytes(w.B, w.H, w.S, S_pad, 128, w.rms_norm, w.rope_dim)
    assert abs(got / 1e9 - gb) < 0.01
    bsh = w.B * w.S * w.H * 128
    smooth = roofline.prepare_smooth_k_bytes(w.B, w.H, w.S, S_pad, 128, w.rms_norm, w.rope_dim)
    assert smooth - got == bsh * 2 + 2 * w.B * w.H * (S_pad // 32) * 128 * 4 + 2 * w.B * w.H * 128 * 4
