"""Pins for the oracle's Q smoothing (CPU only).

The ai-infra handbook ("Kernel acceleration: attention, compilation and
fusion", section "SageAttention: quantizing attention too") describes
SageAttention removing a block mean from Q, and from K, ahead of INT8.
Unlike K's, Q's mean does not cancel in the softmax: q . k = (q - qbar) . k +
qbar . k, so the mean is kept with each 32-row block, in units of the block's
step as binary16 values, and the score product takes Q's operand as
f16(code + mean) (oracle.c, oracle_quant_q_smooth).

Pinned against: numpy's binary16 cast (the encoder); the plain FP64 attention
on exactly representable inputs (blocks built as an integer mean plus integer
deviations that sum to zero, times a power of two per block, including ragged
last blocks -- a wrong mean, order, step or correction moves the result); a
closed form for constant blocks; the reconstruction bound (code + mean) x step
within half a step plus the binary16 rounding of the mean; the accuracy gain
the smoothing exists for (Q with per-channel offsets); and planted mistakes.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from parity import metrics
from workloads import make_inputs, small_case


def test_f16_encoder_matches_numpy():
    rng = np.random.default_rng(11)
    x = np.concatenate([rng.standard_normal(200000) * 10.0 ** rng.integers(-9, 5, 200000),
                        np.ldexp(1.0, np.arange(-30, 16)).astype(np.float64)])
    x = x[np.abs(x) < 65504]
    assert np.array_equal(oracle.f16_encode(x), x.astype(np.float16).view(np.uint16))
    # every finite binary16 value round-trips, and midpoints go to the even pattern
    pats = np.arange(0, 0x7c00, dtype=np.uint16)
    vals = pats.view(np.float16).astype(np.float64)
    assert np.array_equal(oracle.f16_encode(vals), pats)
    mids = (vals[:-1] + vals[1:]) / 2
    want = np.where(pats[:-1] % 2 == 0, pats[:-1], pats[1:])
    assert np.array_equal(oracle.f16_encode(mids), want)
    assert np.array_equal(oracle.f16_encode(-vals[1:]), pats[1:] | 0x8000)


def mean_plus_deviation(g, B, S, H, exps, mu_max=100):
    """Q = (mu_B + d) * 2^e_B per 32-row block: mu_B integer per (block, head, channel)
    with |mu_B| <= mu_max, d integer with every channel's deviations over the block's
    valid rows summing to zero and a 127 in each block: the block mean is mu_B * 2^e
    exactly, the smoothed maximum 127 * 2^e, so the step is 2^e, the codes are d and
    the mean in step units is mu_B -- all exact."""
    q = torch.zeros((B, S, H, 128), dtype=torch.float64)
    for blk in range((S + 31) // 32):
        r0, r1 = 32 * blk, min(32 * blk + 32, S)
        n = r1 - r0
        # rows in +- pairs (an odd last row is zero): every channel's deviations sum to 0
        half = torch.randint(-126, 127, (B, n // 2, H, 128), generator=g).double()
        if n >= 2:
            half[:, 0, :, 3] = 127.0                           # the block's maximum |d| = 127
        d = torch.zeros((B, n, H, 128), dtype=torch.float64)
        d[:, 0:2 * (n // 2):2] = half
        d[:, 1:2 * (n // 2):2] = -half
        mu = torch.randint(-mu_max, mu_max + 1, (B, 1, H, 128), generator=g).double()
        if n == 1:
            mu[..., 3] = 127.0 * 256                          # a single row: the floor sets the step
        q[:, r0:r1] = (mu + d) * 2.0 ** exps[blk % len(exps)]
    return q


@pytest.mark.parametrize("S", [96, 113, 129])
def test_exact_construction_gives_codes_and_means(S):
    g = torch.Generator().manual_seed(2100 + S)
    B, H = 1, 2
    exps = [0, -2, 1, -1]
    q = mean_plus_deviation(g, B, S, H, exps)
    assert torch.equal(q.to(torch.bfloat16).double(), q)       # exactly representable
    c = oracle.softmax_log2_factor(0.01)
    codes, scales, m16 = oracle.quant_q_smooth(q.to(torch.bfloat16), 160, c)
    for blk in range((S + 31) // 32):
        r0, r1 = 32 * blk, min(32 * blk + 32, S)
        if r1 - r0 < 2:
            continue
        step = 2.0 ** exps[blk % len(exps)]
        mu = q[:, r0:r1].mean(dim=1)                            # exact here
        assert torch.equal(codes[:, :, r0:r1].permute(0, 2, 1, 3).double(), (q[:, r0:r1] - mu[:, None]) / step)
        got = np.vectorize(oracle.f16_decode)(m16[:, :, blk].numpy())
        assert np.array_equal(got, (mu / step).numpy())
        assert torch.equal(scales[:, :, blk].double(), torch.full((B, H), float(np.float32(np.float32(step) * c)),
                                                                  dtype=torch.float64))
    assert (codes[:, :, S:] == 0).all() and (scales[:, :, (S + 31) // 32:] == 0).all()


@pytest.mark.parametrize("S", [96, 113])
def test_exact_construction_reduces_to_plain_attention(S):
    """With exactly representable Q (smoothed), K (plain codes, per-block powers of two)
    and V (e4m3 values, channel maximum 448), both format values equal the plain FP64
    attention up to the binary32 rounding of the softmax factor."""
    g = torch.Generator().manual_seed(2200 + S)
    B, H = 1, 2
    q = mean_plus_deviation(g, B, S, H, [0, -1, 1]).to(torch.bfloat16)
    k = torch.randint(-127, 128, (B, S, H, 128), generator=g).double()
    k[:, ::32, :, 7] = 127.0
    for blk in range((S + 31) // 32):
        k[:, 32 * blk:32 * blk + 32] *= 2.0 ** [-1, 1, 0, -2][blk % 4]
    k = k.to(torch.bfloat16)
    codes = torch.randint(0, 126, (B, S, H, 128), generator=g, dtype=torch.uint8)
    v = torch.from_numpy(oracle.e4m3_decode(codes.numpy())).float()
    v = v * torch.where(torch.rand(v.shape, generator=g) < 0.5, -1.0, 1.0)
    v[:, 0] = 448.0
    v = v.to(torch.bfloat16)
    scale = 1.0 / (160.0 * 127.0 * math.sqrt(128))
    prep = oracle.prepare(q, k, v, scale, smooth_q=True)
    rows = oracle.all_rows(B, S, H)
    ref = oracle.attention(q, k, v, scale, rows=rows)
    t = (q.double()[0].permute(1, 0, 2) @ k.double()[0].permute(1, 2, 0)).abs().max().item() * scale * 1.4427
    assert 4 < t < 60                                          # a softmax that is neither flat nor one-hot
    for got, vmax in ((oracle.sage_attention(prep, S, rows, H), 448.0),
                      (oracle.sage_attention_v16(prep, v, rows), 448.0)):
        assert np.abs(got - ref).max() <= 2e-5 * vmax
    # planted mistakes: the correction dropped, or one block's mean moved by four steps
    no_mean = dict(prep, q_mean16=torch.zeros_like(prep["q_mean16"]))
    assert np.abs(oracle.sage_attention_v16(no_mean, v, rows) - ref).max() > 100 * 2e-5 * 448
    shifted = prep["q_mean16"].numpy().view(np.uint16).copy()
    dec = np.vectorize(oracle.f16_decode)(shifted[:, :, 1])
    shifted[:, :, 1] = oracle.f16_encode(dec + 4.0)
    moved = dict(prep, q_mean16=torch.from_numpy(shifted.view(np.int16)))
    assert np.abs(oracle.sage_attention_v16(moved, v, rows) - ref).max() > 10 * 2e-5 * 448


def test_constant_and_zero_blocks():
    """A block whose rows are all equal has zero deviations: the step is the floor
    max|mean| / (256 * 127), the codes are 0 and the mean in step units is +-32512 on
    the largest channel.  An all-zero block and one below 127/FLT_MAX are stored as
    zeros with scale 0."""
    B, H, S = 1, 1, 96
    x = torch.zeros((B, S, H, 128))
    row = torch.linspace(-3.0, 2.0, 128)
    x[:, 0:32] = row
    x[:, 64:96] = torch.full((128,), 1e-38)
    xb = x.to(torch.bfloat16)
    c = oracle.softmax_log2_factor(1 / math.sqrt(128))
    codes, scales, m16 = oracle.quant_q_smooth(xb, 96, c)
    assert (codes == 0).all()
    rowb = xb[0, 0, 0].float()
    cm = rowb.abs().max().item()
    step32 = np.float32(np.float32(np.float32(cm) * np.float32(1 / 256)) / np.float32(127))
    assert scales[0, 0, 0].item() == float(np.float32(step32 * np.float32(c)))
    m = np.vectorize(oracle.f16_decode)(m16[0, 0, 0].numpy())
    assert m[rowb.abs().argmax()] == math.copysign(32512.0, rowb[rowb.abs().argmax()].item())
    inv = np.float32(127) / np.float32(np.float32(cm) * np.float32(1 / 256))
    want = oracle.f16_encode((rowb.numpy() * inv).astype(np.float32).astype(np.float64))
    assert np.array_equal(m16[0, 0, 0].numpy().view(np.uint16), want)
    for blk in (1, 2):
        assert scales[0, 0, blk] == 0 and (m16[0, 0, blk] == 0).all()


@pytest.mark.parametrize("seed,offset", [(1, 0.0), (2, 3.0), (3, 40.0)])
def test_reconstruction_bound(seed, offset):
    """(code + mean) x step reconstructs every valid Q element within half a step plus
    the binary16 rounding of the mean (half a binary16 ulp of |mean|, in steps)."""
    g = torch.Generator().manual_seed(seed)
    B, H, S = 2, 3, 150
    q = (torch.randn((B, S, H, 128), generator=g) + offset * torch.randn((1, 1, H, 128), generator=g))
    qb = q.to(torch.bfloat16)
    c = 0.25
    codes, scales, m16 = oracle.quant_q_smooth(qb, 256, c)
    step = scales.double() / float(np.float32(c))                       # the binary32 step a_eff/127, near enough
    mean = torch.from_numpy(np.vectorize(oracle.f16_decode)(m16.numpy()))
    rec = (codes[:, :, :S].double() + mean.repeat_interleave(32, dim=2)[:, :, :S]) * \
        step.repeat_interleave(32, dim=2)[:, :, :S, None]
    err = (rec - qb.double().permute(0, 2, 1, 3)).abs()
    m_abs = mean.abs().repeat_interleave(32, dim=2)[:, :, :S]
    ulp_half = torch.where(m_abs >= 2 ** -14, 2.0 ** (torch.floor(torch.log2(m_abs.clamp_min(2 ** -14))) - 11), 2 ** -25)
    bound = (0.5 + ulp_half + 1e-5 * (m_abs + 127)) * step.repeat_interleave(32, dim=2)[:, :, :S, None]
    assert (err <= bound).all()


def test_smoothing_helps_offset_queries():
    """Q with large per-channel offsets: the smoothed format is much closer to the exact
    attention than the plain INT8 format (the reason for the smoothing)."""
    inp = make_inputs(small_case(1, 2, 512, 2300))
    g = torch.Generator().manual_seed(2301)
    q = (inp.q.float() + 4.0 * torch.randn((1, 1, 2, 128), generator=g)).to(torch.bfloat16)
    sm = 1 / math.sqrt(128)
    rows = oracle.all_rows(1, 512, 2)
    exact = oracle.attention(q, inp.k, inp.v, sm, rows=rows)
    plain = oracle.sage_attention_v16(oracle.prepare(q, inp.k, inp.v, sm), inp.v, rows)
    smooth = oracle.sage_attention_v16(oracle.prepare(q, inp.k, inp.v, sm, smooth_q=True), inp.v, rows)
    assert metrics(smooth, exact)["rel_l2"] < 0.5 * metrics(plain, exact)["rel_l2"]
