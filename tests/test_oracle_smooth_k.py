"""Pins for the oracle's K smoothing (CPU only).

SageAttention subtracts the mean of K before quantising it, which takes out
K's outlier channels (ai-infra handbook, "Kernel acceleration: attention,
compilation and fusion", section "SageAttention: quantizing attention too").
The oracle's reading: one mean per (batch, head, channel) over the S tokens,
summed in a fixed binary32 order (oracle.c, oracle_k_mean), then K - mean is
quantised like K.

The pins: the mean against an FP64 mean within the summation's rounding
bound; the smoothed codes against K - mean within half a quantisation step;
exactness (the FP64 attention of the smoothed format, evaluated by the oracle,
equals an independent numpy evaluation with the mean added back into K); and
the point of the step (smaller error on K with per-channel offsets).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from parity import metrics
from workloads import make_inputs, small_case

U = 2.0 ** -24   # binary32 unit roundoff


@pytest.mark.parametrize("B,H,S,off", [(1, 2, 200, 0.0), (2, 1, 77, 3.0), (1, 3, 1000, 0.5), (1, 1, 32, 0.0)])
def test_k_mean_within_summation_bound_of_fp64_mean(B, H, S, off):
    inp = make_inputs(small_case(B, H, S, 900 + S, k_channel_offset_std=off))
    S_pad = oracle.padded_len(S)
    mu = oracle.k_mean(inp.k, S_pad).double().numpy()                 # [B, H, 128]
    x = inp.k.double().permute(0, 2, 1, 3).numpy()                      # [B, H, S, 128]
    m64 = x.mean(axis=2)
    abs_sum = np.abs(x).sum(axis=2)
    depth = 8 + 2 + S_pad // 32        # additions on the longest path of the documented order
    bound = (depth + 2) * U * abs_sum / S + U * np.abs(m64)
    assert (np.abs(mu - m64) <= bound).all(), np.abs(mu - m64).max()


def test_k_mean_exact_for_a_constant_k():
    # 0.75 * n is exact in binary32 for every partial sum here, so the mean is 0.75 exactly,
    # K - mean is 0, and every smoothed code and scale is 0
    S = 300
    k = torch.full((1, S, 2, 128), 0.75).to(torch.bfloat16)
    S_pad = oracle.padded_len(S)
    mu = oracle.k_mean(k, S_pad)
    assert (mu == 0.75).all()
    codes, scales = oracle.quant_qk(k, S_pad, 1.0, mu)
    assert (codes == 0).all() and (scales == 0).all()


def test_k_mean_ignores_padding_rows():
    # the same tokens, S = 100, give the same mean whatever S_pad is
    inp = make_inputs(small_case(1, 2, 100, 31))
    assert torch.equal(oracle.k_mean(inp.k, 128), oracle.k_mean(inp.k, 256))


@pytest.mark.parametrize("S,off", [(200, 2.0), (61, 0.5)])
def test_smoothed_codes_reconstruct_k_minus_mean(S, off):
    inp = make_inputs(small_case(1, 2, S, 950 + S, k_channel_offset_std=off))
    S_pad = oracle.padded_len(S)
    mu = oracle.k_mean(inp.k, S_pad)
    codes, scales = oracle.quant_qk(inp.k, S_pad, 1.0, mu)
    x = inp.k.double().permute(0, 2, 1, 3)                               # [B, H, S, 128]
    xs = x - mu.double()[:, :, None, :]
    c = codes.double()
    for h in range(2):
        for j in range(S_pad // 32):
            r0, r1 = 32 * j, min(32 * j + 32, S)
            sc = scales[0, h, j].item()
            if r0 >= S:
                assert sc == 0.0 and (codes[0, h, r0:r0 + 32] == 0).all()
                continue
            blk = xs[0, h, r0:r1]
            a32 = np.float32(blk.abs().max().item())
            # the block's scale comes from the largest |K - mean| (up to the binary32 subtraction)
            assert abs(sc - float(np.float32(a32 / np.float32(127)))) <= 2 * U * sc
            err = (blk - c[0, h, r0:r1] * sc).abs()
            assert (err <= 0.5 * sc * (1 + 1e-5) + 2 * U * blk.abs()).all()
            idx = blk.abs().argmax()
            assert abs(c[0, h, r0:r1].flatten()[idx].item()) == 127
            assert (codes[0, h, r1:r0 + 32] == 0).all()


def _numpy_attention_log2(q2, kd, vd, rows):
    """softmax in base 2 of q2 . k (q2 already carries softmax_scale * log2 e)."""
    out = np.empty((len(rows), 128))
    for n, (b, s, h) in enumerate(rows.tolist()):
        t = kd[b, :, h, :] @ q2[b, s, h, :]
        w = np.exp2(t - t.max())
        out[n] = (w @ vd[b, :, h, :]) / w.sum()
    return out


def test_smoothing_is_exact_in_the_attention():
    """The oracle's FP64 attention of the smoothed codes equals a numpy FP64
    attention of the same codes with the mean added back into K: the shift
    by q . mean cancels in the softmax."""
    S, H = 150, 2
    sm = 1 / math.sqrt(128)
    inp = make_inputs(small_case(1, H, S, 961, k_channel_offset_std=2.0))
    prep = oracle.prepare(inp.q, inp.k, inp.v, sm, smooth_k=True)
    rows = oracle.all_rows(1, S, H)
    got = oracle.sage_attention(prep, S, rows, H)
    _, kd, vd = (t.numpy() for t in oracle.dequantized(prep, S))
    # Q in the log2 units the format uses: code * q_scale (q_scale carries softmax_scale * log2 e)
    q2 = (prep["q_i8"].double() * prep["q_scale"].double().repeat_interleave(32, dim=2)[..., None])
    q2 = q2[:, :, :S].permute(0, 2, 1, 3).numpy()
    mu = prep["k_mean"].double().numpy()                                   # [B, H, 128]
    kd_back = kd + mu[:, None, :, :]
    ref_back = _numpy_attention_log2(q2, kd_back, vd, rows)
    ref_plain = _numpy_attention_log2(q2, kd, vd, rows)
    assert np.abs(got - ref_back).max() <= 1e-10
    assert np.abs(got - ref_plain).max() <= 1e-10


def test_smoothing_reduces_error_on_channel_offsets():
    """K with per-(head, channel) offsets (the FLUX 1024 recipe, offsets
    scaled up): the quantised format with smoothing is closer to the FP64
    attention of the BF16 inputs than without."""
    S, H = 512, 2
    sm = 1 / math.sqrt(128)
    inp = make_inputs(small_case(1, H, S, 971, k_channel_offset_std=4.0))
    rows = oracle.all_rows(1, S, H)
    exact = oracle.attention(inp.q, inp.k, inp.v, sm, rows=rows)
    plain = oracle.sage_attention(oracle.prepare(inp.q, inp.k, inp.v, sm), S, rows, H)
    smooth = oracle.sage_attention(oracle.prepare(inp.q, inp.k, inp.v, sm, smooth_k=True), S, rows, H)
    e_plain = metrics(plain, exact)["rel_l2"]
    e_smooth = metrics(smooth, exact)["rel_l2"]
    assert e_smooth < 0.7 * e_plain, (e_smooth, e_plain)


def test_smoothing_changes_only_k():
    inp = make_inputs(small_case(1, 2, 130, 981, k_channel_offset_std=1.0))
    sm = 1 / math.sqrt(128)
    a = oracle.prepare(inp.q, inp.k, inp.v, sm)
    b = oracle.prepare(inp.q, inp.k, inp.v, sm, smooth_k=True)
    for key in ("q_i8", "q_scale", "v_fp8", "v_scale"):
        assert torch.equal(a[key], b[key]), key
    assert a["k_mean"] is None and b["k_mean"].shape == (1, 2, 128)
    assert not torch.equal(a["k_i8"], b["k_i8"])
