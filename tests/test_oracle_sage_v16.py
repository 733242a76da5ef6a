"""Pins for the oracle's Sage attention with a 16-bit P V product (CPU only).

The handbook's SageAttention section has P and V "in FP8 or FP16" (ai-infra
handbook, "Kernel acceleration: attention, compilation and fusion", section
"SageAttention: quantizing attention too"); the oracle's reading of the
16-bit mode: scores from the INT8 Q/K codes exactly as in the FP8 mode, V
taken from the BF16 input, nothing rounded.

Pinned against the plain FP64 attention on exactly representable inputs
(integer codes times a power of two per 32-row block, so that every block's
scale is that power of two exactly and a wrong scale index, block edge or
factor changes the result), including ragged lengths whose last Q and K
blocks are partial; against a closed form (all scores equal: the output is
the plain mean of V); and against the ordering that motivates the mode
(closer to the exact attention than the e4m3 format).  The numpy evaluation
below repeats the oracle's formula and only guards the marshalling.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from parity import metrics
from workloads import make_inputs, small_case


def numpy_reference(prep, v, rows):
    q2 = prep["q_i8"].double() * prep["q_scale"].double().repeat_interleave(32, dim=2)[..., None]
    k2 = prep["k_i8"].double() * prep["k_scale"].double().repeat_interleave(32, dim=2)[..., None]
    S = v.shape[1]
    q2 = q2[:, :, :S].permute(0, 2, 1, 3).numpy()       # [B, S, H, 128], log2 units
    k2 = k2[:, :, :S].permute(0, 2, 1, 3).numpy()
    vd = v.double().numpy()
    out = np.empty((len(rows), 128))
    for n, (b, s, h) in enumerate(rows.tolist()):
        t = k2[b, :, h, :] @ q2[b, s, h, :]
        w = np.exp2(t - t.max())
        out[n] = (w @ vd[b, :, h, :]) / w.sum()
    return out


def blockwise_pow2_codes(g, B, S, H, exps):
    """Integer codes in [-127, 127] with a 127 in every 32-row block (and head), times
    2^exps[block]: the block's maximum is 127 * 2^e, so its scale a/127 is 2^e exactly and
    its codes are the integers themselves."""
    x = torch.randint(-127, 128, (B, S, H, 128), generator=g).double()
    x[:, ::32, :, 5] = 127.0
    for blk in range((S + 31) // 32):
        x[:, 32 * blk:32 * blk + 32] *= 2.0 ** exps[blk % len(exps)]
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("S", [96, 113, 161])
def test_exact_codes_reduce_to_plain_attention(S):
    """Q and K exactly representable by the format (per-block power-of-two scales that
    differ from block to block), V any BF16: the 16-bit mode's format value is the plain
    FP64 attention of the same inputs, up to the binary32 rounding of the softmax factor
    that Q's scale carries (relative 2^-24 on each score).  S = 113 and 161 leave the
    last Q and K blocks partial."""
    g = torch.Generator().manual_seed(1204 + S)
    B, H = 1, 2
    q = blockwise_pow2_codes(g, B, S, H, [0, -1, 1, -2])
    k = blockwise_pow2_codes(g, B, S, H, [-1, 2, 0, -3, 1])
    v = torch.randn((B, S, H, 128), generator=g).to(torch.bfloat16)
    # scores |t| = |q.k| * scale * log2(e) of order 10
    scale = 1.0 / (127.0 * 127.0 * math.sqrt(128))
    prep = oracle.prepare(q, k, v, scale)
    nblk = (S + 31) // 32
    kexp = torch.tensor([[-1, 2, 0, -3, 1][b % 5] for b in range(nblk)], dtype=torch.float64)
    assert torch.equal(prep["k_scale"][0, 0, :nblk].double(), 2.0 ** kexp)
    assert torch.equal(prep["k_i8"][:, :, :S].permute(0, 2, 1, 3).double(),
                       k.double() / (2.0 ** kexp).repeat_interleave(32)[:S].view(1, S, 1, 1))
    rows = oracle.all_rows(B, S, H)
    got = oracle.sage_attention_v16(prep, v, rows)
    ref = oracle.attention(q, k, v, scale, rows=rows)
    vmax = v.double().abs().max().item()
    assert np.abs(got - ref).max() <= 1e-5 * vmax


def test_planted_scale_mistakes_are_caught():
    """The same exactly representable case with the K scale of one block doubled, or
    the Q scale taken from the neighbouring block: the oracle's value moves far
    outside the tolerance of the test above (by a factor of 100 at least)."""
    g = torch.Generator().manual_seed(1210)
    B, H, S = 1, 2, 113
    q = blockwise_pow2_codes(g, B, S, H, [0, -1, 1, -2])
    k = blockwise_pow2_codes(g, B, S, H, [-1, 2, 0, -3, 1])
    v = torch.randn((B, S, H, 128), generator=g).to(torch.bfloat16)
    scale = 1.0 / (127.0 * 127.0 * math.sqrt(128))
    prep = oracle.prepare(q, k, v, scale)
    rows = oracle.all_rows(B, S, H)
    ref = oracle.attention(q, k, v, scale, rows=rows)
    tol = 1e-5 * v.double().abs().max().item()
    bad_k = dict(prep, k_scale=prep["k_scale"].clone())
    bad_k["k_scale"][:, :, 3] *= 2
    bad_q = dict(prep, q_scale=torch.roll(prep["q_scale"], 1, dims=2))
    for bad in (bad_k, bad_q):
        assert np.abs(oracle.sage_attention_v16(bad, v, rows) - ref).max() > 100 * tol


def test_matches_numpy_fp64():
    B, H, S = 2, 2, 137
    inp = make_inputs(small_case(B, H, S, 1201))
    prep = oracle.prepare(inp.q, inp.k, inp.v, 1 / math.sqrt(128))
    rows = oracle.all_rows(B, S, H)
    got = oracle.sage_attention_v16(prep, inp.v, rows)
    assert np.abs(got - numpy_reference(prep, inp.v, rows)).max() <= 1e-11
    got_abs = oracle.sage_attention_v16(prep, inp.v, rows, abs_v=True)
    assert np.abs(got_abs - numpy_reference(prep, inp.v.abs(), rows)).max() <= 1e-11


def test_zero_query_gives_the_mean_of_v():
    # Q = 0: every score is 0, the softmax is uniform and O is the plain mean of V over the keys
    B, H, S = 1, 2, 45
    inp = make_inputs(small_case(B, H, S, 1202))
    q = torch.zeros_like(inp.q)
    prep = oracle.prepare(q, inp.k, inp.v, 1 / math.sqrt(128))
    rows = oracle.all_rows(B, S, H)
    got = oracle.sage_attention_v16(prep, inp.v, rows)
    mean_v = inp.v.double().mean(dim=1)                 # [B, H, 128]
    ref = mean_v[rows[:, 0], rows[:, 2]].numpy()
    assert np.abs(got - ref).max() <= 1e-13


def test_closer_to_exact_than_the_e4m3_format():
    B, H, S = 1, 2, 400
    sm = 1 / math.sqrt(128)
    inp = make_inputs(small_case(B, H, S, 1203))
    prep = oracle.prepare(inp.q, inp.k, inp.v, sm)
    rows = oracle.all_rows(B, S, H)
    exact = oracle.attention(inp.q, inp.k, inp.v, sm, rows=rows)
    v16 = oracle.sage_attention_v16(prep, inp.v, rows)
    e4m3 = oracle.sage_attention(prep, S, rows, H)
    assert metrics(v16, exact)["rel_l2"] < metrics(e4m3, exact)["rel_l2"]
