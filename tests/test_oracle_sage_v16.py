"""Pins for the oracle's Sage attention with a 16-bit P V product (CPU only).

The handbook's SageAttention section has P and V "in FP8 or FP16" (ai-infra
handbook, "Kernel acceleration: attention, compilation and fusion", section
"SageAttention: quantizing attention too"); the oracle's reading of the
16-bit mode: scores from the INT8 Q/K codes exactly as in the FP8 mode, V
taken from the BF16 input, nothing rounded.

Pinned against an independent numpy FP64 evaluation, a closed form (all
scores equal: the output is the plain mean of V), and the ordering that
motivates the mode (closer to the exact attention than the e4m3 format).
"""
import math

import numpy as np
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
