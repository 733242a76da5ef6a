"""Pins for the oracle's FP64 attention on prepared (INT8 / e4m3) tensors (CPU only)."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import make_inputs, small_case

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_exactly_representable_inputs_reduce_to_plain_attention():
    """Integer Q/K whose every 32-row block holds a 127 quantise with scale 1 (codes equal
    the values, Q's scale is the log2 softmax factor); V whose channels are e4m3 values with
    maximum 448 quantise with scale 1.  The format's attention is then the plain attention
    of the same inputs, up to the binary32 rounding of the softmax factor."""
    g = torch.Generator().manual_seed(3)
    B, S, H = 1, 96, 2
    q = torch.randint(-127, 128, (B, S, H, 128), generator=g).float()
    k = torch.randint(-127, 128, (B, S, H, 128), generator=g).float()
    for t in (q, k):
        t[:, ::32, :, 0] = 127.0
    codes = torch.randint(0, 126, (B, S, H, 128), generator=g, dtype=torch.uint8)
    vals = torch.from_numpy(oracle.e4m3_decode(codes.numpy())).float()
    vals = vals * torch.where(torch.rand(vals.shape, generator=g) < 0.5, -1.0, 1.0)
    vals[:, 0, :, :] = 448.0
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, vals))
    scale = 1.0 / (math.sqrt(128) * 127 * 127 / 3)
    prep = oracle.prepare(q, k, v, scale)
    assert (prep["k_scale"][:, :, :3] == 1.0).all() and (prep["v_scale"] == 1.0).all()
    assert torch.equal(prep["q_i8"][:, :, :S].permute(0, 2, 1, 3), q.to(torch.int8))
    rows = oracle.all_rows(B, S, H)
    got = oracle.sage_attention(prep, S, rows, H)
    ref = oracle.attention(q, k, v, scale, rows=rows)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-5 * 448)


def test_abs_values_give_weighted_mean_magnitude():
    inp = make_inputs(small_case(1, 2, 200, 4))
    prep = oracle.prepare(inp.q, inp.k, inp.v, 1 / math.sqrt(128))
    rows = oracle.all_rows(1, 200, 2)
    a = oracle.sage_attention(prep, 200, rows, 2, abs_v=True)
    o = oracle.sage_attention(prep, 200, rows, 2)
    assert (a >= np.abs(o) - 1e-12).all()


def test_rounded_p_reproduces_the_printed_accuracy_band():
    """The Sage format with e4m3 probabilities, on N(0,1) BF16 inputs, lands in the
    accuracy band the aiter pull request prints for its op on randn inputs."""
    band = {}
    for line in open(os.path.join(GOLDEN, "aiter_sage_accuracy.txt")):
        f = line.split("#")[0].split()
        if len(f) == 2:
            band[f[0]] = float(f[1])
    inp = make_inputs(small_case(1, 4, 2048, 5))
    scale = 1 / math.sqrt(128)
    prep = oracle.prepare(inp.q, inp.k, inp.v, scale)
    rows = oracle.all_rows(1, 2048, 4)[::7]
    got = oracle.sage_attention(prep, 2048, rows, 4, p_e4m3=True)
    ref = oracle.attention(inp.q, inp.k, inp.v, scale, rows=rows)
    cos = float((got * ref).sum() / (np.linalg.norm(got) * np.linalg.norm(ref)))
    rel = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    # the page gives one band over its (unprinted) shapes; allow its width again on each side
    w_cos = band["cos_max"] - band["cos_min"]
    w_rel = band["rel_l2_max"] - band["rel_l2_min"]
    assert band["cos_min"] - 2 * w_cos <= cos <= band["cos_max"] + 2 * w_cos, cos
    assert band["rel_l2_min"] - 2 * w_rel <= rel <= band["rel_l2_max"] + 2 * w_rel, rel
    # without the rounding of P the format alone is clearly more accurate
    exact = oracle.sage_attention(prep, 2048, rows, 4)
    assert np.linalg.norm(exact - ref) / np.linalg.norm(ref) < 0.8 * rel


def test_key_value_reversal_permutes_codes_and_keeps_the_format_value():
    """With S a multiple of 32, reversing the K/V tokens maps whole K blocks
    onto blocks and keeps V's per-channel maxima, so the oracle's codes are the
    forward order's, permuted, and the FP64 attention of the format is the same
    up to summation order.  A wrong block index, or V's transpose taken on the
    wrong axis, breaks the permutation."""
    S, H = 192, 2
    inp = make_inputs(small_case(1, H, S, 57))
    sm = 1 / math.sqrt(128)
    rev = torch.arange(S - 1, -1, -1)
    a = oracle.prepare(inp.q, inp.k, inp.v, sm)
    b = oracle.prepare(inp.q, inp.k[:, rev], inp.v[:, rev], sm)
    assert torch.equal(b["q_i8"], a["q_i8"]) and torch.equal(b["q_scale"], a["q_scale"])
    nb = S // 32
    assert torch.equal(b["k_i8"][:, :, :S], a["k_i8"][:, :, rev])
    assert torch.equal(b["k_scale"][..., :nb], a["k_scale"][..., :nb].flip(-1))
    assert torch.equal(b["v_fp8"][..., :S], a["v_fp8"][..., rev])
    assert torch.equal(b["v_scale"], a["v_scale"])
    rows = oracle.all_rows(1, S, H)
    oa = oracle.sage_attention(a, S, rows, H)
    ob = oracle.sage_attention(b, S, rows, H)
    assert np.abs(oa - ob).max() <= 1e-12


@pytest.mark.parametrize("S,kw", [(1000, {}), (2000, dict(outlier_frac=0.05, outlier_gain=8.0)),
                                  (700, dict(k_channel_offset_std=2.0))])
def test_format_gate_covers_e4m3_rounding_of_p(S, kw):
    """The Sage kernel's gate against the exact format value, 1e-3 + (2^-4 + 2^-8) A|V|,
    is derived from rounding every probability to e4m3 (relative error <= 2^-4) with the
    denominator left unrounded.  The oracle's own e4m3-P evaluation must therefore sit
    inside it, outlier-dominated rows included, and well inside for the cosine."""
    from parity import SAGE_A, SAGE_B, metrics
    inp = make_inputs(small_case(1, 2, S, 520 + S, **kw))
    sm = 1 / math.sqrt(128)
    prep = oracle.prepare(inp.q, inp.k, inp.v, sm)
    rows = oracle.all_rows(1, S, 2)[::5]
    exact = oracle.sage_attention(prep, S, rows, 2)
    abs_v = oracle.sage_attention(prep, S, rows, 2, abs_v=True)
    rounded = oracle.sage_attention(prep, S, rows, 2, p_e4m3=True)
    m = metrics(rounded, exact, abs_v, SAGE_A, SAGE_B)
    assert m["bound_ratio"] <= 1.0 and m["cos"] >= 0.999, m
