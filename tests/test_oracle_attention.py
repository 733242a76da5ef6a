"""Pins for the oracle's FP64 attention (CPU only).

Each test checks the oracle against something other than itself: closed
forms, invariants of softmax attention, a second algorithm written from the
ai-infra handbook's blocked online-softmax example ("Kernel acceleration:
attention, compilation and fusion", section "Attention: from O(N^2) memory to
blocks"), and torch's own scaled_dot_product_attention in float64.
"""
import functools
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from workloads import make_inputs, small_case

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


def sdpa64(q, k, v, scale):
    qd, kd, vd = (t.double().permute(0, 2, 1, 3) for t in (q, k, v))
    return F.scaled_dot_product_attention(qd, kd, vd, scale=scale).permute(0, 2, 1, 3).numpy()


def chunked_softmax_attention(q, k, v, scale, chunk):
    """FP64 attention the blocked way, so that the full S x S score matrix never
    exists: the keys are taken `chunk` at a time, each chunk is reduced to a
    partial softmax state (per query row: the chunk's largest score, the sum of
    exp(t - that maximum) and the same weights applied to the chunk's V rows), and
    the states are merged left to right by bringing both to the larger maximum.
    This is the running-maximum bookkeeping of the handbook's blocked online
    softmax written as a fold; only the final division by the weight sum remains."""
    qd, kd, vd = (t.double().numpy() for t in (q, k, v))   # [B, S, H, D]

    def reduce_chunk(c0):
        t = np.einsum("bqhd,bkhd->bhqk", qd, kd[:, c0:c0 + chunk]) * scale
        top = t.max(axis=-1)
        w = np.exp(t - top[..., None])
        return top, w.sum(axis=-1), np.einsum("bhqk,bkhd->bhqd", w, vd[:, c0:c0 + chunk])

    def merge(a, b):
        peak = np.maximum(a[0], b[0])
        fa, fb = np.exp(a[0] - peak), np.exp(b[0] - peak)
        return peak, a[1] * fa + b[1] * fb, a[2] * fa[..., None] + b[2] * fb[..., None]

    _, weight, weighted_v = functools.reduce(merge, map(reduce_chunk, range(0, qd.shape[1], chunk)))
    return (weighted_v / weight[..., None]).transpose(0, 2, 1, 3)


def test_single_key_returns_its_value_exactly():
    g = torch.Generator().manual_seed(1)
    q, k, v = (torch.randn(2, 1, 3, 128, generator=g).to(torch.bfloat16) for _ in range(3))
    o = oracle.attention(q, k, v, 1 / math.sqrt(128))
    assert np.array_equal(o, v.double().numpy())


def test_two_keys_closed_form():
    g = torch.Generator().manual_seed(2)
    q, k, v = (torch.randn(1, 2, 1, 64, generator=g).to(torch.bfloat16) for _ in range(3))
    scale = 0.125
    o = oracle.attention(q, k, v, scale)
    qd, kd, vd = (t.double().numpy()[0, :, 0] for t in (q, k, v))
    for i in range(2):
        t0, t1 = scale * qd[i] @ kd[0], scale * qd[i] @ kd[1]
        s0 = 1.0 / (1.0 + math.exp(t1 - t0))   # logistic sigma(t0 - t1)
        expect = s0 * vd[0] + (1 - s0) * vd[1]
        np.testing.assert_allclose(o[0, i, 0], expect, rtol=0, atol=1e-14)


def test_uniform_values_are_returned():
    g = torch.Generator().manual_seed(3)
    B, S, H, D = 1, 77, 2, 128
    q, k = (torch.randn(B, S, H, D, generator=g).to(torch.bfloat16) for _ in range(2))
    row = torch.randn(D, generator=g).to(torch.bfloat16)
    v = row.expand(B, S, H, D).contiguous()
    o = oracle.attention(q, k, v, 1 / math.sqrt(D))
    np.testing.assert_allclose(o, np.broadcast_to(row.double().numpy(), o.shape), rtol=0, atol=1e-13)


def test_one_hot_scores_select_one_value():
    # K rows are scaled unit vectors; query i points along key i, so its score
    # gap to every other key is alpha^2 * scale and O_i -> V_i.
    D, S = 128, 32
    alpha = 20.0
    k = torch.zeros(1, S, 1, D)
    for j in range(S):
        k[0, j, 0, j] = alpha
    q = k.clone()
    g = torch.Generator().manual_seed(4)
    v = torch.randn(1, S, 1, D, generator=g)
    q, k, v = bf16(q), bf16(k), bf16(v)
    scale = 1 / math.sqrt(D)
    o = oracle.attention(q, k, v, scale)
    gap = alpha * alpha * scale
    bound = (S - 1) * math.exp(-gap) * 2 * v.double().abs().max().item()
    assert bound < 1e-8
    np.testing.assert_allclose(o[0, :, 0], v.double().numpy()[0, :, 0], rtol=0, atol=bound)


def test_affine_equivariance_in_values():
    g = torch.Generator().manual_seed(5)
    B, S, H, D = 1, 64, 2, 128
    q, k = (torch.randn(B, S, H, D, generator=g).to(torch.bfloat16) for _ in range(2))
    vi = torch.randint(-8, 9, (B, S, H, D), generator=g).float() / 4
    v = bf16(vi)
    v2 = bf16(2 * vi + 1)          # exact in BF16 for these small dyadics
    scale = 1 / math.sqrt(D)
    o1 = oracle.attention(q, k, v, scale)
    o2 = oracle.attention(q, k, v2, scale)
    np.testing.assert_allclose(o2, 2 * o1 + 1, rtol=0, atol=1e-12)


def test_key_value_permutation_invariance():
    inp = make_inputs(small_case(1, 3, 200, 11))
    perm = torch.randperm(200, generator=torch.Generator().manual_seed(6))
    scale = inp.wl.softmax_scale
    o1 = oracle.attention(inp.q, inp.k, inp.v, scale)
    o2 = oracle.attention(inp.q, inp.k[:, perm].contiguous(), inp.v[:, perm].contiguous(), scale)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)


def _golden(name):
    vals = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#")[0].split()
        if len(line) == 2:
            vals[line[0]] = float(line[1])
    return vals


def test_blocked_online_softmax_equals_definition_at_handbook_example():
    gd = _golden("handbook_blocked_example.txt")
    B, H, N, D, block = (int(gd[k]) for k in ("B", "H", "N", "D", "block"))
    g = torch.Generator().manual_seed(0)
    q, k, v = (torch.randn(B, N, H, D, generator=g).to(torch.bfloat16) for _ in range(3))
    scale = 1 / math.sqrt(D)
    o = oracle.attention(q, k, v, scale)
    ob = chunked_softmax_attention(q, k, v, scale, block)
    # the handbook prints agreement at atol 1e-5 in float32; in FP64 the two forms agree to rounding
    assert np.allclose(o, ob, atol=gd["atol"])
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
    # the example's printed memory figures: N x N float32 scores vs one block x N slab
    assert B * H * N * N * 4 / 1024 == gd["naive_scores_kb"]
    assert B * H * block * N * 4 / 1024 == gd["blocked_peak_kb"]


@pytest.mark.parametrize("B,H,S,D", [(1, 4, 256, 32), (2, 3, 129, 128), (1, 1, 1, 128), (1, 2, 300, 128)])
def test_matches_torch_sdpa_float64(B, H, S, D):
    g = torch.Generator().manual_seed(B * 1000 + S)
    q, k, v = (torch.randn(B, S, H, D, generator=g).to(torch.bfloat16) for _ in range(3))
    scale = 1 / math.sqrt(D)
    o = oracle.attention(q, k, v, scale)
    np.testing.assert_allclose(o, sdpa64(q, k, v, scale), rtol=0, atol=1e-12)


def test_row_sampling_matches_full_evaluation():
    inp = make_inputs(small_case(2, 3, 150, 12))
    full = oracle.attention(inp.q, inp.k, inp.v, inp.wl.softmax_scale)
    rows = torch.tensor([[0, 0, 0], [1, 149, 2], [0, 77, 1], [1, 128, 0]])
    part = oracle.attention(inp.q, inp.k, inp.v, inp.wl.softmax_scale, rows=rows)
    for i, (b, s, h) in enumerate(rows.tolist()):
        assert np.array_equal(part[i], full[b, s, h])


def test_strided_views_read_like_contiguous():
    inp = make_inputs(small_case(1, 3, 100, 13, head_major_storage=True))
    assert not inp.q.is_contiguous()
    o1 = oracle.attention(inp.q, inp.k, inp.v, inp.wl.softmax_scale)
    o2 = oracle.attention(inp.q.contiguous(), inp.k.contiguous(), inp.v.contiguous(), inp.wl.softmax_scale)
    assert np.array_equal(o1, o2)


def test_planted_scale_mistake_is_caught():
    """A pin must fail on a plausible oracle mistake: evaluate the definition with a
    dropped softmax scale and check the torch comparison would reject it."""
    g = torch.Generator().manual_seed(9)
    q, k, v = (torch.randn(1, 64, 2, 128, generator=g).to(torch.bfloat16) for _ in range(3))
    wrong = oracle.attention(q, k, v, 1.0)
    right = sdpa64(q, k, v, 1 / math.sqrt(128))
    assert np.abs(wrong - right).max() > 1e-3


def _bf16(x):
    """float64 -> nearest BF16 value, through binary32 as the kernel's conversions do."""
    x32 = np.asarray(x, dtype=np.float32)
    return (oracle.f32_to_bf16(x32).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("S,kw", [(1000, {}), (2000, dict(outlier_frac=0.05, outlier_gain=8.0))])
def test_bf16_gate_covers_the_bf16_roundings(S, kw):
    """The BF16 path's gate, 2e-2 + 2^-7 A|V| with cosine >= 0.99999, is derived from what
    the kernel rounds: every probability to BF16 for the P V product (the denominator from
    the unrounded ones) and O once to BF16.  Emulated in FP64 on plain and outlier-dominated
    rows, that rounding stays inside the gate."""
    from parity import BF16_A, BF16_B, metrics
    inp = make_inputs(small_case(1, 2, S, 540 + S, **kw))
    sm = 1 / math.sqrt(128)
    rows = oracle.all_rows(1, S, 2)[::7]
    exact = oracle.attention(inp.q, inp.k, inp.v, sm, rows=rows)
    q, k, v = (x.double().numpy() for x in (inp.q, inp.k, inp.v))
    got = np.empty_like(exact)
    av = np.empty_like(exact)
    for n, (b, s, h) in enumerate(rows.tolist()):
        t = (k[b, :, h] @ q[b, s, h]) * sm
        w = np.exp(t - t.max())
        got[n] = _bf16((_bf16(w) @ v[b, :, h]) / w.sum())
        av[n] = (w @ np.abs(v[b, :, h])) / w.sum()
    m = metrics(got, exact, av, BF16_A, BF16_B)
    assert m["bound_ratio"] <= 1.0 and m["cos"] >= 0.99999, m
