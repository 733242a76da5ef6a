"""The attention kernels' online softmax with a lazily moved reference,
emulated tile by tile in FP64 (CPU): per 128-key tile, the reference m moves
only when the tile's maximum passes it by more than tau, O and l are then
scaled by 2^(m_old - m_new), and p = c * 2^(t - m) with c = 1 (BF16 P, tau = 64)
or c = 448 * 2^-tau (e4m3 P, tau = 4; the largest p then stays <= 448).  In
exact arithmetic O / l is the softmax-weighted mean whatever the schedule of
moves (the handbook's blocked online softmax, section "Attention: from O(N^2)
memory to blocks", with the rescale deferred), so the emulation equals the
oracle's FP64 attention; a planted mistake (the reference moved without
rescaling l) is caught."""
import math

import numpy as np
import pytest
import torch

import oracle
from workloads import make_inputs, small_case


def lazy_flash(t2, v, tau, c, bug=False):
    """t2: [S] scores in log2 units, v: [S, D]; tiles of 128 keys in order."""
    m, l, o, p_max = -math.inf, 0.0, np.zeros(v.shape[1]), 0.0
    for j0 in range(0, t2.size, 128):
        t = t2[j0:j0 + 128]
        mt = t.max()
        if mt > m + tau:
            sc = 2.0 ** (m - mt) if m > -math.inf else 0.0
            if not bug:
                l *= sc
            o *= sc
            m = mt
        p = c * np.exp2(t - m)
        p_max = max(p_max, p.max())
        l += p.sum()
        o += p @ v[j0:j0 + 128]
    return o / l, p_max


@pytest.mark.parametrize("tau,c", [(64.0, 1.0), (4.0, 448.0 * 2.0 ** -4)])
@pytest.mark.parametrize("S,kw", [(1000, {}), (2000, dict(outlier_frac=0.05, outlier_gain=8.0))])
def test_lazy_reference_is_exact(tau, c, S, kw):
    inp = make_inputs(small_case(1, 2, S, 300 + S, **kw))
    sm = 1 / math.sqrt(128)
    rows = oracle.all_rows(1, S, 2)[:: 37]
    ref = oracle.attention(inp.q, inp.k, inp.v, sm, rows=rows)
    q = inp.q.double().numpy()
    k = inp.k.double().numpy()
    v = inp.v.double().numpy()
    for n, (b, s, h) in enumerate(rows.tolist()):
        t2 = (k[b, :, h] @ q[b, s, h]) * sm / math.log(2)       # softmax in base 2
        o, p_max = lazy_flash(t2, v[b, :, h], tau, c)
        assert np.abs(o - ref[n]).max() <= 1e-12
        if c != 1.0:
            assert p_max <= 448.0 * (1 + 1e-12)                   # e4m3 range never exceeded


def test_a_planted_mistake_is_caught():
    inp = make_inputs(small_case(1, 1, 1000, 333, outlier_frac=0.05, outlier_gain=8.0))
    sm = 1 / math.sqrt(128)
    rows = oracle.all_rows(1, 1000, 1)[:: 50]
    ref = oracle.attention(inp.q, inp.k, inp.v, sm, rows=rows)
    q, k, v = (x.double().numpy() for x in (inp.q, inp.k, inp.v))
    worst = 0.0
    for n, (b, s, h) in enumerate(rows.tolist()):
        t2 = (k[b, :, h] @ q[b, s, h]) * sm / math.log(2)
        o, _ = lazy_flash(t2, v[b, :, h], 4.0, 28.0, bug=True)
        worst = max(worst, np.abs(o - ref[n]).max())
    assert worst > 1e-3
