"""Property-based pins of the oracle's quantisers (hypothesis drives shapes,
ragged lengths and magnitudes 2^-60..2^60; CPU only).  Against the
definitions, per block or channel:
  * quant_qk (the aiter pull request, Technical Details: INT8, one scale per
    32-row block): scale = fl32(a / 127) for the block's largest |x| = a; the
    largest element codes to +-127; every code is round(x * 127 / a) to within
    the binary32 rounding of the product (and +-127 for every nonzero element
    where 127 / a overflows, the reading's literal result); padding codes 0.
  * quant_v (same section: e4m3, one scale per channel over all positions):
    scale = fl32(a / 448); the largest element decodes to +-448; every decoded
    code is within e4m3's rounding of v * 448 / a (relative 2^-4 on normal
    values, 2^-10 absolute below them); padding 0."""
import numpy as np
import pytest

pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402
from workloads import wide_bf16  # noqa: E402

shapes = st.tuples(st.integers(1, 2), st.integers(1, 3), st.integers(1, 300))
ranges = st.tuples(st.integers(-60, 60), st.integers(0, 30)).map(lambda t: (t[0], t[0] + t[1] + 1))


@settings(max_examples=30, deadline=None)
@given(shape=shapes, rng=ranges, seed=st.integers(0, 10_000))
def test_quant_qk_block_properties(shape, rng, seed):
    B, H, S = shape
    x = wide_bf16(seed, (B, S, H, 128), *rng)
    S_pad = oracle.padded_len(S)
    codes, scales = oracle.quant_qk(x, S_pad)
    xf = x.float().numpy().transpose(0, 2, 1, 3)          # [B, H, S, 128], exact
    c = codes.numpy().astype(np.int64)
    sc = scales.numpy()
    for b in range(B):
        for h in range(H):
            for j in range(S_pad // 32):
                r0, r1 = 32 * j, min(32 * j + 32, S)
                blk_c = c[b, h, 32 * j:32 * j + 32]
                if r0 >= S:
                    assert sc[b, h, j] == 0 and (blk_c == 0).all()
                    continue
                blk = xf[b, h, r0:r1].astype(np.float32)
                a = np.float32(np.abs(blk).max())
                assert sc[b, h, j] == np.float32(a / np.float32(127))
                assert (np.abs(blk_c) <= 127).all() and (blk_c[r1 - r0:] == 0).all()
                live = blk_c[:r1 - r0]
                assert np.abs(live).max() == 127
                inv = np.float32(127) / a
                if np.isfinite(inv):
                    t = (blk.astype(np.float64) * (127.0 / np.float64(a)))
                    assert (np.abs(live - t) <= 0.5 + 1e-4 * np.maximum(1.0, np.abs(t))).all()
                else:
                    assert (np.abs(live[blk != 0]) == 127).all() and (live[blk == 0] == 0).all()


@settings(max_examples=30, deadline=None)
@given(shape=shapes, rng=ranges, seed=st.integers(0, 10_000))
def test_quant_v_channel_properties(shape, rng, seed):
    B, H, S = shape
    v = wide_bf16(seed, (B, S, H, 128), *rng)
    S_pad = oracle.padded_len(S)
    codes, scales = oracle.quant_v(v, S_pad)
    vf = v.float().numpy().transpose(0, 2, 3, 1).astype(np.float64)   # [B, H, 128, S]
    dec = oracle.e4m3_decode(codes.numpy())                          # [B, H, 128, S_pad]
    sc = scales.numpy()
    assert (dec[..., S:] == 0).all()
    a = np.abs(vf).max(axis=-1)                                      # [B, H, 128]
    assert (sc == (a.astype(np.float32) / np.float32(448))).all()
    live = dec[..., :S]
    assert (np.abs(live).max(axis=-1)[a > 0] == 448).all()
    inv = (np.float32(448) / a.astype(np.float32)).astype(np.float64)
    fin = np.isfinite(inv)
    t = vf * (448.0 / np.where(a > 0, a, 1.0))[..., None]
    err = np.abs(live - t)
    bound = np.maximum(2.0 ** -4 * np.abs(t), 2.0 ** -10) * (1 + 1e-5) + 1e-5 * np.abs(t)
    ok = err <= bound
    assert ok[fin].all()
