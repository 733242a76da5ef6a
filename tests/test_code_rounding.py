"""The code formation the prepare and the forward's quantise-on-load use (CPU
check of the argument, in binary32 arithmetic as the kernels do it): for a
block with largest |x| = a and inv = fl32(127 / a) finite, the code
clamp(rne(fl32(x * inv)), -127, 127) equals the integer n that
fl32(fl32(x * inv) + 1.5 * 2^23) carries in its low mantissa bits
(bits = 0x4B400000 + n), the clamp never binds (|fl32(x * inv)| <= 127 after
rounding), its low byte is n's two's-complement byte, and
fl32(that sum - 1.5 * 2^23) is n exactly (so its FP16 conversion is exact)."""
import numpy as np

MAGIC = np.float32(12582912.0)


def blocks(seed, n_blocks):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n_blocks):
        e = rng.integers(-120, 120)
        x = (rng.standard_normal(4096) * np.exp2(float(e))).astype(np.float32)
        if i % 7 == 0:
            x[rng.integers(0, 4096)] *= np.float32(16)          # an outlier sets a
        out.append(x)
    return out


def test_magic_rounding_equals_clamped_rne():
    for x in blocks(11, 300):
        a = np.abs(x).max()
        inv = np.float32(127) / a
        assert np.isfinite(inv)
        t = x * inv                                              # fl32(x * inv)
        assert np.abs(t).max() <= np.float32(127.5)              # never a tie at or past 127.5
        ref = np.clip(np.rint(t), -127, 127).astype(np.int64)    # rne, then the clamp
        assert np.array_equal(np.rint(t).astype(np.int64), ref)  # the clamp never binds
        y = t + MAGIC                                            # fl32(t + 1.5 * 2^23)
        n = y.view(np.int32).astype(np.int64) - 0x4B400000
        assert np.array_equal(n, ref)
        assert np.array_equal((y.view(np.uint32) & 0xFF).astype(np.uint8), ref.astype(np.int8).view(np.uint8))
        back = y - MAGIC
        assert np.array_equal(back.astype(np.int64), ref) and np.array_equal(back, ref.astype(np.float32))
        assert np.array_equal(back.astype(np.float16).astype(np.float32), back)


def test_ties_go_to_even():
    # exact x.5 products: rne sends them to the even neighbour, as the magic addition does
    t = np.array([0.5, 1.5, 2.5, -0.5, -1.5, 126.5, -126.5], dtype=np.float32)
    y = t + MAGIC
    n = y.view(np.int32).astype(np.int64) - 0x4B400000
    assert n.tolist() == [0, 2, 2, 0, -2, 126, -126]


def test_int8_to_fp16_widening_is_exact():
    # the two-call path's widening: byte u = code + 128 as the FP16 pattern 0x6400 | u is
    # 1024 + u, and 1024 + u - 1152 is the code -- for all 256 codes, in FP16 arithmetic
    codes = np.arange(-128, 128, dtype=np.int64)
    u = (codes + 128).astype(np.uint16)
    h = (np.uint16(0x6400) | u).view(np.float16)
    assert np.array_equal(h.astype(np.float64), 1024.0 + u)
    widened = (h - np.float16(1152)).astype(np.float64)       # one FP16 subtraction, exact
    assert np.array_equal(widened, codes.astype(np.float64))


def test_int8_score_products_accumulate_exactly_in_fp32():
    # Q K^T on the FP16 codes with an FP32 accumulator: every product (<= 127^2) and every
    # partial sum over the 128 channels (<= 128 * 127^2 < 2^24) is an integer binary32 holds
    assert 128 * 127 * 127 < 2 ** 24
    rng = np.random.default_rng(5)
    q = rng.integers(-127, 128, size=(64, 128)).astype(np.float32)
    k = rng.integers(-127, 128, size=(64, 128)).astype(np.float32)
    acc = np.zeros((64, 64), dtype=np.float32)
    for c in range(128):                                       # sequential binary32 accumulation
        acc = acc + np.outer(q[:, c], k[:, c]).astype(np.float32)
    assert np.array_equal(acc.astype(np.int64), q.astype(np.int64) @ k.astype(np.int64).T)
