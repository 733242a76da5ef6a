"""The rounding argument behind the prepare's BF16 arithmetic (CPU only): for
finite BF16 operands, eager BF16 -- compute in binary32, round to BF16 -- gives
the same value as rounding the exact product or sum to BF16 once, which is what
mul/add.rn.bf16x2 compute.  A BF16 x BF16 product has a 16-bit significand, so
it is exact in binary32 down to 2^-149 and below that it lies under the
smallest BF16 rounding midpoint; a sum is exact in binary32 unless the
exponents differ by more than 15, and then the smaller term is far below half a
BF16 ulp of the larger.  Checked on random operands over the whole finite
range plus the subnormal and overflow edges, with exact float64 arithmetic
(products exact, sums exact or far from any BF16 midpoint)."""
import numpy as np

import oracle


def bf16_rne(x):
    """float64 -> the nearest BF16 value (ties to even), as float64; +-inf beyond the range."""
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, copy=True)
    fin = np.isfinite(x) & (x != 0)
    _, e = np.frexp(np.abs(x[fin]))               # |x| = m 2^e, m in [1/2, 1)
    spacing = np.exp2(np.maximum(e - 1, -126) - 7)  # 8 significant bits; subnormal spacing 2^-133
    r = np.rint(x[fin] / spacing) * spacing
    r[np.abs(r) >= 2.0 ** 128] = np.inf * np.sign(r[np.abs(r) >= 2.0 ** 128])
    out[fin] = r
    return out


def eager(x64):
    """Eager BF16: the binary32 result, then rounded to BF16."""
    with np.errstate(over="ignore"):
        f32 = x64.astype(np.float32)
    return bf16_rne(f32.astype(np.float64))


def operands(n, seed):
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 1 << 16, size=2 * n, dtype=np.uint32).astype(np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80][: n]                  # finite only
    # edges: subnormals, the smallest normals, values next to the largest
    edge = np.concatenate([np.arange(1, 0x100), np.arange(0x7E00, 0x7F80)]).astype(np.uint16)
    edge = np.concatenate([edge, edge | 0x8000])
    b = np.concatenate([bits, edge])
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_bf16_rne_matches_the_oracle_cast():
    x = np.random.default_rng(3).standard_normal(200000).astype(np.float32) * np.float32(1e3)
    ours = bf16_rne(x.astype(np.float64))
    ref = (oracle.f32_to_bf16(x).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.array_equal(ours, ref)


def test_products_round_once():
    a, b = operands(400000, 1), operands(400000, 2)[::-1]
    n = min(a.size, b.size)
    a, b = a[:n], b[:n]
    prod = a * b                                   # exact in binary64
    assert np.array_equal(eager(prod), bf16_rne(prod))


def test_sums_round_once():
    a, b = operands(400000, 5), operands(400000, 6)[::-1]
    n = min(a.size, b.size)
    a, b = a[:n], b[:n]
    s = a + b                                      # exact, or far from every BF16 midpoint
    assert np.array_equal(eager(s), bf16_rne(s))


def test_the_comparison_sees_double_rounding():
    # 2^-30 above the BF16 midpoint between 1 and 1 + 2^-7: binary32 rounds onto the midpoint,
    # whose tie goes to even (1), while the single rounding goes up -- the two paths differ,
    # so the equalities above are not vacuous
    x = np.array([1.0 + 2.0 ** -8 + 2.0 ** -30, -(1.0 + 2.0 ** -8 + 2.0 ** -30)])
    assert np.array_equal(eager(x), [1.0, -1.0])
    assert np.array_equal(bf16_rne(x), [1.0 + 2.0 ** -7, -(1.0 + 2.0 ** -7)])
