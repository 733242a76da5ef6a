"""The hardware e4m3 conversion against the oracle's encoder, exhaustively.

`cvt.rn.satfinite.e4m3x2.f32` turns the prepare's scaled V into its e4m3 codes
and the Sage forward's P into the operand of its FP8 P V product (the aiter pull
request "gfx1201_sage_prepare / gfx1201_sage_attention", Technical Details and
commit message of gfx1201_sage_attention).  sage_e4m3_encode runs the same
packing on arbitrary binary32 values, so the conversion is compared here with
`oracle.e4m3_encode` on every binary32 bit pattern of magnitude up to 448, both
signs, on a stride through the rest of the finite range, where both must
saturate to +-448, and on the special values (infinities, NaN, signed zeros).  The oracle's encoder is itself pinned against torch's cast on
the same patterns below 448 (tests/test_oracle_prepare.py).
"""
import numpy as np
import pytest
import torch

import oracle
import sage_attention_forward_gb300 as sa

TOP = 0x43E00000          # the bit pattern of 448.0
FINITE_END = 0x7F800000   # the first non-finite pattern


def _compare(bits: np.ndarray, dev) -> None:
    x = bits.view(np.float32)
    want = oracle.e4m3_encode(x)
    got = sa.e4m3_encode(torch.from_numpy(x).to(dev)).cpu().numpy()
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, (f"{bad.size} mismatches; first at bits {int(bits[bad[0]]):#010x}: "
                           f"hardware {int(got[bad[0]]):#04x}, oracle {int(want[bad[0]]):#04x}")


@pytest.mark.gpu
@pytest.mark.parametrize("sign", [0, 0x80000000])
def test_every_binary32_up_to_448(cuda_dev, sign):
    chunk = 1 << 27
    for start in range(0, TOP + 1, chunk):
        bits = np.arange(start, min(start + chunk, TOP + 1), dtype=np.uint32) | np.uint32(sign)
        _compare(bits, cuda_dev)


@pytest.mark.gpu
def test_saturation_beyond_448(cuda_dev):
    # every 4093rd finite pattern above 448 (with the largest finite one), both signs
    pos = np.append(np.arange(TOP + 1, FINITE_END, 4093, dtype=np.uint32), np.uint32(FINITE_END - 1))
    bits = np.concatenate([pos, pos | np.uint32(0x80000000)])
    _compare(bits, cuda_dev)
    got = sa.e4m3_encode(torch.from_numpy(bits.view(np.float32)).to(cuda_dev)).cpu().numpy()
    assert np.all((got & 0x7F) == 126)


@pytest.mark.gpu
def test_ragged_lengths_and_offsets(cuda_dev):
    # lengths that leave 1-3 values after the last group of four, and inputs that start
    # off a 16-byte boundary: every value written, nothing past n
    g = np.random.default_rng(5)
    for n in (1, 2, 3, 5, 1023, 4097):
        x = (g.standard_normal(n + 3) * 100).astype(np.float32)
        xd = torch.from_numpy(x).to(cuda_dev)
        for off in (0, 1, 3):
            out = torch.full((n + 8,), 0xAB, dtype=torch.uint8, device=cuda_dev)
            sa.e4m3_encode(xd[off:off + n], out=out[:n])
            o = out.cpu().numpy()
            assert np.array_equal(o[:n], oracle.e4m3_encode(x[off:off + n]))
            assert (o[n:] == 0xAB).all()


@pytest.mark.gpu
def test_special_values(cuda_dev):
    # +-inf saturate to +-448 like every magnitude beyond it; NaN gives an e4m3 NaN (S.1111.111),
    # whose sign bit neither side fixes; signed zeros keep their sign
    x = np.array([np.inf, -np.inf, np.nan, -np.nan, 0.0, -0.0, 448.0, -448.0, 464.0, -464.0], dtype=np.float32)
    got = sa.e4m3_encode(torch.from_numpy(x).to(cuda_dev)).cpu().numpy()
    want = oracle.e4m3_encode(x)
    assert np.array_equal(got[:2], np.array([0x7E, 0xFE], dtype=np.uint8))
    assert np.array_equal(got[:2], want[:2])
    assert ((got[2:4] & 0x7F) == 0x7F).all() and ((want[2:4] & 0x7F) == 0x7F).all()
    assert np.array_equal(got[4:], want[4:])
    assert np.array_equal(got[4:6], np.array([0x00, 0x80], dtype=np.uint8))
