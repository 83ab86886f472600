"""Oracle pins: the oracle's own IEEE binary16 conversions.

Checked against numpy's float16 conversion (an independent library routine):
exhaustively for binary16 -> binary32, and for binary32 -> binary16 on every
boundary class plus a large random sweep of bit patterns.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.filterwarnings("ignore:overflow encountered in cast")


def test_f16_to_f32_exhaustive(orc):
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = orc.f16_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(got.view(np.uint32)[~nan], ref.view(np.uint32)[~nan])
    assert np.isnan(got[nan]).all()


def test_f16_roundtrip_exhaustive(orc):
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = orc.f16_to_f32(h)
    back = orc.f32_to_f16(f)
    nan = np.isnan(f)
    assert np.array_equal(back[~nan], h[~nan])
    assert np.isnan(back[nan].view(np.float16)).all()


def test_f32_to_f16_boundaries(orc):
    # every binary16 value, and the midpoints between neighbours (ties), and
    # points just off the midpoints, covers the rounding rule everywhere
    h = np.arange(0, 0x7C00, dtype=np.uint32).astype(np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    mid = ((lo + hi) / 2).astype(np.float32)          # exact in fp32
    for v in (lo.astype(np.float32), mid,
              np.nextafter(mid, np.float32(np.inf)),
              np.nextafter(mid, np.float32(0))):
        for s in (1.0, -1.0):
            x = (v * np.float32(s)).astype(np.float32)
            assert np.array_equal(orc.f32_to_f16(x), x.astype(np.float16).view(np.uint16))
    special = np.array([65504.0, 65519.996, 65520.0, 1e30, np.inf, -np.inf, 0.0, -0.0,
                        2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -26, 1e-40,
                        2.0 ** -14, 2.0 ** -14 - 2.0 ** -25], dtype=np.float32)
    assert np.array_equal(orc.f32_to_f16(special), special.astype(np.float16).view(np.uint16))


def test_f32_to_f16_random_bits(orc):
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 1 << 32, size=1 << 23, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[~np.isnan(x)]
    assert np.array_equal(orc.f32_to_f16(x), x.astype(np.float16).view(np.uint16))
    # and the range that matters for activations: |x| < 2^17
    y = (rng.standard_normal(1 << 22) * rng.choice([1e-6, 1e-3, 1.0, 1e3, 6e4], 1 << 22)
         ).astype(np.float32)
    assert np.array_equal(orc.f32_to_f16(y), y.astype(np.float16).view(np.uint16))
