"""Pins of the exactness the matvec's fixed order rests on.

* Every product of an fp16 activation and a code is exact in fp32, for all
  three widths. An fp16 significand has 11 bits and a code at most 8, and
  11 + 8 <= 24. Only the additions round, so the result depends on their
  order alone, and an FMA in the inner dot gives the same value as a
  multiply followed by an add. This is checked exhaustively: every finite
  fp16 value against every int8 code, which includes every int2 and int4
  code, through the oracle's own matvec with K = 1 and scale 1.
* For int2, x*c is also representable in fp16 whenever |x| <= 32752, the
  largest fp16 whose double is still finite.
"""
import numpy as np


def _finite_f16():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = h.view(np.float16)
    return f[np.isfinite(f)]


def test_every_product_exact_in_fp32(orc):
    y = _finite_f16()                                     # 63488 values
    codes = np.arange(-128, 128, dtype=np.int64).astype(np.int8)[:, None]   # N = 256, K = 1
    ones = np.ones((256, 1), np.float16)
    out = orc.gemv(codes, ones, 1, y[:, None])            # [M = 63488, N = 256]
    exact = y.astype(np.float64)[:, None] * codes[:, 0].astype(np.float64)[None, :]
    assert np.array_equal(out.astype(np.float64), exact)


def test_int2_products_representable_in_fp16():
    y = _finite_f16().astype(np.float64)
    y = y[np.abs(y) <= 32752.0]
    for c in (-2, -1, 0, 1):
        p = y * c
        assert np.array_equal(p.astype(np.float16).astype(np.float64), p)
    # the bound is tight: the next fp16, 32768, doubles past the largest fp16
    assert 32768.0 * 2.0 > float(np.finfo(np.float16).max) == 65504.0
