"""Oracle pins: the matvec.

* brute force over every int2 code vector of length 8, on inputs chosen so
  that every fp32 partial sum is exact: the oracle must then equal the exact
  rational value (computed here in integers), whatever the order;
* the same for int4 / int8 code ranges on random rows;
* hand-derived cases whose fp32 result depends on the accumulation order
  (serial in k inside a block, serial over groups, scale applied with its own
  rounding and no fused multiply-add, one scale per row for group == K);
* the sequential-summation error bound against the exact value on general
  fp16 inputs;
* special cases (all codes zero; one live group).
"""
import itertools
from fractions import Fraction

import numpy as np
import pytest

F16 = np.float16


def h(vals):
    return np.asarray(vals, dtype=np.float64).astype(F16)


def test_bruteforce_int2_k8_exact(orc):
    K = 8
    codes = np.array(list(itertools.product([-2, -1, 0, 1], repeat=K)), np.int8)  # 65536 x 8
    N = codes.shape[0]
    rng = np.random.default_rng(1)
    for group in (8, 4, 2):
        G = K // group
        for trial in range(3):
            y8 = rng.integers(-64, 65, size=K)                    # y = y8 / 8
            s4 = rng.integers(1, 8, size=(N, G))                   # s = s4 / 4
            y = h(y8 / 8.0)
            s = h(s4 / 4.0)
            out = orc.gemv(codes, s, group, y[None])[0]
            # exact: sum_g (sum_{k in g} y8_k v_k) * s4_g / 32
            prod = codes.astype(np.int64) * y8[None, :]
            gsum = prod.reshape(N, G, group).sum(axis=2)
            exact32 = (gsum * s4).sum(axis=1)
            assert np.array_equal(out.astype(np.float64) * 32.0, exact32.astype(np.float64))


@pytest.mark.parametrize("bits", [4, 8])
def test_wide_codes_exact(orc, bits):
    rng = np.random.default_rng(bits)
    N, K, group = 512, 128, 32
    lo, hi = -(1 << (bits - 1)), 1 << (bits - 1)
    codes = rng.integers(lo, hi, size=(N, K)).astype(np.int8)
    y8 = rng.integers(-8, 9, size=K)
    s4 = rng.integers(1, 8, size=(N, K // group))
    out = orc.gemv(codes, h(s4 / 4.0), group, h(y8 / 8.0)[None])[0]
    gsum = (codes.astype(np.int64) * y8).reshape(N, K // group, group).sum(axis=2)
    exact32 = (gsum * s4).sum(axis=1)
    assert np.array_equal(out.astype(np.float64) * 32.0, exact32.astype(np.float64))


def test_per_row_group_exact(orc):
    rng = np.random.default_rng(3)
    N, K = 256, 96
    codes = rng.integers(-128, 128, size=(N, K)).astype(np.int8)
    y8 = rng.integers(-4, 5, size=K)
    s4 = rng.integers(1, 8, size=(N, 1))
    out = orc.gemv(codes, h(s4 / 4.0), K, h(y8 / 8.0)[None])[0]
    exact32 = (codes.astype(np.int64) * y8).sum(axis=1) * s4[:, 0]
    assert np.array_equal(out.astype(np.float64) * 32.0, exact32.astype(np.float64))


A = 65504.0          # largest fp16; fp32 spacing at A is 2^-8
E = 2.0 ** -10       # a quarter of that spacing


def _one_row(y, v, s, group):
    y = h(y)
    codes = np.asarray(v, np.int8)[None]
    return float(orc_gemv(codes, h(s)[None], group, y[None]))


def orc_gemv(codes, s, group, y):
    import oracle
    return oracle.gemv(codes, s, group, y)[0, 0]


def test_serial_order_inside_block():
    # [A, e x7]: a serial fp32 chain absorbs every e -> exactly A.
    # (a pairwise tree gives A + 2^-8; a float64 accumulator A + 7e rounded.)
    y = [A] + [E] * 7 + [0.0] * 24
    assert _one_row(y, [1] * 32, [1.0], 32) == A
    # [e x7, A]: the small terms add exactly first -> A + 7e rounds to A + 2^-7.
    # (reverse order would absorb them -> A.)
    y = [E] * 7 + [A] + [0.0] * 24
    assert _one_row(y, [1] * 32, [1.0], 32) == A + 2.0 ** -7
    # [A, e x4, -A]: fp32 result 0 although the exact value is 2^-8
    y = [A] + [E] * 4 + [-A] + [0.0] * 26
    assert _one_row(y, [1] * 32, [1.0], 32) == 0.0
    # [A, 0 x15, e x16]: one 32-code chain absorbs all sixteen e -> A.
    # (two 16-code chains added would keep 16e = 2^-6: A + 2^-6.)
    y = [A] + [0.0] * 15 + [E] * 16
    assert _one_row(y, [1] * 32, [1.0], 32) == A


def test_blocks_inside_a_long_group():
    # group == K == 64 is summed as two 32-code blocks, then the block sums
    # are added: [A, 0 x31, e x32] -> block 1 is 32e = 2^-5 exactly and
    # A + 2^-5 is representable.  One serial chain over all 64 codes would
    # absorb every e and give A.  With group 32 the two groups add the same way.
    y = [A] + [0.0] * 31 + [E] * 32
    assert _one_row(y, [1] * 64, [1.0], 64) == A + 2.0 ** -5
    assert _one_row(y, [1] * 64, [1.0, 1.0], 32) == A + 2.0 ** -5


def test_block_sums_of_a_group_added_in_fp32():
    # group == K == 128: four 32-code blocks whose sums are A, e, e, e.  Added
    # serially in fp32, each e (a quarter of the spacing at A) is absorbed:
    # the group's dot is A.  Kept in a wider type, the three e would reach
    # three quarters of a spacing and round up to A + 2^-8.
    K = 128
    y = np.zeros(K)
    y[0] = A
    y[32] = y[64] = y[96] = E
    assert _one_row(y, [1] * K, [1.0], K) == A


def test_serial_order_over_groups():
    # eight groups, each with one live term: group partials A, e, e, ... in
    # order -> every e absorbed; reversed placement -> A + 2^-7
    K = 256
    y = np.zeros(K)
    y[0] = A
    y[32::32] = E
    assert _one_row(y, [1] * K, [1.0] * 8, 32) == A
    y = np.zeros(K)
    y[0:224:32] = E
    y[224] = A
    assert _one_row(y, [1] * K, [1.0] * 8, 32) == A + 2.0 ** -7


def _fma_case():
    # group 0: y0 = 1, v = -1, s0 = 1         -> t0 = -1
    # group 1: y32 = 1 + 2^-10, y33 = 2^-13 + 2^-23, v = 1  -> p1 = 1 + 2^-10 + 2^-13 + 2^-23 (exact)
    #          s1 = 1 + 3*2^-10
    # p1*s1 = 1 + 2^-8 + 2^-13 + 3*2^-20 + 2^-21 + 3*2^-33 ; rounded to fp32 the
    # 3*2^-33 tail is dropped, so acc = -1 + fl(p1*s1) = 2^-8 + 2^-13 + 3*2^-20 + 2^-21.
    # A fused multiply-add would round 2^-8 + ... + 3*2^-33 instead and keep 2^-31.
    y = np.zeros(64)
    v = np.zeros(64, np.int64)
    y[0], v[0] = 1.0, -1
    y[32], v[32] = 1.0 + 2.0 ** -10, 1
    y[33], v[33] = 2.0 ** -13 + 2.0 ** -23, 1
    return y, v


def test_scale_step_not_fused():
    y, v = _fma_case()
    got = _one_row(y, v, [1.0, 1.0 + 3 * 2.0 ** -10], 32)
    assert got == 2.0 ** -8 + 2.0 ** -13 + 3 * 2.0 ** -20 + 2.0 ** -21
    assert got != 2.0 ** -8 + 2.0 ** -13 + 3 * 2.0 ** -20 + 2.0 ** -21 + 2.0 ** -31


def test_per_row_scale_applied_once():
    # Same codes with one scale for the whole row (group == K == 64): the two
    # 32-blocks are added first (q = 2^-10 + 2^-13 + 2^-23, exact) and q*s is
    # exact too: 2^-10 + 2^-13 + 3*2^-20 + 2^-21 + 3*2^-33.  Scaling each
    # block separately (group-32 style) would lose the 3*2^-33 tail.
    y, v = _fma_case()
    s = 1.0 + 3 * 2.0 ** -10
    got = _one_row(y, v, [s], 64)
    assert got == 2.0 ** -10 + 2.0 ** -13 + 3 * 2.0 ** -20 + 2.0 ** -21 + 3 * 2.0 ** -33
    assert _one_row(y, v, [s, s], 32) == 2.0 ** -10 + 2.0 ** -13 + 3 * 2.0 ** -20 + 2.0 ** -21


def test_zero_codes_and_single_group(orc):
    rng = np.random.default_rng(5)
    K, N = 256, 16
    y = h(rng.standard_normal(K))
    s = h(rng.uniform(0.005, 0.02, size=(N, K // 32)))
    assert np.all(orc.gemv(np.zeros((N, K), np.int8), s, 32, y[None]) == 0.0)
    # one live group with all codes 1: the result is fl(fl(sum y) * s) with the
    # sum exact when y are small integers
    yi = h(rng.integers(-20, 21, size=K).astype(np.float64))
    codes = np.zeros((N, K), np.int8)
    codes[:, 64:96] = 1
    out = orc.gemv(codes, s, 32, yi[None])[0]
    ysum = np.float32(yi[64:96].astype(np.float64).sum())
    assert np.array_equal(out, (ysum * s[:, 2].astype(np.float32)).astype(np.float32))


def _exact(codes, s, group, y):
    # exact rational value: every fp16 is an integer multiple of 2^-24
    N, K = codes.shape
    G = K // group
    yi = [int(Fraction(float(t)) * 2 ** 24) for t in y]
    out = []
    for n in range(N):
        tot = 0
        for g in range(G):
            si = int(Fraction(float(s[n, g])) * 2 ** 24)
            dot = sum(yi[k] * int(codes[n, k]) for k in range(g * group, (g + 1) * group))
            tot += dot * si
        out.append(Fraction(tot, 2 ** 48))
    return out


@pytest.mark.parametrize("bits,group,K", [(2, 32, 64), (2, 32, 128), (4, 32, 96), (8, 96, 96), (8, 32, 64)])
def test_error_bound_general_inputs(orc, bits, group, K):
    rng = np.random.default_rng(K + bits)
    N = 24
    lo, hi = -(1 << (bits - 1)), 1 << (bits - 1)
    codes = rng.integers(lo, hi, size=(N, K)).astype(np.int8)
    y = h(rng.standard_normal(K) * 3)
    s = h(rng.uniform(0.005, 0.02, size=(N, K // group)))
    got = orc.gemv(codes, s, group, y[None])[0]
    exact = _exact(codes, s, group, y)
    u = 2.0 ** -24
    n_ops = min(group, 32) + (group // 32 if group > 32 else 0) + K // group + 1
    gam = n_ops * u / (1 - n_ops * u)
    for n in range(N):
        mag = sum(abs(float(y[k]) * int(codes[n, k]) * float(s[n, k // group])) for k in range(K))
        err = abs(Fraction(float(got[n])) - exact[n])
        assert float(err) <= gam * mag + 1e-45, (n, float(err), gam * mag)


def test_columns_independent(orc):
    # M columns give the same result as M separate calls
    rng = np.random.default_rng(9)
    N, K, M = 40, 128, 5
    codes = rng.integers(-2, 2, size=(N, K)).astype(np.int8)
    s = h(rng.uniform(0.005, 0.02, size=(N, K // 32)))
    y = h(rng.standard_normal((M, K)))
    out = orc.gemv(codes, s, 32, y)
    for m in range(M):
        assert np.array_equal(out[m], orc.gemv(codes, s, 32, y[m:m + 1])[0])
