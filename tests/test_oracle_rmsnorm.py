"""Oracle pins: residual add + RMSNorm.

* fused == unfused, bitwise (two separately written code paths);
* zero input, constant input, tiny input (eps inside the root), each against
  the definition y = h / sqrt(mean(h^2) + eps) * gamma evaluated in float64;
* random inputs within 2 fp16 ulp of the float64 definition;
* the blocked sum-of-squares order on a hand-derived case.
"""
import numpy as np
import pytest

F16 = np.float16
EPS = 1e-6


def _ref64(h, gamma, eps=EPS):
    h = h.astype(np.float64)
    return h / np.sqrt(np.mean(h * h) + eps) * gamma.astype(np.float64)


def _ulp16(v):
    v = np.abs(v.astype(np.float64))
    e = np.floor(np.log2(np.maximum(v, 2.0 ** -14)))
    return 2.0 ** (e - 10)


@pytest.mark.parametrize("K", [32, 96, 1024, 2048, 5376, 50])
def test_fused_equals_unfused(orc, K):
    rng = np.random.default_rng(K)
    M = 3
    x = rng.standard_normal((M, K)).astype(F16)
    r = rng.standard_normal((M, K)).astype(F16)
    g = (1 + 0.1 * rng.standard_normal(K)).astype(F16)
    hf, yf = orc.fused_residual_rmsnorm(x, r, g, EPS)
    for m in range(M):
        hu = orc.residual_add(x[m], r[m])
        yu = orc.rmsnorm(hu, g, EPS, order=0)
        assert np.array_equal(hf[m], hu)
        assert np.array_equal(yf[m], yu)


def test_zero_input(orc):
    K = 256
    z = np.zeros(K, F16)
    g = np.full(K, 1.5, F16)
    h, y = orc.fused_residual_rmsnorm(z, z, g, EPS)
    assert np.all(y == 0) and np.all(h == 0)
    x = np.linspace(-3, 3, K).astype(F16)
    h, y = orc.fused_residual_rmsnorm(x, -x, g, EPS)      # x + (-x) = 0 exactly
    assert np.all(y.view(F16).astype(np.float32) == 0)


@pytest.mark.parametrize("a", [3.0, -0.75, 100.0, 2.0 ** -12])
def test_constant_input(orc, a):
    K = 512
    h = np.full(K, a, F16)
    g = np.linspace(0.8, 1.2, K).astype(F16)
    y = orc.rmsnorm(h, g, EPS).view(F16)
    ref = _ref64(h, g)
    assert np.all(np.abs(y.astype(np.float64) - ref) <= _ulp16(ref))


def test_eps_inside_root(orc):
    # h = 2^-12: mean(h^2) = 2^-24 ~ 6e-8 is small next to eps = 1e-6, so
    # y = 2^-12 / sqrt(2^-24 + 1e-6) = 0.2372...; without eps it would be 1.0,
    # with eps outside the root 0.996.
    K = 64
    h = np.full(K, 2.0 ** -12, F16)
    g = np.ones(K, F16)
    y = orc.rmsnorm(h, g, EPS).view(F16).astype(np.float64)
    assert np.all(np.abs(y - 0.23717) < 2e-4)


def test_gamma_used_as_is(orc):
    # h = 3 everywhere, gamma = 0.5 -> y = 0.5 (a (1 + gamma) form would give 0.75)
    K = 32
    y = orc.rmsnorm(np.full(K, 3.0, F16), np.full(K, 0.5, F16), EPS).view(F16)
    assert np.all(y == F16(0.5))


@pytest.mark.parametrize("K", [1024, 2048, 5376])
def test_random_within_2ulp(orc, K):
    rng = np.random.default_rng(K + 1)
    x = rng.standard_normal(K).astype(F16)
    r = rng.standard_normal(K).astype(F16)
    g = (1 + 0.1 * rng.standard_normal(K)).astype(F16)
    hb, yb = orc.fused_residual_rmsnorm(x, r, g, EPS)
    hh = hb[0].view(F16)
    assert np.all(hh == (x.astype(np.float32) + r.astype(np.float32)).astype(F16))
    ref = _ref64(hh, g)
    y = yb[0].view(F16).astype(np.float64)
    assert np.all(np.abs(y - ref) <= 2 * _ulp16(ref))


def test_sumsq_block_order(orc):
    # h0 = 2048 (h0^2 = 2^22), h1..31 = 2^-7 (squares 2^-14), h32..63 = 0.25
    # (squares 2^-4).  fp32 spacing at 2^22 is 0.5, so every small square is
    # absorbed by a serial chain: 2^22.  Blocked: block 0 -> 2^22, block 1 -> 2
    # exactly, total 2^22 + 2.
    h = np.array([2048.0] + [2.0 ** -7] * 31 + [0.25] * 32, F16)
    assert orc.sumsq(h, order=0) == 2.0 ** 22 + 2
    assert orc.sumsq(h, order=1) == 2.0 ** 22
    # The block is 32 values long: h16..31 = 0.25 (squares 2^-4) sit in
    # block 0 behind h0^2 = 2^22 and are each absorbed -> 2^22.  A 16-value
    # block would sum them first to 1 and give 2^22 + 1.
    h = np.array([2048.0] + [0.0] * 15 + [0.25] * 16, F16)
    assert orc.sumsq(h, order=0) == 2.0 ** 22
    hb, yb = orc.fused_residual_rmsnorm(h, np.zeros(32, F16), np.ones(32, F16), EPS)
    assert np.array_equal(yb[0], orc.rmsnorm(h, np.ones(32, F16), EPS, order=0))


def test_normalise_then_scale_order(orc):
    # y = fp16((h * inv) * gamma): the product with inv comes first.  With
    # h = [3, 13] (K = 2), eps = 0 and gamma0 = 1557/1024, each step exactly:
    #   ss = 178, mean = 89, rt = RN(sqrt 89) = 4946123 * 2^-19,
    #   inv = RN(1 / rt) = 14227051 * 2^-27,
    #   h0 * inv = 42681153 * 2^-27 -> RN 666893 * 2^-21,
    #   times gamma0 = 1038352401 * 2^-31 -> RN 16224256 * 2^-25 = 1980.5 * 2^-12,
    # exactly halfway between two fp16 values: ties to even give 1980 * 2^-12.
    # The other order, RN(h0 * gamma0) = 4671 * 2^-10 times inv, rounds to
    # 16224257 * 2^-25, above the halfway point, and would give 1981 * 2^-12.
    h = np.array([3.0, 13.0], F16)
    g = np.array([1557 / 1024, 1.0], F16)
    y = orc.rmsnorm(h, g, 0.0).view(F16)
    assert float(y[0]) == 1980 * 2.0 ** -12
    _, yb = orc.fused_residual_rmsnorm(h, np.zeros(2, F16), g, 0.0)
    assert float(yb[0].view(F16)[0]) == 1980 * 2.0 ** -12


def test_inv_steps_each_rounded_in_fp32(orc):
    # mean = RN(ss / K), then RN(sqrt), then RN(1 / rt), each one fp32
    # operation.  With h = [7, 0, 5] (K = 3), eps = 0, gamma0 = 1485/1024:
    #   ss = 74, mean = RN(74/3) = 12932437 * 2^-19,
    #   rt = RN(sqrt mean) = 2603905 * 2^-19, inv = RN(1 / rt) = 13512157 * 2^-26,
    #   h0 * inv = 94585099 * 2^-26 -> RN 11823137 * 2^-23,
    #   times gamma0 = 17557358445 * 2^-33 -> RN 8572929 * 2^-22,
    # just above the fp16 halfway point 1046.5 * 2^-9: y0 = 1047 * 2^-9.
    # inv from a double-precision 1/sqrt (13512156 * 2^-26) or a mean taken as
    # ss * RN(1/3) (inv 13512155 * 2^-26) both give h0 * inv = 11823136 * 2^-23
    # and a product exactly on the halfway point: ties to even, 1046 * 2^-9.
    h = np.array([7.0, 0.0, 5.0], F16)
    g = np.array([1485 / 1024, 1.0, 1.0], F16)
    y = orc.rmsnorm(h, g, 0.0).view(F16)
    assert float(y[0]) == 1047 * 2.0 ** -9
    _, yb = orc.fused_residual_rmsnorm(h, np.zeros(3, F16), g, 0.0)
    assert float(yb[0].view(F16)[0]) == 1047 * 2.0 ** -9


def test_norm_uses_the_blocked_sum_of_squares(orc):
    # RMSNorm itself sums the squares in blocks of 32, then over the blocks,
    # not in one serial chain.  h0 = 100, h1..31 = 0, h32..63 = 27/64 (K = 64),
    # eps = 0, gamma0 = 1757/1024:
    #   blocked: ss = 10000 + 32 * 729/4096 = 1280729 * 2^-7,
    #     mean = 1280729 * 2^-13, rt = 3277733 * 2^-18, inv = 5367181 * 2^-26,
    #     h0 * inv -> 16772441 * 2^-21, times gamma0 -> 14389247 * 2^-20,
    #     one fp32 ulp below the fp16 halfway point 1756.5 * 2^-7: y0 = 1756 * 2^-7;
    #   one serial chain rounds each 729/4096 added to 10000 down to 182/1024:
    #     ss = 160091 * 2^-4, inv = 5367183 * 2^-26, product 14389253 * 2^-20,
    #     above the halfway point, which would give 1757 * 2^-7.
    h = np.array([100.0] + [0.0] * 31 + [27 / 64] * 32, F16)
    g = np.ones(64, F16)
    g[0] = 1757 / 1024
    assert orc.sumsq(h, order=0) == 1280729 * 2.0 ** -7
    y = orc.rmsnorm(h, g, 0.0).view(F16)
    assert float(y[0]) == 1756 * 2.0 ** -7
    _, yb = orc.fused_residual_rmsnorm(h, np.zeros(64, F16), g, 0.0)
    assert float(yb[0].view(F16)[0]) == 1756 * 2.0 ** -7
