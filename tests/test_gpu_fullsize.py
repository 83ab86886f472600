"""Parity at the full sizes of the five workloads, in the launch
configurations the bench uses (fast mode, within 1e-3*(1+|ref|)) and in exact
mode (bit-exact up to 32 columns), on sampled output rows the oracle computes one
by one (first and last rows plus random ones; inputs regenerated on the host
from the same seeded streams, never read back from the GPU).

  1  single int2 GEMV 1024x1024 with the fused RMSNorm prologue (every row)
  2/3 decode layer (d_model 2048): fused q/k/v int4 2560x2048, o int4, fused
      gate/up int2 2*d_ff x 2048, down int2 2048 x d_ff (d_ff 8192 and 16384),
      per-row int8 2048x2048 projection, int2 lm_head 262144x2048
  4  int2 FFN d_model 4096: gate/up 28672x4096, down 4096x14336, M in
      {1,4,8,16} bit-exact and {64,128} within tolerance (tensor tiles)
  5  int4/int8 d_model 5376, d_ff 21504, 0.1% outliers, fused prologue,
      M in {1, 8, 32}; lm_head int4 262144x5376
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import (EPS, Mat, acts, bits_equal, first_diff, max_rel_err, sample_rows, to_dev,
                      within_tol, qmv)

pytestmark = pytest.mark.gpu


def _check_rows(ys, mat, rows, y16_in):
    """ys: {"fast": y, "exact": y or None}; fast within tolerance, exact bit-exact"""
    codes, scales = mat.host(rows)
    ref = oracle.gemv(codes, scales, mat.group, y16_in)
    got = ys["fast"].cpu().numpy()[:, rows]
    assert within_tol(got, ref), max_rel_err(got, ref)
    if ys.get("exact") is not None:
        got = ys["exact"].cpu().numpy()[:, rows]
        assert bits_equal(got, ref), first_diff(got, ref)


def _both(fn, exact=True):
    """run fn(mode) in fast mode (the bench's) and, if asked, in exact mode"""
    q = qmv()
    ys = {"fast": fn(q.QMV_FAST), "exact": fn(q.QMV_EXACT) if exact else None}
    torch.cuda.synchronize()
    return ys


def _fused(mat, M, name, outliers=False, exact_rows=None):
    q = qmv()
    x, r, g = acts(name, M, mat.K, outliers)
    h = torch.empty(M, mat.K, dtype=torch.float16, device="cuda")
    ys = _both(lambda md: q.qmv_fused_rmsnorm_gemv(mat.pack, to_dev(x), to_dev(r), to_dev(g), EPS,
                                                   h_out=h, mode=md))
    h_ref, y16, _ = oracle.fused_rmsnorm_gemv(np.zeros((1, mat.K), np.int8),
                                              np.zeros((1, mat.K // mat.group), np.float16),
                                              mat.group, x, r, g, EPS)
    assert np.array_equal(h.cpu().numpy().view(np.uint16), h_ref)
    rows = sample_rows(mat.N) if exact_rows is None else exact_rows
    _check_rows(ys, mat, rows, y16)


def test_config1_single_int2_gemv_all_rows():
    m = Mat("full.c1", 1024, 1024, 2, 32)
    _fused(m, 1, "full.c1", exact_rows=np.arange(1024))


@pytest.mark.parametrize("d_ff", [8192, 16384])
def test_decode_layer(d_ff):
    q = qmv()
    qkv = Mat(f"full.L{d_ff}.qkv", 2560, 2048, 4, 32)
    o = Mat(f"full.L{d_ff}.o", 2048, 2048, 4, 32)
    gu = Mat(f"full.L{d_ff}.gateup", 2 * d_ff, 2048, 2, 32)
    dn = Mat(f"full.L{d_ff}.down", 2048, d_ff, 2, 32)
    _fused(qkv, 1, f"full.L{d_ff}.qkv")
    _fused(gu, 1, f"full.L{d_ff}.gu")
    for mat in (o, dn):
        x, _, _ = acts(f"full.L{d_ff}.{mat.name}", 1, mat.K)
        ys = _both(lambda md: q.qmv_gemv(mat.pack, to_dev(x), mode=md))
        _check_rows(ys, mat, sample_rows(mat.N), x)


def test_per_row_int8_projection_and_int2_lm_head():
    q = qmv()
    ple = Mat("full.ple", 2048, 2048, 8, 2048)
    x, _, _ = acts("full.ple", 1, 2048)
    ys = _both(lambda md: q.qmv_gemv(ple.pack, to_dev(x), mode=md))
    _check_rows(ys, ple, np.arange(2048), x)
    head = Mat("full.head2", 262144, 2048, 2, 32)
    x, _, _ = acts("full.head2", 1, 2048)
    ys = _both(lambda md: q.qmv_gemv(head.pack, to_dev(x), mode=md))
    _check_rows(ys, head, sample_rows(262144, 512), x)


@pytest.fixture(scope="module")
def ffn4096():
    return (Mat("full.c4.gateup", 28672, 4096, 2, 32), Mat("full.c4.down", 4096, 14336, 2, 32))


@pytest.mark.parametrize("M", [1, 4, 8, 16, 64, 128])
def test_config4_chunk_sweep(ffn4096, M):
    q = qmv()
    for mat in ffn4096:
        x, _, _ = acts(f"full.c4.{mat.name}.m{M}", M, mat.K)
        rows = sample_rows(mat.N, 128)
        ys = _both(lambda md: q.qmv_chunk_gemm(mat.pack, to_dev(x), mode=md))
        _check_rows(ys, mat, rows, x)
        if M > 1:
            y1 = _both(lambda md: q.qmv_gemv(mat.pack, to_dev(x[M - 1:M]), mode=md))
            # the last column of the tile equals the M = 1 result bit for bit:
            # always in exact mode, and in fast mode for the CUDA-core tiles
            assert bits_equal(ys["exact"].cpu().numpy()[M - 1], y1["exact"].cpu().numpy()[0])
            if M <= 32:
                assert bits_equal(ys["fast"].cpu().numpy()[M - 1], y1["fast"].cpu().numpy()[0])
    assert q.qmv_device_error(clear=True) == 0


@pytest.fixture(scope="module")
def set5():
    return {
        "gateup": Mat("full.c5.gateup", 43008, 5376, 4, 32),
        "down": Mat("full.c5.down", 5376, 21504, 4, 32),
        "q": Mat("full.c5.q", 8192, 5376, 8, 5376),
        "k": Mat("full.c5.k", 2048, 5376, 8, 5376),
        "v": Mat("full.c5.v", 2048, 5376, 8, 5376),
    }


@pytest.mark.parametrize("M", [1, 8, 32])
def test_config5_mixed_int4_int8_with_outliers(set5, M):
    q = qmv()
    for name in ("gateup", "q", "k", "v"):
        _fused(set5[name], M, f"full.c5.{name}.m{M}", outliers=True,
               exact_rows=sample_rows(set5[name].N, 96))
    x, _, _ = acts(f"full.c5.down.m{M}", M, 21504, outliers=True)
    dn = set5["down"].pack
    ys = _both(lambda md: q.qmv_chunk_gemm(dn, to_dev(x), mode=md) if M > 1
               else q.qmv_gemv(dn, to_dev(x), mode=md))
    _check_rows(ys, set5["down"], sample_rows(5376, 96), x)


def test_config5_int4_lm_head():
    q = qmv()
    head = Mat("full.c5.head", 262144, 5376, 4, 32)
    for M in (1, 8):
        x, _, _ = acts(f"full.c5.head.m{M}", M, 5376, outliers=True)
        ys = _both(lambda md: q.qmv_gemv(head.pack, to_dev(x), mode=md) if M == 1
                   else q.qmv_chunk_gemm(head.pack, to_dev(x), mode=md))
        _check_rows(ys, head, sample_rows(262144, 128), x)
