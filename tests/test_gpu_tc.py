"""GPU parity of the tcgen05 tensor-core tiles (M > 32 token columns, fast
mode, int2 weights) against the oracle, within max |y - ref| <= 1e-3*(1+|ref|);
the exact mode at M > 32, which stays bit-exact; and the fast int4/int8 tiles
at M > 32."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import Mat, acts, bits_equal, first_diff, max_rel_err, to_dev, within_tol, qmv, qmv_guarded

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,K,group", [(300, 1024, 32), (128, 4096, 32), (1000, 2048, 2048),
                                       (64, 64, 32), (2048, 4096, 32)])
@pytest.mark.parametrize("M", [33, 64, 65, 100, 128, 200])
def test_tensor_tiles_within_tolerance(N, K, group, M):
    q = qmv_guarded()
    m = Mat(f"tc{N}x{K}g{group}", N, K, 2, group)
    x, _, _ = acts(f"tc{N}x{K}m{M}", M, K)
    y = q.qmv_chunk_gemm(m.pack, to_dev(x), mode=q.QMV_FAST)
    torch.cuda.synchronize()
    codes, scales = m.host()
    ref = oracle.gemv(codes, scales, group, x)
    got = y.cpu().numpy()
    err = np.max(np.abs(got.astype(np.float64) - ref) / (1 + np.abs(ref)))
    assert within_tol(got, ref), f"max scaled error {err}"
    assert q.qmv_device_error(clear=True) == 0


def test_tensor_tiles_fp16_output():
    q = qmv_guarded()
    m = Mat("tc_f16", 512, 2048, 2, 32)
    x, _, _ = acts("tc_f16", 64, 2048)
    y = q.qmv_chunk_gemm(m.pack, to_dev(x), y_dtype=q.QMV_F16, mode=q.QMV_FAST)
    torch.cuda.synchronize()
    codes, scales = m.host()
    ref = oracle.gemv(codes, scales, 32, x)
    assert within_tol(y.cpu().float().numpy(), ref, 2e-3)


@pytest.mark.parametrize("N,K", [(4096, 1024), (2048, 8192), (28672, 4096)])
def test_tensor_tiles_repeatable(N, K):
    """split-K partials are added in split order by a second kernel: the same
    call gives the same bits every time (16 to 224 row tiles, splits 1 to 8)"""
    q = qmv_guarded()
    m = Mat(f"tc_rep{N}x{K}", N, K, 2, 32)
    x, _, _ = acts(f"tc_rep{N}", 128, K)
    xd = to_dev(x)
    ys = [q.qmv_chunk_gemm(m.pack, xd) for _ in range(3)]
    torch.cuda.synchronize()
    for y in ys[1:]:
        assert torch.equal(y.view(torch.int32), ys[0].view(torch.int32))
    assert q.qmv_device_error(clear=True) == 0


@pytest.mark.parametrize("M", [64, 128])
def test_tensor_tiles_split_fp16_is_rne_of_fp32(M):
    """down-projection shape (16 row tiles, split K): the fp16 output is the RNE
    of the fp32 output, and both are within tolerance of the oracle"""
    q = qmv_guarded()
    N, K = 2048, 8192
    m = Mat("tc_split16", N, K, 2, 32)
    x, _, _ = acts(f"tc_split16m{M}", M, K)
    xd = to_dev(x)
    y = q.qmv_chunk_gemm(m.pack, xd, mode=q.QMV_FAST)
    y16 = q.qmv_chunk_gemm(m.pack, xd, y_dtype=q.QMV_F16, mode=q.QMV_FAST)
    torch.cuda.synchronize()
    got = y.cpu().numpy()
    assert np.array_equal(y16.cpu().numpy().view(np.uint16), oracle.f32_to_f16(got))
    rows = np.arange(0, N, 7)
    codes, scales = m.host(rows)
    ref = oracle.gemv(codes, scales, 32, x)
    assert within_tol(got[:, rows], ref), max_rel_err(got[:, rows], ref)


@pytest.mark.parametrize("bits,M", [(4, 64), (8, 40), (2, 48)])
def test_exact_above_32_columns_bit_exact(bits, M):
    q = qmv_guarded()
    m = Mat(f"ex{bits}", 200, 1024, bits, 32)
    x, _, _ = acts(f"ex{bits}m{M}", M, 1024)
    y = q.qmv_chunk_gemm(m.pack, to_dev(x), mode=q.QMV_EXACT)
    torch.cuda.synchronize()
    codes, scales = m.host()
    ref = oracle.gemv(codes, scales, 32, x)
    assert bits_equal(y.cpu().numpy(), ref), first_diff(y.cpu().numpy(), ref)


@pytest.mark.parametrize("bits,M", [(4, 64), (8, 40)])
def test_fast_wide_codes_above_32_columns(bits, M):
    """int4/int8 above 32 columns run the CUDA-core tiles in 32-column chunks:
    within tolerance, and every column equal to the fast M = 1 result."""
    q = qmv_guarded()
    m = Mat(f"ex{bits}", 200, 1024, bits, 32)
    x, _, _ = acts(f"ex{bits}m{M}", M, 1024)
    y = q.qmv_chunk_gemm(m.pack, to_dev(x), mode=q.QMV_FAST)
    y1 = [q.qmv_gemv(m.pack, to_dev(x[i:i + 1]), mode=q.QMV_FAST) for i in (0, 31, 32, M - 1)]
    torch.cuda.synchronize()
    codes, scales = m.host()
    ref = oracle.gemv(codes, scales, 32, x)
    got = y.cpu().numpy()
    assert within_tol(got, ref), max_rel_err(got, ref)
    for yi, i in zip(y1, (0, 31, 32, M - 1)):
        assert bits_equal(got[i], yi.cpu().numpy()[0])
