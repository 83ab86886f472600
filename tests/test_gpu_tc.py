"""GPU parity of the tcgen05 tensor-core tiles (M > 32 token columns, fast
mode, int2 weights) against the oracle, within max |y - ref| <= 1e-3*(1+|ref|);
and the exact-mode / int4 paths at M > 32, which stay bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import Mat, acts, bits_equal, first_diff, to_dev, within_tol, qmv

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,K,group", [(300, 1024, 32), (128, 4096, 32), (1000, 2048, 2048),
                                       (64, 64, 32), (2048, 4096, 32)])
@pytest.mark.parametrize("M", [33, 64, 65, 100, 128, 200])
def test_tensor_tiles_within_tolerance(N, K, group, M):
    q = qmv()
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
    q = qmv()
    m = Mat("tc_f16", 512, 2048, 2, 32)
    x, _, _ = acts("tc_f16", 64, 2048)
    y = q.qmv_chunk_gemm(m.pack, to_dev(x), y_dtype=q.QMV_F16, mode=q.QMV_FAST)
    torch.cuda.synchronize()
    codes, scales = m.host()
    ref = oracle.gemv(codes, scales, 32, x)
    assert within_tol(y.cpu().float().numpy(), ref, 2e-3)


def test_tensor_tiles_repeatable_without_split():
    q = qmv()
    m = Mat("tc_rep", 4096, 1024, 2, 32)          # 32 row tiles: no split
    x, _, _ = acts("tc_rep", 128, 1024)
    a = q.qmv_chunk_gemm(m.pack, to_dev(x))
    b = q.qmv_chunk_gemm(m.pack, to_dev(x))
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("bits,M", [(4, 64), (8, 40), (2, 48)])
def test_exact_or_wide_codes_above_32_columns_bit_exact(bits, M):
    q = qmv()
    m = Mat(f"ex{bits}", 200, 1024, bits, 32)
    x, _, _ = acts(f"ex{bits}m{M}", M, 1024)
    mode = q.QMV_EXACT if bits == 2 else q.QMV_FAST
    y = q.qmv_chunk_gemm(m.pack, to_dev(x), mode=mode)
    torch.cuda.synchronize()
    codes, scales = m.host()
    ref = oracle.gemv(codes, scales, 32, x)
    assert bits_equal(y.cpu().numpy(), ref), first_diff(y.cpu().numpy(), ref)
