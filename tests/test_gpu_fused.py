"""GPU parity of the fused residual-add + RMSNorm + matvec against the
oracle (bitwise for h, y16 through the matvec output, and the outputs)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import EPS, Mat, acts, bits_equal, first_diff, to_dev, within_tol, qmv, qmv_guarded

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,K,bits,group,M,outliers", [
    (1024, 1024, 2, 32, 1, False),     # single int2 GEMV with the fused prologue
    (2560, 2048, 4, 32, 1, False),     # fused prologue before q/k/v
    (16384, 2048, 2, 32, 1, False),    # fused prologue before gate/up
    (300, 5376, 4, 32, 1, True),       # d_model 5376 with 0.1% outliers at +-50
    (300, 5376, 8, 5376, 8, True),     # per-row int8 q/k/v, M = 8
    (200, 5376, 4, 32, 32, True),      # M = 32
    (77, 2048, 2, 32, 4, False),
    (50, 2048, 4, 32, 3, False),
    (33, 64, 2, 32, 1, False),
])
def test_fused_bit_exact(N, K, bits, group, M, outliers):
    q = qmv_guarded()
    m = Mat(f"fu{N}x{K}b{bits}", N, K, bits, group)
    x, r, g = acts(f"fu{N}x{K}m{M}", M, K, outliers)
    h = torch.empty(M, K, dtype=torch.float16, device="cuda")
    y = q.qmv_fused_rmsnorm_gemv(m.pack, to_dev(x), to_dev(r), to_dev(g), EPS, h_out=h,
                                 mode=q.QMV_EXACT)
    torch.cuda.synchronize()
    codes, scales = m.host()
    h_ref, y16_ref, ref = oracle.fused_rmsnorm_gemv(codes, scales, group, x, r, g, EPS)
    assert np.array_equal(h.cpu().numpy().view(np.uint16), h_ref)
    got = y.cpu().numpy()
    assert bits_equal(got, ref), first_diff(got, ref)
    # fused == unfused: the matvec of the oracle's normalised input
    y2 = q.qmv_gemv(m.pack, to_dev(y16_ref.view(np.float16)), mode=q.QMV_EXACT)
    torch.cuda.synchronize()
    assert bits_equal(y2.cpu().numpy(), got)


def test_fused_without_h_out():
    q = qmv_guarded()
    m = Mat("fu_noh", 512, 2048, 2, 32)
    x, r, g = acts("fu_noh", 1, 2048)
    y = q.qmv_fused_rmsnorm_gemv(m.pack, to_dev(x), to_dev(r), to_dev(g), EPS, mode=q.QMV_EXACT)
    yf = q.qmv_fused_rmsnorm_gemv(m.pack, to_dev(x), to_dev(r), to_dev(g), EPS, mode=q.QMV_FAST)
    torch.cuda.synchronize()
    codes, scales = m.host()
    _, _, ref = oracle.fused_rmsnorm_gemv(codes, scales, 32, x, r, g, EPS)
    assert bits_equal(y.cpu().numpy(), ref)
    assert within_tol(yf.cpu().numpy(), ref)


def test_fused_zero_input():
    q = qmv_guarded()
    m = Mat("fu_zero", 128, 1024, 2, 32)
    z = np.zeros((1, 1024), np.float16)
    _, _, g = acts("fu_zero", 1, 1024)
    for mode in (q.QMV_FAST, q.QMV_EXACT):
        y = q.qmv_fused_rmsnorm_gemv(m.pack, to_dev(z), to_dev(z), to_dev(g), EPS, mode=mode)
        torch.cuda.synchronize()
        assert torch.all(y == 0)
