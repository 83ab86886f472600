"""GPU parity of the 8-column M-tiles.  The tile-shape chooser takes them
for wide matrices at M >= 5 (each code's mask then serves twice the paired
FMAs).  The shapes below are ones it sends there, checked through the
workspace size, which counts 17408-byte table records per 8 columns only
for them.  Exact mode must equal the oracle bit for bit.  In both modes every
column must equal the M = 1 result for that column bit for bit, including
the padded columns of a last partial chunk."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import (EPS, Mat, acts, bits_equal, first_diff, max_rel_err, to_dev, within_tol, qmv,
                      qmv_guarded)

pytestmark = pytest.mark.gpu

# (N, K, bits, group, M): int2 128-row tiles, int4 and int8 64-row tiles,
# a ragged row tile, a padded last chunk (M = 13) and a half last segment
CASES = [
    (28672, 512, 2, 32, 16),
    (28672, 768, 2, 32, 13),
    (19456, 512, 4, 32, 16),
    (19400, 512, 4, 32, 24),
    (9728, 512, 8, 512, 16),
]


def _is_eight(q, p, M, fused=False):
    n = q.qmv_workspace_bytes(p, M, q.QMV_F32, q.QMV_FAST, fused)
    return n == -(-M // 8) * -(-p.K // 512) * 17408


@pytest.mark.parametrize("N,K,bits,group,M", CASES)
@pytest.mark.parametrize("mode", ["exact", "fast"])
def test_eight_column_tiles(N, K, bits, group, M, mode):
    q = qmv_guarded()
    md = q.QMV_EXACT if mode == "exact" else q.QMV_FAST
    m = Mat(f"mt8.{N}x{K}b{bits}", N, K, bits, group)
    assert _is_eight(q, m.pack, M), "the chooser no longer takes 8-column tiles here"
    x, _, _ = acts(f"mt8.{N}x{K}m{M}", M, K)
    xd = to_dev(x)
    y = q.qmv_chunk_gemm(m.pack, xd, mode=md)
    y16 = q.qmv_chunk_gemm(m.pack, xd, y_dtype=q.QMV_F16, mode=md)
    y1 = [q.qmv_gemv(m.pack, xd[i:i + 1], mode=md) for i in range(M)]
    torch.cuda.synchronize()
    got = y.cpu().numpy()
    for i in range(M):
        assert bits_equal(got[i], y1[i].cpu().numpy()[0]), (i, first_diff(got[i], y1[i].cpu().numpy()[0]))
    assert np.array_equal(y16.cpu().numpy().view(np.uint16), oracle.f32_to_f16(got))
    codes, scales = m.host()
    ref = oracle.gemv(codes, scales, group, x)
    if mode == "exact":
        assert bits_equal(got, ref), first_diff(got, ref)
    else:
        assert within_tol(got, ref), max_rel_err(got, ref)
    assert q.qmv_device_error(clear=True) == 0


@pytest.mark.parametrize("mode", ["exact", "fast"])
def test_eight_column_tiles_fused(mode):
    q = qmv_guarded()
    md = q.QMV_EXACT if mode == "exact" else q.QMV_FAST
    N, K, M = 28672, 512, 16
    m = Mat("mt8.fused", N, K, 2, 32)
    assert _is_eight(q, m.pack, M, fused=True)
    x, r, g = acts("mt8.fused", M, K)
    h = torch.empty(M, K, dtype=torch.float16, device="cuda")
    y = q.qmv_fused_rmsnorm_gemv(m.pack, to_dev(x), to_dev(r), to_dev(g), EPS, h_out=h, mode=md)
    torch.cuda.synchronize()
    codes, scales = m.host()
    h_ref, y16, ref = oracle.fused_rmsnorm_gemv(codes, scales, 32, x, r, g, EPS)
    assert np.array_equal(h.cpu().numpy().view(np.uint16), h_ref)
    got = y.cpu().numpy()
    if mode == "exact":
        assert bits_equal(got, ref), first_diff(got, ref)
    else:
        assert within_tol(got, ref), max_rel_err(got, ref)
        y1 = [q.qmv_gemv(m.pack, to_dev(y16[i:i + 1].view(np.float16)), mode=md) for i in range(M)]
        torch.cuda.synchronize()
        for i in range(M):
            assert bits_equal(got[i], y1[i].cpu().numpy()[0]), i
    assert q.qmv_device_error(clear=True) == 0
