"""GPU parity of the pipelined M-column tiles (any M >= 2 token columns, K a
multiple of 256): the "raw-metal-loop-playbook" prefill-regimes rule that each
output scalar keeps the single-token K order.  Exact mode: every element
bit-identical to the oracle.  Fast mode: every column bit-identical to the
fast M = 1 result for that column, and within 1e-3 * (1 + |ref|) of the
oracle.  Shapes cover ragged row tiles (N not a multiple of 64 or 128), a
last segment shorter than 512 codes (K = 768, 2304, 5376), column chunks
with padding (M not a multiple of 4 or 8), per-row and group-32 scales, fp16
outputs, and the full-size gate/up and down projections (sampled rows)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import (EPS, Mat, acts, bits_equal, first_diff, max_rel_err, sample_rows, to_dev,
                      within_tol, qmv, qmv_guarded)

pytestmark = pytest.mark.gpu

SHAPES = [
    # (N, K, bits, group)
    (1000, 768, 2, 32),
    (333, 2304, 4, 32),
    (200, 5376, 8, 32),
    (130, 1024, 2, 1024),     # one scale per row
    (77, 2304, 8, 2304),
    (4100, 2048, 4, 32),
]
MS = [2, 3, 4, 7, 9, 16, 24, 33, 70]


@pytest.mark.parametrize("N,K,bits,group", SHAPES)
@pytest.mark.parametrize("M", MS)
def test_mtile_exact_equals_oracle(N, K, bits, group, M):
    q = qmv_guarded()
    m = Mat(f"mt{N}x{K}b{bits}g{group}", N, K, bits, group)
    x, _, _ = acts(f"mt{N}x{K}m{M}", M, K)
    y = q.qmv_chunk_gemm(m.pack, to_dev(x), mode=q.QMV_EXACT)
    torch.cuda.synchronize()
    codes, scales = m.host()
    ref = oracle.gemv(codes, scales, group, x)
    got = y.cpu().numpy()
    assert bits_equal(got, ref), first_diff(got, ref)
    assert q.qmv_device_error(clear=True) == 0


@pytest.mark.parametrize("N,K,bits,group", SHAPES)
@pytest.mark.parametrize("M", [2, 5, 8, 13, 32, 40])
def test_mtile_fast_columns_equal_m1(N, K, bits, group, M):
    q = qmv_guarded()
    if bits == 2 and M > 32:
        pytest.skip("int2 at M > 32 in fast mode runs the tensor tiles (hardware order)")
    m = Mat(f"mf{N}x{K}b{bits}g{group}", N, K, bits, group)
    x, _, _ = acts(f"mf{N}x{K}m{M}", M, K)
    xd = to_dev(x)
    y = q.qmv_chunk_gemm(m.pack, xd, mode=q.QMV_FAST)
    y1 = [q.qmv_gemv(m.pack, xd[i:i + 1].contiguous(), mode=q.QMV_FAST) for i in range(M)]
    torch.cuda.synchronize()
    got = y.cpu().numpy()
    for i in range(M):
        g1 = y1[i].cpu().numpy()[0]
        assert bits_equal(got[i], g1), (i, first_diff(got[i], g1))
    codes, scales = m.host()
    ref = oracle.gemv(codes, scales, group, x)
    assert within_tol(got, ref), max_rel_err(got, ref)


@pytest.mark.parametrize("mode", ["exact", "fast"])
def test_mtile_fp16_output_is_rne_of_fp32(mode):
    q = qmv_guarded()
    md = q.QMV_EXACT if mode == "exact" else q.QMV_FAST
    m = Mat("mt16out", 700, 2304, 2, 32)
    x, _, _ = acts("mt16out", 11, 2304)
    y = q.qmv_chunk_gemm(m.pack, to_dev(x), mode=md)
    y16 = q.qmv_chunk_gemm(m.pack, to_dev(x), y_dtype=q.QMV_F16, mode=md)
    torch.cuda.synchronize()
    assert np.array_equal(y16.cpu().numpy().view(np.uint16), oracle.f32_to_f16(y.cpu().numpy()))


def test_mtile_repeated_calls_identical():
    q = qmv_guarded()
    m = Mat("mtrep", 2000, 2048, 2, 32)
    x, _, _ = acts("mtrep", 16, 2048)
    xd = to_dev(x)
    ys = [q.qmv_chunk_gemm(m.pack, xd, mode=q.QMV_FAST) for _ in range(3)]
    torch.cuda.synchronize()
    for y in ys[1:]:
        assert torch.equal(y.view(torch.int32), ys[0].view(torch.int32))


@pytest.mark.parametrize("name,N,K,M", [("gateup", 28672, 4096, 16), ("down", 4096, 14336, 8)])
def test_mtile_full_size_sampled(name, N, K, M):
    """the full projections at prefill chunk sizes: exact mode on sampled rows
    equals the oracle; fast mode equals the fast M = 1 results"""
    q = qmv_guarded()
    m = Mat(f"mtfull.{name}", N, K, 2, 32)
    x, _, _ = acts(f"mtfull.{name}", M, K)
    xd = to_dev(x)
    ye = q.qmv_chunk_gemm(m.pack, xd, mode=q.QMV_EXACT)
    yf = q.qmv_chunk_gemm(m.pack, xd, mode=q.QMV_FAST)
    y1 = [q.qmv_gemv(m.pack, xd[i:i + 1].contiguous(), mode=q.QMV_FAST) for i in (0, M - 1)]
    torch.cuda.synchronize()
    rows = sample_rows(N, n=96)
    codes, scales = m.host(rows)
    ref = oracle.gemv(codes, scales, 32, x)
    got = ye.cpu().numpy()[:, rows]
    assert bits_equal(got, ref), first_diff(got, ref)
    gf = yf.cpu().numpy()
    assert bits_equal(gf[0], y1[0].cpu().numpy()[0])
    assert bits_equal(gf[M - 1], y1[1].cpu().numpy()[0])
    assert within_tol(gf[:, rows], ref), max_rel_err(gf[:, rows], ref)
    assert q.qmv_device_error(clear=True) == 0


@pytest.mark.parametrize("N,K,bits,group,M", [(1000, 2048, 2, 32, 16), (333, 2304, 4, 32, 5),
                                              (130, 1024, 2, 1024, 8), (200, 5376, 8, 32, 3),
                                              (4100, 4096, 2, 32, 32)])
def test_mtile_fused_prologue(N, K, bits, group, M):
    """fused residual-add + RMSNorm before the tiles: h bit-exact, the exact
    mode bit-exact against the oracle, and every fast-mode column equal to the
    fused fast M = 1 result for that column"""
    q = qmv_guarded()
    m = Mat(f"mfu{N}x{K}b{bits}g{group}", N, K, bits, group)
    x, r, g = acts(f"mfu{N}x{K}m{M}", M, K, outliers=(K == 5376))
    xd, rd, gd = to_dev(x), to_dev(r), to_dev(g)
    h = torch.empty(M, K, dtype=torch.float16, device="cuda")
    ye = q.qmv_fused_rmsnorm_gemv(m.pack, xd, rd, gd, EPS, h_out=h, mode=q.QMV_EXACT)
    yf = q.qmv_fused_rmsnorm_gemv(m.pack, xd, rd, gd, EPS, mode=q.QMV_FAST)
    y1 = [q.qmv_fused_rmsnorm_gemv(m.pack, xd[i:i + 1].contiguous(), rd[i:i + 1].contiguous(), gd, EPS,
                                   mode=q.QMV_FAST) for i in range(M)]
    torch.cuda.synchronize()
    codes, scales = m.host()
    h_ref, _, ref = oracle.fused_rmsnorm_gemv(codes, scales, group, x, r, g, EPS)
    assert np.array_equal(h.cpu().numpy().view(np.uint16), h_ref)
    got = ye.cpu().numpy()
    assert bits_equal(got, ref), first_diff(got, ref)
    gf = yf.cpu().numpy()
    for i in range(M):
        assert bits_equal(gf[i], y1[i].cpu().numpy()[0]), i
    assert within_tol(gf, ref), max_rel_err(gf, ref)
    assert q.qmv_device_error(clear=True) == 0


@pytest.mark.parametrize("N,K,bits,group", [(150, 1024, 2, 32), (90, 320, 4, 32)])
def test_fused_above_32_columns(N, K, bits, group):
    """the fused prologue at M = 40: the pipelined tiles (K % 256 == 0) and the
    plain tiles in 32-column launches (K % 256 != 0) -- h and y bit-exact
    against the oracle in exact mode, fast columns equal to fused fast M = 1"""
    q = qmv_guarded()
    M = 40
    m = Mat(f"fu40.{N}x{K}b{bits}", N, K, bits, group)
    x, r, g = acts(f"fu40.{N}x{K}", M, K)
    xd, rd, gd = to_dev(x), to_dev(r), to_dev(g)
    h = torch.empty(M, K, dtype=torch.float16, device="cuda")
    ye = q.qmv_fused_rmsnorm_gemv(m.pack, xd, rd, gd, EPS, h_out=h, mode=q.QMV_EXACT)
    yf = q.qmv_fused_rmsnorm_gemv(m.pack, xd, rd, gd, EPS, mode=q.QMV_FAST)
    y1 = [q.qmv_fused_rmsnorm_gemv(m.pack, xd[i:i + 1].contiguous(), rd[i:i + 1].contiguous(), gd, EPS,
                                   mode=q.QMV_FAST) for i in (0, M - 1)]
    torch.cuda.synchronize()
    codes, scales = m.host()
    h_ref, _, ref = oracle.fused_rmsnorm_gemv(codes, scales, group, x, r, g, EPS)
    assert np.array_equal(h.cpu().numpy().view(np.uint16), h_ref)
    assert bits_equal(ye.cpu().numpy(), ref), first_diff(ye.cpu().numpy(), ref)
    gf = yf.cpu().numpy()
    assert bits_equal(gf[0], y1[0].cpu().numpy()[0])
    assert bits_equal(gf[M - 1], y1[1].cpu().numpy()[0])
    assert within_tol(gf, ref), max_rel_err(gf, ref)


def test_mtile_max_columns():
    """M = 4096 (the largest chunk the ABI takes) on a small matrix: 1024 column
    chunks of one row tile each; exact mode bit-exact against the oracle"""
    q = qmv_guarded()
    N, K, M = 100, 256, 4096
    m = Mat("mtmax", N, K, 2, 32)
    x, _, _ = acts("mtmax", M, K)
    y = q.qmv_chunk_gemm(m.pack, to_dev(x), mode=q.QMV_EXACT)
    torch.cuda.synchronize()
    codes, scales = m.host()
    ref = oracle.gemv(codes, scales, 32, x)
    got = y.cpu().numpy()
    assert bits_equal(got, ref), first_diff(got, ref)
    assert q.qmv_device_error(clear=True) == 0
