"""Calls that need scratch take it from the caller's workspace: the M-column
tiles' segment tables (fused or not) and the tensor tiles' split-K partial
tiles.  On an explicit workspace whose
contents are garbage, results equal the oracle (exact mode bit for bit;
tensor tiles within tolerance) and the binding's own path; a missing or short
workspace is refused before any launch, and the workspace's guard bands stay
intact."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import (EPS, GuardBuf, Mat, acts, bits_equal, first_diff, max_rel_err, sample_rows, to_dev,
                      within_tol, qmv)

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.float16 else t.view(torch.int32)


def _tables(M, K):
    """The possible bytes of the M-column tiles' table records: per 512 codes,
    8960 per 4 columns, or 17408 per 8 (8-column tiles, M >= 5)."""
    segs = -(-K // 512)
    four = -(-M // 4) * segs * 8960
    return {four} if M < 5 else {four, -(-M // 8) * segs * 17408}


def _ws(q, p, M, y_dtype, mode, fused):
    n = q.qmv_workspace_bytes(p, M, y_dtype, mode, fused)
    assert n > 0 and n % 256 == 0
    g = GuardBuf(n, fill=0x5A)
    return g, g.view(torch.uint8, (n,))


@pytest.mark.parametrize("mode", ["exact", "fast"])
def test_fused_m16_on_caller_workspace(mode):
    q = qmv()
    md = q.QMV_EXACT if mode == "exact" else q.QMV_FAST
    N, K, M = 1024, 2048, 16
    m = Mat("ws.fused", N, K, 2, 32)
    x, r, g = acts("ws.fused", M, K)
    xd, rd, gd = to_dev(x), to_dev(r), to_dev(g)
    gw, ws = _ws(q, m.pack, M, q.QMV_F32, md, True)
    assert gw.nbytes in _tables(M, K)
    h = torch.empty(M, K, dtype=torch.float16, device="cuda")
    y = q.qmv_fused_rmsnorm_gemv(m.pack, xd, rd, gd, EPS, h_out=h, mode=md, workspace=ws)
    y_auto = q.qmv_fused_rmsnorm_gemv(m.pack, xd, rd, gd, EPS, mode=md)
    torch.cuda.synchronize()
    gw.check("workspace")
    assert torch.equal(_bits(y), _bits(y_auto))
    codes, scales = m.host()
    for i in (0, 7, M - 1):
        h_ref, _, y_ref = oracle.fused_rmsnorm_gemv(codes, scales, 32, x[i:i + 1], r[i:i + 1], g, EPS)
        assert np.array_equal(h[i].cpu().numpy().view(np.uint16), h_ref.reshape(-1)), i
        yi = y[i].cpu().numpy()
        if mode == "exact":
            assert bits_equal(yi, y_ref.reshape(-1)), (i, first_diff(yi, y_ref.reshape(-1)))
        else:
            assert within_tol(yi, y_ref.reshape(-1)), (i, max_rel_err(yi, y_ref.reshape(-1)))
    assert q.qmv_device_error(clear=True) == 0


@pytest.mark.parametrize("y_dtype", ["f32", "f16"])
def test_split_k_m128_on_caller_workspace(y_dtype):
    q = qmv()
    dt = q.QMV_F32 if y_dtype == "f32" else q.QMV_F16
    N, K, M = 512, 4096, 128
    m = Mat("ws.tc", N, K, 2, 32)
    x, _, _ = acts("ws.tc", M, K)
    xd = to_dev(x)
    gw, ws = _ws(q, m.pack, M, dt, q.QMV_FAST, False)
    y = q.qmv_chunk_gemm(m.pack, xd, y_dtype=dt, mode=q.QMV_FAST, workspace=ws)
    # the same workspace, garbage again, serves a second call
    ws.fill_(0xC3)
    y2 = q.qmv_chunk_gemm(m.pack, xd, y_dtype=dt, mode=q.QMV_FAST, workspace=ws)
    y_auto = q.qmv_chunk_gemm(m.pack, xd, y_dtype=dt, mode=q.QMV_FAST)
    torch.cuda.synchronize()
    gw.check("workspace")
    assert torch.equal(_bits(y), _bits(y_auto)) and torch.equal(_bits(y2), _bits(y_auto))
    rows = sample_rows(N, n=48)
    codes, scales = m.host(rows)
    for i in (0, 61, M - 1):
        ref = oracle.gemv(codes, scales, 32, x[i:i + 1]).reshape(-1)
        got = y[i, rows].float().cpu().numpy()
        tol = 1e-3 if y_dtype == "f32" else 2e-3
        assert within_tol(got, ref, tol), (i, max_rel_err(got, ref))
    assert q.qmv_device_error(clear=True) == 0


def test_missing_or_short_workspace_is_refused():
    q = qmv()
    N, K, M = 512, 4096, 128
    m = Mat("ws.short", N, K, 2, 32)
    xd = torch.zeros(M, K, dtype=torch.float16, device="cuda")
    y = torch.zeros(M, N, dtype=torch.float16, device="cuda")
    n = q.qmv_workspace_bytes(m.pack, M, q.QMV_F16, q.QMV_FAST, False)
    lib, s = q.lib(), torch.cuda.current_stream().cuda_stream
    assert lib.qmv_chunk_gemm(m.pack.handle, M, xd.data_ptr(), y.data_ptr(), 1, 0, None, 0, s) == q.QMV_ERR_WORKSPACE
    short = torch.empty(n - 256, dtype=torch.uint8, device="cuda")
    assert lib.qmv_chunk_gemm(m.pack.handle, M, xd.data_ptr(), y.data_ptr(), 1, 0, short.data_ptr(), n - 256,
                              s) == q.QMV_ERR_WORKSPACE
    full = torch.empty(n + 256, dtype=torch.uint8, device="cuda")
    assert lib.qmv_chunk_gemm(m.pack.handle, M, xd.data_ptr(), y.data_ptr(), 1, 0, full.data_ptr() + 16, n,
                              s) == q.QMV_ERR_ALIGNMENT
    # a call that needs none accepts none
    assert q.qmv_workspace_bytes(m.pack, 1, q.QMV_F16, q.QMV_FAST, False) == 0
    assert lib.qmv_gemv(m.pack.handle, 1, N, K, 2, 32, xd.data_ptr(), y.data_ptr(), 1, 0, None, 0, s) == 0
    torch.cuda.synchronize()


@pytest.mark.parametrize("mode", ["exact", "fast"])
@pytest.mark.parametrize("M", [2, 7, 16])
def test_mtile_tables_on_caller_workspace(mode, M):
    # the tables are built into a garbage-filled workspace, which then serves a
    # second call; every column equals the M = 1 result bit for bit
    q = qmv()
    md = q.QMV_EXACT if mode == "exact" else q.QMV_FAST
    N, K = 700, 4352          # a ragged row tile and a half last segment
    m = Mat("ws.mt", N, K, 4, 32)
    x, _, _ = acts("ws.mt", M, K)
    xd = to_dev(x)
    gw, ws = _ws(q, m.pack, M, q.QMV_F32, md, False)
    assert gw.nbytes in _tables(M, K)
    y = q.qmv_chunk_gemm(m.pack, xd, mode=md, workspace=ws)
    ws.fill_(0xC3)
    y2 = q.qmv_chunk_gemm(m.pack, xd, mode=md, workspace=ws)
    y1 = [q.qmv_gemv(m.pack, xd[i:i + 1], mode=md) for i in range(M)]
    torch.cuda.synchronize()
    gw.check("workspace")
    assert torch.equal(_bits(y), _bits(y2))
    for i in range(M):
        assert torch.equal(_bits(y[i]), _bits(y1[i][0])), i
    if mode == "exact":
        codes, scales = m.host()
        ref = oracle.gemv(codes, scales, 32, x)
        got = y.cpu().numpy()
        assert bits_equal(got, ref), first_diff(got, ref)
    assert q.qmv_device_error(clear=True) == 0


def test_calls_in_turn_share_one_workspace_under_pdl():
    # gate/up-like then down-like then gate/up-like again on one workspace,
    # with programmatic dependent launch: a call's table kernel must not
    # overwrite the records while the previous call's tiles still read them
    q = qmv()
    A = Mat("ws.pdlA", 2048, 4096, 2, 32)
    B = Mat("ws.pdlB", 1024, 8192, 4, 32)
    M = 16
    xa, _, _ = acts("ws.pdlA", M, 4096)
    xb, _, _ = acts("ws.pdlB", M, 8192)
    xad, xbd = to_dev(xa), to_dev(xb)
    ref = [q.qmv_chunk_gemm(A.pack, xad), q.qmv_chunk_gemm(B.pack, xbd)]
    n = max(q.qmv_workspace_bytes(A.pack, M), q.qmv_workspace_bytes(B.pack, M))
    gw = GuardBuf(n, fill=0x5A)
    ws = gw.view(torch.uint8, (n,))
    torch.cuda.synchronize()
    q.qmv_set_pdl(True)
    try:
        outs = []
        for _ in range(3):
            outs.append(q.qmv_chunk_gemm(A.pack, xad, workspace=ws))
            outs.append(q.qmv_chunk_gemm(B.pack, xbd, workspace=ws))
        torch.cuda.synchronize()
    finally:
        q.qmv_set_pdl(False)
    gw.check("workspace")
    for i, o in enumerate(outs):
        assert torch.equal(_bits(o), _bits(ref[i % 2])), i
    assert q.qmv_device_error(clear=True) == 0


def test_mtile_missing_workspace_is_refused():
    q = qmv()
    N, K, M = 256, 1024, 8
    m = Mat("ws.mtshort", N, K, 2, 32)
    xd = torch.zeros(M, K, dtype=torch.float16, device="cuda")
    y = torch.zeros(M, N, dtype=torch.float32, device="cuda")
    n = q.qmv_workspace_bytes(m.pack, M, q.QMV_F32, q.QMV_EXACT, False)
    assert n in _tables(M, K)
    lib, s = q.lib(), torch.cuda.current_stream().cuda_stream
    for mode in (0, 1):
        assert lib.qmv_chunk_gemm(m.pack.handle, M, xd.data_ptr(), y.data_ptr(), 0, mode, None, 0,
                                  s) == q.QMV_ERR_WORKSPACE
        assert lib.qmv_gemv(m.pack.handle, M, N, K, 2, 32, xd.data_ptr(), y.data_ptr(), 0, mode, None, 0,
                            s) == q.QMV_ERR_WORKSPACE
    short = torch.empty(n, dtype=torch.uint8, device="cuda")
    assert lib.qmv_chunk_gemm(m.pack.handle, M, xd.data_ptr(), y.data_ptr(), 0, 1, short.data_ptr(), n - 16,
                              s) == q.QMV_ERR_WORKSPACE
    torch.cuda.synchronize()
