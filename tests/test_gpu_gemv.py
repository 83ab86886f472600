"""GPU parity of the matvec through the C ABI against the CPU oracle.

Exact mode keeps the oracle's accumulation order in every CUDA-core kernel
(M <= 32), so its fp32 outputs must be bit-identical to the oracle's, its
fp16 outputs the RNE of them, and every column of an M-tile bit-identical to
the M = 1 result for that column.  Fast mode (the folded-offset form where
K % 256 == 0) must stay within max |y - ref| <= 1e-3 * (1 + |ref|), and its
M-tile columns must equal its own M = 1 results bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import Mat, acts, bits_equal, first_diff, max_rel_err, to_dev, within_tol, qmv, qmv_guarded

pytestmark = pytest.mark.gpu

SHAPES = [
    # (N, K, bits, group)
    (1024, 1024, 2, 32),      # single int2 GEMV (1024 x 1024)
    (2560, 2048, 4, 32),      # fused q/k/v, int4
    (2048, 2048, 4, 32),      # o_proj, int4
    (16384, 2048, 2, 32),     # fused gate/up, int2
    (2048, 8192, 2, 32),      # down, int2
    (2048, 2048, 8, 2048),    # per-row int8 projection
    (1, 64, 2, 32), (3, 128, 2, 128), (33, 96, 4, 32), (65, 160, 8, 32), (100, 5376, 4, 32),
    (37, 5376, 8, 5376), (19, 21504, 4, 32), (29, 14336, 2, 32), (5, 16384, 2, 32),
    # few rows over a long K: 4096-code segments, a ragged last row group
    (2047, 20480, 2, 32), (700, 16384, 4, 32),
]


@pytest.mark.parametrize("N,K,bits,group", SHAPES)
def test_gemv_m1_bit_exact(N, K, bits, group):
    q = qmv_guarded()
    m = Mat(f"g{N}x{K}b{bits}g{group}", N, K, bits, group)
    x, _, _ = acts(f"g{N}x{K}", 1, K)
    y = q.qmv_gemv(m.pack, to_dev(x), mode=q.QMV_EXACT)
    y16 = q.qmv_gemv(m.pack, to_dev(x), y_dtype=q.QMV_F16, mode=q.QMV_EXACT)
    torch.cuda.synchronize()
    codes, scales = m.host()
    ref = oracle.gemv(codes, scales, group, x)
    got = y.cpu().numpy()
    assert bits_equal(got, ref), first_diff(got, ref)
    assert np.array_equal(y16.cpu().numpy().view(np.uint16), oracle.f32_to_f16(ref))


@pytest.mark.parametrize("N,K,bits,group", SHAPES)
def test_gemv_m1_fast_within_tolerance(N, K, bits, group):
    q = qmv_guarded()
    m = Mat(f"g{N}x{K}b{bits}g{group}", N, K, bits, group)
    x, _, _ = acts(f"g{N}x{K}", 1, K)
    y = q.qmv_gemv(m.pack, to_dev(x), mode=q.QMV_FAST)
    y16 = q.qmv_gemv(m.pack, to_dev(x), y_dtype=q.QMV_F16, mode=q.QMV_FAST)
    torch.cuda.synchronize()
    codes, scales = m.host()
    ref = oracle.gemv(codes, scales, group, x)
    got = y.cpu().numpy()
    assert within_tol(got, ref), max_rel_err(got, ref)
    # the fp16 output is the RNE of the same fp32 result
    assert np.array_equal(y16.cpu().numpy().view(np.uint16), oracle.f32_to_f16(got))


@pytest.mark.parametrize("N,K,bits,group", [(1024, 1024, 2, 32), (2560, 2048, 4, 32),
                                            (2048, 2048, 8, 2048), (300, 5376, 4, 32),
                                            (65, 256, 8, 32), (33, 2048, 2, 2048)])
@pytest.mark.parametrize("M", [2, 5, 8, 16, 17, 32])
def test_fast_tile_columns_equal_fast_m1(N, K, bits, group, M):
    q = qmv_guarded()
    m = Mat(f"f{N}x{K}b{bits}g{group}", N, K, bits, group)
    x, _, _ = acts(f"f{N}x{K}m{M}", M, K)
    y = q.qmv_chunk_gemm(m.pack, to_dev(x), mode=q.QMV_FAST)
    y1 = [q.qmv_gemv(m.pack, to_dev(x[i:i + 1]), mode=q.QMV_FAST) for i in range(M)]
    torch.cuda.synchronize()
    codes, scales = m.host()
    ref = oracle.gemv(codes, scales, group, x)
    got = y.cpu().numpy()
    assert within_tol(got, ref), max_rel_err(got, ref)
    for i in range(M):
        assert bits_equal(got[i], y1[i].cpu().numpy()[0]), (i, first_diff(got[i], y1[i].cpu().numpy()[0]))


@pytest.mark.parametrize("N,K,bits,group", [(1024, 1024, 2, 32), (2560, 2048, 4, 32),
                                            (2048, 2048, 8, 2048), (100, 5376, 4, 32),
                                            (37, 5376, 8, 5376), (33, 128, 2, 32)])
@pytest.mark.parametrize("M", [2, 3, 4, 5, 8, 16, 17, 32, 33, 40])
def test_chunk_columns_bit_exact(N, K, bits, group, M):
    q = qmv_guarded()
    m = Mat(f"c{N}x{K}b{bits}g{group}", N, K, bits, group)
    x, _, _ = acts(f"c{N}x{K}m{M}", M, K)
    y = q.qmv_chunk_gemm(m.pack, to_dev(x), mode=q.QMV_EXACT)
    yg = q.qmv_gemv(m.pack, to_dev(x), mode=q.QMV_EXACT)
    y1 = [q.qmv_gemv(m.pack, to_dev(x[i:i + 1]), mode=q.QMV_EXACT) for i in (0, M - 1)]
    torch.cuda.synchronize()
    codes, scales = m.host()
    ref = oracle.gemv(codes, scales, group, x)
    got = y.cpu().numpy()
    assert bits_equal(got, ref), first_diff(got, ref)
    assert bits_equal(yg.cpu().numpy(), ref)
    assert bits_equal(got[0], y1[0].cpu().numpy()[0])
    assert bits_equal(got[M - 1], y1[1].cpu().numpy()[0])


def test_output_fp16_rne_small_tile():
    q = qmv_guarded()
    m = Mat("f16tile", 300, 2048, 2, 32)
    x, _, _ = acts("f16tile", 8, 2048)
    y = q.qmv_chunk_gemm(m.pack, to_dev(x), y_dtype=q.QMV_F16, mode=q.QMV_EXACT)
    torch.cuda.synchronize()
    codes, scales = m.host()
    ref = oracle.gemv(codes, scales, 32, x)
    assert np.array_equal(y.cpu().numpy().view(np.uint16), oracle.f32_to_f16(ref))


def test_zero_codes_give_zero():
    q = qmv_guarded()
    N, K = 64, 256
    p = q.Pack(N, K, 2, 32).pack_weights(torch.zeros(N, K, dtype=torch.int8, device="cuda"),
                                         torch.full((N, K // 32), 0.01, dtype=torch.float16,
                                                    device="cuda"))
    x, _, _ = acts("zero", 4, K)
    for M in (1, 4):
        for mode in (q.QMV_FAST, q.QMV_EXACT):
            y = q.qmv_gemv(p, to_dev(x[:M]), mode=mode)
            torch.cuda.synchronize()
            assert torch.all(y == 0)


def test_repeated_calls_identical():
    q = qmv_guarded()
    m = Mat("repeat", 4096, 2048, 2, 32)
    x, _, _ = acts("repeat", 1, 2048)
    xd = to_dev(x)
    ys = [q.qmv_gemv(m.pack, xd) for _ in range(3)]
    torch.cuda.synchronize()
    for y in ys[1:]:
        assert torch.equal(y.view(torch.int32), ys[0].view(torch.int32))


def test_shape_mismatch_rejected():
    q = qmv_guarded()
    m = Mat("mismatch", 64, 128, 2, 32)
    x = torch.zeros(1, 128, dtype=torch.float16, device="cuda")
    y = torch.zeros(1, 64, dtype=torch.float32, device="cuda")
    lib = q.lib()
    s = torch.cuda.current_stream().cuda_stream
    assert lib.qmv_gemv(m.pack.handle, 1, 65, 128, 2, 32, x.data_ptr(), y.data_ptr(), 0, 0, None, 0, s) == -4
    assert lib.qmv_gemv(m.pack.handle, 1, 64, 128, 4, 32, x.data_ptr(), y.data_ptr(), 0, 0, None, 0, s) == -4
    assert lib.qmv_gemv(m.pack.handle, 0, 64, 128, 2, 32, x.data_ptr(), y.data_ptr(), 0, 0, None, 0, s) == -1
    assert lib.qmv_gemv(m.pack.handle, 1, 64, 128, 2, 32, x.data_ptr() + 2, y.data_ptr(), 0, 0, None, 0, s) == -3
    assert lib.qmv_gemv(m.pack.handle, 1, 64, 128, 2, 32, x.data_ptr(), y.data_ptr(), 7, 0, None, 0, s) == -1


def test_device_error_word_clear_after_runs():
    q = qmv_guarded()
    m = Mat("errword", 8192, 2048, 2, 32)
    x, _, _ = acts("errword", 1, 2048)
    for _ in range(3):
        q.qmv_gemv(m.pack, to_dev(x))
    torch.cuda.synchronize()
    assert q.qmv_device_error(clear=True) == 0


def _chain(q, packs, x, reps):
    """x -> A -> B -> A -> ... with fp16 outputs feeding the next matvec."""
    outs = []
    cur = x
    for i in range(reps):
        p = packs[i % len(packs)]
        cur = q.qmv_gemv(p, cur, y_dtype=q.QMV_F16)
        outs.append(cur)
    return outs


def test_pdl_chain_matches_plain_launches():
    q = qmv()
    A = Mat("pdlA", 2048, 2048, 2, 32)
    B = Mat("pdlB", 2048, 2048, 4, 32)
    x, _, _ = acts("pdl", 1, 2048)
    xd = to_dev(x)
    ref = [t.clone() for t in _chain(q, [A.pack, B.pack], xd, 8)]
    torch.cuda.synchronize()
    q.qmv_set_pdl(True)
    try:
        got = _chain(q, [A.pack, B.pack], xd, 8)
        torch.cuda.synchronize()
        for r, g in zip(ref, got):
            assert torch.equal(r.view(torch.int16), g.view(torch.int16))
        # the same chain captured in a CUDA graph (programmatic edges)
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            _chain(q, [A.pack, B.pack], xd, 2)           # warm-up on the capture stream
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            gout = _chain(q, [A.pack, B.pack], xd, 8)
        g.replay()
        torch.cuda.synchronize()
        for r, t in zip(ref, gout):
            assert torch.equal(r.view(torch.int16), t.view(torch.int16))
    finally:
        q.qmv_set_pdl(False)
    assert q.qmv_device_error(clear=True) == 0
