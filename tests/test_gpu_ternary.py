"""Ternary weights {-1, 0, 1} ("raw-metal-loop-playbook", ranked-targets
table, BitCPM-8B row) on the int2 decoder family: packed as int2 fields
u in {1, 2, 3} and run through every path -- M = 1 (exact bit-exact, fast
within tolerance), the fused prologue, the M-column tiles and the tensor-core
tiles -- at a BitCPM-8B-like d_model of 4096."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import EPS, Mat, acts, bits_equal, first_diff, max_rel_err, sample_rows, to_dev, \
    within_tol, qmv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tern():
    return {"up": Mat("tern.up", 14336, 4096, 2, 32, ternary=True),
            "down": Mat("tern.down", 4096, 14336, 2, 32, ternary=True)}


@pytest.mark.parametrize("M", [1, 8, 128])
def test_ternary_matvec_paths(tern, M):
    q = qmv()
    for name, m in tern.items():
        x, _, _ = acts(f"tern.{name}.m{M}", M, m.K)
        rows = sample_rows(m.N, 96)
        codes, scales = m.host(rows)
        assert set(np.unique(codes)) <= {-1, 0, 1}
        ref = oracle.gemv(codes, scales, 32, x)
        yf = q.qmv_chunk_gemm(m.pack, to_dev(x), mode=q.QMV_FAST) if M > 1 else \
            q.qmv_gemv(m.pack, to_dev(x), mode=q.QMV_FAST)
        ye = q.qmv_chunk_gemm(m.pack, to_dev(x), mode=q.QMV_EXACT) if M > 1 else \
            q.qmv_gemv(m.pack, to_dev(x), mode=q.QMV_EXACT)
        torch.cuda.synchronize()
        gf, ge = yf.cpu().numpy()[:, rows], ye.cpu().numpy()[:, rows]
        assert within_tol(gf, ref), max_rel_err(gf, ref)
        assert bits_equal(ge, ref), first_diff(ge, ref)


def test_ternary_fused_prologue_exact(tern):
    q = qmv()
    m = tern["up"]
    x, r, g = acts("tern.fused", 1, m.K)
    h = torch.empty(1, m.K, dtype=torch.float16, device="cuda")
    y = q.qmv_fused_rmsnorm_gemv(m.pack, to_dev(x), to_dev(r), to_dev(g), EPS, h_out=h, mode=q.QMV_EXACT)
    torch.cuda.synchronize()
    rows = sample_rows(m.N, 96)
    codes, scales = m.host(rows)
    h_ref, _, ref = oracle.fused_rmsnorm_gemv(codes, scales, 32, x, r, g, EPS)
    assert np.array_equal(h.cpu().numpy().view(np.uint16), h_ref)
    assert bits_equal(y.cpu().numpy()[:, rows], ref)
