"""GPU parity of the expert-gather matvec (qmv_gemv_gather): the selected
experts' rows of a stacked pack times x, with no gathered weight copy
("raw-metal-loop-playbook", ranked-targets table, MoE row).  Exact mode equals
the oracle on the gathered rows bit for bit; fast mode equals the dense fast
matvec's rows bit for bit (a row's arithmetic does not depend on how rows are
grouped) and the oracle within tolerance."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import Mat, acts, bits_equal, first_diff, max_rel_err, to_dev, within_tol, qmv, qmv_guarded

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("E,rows,K,bits,group", [(64, 1024, 2048, 2, 32), (16, 1000, 2048, 4, 32),
                                                 (8, 700, 5376, 8, 5376), (32, 96, 256, 2, 32)])
@pytest.mark.parametrize("mode", ["fast", "exact"])
def test_gather_equals_gathered_rows(E, rows, K, bits, group, mode):
    q = qmv_guarded()
    md = q.QMV_FAST if mode == "fast" else q.QMV_EXACT
    m = Mat(f"ga{E}x{rows}x{K}b{bits}", E * rows, K, bits, group)
    x, _, _ = acts(f"ga{E}x{rows}", 1, K)
    rng = np.random.default_rng(E + rows)
    ids = rng.integers(0, E, size=8).astype(np.int32)
    ids[3] = ids[1]                                     # a repeated expert
    y = q.qmv_gemv_gather(m.pack, rows, to_dev(ids), to_dev(x), mode=md)
    dense = q.qmv_gemv(m.pack, to_dev(x), mode=md)
    torch.cuda.synchronize()
    sel = np.concatenate([np.arange(e * rows, (e + 1) * rows) for e in ids])
    got = y.cpu().numpy()[0]
    assert bits_equal(got, dense.cpu().numpy()[0][sel])
    codes, scales = m.host(sel)
    ref = oracle.gemv(codes, scales, group, x)[0]
    if mode == "exact":
        assert bits_equal(got, ref), first_diff(got, ref)
    else:
        assert within_tol(got, ref), max_rel_err(got, ref)
    assert q.qmv_device_error(clear=True) == 0


def test_gather_ids_from_the_previous_kernel_with_pdl():
    """ids computed on the device right before the call (programmatic launch
    on): the kernel reads them only after that kernel completes"""
    q = qmv_guarded()
    E, rows, K = 128, 512, 2048
    m = Mat("gapdl", E * rows, K, 2, 32)
    x = to_dev(acts("gapdl", 1, K)[0])
    q.qmv_set_pdl(True)
    try:
        base = torch.arange(8, dtype=torch.int32, device="cuda")
        outs, idss = [], []
        for t in range(4):
            ids = (base * 13 + 7 * t) % E               # a small kernel writes the ids
            idss.append(ids)
            outs.append(q.qmv_gemv_gather(m.pack, rows, ids, x))
        dense = q.qmv_gemv(m.pack, x)
        torch.cuda.synchronize()
    finally:
        q.qmv_set_pdl(False)
    for ids, y in zip(idss, outs):
        sel = np.concatenate([np.arange(e * rows, (e + 1) * rows) for e in ids.cpu().numpy()])
        assert bits_equal(y.cpu().numpy()[0], dense.cpu().numpy()[0][sel])


def test_gather_invalid_id_gives_zeros_and_error_word():
    q = qmv_guarded()
    m = Mat("gabad", 4 * 256, 256, 2, 32)
    x = to_dev(acts("gabad", 1, 256)[0])
    q.qmv_device_error(clear=True)
    ids = torch.tensor([1, 9, 0], dtype=torch.int32, device="cuda")   # 9 >= E = 4
    y = q.qmv_gemv_gather(m.pack, 256, ids, x)
    dense = q.qmv_gemv(m.pack, x)
    torch.cuda.synchronize()
    assert q.qmv_device_error(clear=True) == 8
    got = y.cpu().numpy()[0]
    d = dense.cpu().numpy()[0]
    assert bits_equal(got[:256], d[256:512]) and bits_equal(got[512:], d[:256])
    assert np.all(got[256:512] == 0)


def test_gather_argument_errors():
    q = qmv()
    m = Mat("gaerr", 1000, 256, 2, 32)
    x = torch.zeros(1, 256, dtype=torch.float16, device="cuda")
    ids = torch.zeros(4, dtype=torch.int32, device="cuda")
    with pytest.raises(q.QmvError) as e:
        q.qmv_gemv_gather(m.pack, 300, ids, x)          # 300 does not divide 1000
    assert e.value.status == q.QMV_ERR_SHAPE
    with pytest.raises(q.QmvError) as e:
        q.qmv_gemv_gather(m.pack, 100, torch.zeros(257, dtype=torch.int32, device="cuda"), x)
    assert e.value.status == q.QMV_ERR_INVALID_ARG
