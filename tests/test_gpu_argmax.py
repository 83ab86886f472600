"""GPU parity of the fused argmax epilogue (qmv_gemv_argmax): the greedy token
after the lm_head matvec, first-max tie-break ("Gemma4 raw-Metal loop on
A19", "The parked levers" table, argmax row).  Exact mode: the index and the
value equal the oracle's argmax of the oracle's output.  Fast mode: the index
is the first maximum of the kernel's own stored logits, and the oracle's
value at that index is within the tolerance of the oracle's maximum."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import EPS, TOL, Mat, acts, bits_equal, to_dev, qmv, qmv_guarded

pytestmark = pytest.mark.gpu


def _ws():
    return qmv().qmv_argmax_workspace()


@pytest.mark.parametrize("N,K,bits,group", [(32768, 2048, 2, 32), (20000, 5376, 4, 32),
                                            (4099, 2048, 8, 2048), (300, 256, 2, 32)])
@pytest.mark.parametrize("fused", [False, True])
def test_argmax_exact_equals_oracle(N, K, bits, group, fused):
    q = qmv_guarded()
    m = Mat(f"am{N}x{K}b{bits}", N, K, bits, group)
    x, r, g = acts(f"am{N}x{K}", 1, K, outliers=(K == 5376))
    ws = _ws()
    y = torch.zeros(1, N, dtype=torch.float32, device="cuda")
    if fused:
        idx, val = q.qmv_gemv_argmax(m.pack, to_dev(x), ws, residual=to_dev(r), gamma=to_dev(g),
                                     eps=EPS, y=y, mode=q.QMV_EXACT)
    else:
        idx, val = q.qmv_gemv_argmax(m.pack, to_dev(x), ws, y=y, mode=q.QMV_EXACT)
    torch.cuda.synchronize()
    codes, scales = m.host(np.arange(N))
    if fused:
        _, _, ref = oracle.fused_rmsnorm_gemv(codes, scales, group, x, r, g, EPS)
    else:
        ref = oracle.gemv(codes, scales, group, x)
    ri, rv = oracle.argmax(ref[0])
    assert int(idx.item()) == ri
    assert float(val.item()) == rv
    assert bits_equal(y.cpu().numpy(), ref)
    assert torch.count_nonzero(ws).item() == 0          # left zero for the next call


@pytest.mark.parametrize("N,K,bits,group", [(32768, 2048, 2, 32), (20000, 5376, 4, 32)])
def test_argmax_fast_is_a_true_maximum(N, K, bits, group):
    q = qmv_guarded()
    m = Mat(f"amf{N}x{K}b{bits}", N, K, bits, group)
    x, _, _ = acts(f"amf{N}x{K}", 1, K)
    y = torch.zeros(1, N, dtype=torch.float32, device="cuda")
    idx, val = q.qmv_gemv_argmax(m.pack, to_dev(x), _ws(), y=y, mode=q.QMV_FAST)
    torch.cuda.synchronize()
    i = int(idx.item())
    yg = y.cpu().numpy()[0]
    # consistent with the kernel's own logits: their first maximum
    assert i == int(np.argmax(yg)) and float(val.item()) == float(yg.max())
    codes, scales = m.host(np.arange(N))
    ref = oracle.gemv(codes, scales, group, x)[0]
    rmax = float(ref.max())
    assert float(ref[i]) >= rmax - TOL * (1.0 + abs(rmax))


@pytest.mark.parametrize("mode", ["fast", "exact"])
def test_argmax_ties_take_the_first(mode):
    """three identical maximal rows planted among random ones: the lowest wins"""
    q = qmv_guarded()
    N, K = 40000, 2048
    codes = synth.codes(7, "amtie", N, K, 2)
    scales = synth.scales(7, "amtie", N, K // 32)
    for row in (31000, 777, 5000):
        codes[row] = 1
        scales[row] = torch.tensor(0.02, dtype=torch.float16)
    p = q.Pack(N, K, 2, 32).pack_weights(codes.cuda(), scales.cuda())
    x = np.abs(synth.normal_f16(7, "amtie.x", (1, K)))
    md = q.QMV_FAST if mode == "fast" else q.QMV_EXACT
    ws = _ws()
    for _ in range(2):                                  # the workspace resets itself
        idx, val = q.qmv_gemv_argmax(p, to_dev(x), ws, mode=md)   # logits not stored
        torch.cuda.synchronize()
        assert int(idx.item()) == 777
    ref = oracle.gemv(codes[[777]].numpy(), scales[[777]].numpy(), 32, x)[0, 0]
    if mode == "exact":
        assert float(val.item()) == float(ref)
    else:
        assert abs(float(val.item()) - float(ref)) <= TOL * (1 + abs(float(ref)))


def test_argmax_full_size_lm_head_int2():
    """262144 x 2048 int2 (the decode token's lm_head), exact mode: the index is
    the first maximum of the stored logits and the oracle computes that row's
    value bit for bit"""
    q = qmv_guarded()
    head = Mat("full.head2", 262144, 2048, 2, 32)
    x, _, _ = acts("full.head2.am", 1, 2048)
    y = torch.zeros(1, 262144, dtype=torch.float32, device="cuda")
    idx, val = q.qmv_gemv_argmax(head.pack, to_dev(x), _ws(), y=y, mode=q.QMV_EXACT)
    torch.cuda.synchronize()
    i = int(idx.item())
    yg = y.cpu().numpy()[0]
    assert i == int(np.argmax(yg)) and float(val.item()) == float(yg[i])
    codes, scales = head.host(np.array([i]))
    ref = oracle.gemv(codes, scales, 32, x)[0, 0]
    assert float(val.item()) == float(ref)
    assert q.qmv_device_error(clear=True) == 0


def test_argmax_argument_errors():
    q = qmv()
    m = Mat("amerr", 64, 128, 2, 32)                    # K % 256 != 0: not on the pipeline
    x = torch.zeros(1, 128, dtype=torch.float16, device="cuda")
    with pytest.raises(q.QmvError) as e:
        q.qmv_gemv_argmax(m.pack, x, _ws())
    assert e.value.status == q.QMV_ERR_UNSUPPORTED
    m2 = Mat("amerr2", 64, 256, 2, 32)
    x2 = torch.zeros(1, 256, dtype=torch.float16, device="cuda")
    bad = torch.zeros(24, dtype=torch.uint8, device="cuda")[4:]   # misaligned workspace
    with pytest.raises(q.QmvError) as e:
        q.qmv_gemv_argmax(m2.pack, x2, bad)
    assert e.value.status == q.QMV_ERR_ALIGNMENT
