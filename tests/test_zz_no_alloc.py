"""qmv_chain_create_no_alloc: a chain whose scratch (barrier words and op
table) is the library's own device array.  Two runs in a row of a chain made
this way must give, bit for bit, what the same chain on a caller-provided
workspace (qmv_chain_create) gives; and a second no-alloc chain run in between
must not disturb the first one's op table."""
import pytest
import torch

from gpu_util import EPS, Mat, acts, to_dev, qmv

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.float16 else t.view(torch.int32)


def test_no_alloc_chain_equals_workspace_chain_twice():
    q = qmv()
    A = Mat("na.A", 2560, 2048, 4, 32)
    B = Mat("na.B", 2048, 2048, 2, 32)
    x, r, g = (to_dev(v) for v in acts("na", 1, 2048))
    outs = {}

    def build(ch, tag):
        h = torch.zeros(1, 2048, dtype=torch.float16, device="cuda")
        y1 = torch.zeros(1, 2560, dtype=torch.float16, device="cuda")
        y2 = torch.zeros(1, 2048, dtype=torch.float32, device="cuda")
        ch.add_fused_rmsnorm_gemv(A.pack, x, r, g, EPS, h, y1, y_dtype=q.QMV_F16)
        ch.add_gemv(B.pack, y1[:, :2048], y2)          # depends on the first op
        outs[tag] = (h, y1, y2)
        return ch

    ref = build(q.Chain(4), "ws")
    na = build(q.Chain(4, no_alloc=True), "na")
    other = q.Chain(2, no_alloc=True)
    y_other = torch.zeros(1, 2048, dtype=torch.float32, device="cuda")
    other.add_gemv(B.pack, x, y_other)
    ref.run()
    torch.cuda.synchronize()
    for call in range(2):
        for t in outs["na"]:
            t.zero_()
        na.run()
        other.run()                                    # uses the same scratch array next
        torch.cuda.synchronize()
        for a, b in zip(outs["na"], outs["ws"]):
            assert torch.equal(_bits(a), _bits(b)), call
    assert torch.equal(_bits(y_other), _bits(q.qmv_gemv(B.pack, x)))
    assert q.qmv_device_error(clear=True) == 0


def test_no_alloc_chains_alternate_on_one_stream():
    """Two no-alloc chains queued one after another on a side stream (no
    synchronisation between the runs): each run's op-table copy is ordered on
    that stream after the other chain's kernel, so both keep their results."""
    q = qmv()
    A = Mat("na2.A", 2048, 2048, 2, 32)
    B = Mat("na2.B", 2560, 2048, 4, 32)
    x = to_dev(acts("na2", 1, 2048)[0])
    ya = torch.zeros(1, 2048, dtype=torch.float32, device="cuda")
    yb = torch.zeros(1, 2560, dtype=torch.float32, device="cuda")
    ca = q.Chain(1, no_alloc=True).add_gemv(A.pack, x, ya)
    cb = q.Chain(1, no_alloc=True).add_gemv(B.pack, x, yb)
    ref_a, ref_b = q.qmv_gemv(A.pack, x), q.qmv_gemv(B.pack, x)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(4):
            ca.run(s)
            cb.run(s)
    s.synchronize()
    assert torch.equal(_bits(ya), _bits(ref_a))
    assert torch.equal(_bits(yb), _bits(ref_b))
    assert q.qmv_device_error(clear=True) == 0


def test_no_alloc_rejects_oversize():
    q = qmv()
    with pytest.raises(q.QmvError) as e:
        q.Chain(1025, no_alloc=True)
    assert e.value.status == q.QMV_ERR_UNSUPPORTED
