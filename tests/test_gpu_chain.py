"""GPU parity of the persistent matvec chain (qmv_chain_*): every op of a
chain must equal, bit for bit, the same qmv_gemv / qmv_fused_rmsnorm_gemv
call run on its own (same mode), including h_out; in exact mode the chain's
outputs are therefore also bit-identical to the oracle.  Grid barriers are
inserted exactly where an op's activations or outputs conflict with earlier
ops since the last barrier."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import EPS, GuardBuf, Mat, acts, bits_equal, first_diff, to_dev, qmv

pytestmark = pytest.mark.gpu


def _eq(a, b):
    return torch.equal(a.contiguous().view(torch.int16 if a.dtype == torch.float16 else torch.int32),
                       b.contiguous().view(torch.int16 if b.dtype == torch.float16 else torch.int32))


def _layer_mats(tag):
    return {"qkv": Mat(f"ch.{tag}.qkv", 2560, 2048, 4, 32),
            "o": Mat(f"ch.{tag}.o", 2048, 2048, 4, 32),
            "gateup": Mat(f"ch.{tag}.gu", 16384, 2048, 2, 32),
            "down": Mat(f"ch.{tag}.down", 2048, 8192, 2, 32)}


def _bufs(tag):
    d = {}
    for name, K in (("x", 2048), ("r", 2048), ("attn", 2048), ("act", 8192)):
        x, _, _ = acts(f"ch.{tag}.{name}", 1, K)
        d[name] = to_dev(x)
    _, _, g1 = acts(f"ch.{tag}.g1", 1, 2048)
    _, _, g2 = acts(f"ch.{tag}.g2", 1, 2048)
    d["g1"], d["g2"] = to_dev(g1), to_dev(g2)
    return d


def _outs(guards=None):
    """the layer's outputs; with a guards list, each sits between guard
    bands (appended to the list, to be checked after the chain runs)"""
    def mk(n, dt):
        if guards is None:
            return torch.zeros(1, n, dtype=dt, device="cuda")
        g = GuardBuf(n * (2 if dt == torch.float16 else 4))
        guards.append(g)
        return g.view(dt, (1, n))
    f = lambda n: mk(n, torch.float32)
    h = lambda n: mk(n, torch.float16)
    return {"h": h(2048), "h2": h(2048), "y_qkv": f(2560), "y_o": f(2048), "y_gu": f(16384),
            "y_down": f(2048)}


def _layer_ops(layer, b, o):
    """the decode-layer op list (same buffers as the benchmark's layer)"""
    return [("fused", layer["qkv"], b["x"], b["r"], b["g1"], o["h"], o["y_qkv"]),
            ("gemv", layer["o"], b["attn"], o["y_o"]),
            ("fused", layer["gateup"], b["attn"], o["h"], b["g2"], o["h2"], o["y_gu"]),
            ("gemv", layer["down"], b["act"], o["y_down"])]


def _run_single(q, op, mode):
    if op[0] == "fused":
        _, m, x, r, g, h, y = op
        q.qmv_fused_rmsnorm_gemv(m.pack, x, r, g, EPS, h_out=h, y=y, mode=mode)
    else:
        _, m, x, y = op
        q.qmv_gemv(m.pack, x, y=y, mode=mode)


def _add(q, ch, op, mode):
    if op[0] == "fused":
        _, m, x, r, g, h, y = op
        ch.add_fused_rmsnorm_gemv(m.pack, x, r, g, EPS, h, y, mode=mode)
    else:
        _, m, x, y = op
        ch.add_gemv(m.pack, x, y, mode=mode)


@pytest.fixture(scope="module")
def layers():
    return [_layer_mats("L0"), _layer_mats("L1")]


@pytest.mark.parametrize("mode", ["fast", "exact"])
def test_decode_layers_chain_equals_calls(layers, mode):
    q = qmv()
    md = q.QMV_FAST if mode == "fast" else q.QMV_EXACT
    b = _bufs("L")
    guards = []
    ref_o, got_o = _outs(), _outs(guards)
    # reference: the calls one by one, outputs snapshotted after each op
    ref = []
    for lay in layers:
        for op in _layer_ops(lay, b, ref_o):
            _run_single(q, op, md)
            ref.append([t.clone() for t in op[5:]] if op[0] == "fused" else [op[3].clone()])
    ch = q.Chain(8)
    ops = [op for lay in layers for op in _layer_ops(lay, b, got_o)]
    for op in ops:
        _add(q, ch, op, md)
    # gate/up reads h written by q/k/v; the next layer's q/k/v rewrites h
    assert ch.info()["barriers"] == 3
    ch.run()
    torch.cuda.synchronize()
    assert q.qmv_device_error(clear=True) == 0
    for i, g in enumerate(guards):
        g.check(f"chain output {i}")
    # the last layer's outputs equal the last calls' outputs
    for op, r in zip(ops[4:], ref[4:]):
        outs = list(op[5:]) if op[0] == "fused" else [op[3]]
        for t, rt in zip(outs, r):
            assert _eq(t, rt)
    if mode == "exact":
        codes, scales = layers[1]["o"].host()
        y_ref = oracle.gemv(codes, scales, 32, b["attn"].cpu().numpy())
        assert bits_equal(got_o["y_o"].cpu().numpy(), y_ref), first_diff(got_o["y_o"].cpu().numpy(), y_ref)


def test_dependent_chain_fp16_outputs_feed_next_op():
    """x -> A -> B -> A -> ... through fp16 outputs: a barrier before every op
    after the first, and every intermediate equal to the plain calls."""
    q = qmv()
    A = Mat("chdepA", 2048, 2048, 2, 32)
    B = Mat("chdepB", 2048, 2048, 4, 32)
    x, _, _ = acts("chdep", 1, 2048)
    xd = to_dev(x)
    n = 10
    ys = [torch.zeros(1, 2048, dtype=torch.float16, device="cuda") for _ in range(n)]
    ch = q.Chain(n)
    cur = xd
    for i in range(n):
        ch.add_gemv((A if i % 2 == 0 else B).pack, cur, ys[i], y_dtype=q.QMV_F16)
        cur = ys[i]
    assert ch.info()["barriers"] == n - 1
    ch.run()
    ref = []
    cur = xd
    for i in range(n):
        cur = q.qmv_gemv((A if i % 2 == 0 else B).pack, cur, y_dtype=q.QMV_F16)
        ref.append(cur)
    torch.cuda.synchronize()
    for g, r in zip(ys, ref):
        assert _eq(g, r)
    assert q.qmv_device_error(clear=True) == 0


@pytest.mark.parametrize("N,K,bits,group", [(1000, 5376, 8, 5376), (777, 5376, 4, 32),
                                            (3, 256, 2, 32), (5000, 1024, 8, 32),
                                            (300, 16384, 2, 32)])
@pytest.mark.parametrize("mode", ["fast", "exact"])
def test_ragged_and_wide_ops_equal_calls(N, K, bits, group, mode):
    """ragged row counts, three K segments, per-row int8, tiny N; the same
    pack run twice on different inputs in one chain (no conflict: no barrier)"""
    q = qmv()
    md = q.QMV_FAST if mode == "fast" else q.QMV_EXACT
    m = Mat(f"chr{N}x{K}b{bits}", N, K, bits, group)
    xs = [to_dev(acts(f"chr{N}x{K}.{i}", 1, K)[0]) for i in range(2)]
    _, r, g = acts(f"chr{N}x{K}.rg", 1, K)
    rd, gd = to_dev(r), to_dev(g)
    ys = [torch.zeros(1, N, dtype=torch.float32, device="cuda") for _ in range(3)]
    h = torch.zeros(1, K, dtype=torch.float16, device="cuda")
    ch = q.Chain(3)
    ch.add_gemv(m.pack, xs[0], ys[0], mode=md)
    ch.add_gemv(m.pack, xs[1], ys[1], mode=md)
    ch.add_fused_rmsnorm_gemv(m.pack, xs[0], rd, gd, EPS, h, ys[2], mode=md)
    assert ch.info()["barriers"] == 0
    ch.run()
    r0 = q.qmv_gemv(m.pack, xs[0], mode=md)
    r1 = q.qmv_gemv(m.pack, xs[1], mode=md)
    hr = torch.zeros_like(h)
    r2 = q.qmv_fused_rmsnorm_gemv(m.pack, xs[0], rd, gd, EPS, h_out=hr, mode=md)
    torch.cuda.synchronize()
    assert _eq(ys[0], r0) and _eq(ys[1], r1) and _eq(ys[2], r2)
    assert _eq(h, hr)
    if mode == "exact":
        codes, scales = m.host()
        ref = oracle.gemv(codes, scales, group, xs[1].cpu().numpy())
        assert bits_equal(ys[1].cpu().numpy(), ref), first_diff(ys[1].cpu().numpy(), ref)


def test_long_chain_reruns_identically():
    """64 ops over 4 packs (ring and CTA rotation across many ops), run twice,
    and captured in a CUDA graph"""
    q = qmv()
    mats = [Mat(f"chl{i}", n, 2048, b, 32) for i, (n, b) in
            enumerate([(1536, 2), (2560, 4), (4096, 2), (640, 8)])]
    xs = [to_dev(acts(f"chl.x{i}", 1, 2048)[0]) for i in range(4)]
    ys = [torch.zeros(1, mats[i % 4].N, dtype=torch.float32, device="cuda") for i in range(64)]
    ch = q.Chain(64)
    for i in range(64):
        ch.add_gemv(mats[i % 4].pack, xs[(i // 4) % 4], ys[i])
    assert ch.info()["barriers"] == 0
    ch.run()
    torch.cuda.synchronize()
    first = [y.clone() for y in ys]
    for y in ys:
        y.zero_()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ch.run(s)
    torch.cuda.synchronize()
    for y, f in zip(ys, first):
        assert _eq(y, f)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ch.run(s)
    for y in ys:
        y.zero_()
    g.replay()
    torch.cuda.synchronize()
    for y, f in zip(ys, first):
        assert _eq(y, f)
    for i in range(0, 64, 9):
        r = q.qmv_gemv(mats[i % 4].pack, xs[(i // 4) % 4])
        torch.cuda.synchronize()
        assert _eq(ys[i], r)
    assert q.qmv_device_error(clear=True) == 0


def test_chain_argument_errors():
    q = qmv()
    m = Mat("cherr", 64, 2048, 2, 32)
    m96 = Mat("cherr96", 64, 128, 2, 32)
    x = torch.zeros(1, 2048, dtype=torch.float16, device="cuda")
    y = torch.zeros(1, 64, dtype=torch.float32, device="cuda")
    ch = q.Chain(1)
    with pytest.raises(q.QmvError) as e:
        ch.add_gemv(m96.pack, x[:, :128], y)
    assert e.value.status == q.QMV_ERR_UNSUPPORTED
    ch.add_gemv(m.pack, x, y)
    with pytest.raises(q.QmvError) as e:
        ch.add_gemv(m.pack, x, y)          # full
    assert e.value.status == q.QMV_ERR_INVALID_ARG
    lib = q.lib()
    assert lib.qmv_chain_add_gemv(ch.handle, m.pack.handle, x.data_ptr() + 2, y.data_ptr(), 0, 0) in (
        q.QMV_ERR_INVALID_ARG, q.QMV_ERR_ALIGNMENT)
