"""Helpers shared by the GPU parity tests: seeded inputs on both sides, the
CUDA path through the C ABI, the oracle on the CPU, and the comparisons."""
import numpy as np
import torch

import oracle
import synth

SEED = synth.DEFAULT_SEED
EPS = 1e-6
TOL = 1e-3   # fast mode: max |y - ref| <= TOL * (1 + |ref|)


def qmv():
    from bit_weight_only_packed_gb300 import qmv as q
    return q


def dev():
    return torch.device("cuda")


class Mat:
    """One packed matrix: device pack, and a way to get host codes/scales of
    any rows (regenerated from the same seeded streams, never read back from
    the GPU)."""

    def __init__(self, name, N, K, bits, group, seed=SEED, device_gen=None, ternary=False):
        self.name, self.N, self.K, self.bits, self.group, self.seed = name, N, K, bits, group, seed
        self.G = K // group
        self.ternary = ternary
        big = N * K > (1 << 26) if device_gen is None else device_gen
        gdev = dev() if big else "cpu"
        codes = self._codes(device=gdev)
        scales = synth.scales(seed, name, N, self.G, device=gdev)
        self.pack = qmv().Pack(N, K, bits, group).pack_weights(codes.to(dev()), scales.to(dev()))
        self._host = None if big else (codes.numpy(), scales.numpy())
        del codes, scales

    def _codes(self, rows=None, device="cpu"):
        if self.ternary:
            return synth.ternary_codes(self.seed, self.name, self.N, self.K, rows=rows, device=device)
        return synth.codes(self.seed, self.name, self.N, self.K, self.bits, rows=rows, device=device)

    def host(self, rows=None):
        if rows is None:
            if self._host is None:
                raise ValueError("full host copy not kept for large matrices; pass rows")
            return self._host
        if self._host is not None:
            c, s = self._host
            return c[rows], s[rows]
        c = self._codes(rows=rows).numpy()
        s = synth.scales(self.seed, self.name, self.N, self.G, rows=rows).numpy()
        return c, s


def acts(name, M, K, outliers=False, seed=SEED):
    every = 1000 if outliers else 0
    x = synth.normal_f16(seed, name + ".x", (M, K), outlier_every=every)
    r = synth.normal_f16(seed, name + ".r", (M, K), outlier_every=every)
    g = synth.normal_f16(seed, name + ".gamma", (K,), mean=1.0, std=0.1)
    return x, r, g


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


def sample_rows(N, n=256, seed=1):
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([np.arange(min(N, 8)), np.arange(max(0, N - 8), N),
                                     rng.integers(0, N, size=n)]))
    return rows


def bits_equal(a, b):
    a = np.ascontiguousarray(a, dtype=np.float32)
    b = np.ascontiguousarray(b, dtype=np.float32)
    return a.shape == b.shape and np.array_equal(a.view(np.uint32), b.view(np.uint32))


def first_diff(a, b):
    a = np.asarray(a, np.float32).ravel()
    b = np.asarray(b, np.float32).ravel()
    d = np.nonzero(a.view(np.uint32) != b.view(np.uint32))[0]
    if d.size == 0:
        return "equal"
    i = d[0]
    return f"{d.size} differ; first at {i}: gpu {a[i]!r} oracle {b[i]!r}"


def within_tol(y, ref, tol=TOL):
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    return np.all(np.abs(y - ref) <= tol * (1.0 + np.abs(ref)))


def max_rel_err(y, ref):
    """max |y - ref| / (1 + |ref|), for failure messages"""
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.max(np.abs(y - ref) / (1.0 + np.abs(ref))))


# ------------------------------------------------------------ guard bands --
# compute-sanitizer is not available, so out-of-bounds stores are caught by
# guard bands: every output (and workspace) of a guarded call sits between
# two 4 KiB bands of 0xA5 that must be intact after the call.

GUARD = 4096
CANARY = 0xA5


class GuardBuf:
    """nbytes of device memory between two GUARD-byte bands of CANARY (the
    payload itself filled with `fill`); the payload is 256-byte aligned."""

    def __init__(self, nbytes, fill=CANARY):
        self.nbytes = int(nbytes)
        self.raw = torch.full((2 * GUARD + self.nbytes,), CANARY, dtype=torch.uint8, device="cuda")
        if fill != CANARY:
            self.raw[GUARD:GUARD + self.nbytes].fill_(fill)

    def view(self, dtype, shape):
        return self.raw[GUARD:GUARD + self.nbytes].view(dtype).view(shape)

    def check(self, what):
        lo = torch.nonzero(self.raw[:GUARD] != CANARY)
        hi = torch.nonzero(self.raw[GUARD + self.nbytes:] != CANARY)
        assert lo.numel() == 0, f"{what}: {lo.numel()} bytes written before the buffer (first at -{GUARD - int(lo[0])})"
        assert hi.numel() == 0, f"{what}: {hi.numel()} bytes written past the buffer (first at +{int(hi[0])})"


def _esize(dtype):
    return torch.tensor([], dtype=dtype).element_size()


def guarded_like(t):
    """A guarded buffer shaped and typed like tensor t (payload 0xA5)."""
    g = GuardBuf(t.numel() * _esize(t.dtype))
    return g, g.view(t.dtype, t.shape)


class _GuardedQmv:
    """The binding with guard bands around every output, h_out and workspace
    of the matvec calls (the workspace payload is filled with 0x5A: its
    contents on entry must not matter); each call synchronises, checks the
    bands, and returns (or fills) the caller's outputs as the binding does."""

    def __init__(self, q):
        self._q = q

    def __getattr__(self, name):
        return getattr(self._q, name)

    def _ydt(self, y_dtype):
        return torch.float16 if y_dtype == self._q.QMV_F16 else torch.float32

    def _ws(self, p, M, y_dtype, mode, fused):
        n = self._q.qmv_workspace_bytes(p, M, y_dtype, mode, fused)
        if n == 0:
            return None, None
        g = GuardBuf(n, fill=0x5A)
        return g, g.view(torch.uint8, (n,))

    def _finish(self, bufs, outs):
        torch.cuda.synchronize()
        for name, g in bufs:
            if g is not None:
                g.check(name)
        for dst, src in outs:
            if dst is not None:
                dst.copy_(src)

    def _call(self, fn, p, M, N, y, y_dtype, mode, fused, h_out, **kw):
        gy = GuardBuf(M * N * _esize(self._ydt(y_dtype)))
        yv = gy.view(self._ydt(y_dtype), (M, N))
        gh, hv = (None, None) if h_out is None else guarded_like(h_out)
        gw, wv = self._ws(p, M, y_dtype, mode, fused)
        if fused:
            kw["h_out"] = hv
        fn(y=yv, y_dtype=y_dtype, mode=mode, workspace=wv, **kw)
        self._finish([("y", gy), ("h_out", gh), ("workspace", gw)], [(h_out, hv)])
        if y is not None:
            y.copy_(yv.view_as(y))
            return y
        return yv.clone()

    def qmv_gemv(self, p, x, y=None, y_dtype=0, mode=0, stream=None, M=None, workspace=None):
        M = x.shape[0] if (M is None and x.dim() == 2) else (M or 1)
        return self._call(lambda **kw: self._q.qmv_gemv(p, x, stream=stream, M=M, **kw),
                          p, M, p.N, y, y_dtype, mode, False, None)

    def qmv_chunk_gemm(self, p, x, y=None, y_dtype=0, mode=0, stream=None, workspace=None):
        return self._call(lambda **kw: self._q.qmv_chunk_gemm(p, x, stream=stream, **kw),
                          p, x.shape[0], p.N, y, y_dtype, mode, False, None)

    def qmv_fused_rmsnorm_gemv(self, p, x, residual, gamma, eps=1e-6, h_out=None, y=None, y_dtype=0,
                               mode=0, stream=None, workspace=None):
        M = x.shape[0] if x.dim() == 2 else 1
        return self._call(lambda **kw: self._q.qmv_fused_rmsnorm_gemv(p, x, residual, gamma, eps,
                                                                      stream=stream, **kw),
                          p, M, p.N, y, y_dtype, mode, True, h_out)

    def qmv_gemv_gather(self, p, rows_per_expert, expert_ids, x, y=None, y_dtype=0, mode=0, stream=None):
        n = expert_ids.numel() * rows_per_expert
        gy = GuardBuf(n * _esize(self._ydt(y_dtype)))
        yv = gy.view(self._ydt(y_dtype), (1, n))
        self._q.qmv_gemv_gather(p, rows_per_expert, expert_ids, x, y=yv, y_dtype=y_dtype, mode=mode,
                                stream=stream)
        self._finish([("y", gy)], [])
        if y is not None:
            y.copy_(yv.view_as(y))
            return y
        return yv.clone()

    def qmv_gemv_argmax(self, p, x, workspace, residual=None, gamma=None, eps=1e-6, h_out=None, y=None,
                        y_dtype=0, mode=0, stream=None, index=None, value=None):
        gi = GuardBuf(4)
        gv = GuardBuf(4)
        iv, vv = gi.view(torch.int32, (1,)), gv.view(torch.float32, (1,))
        gy, yv = (None, None) if y is None else guarded_like(y)
        gh, hv = (None, None) if h_out is None else guarded_like(h_out)
        gw = GuardBuf(workspace.numel() * workspace.element_size(), fill=0)
        wv = gw.view(torch.uint8, (gw.nbytes,))
        wv.copy_(workspace.view(torch.uint8).view(-1))
        self._q.qmv_gemv_argmax(p, x, wv, residual=residual, gamma=gamma, eps=eps, h_out=hv, y=yv,
                                y_dtype=y_dtype, mode=mode, stream=stream, index=iv, value=vv)
        self._finish([("index", gi), ("value", gv), ("y", gy), ("h_out", gh), ("workspace", gw)],
                     [(y, yv), (h_out, hv)])
        workspace.view(torch.uint8).view(-1).copy_(wv)
        if index is not None:
            index.copy_(iv)
        if value is not None:
            value.copy_(vv)
        return (index if index is not None else iv.clone()), (value if value is not None else vv.clone())


def qmv_guarded():
    """The binding with guard-band checks around every matvec output."""
    return _GuardedQmv(qmv())
