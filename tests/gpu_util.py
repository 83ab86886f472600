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
