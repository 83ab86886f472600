"""Seeded synthetic inputs shared by the oracle side and the GPU side.

This module holds none of the method's arithmetic: no packing, no decode, no
norm, no dot.  It only draws numbers.  The same functions run on the CPU
(oracle inputs, small cases) and on a CUDA device (full-size weights, so that
gigabyte-sized code matrices need not cross PCIe/C2C); both give identical
integers because every step is 64-bit integer arithmetic or a single IEEE
binary32 operation.

Generator: SplitMix64 (G. L. Steele, D. Lea, C. H. Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014), used counter-style: the i-th
output of a stream with starting state s0 is mix64(s0 + (i + 1) * GAMMA).
A stream's starting state is mix64(seed ^ mix64(stream_id + GAMMA)), where
stream_id is the FNV-1a 64-bit hash of the stream's name.

Recipes (the shapes and value distributions of the decode workloads):
  codes   field u = top `bits` bits of draw(n*K + k); signed code v = u - 2^(bits-1)
          -- uniform over all 2^bits codes ({-2,-1,0,1} for int2);
  scales  s = fp16( 0.005f + 0.015f * (float(draw >> 40) * 2^-24) ), fp32 ops,
          i.e. uniform in [0.005, 0.02];
  normal  Box-Muller in float64 from two draws, then mean + std * z rounded to
          fp16 (activations, residuals ~ N(0,1); RMSNorm gamma ~ N(1, 0.1));
  outliers  element i becomes +-50 when draw(i) mod 1000 == 0 (0.1 %).
"""
from __future__ import annotations

import numpy as np
import torch

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
DEFAULT_SEED = 20261202


def _signed(c: int) -> int:
    c &= MASK64
    return c - (1 << 64) if c >= (1 << 63) else c


def mix64_int(z: int) -> int:
    """SplitMix64 finaliser on a Python int (reference form)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * _M1) & MASK64
    z = ((z ^ (z >> 27)) * _M2) & MASK64
    return z ^ (z >> 31)


def fnv1a64(data: bytes) -> int:
    h = 0xCBF29CE484222325
    for b in data:
        h ^= b
        h = (h * 0x100000001B3) & MASK64
    return h


def stream_id(name: str) -> int:
    return fnv1a64(name.encode())


def stream_key(seed: int, name: str) -> int:
    return mix64_int((seed & MASK64) ^ mix64_int(stream_id(name) + GAMMA))


def draw_int(key: int, i: int) -> int:
    """The i-th output of a stream, pure Python (reference for the tensor form)."""
    return mix64_int(key + (i + 1) * GAMMA)


def _lsr(z: torch.Tensor, s: int) -> torch.Tensor:
    """Logical shift right of int64 bit patterns."""
    return (z >> s) & ((1 << (64 - s)) - 1)


def draws(key: int, idx: torch.Tensor) -> torch.Tensor:
    """SplitMix64 outputs for counters `idx` (int64 tensor), as int64 bit patterns."""
    z = idx + 1
    z = z * _signed(GAMMA) + _signed(key)
    z = (z ^ _lsr(z, 30)) * _signed(_M1)
    z = (z ^ _lsr(z, 27)) * _signed(_M2)
    return z ^ _lsr(z, 31)


def _row_index(rows, N: int, device) -> torch.Tensor:
    if rows is None:
        return torch.arange(N, dtype=torch.int64, device=device)
    return torch.as_tensor(np.asarray(rows, dtype=np.int64), device=device)


def codes(seed: int, name: str, N: int, K: int, bits: int, rows=None,
          device="cpu", chunk_elems: int = 1 << 26) -> torch.Tensor:
    """Signed codes [len(rows) or N, K] (int8) for matrix `name`."""
    key = stream_key(seed, name + ".codes")
    r = _row_index(rows, N, device)
    out = torch.empty((r.numel(), K), dtype=torch.int8, device=device)
    rows_per_chunk = max(1, chunk_elems // max(K, 1))
    kk = torch.arange(K, dtype=torch.int64, device=device)
    bias = 1 << (bits - 1)
    for r0 in range(0, r.numel(), rows_per_chunk):
        rr = r[r0:r0 + rows_per_chunk]
        idx = rr[:, None] * K + kk[None, :]
        u = _lsr(draws(key, idx), 64 - bits)
        out[r0:r0 + rr.numel()] = (u - bias).to(torch.int8)
    return out


def ternary_codes(seed: int, name: str, N: int, K: int, rows=None,
                  device="cpu") -> torch.Tensor:
    """Ternary codes [len(rows) or N, K] (int8), uniform over {-1, 0, 1}
    (the top 31 bits of each draw, modulo 3, minus 1)."""
    key = stream_key(seed, name + ".tcodes")
    r = _row_index(rows, N, device)
    kk = torch.arange(K, dtype=torch.int64, device=device)
    u = _lsr(draws(key, r[:, None] * K + kk[None, :]), 33)
    return (torch.remainder(u, 3) - 1).to(torch.int8)


def scales(seed: int, name: str, N: int, G: int, rows=None, device="cpu",
           lo: float = 0.005, hi: float = 0.02) -> torch.Tensor:
    """fp16 scales [len(rows) or N, G], uniform in [lo, hi]."""
    key = stream_key(seed, name + ".scales")
    r = _row_index(rows, N, device)
    gg = torch.arange(G, dtype=torch.int64, device=device)
    idx = r[:, None] * G + gg[None, :]
    u24 = _lsr(draws(key, idx), 40).to(torch.float32)          # exact (24 bits)
    unit = u24 * torch.tensor(2.0 ** -24, dtype=torch.float32, device=device)
    span = torch.tensor(hi - lo, dtype=torch.float32, device=device)
    base = torch.tensor(lo, dtype=torch.float32, device=device)
    return (unit * span + base).to(torch.float16)


def normal_f16(seed: int, name: str, shape, mean: float = 0.0, std: float = 1.0,
               outlier_every: int = 0, outlier_mag: float = 50.0) -> np.ndarray:
    """Host-side fp16 normal samples (Box-Muller in float64)."""
    n = int(np.prod(shape))
    key = stream_key(seed, name)
    idx = torch.arange(2 * n, dtype=torch.int64)
    d = draws(key, idx).numpy().view(np.uint64)
    u1 = ((d[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
    u2 = (d[1::2] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    v = mean + std * z
    if outlier_every:
        ko = stream_key(seed, name + ".outliers")
        o = draws(ko, torch.arange(n, dtype=torch.int64)).numpy().view(np.uint64)
        hit = (o % np.uint64(outlier_every)) == 0
        sign = np.where((o >> np.uint64(63)) & np.uint64(1), -1.0, 1.0)
        v = np.where(hit, sign * outlier_mag, v)
    return v.astype(np.float16).reshape(shape)


def checksum(a) -> int:
    """FNV-1a 64 of a buffer's bytes (for recording inputs)."""
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu().numpy()
    return fnv1a64(np.ascontiguousarray(a).tobytes())
