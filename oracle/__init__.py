"""CPU oracle for the weight-only mixed-bit packed matvec.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg (and its ``--impl reference`` arm) import this
package.  The library under ``bit_weight_only_packed_gb300`` never imports it,
and this package imports nothing from the library.

The arithmetic lives in ``qmv_oracle.c`` (plain C99, single-threaded, built
with ``-ffp-contract=off -fno-fast-math``).  This module compiles it with gcc
on first use and wraps it with ctypes + numpy.  fp16 data crosses the boundary
as ``uint16`` bit patterns.

What each function computes, and the passage it follows, is stated in the C
file's header: the decode of 16 int2 codes per 32-bit word and the exact
products accumulated in fp32 in code order ("Gemma4 raw-Metal loop on A19 --
findings + the remaining (parked) levers", section "What moved the needle"),
K-order-fixed accumulation ("raw-metal-loop-playbook", prefill-regimes table),
and the residual-add + RMSNorm fold (A19 page, dispatch-count fusion item).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmv_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
CFLAGS = ["-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math",
          "-fno-strict-aliasing", "-shared", "-fPIC"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``qmv_oracle.c`` into ``oracle/_build/liboracle.so``."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i64 = ctypes.c_int64
            lib.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
            lib.orc_f16_to_f32.restype = ctypes.c_float
            lib.orc_f32_to_f16.argtypes = [ctypes.c_float]
            lib.orc_f32_to_f16.restype = ctypes.c_uint16
            lib.orc_f16_to_f32_array.argtypes = [P, P, i64]
            lib.orc_f32_to_f16_array.argtypes = [P, P, i64]
            lib.orc_pack.argtypes = [P, i64, i64, ctypes.c_int, P]
            lib.orc_pack.restype = ctypes.c_int
            lib.orc_unpack.argtypes = [P, i64, i64, ctypes.c_int, P]
            lib.orc_unpack.restype = ctypes.c_int
            lib.orc_residual_add.argtypes = [P, P, i64, P]
            lib.orc_sumsq.argtypes = [P, i64, ctypes.c_int]
            lib.orc_sumsq.restype = ctypes.c_float
            lib.orc_rms_inv.argtypes = [ctypes.c_float, i64, ctypes.c_float]
            lib.orc_rms_inv.restype = ctypes.c_float
            lib.orc_rmsnorm.argtypes = [P, P, i64, ctypes.c_float, ctypes.c_int, P]
            lib.orc_fused_residual_rmsnorm.argtypes = [P, P, P, i64, i64,
                                                       ctypes.c_float, P, P]
            lib.orc_gemv.argtypes = [P, P, i64, i64, i64, P, i64, P]
            lib.orc_gemv.restype = ctypes.c_int
            lib.orc_argmax.argtypes = [P, i64, P]
            lib.orc_argmax.restype = i64
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _h16(a) -> np.ndarray:
    """Accept float16 arrays or uint16 bit patterns; return uint16 bits."""
    a = np.asarray(a)
    if a.dtype == np.float16:
        return np.ascontiguousarray(a).view(np.uint16)
    return _c(a, np.uint16)


# ------------------------------------------------------------------ fp16 --

def f16_to_f32(h) -> np.ndarray:
    h = _h16(h)
    out = np.empty(h.shape, np.float32)
    _load().orc_f16_to_f32_array(_ptr(h), _ptr(out), h.size)
    return out


def f32_to_f16(f) -> np.ndarray:
    """fp32 -> fp16 bits (uint16), round to nearest even."""
    f = _c(f, np.float32)
    out = np.empty(f.shape, np.uint16)
    _load().orc_f32_to_f16_array(_ptr(f), _ptr(out), f.size)
    return out


# ------------------------------------------------------------ pack/unpack --

def pack(codes, bits: int) -> np.ndarray:
    """Signed codes [N, K] (int8) -> packed words [N, K*bits/32] (uint32)."""
    codes = _c(codes, np.int8)
    N, K = codes.shape
    words = np.empty((N, K * bits // 32), np.uint32)
    rc = _load().orc_pack(_ptr(codes), N, K, bits, _ptr(words))
    if rc != 0:
        raise ValueError(f"orc_pack failed ({rc})")
    return words


def unpack(words, K: int, bits: int) -> np.ndarray:
    words = _c(words, np.uint32)
    N = words.shape[0]
    codes = np.empty((N, K), np.int8)
    rc = _load().orc_unpack(_ptr(words), N, K, bits, _ptr(codes))
    if rc != 0:
        raise ValueError(f"orc_unpack failed ({rc})")
    return codes


# ------------------------------------------------------ residual/RMSNorm --

def residual_add(x, r) -> np.ndarray:
    x, r = _h16(x), _h16(r)
    h = np.empty(x.shape, np.uint16)
    _load().orc_residual_add(_ptr(x), _ptr(r), x.size, _ptr(h))
    return h


def sumsq(h, order: int = 0) -> float:
    h = _h16(h)
    return float(_load().orc_sumsq(_ptr(h), h.size, order))


def rms_inv(ss: float, K: int, eps: float) -> float:
    return float(_load().orc_rms_inv(ss, K, eps))


def rmsnorm(h, gamma, eps: float = 1e-6, order: int = 0) -> np.ndarray:
    """Unfused RMSNorm of one K-vector (fp16 bits in, fp16 bits out)."""
    h, gamma = _h16(h), _h16(gamma)
    y = np.empty(h.shape, np.uint16)
    _load().orc_rmsnorm(_ptr(h), _ptr(gamma), h.size, eps, order, _ptr(y))
    return y


def fused_residual_rmsnorm(x, r, gamma, eps: float = 1e-6):
    """x, r: [M, K] fp16; gamma: [K].  Returns (h, y), both [M, K] fp16 bits."""
    x, r, gamma = _h16(x), _h16(r), _h16(gamma)
    if x.ndim == 1:
        x, r = x[None], r[None]
    M, K = x.shape
    h = np.empty((M, K), np.uint16)
    y = np.empty((M, K), np.uint16)
    _load().orc_fused_residual_rmsnorm(_ptr(x), _ptr(r), _ptr(gamma), M, K, eps,
                                       _ptr(h), _ptr(y))
    return h, y


# ---------------------------------------------------------------- matvec --

def gemv(codes, scales, group: int, y) -> np.ndarray:
    """codes [N, K] int8, scales [N, K/group] fp16, y [M, K] fp16 -> [M, N] fp32."""
    codes = _c(codes, np.int8)
    scales = _h16(scales)
    y = _h16(y)
    if y.ndim == 1:
        y = y[None]
    N, K = codes.shape
    M = y.shape[0]
    assert y.shape[1] == K and scales.shape == (N, K // group)
    out = np.empty((M, N), np.float32)
    rc = _load().orc_gemv(_ptr(codes), _ptr(scales), N, K, group, _ptr(y), M, _ptr(out))
    if rc != 0:
        raise ValueError(f"orc_gemv failed ({rc})")
    return out


def argmax(y):
    """(index, value) of the largest of the fp32 vector y, first max on ties;
    (-1, nan) if there is none."""
    y = _c(np.asarray(y, np.float32).ravel(), np.float32)
    v = ctypes.c_float(float("nan"))
    lib = _load()
    idx = lib.orc_argmax(_ptr(y), y.size, ctypes.byref(v))
    return int(idx), float(v.value)


def fused_rmsnorm_gemv(codes, scales, group: int, x, r, gamma, eps: float = 1e-6):
    """The whole fused path: (h, y16, out) for M columns."""
    h, y16 = fused_residual_rmsnorm(x, r, gamma, eps)
    return h, y16, gemv(codes, scales, group, y16)
