"""The C-ABI library loads, exports every entry point that include/qmv.h
declares, and validates arguments on the host (no device is touched)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "qmv.h")


def _declared():
    txt = open(HEADER).read()
    return re.findall(r"QMV_API\s+[\w\s\*]*?\b(qmv_\w+)\s*\(", txt)


@pytest.fixture(scope="module")
def q():
    from bit_weight_only_packed_gb300 import build
    build.build()
    from bit_weight_only_packed_gb300 import qmv
    return qmv


def test_header_declares_the_abi():
    names = set(_declared())
    for n in ("qmv_create_pack", "qmv_pack_weights", "qmv_gemv", "qmv_fused_rmsnorm_gemv",
              "qmv_chunk_gemm", "qmv_destroy_pack", "qmv_status_string", "qmv_last_cuda_error"):
        assert n in names


def test_library_exports_every_declared_symbol(q):
    lib = ctypes.CDLL(q.LIB_PATH)
    for n in _declared():
        assert hasattr(lib, n), n
        assert n in q.SIGNATURES, n


@pytest.mark.parametrize("N,K,bits,group,status", [
    (16, 64, 3, 32, -1),      # bad width
    (16, 48, 2, 32, -4),      # int2 row not a whole number of 16-byte units
    (16, 96, 4, 32, 0),
    (16, 80, 8, 32, -4),      # K not a multiple of 32
    (0, 64, 2, 32, -4),       # N < 1
    (16, 64, 2, 64, 0),       # group == K (one scale per row)
    (16, 128, 2, 64, -1),     # group neither 32 nor K
    (8, 5376, 4, 32, 0),
])
def test_create_pack_validation(q, N, K, bits, group, status):
    h = ctypes.c_void_p()
    cb, sb = ctypes.c_size_t(), ctypes.c_size_t()
    rc = q.lib().qmv_create_pack(ctypes.byref(h), N, K, bits, group, ctypes.byref(cb), ctypes.byref(sb))
    assert rc == status
    if rc == 0:
        assert cb.value == N * K * bits // 8 and sb.value == N * (K // group) * 2
        n, k, b, g = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
        assert q.lib().qmv_pack_info(h, ctypes.byref(n), ctypes.byref(k), ctypes.byref(b),
                                     ctypes.byref(g)) == 0
        assert (n.value, k.value, b.value, g.value) == (N, K, bits, group)
        assert q.lib().qmv_destroy_pack(h) == 0
    else:
        assert not h.value


def test_calls_on_unbound_pack_fail_on_host(q):
    p = q.Pack(64, 128, 2, 32)
    lib = q.lib()
    # not packed yet -> invalid argument, before any CUDA call
    assert lib.qmv_gemv(p.handle, 1, 64, 128, 2, 32, 16, 32, 0, 0, None) == -1
    assert lib.qmv_chunk_gemm(p.handle, 4, 16, 32, 0, 0, None) == -1
    assert lib.qmv_fused_rmsnorm_gemv(p.handle, 1, 16, 16, 16, 1e-6, None, 32, 0, 0, None) == -1
    assert lib.qmv_unpack_codes(p.handle, 16, None) == -1
    # null and misaligned pointers are rejected on the host
    assert lib.qmv_pack_weights(p.handle, None, 16, 16, 16, None) == -1
    assert lib.qmv_pack_weights(p.handle, 8, 16, 16, 16, None) == -3
    assert lib.qmv_pack_weights(p.handle, 16, 16, 16, 24, None) == -3
    assert lib.qmv_gemv(None, 1, 64, 128, 2, 32, 16, 32, 0, 0, None) == -1
    assert lib.qmv_destroy_pack(None) == -1


def test_status_strings(q):
    for s in range(-6, 1):
        assert q.qmv_status_string(s) and q.qmv_status_string(s) != "unknown status"
    assert q.qmv_status_string(-99) == "unknown status"
    assert q.qmv_last_cuda_error() == 0
