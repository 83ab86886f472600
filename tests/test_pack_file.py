"""Saved packs: the versioned 64-byte header round-trips a pack's shape, and
every malformed header is refused on the host before anything is bound (no
GPU: these calls touch no device)."""
import ctypes
import struct

import pytest


@pytest.fixture(scope="module")
def q():
    from bit_weight_only_packed_gb300 import build
    build.build()
    from bit_weight_only_packed_gb300 import qmv
    return qmv


def _fields(h):
    magic, version, size, N, K, bits, group, cb, sb = struct.unpack_from("<8sIIiiiiQQ", h, 0)
    return magic, version, size, N, K, bits, group, cb, sb, h[48:]


@pytest.mark.parametrize("N,K,bits,group", [(1, 64, 2, 32), (2560, 2048, 4, 32), (37, 5376, 8, 5376),
                                            (4096, 14336, 2, 32)])
def test_header_round_trip(q, N, K, bits, group):
    p = q.Pack(N, K, bits, group)
    h = p.header()
    assert len(h) == q.QMV_PACK_HEADER_BYTES == 64
    magic, version, size, n, k, b, g, cb, sb, rest = _fields(h)
    assert magic == b"QMVPACK\0" and version == q.QMV_PACK_VERSION and size == 64
    assert (n, k, b, g) == (N, K, bits, group)
    assert cb == N * K * bits // 8 and sb == N * (K // group) * 2
    assert rest == bytes(16)
    r = q.Pack.from_header(h)
    assert (r.N, r.K, r.bits, r.group) == (N, K, bits, group)
    assert (r.codes_bytes, r.scales_bytes) == (p.codes_bytes, p.scales_bytes)
    assert r.header() == h


def _patched(q, off, fmt, value):
    h = bytearray(q.Pack(256, 1024, 2, 32).header())
    struct.pack_into(fmt, h, off, value)
    return bytes(h)


@pytest.mark.parametrize("what,off,fmt,value,status", [
    ("magic", 0, "<8s", b"QMVPACX\0", "QMV_ERR_INVALID_ARG"),
    ("header size", 12, "<I", 128, "QMV_ERR_INVALID_ARG"),
    ("reserved byte", 60, "<B", 1, "QMV_ERR_INVALID_ARG"),
    ("layout version", 8, "<I", 2, "QMV_ERR_UNSUPPORTED"),
    ("bits", 24, "<i", 3, "QMV_ERR_INVALID_ARG"),
    ("group", 28, "<i", 64, "QMV_ERR_INVALID_ARG"),
    ("K", 20, "<i", 1000, "QMV_ERR_SHAPE"),
    ("N", 16, "<i", 0, "QMV_ERR_SHAPE"),
    ("codes bytes", 32, "<Q", 1, "QMV_ERR_SHAPE"),
    ("scales bytes", 40, "<Q", 2 * 256 * 32 + 2, "QMV_ERR_SHAPE"),
])
def test_malformed_headers_are_refused(q, what, off, fmt, value, status):
    h = _patched(q, off, fmt, value)
    out = ctypes.c_void_p(1)
    buf = ctypes.create_string_buffer(h, len(h))
    st = q.lib().qmv_create_pack_from_header(ctypes.byref(out), buf, None, None)
    assert st == getattr(q, status), what
    assert not out.value, what   # nothing is handed out on failure
    with pytest.raises(q.QmvError):
        q.Pack.from_header(h)


def test_binding_checks_the_header_length_and_bind_arguments(q):
    with pytest.raises(ValueError):
        q.Pack.from_header(bytes(63))
    lib = q.lib()
    p = q.Pack(256, 1024, 2, 32)
    assert lib.qmv_bind_packed(p.handle, None, None) == q.QMV_ERR_INVALID_ARG
    assert lib.qmv_bind_packed(p.handle, 1 << 20, (1 << 20) + 8) == q.QMV_ERR_ALIGNMENT
    assert lib.qmv_pack_header(p.handle, None) == q.QMV_ERR_INVALID_ARG
    assert lib.qmv_pack_header(None, ctypes.create_string_buffer(64)) == q.QMV_ERR_INVALID_ARG
