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
    assert lib.qmv_gemv(p.handle, 1, 64, 128, 2, 32, 16, 32, 0, 0, None, 0, None) == -1
    assert lib.qmv_chunk_gemm(p.handle, 4, 16, 32, 0, 0, None, 0, None) == -1
    assert lib.qmv_fused_rmsnorm_gemv(p.handle, 1, 16, 16, 16, 1e-6, None, 32, 0, 0, None, 0, None) == -1
    assert lib.qmv_unpack_codes(p.handle, 16, None) == -1
    # null and misaligned pointers are rejected on the host
    assert lib.qmv_pack_weights(p.handle, None, 16, 16, 16, None) == -1
    assert lib.qmv_pack_weights(p.handle, 8, 16, 16, 16, None) == -3
    assert lib.qmv_pack_weights(p.handle, 16, 16, 16, 24, None) == -3
    assert lib.qmv_gemv(None, 1, 64, 128, 2, 32, 16, 32, 0, 0, None, 0, None) == -1
    assert lib.qmv_destroy_pack(None) == -1


def test_status_strings(q):
    for s in range(-7, 1):
        assert q.qmv_status_string(s) and q.qmv_status_string(s) != "unknown status"
    assert q.qmv_status_string(-99) == "unknown status"
    assert q.qmv_last_cuda_error() == 0


def test_workspace_sizes_follow_the_dispatch(q):
    # qmv_workspace_bytes, host only.  Nothing for M = 1, or where K is not a
    # multiple of 256 (the 32-column tiles need no scratch).  The pipelined
    # M-column tiles take one table record per 512 codes and column chunk:
    # 8960 bytes per 4 columns, or 17408 per 8 where the tile-shape chooser
    # takes 8-column tiles (never below 5 columns); the fused prologue needs
    # no scratch of its own.  The int2 tensor tiles
    # (M > 32, fast mode) take split-K partial tiles only, never more than a
    # split of 8 over 128 columns.
    def tables(M, K):
        segs = -(-K // 512)
        four = -(-M // 4) * segs * 8960
        if M < 5:
            return {four}
        return {four, -(-M // 8) * segs * 17408}

    p2 = q.Pack(28672, 4096, 2, 32)
    p4 = q.Pack(4096, 4096, 4, 32)
    assert q.qmv_workspace_bytes(p2, 1, q.QMV_F32, q.QMV_FAST, fused=True) == 0
    assert q.qmv_workspace_bytes(p2, 1, q.QMV_F32, q.QMV_FAST) == 0
    assert q.qmv_workspace_bytes(p2, 16, q.QMV_F32, q.QMV_FAST, fused=True) in tables(16, 4096)
    assert q.qmv_workspace_bytes(p2, 3, q.QMV_F16, q.QMV_EXACT, fused=True) == 8 * 8960
    assert q.qmv_workspace_bytes(p2, 16, q.QMV_F32, q.QMV_FAST) in tables(16, 4096)
    assert q.qmv_workspace_bytes(p2, 2, q.QMV_F16, q.QMV_EXACT) == 8 * 8960
    assert q.qmv_workspace_bytes(p2, 128, q.QMV_F32, q.QMV_EXACT) in tables(128, 4096)
    assert q.qmv_workspace_bytes(p4, 128, q.QMV_F16, q.QMV_FAST) in tables(128, 4096)
    assert q.qmv_workspace_bytes(p4, 128, q.QMV_F16, q.QMV_FAST, fused=True) in tables(128, 4096)
    # the size does not depend on the output type or, for these tiles, the mode
    for M in (2, 5, 8, 16, 32, 40):
        n = q.qmv_workspace_bytes(p4, M, q.QMV_F32, q.QMV_EXACT)
        assert n in tables(M, 4096), (M, n)
        assert n == q.qmv_workspace_bytes(p4, M, q.QMV_F16, q.QMV_FAST), M
    # a partial last segment (K = 4352 = 8.5 segments) takes a whole record
    p5 = q.Pack(64, 4352, 4, 32)
    assert q.qmv_workspace_bytes(p5, 5, q.QMV_F32, q.QMV_FAST) in {2 * 9 * 8960, 9 * 17408}
    # K not a multiple of 256: the 32-column tiles, no scratch
    p6 = q.Pack(64, 320, 4, 32)
    assert q.qmv_workspace_bytes(p6, 16, q.QMV_F32, q.QMV_FAST) == 0
    assert q.qmv_workspace_bytes(p6, 16, q.QMV_F32, q.QMV_FAST, fused=True) == 0
    for M in (33, 64, 128, 200):
        for dt in (q.QMV_F32, q.QMV_F16):
            n = q.qmv_workspace_bytes(p2, M, dt, q.QMV_FAST)
            assert n % 256 == 0 and n <= 8 * 128 * 28672 * 4, (M, dt, n)
    # the down projection's shape splits K with fp16 output: it needs scratch
    pd = q.Pack(4096, 14336, 2, 32)
    assert q.qmv_workspace_bytes(pd, 128, q.QMV_F16, q.QMV_FAST) > 0


def test_binding_checks_tensors_before_any_call(q):
    # The ABI takes bare pointers, so the binding checks the dtype and size of
    # every tensor first: a short or mistyped buffer is rejected on the host
    # (these tensors live on the CPU; no call reaches the library or a device).
    import torch
    f16 = lambda *s: torch.zeros(*s, dtype=torch.float16)
    p = q.Pack(64, 128, 2, 32)
    x = f16(1, 128)
    cases = [
        (lambda: q.qmv_gemv(p, torch.zeros(1, 128)), "x: expected torch.float16"),
        (lambda: q.qmv_gemv(p, f16(1, 64)), "x: needs at least 128"),
        (lambda: q.qmv_gemv(p, x, y=torch.zeros(1, 32)), "y: needs at least 64"),
        (lambda: q.qmv_gemv(p, x, y=torch.zeros(1, 64), y_dtype=q.QMV_F16), "y: expected torch.float16"),
        (lambda: q.qmv_chunk_gemm(p, f16(4, 100)), "x: needs at least 512"),
        (lambda: q.qmv_fused_rmsnorm_gemv(p, f16(2, 128), f16(1, 128), f16(128)), "residual: needs at least 256"),
        (lambda: q.qmv_fused_rmsnorm_gemv(p, x, x, f16(64)), "gamma: needs at least 128"),
        (lambda: q.qmv_fused_rmsnorm_gemv(p, x, x, f16(128), h_out=f16(100)), "h_out: needs at least 128"),
        (lambda: q.qmv_gemv_gather(p, 16, torch.zeros(2, dtype=torch.int64), x), "expert_ids: expected torch.int32"),
        (lambda: q.qmv_gemv_gather(p, 16, torch.zeros(2, dtype=torch.int32), x, y=torch.zeros(31)),
         "y: needs at least 32"),
        (lambda: q.qmv_gemv_argmax(p, x, torch.zeros(8, dtype=torch.uint8)), "workspace: needs at least 16 bytes"),
        (lambda: q.qmv_gemv_argmax(p, x, torch.zeros(16, dtype=torch.uint8),
                                   index=torch.zeros(1, dtype=torch.int64)), "index: expected torch.int32"),
        (lambda: q.qmv_pack_weights(p, torch.zeros(64, 128, dtype=torch.int16), f16(64, 4),
                                    torch.zeros(512, dtype=torch.int32), f16(256)), "codes: expected torch.int8"),
        (lambda: q.qmv_pack_weights(p, torch.zeros(64, 128, dtype=torch.int8), f16(64, 4),
                                    torch.zeros(511, dtype=torch.int32), f16(256)), "d_codes: needs at least 2048 bytes"),
        (lambda: q.qmv_unpack_codes(p, out=torch.zeros(64, 127, dtype=torch.int8)), "out: needs at least 8192"),
    ]
    ch = q.Chain.__new__(q.Chain)          # no workspace: the checks come first
    ch.handle, ch._keep = None, []
    cases += [
        (lambda: ch.add_gemv(p, f16(1, 100), torch.zeros(1, 64)), "x: needs at least 128"),
        (lambda: ch.add_fused_rmsnorm_gemv(p, x, x, f16(128), 1e-6, None, f16(1, 64)), "y: expected torch.float32"),
    ]
    for call, msg in cases:
        with pytest.raises(ValueError, match=msg):
            call()
    # a well-formed call gets past the checks and stops at the device pointer
    with pytest.raises(ValueError, match="contiguous CUDA tensor"):
        q.qmv_gemv(p, x, y=torch.zeros(1, 64))


def test_header_is_plain_c_and_links(q, tmp_path):
    # A C99 program that includes only include/qmv.h, links libqmv.so and
    # uses the host-only entry points (no device is touched).
    import subprocess
    src = tmp_path / "abi_c.c"
    src.write_text(r'''
#include <stdio.h>
#include "qmv.h"
int main(void) {
    qmv_pack *p = NULL;
    size_t cb = 0, sb = 0;
    int N = 0, K = 0, bits = 0, group = 0;
    if (qmv_create_pack(&p, 48, 256, 4, 32, &cb, &sb) != QMV_OK) return 1;
    if (cb != 48 * 256 / 2 || sb != 48 * 8 * 2) return 2;
    if (qmv_pack_info(p, &N, &K, &bits, &group) != QMV_OK) return 3;
    if (N != 48 || K != 256 || bits != 4 || group != 32) return 4;
    if (qmv_gemv(p, 1, 48, 256, 4, 32, NULL, NULL, QMV_F32, QMV_FAST, NULL, 0, NULL) != QMV_ERR_INVALID_ARG) return 5;
    if (qmv_workspace_bytes(p, 1, QMV_F32, QMV_FAST, 1) != 0) return 7;
    if (qmv_workspace_bytes(p, 16, QMV_F32, QMV_EXACT, 1) != 4 * 8960 &&
        qmv_workspace_bytes(p, 16, QMV_F32, QMV_EXACT, 1) != 2 * 17408) return 8;
    if (qmv_workspace_bytes(p, 64, QMV_F16, QMV_FAST, 0) != 16 * 8960 &&
        qmv_workspace_bytes(p, 64, QMV_F16, QMV_FAST, 0) != 8 * 17408) return 9;
    if (qmv_destroy_pack(p) != QMV_OK) return 6;
    printf("%s\n", qmv_status_string(QMV_ERR_SHAPE));
    return 0;
}
''')
    exe = tmp_path / "abi_c"
    libdir = os.path.dirname(q.LIB_PATH)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), "-L", libdir, "-lqmv", f"-Wl,-rpath,{libdir}"],
                   check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stderr)
    assert r.stdout.strip() == q.qmv_status_string(q.QMV_ERR_SHAPE)


def test_binding_fails_loudly_without_the_library(tmp_path):
    # The binding module, copied where no _lib/libqmv.so sits beside it,
    # raises at import: there is no fallback of any kind.
    import importlib.util
    import shutil
    src = os.path.join(ROOT, "bit_weight_only_packed_gb300", "qmv.py")
    shutil.copy(src, tmp_path / "qmv_nolib.py")
    spec = importlib.util.spec_from_file_location("qmv_nolib", tmp_path / "qmv_nolib.py")
    mod = importlib.util.module_from_spec(spec)
    with pytest.raises(ImportError, match="libqmv.so is not built"):
        spec.loader.exec_module(mod)


def test_product_never_touches_the_oracle():
    # The library and its binding neither import nor load the oracle, the
    # generator or scratch files; the oracle is test infrastructure only.
    pkg = os.path.join(ROOT, "bit_weight_only_packed_gb300")
    bad = re.compile(r"\b(import\s+oracle|from\s+oracle|import\s+synth|from\s+synth|liboracle|_work)\b")
    for dirpath, _, files in os.walk(pkg):
        if "__pycache__" in dirpath or "_lib" in dirpath:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not bad.search(text), (f, bad.search(text).group(0))


def test_oracle_shares_no_code_with_the_library():
    # The oracle includes only the C standard headers and imports nothing of
    # the library; the two sides share only the input generator.
    c = open(os.path.join(ROOT, "oracle", "qmv_oracle.c")).read()
    assert sorted(set(re.findall(r'#include\s*[<"]([^>"]+)[>"]', c))) == ["math.h", "stdint.h", "string.h"]
    py = open(os.path.join(ROOT, "oracle", "__init__.py")).read()
    imports = re.findall(r"^\s*(?:from\s+(\S+)\s+import|import\s+(\S+))", py, re.M)
    mods = {a or b for a, b in imports}
    assert not {m for m in mods if m.split(".")[0] in ("bit_weight_only_packed_gb300", "synth", "bench")}, mods


def test_binding_signatures_match_the_header():
    # every ctypes signature has as many arguments as the C declaration, and
    # pointer parameters are passed as pointers (a mismatch would only show as
    # a corrupted call on a GPU)
    import ctypes
    from bit_weight_only_packed_gb300 import qmv as q
    txt = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    decls = re.findall(r"QMV_API\s+([\w\s\*]*?)\b(qmv_\w+)\s*\(([^)]*)\)\s*;", txt)
    assert len(decls) == len(q.SIGNATURES)
    for ret, name, params in decls:
        ps = [p.strip() for p in params.split(",") if p.strip() and p.strip() != "void"]
        restype, argtypes = q.SIGNATURES[name]
        ret = " ".join(ret.split())
        want_ret = {"int": ctypes.c_int, "size_t": ctypes.c_size_t, "const char *": ctypes.c_char_p}[ret]
        assert restype is want_ret, (name, ret, restype)
        assert len(ps) == len(argtypes), (name, ps, argtypes)
        for p, a in zip(ps, argtypes):
            if "*" in p:
                assert a is ctypes.c_void_p or issubclass(a, ctypes._Pointer), (name, p, a)
            elif p.split()[0] in ("int", "float", "size_t"):
                want = {"int": ctypes.c_int, "float": ctypes.c_float, "size_t": ctypes.c_size_t}[p.split()[0]]
                assert a is want, (name, p, a)
