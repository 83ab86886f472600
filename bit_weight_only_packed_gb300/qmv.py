"""Thin ctypes binding of the C ABI in include/qmv.h (libqmv.so).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the ABI.  torch is used for device memory and streams.  If the
native library is missing the import of this module raises (there is no
fallback of any kind).
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libqmv.so")

QMV_OK = 0
QMV_ERR_INVALID_ARG = -1
QMV_ERR_UNSUPPORTED = -2
QMV_ERR_ALIGNMENT = -3
QMV_ERR_SHAPE = -4
QMV_ERR_CUDA = -5
QMV_ERR_TIMEOUT = -6
QMV_ERR_WORKSPACE = -7
QMV_F32, QMV_F16 = 0, 1
QMV_FAST, QMV_EXACT = 0, 1
QMV_PACK_HEADER_BYTES, QMV_PACK_VERSION = 64, 1

# every entry point declared in include/qmv.h, with its ctypes signature
_P, _I, _F, _SZP = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.POINTER(ctypes.c_size_t)
SIGNATURES = {
    "qmv_create_pack": (_I, [ctypes.POINTER(_P), _I, _I, _I, _I, _SZP, _SZP]),
    "qmv_pack_weights": (_I, [_P, _P, _P, _P, _P, _P]),
    "qmv_workspace_bytes": (ctypes.c_size_t, [_P, _I, _I, _I, _I]),
    "qmv_gemv": (_I, [_P, _I, _I, _I, _I, _I, _P, _P, _I, _I, _P, ctypes.c_size_t, _P]),
    "qmv_fused_rmsnorm_gemv": (_I, [_P, _I, _P, _P, _P, _F, _P, _P, _I, _I, _P, ctypes.c_size_t, _P]),
    "qmv_chunk_gemm": (_I, [_P, _I, _P, _P, _I, _I, _P, ctypes.c_size_t, _P]),
    "qmv_unpack_codes": (_I, [_P, _P, _P]),
    "qmv_pack_info": (_I, [_P, ctypes.POINTER(_I), ctypes.POINTER(_I), ctypes.POINTER(_I),
                           ctypes.POINTER(_I)]),
    "qmv_destroy_pack": (_I, [_P]),
    "qmv_pack_header": (_I, [_P, _P]),
    "qmv_create_pack_from_header": (_I, [ctypes.POINTER(_P), _P, _SZP, _SZP]),
    "qmv_bind_packed": (_I, [_P, _P, _P]),
    "qmv_status_string": (ctypes.c_char_p, [_I]),
    "qmv_last_cuda_error": (_I, []),
    "qmv_device_error": (_I, [ctypes.POINTER(_I), _I]),
    "qmv_set_pdl": (_I, [_I]),
    "qmv_gemv_gather": (_I, [_P, _I, _P, _I, _P, _P, _I, _I, _P]),
    "qmv_argmax_workspace_bytes": (ctypes.c_size_t, []),
    "qmv_gemv_argmax": (_I, [_P, _P, _P, _P, _F, _P, _P, _I, _I, _P, _P, _P, _P]),
    "qmv_chain_workspace_bytes": (ctypes.c_size_t, [_I]),
    "qmv_chain_create": (_I, [ctypes.POINTER(_P), _I, _P, ctypes.c_size_t]),
    "qmv_chain_create_no_alloc": (_I, [ctypes.POINTER(_P), _I]),
    "qmv_chain_add_gemv": (_I, [_P, _P, _P, _P, _I, _I]),
    "qmv_chain_add_fused_rmsnorm_gemv": (_I, [_P, _P, _P, _P, _P, _F, _P, _P, _I, _I]),
    "qmv_chain_run": (_I, [_P, _P]),
    "qmv_chain_info": (_I, [_P, ctypes.POINTER(_I), ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "qmv_chain_destroy": (_I, [_P]),
}


class QmvError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = _lib.qmv_status_string(status).decode()
        if status == QMV_ERR_CUDA:
            msg += f" (cudaError {_lib.qmv_last_cuda_error()})"
        super().__init__(f"{fn}: {msg} [{status}]")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libqmv.so is not built ({LIB_PATH}); run "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


_lib = _load()


def lib() -> ctypes.CDLL:
    return _lib


def _check(fn: str, rc: int):
    if rc != QMV_OK:
        raise QmvError(fn, rc)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dptr(t):
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("expected a contiguous CUDA tensor")
    return t.data_ptr()


_YDT = {QMV_F32: torch.float32, QMV_F16: torch.float16}


def _need(name, t, dtype, n):
    """The tensor behind a pointer argument has the dtype the kernels read or
    write and at least the n elements they touch from its start.  The ABI
    takes bare pointers and cannot check sizes, so this is checked here,
    before any call.  A y_dtype outside QMV_F32/QMV_F16 skips the dtype
    check; the ABI rejects that value itself."""
    if t is None:
        return
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name}: expected {dtype}, got {t.dtype}")
    if t.numel() < n:
        raise ValueError(f"{name}: needs at least {n} elements, has {t.numel()}")


def _need_bytes(name, t, n):
    if t.numel() * t.element_size() < n:
        raise ValueError(f"{name}: needs at least {n} bytes, has {t.numel() * t.element_size()}")


class Pack:
    """A packed weight matrix: the host descriptor plus the device buffers
    (allocated with torch) that hold the packed codes and scales."""

    def __init__(self, N: int, K: int, bits: int, group: int, header: bytes = None):
        h = _P()
        cb, sb = ctypes.c_size_t(), ctypes.c_size_t()
        if header is None:
            _check("qmv_create_pack", _lib.qmv_create_pack(ctypes.byref(h), N, K, bits, group,
                                                            ctypes.byref(cb), ctypes.byref(sb)))
        else:
            if len(header) != QMV_PACK_HEADER_BYTES:
                raise ValueError(f"a pack header is {QMV_PACK_HEADER_BYTES} bytes, got {len(header)}")
            buf = ctypes.create_string_buffer(bytes(header), QMV_PACK_HEADER_BYTES)
            _check("qmv_create_pack_from_header", _lib.qmv_create_pack_from_header(
                ctypes.byref(h), buf, ctypes.byref(cb), ctypes.byref(sb)))
        self.handle = h
        if header is not None:
            n, k, b, g = _I(), _I(), _I(), _I()
            _check("qmv_pack_info", _lib.qmv_pack_info(h, ctypes.byref(n), ctypes.byref(k), ctypes.byref(b),
                                                       ctypes.byref(g)))
            N, K, bits, group = n.value, k.value, b.value, g.value
        self.N, self.K, self.bits, self.group = N, K, bits, group
        self.codes_bytes, self.scales_bytes = cb.value, sb.value
        self.words = None
        self.scales = None

    @classmethod
    def from_header(cls, header: bytes) -> "Pack":
        """The pack described by a saved header (qmv_create_pack_from_header);
        bind its reloaded buffers with bind_packed."""
        return cls(0, 0, 0, 0, header=header)

    def header(self) -> bytes:
        return qmv_pack_header(self)

    def bind_packed(self, words: torch.Tensor, scales: torch.Tensor):
        """words, scales: device buffers holding the packed words and scales of
        this shape (as pack_weights left them, e.g. reloaded from a file)."""
        qmv_bind_packed(self, words, scales)
        self.words, self.scales = words, scales
        return self

    @property
    def packed_bytes(self) -> int:
        return self.codes_bytes + self.scales_bytes

    def pack_weights(self, codes: torch.Tensor, scales: torch.Tensor, stream=None, device=None):
        """codes: device int8 [N, K] signed codes; scales: device fp16 [N, K/group]."""
        dev = codes.device if device is None else device
        self.words = torch.empty(self.codes_bytes // 4, dtype=torch.int32, device=dev)
        self.scales = torch.empty(self.scales_bytes // 2, dtype=torch.float16, device=dev)
        qmv_pack_weights(self, codes, scales, self.words, self.scales, stream)
        return self

    def close(self):
        if self.handle is not None and self.handle.value:
            _lib.qmv_destroy_pack(self.handle)
        self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def qmv_create_pack(N: int, K: int, bits: int, group: int) -> Pack:
    return Pack(N, K, bits, group)


def qmv_pack_weights(p: Pack, codes, scales, d_codes, d_scales, stream=None):
    G = p.K // p.group
    _need("codes", codes, torch.int8, p.N * p.K)
    _need("scales", scales, torch.float16, p.N * G)
    _need_bytes("d_codes", d_codes, p.codes_bytes)
    _need_bytes("d_scales", d_scales, p.scales_bytes)
    _check("qmv_pack_weights", _lib.qmv_pack_weights(
        p.handle, _dptr(codes), _dptr(scales), _dptr(d_codes), _dptr(d_scales), _stream(stream)))


def _out(y, M, N, y_dtype, like):
    if y is None:
        dt = torch.float16 if y_dtype == QMV_F16 else torch.float32
        y = torch.empty((M, N), dtype=dt, device=like.device)
    return y


def qmv_workspace_bytes(p: Pack, M: int, y_dtype=QMV_F32, mode=QMV_FAST, fused=False) -> int:
    """Device scratch bytes a call needs (0 for none)."""
    return int(_lib.qmv_workspace_bytes(p.handle, M, y_dtype, mode, 1 if fused else 0))


def workspace(p: Pack, M: int, y_dtype=QMV_F32, mode=QMV_FAST, fused=False, device=None):
    """A workspace tensor for such calls (None when they need none)."""
    n = qmv_workspace_bytes(p, M, y_dtype, mode, fused)
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda") if n else None


def _ws(p, M, y_dtype, mode, fused, ws, like, stream=None):
    """The caller's workspace, checked, or (when none is given) a fresh torch
    allocation of the size the call needs: (pointer, bytes, tensor).  A fresh
    one used on another stream than torch's current one is recorded on that
    stream, so the allocator does not hand it out again before the call ends."""
    n = qmv_workspace_bytes(p, M, y_dtype, mode, fused)
    if ws is None:
        if n == 0:
            return None, 0, None
        ws = torch.empty(n, dtype=torch.uint8, device=like.device)
        if stream is not None:
            cur = torch.cuda.current_stream(like.device)
            if _stream(stream) != cur.cuda_stream:
                ts = stream if isinstance(stream, torch.cuda.Stream) else torch.cuda.ExternalStream(
                    int(stream), device=like.device)
                ws.record_stream(ts)
    _need_bytes("workspace", ws, n)
    return _dptr(ws), ws.numel() * ws.element_size(), ws


def qmv_gemv(p: Pack, x, y=None, y_dtype=QMV_F32, mode=QMV_FAST, stream=None, M=None, workspace=None):
    M = x.shape[0] if (M is None and x.dim() == 2) else (M or 1)
    _need("x", x, torch.float16, M * p.K)
    _need("y", y, _YDT.get(y_dtype), M * p.N)
    y = _out(y, M, p.N, y_dtype, x)
    wp, wb, _keep = _ws(p, M, y_dtype, mode, False, workspace, x, stream)
    _check("qmv_gemv", _lib.qmv_gemv(p.handle, M, p.N, p.K, p.bits, p.group, _dptr(x), _dptr(y),
                                     y_dtype, mode, wp, wb, _stream(stream)))
    return y


def qmv_chunk_gemm(p: Pack, x, y=None, y_dtype=QMV_F32, mode=QMV_FAST, stream=None, workspace=None):
    M = x.shape[0]
    _need("x", x, torch.float16, M * p.K)
    _need("y", y, _YDT.get(y_dtype), M * p.N)
    y = _out(y, M, p.N, y_dtype, x)
    wp, wb, _keep = _ws(p, M, y_dtype, mode, False, workspace, x, stream)
    _check("qmv_chunk_gemm", _lib.qmv_chunk_gemm(p.handle, M, _dptr(x), _dptr(y), y_dtype, mode,
                                                 wp, wb, _stream(stream)))
    return y


def qmv_fused_rmsnorm_gemv(p: Pack, x, residual, gamma, eps=1e-6, h_out=None, y=None,
                           y_dtype=QMV_F32, mode=QMV_FAST, stream=None, workspace=None):
    M = x.shape[0] if x.dim() == 2 else 1
    _need("x", x, torch.float16, M * p.K)
    _need("residual", residual, torch.float16, M * p.K)
    _need("gamma", gamma, torch.float16, p.K)
    _need("h_out", h_out, torch.float16, M * p.K)
    _need("y", y, _YDT.get(y_dtype), M * p.N)
    y = _out(y, M, p.N, y_dtype, x)
    wp, wb, _keep = _ws(p, M, y_dtype, mode, True, workspace, x, stream)
    _check("qmv_fused_rmsnorm_gemv", _lib.qmv_fused_rmsnorm_gemv(
        p.handle, M, _dptr(x), _dptr(residual), _dptr(gamma), float(eps), _dptr(h_out), _dptr(y),
        y_dtype, mode, wp, wb, _stream(stream)))
    return y


def qmv_gemv_gather(p: Pack, rows_per_expert: int, expert_ids, x, y=None, y_dtype=QMV_F32,
                    mode=QMV_FAST, stream=None):
    """y [1, n_selected * rows_per_expert]: the selected experts' rows times x."""
    n = expert_ids.numel()
    _need("expert_ids", expert_ids, torch.int32, n)
    _need("x", x, torch.float16, p.K)
    _need("y", y, _YDT.get(y_dtype), n * rows_per_expert)
    y = _out(y, 1, n * rows_per_expert, y_dtype, x)
    _check("qmv_gemv_gather", _lib.qmv_gemv_gather(p.handle, rows_per_expert, _dptr(expert_ids), n,
                                                   _dptr(x), _dptr(y), y_dtype, mode, _stream(stream)))
    return y


def qmv_argmax_workspace(device=None):
    """A zeroed workspace for qmv_gemv_argmax (left zero by every completed call)."""
    return torch.zeros(_lib.qmv_argmax_workspace_bytes(), dtype=torch.uint8, device=device or "cuda")


def qmv_gemv_argmax(p: Pack, x, workspace, residual=None, gamma=None, eps=1e-6, h_out=None, y=None,
                    y_dtype=QMV_F32, mode=QMV_FAST, stream=None, index=None, value=None):
    """(index, value) device tensors of the greedy token; y (logits) is stored
    only if given."""
    _need("x", x, torch.float16, p.K)
    _need("residual", residual, torch.float16, p.K)
    _need("gamma", gamma, torch.float16, p.K)
    _need("h_out", h_out, torch.float16, p.K)
    _need("y", y, _YDT.get(y_dtype), p.N)
    _need("index", index, torch.int32, 1)
    _need("value", value, torch.float32, 1)
    _need_bytes("workspace", workspace, _lib.qmv_argmax_workspace_bytes())
    if index is None:
        index = torch.empty(1, dtype=torch.int32, device=x.device)
    if value is None:
        value = torch.empty(1, dtype=torch.float32, device=x.device)
    _check("qmv_gemv_argmax", _lib.qmv_gemv_argmax(
        p.handle, _dptr(x), _dptr(residual), _dptr(gamma), float(eps), _dptr(h_out), _dptr(y), y_dtype,
        mode, _dptr(index), _dptr(value), _dptr(workspace), _stream(stream)))
    return index, value


def qmv_unpack_codes(p: Pack, out=None, stream=None):
    if out is None:
        out = torch.empty((p.N, p.K), dtype=torch.int8, device=p.words.device)
    _need("out", out, torch.int8, p.N * p.K)
    _check("qmv_unpack_codes", _lib.qmv_unpack_codes(p.handle, _dptr(out), _stream(stream)))
    return out


def qmv_pack_info(p: Pack):
    n, k, b, g = _I(), _I(), _I(), _I()
    _check("qmv_pack_info", _lib.qmv_pack_info(p.handle, ctypes.byref(n), ctypes.byref(k),
                                               ctypes.byref(b), ctypes.byref(g)))
    return n.value, k.value, b.value, g.value


def qmv_pack_header(p: Pack) -> bytes:
    buf = ctypes.create_string_buffer(QMV_PACK_HEADER_BYTES)
    _check("qmv_pack_header", _lib.qmv_pack_header(p.handle, buf))
    return buf.raw


def qmv_create_pack_from_header(header: bytes) -> Pack:
    return Pack.from_header(header)


def qmv_bind_packed(p: Pack, d_codes, d_scales):
    _need_bytes("d_codes", d_codes, p.codes_bytes)
    _need_bytes("d_scales", d_scales, p.scales_bytes)
    _check("qmv_bind_packed", _lib.qmv_bind_packed(p.handle, _dptr(d_codes), _dptr(d_scales)))


def qmv_status_string(status: int) -> str:
    return _lib.qmv_status_string(status).decode()


def qmv_last_cuda_error() -> int:
    return _lib.qmv_last_cuda_error()


def qmv_set_pdl(enable: bool):
    _check("qmv_set_pdl", _lib.qmv_set_pdl(1 if enable else 0))


def qmv_device_error(clear: bool = True) -> int:
    v = _I()
    _check("qmv_device_error", _lib.qmv_device_error(ctypes.byref(v), 1 if clear else 0))
    return v.value


class Chain:
    """A chain of M = 1 matvecs run by one persistent launch (qmv_chain_*).
    The workspace is a torch uint8 device tensor; the tensors of every added
    op are kept referenced for the chain's lifetime."""

    def __init__(self, max_ops: int, device=None, no_alloc: bool = False):
        """no_alloc: use the library's own scratch array (qmv_chain_create_no_alloc)
        instead of a workspace tensor."""
        h = _P()
        if no_alloc:
            self.ws = None
            _check("qmv_chain_create_no_alloc", _lib.qmv_chain_create_no_alloc(ctypes.byref(h), max_ops))
        else:
            n = _lib.qmv_chain_workspace_bytes(max_ops)
            self.ws = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
            _check("qmv_chain_create", _lib.qmv_chain_create(ctypes.byref(h), max_ops, _dptr(self.ws), n))
        self.handle = h
        self._keep = []

    def add_gemv(self, p: Pack, x, y, y_dtype=QMV_F32, mode=QMV_FAST):
        _need("x", x, torch.float16, p.K)
        _need("y", y, _YDT.get(y_dtype), p.N)
        _check("qmv_chain_add_gemv", _lib.qmv_chain_add_gemv(self.handle, p.handle, _dptr(x), _dptr(y),
                                                             y_dtype, mode))
        self._keep += [p, x, y]
        return self

    def add_fused_rmsnorm_gemv(self, p: Pack, x, residual, gamma, eps, h_out, y, y_dtype=QMV_F32,
                               mode=QMV_FAST):
        _need("x", x, torch.float16, p.K)
        _need("residual", residual, torch.float16, p.K)
        _need("gamma", gamma, torch.float16, p.K)
        _need("h_out", h_out, torch.float16, p.K)
        _need("y", y, _YDT.get(y_dtype), p.N)
        _check("qmv_chain_add_fused_rmsnorm_gemv", _lib.qmv_chain_add_fused_rmsnorm_gemv(
            self.handle, p.handle, _dptr(x), _dptr(residual), _dptr(gamma), float(eps), _dptr(h_out),
            _dptr(y), y_dtype, mode))
        self._keep += [p, x, residual, gamma, h_out, y]
        return self

    def run(self, stream=None):
        _check("qmv_chain_run", _lib.qmv_chain_run(self.handle, _stream(stream)))

    def info(self):
        n, b, sm = _I(), _I(), _I()
        _check("qmv_chain_info", _lib.qmv_chain_info(self.handle, ctypes.byref(n), ctypes.byref(b),
                                                     ctypes.byref(sm)))
        return {"ops": n.value, "barriers": b.value, "smem": sm.value}

    def close(self):
        if self.handle is not None and self.handle.value:
            _lib.qmv_chain_destroy(self.handle)
        self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
