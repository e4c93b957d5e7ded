"""Python binding of libq4gemv.so, the GB300 int4 weight-streaming GEMV library.

The functions here carry the C ABI's names (include/q4gemv.h) and only
marshal arguments: torch tensors (or raw integer device addresses) become
pointers, sizes are read off the tensors when not given, and the current
torch CUDA stream is passed unless another is named.  Every step of the
computation runs in the library's CUDA kernels; there is no fallback of any
kind -- if the shared library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

__all__ = [
    "Q4Error", "lib", "library_path", "exported_names",
    "q4gemv_pack_info", "q4gemv_run", "q4gemv_fused_run", "q4gemv_grouped_run", "q4_0_gemv_run", "q8_0_gemv_run",
    "q4gemm_run", "q4gemv_run_ex", "q4gemv_fused_run_ex", "q4gemv_grouped_run_ex", "q4gemm_run_ex",
    "f32gemv_run",
    "q4gemv_status_string", "q4gemv_last_cuda_error",
    "q4_dequant_f32_run", "q4_dequant_bf16_run", "vec4_read_probe_run",
    "q4gemv_device_status", "q4gemm_set_wait_timeout_ns", "q4gemv_set_overlapped_launch",
    "q4gemv_bounds_violations", "q4gemv_grouped_split",
    "Q4_OK", "Q4_ERR_INVALID_ARG", "Q4_ERR_UNSUPPORTED", "Q4_ERR_MISALIGNED",
    "Q4_ERR_CUDA", "Q4_ERR_TIMEOUT", "Q4_EPILOGUE_NONE", "Q4_EPILOGUE_SWIGLU",
    "Q4_RUN_OVERLAPPED", "Q4_RUN_EXACT_X", "Q4_RUN_WAIT_TIMEOUT",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
HEADER = os.path.join(_ROOT, "include", "q4gemv.h")

Q4_OK, Q4_ERR_INVALID_ARG, Q4_ERR_UNSUPPORTED, Q4_ERR_MISALIGNED, Q4_ERR_CUDA, Q4_ERR_TIMEOUT = range(6)
Q4_EPILOGUE_NONE, Q4_EPILOGUE_SWIGLU = 0, 1
Q4_RUN_OVERLAPPED, Q4_RUN_EXACT_X, Q4_RUN_WAIT_TIMEOUT = 0x1, 0x2, 0x4


def library_path() -> str:
    return os.path.join(_HERE, "libq4gemv.so")


class Q4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {q4gemv_status_string(status)} (status {status})"
        if status == Q4_ERR_CUDA:
            msg += f" [{q4gemv_last_cuda_error()}]"
        super().__init__(msg)


class _PackInfo(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int64), ("k", ctypes.c_int64), ("group", ctypes.c_int32),
                ("blocks_per_row", ctypes.c_int32), ("codes_row_bytes", ctypes.c_int64),
                ("codes_bytes", ctypes.c_int64), ("scales_row_bytes", ctypes.c_int64),
                ("scales_bytes", ctypes.c_int64), ("zeros_row_bytes", ctypes.c_int64),
                ("zeros_bytes", ctypes.c_int64), ("base_alignment", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class _RunOptions(ctypes.Structure):
    _fields_ = [("flags", ctypes.c_uint32), ("reserved", ctypes.c_uint32), ("wait_timeout_ns", ctypes.c_uint64)]


class _Segment(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales_f16", ctypes.c_void_p), ("zeros_u4_or_null", ctypes.c_void_p),
                ("x", ctypes.c_void_p), ("y", ctypes.c_void_p), ("N", ctypes.c_int64)]


_lock = threading.Lock()
_lib = None
_vp, _i32, _i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64


def lib() -> ctypes.CDLL:
    """Load libq4gemv.so (built by gemm_decode_gb300.build); raises if absent."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise OSError(f"{path} is missing: build it with "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(path)
            L.q4gemv_pack_info.argtypes = [_i64, _i64, _i32, ctypes.POINTER(_PackInfo)]
            L.q4gemv_run.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _i64, _i64, _i32, _vp]
            L.q4gemv_fused_run.argtypes = [_vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _i32, _i64, _i64,
                                           _i32, _i32, _vp]
            L.q4gemm_run.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _i64, _i64, _i32, _vp]
            _opt = ctypes.POINTER(_RunOptions)
            L.q4gemv_run_ex.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _i64, _i64, _i32, _opt, _vp]
            L.q4gemv_fused_run_ex.argtypes = [_vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _i32, _i64, _i64,
                                              _i32, _i32, _opt, _vp]
            L.q4gemv_grouped_run_ex.argtypes = [ctypes.POINTER(_Segment), _i32, _i64, _i32, _opt, _vp]
            L.q4gemm_run_ex.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _i64, _i64, _i32, _opt, _vp]
            L.q4_0_gemv_run.argtypes = [_vp, _vp, _vp, _i32, _i64, _i64, _vp]
            L.q8_0_gemv_run.argtypes = [_vp, _vp, _vp, _i32, _i64, _i64, _vp]
            L.q4gemv_grouped_run.argtypes = [ctypes.POINTER(_Segment), _i32, _i64, _i32, _vp]
            L.f32gemv_run.argtypes = [_vp, _vp, _vp, _i32, _i64, _i64, _vp]
            L.q4gemv_status_string.argtypes = [ctypes.c_int]
            L.q4gemv_status_string.restype = ctypes.c_char_p
            L.q4gemv_last_cuda_error.argtypes = []
            L.q4gemv_last_cuda_error.restype = ctypes.c_char_p
            L.q4_dequant_f32_run.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i32, _vp]
            L.q4_dequant_bf16_run.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i32, _vp]
            L.vec4_read_probe_run.argtypes = [_vp, _i64, _vp, _i32, ctypes.POINTER(_i32), _vp]
            L.q4gemv_device_status.argtypes = [_vp]
            L.q4gemm_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
            L.q4gemv_set_overlapped_launch.argtypes = [ctypes.c_int]
            L.q4gemv_bounds_violations.argtypes = [_vp]
            L.q4gemv_grouped_split.argtypes = [ctypes.POINTER(_i64), _i32, _i64, _i32, _i32,
                                               ctypes.POINTER(_i32), ctypes.POINTER(_i32)]
            for f in ("q4gemv_pack_info", "q4gemv_run", "q4gemv_fused_run", "q4gemv_grouped_run", "q4_0_gemv_run",
                      "q8_0_gemv_run",
                      "q4gemm_run", "f32gemv_run", "q4gemv_run_ex", "q4gemv_fused_run_ex", "q4gemv_grouped_run_ex",
                      "q4gemm_run_ex",
                      "q4_dequant_f32_run", "q4_dequant_bf16_run", "vec4_read_probe_run",
                      "q4gemv_device_status", "q4gemm_set_wait_timeout_ns",
                      "q4gemv_set_overlapped_launch", "q4gemv_bounds_violations", "q4gemv_grouped_split"):
                getattr(L, f).restype = ctypes.c_int
            _lib = L
        return _lib


def exported_names():
    """Function names declared in include/q4gemv.h."""
    text = open(HEADER).read()
    return re.findall(r"^Q4_API\s+[\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M)


# ------------------------------------------------------------------ marshalling

def _addr(t, name="argument", esize=0):
    """Address of an array argument: None and integer addresses pass through as given;
    a tensor must be contiguous (the library reads packed row-major arrays) and, where
    esize is set, hold elements of esize bytes.  Metadata checks only: where the memory
    lives and how large it is stay the caller's responsibility, as in the C ABI."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError(f"{name}: a contiguous tensor is required (got strides {tuple(t.stride())})")
    if esize and t.element_size() != esize:
        raise ValueError(f"{name}: {esize}-byte elements expected, got {t.dtype}")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(st: int, where: str):
    if st != Q4_OK:
        raise Q4Error(st, where)


def q4gemv_status_string(status: int) -> str:
    return lib().q4gemv_status_string(int(status)).decode()


def q4gemv_last_cuda_error() -> str:
    return lib().q4gemv_last_cuda_error().decode()


def q4gemv_pack_info(N: int, K: int, group: int) -> dict:
    info = _PackInfo()
    _check(lib().q4gemv_pack_info(N, K, group, ctypes.byref(info)), "q4gemv_pack_info")
    return {name: getattr(info, name) for name, _ in _PackInfo._fields_ if name != "reserved"}


def _mnk_q4(codes, x, M, N, K):
    if M is None:
        M = x.shape[0]
    if N is None:
        N = codes.shape[0]
    if K is None:
        K = x.shape[1]
    return int(M), int(N), int(K)


def q4gemv_run(codes, scales_f16, zeros_u4_or_null, x, y, M=None, N=None, K=None, group=32,
               stream=None, check=True) -> int:
    M, N, K = _mnk_q4(codes, x, M, N, K)
    st = lib().q4gemv_run(_addr(codes, "codes", 1), _addr(scales_f16, "scales_f16", 2),
                          _addr(zeros_u4_or_null, "zeros_u4_or_null", 1), _addr(x, "x", 4),
                          _addr(y, "y", 4), M, N, K, int(group), _stream(stream))
    if check:
        _check(st, "q4gemv_run")
    return st


def q4gemv_fused_run(codes, scales_f16, zeros_u4_or_null, x, gamma, eps, y, M=None, N=None, K=None, group=32,
                     epilogue=Q4_EPILOGUE_NONE, stream=None, check=True) -> int:
    M, N, K = _mnk_q4(codes, x, M, N, K)
    st = lib().q4gemv_fused_run(_addr(codes, "codes", 1), _addr(scales_f16, "scales_f16", 2),
                                _addr(zeros_u4_or_null, "zeros_u4_or_null", 1), _addr(x, "x", 4),
                                _addr(gamma, "gamma", 4), float(eps), _addr(y, "y", 4), M, N, K, int(group),
                                int(epilogue), _stream(stream))
    if check:
        _check(st, "q4gemv_fused_run")
    return st


def q4gemv_grouped_run(segments, K, group=32, stream=None, check=True) -> int:
    """segments: (codes, scales_f16, zeros_or_None, x, y[, N]) per matrix, M = 1 each;
    N defaults to codes.shape[0]."""
    arr = (_Segment * max(1, len(segments)))()
    for i, sg in enumerate(segments):
        codes, scales, zeros, x, y = sg[:5]
        N = int(sg[5]) if len(sg) > 5 else int(codes.shape[0])
        arr[i] = _Segment(_addr(codes, "codes", 1), _addr(scales, "scales_f16", 2), _addr(zeros, "zeros_u4_or_null", 1),
                          _addr(x, "x", 4), _addr(y, "y", 4), N)
    st = lib().q4gemv_grouped_run(arr, len(segments), int(K), int(group), _stream(stream))
    if check:
        _check(st, "q4gemv_grouped_run")
    return st


def _options(flags, wait_timeout_ns, reserved=0):
    """Per-call options of the *_ex entry points (None: a NULL pointer, the defaults)."""
    if flags is None and wait_timeout_ns is None and not reserved:
        return None
    f = int(flags or 0)
    if wait_timeout_ns is not None:
        f |= Q4_RUN_WAIT_TIMEOUT
    o = _RunOptions(f, int(reserved), int(wait_timeout_ns or 0))
    return ctypes.byref(o)


def q4gemv_run_ex(codes, scales_f16, zeros_u4_or_null, x, y, M=None, N=None, K=None, group=32,
                  flags=None, wait_timeout_ns=None, stream=None, check=True, _reserved=0) -> int:
    """q4gemv_run with per-call options: flags (Q4_RUN_*), and wait_timeout_ns, which sets
    Q4_RUN_WAIT_TIMEOUT when given."""
    M, N, K = _mnk_q4(codes, x, M, N, K)
    st = lib().q4gemv_run_ex(_addr(codes, "codes", 1), _addr(scales_f16, "scales_f16", 2),
                             _addr(zeros_u4_or_null, "zeros_u4_or_null", 1), _addr(x, "x", 4),
                             _addr(y, "y", 4), M, N, K, int(group), _options(flags, wait_timeout_ns, _reserved),
                             _stream(stream))
    if check:
        _check(st, "q4gemv_run_ex")
    return st


def q4gemv_fused_run_ex(codes, scales_f16, zeros_u4_or_null, x, gamma, eps, y, M=None, N=None, K=None, group=32,
                        epilogue=Q4_EPILOGUE_NONE, flags=None, wait_timeout_ns=None, stream=None, check=True) -> int:
    M, N, K = _mnk_q4(codes, x, M, N, K)
    st = lib().q4gemv_fused_run_ex(_addr(codes, "codes", 1), _addr(scales_f16, "scales_f16", 2),
                                   _addr(zeros_u4_or_null, "zeros_u4_or_null", 1), _addr(x, "x", 4),
                                   _addr(gamma, "gamma", 4), float(eps), _addr(y, "y", 4), M, N, K, int(group),
                                   int(epilogue), _options(flags, wait_timeout_ns), _stream(stream))
    if check:
        _check(st, "q4gemv_fused_run_ex")
    return st


def q4gemv_grouped_run_ex(segments, K, group=32, flags=None, wait_timeout_ns=None, stream=None, check=True) -> int:
    arr = (_Segment * max(1, len(segments)))()
    for i, sg in enumerate(segments):
        codes, scales, zeros, x, y = sg[:5]
        N = int(sg[5]) if len(sg) > 5 else int(codes.shape[0])
        arr[i] = _Segment(_addr(codes, "codes", 1), _addr(scales, "scales_f16", 2), _addr(zeros, "zeros_u4_or_null", 1),
                          _addr(x, "x", 4), _addr(y, "y", 4), N)
    st = lib().q4gemv_grouped_run_ex(arr, len(segments), int(K), int(group), _options(flags, wait_timeout_ns),
                                     _stream(stream))
    if check:
        _check(st, "q4gemv_grouped_run_ex")
    return st


def q4gemm_run_ex(codes, scales_f16, zeros_u4_or_null, a_bf16, c, M=None, N=None, K=None, group=32,
                  flags=None, wait_timeout_ns=None, stream=None, check=True) -> int:
    M, N, K = _mnk_q4(codes, a_bf16, M, N, K)
    st = lib().q4gemm_run_ex(_addr(codes, "codes", 1), _addr(scales_f16, "scales_f16", 2),
                             _addr(zeros_u4_or_null, "zeros_u4_or_null", 1), _addr(a_bf16, "a_bf16", 2),
                             _addr(c, "c", 4), M, N, K, int(group), _options(flags, wait_timeout_ns),
                             _stream(stream))
    if check:
        _check(st, "q4gemm_run_ex")
    return st


def q4_0_gemv_run(blocks, x, y, M=None, N=None, K=None, stream=None, check=True) -> int:
    M = int(x.shape[0] if M is None else M)
    K = int(x.shape[1] if K is None else K)
    N = int(blocks.shape[0] if N is None else N)
    st = lib().q4_0_gemv_run(_addr(blocks, "blocks", 1), _addr(x, "x", 4), _addr(y, "y", 4), M, N, K,
                             _stream(stream))
    if check:
        _check(st, "q4_0_gemv_run")
    return st


def q8_0_gemv_run(blocks, x, y, M=None, N=None, K=None, stream=None, check=True) -> int:
    M = int(x.shape[0] if M is None else M)
    K = int(x.shape[1] if K is None else K)
    N = int(blocks.shape[0] if N is None else N)
    st = lib().q8_0_gemv_run(_addr(blocks, "blocks", 1), _addr(x, "x", 4), _addr(y, "y", 4), M, N, K,
                             _stream(stream))
    if check:
        _check(st, "q8_0_gemv_run")
    return st


def q4gemm_run(codes, scales_f16, zeros_u4_or_null, a_bf16, c, M=None, N=None, K=None, group=32,
               stream=None, check=True) -> int:
    M, N, K = _mnk_q4(codes, a_bf16, M, N, K)
    st = lib().q4gemm_run(_addr(codes, "codes", 1), _addr(scales_f16, "scales_f16", 2),
                          _addr(zeros_u4_or_null, "zeros_u4_or_null", 1), _addr(a_bf16, "a_bf16", 2),
                          _addr(c, "c", 4), M, N, K, int(group), _stream(stream))
    if check:
        _check(st, "q4gemm_run")
    return st


def f32gemv_run(W, x, y, M=None, N=None, K=None, stream=None, check=True) -> int:
    M = int(x.shape[0] if M is None else M)
    N = int(W.shape[0] if N is None else N)
    K = int(W.shape[1] if K is None else K)
    st = lib().f32gemv_run(_addr(W, "W", 4), _addr(x, "x", 4), _addr(y, "y", 4), M, N, K, _stream(stream))
    if check:
        _check(st, "f32gemv_run")
    return st


def q4_dequant_f32_run(codes, scales_f16, zeros_u4_or_null, w, N=None, K=None, group=32,
                       stream=None, check=True) -> int:
    N = int(codes.shape[0] if N is None else N)
    K = int(codes.shape[1] * 2 if K is None else K)
    st = lib().q4_dequant_f32_run(_addr(codes, "codes", 1), _addr(scales_f16, "scales_f16", 2),
                                  _addr(zeros_u4_or_null, "zeros_u4_or_null", 1), _addr(w, "w", 4),
                                  N, K, int(group), _stream(stream))
    if check:
        _check(st, "q4_dequant_f32_run")
    return st


def q4_dequant_bf16_run(codes, scales_f16, zeros_u4_or_null, wb, N=None, K=None, group=32,
                        stream=None, check=True) -> int:
    N = int(codes.shape[0] if N is None else N)
    K = int(codes.shape[1] * 2 if K is None else K)
    st = lib().q4_dequant_bf16_run(_addr(codes, "codes", 1), _addr(scales_f16, "scales_f16", 2),
                                   _addr(zeros_u4_or_null, "zeros_u4_or_null", 1), _addr(wb, "wb", 2),
                                   N, K, int(group), _stream(stream))
    if check:
        _check(st, "q4_dequant_bf16_run")
    return st


def q4gemv_device_status(stream=None) -> int:
    """Synchronise the stream; Q4_OK or Q4_ERR_TIMEOUT (clears the flag)."""
    return lib().q4gemv_device_status(_stream(stream))


def q4gemm_set_wait_timeout_ns(ns: int) -> int:
    return lib().q4gemm_set_wait_timeout_ns(int(ns))


def q4gemv_bounds_violations(stream=None) -> int:
    """Out-of-range accesses counted since the last call (bounds-checking builds), -1
    in a library built without the checks."""
    return lib().q4gemv_bounds_violations(_stream(stream) if stream is not None else None)


def q4gemv_grouped_split(Ns, K, group, grid_max):
    """Host-only test export: (grid, nblocks per matrix, first CTA per matrix) of the CTA
    split a grouped launch makes; raises Q4Error on a negated status."""
    n = len(Ns)
    arr = (_i64 * max(1, n))(*[int(v) for v in Ns])
    nb = (_i32 * max(1, n))()
    cb = (_i32 * max(1, n))()
    grid = lib().q4gemv_grouped_split(arr, n, int(K), int(group), int(grid_max), nb, cb)
    if grid < 0:
        raise Q4Error(-grid, "q4gemv_grouped_split")
    return grid, list(nb[:n]), list(cb[:n])


def q4gemv_set_overlapped_launch(enable: bool) -> int:
    """Programmatic dependent launch for later q4gemv_run calls; returns the old setting."""
    return lib().q4gemv_set_overlapped_launch(1 if enable else 0)


def vec4_read_probe_run(buf, nbytes, partial, blocks=0, stream=None, check=True):
    used = _i32(0)
    st = lib().vec4_read_probe_run(_addr(buf, "buf"), int(nbytes), _addr(partial, "partial", 4), int(blocks),
                                   ctypes.byref(used), _stream(stream))
    if check:
        _check(st, "vec4_read_probe_run")
    return used.value
