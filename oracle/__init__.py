"""CPU oracle for the int4 weight-streaming GEMV (test infrastructure only).

This package is the plain, slow, obviously correct restatement of what the
GPU library computes.  Only the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg (and its ``--impl reference`` arm) may import it;
the product path never does, and it shares no code with the CUDA library.

The arithmetic lives in ``q4_oracle.c`` (plain C99, binary64 accumulation);
this module only compiles it with ``gcc`` and marshals numpy arrays into it.

Array conventions (all C-contiguous numpy arrays):

* ``codes``  uint8  [N, K/2]          two 4-bit codes per byte, even k low
* ``scales`` uint16 [N, K/g]          fp16 bit patterns
* ``zeros``  uint8  [N, ceil(K/g/2)]  two 4-bit zero points per byte, even
                                      group low; ``None`` = symmetric (8)
* ``x``      float32 [M, K];  ``a_bf16`` uint16 [M, K] (bfloat16 bits)
* results    float32 [M, N] plus the binary64 bound sum_k |w*x| [M, N]
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q4_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_q4.so")
# A test may point the wrapper at a separately compiled copy of the oracle
# (the planted-mistake tests compile altered copies to show the pins catch
# them); the environment variable names that shared object.
_LIB_OVERRIDE = os.environ.get("Q4_ORACLE_LIB")

# ISO C mode and -ffp-contract=off: the products and sums are rounded exactly
# as written (no fused multiply-add contraction on either host architecture).
_CFLAGS = ["-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared"]

_lock = threading.Lock()
_lib = None

_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_i64 = ctypes.c_int64


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile ``q4_oracle.c`` into ``liboracle_q4.so`` next to it."""
    stale = (not os.path.exists(out)
             or os.path.getmtime(out) < os.path.getmtime(src))
    if force or stale:
        tmp = out + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *_CFLAGS, src, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, out)
    return out


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            if _LIB_OVERRIDE:
                L = ctypes.CDLL(_LIB_OVERRIDE)
            else:
                build()
                L = ctypes.CDLL(_LIB_PATH)
            L.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
            L.orc_f16_to_f32.restype = ctypes.c_float
            L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
            L.orc_bf16_to_f32.restype = ctypes.c_float
            L.orc_f32_to_bf16.argtypes = [ctypes.c_float]
            L.orc_f32_to_bf16.restype = ctypes.c_uint16
            L.orc_q4_code.argtypes = [_u8p, _i64, _i64, _i64]
            L.orc_q4_code.restype = ctypes.c_int
            L.orc_q4_zero.argtypes = [_u8p, _i64, _i64, _i64]
            L.orc_q4_zero.restype = ctypes.c_int
            L.orc_q4_dequant.argtypes = [_u8p, _u16p, _u8p, _i64, _i64, _i64, _f32p]
            L.orc_q4_dequant.restype = None
            L.orc_q4_dequant_bf16.argtypes = [_u8p, _u16p, _u8p, _i64, _i64, _i64, _u16p]
            L.orc_q4_dequant_bf16.restype = None
            L.orc_q4_gemv.argtypes = [_u8p, _u16p, _u8p, _f32p, _i64, _i64, _i64,
                                      _i64, _f32p, _f64p]
            L.orc_q4_gemv.restype = None
            L.orc_q4_gemm.argtypes = [_u8p, _u16p, _u8p, _u16p, _i64, _i64, _i64,
                                      _i64, _f32p, _f64p]
            L.orc_q4_gemm.restype = None
            L.orc_f32_gemv.argtypes = [_f32p, _f32p, _i64, _i64, _i64, _f32p, _f64p]
            L.orc_f32_gemv.restype = None
            L.orc_sum_f32.argtypes = [_f32p, _i64]
            L.orc_sum_f32.restype = ctypes.c_double
            L.orc_rmsnorm.argtypes = [_f32p, _f32p, ctypes.c_double, _i64, _i64, _f64p]
            L.orc_rmsnorm.restype = None
            L.orc_q4_gemv_f64.argtypes = [_u8p, _u16p, _u8p, _f64p, _i64, _i64, _i64,
                                          _i64, _f64p, _f64p]
            L.orc_q4_gemv_f64.restype = None
            L.orc_silu.argtypes = [ctypes.c_double]
            L.orc_silu.restype = ctypes.c_double
            L.orc_swiglu.argtypes = [_f64p, _f64p, _i64, _f64p]
            L.orc_swiglu.restype = None
            L.orc_q40_weight.argtypes = [_u8p, _i64, _i64, _i64]
            L.orc_q40_weight.restype = ctypes.c_float
            L.orc_q40_gemv.argtypes = [_u8p, _f32p, _i64, _i64, _i64, _f32p, _f64p]
            L.orc_q40_gemv.restype = None
            L.orc_q80_weight.argtypes = [_u8p, _i64, _i64, _i64]
            L.orc_q80_weight.restype = ctypes.c_float
            L.orc_q80_gemv.argtypes = [_u8p, _f32p, _i64, _i64, _i64, _f32p, _f64p]
            L.orc_q80_gemv.restype = None
            _lib = L
        return _lib


# --------------------------------------------------------------------------
# marshalling helpers
# --------------------------------------------------------------------------

def _ptr(a, ctype, offset_elems: int = 0):
    if a is None:
        return ctypes.cast(None, ctype)
    assert a.flags.c_contiguous
    return ctypes.cast(a.ctypes.data + offset_elems * a.itemsize, ctype)


def _check_q4(codes, scales, zeros, K, g):
    N = codes.shape[0]
    nb = K // g
    assert codes.dtype == np.uint8 and codes.shape == (N, K // 2)
    assert scales.dtype == np.uint16 and scales.shape == (N, nb)
    if zeros is not None:
        assert zeros.dtype == np.uint8 and zeros.shape == (N, (nb + 1) // 2)
    return N, nb


def f16_to_f32(h: int) -> float:
    return lib().orc_f16_to_f32(int(h))


def bf16_to_f32(b: int) -> float:
    return lib().orc_bf16_to_f32(int(b))


def f32_to_bf16(f: float) -> int:
    return lib().orc_f32_to_bf16(ctypes.c_float(float(f)))


def q4_code(codes, K: int, n: int, k: int) -> int:
    return lib().orc_q4_code(_ptr(codes, _u8p), K, n, k)


def q4_dequant(codes, scales, zeros, K: int, g: int) -> np.ndarray:
    N, _ = _check_q4(codes, scales, zeros, K, g)
    w = np.empty((N, K), np.float32)
    lib().orc_q4_dequant(_ptr(codes, _u8p), _ptr(scales, _u16p), _ptr(zeros, _u8p),
                         N, K, g, _ptr(w, _f32p))
    return w


def q4_dequant_bf16(codes, scales, zeros, K: int, g: int) -> np.ndarray:
    N, _ = _check_q4(codes, scales, zeros, K, g)
    w = np.empty((N, K), np.uint16)
    lib().orc_q4_dequant_bf16(_ptr(codes, _u8p), _ptr(scales, _u16p), _ptr(zeros, _u8p),
                              N, K, g, _ptr(w, _u16p))
    return w


def q4_gemv(codes, scales, zeros, x, g: int):
    """y[M,N] (float32) and bound[M,N] (float64) for x[M,K] float32."""
    x = np.ascontiguousarray(x, np.float32)
    M, K = x.shape
    N, _ = _check_q4(codes, scales, zeros, K, g)
    y = np.empty((M, N), np.float32)
    b = np.empty((M, N), np.float64)
    lib().orc_q4_gemv(_ptr(codes, _u8p), _ptr(scales, _u16p), _ptr(zeros, _u8p),
                      _ptr(x, _f32p), M, N, K, g, _ptr(y, _f32p), _ptr(b, _f64p))
    return y, b


def q4_gemv_rows(codes, scales, zeros, x, g: int, rows):
    """The oracle on selected output rows only: y[M, len(rows)], bound."""
    x = np.ascontiguousarray(x, np.float32)
    M, K = x.shape
    N, nb = _check_q4(codes, scales, zeros, K, g)
    rows = [int(r) for r in rows]
    y = np.empty((M, len(rows)), np.float32)
    b = np.empty((M, len(rows)), np.float64)
    yr = np.empty((M, 1), np.float32)
    br = np.empty((M, 1), np.float64)
    zrow = (nb + 1) // 2
    for j, n in enumerate(rows):
        lib().orc_q4_gemv(_ptr(codes, _u8p, n * (K // 2)), _ptr(scales, _u16p, n * nb),
                          None if zeros is None else _ptr(zeros, _u8p, n * zrow),
                          _ptr(x, _f32p), M, 1, K, g, _ptr(yr, _f32p), _ptr(br, _f64p))
        y[:, j] = yr[:, 0]
        b[:, j] = br[:, 0]
    return y, b


def q4_gemv_threaded(codes, scales, zeros, x, g: int, threads: int):
    """The same oracle, run on `threads` contiguous row slices at once (the C
    routine is called unchanged on each slice; ctypes releases the GIL)."""
    x = np.ascontiguousarray(x, np.float32)
    M, K = x.shape
    N, nb = _check_q4(codes, scales, zeros, K, g)
    zrow = (nb + 1) // 2
    y = np.empty((M, N), np.float32)
    b = np.empty((M, N), np.float64)
    threads = max(1, min(threads, N))
    bounds = [N * t // threads for t in range(threads + 1)]
    parts = [(bounds[t], bounds[t + 1]) for t in range(threads)]
    outs = [(np.empty((M, n1 - n0), np.float32), np.empty((M, n1 - n0), np.float64))
            for n0, n1 in parts]
    L = lib()

    def run(t):
        n0, n1 = parts[t]
        L.orc_q4_gemv(_ptr(codes, _u8p, n0 * (K // 2)), _ptr(scales, _u16p, n0 * nb),
                      None if zeros is None else _ptr(zeros, _u8p, n0 * zrow),
                      _ptr(x, _f32p), M, n1 - n0, K, g,
                      _ptr(outs[t][0], _f32p), _ptr(outs[t][1], _f64p))

    ths = [threading.Thread(target=run, args=(t,)) for t in range(threads)]
    for th in ths:
        th.start()
    for th in ths:
        th.join()
    for (n0, n1), (yo, bo) in zip(parts, outs):
        y[:, n0:n1] = yo
        b[:, n0:n1] = bo
    return y, b


def q4_gemm(codes, scales, zeros, a_bf16, g: int):
    a_bf16 = np.ascontiguousarray(a_bf16, np.uint16)
    M, K = a_bf16.shape
    N, _ = _check_q4(codes, scales, zeros, K, g)
    c = np.empty((M, N), np.float32)
    b = np.empty((M, N), np.float64)
    lib().orc_q4_gemm(_ptr(codes, _u8p), _ptr(scales, _u16p), _ptr(zeros, _u8p),
                      _ptr(a_bf16, _u16p), M, N, K, g, _ptr(c, _f32p), _ptr(b, _f64p))
    return c, b


def q4_gemm_rows(codes, scales, zeros, a_bf16, g: int, m_rows, n_cols):
    """The oracle on a sample of output elements C[m, n] for m in m_rows and
    n in n_cols: returns c[len(m_rows), len(n_cols)] and the bound."""
    a_bf16 = np.ascontiguousarray(a_bf16, np.uint16)
    M, K = a_bf16.shape
    N, nb = _check_q4(codes, scales, zeros, K, g)
    zrow = (nb + 1) // 2
    c = np.empty((len(m_rows), len(n_cols)), np.float32)
    b = np.empty((len(m_rows), len(n_cols)), np.float64)
    cr = np.empty((1, 1), np.float32)
    br = np.empty((1, 1), np.float64)
    for i, m in enumerate(m_rows):
        for j, n in enumerate(n_cols):
            lib().orc_q4_gemm(_ptr(codes, _u8p, int(n) * (K // 2)),
                              _ptr(scales, _u16p, int(n) * nb),
                              None if zeros is None else _ptr(zeros, _u8p, int(n) * zrow),
                              _ptr(a_bf16, _u16p, int(m) * K), 1, 1, K, g,
                              _ptr(cr, _f32p), _ptr(br, _f64p))
            c[i, j] = cr[0, 0]
            b[i, j] = br[0, 0]
    return c, b


def f32_gemv(W, x):
    W = np.ascontiguousarray(W, np.float32)
    x = np.ascontiguousarray(x, np.float32)
    N, K = W.shape
    M = x.shape[0]
    assert x.shape == (M, K)
    y = np.empty((M, N), np.float32)
    b = np.empty((M, N), np.float64)
    lib().orc_f32_gemv(_ptr(W, _f32p), _ptr(x, _f32p), M, N, K, _ptr(y, _f32p),
                       _ptr(b, _f64p))
    return y, b


def f32_gemv_rows(W, x, rows):
    W = np.ascontiguousarray(W, np.float32)
    x = np.ascontiguousarray(x, np.float32)
    N, K = W.shape
    M = x.shape[0]
    y = np.empty((M, len(rows)), np.float32)
    b = np.empty((M, len(rows)), np.float64)
    yr = np.empty((M, 1), np.float32)
    br = np.empty((M, 1), np.float64)
    for j, n in enumerate(rows):
        lib().orc_f32_gemv(_ptr(W, _f32p, int(n) * K), _ptr(x, _f32p), M, 1, K,
                           _ptr(yr, _f32p), _ptr(br, _f64p))
        y[:, j] = yr[:, 0]
        b[:, j] = br[:, 0]
    return y, b


def sum_f32(buf) -> float:
    buf = np.ascontiguousarray(buf, np.float32).reshape(-1)
    return lib().orc_sum_f32(_ptr(buf, _f32p), buf.size)


# --------------------------------------------------------------------------
# the fused decode variants: RMSNorm prologue, SwiGLU epilogue
# --------------------------------------------------------------------------

SILU_SLOPE_MAX = 1.1   # |d silu / dv| <= 1.0998 for every real v


def rmsnorm(x, gamma, eps: float) -> np.ndarray:
    """binary64 [M, K]: x[m][k] / sqrt(mean_k x[m][k]^2 + eps) * gamma[k]."""
    x = np.ascontiguousarray(x, np.float32)
    gamma = np.ascontiguousarray(gamma, np.float32)
    M, K = x.shape
    assert gamma.shape == (K,)
    out = np.empty((M, K), np.float64)
    lib().orc_rmsnorm(_ptr(x, _f32p), _ptr(gamma, _f32p), float(eps), M, K, _ptr(out, _f64p))
    return out


def silu(v: float) -> float:
    return lib().orc_silu(float(v))


def swiglu(gate, up) -> np.ndarray:
    gate = np.ascontiguousarray(gate, np.float64)
    up = np.ascontiguousarray(up, np.float64)
    assert gate.shape == up.shape
    out = np.empty(gate.shape, np.float64)
    lib().orc_swiglu(_ptr(gate, _f64p), _ptr(up, _f64p), gate.size, _ptr(out, _f64p))
    return out


def _q4_gemv_f64_rows(codes, scales, zeros, xf, g: int, rows):
    M, K = xf.shape
    N, nb = _check_q4(codes, scales, zeros, K, g)
    zrow = (nb + 1) // 2
    y = np.empty((M, len(rows)), np.float64)
    b = np.empty((M, len(rows)), np.float64)
    yr = np.empty((M, 1), np.float64)
    br = np.empty((M, 1), np.float64)
    for j, n in enumerate(rows):
        lib().orc_q4_gemv_f64(_ptr(codes, _u8p, n * (K // 2)), _ptr(scales, _u16p, n * nb),
                              None if zeros is None else _ptr(zeros, _u8p, n * zrow),
                              _ptr(xf, _f64p), M, 1, K, g, _ptr(yr, _f64p), _ptr(br, _f64p))
        y[:, j] = yr[:, 0]
        b[:, j] = br[:, 0]
    return y, b


def q4_gemv_fused(codes, scales, zeros, x, gamma, eps: float, g: int, swiglu_epilogue: bool,
                  outputs=None):
    """The fused variant: y = W . RMSNorm(x) (or W . x when gamma is None), and with
    the SwiGLU epilogue h[m][i] = silu(y[m][2i]) * y[m][2i+1] (rows 2i, 2i+1 of W are
    the gate / up pair of output i).  `outputs` selects output columns (all when None).
    Returns the reference (binary64) and the tolerance bound per output:
      plain:  1e-3 * sum_k |w x'| + 1e-6, x' the (normalised) input, as for the GEMV;
      SwiGLU: with B_g, B_u those bounds of the pair,
              SILU_SLOPE_MAX * B_g * (|u| + B_u) + (|silu(g)| + SILU_SLOPE_MAX * B_g) * B_u
              + 2^-20 |h| + 1e-6
              (the first-order propagation of the pair's errors through silu(g) * u, and
              binary32 rounding of the combine)."""
    x = np.ascontiguousarray(x, np.float32)
    M, K = x.shape
    N, _ = _check_q4(codes, scales, zeros, K, g)
    if gamma is None:
        xf = x.astype(np.float64)
    else:
        xf = rmsnorm(x, gamma, eps)
    if not swiglu_epilogue:
        cols = list(range(N)) if outputs is None else [int(c) for c in outputs]
        y, mag = _q4_gemv_f64_rows(codes, scales, zeros, xf, g, cols)
        return y, 1e-3 * mag + 1e-6
    assert N % 2 == 0
    cols = list(range(N // 2)) if outputs is None else [int(c) for c in outputs]
    rows = []
    for i in cols:
        rows += [2 * i, 2 * i + 1]
    y, mag = _q4_gemv_f64_rows(codes, scales, zeros, xf, g, rows)
    gate, up = y[:, 0::2], y[:, 1::2]
    bg, bu = 1e-3 * mag[:, 0::2] + 1e-6, 1e-3 * mag[:, 1::2] + 1e-6
    h = swiglu(gate, up)
    sg = np.abs(swiglu(gate, np.ones_like(gate)))
    bound = (SILU_SLOPE_MAX * bg * (np.abs(up) + bu) + (sg + SILU_SLOPE_MAX * bg) * bu
             + 2.0 ** -20 * np.abs(h) + 1e-6)
    return h, bound


# --------------------------------------------------------------------------
# the second format: Q4_0 blocks (32 elements in 18 bytes)
# --------------------------------------------------------------------------

def q40_weight(blocks, K: int, n: int, k: int) -> float:
    blocks = np.ascontiguousarray(blocks, np.uint8)
    return lib().orc_q40_weight(_ptr(blocks, _u8p), K, n, k)


def q40_gemv(blocks, x):
    """y[M,N] (float32) and bound[M,N] (float64) for Q4_0 blocks uint8 [N, K/32, 18]."""
    x = np.ascontiguousarray(x, np.float32)
    M, K = x.shape
    blocks = np.ascontiguousarray(blocks, np.uint8)
    N = blocks.shape[0]
    assert blocks.shape == (N, K // 32, 18)
    y = np.empty((M, N), np.float32)
    b = np.empty((M, N), np.float64)
    lib().orc_q40_gemv(_ptr(blocks, _u8p), _ptr(x, _f32p), M, N, K, _ptr(y, _f32p), _ptr(b, _f64p))
    return y, b


def q40_gemv_rows(blocks, x, rows):
    """The Q4_0 oracle on selected output rows only."""
    x = np.ascontiguousarray(x, np.float32)
    M, K = x.shape
    blocks = np.ascontiguousarray(blocks, np.uint8)
    rows = [int(r) for r in rows]
    y = np.empty((M, len(rows)), np.float32)
    b = np.empty((M, len(rows)), np.float64)
    yr = np.empty((M, 1), np.float32)
    br = np.empty((M, 1), np.float64)
    row_bytes = (K // 32) * 18
    for j, n in enumerate(rows):
        lib().orc_q40_gemv(_ptr(blocks, _u8p, n * row_bytes), _ptr(x, _f32p), M, 1, K,
                           _ptr(yr, _f32p), _ptr(br, _f64p))
        y[:, j] = yr[:, 0]
        b[:, j] = br[:, 0]
    return y, b


# --------------------------------------------------------------------------
# the third format: Q8_0 blocks (32 elements in 34 bytes)
# --------------------------------------------------------------------------

def q80_weight(blocks, K: int, n: int, k: int) -> float:
    blocks = np.ascontiguousarray(blocks, np.uint8)
    return lib().orc_q80_weight(_ptr(blocks, _u8p), K, n, k)


def q80_gemv(blocks, x):
    """y[M,N] (float32) and bound[M,N] (float64) for Q8_0 blocks uint8 [N, K/32, 34]."""
    x = np.ascontiguousarray(x, np.float32)
    M, K = x.shape
    blocks = np.ascontiguousarray(blocks, np.uint8)
    N = blocks.shape[0]
    assert blocks.shape == (N, K // 32, 34)
    y = np.empty((M, N), np.float32)
    b = np.empty((M, N), np.float64)
    lib().orc_q80_gemv(_ptr(blocks, _u8p), _ptr(x, _f32p), M, N, K, _ptr(y, _f32p), _ptr(b, _f64p))
    return y, b


def q80_gemv_rows(blocks, x, rows):
    """The Q8_0 oracle on selected output rows only."""
    x = np.ascontiguousarray(x, np.float32)
    M, K = x.shape
    blocks = np.ascontiguousarray(blocks, np.uint8)
    rows = [int(r) for r in rows]
    y = np.empty((M, len(rows)), np.float32)
    b = np.empty((M, len(rows)), np.float64)
    yr = np.empty((M, 1), np.float32)
    br = np.empty((M, 1), np.float64)
    row_bytes = (K // 32) * 34
    for j, n in enumerate(rows):
        lib().orc_q80_gemv(_ptr(blocks, _u8p, n * row_bytes), _ptr(x, _f32p), M, 1, K,
                           _ptr(yr, _f32p), _ptr(br, _f64p))
        y[:, j] = yr[:, 0]
        b[:, j] = br[:, 0]
    return y, b
