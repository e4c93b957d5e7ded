"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module only draws random data in the storage layout the library reads;
it holds none of the method's arithmetic (no unpacking, no dequantisation, no
dot products).  Both sides -- the CUDA library and the CPU oracle -- receive
exactly these arrays.

Recipe (the decode-projection and prefill workloads of a 0.5B-class and an
8B-class transformer, synthetic stand-ins for model weights):

* codes:  4-bit values uniform on 0..15, two per byte, the even k in the low
          nibble.  Drawing whole bytes uniformly on 0..255 gives exactly
          that: both nibbles are independent and uniform.
* scales: binary32 uniform on [lo, hi], rounded to fp16 (nearest-even);
          [0.005, 0.02] for the 0.5B-class shapes, the prefill shapes and the
          sweep, [0.001, 0.01] for the 8B-class shapes.
* zeros:  4-bit values uniform on 0..15, two per byte (even group low); a
          row with an odd number of groups ends in a pad nibble written as 0.
          The symmetric variant has no zero-point array (zero = 8).
* x:      binary32 ~ N(0, 1).
* A:      N(0, 1) rounded to bfloat16 (nearest-even) for the matmul path.
* W:      binary32 ~ N(0, 0.02) (0.02 = standard deviation) for the dense
          f32 control.
"""
from __future__ import annotations

import zlib
from dataclasses import dataclass
from typing import Optional

import numpy as np

SCALE_05B = (0.005, 0.02)
SCALE_8B = (0.001, 0.01)


def _rng(seed: int, tag: str) -> np.random.Generator:
    return np.random.default_rng([int(seed) & 0xFFFFFFFF, zlib.crc32(tag.encode())])


@dataclass
class Q4Weights:
    codes: np.ndarray            # uint8  [N, K/2]
    scales: np.ndarray           # uint16 [N, K/g]   (fp16 bit patterns)
    zeros: Optional[np.ndarray]  # uint8  [N, ceil(K/g/2)] or None
    N: int
    K: int
    group: int

    @property
    def nbytes(self) -> int:
        z = 0 if self.zeros is None else self.zeros.nbytes
        return self.codes.nbytes + self.scales.nbytes + z


def q4_weights(seed: int, N: int, K: int, group: int, scale_range=SCALE_05B,
               symmetric: bool = False, tag: str = "w") -> Q4Weights:
    if K % group or K % 2:
        raise ValueError("K must be a multiple of the group size and even")
    nb = K // group
    r = _rng(seed, tag + ":codes")
    codes = np.frombuffer(r.bytes(N * (K // 2)), np.uint8).reshape(N, K // 2).copy()
    r = _rng(seed, tag + ":scales")
    lo, hi = scale_range
    scales = r.uniform(lo, hi, size=(N, nb)).astype(np.float32).astype(np.float16)
    scales = scales.view(np.uint16).copy()
    zeros = None
    if not symmetric:
        r = _rng(seed, tag + ":zeros")
        zb = (nb + 1) // 2
        zeros = np.frombuffer(r.bytes(N * zb), np.uint8).reshape(N, zb).copy()
        if nb % 2:
            zeros[:, -1] &= 0x0F
    return Q4Weights(codes, scales, zeros, N, K, group)


def q40_blocks(seed: int, N: int, K: int, scale_range=SCALE_05B, tag: str = "q40") -> np.ndarray:
    """Q4_0-format weights, uint8 [N, K/32, 18]: per block the binary16 scale bits
    (little-endian) from U[scale_range], then 16 bytes of uniform random codes."""
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    nblk = K // 32
    r = _rng(seed, tag + ":scales")
    lo, hi = scale_range
    d = r.uniform(lo, hi, size=(N, nblk)).astype(np.float32).astype(np.float16).view(np.uint16)
    r = _rng(seed, tag + ":codes")
    codes = np.frombuffer(r.bytes(N * nblk * 16), np.uint8).reshape(N, nblk, 16)
    out = np.empty((N, nblk, 18), np.uint8)
    out[:, :, 0] = (d & 0xFF).astype(np.uint8)
    out[:, :, 1] = (d >> 8).astype(np.uint8)
    out[:, :, 2:] = codes
    return out


# Q8_0 codes span -128..127, sixteen times the int4 span: scales a sixteenth of the
# 0.5B-class range keep the weights of the same magnitude.
SCALE_Q80 = (0.005 / 16, 0.02 / 16)


def q80_blocks(seed: int, N: int, K: int, scale_range=SCALE_Q80, tag: str = "q80") -> np.ndarray:
    """Q8_0-format weights, uint8 [N, K/32, 34]: per block the binary16 scale bits
    (little-endian) from U[scale_range], then 32 uniform random bytes (the codes,
    read as two's-complement int8)."""
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    nblk = K // 32
    r = _rng(seed, tag + ":scales")
    lo, hi = scale_range
    d = r.uniform(lo, hi, size=(N, nblk)).astype(np.float32).astype(np.float16).view(np.uint16)
    r = _rng(seed, tag + ":codes")
    codes = np.frombuffer(r.bytes(N * nblk * 32), np.uint8).reshape(N, nblk, 32)
    out = np.empty((N, nblk, 34), np.uint8)
    out[:, :, 0] = (d & 0xFF).astype(np.uint8)
    out[:, :, 1] = (d >> 8).astype(np.uint8)
    out[:, :, 2:] = codes
    return out


def activations_f32(seed: int, M: int, K: int, tag: str = "x") -> np.ndarray:
    return _rng(seed, tag).standard_normal((M, K), dtype=np.float32)


def activations_bf16(seed: int, M: int, K: int, tag: str = "a") -> np.ndarray:
    """N(0,1) rounded to bfloat16; returned as the uint16 bit patterns."""
    import torch
    x = _rng(seed, tag).standard_normal((M, K), dtype=np.float32)
    t = torch.from_numpy(x).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def dense_f32(seed: int, N: int, K: int, std: float = 0.02, tag: str = "W") -> np.ndarray:
    return (_rng(seed, tag).standard_normal((N, K), dtype=np.float32) * np.float32(std))


def uniform_f32(seed: int, n: int, tag: str = "buf") -> np.ndarray:
    """Small integers 0..7 as binary32, for the read probe (exact partial sums)."""
    r = _rng(seed, tag)
    return r.integers(0, 8, size=n, dtype=np.int32).astype(np.float32)


# --------------------------------------------------------------------------
# The workloads (shapes are (name, N, K); M and the group size per set).
# --------------------------------------------------------------------------

# Single GEMV, 896 x 896, group 32, plus the dense control of the same shape.
SINGLE_896 = dict(name="single_896", M=1, group=32, scale=SCALE_05B,
                  shapes=[("proj", 896, 896)])

# Decode projection set of a 0.5B-class transformer, M = 1, group 32.
DECODE_05B = dict(name="decode_0.5b", M=1, group=32, scale=SCALE_05B,
                  shapes=[("q_proj", 896, 896), ("k_proj", 128, 896),
                          ("v_proj", 128, 896), ("gate_proj", 4864, 896),
                          ("up_proj", 4864, 896), ("down_proj", 896, 4864),
                          ("lm_head", 151936, 896)])

# 8B-class decode shapes, group 128, M in {1, 2, 4, 8}.
DECODE_8B = dict(name="decode_8b", Ms=(1, 2, 4, 8), group=128, scale=SCALE_8B,
                 shapes=[("qo_proj", 4096, 4096), ("gate_up_proj", 14336, 4096),
                         ("down_proj", 4096, 14336), ("lm_head", 128256, 4096)])

# Prefill-shaped int4 matmul on the tensor cores, group 32: (name, M, N, K).
PREFILL = dict(name="prefill", group=32, scale=SCALE_05B,
               shapes=[("gate_128tok", 128, 512, 2048),
                       ("ffn_2048tok", 2048, 14336, 4096)])

# Sweep axes.
SWEEP = dict(Ms=(1, 16), Ks=(896, 2048, 4096, 8192, 16384),
             Ns=(512, 4096, 32768, 151936), groups=(32, 64, 128),
             symmetric=(True, False), scale=SCALE_05B)

