"""GPU parity of the Q8_0 GEMV (q8_0_gemv_run: 32-element blocks of 34 bytes, int8 codes
and a binary16 scale) against the CPU oracle, within the GEMV tolerance
1e-3 * sum_k |w x| + 1e-6: the CUDA-core kernel (every M, short matrices) and the
streamed kernel's Q8_0 instances (M = 1 on long matrices: ragged last blocks of rows,
runtime geometries).  Marked gpu.
"""
import os

import numpy as np
import pytest

import gemm_decode_gb300 as q4
import oracle
import synth
from gpu_util import assert_within_bound, dev, host, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    t = torch_cuda()
    q4.lib()
    return t


def run(torch, blocks, x):
    M, K = x.shape
    N = blocks.shape[0]
    guard = 64
    buf = torch.full((M * N + 2 * guard,), 12345.0, dtype=torch.float32, device="cuda")
    y = buf[guard:guard + M * N]
    q4.q8_0_gemv_run(dev(blocks, torch), dev(x, torch), y, M, N, K)
    torch.cuda.synchronize()
    b = host(buf)
    assert np.all(b[:guard] == 12345.0) and np.all(b[guard + M * N:] == 12345.0), "guard words written"
    return b[guard:guard + M * N].reshape(M, N)


# On 152 SMs these reach every plan of the CUDA-core kernel (a warp takes 8 blocks of each
# of its rows per step): 4 weight rows per warp (M <= 4) with the blocks unsplit
# (40003 x 896; 20001 x 608, whose 19 blocks leave a partial last step) or split over 4 or
# 8 warps (4864 x 896, 4096 x 4096); 2 rows per warp (M > 4) split over 2 or 4 warps
# (9001 x 864 at M = 16, 27 blocks; 4099 x 1056, 33 blocks); one row per warp unsplit
# (77 x 32, 1 x 64) or split over 2, 4 or 8 warps (3001 x 608, 2051 x 4096, 896 x 4864,
# 512 x 2048 at M = 16); ragged last CTAs, a single block per row (K = 32: the lanes past
# it idle) and single rows.
@pytest.mark.parametrize("M,N,K", [(1, 896, 896), (2, 4864, 896), (1, 896, 4864), (3, 1000, 2048), (4, 4096, 4096),
                                   (8, 300, 16384), (16, 512, 2048), (5, 77, 32), (1, 1, 64), (2, 33, 4864),
                                   (4, 40003, 896), (3, 20001, 608), (16, 9001, 864), (2, 2051, 4096),
                                   (1, 3001, 608), (7, 4099, 1056)])
def test_cuda_core_kernel_against_oracle(torch, M, N, K):
    blocks = synth.q80_blocks(M + N + K, N, K)
    x = synth.activations_f32(M * N + K, M, K)
    y = run(torch, blocks, x)
    y_ref, bound = oracle.q80_gemv(blocks, x)
    assert_within_bound(y, y_ref, bound, f"Q8_0 M={M} N={N} K={K}")


@pytest.mark.parametrize("N,K", [(9765, 896), (8195, 2048), (4901, 4096), (4101, 14336), (4099, 16384), (40003, 608)])
def test_streamed_kernel(torch, N, K):
    # M = 1 on long matrices: the streamed kernel's Q8_0 instances (a block of rows is one
    # stretch of 34-byte blocks; 9765 x 896: a last block of 21 rows); 14336 and 608 take
    # the runtime geometry, 608 with 19 chunks per row.  Every row against the oracle.
    blocks = synth.q80_blocks(N + K, N, K)
    x = synth.activations_f32(N - K, 1, K)
    y = run(torch, blocks, x)
    y_ref, bound = _rows_threaded(blocks, x)
    assert_within_bound(y, y_ref, bound, f"Q8_0 streamed N={N} K={K}")


def _rows_threaded(blocks, x):
    """The oracle on every row, over the host cores in contiguous row slices."""
    from concurrent.futures import ThreadPoolExecutor
    N = blocks.shape[0]
    cuts = np.linspace(0, N, (os.cpu_count() or 1) + 1).astype(int)
    with ThreadPoolExecutor(max_workers=len(cuts) - 1) as ex:
        parts = list(ex.map(lambda i: oracle.q80_gemv(np.ascontiguousarray(blocks[cuts[i]:cuts[i + 1]]), x),
                            range(len(cuts) - 1)))
    return np.concatenate([p[0] for p in parts], axis=1), np.concatenate([p[1] for p in parts], axis=1)


def test_lm_head(torch):
    N, K = 151936, 896
    blocks = synth.q80_blocks(7, N, K)
    x = synth.activations_f32(8, 1, K)
    y = run(torch, blocks, x)
    y_ref, bound = _rows_threaded(blocks, x)
    r = assert_within_bound(y, y_ref, bound, "Q8_0 LM head")
    assert r < 0.05, r   # N(0, 1) activations: far inside the tolerance


@pytest.mark.parametrize("M,N,K", [(4, 128256, 4096), (2, 128256, 4096), (16, 151936, 896), (8, 14336, 4096)])
def test_cuda_core_kernel_full_size_sampled(torch, M, N, K):
    # the decode shapes at M > 1 (the CUDA-core kernel): every output finite, 257 rows
    # (both ends, random ones in between) against the oracle
    blocks = synth.q80_blocks(M + 31, N, K)
    x = synth.activations_f32(M + 37, M, K)
    y = run(torch, blocks, x)
    assert np.all(np.isfinite(y)), f"{int(np.sum(~np.isfinite(y)))} outputs not finite"
    rows = np.unique(np.concatenate([[0, 1, N - 2, N - 1],
                                     np.random.default_rng(N + M).choice(N, size=253, replace=False)]))
    y_ref, bound = oracle.q80_gemv(np.ascontiguousarray(blocks[rows]), x)
    assert_within_bound(y[:, rows], y_ref, bound, f"Q8_0 full size M={M} N={N} K={K}")


def test_matches_q4_0_on_the_int4_range(torch):
    # codes -8..7 as Q8_0 are the Q4_0 weights of codes 0..15 with the same scales: the two
    # entry points agree within the tolerance of the one oracle
    N, K = 4864, 896
    q40 = synth.q40_blocks(9, N, K)
    codes4 = np.empty((N, K // 32, 32), np.int16)
    codes4[:, :, 0::2] = q40[:, :, 2:] & 0xF
    codes4[:, :, 1::2] = q40[:, :, 2:] >> 4
    q80 = np.empty((N, K // 32, 34), np.uint8)
    q80[:, :, :2] = q40[:, :, :2]
    q80[:, :, 2:] = (codes4 - 8).astype(np.int8).view(np.uint8)
    for M in (1, 3):
        x = synth.activations_f32(10 + M, M, K)
        y_ref, bound = oracle.q40_gemv(q40, x)
        assert_within_bound(run(torch, q80, x), y_ref, bound, f"Q8_0 of the Q4_0 weights M={M}")


def test_deterministic_and_empty(torch):
    blocks = synth.q80_blocks(11, 8192, 2048)
    x = synth.activations_f32(12, 1, 2048)
    np.testing.assert_array_equal(run(torch, blocks, x), run(torch, blocks, x))
    x4 = synth.activations_f32(13, 4, 2048)
    np.testing.assert_array_equal(run(torch, blocks, x4), run(torch, blocks, x4))
    assert q4.q8_0_gemv_run(None, None, None, 0, 64, 64, check=False) == q4.Q4_OK
