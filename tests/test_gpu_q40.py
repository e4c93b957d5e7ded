"""GPU parity of the Q4_0 GEMV (q4_0_gemv_run: 32-element blocks of 18 bytes) against the
CPU oracle, within the GEMV tolerance 1e-3 * sum_k |w x| + 1e-6, on every path of the
general kernel it runs on (lanes per row, split-K clusters, M tiles, ragged rows).
Marked gpu.
"""
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
    q4.q4_0_gemv_run(dev(blocks, torch), dev(x, torch), y, M, N, K)
    torch.cuda.synchronize()
    b = host(buf)
    assert np.all(b[:guard] == 12345.0) and np.all(b[guard + M * N:] == 12345.0), "guard words written"
    return b[guard:guard + M * N].reshape(M, N)


@pytest.mark.parametrize("M,N,K", [(1, 896, 896), (2, 4864, 896), (1, 896, 4864), (3, 1000, 2048), (4, 4096, 4096),
                                   (8, 300, 16384), (16, 512, 2048), (5, 77, 32), (1, 1, 64)])
def test_shapes_against_oracle(torch, M, N, K):
    blocks = synth.q40_blocks(M + N + K, N, K)
    x = synth.activations_f32(M * N + K, M, K)
    y = run(torch, blocks, x)
    y_ref, bound = oracle.q40_gemv(blocks, x)
    assert_within_bound(y, y_ref, bound, f"Q4_0 M={M} N={N} K={K}")


def test_lm_head_sampled(torch):
    N, K = 151936, 896
    blocks = synth.q40_blocks(7, N, K)
    x = synth.activations_f32(8, 1, K)
    y = run(torch, blocks, x)
    rows = sorted(set(np.random.default_rng(2).choice(N, 200, replace=False).tolist()) | {0, N - 1})
    y_ref, bound = oracle.q40_gemv_rows(blocks, x, rows)
    assert_within_bound(y[:, rows], y_ref, bound, "Q4_0 LM head")


def test_matches_the_symmetric_group32_gemv(torch):
    # the same weights in the two layouts through the two entry points
    N, K = 4864, 896
    w = synth.q4_weights(9, N, K, 32, symmetric=True)
    nblk = K // 32
    blocks = np.empty((N, nblk, 18), np.uint8)
    blocks[:, :, 0] = (w.scales & 0xFF).astype(np.uint8)
    blocks[:, :, 1] = (w.scales >> 8).astype(np.uint8)
    blocks[:, :, 2:] = w.codes.reshape(N, nblk, 16)
    x = synth.activations_f32(10, 2, K)
    y40 = run(torch, blocks, x)
    y = torch.empty((2, N), dtype=torch.float32, device="cuda")
    q4.q4gemv_run(dev(w.codes, torch), dev(w.scales, torch), None, dev(x, torch), y, 2, N, K, 32)
    y_ref, bound = oracle.q4_gemv(w.codes, w.scales, None, x, 32)
    assert_within_bound(y40, y_ref, bound, "Q4_0 layout")
    assert_within_bound(host(y), y_ref, bound, "MatMulNBits layout")


def test_deterministic_and_empty(torch):
    blocks = synth.q40_blocks(11, 2048, 2048)
    x = synth.activations_f32(12, 4, 2048)
    np.testing.assert_array_equal(run(torch, blocks, x), run(torch, blocks, x))
    assert q4.q4_0_gemv_run(None, None, None, 0, 64, 64, check=False) == q4.Q4_OK


@pytest.mark.parametrize("N,K", [(9765, 896), (8195, 2048), (4901, 4096), (4101, 14336), (40003, 608)])
def test_streamed_kernel(torch, N, K):
    # M = 1 on long matrices: the streamed kernel's Q4_0 instances (a block of rows is one
    # stretch of 18-byte blocks).  9765 x 896: a last block of 21 rows, 8 bytes past a
    # 16-byte multiple; 14336 and 608: the runtime geometry, 608 with 19 chunks per row
    blocks = synth.q40_blocks(N + K, N, K)
    x = synth.activations_f32(N - K, 1, K)
    y = run(torch, blocks, x)
    rows = sorted(set(np.random.default_rng(4).choice(N, 300, replace=False).tolist()) | set(range(N - 70, N)) | {0})
    y_ref, bound = oracle.q40_gemv_rows(blocks, x, rows)
    assert_within_bound(y[:, rows], y_ref, bound, f"Q4_0 streamed N={N} K={K}")
