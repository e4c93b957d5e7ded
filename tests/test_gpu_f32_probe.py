"""GPU parity of the dense f32 GEMV control and the read-bandwidth probe."""
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


@pytest.mark.parametrize("M", [1, 2, 3, 4, 8, 16])
def test_f32_control_small(torch, M):
    for N, K in [(1, 4), (33, 100), (896, 896), (130, 4864), (64, 16384)]:
        W = synth.dense_f32(N + K, N, K)
        x = synth.activations_f32(N + K, M, K)
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        q4.f32gemv_run(dev(W, torch), dev(x, torch), y)
        torch.cuda.synchronize()
        y_ref, bound = oracle.f32_gemv(W, x)
        assert_within_bound(host(y), y_ref, bound, f"f32 N={N} K={K} M={M}")


@pytest.mark.parametrize("N,K", [(896, 896), (151936, 896), (4096, 14336)])
def test_f32_control_full_size_sampled(torch, N, K):
    W = synth.dense_f32(7, N, K)
    x = synth.activations_f32(7, 1, K)
    y = torch.empty((1, N), dtype=torch.float32, device="cuda")
    q4.f32gemv_run(dev(W, torch), dev(x, torch), y)
    torch.cuda.synchronize()
    rows = sorted(set(np.random.default_rng(1).choice(N, 64, replace=False).tolist()) | {0, N - 1})
    y_ref, bound = oracle.f32_gemv_rows(W, x, rows)
    assert_within_bound(host(y)[:, rows], y_ref, bound, "f32 sampled")


@pytest.mark.parametrize("n", [4, 1000, 1 << 20, (1 << 22) + 12])
@pytest.mark.parametrize("blocks", [0, 1, 7])
def test_read_probe_sums(torch, n, blocks):
    buf = synth.uniform_f32(n, n)
    d = dev(buf, torch)
    partial = torch.zeros(4096, dtype=torch.float32, device="cuda")
    used = q4.vec4_read_probe_run(d, n * 4, partial, blocks)
    torch.cuda.synchronize()
    p = host(partial)[:used].astype(np.float64)
    # integer data below 2^24 per partial: every partial sum is exact
    assert p.sum() == oracle.sum_f32(buf)
