"""The bounds-checking build (libq4gemv_check.so, -DQ4_BOUNDS_CHECK): every checked
shared- and global-memory index of the streamed, tensor-core and register-resident GEMV
kernels, the split matmul and the Q8_0 CUDA-core GEMV (whose loads are also checked for
alignment) is compared with its buffer; one out of range is counted on a device counter
and skipped.  With a memory checker unavailable, these tests run the shapes with the
most index arithmetic (ragged last blocks and tiles, K tails, runtime geometry) through
that build and require zero counted violations and results within tolerance.  Marked gpu.
"""
import numpy as np
import pytest

import gemm_decode_gb300 as q4
import oracle
import synth
from gemm_decode_gb300 import build as q4build
from gpu_util import assert_within_bound, dev, host, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    t = torch_cuda()
    path = q4build.build(variant="check")
    saved_lib, saved_path = q4._lib, q4.library_path
    q4._lib = None
    q4.library_path = lambda: path
    try:
        q4.lib()
        assert q4.q4gemv_bounds_violations() == 0   # a checking build, counter clear
        yield t
    finally:
        q4._lib, q4.library_path = saved_lib, saved_path


def run_checked(torch, w, x, what, rows=None):
    M, K = x.shape
    y = torch.full((M, w.N), float("nan"), dtype=torch.float32, device="cuda")
    q4.q4gemv_run(dev(w.codes, torch), dev(w.scales, torch), dev(w.zeros, torch), dev(x, torch), y,
                  M, w.N, K, w.group)
    assert q4.q4gemv_bounds_violations() == 0, f"{what}: out-of-range accesses counted"
    yh = host(y)
    if rows is None:
        y_ref, bound = oracle.q4_gemv(w.codes, w.scales, w.zeros, x, w.group)
        assert_within_bound(yh, y_ref, bound, what)
    else:
        y_ref, bound = oracle.q4_gemv_rows(w.codes, w.scales, w.zeros, x, w.group, rows)
        assert_within_bound(yh[:, rows], y_ref, bound, what)


@pytest.mark.parametrize("symmetric", [False, True])
@pytest.mark.parametrize("N,K,g", [(9765, 896, 32), (4899, 4096, 128), (4101, 14336, 128), (4099, 16384, 32)])
def test_streamed_kernel(torch, N, K, g, symmetric):
    # M = 1, many rows: the TMA-streamed kernel, partial last block; K = 14336 has no
    # compile-time instance (runtime geometry)
    w = synth.q4_weights(N + K, N, K, g, symmetric=symmetric, tag="bounds")
    x = synth.activations_f32(N, 1, K)
    run_checked(torch, w, x, f"streamed N={N} K={K} g={g}")


@pytest.mark.parametrize("N,K,g", [(4899, 4096, 128), (4101, 14336, 128), (9777, 2048, 32)])
def test_streamed_kernel_two_rows(torch, N, K, g):
    # M = 2: the two-row instances (and the runtime geometry at K = 14336), partial last block
    w = synth.q4_weights(N + K + 2, N, K, g, tag="bounds-two-rows")
    x = synth.activations_f32(N + 3, 2, K)
    run_checked(torch, w, x, f"streamed two rows N={N} K={K} g={g}")


@pytest.mark.parametrize("M,N,K,g", [(16, 8323, 4128, 32), (5, 8196, 2048, 64), (9, 4100, 896, 128),
                                     (8, 4100, 4128, 32), (3, 900, 4864, 64)])
def test_tensor_core_kernel(torch, M, N, K, g):
    # partial last 128-row tile; K = 4128 leaves the last K-block half empty; with these
    # few tiles each tile's K-blocks are split over a cluster (2 to 8 CTAs, uneven shares)
    w = synth.q4_weights(M + N + K, N, K, g, tag="bounds-tc")
    x = synth.activations_f32(M + K, M, K)
    run_checked(torch, w, x, f"tensor-core M={M} N={N} K={K}")


@pytest.mark.parametrize("M,N,K,g", [(16, 39100, 4128, 32), (9, 78000, 896, 128)])
def test_tensor_core_kernel_unsplit(torch, M, N, K, g):
    # enough tiles for no K split: 306 tiles of 128 rows, and 305 of 256 rows (two MMAs per
    # CTA); partial last tiles, a half-empty last K-block
    w = synth.q4_weights(41 + M, N, K, g, tag="bounds-tc-unsplit")
    x = synth.activations_f32(42 + M, M, K)
    rows = sorted(set(np.random.default_rng(6).choice(N, size=64, replace=False).tolist()) | {0, N - 1})
    run_checked(torch, w, x, f"tensor-core unsplit M={M} N={N} K={K}", rows=rows)


@pytest.mark.parametrize("M,N,K,g", [(1, 896, 896, 32), (1, 128, 896, 32), (1, 4864, 896, 32),
                                     (1, 896, 4864, 32), (2, 1000, 2048, 64), (2, 77, 4096, 128)])
@pytest.mark.parametrize("symmetric", [False, True])
def test_register_resident_kernel(torch, M, N, K, g, symmetric):
    # M <= 2 below the streamed kernel's row count: per-thread cp.async rings, ragged
    # row tails, split-K clusters for the long rows
    w = synth.q4_weights(M * 3 + N + K, N, K, g, symmetric=symmetric, tag="bounds-xreg")
    x = synth.activations_f32(N + M, M, K)
    run_checked(torch, w, x, f"register-resident M={M} N={N} K={K}")


@pytest.mark.parametrize("N,K,g", [(1152, 896, 32), (896, 4864, 32), (9730, 896, 64), (4098, 14336, 128)])
def test_fused_kernels(torch, N, K, g):
    # the fused instances (RMSNorm and SwiGLU): register-resident (the first two) and
    # streamed (a partial last block; runtime geometry for K = 14336)
    w = synth.q4_weights(N + 5, N, K, g, tag="bounds-fused")
    x = synth.activations_f32(N + 6, 1, K)
    gamma = np.random.default_rng(N).uniform(0.5, 1.5, K).astype(np.float32)
    y = torch.full((1, N // 2), float("nan"), dtype=torch.float32, device="cuda")
    q4.q4gemv_fused_run(dev(w.codes, torch), dev(w.scales, torch), dev(w.zeros, torch), dev(x, torch),
                        dev(gamma, torch), 1e-6, y, 1, N, K, g, epilogue=q4.Q4_EPILOGUE_SWIGLU)
    assert q4.q4gemv_bounds_violations() == 0, f"fused N={N} K={K}: out-of-range accesses counted"
    outs = sorted(set(np.random.default_rng(1).choice(N // 2, size=min(N // 2, 64), replace=False).tolist())
                  | {0, N // 2 - 1})
    ref, tol = oracle.q4_gemv_fused(w.codes, w.scales, w.zeros, x, gamma, 1e-6, g, True, outputs=outs)
    assert np.all(np.abs(host(y)[:, outs] - ref) <= tol)


@pytest.mark.parametrize("N,K", [(9765, 896), (40003, 608)])
def test_q40_streamed_kernel(torch, N, K):
    blocks = synth.q40_blocks(N + 7, N, K)
    x = synth.activations_f32(N + 8, 1, K)
    y = torch.full((1, N), float("nan"), dtype=torch.float32, device="cuda")
    q4.q4_0_gemv_run(dev(blocks, torch), dev(x, torch), y, 1, N, K)
    assert q4.q4gemv_bounds_violations() == 0, f"Q4_0 N={N} K={K}: out-of-range accesses counted"
    rows = sorted(set(np.random.default_rng(3).choice(N, 64, replace=False).tolist()) | {0, N - 1})
    y_ref, bound = oracle.q40_gemv_rows(blocks, x, rows)
    assert_within_bound(host(y)[:, rows], y_ref, bound, f"Q4_0 bounds N={N} K={K}")


@pytest.mark.parametrize("K,g", [(896, 32), (4096, 128)])
def test_grouped_streamed_kernel(torch, K, g):
    # several matrices in one streamed launch, each with its own CTAs, x and y; partial
    # last blocks and a matrix smaller than one block
    specs = [4099, 37, 1, 9001]
    ws = [synth.q4_weights(K + N, N, K, g, tag="bounds-grouped") for N in specs]
    xs = [synth.activations_f32(N + 5, 1, K) for N in specs]
    ys = [torch.full((1, N), float("nan"), dtype=torch.float32, device="cuda") for N in specs]
    segs = [(dev(w.codes, torch), dev(w.scales, torch), dev(w.zeros, torch), dev(x, torch), y, w.N)
            for w, x, y in zip(ws, xs, ys)]
    q4.q4gemv_grouped_run(segs, K, g)
    assert q4.q4gemv_bounds_violations() == 0, f"grouped K={K}: out-of-range accesses counted"
    for w, x, y in zip(ws, xs, ys):
        y_ref, bound = oracle.q4_gemv(w.codes, w.scales, w.zeros, x, g)
        assert_within_bound(host(y), y_ref, bound, f"grouped K={K} N={w.N}")


@pytest.mark.parametrize("M,N,K,g", [(100, 200, 2080, 32), (300, 96, 1024, 64), (256, 1000, 4096, 128),
                                     (1030, 4100, 160, 32)])
def test_split_matmul_kernel(torch, M, N, K, g):
    # the matmul's split kernel: ragged tiles of A and of weight rows, a half-empty last
    # K-block, 32- and 64-row tiles, 4- and 8-CTA clusters; and (the last case) the
    # 128 x 128-tile kernel with a 6-row last tile of A, a 4-row last tile of weights, a K tail
    w = synth.q4_weights(M + N + K, N, K, g, tag="bounds-split")
    a = synth.activations_bf16(M + 1, M, K)
    c = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    q4.q4gemm_run(dev(w.codes, torch), dev(w.scales, torch), dev(w.zeros, torch), dev(a, torch), c, M, N, K, g)
    assert q4.q4gemv_bounds_violations() == 0, f"split matmul M={M} N={N} K={K}: out-of-range accesses counted"
    c_ref, bound = oracle.q4_gemm(w.codes, w.scales, w.zeros, a, g)
    err = np.abs(host(c).astype(np.float64) - c_ref.astype(np.float64))
    assert np.all(err <= (2.0 ** -9 + 2e-6) * bound + 1e-6)


@pytest.mark.parametrize("N,K", [(9765, 896), (4101, 14336), (4901, 4096)])
def test_q80_streamed_kernel(torch, N, K):
    blocks = synth.q80_blocks(N + 9, N, K)
    x = synth.activations_f32(N + 10, 1, K)
    y = torch.full((1, N), float("nan"), dtype=torch.float32, device="cuda")
    q4.q8_0_gemv_run(dev(blocks, torch), dev(x, torch), y, 1, N, K)
    assert q4.q4gemv_bounds_violations() == 0, f"Q8_0 N={N} K={K}: out-of-range accesses counted"
    rows = sorted(set(np.random.default_rng(3).choice(N, 64, replace=False).tolist()) | {0, N - 1})
    y_ref, bound = oracle.q80_gemv_rows(blocks, x, rows)
    assert_within_bound(host(y)[:, rows], y_ref, bound, f"Q8_0 bounds N={N} K={K}")


@pytest.mark.parametrize("offset", [0, 2])
@pytest.mark.parametrize("M,N,K", [(5, 77, 32), (3, 2001, 608), (7, 999, 1056), (4, 4099, 896), (16, 301, 864),
                                   (1, 896, 4864), (2, 33, 4864)])
def test_q80_cuda_core_kernel(torch, M, N, K, offset):
    # the CUDA-core Q8_0 kernel: 32- and 16-bit code loads at addresses that are only 2-byte
    # aligned; rows of an odd number of blocks alternate between the two alignments, and a
    # blocks array 2 bytes past a 4-byte boundary swaps them; every load is checked for range
    # and alignment
    blocks = synth.q80_blocks(N + K + offset, N, K)
    raw = torch.zeros(blocks.size + 16, dtype=torch.uint8, device="cuda")
    raw[offset:offset + blocks.size] = torch.from_numpy(blocks.reshape(-1)).cuda()
    x = synth.activations_f32(N + M, M, K)
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    q4.q8_0_gemv_run(raw.data_ptr() + offset, dev(x, torch), y, M, N, K)
    assert q4.q4gemv_bounds_violations() == 0, f"Q8_0 CUDA-core M={M} N={N} K={K}: out-of-range accesses counted"
    y_ref, bound = oracle.q80_gemv(blocks, x)
    assert_within_bound(host(y), y_ref, bound, f"Q8_0 CUDA-core bounds M={M} N={N} K={K} offset={offset}")

