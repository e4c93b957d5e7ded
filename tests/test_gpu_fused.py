"""GPU parity of the fused decode GEMV (q4gemv_fused_run) against the CPU oracle.

The fused call applies the RMSNorm prologue (x / sqrt(mean(x^2) + eps) * gamma) and
the SwiGLU epilogue (rows 2i / 2i+1 a gate / up pair, output silu(gate) * up) around
the int4 GEMV.  M = 1 on long matrices runs the streamed kernel's fused instances; every
other shape the general kernel's fused instance, launched per tile of rows of x.  Each
output is checked against the oracle's binary64 reference within its tolerance: for a
plain output 1e-3 * sum_k |w x'| + 1e-6 (x' the normalised input), for a SwiGLU output
that bound propagated through silu(g) * u.  Marked gpu.
"""
import numpy as np
import pytest

import gemm_decode_gb300 as q4
import oracle
import synth
from gpu_util import dev, host, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    t = torch_cuda()
    q4.lib()
    return t


def gamma_for(K, seed):
    return np.random.default_rng(seed).uniform(0.5, 1.5, K).astype(np.float32)


def run_fused(torch, w, x, gamma, eps, swiglu):
    M, K = x.shape
    cols = w.N // 2 if swiglu else w.N
    guard = 64
    buf = torch.full((M * cols + 2 * guard,), 12345.0, dtype=torch.float32, device="cuda")
    y = buf[guard:guard + M * cols]
    q4.q4gemv_fused_run(dev(w.codes, torch), dev(w.scales, torch), dev(w.zeros, torch), dev(x, torch),
                        None if gamma is None else dev(gamma, torch), eps, y, M, w.N, K, w.group,
                        epilogue=q4.Q4_EPILOGUE_SWIGLU if swiglu else q4.Q4_EPILOGUE_NONE)
    torch.cuda.synchronize()
    b = host(buf)
    assert np.all(b[:guard] == 12345.0) and np.all(b[guard + M * cols:] == 12345.0), "guard words written"
    return b[guard:guard + M * cols].reshape(M, cols)


def check(torch, w, x, gamma, eps, swiglu, what, outputs=None):
    y = run_fused(torch, w, x, gamma, eps, swiglu)
    ref, tol = oracle.q4_gemv_fused(w.codes, w.scales, w.zeros, x, gamma, eps, w.group, swiglu, outputs=outputs)
    yy = y if outputs is None else y[:, outputs]
    assert np.all(np.isfinite(yy)), f"{what}: non-finite output"
    err = np.abs(yy.astype(np.float64) - ref)
    worst = float(np.max(err / tol))
    assert worst <= 1.0, f"{what}: outside tolerance, worst {worst:.3f} of the bound"
    return y


def sample(n, count, seed):
    r = np.random.default_rng(seed)
    return sorted(set(r.choice(n, size=min(n, count), replace=False).tolist()) | {0, n - 1})


@pytest.mark.parametrize("N,K,g", [(9728, 896, 32), (8192, 2048, 64), (4096, 4096, 128), (4096, 14336, 128)])
@pytest.mark.parametrize("symmetric", [False, True])
def test_streamed_rmsnorm_and_swiglu(torch, N, K, g, symmetric):
    # M = 1, long matrices: the streamed kernel's fused instances (K = 14336: the runtime
    # geometry); gate / up rows interleaved, every output checked
    w = synth.q4_weights(N + K + g, N, K, g, symmetric=symmetric, tag="fused")
    x = synth.activations_f32(N + 1, 1, K)
    gamma = gamma_for(K, K)
    check(torch, w, x, gamma, 1e-6, True, f"norm+swiglu N={N} K={K} g={g} sym={symmetric}")
    check(torch, w, x, None, 0.0, True, f"swiglu N={N} K={K} g={g} sym={symmetric}")
    outs = sample(N, 200, 3)
    check(torch, w, x, gamma, 1e-5, False, f"norm N={N} K={K} g={g} sym={symmetric}", outputs=outs)


def test_streamed_lm_head_rmsnorm(torch):
    N, K = 151936, 896
    w = synth.q4_weights(77, N, K, 32, scale_range=synth.SCALE_05B, tag="fused-lm")
    x = synth.activations_f32(78, 1, K) * np.float32(7.0)   # the norm removes the scale
    gamma = gamma_for(K, 79)
    check(torch, w, x, gamma, 1e-6, False, "LM head, RMSNorm", outputs=sample(N, 256, 5))
    check(torch, w, x, gamma, 1e-6, True, "LM head rows as gate/up pairs", outputs=sample(N // 2, 256, 6))


@pytest.mark.parametrize("M", [1, 2, 3, 5, 8, 16])
@pytest.mark.parametrize("N,K,g", [(896, 896, 32), (1152, 896, 32), (4864, 896, 32), (896, 4864, 32),
                                   (258, 2048, 64), (64, 16384, 128)])
def test_general_kernel_fused(torch, M, N, K, g):
    # everything else: the general kernel's fused instance (M = 1 here: fewer than 4096 rows)
    symmetric = (M + N) % 2 == 1
    w = synth.q4_weights(M * 13 + N + K, N, K, g, symmetric=symmetric, tag="fused-general")
    x = synth.activations_f32(M + N + 2, M, K)
    gamma = gamma_for(K, N + M)
    check(torch, w, x, gamma, 1e-6, False, f"norm M={M} N={N} K={K}")
    check(torch, w, x, gamma, 1e-6, True, f"norm+swiglu M={M} N={N} K={K}")
    check(torch, w, x, None, 0.0, True, f"swiglu M={M} N={N} K={K}")


def test_heavy_tailed_activations_fused(torch):
    N, K = 9728, 896
    w = synth.q4_weights(91, N, K, 32, tag="fused-tail")
    x = synth.activations_f32(92, 1, K)
    x[:, np.random.default_rng(3).choice(K, 8, replace=False)] *= 300.0
    check(torch, w, x, gamma_for(K, 93), 1e-6, True, "outliers x300, norm+swiglu")


def test_rmsnorm_removes_the_scale_of_x(torch):
    # RMSNorm(c x) = RMSNorm(x) for eps = 0: the outputs agree to rounding
    N, K = 9728, 896
    w = synth.q4_weights(95, N, K, 32, tag="fused-scale")
    x = synth.activations_f32(96, 1, K)
    gamma = gamma_for(K, 97)
    a = run_fused(torch, w, x, gamma, 0.0, False)
    b = run_fused(torch, w, x * np.float32(1024.0), gamma, 0.0, False)
    ref, tol = oracle.q4_gemv_fused(w.codes, w.scales, w.zeros, x, gamma, 0.0, 32, False)
    assert np.all(np.abs(a - b) <= 2 * tol)


def test_fused_deterministic(torch):
    N, K = 9728, 896
    w = synth.q4_weights(98, N, K, 32, tag="fused-det")
    x = synth.activations_f32(99, 1, K)
    gamma = gamma_for(K, 100)
    np.testing.assert_array_equal(run_fused(torch, w, x, gamma, 1e-6, True), run_fused(torch, w, x, gamma, 1e-6, True))
    x3 = synth.activations_f32(101, 3, K)
    np.testing.assert_array_equal(run_fused(torch, w, x3, gamma, 1e-6, True), run_fused(torch, w, x3, gamma, 1e-6, True))


def test_plain_call_equals_q4gemv_run(torch):
    # no gamma and no epilogue: the call is q4gemv_run
    N, K = 4864, 896
    w = synth.q4_weights(102, N, K, 32, tag="fused-plain")
    x = synth.activations_f32(103, 2, K)
    y = run_fused(torch, w, x, None, 0.0, False)
    y2 = torch.empty((2, N), dtype=torch.float32, device="cuda")
    q4.q4gemv_run(dev(w.codes, torch), dev(w.scales, torch), dev(w.zeros, torch), dev(x, torch), y2, 2, N, K, 32)
    np.testing.assert_array_equal(y, host(y2))
