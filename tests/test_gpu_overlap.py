"""Overlapped (programmatic dependent) launch of the GEMV and matmul kernels.

With the Q4_RUN_OVERLAPPED option of q4gemv_run_ex (or the process-wide
q4gemv_set_overlapped_launch(1) for q4gemv_run) a GEMV may start streaming its
weights while the kernel before it in the stream still runs, and must wait for
that kernel before it reads x or writes y.  These tests run chains in which the y of
one call is the x of the next, so a read of x that does not wait sees the
previous contents of the buffer (NaN, or the previous pass's values) and the
stage disagrees with the oracle evaluated on the GPU's actual input.
Marked gpu: needs an sm_103a device and the built library.
"""
import numpy as np
import pytest

import gemm_decode_gb300 as q4
import oracle
import synth
from gpu_util import assert_within_bound, dev, host, torch_cuda

pytestmark = pytest.mark.gpu

# (N, K, group): each stage's K equals the previous stage's N, except the last of
# each chain, which reads the output of the stage two before it.
CHAIN_05B = [(896, 896, 32), (4864, 896, 32), (896, 4864, 32), (151936, 896, 32), (128, 896, 32)]
CHAIN_8B = [(4096, 4096, 128), (14336, 4096, 128), (4096, 14336, 128), (128256, 4096, 128)]


@pytest.fixture(scope="module")
def torch():
    t = torch_cuda()
    q4.lib()
    return t


@pytest.fixture
def overlapped():
    old = q4.q4gemv_set_overlapped_launch(True)
    try:
        yield
    finally:
        q4.q4gemv_set_overlapped_launch(bool(old))


def _sample_rows(N, count, seed):
    r = np.random.default_rng(seed)
    rows = set(r.choice(N, size=min(N, count), replace=False).tolist())
    return sorted(rows | {0, N - 1})


class Chain:
    def __init__(self, torch, stages, seed, symmetric):
        self.torch = torch
        self.stages = stages
        self.w = [synth.q4_weights(seed + i, N, K, g, symmetric=symmetric, tag="chain")
                  for i, (N, K, g) in enumerate(stages)]
        self.dw = [(dev(w.codes, torch), dev(w.scales, torch), dev(w.zeros, torch)) for w in self.w]
        self.x0 = torch.empty((1, stages[0][1]), dtype=torch.float32, device="cuda")
        self.ys = [torch.full((1, N), float("nan"), dtype=torch.float32, device="cuda") for N, _, _ in stages]
        # input of stage i: x0, then the previous stage's y; a stage whose K differs
        # from the previous N reads the output two stages back
        self.src = []
        for i, (N, K, g) in enumerate(stages):
            if i == 0:
                self.src.append(-1)
            elif stages[i - 1][0] == K:
                self.src.append(i - 1)
            else:
                assert stages[i - 2][0] == K
                self.src.append(i - 2)

    def inp(self, i):
        return self.x0 if self.src[i] < 0 else self.ys[self.src[i]]

    def launch(self, stream=None, per_call=True):
        """The chain; per_call: each launch overlapped by its own option, else through
        q4gemv_run and whatever the process-wide setting is."""
        for i, ((N, K, g), (c, s, z)) in enumerate(zip(self.stages, self.dw)):
            if per_call:
                q4.q4gemv_run_ex(c, s, z, self.inp(i), self.ys[i], 1, N, K, g, flags=q4.Q4_RUN_OVERLAPPED,
                                 stream=stream)
            else:
                q4.q4gemv_run(c, s, z, self.inp(i), self.ys[i], 1, N, K, g, stream=stream)

    def check(self, seed):
        """Every stage against the oracle on the input the GPU actually held."""
        ys = [host(y) for y in self.ys]
        for i, w in enumerate(self.w):
            x = host(self.x0) if self.src[i] < 0 else ys[self.src[i]]
            assert np.all(np.isfinite(x)), f"stage {i}: input not finite"
            rows = list(range(w.N)) if w.N <= 4096 else _sample_rows(w.N, 48, seed + i)
            y_ref, bound = oracle.q4_gemv_rows(w.codes, w.scales, w.zeros, x.reshape(1, -1), w.group, rows)
            assert_within_bound(ys[i][:, rows], y_ref, bound, f"stage {i} N={w.N} K={w.K}")


def test_overlapped_launch_is_off_by_default_and_toggles(torch):
    old = q4.q4gemv_set_overlapped_launch(True)
    try:
        assert old == 0
        assert q4.q4gemv_set_overlapped_launch(True) == 1
        assert q4.q4gemv_set_overlapped_launch(False) == 1
        assert q4.q4gemv_set_overlapped_launch(False) == 0
    finally:
        q4.q4gemv_set_overlapped_launch(bool(old))


@pytest.mark.parametrize("symmetric", [False, True])
@pytest.mark.parametrize("stages", [CHAIN_05B, CHAIN_8B], ids=["0.5b", "8b"])
def test_dependent_chain_eager(torch, stages, symmetric):
    ch = Chain(torch, stages, 40 + len(stages), symmetric)
    for rep in range(2):
        # a new x0 each pass: a stage that read its input before the previous stage
        # finished would see NaN (first pass) or the previous pass's values
        ch.x0.copy_(torch.from_numpy(synth.activations_f32(300 + rep, 1, stages[0][1])).cuda())
        ch.launch()
        torch.cuda.synchronize()
        ch.check(500 + rep)


def test_dependent_chain_process_wide_setting(torch, overlapped):
    # q4gemv_run under the process-wide setting behaves as the per-call option does
    ch = Chain(torch, CHAIN_05B, 45, False)
    for rep in range(2):
        ch.x0.copy_(torch.from_numpy(synth.activations_f32(330 + rep, 1, CHAIN_05B[0][1])).cuda())
        ch.launch(per_call=False)
        torch.cuda.synchronize()
        ch.check(530 + rep)


def test_dependent_chain_in_cuda_graph(torch):
    ch = Chain(torch, CHAIN_05B, 61, False)
    s = torch.cuda.Stream()
    ch.x0.zero_()
    with torch.cuda.stream(s):
        ch.launch(stream=s)          # eager pass before capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):           # the chain three times in one graph
            ch.launch(stream=s)
    for rep in range(2):
        ch.x0.copy_(torch.from_numpy(synth.activations_f32(700 + rep, 1, CHAIN_05B[0][1])).cuda())
        for y in ch.ys:
            y.fill_(float("nan"))
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            g.replay()
        torch.cuda.synchronize()
        ch.check(900 + rep)


# The matmul (q4gemm_run_ex with Q4_RUN_OVERLAPPED): the split kernel (few tiles) and the
# regular one (one and four 128-row halves of A per CTA)
GEMM_SHAPES = [(128, 512, 2048, 32), (200, 1024, 1024, 64), (640, 2048, 1024, 128)]


def _gemm_weights(torch, M, N, K, g):
    w = synth.q4_weights(M + N + K, N, K, g, tag="gemm-overlap")
    return w, (dev(w.codes, torch), dev(w.scales, torch), dev(w.zeros, torch))


@pytest.mark.parametrize("M,N,K,g", GEMM_SHAPES)
def test_matmul_reads_a_written_by_the_kernel_before_it(torch, M, N, K, g):
    # the kernel right before the overlapped matmul converts A to bf16 (A held NaN until
    # then): a read of A that did not wait would see NaN or the previous pass
    w, dw = _gemm_weights(torch, M, N, K, g)
    a32 = dev(synth.activations_f32(M + 1, M, K), torch)
    a = torch.full((M, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    c = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    for rep in range(2):
        a.copy_(a32 * (1.0 + rep))         # a conversion kernel writes A
        q4.q4gemm_run_ex(*dw, a, c, M, N, K, g, flags=q4.Q4_RUN_OVERLAPPED)
        torch.cuda.synchronize()
        a_bits = host(a.view(torch.int16)).view(np.uint16)
        c_ref, bound = oracle.q4_gemm(w.codes, w.scales, w.zeros, a_bits, g)
        err = np.abs(host(c).astype(np.float64) - c_ref.astype(np.float64))
        assert np.all(err <= (2.0 ** -9 + 2e-6) * bound + 1e-6), f"pass {rep} M={M} N={N} K={K}"


@pytest.mark.parametrize("M,N,K,g", GEMM_SHAPES)
def test_matmul_writes_c_after_the_kernel_before_it_read_it(torch, M, N, K, g):
    # the kernel right before the overlapped matmul reads C (a scaled copy); it must see
    # C's old contents, and C must then hold the product
    w, dw = _gemm_weights(torch, M, N, K, g)
    a_bits = (synth.activations_f32(M + 2, M, K).view(np.uint32) >> 16).astype(np.uint16)
    a = dev(a_bits, torch)
    c = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
    seen = torch.empty_like(c)
    torch.cuda.synchronize()
    torch.mul(c, 2.0, out=seen)          # a kernel reads C
    q4.q4gemm_run_ex(*dw, a, c, M, N, K, g, flags=q4.Q4_RUN_OVERLAPPED)
    torch.cuda.synchronize()
    assert np.all(host(seen) == 14.0), "the previous kernel saw C already overwritten"
    c_ref, bound = oracle.q4_gemm(w.codes, w.scales, w.zeros, a_bits, g)
    err = np.abs(host(c).astype(np.float64) - c_ref.astype(np.float64))
    assert np.all(err <= (2.0 ** -9 + 2e-6) * bound + 1e-6)

