"""GPU parity of the tensor-core int4 matmul (q4gemm_run) against the CPU oracle.

Shapes whose 128 x 128 tiles would leave most SMs idle (few weight rows and tokens)
run on the split kernel: 128 x 32 or 128 x 64 tiles with the K-blocks split over a
cluster of up to 8 CTAs and the partials added in rank order; the other shapes on the
128 x 128-tile kernel.  Both are covered below.

The tensor-core path feeds the MMA bf16 weights, each the exact binary32
(q - z) * s rounded once to bfloat16, so a single term can be off by up to
2^-9 of |w a|.  Checks:
  * every case: against the oracle's own bf16-rounded weights multiplied in
    binary64 (numpy) within 2e-6 * sum|w_bf16 a| + 1e-6 -- only binary32
    accumulation differs -- and against the exact oracle within the bound that
    follows from the arithmetic, 2^-9 * sum|w a| + 2e-6 * sum|w a| + 1e-6;
  * the prefill workloads (K >= 2048): against the exact oracle within the
    stated tolerance |c - c_ref| <= 1e-3 * sum_k |w_nk a_mk| + 1e-6.
"""
import os

import numpy as np
import pytest

import gemm_decode_gb300 as q4
import oracle
import synth
from conftest import GOLDEN_FILES, golden_x, load_golden
from gpu_util import assert_within_bound, dev, host, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    t = torch_cuda()
    q4.lib()
    return t


def bf16_to_f64(u16):
    return (u16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def run_gemm(torch, w, a_bf16):
    M, K = a_bf16.shape
    c = torch.full((M, w.N), 7.0, dtype=torch.float32, device="cuda")
    q4.q4gemm_run(dev(w.codes, torch), dev(w.scales, torch), dev(w.zeros, torch), dev(a_bf16, torch), c,
                  M, w.N, K, w.group)
    torch.cuda.synchronize()
    assert q4.q4gemv_device_status() == q4.Q4_OK
    return host(c)


BF16_TERM = 2.0 ** -9


def check_case(torch, w, a, stated_tolerance=False):
    c = run_gemm(torch, w, a)
    c_ref, bound = oracle.q4_gemm(w.codes, w.scales, w.zeros, a, w.group)
    what = f"M={a.shape[0]} N={w.N} K={w.K} g={w.group}"
    if stated_tolerance:
        assert_within_bound(c, c_ref, bound, what)
    err = np.abs(c.astype(np.float64) - c_ref.astype(np.float64))
    assert np.all(err <= (BF16_TERM + 2e-6) * bound + 1e-6), what
    wb = bf16_to_f64(oracle.q4_dequant_bf16(w.codes, w.scales, w.zeros, w.K, w.group))
    af = bf16_to_f64(a)
    ref_b = af @ wb.T
    mag = np.abs(af) @ np.abs(wb).T
    err = np.abs(c.astype(np.float64) - ref_b)
    assert np.all(err <= 2e-6 * mag + 1e-6), f"max {np.max(err / (mag + 1e-30))}"


@pytest.mark.parametrize("name", GOLDEN_FILES)
def test_hand_worked_examples_exact(torch, name):
    d = load_golden(name)
    w = synth.Q4Weights(d["codes"], d["scales"], d["zeros"], d["N"], d["K"], d["group"])
    for kind, y_expect in d["cases"]:
        x = golden_x(kind, d["K"])
        a = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        c = run_gemm(torch, w, a)
        np.testing.assert_array_equal(c[0], y_expect)


@pytest.mark.parametrize("g", [32, 64, 128])
@pytest.mark.parametrize("symmetric", [False, True])
def test_small_shapes(torch, g, symmetric):
    # M > 128 takes tiles of 2, 3 or 4 128-row halves of A per CTA: 130 and 256 use two
    # halves (the second partly empty, then full), 300 and 513 three (one and two
    # tiles), 500 four; the last tile's halves run partly or wholly past M
    for M, N, K in [(1, 128, 128), (7, 200, 256), (128, 128, 2 * 64), (130, 256, 384), (300, 136, 512),
                    (64, 384, 1024 if g <= 64 else 1152), (256, 128, 256), (513, 264, 384), (500, 136, 256)]:
        if K % g:
            continue
        w = synth.q4_weights(M + N + K + g, N, K, g, symmetric=symmetric)
        a = synth.activations_bf16(M + K, M, K)
        check_case(torch, w, a)


@pytest.mark.parametrize("M,N,K,g,symmetric", [
    (128, 512, 2048, 64, True),      # the 128-token prefill shape: 32-row tiles, 8-CTA clusters
    (128, 512, 2048, 128, False),
    (100, 200, 2080, 32, False),     # ragged M and N tiles, a half-empty last K-block, 8-CTA clusters
    (300, 96, 1024, 32, True),       # three 128-row tiles of A, the last 44 rows
    (256, 1000, 4096, 128, False),   # 64-row tiles, 4-CTA clusters, two tiles of A
    (512, 300, 8192, 64, False),     # 64-row tiles, four tiles of A, 32 K-blocks per CTA
    (1, 512, 2048, 32, False),       # one token
    (128, 512, 96, 32, False),       # two K-blocks: no split, 32-row tiles
])
def test_split_kernel_whole_output(torch, M, N, K, g, symmetric):
    w = synth.q4_weights(M * 7 + N + K, N, K, g, symmetric=symmetric, tag="split")
    a = synth.activations_bf16(M + 3 * K, M, K)
    check_case(torch, w, a, stated_tolerance=K >= 2048)


@pytest.mark.parametrize("M,N,K,g", [(130, 10240, 256, 32), (300, 10368, 512, 64), (513, 10240, 384, 128)])
def test_regular_tiles_kernel(torch, M, N, K, g):
    # enough 128 x 128 tiles (at least half the SMs) for the regular kernel: 2, 3 and 4
    # halves of A per CTA, partial last tiles
    w = synth.q4_weights(M + N + K, N, K, g, tag="regular")
    a = synth.activations_bf16(M + K + 1, M, K)
    check_case(torch, w, a)


@pytest.mark.parametrize("M,N,K,g", [(1030, 4100, 256, 32), (2048, 2560, 160, 32), (1536, 3840, 512, 128)])
def test_large_tiles_kernel(torch, M, N, K, g):
    # larger problems on the 128 x 128-tile kernel with several halves of A per CTA: a last
    # tile of A a few rows deep, a last tile of weights with 4 rows, a half-empty last
    # K-block (K = 160)
    w = synth.q4_weights(M + N + K + 1, N, K, g, tag="wide")
    a = synth.activations_bf16(M + K + 2, M, K)
    check_case(torch, w, a)


def test_split_kernel_deterministic(torch):
    # the partials of a cluster are added in rank order: repeated calls agree bit for bit
    w = synth.q4_weights(19, 512, 2048, 32, tag="split-det")
    a = synth.activations_bf16(19, 128, 2048)
    np.testing.assert_array_equal(run_gemm(torch, w, a), run_gemm(torch, w, a))


def test_split_kernel_bounded_wait_reports_timeout_without_fault(torch):
    # every wait that is not already satisfied gives up at once; the CTAs still meet both
    # cluster barriers, release tensor memory and raise the status word
    w = synth.q4_weights(23, 512, 2048, 32, tag="split-timeout")
    a = synth.activations_bf16(23, 128, 2048)
    c = torch.zeros((128, 512), dtype=torch.float32, device="cuda")
    q4.q4gemm_run_ex(dev(w.codes, torch), dev(w.scales, torch), dev(w.zeros, torch), dev(a, torch), c,
                     128, 512, 2048, 32, wait_timeout_ns=0)
    assert q4.q4gemv_device_status() == q4.Q4_ERR_TIMEOUT
    assert q4.q4gemv_device_status() == q4.Q4_OK
    check_case(torch, w, a, stated_tolerance=True)


def test_k_tail_half_block(torch):
    # K = 96: the last 64-wide K-block is half empty
    w = synth.q4_weights(3, 256, 96, 32)
    a = synth.activations_bf16(3, 128, 96)
    check_case(torch, w, a)


def test_prefill_gate_128_tokens(torch):
    name, M, N, K = synth.PREFILL["shapes"][0]
    w = synth.q4_weights(128, N, K, 32, tag=name)
    a = synth.activations_bf16(128, M, K)
    check_case(torch, w, a, stated_tolerance=True)


def test_prefill_ffn_2048_tokens_sampled(torch):
    name, M, N, K = synth.PREFILL["shapes"][1]
    w = synth.q4_weights(2048, N, K, 32, tag=name)
    a = synth.activations_bf16(2048, M, K)
    c = run_gemm(torch, w, a)
    r = np.random.default_rng(5)
    ms = sorted(set(r.choice(M, 24, replace=False).tolist()) | {0, M - 1})
    ns = sorted(set(r.choice(N, 24, replace=False).tolist()) | {0, N - 1})
    c_ref, bound = oracle.q4_gemm_rows(w.codes, w.scales, w.zeros, a, 32, ms, ns)
    assert_within_bound(c[np.ix_(ms, ns)], c_ref, bound, "2048x14336x4096 sampled")
    # a whole strip: 128 tokens (one tile of A, rows 1024..1151) against all 14336 weight
    # rows, the oracle run over the host cores in slices of weight rows
    from concurrent.futures import ThreadPoolExecutor
    m0 = 1024
    strip = np.ascontiguousarray(a[m0:m0 + 128])
    cuts = np.linspace(0, N, (os.cpu_count() or 1) + 1).astype(int)

    def part(i):
        n0, n1 = cuts[i], cuts[i + 1]
        return oracle.q4_gemm(w.codes[n0:n1], w.scales[n0:n1], w.zeros[n0:n1], strip, 32)

    with ThreadPoolExecutor(max_workers=len(cuts) - 1) as ex:
        parts = list(ex.map(part, range(len(cuts) - 1)))
    c_ref = np.concatenate([p[0] for p in parts], axis=1)
    bound = np.concatenate([p[1] for p in parts], axis=1)
    assert_within_bound(c[m0:m0 + 128], c_ref, bound, "2048x14336x4096, a 128-token strip, every column")


def test_deterministic(torch):
    w = synth.q4_weights(9, 512, 2048, 32)
    a = synth.activations_bf16(9, 256, 2048)
    np.testing.assert_array_equal(run_gemm(torch, w, a), run_gemm(torch, w, a))


def test_bounded_wait_reports_timeout_without_fault(torch):
    # every pipeline wait that is not already satisfied gives up at once: the
    # kernel must stop, drain what it issued, release tensor memory and raise the
    # status flag -- and the context must stay usable afterwards
    w = synth.q4_weights(4, 512, 2048, 32)
    a = synth.activations_bf16(4, 256, 2048)
    c = torch.zeros((256, 512), dtype=torch.float32, device="cuda")
    # the bound is this call's own option: nothing process-wide changes
    q4.q4gemm_run_ex(dev(w.codes, torch), dev(w.scales, torch), dev(w.zeros, torch), dev(a, torch), c,
                     256, 512, 2048, 32, wait_timeout_ns=0)
    st = q4.q4gemv_device_status()
    assert st == q4.Q4_ERR_TIMEOUT
    assert q4.q4gemv_device_status() == q4.Q4_OK          # flag cleared
    check_case(torch, w, a)                                # and the next call is correct


def test_process_wide_wait_bound_still_applies_to_calls_without_options(torch):
    # the setter keeps its meaning for q4gemm_run; a call with options ignores it
    w = synth.q4_weights(4, 512, 2048, 32)
    a = synth.activations_bf16(4, 256, 2048)
    c = torch.zeros((256, 512), dtype=torch.float32, device="cuda")
    args = (dev(w.codes, torch), dev(w.scales, torch), dev(w.zeros, torch), dev(a, torch), c, 256, 512, 2048, 32)
    try:
        q4.q4gemm_set_wait_timeout_ns(0)
        q4.q4gemm_run_ex(*args, flags=0)          # built-in 1 s bound: completes
        assert q4.q4gemv_device_status() == q4.Q4_OK
        q4.q4gemm_run(*args)                      # the process-wide bound of 0: gives up
        st = q4.q4gemv_device_status()
    finally:
        q4.q4gemm_set_wait_timeout_ns(1_000_000_000)
    assert st == q4.Q4_ERR_TIMEOUT
    check_case(torch, w, a)
