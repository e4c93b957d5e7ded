"""GPU parity of the int4 GEMV (q4gemv_run) and its dequantisation exports
against the CPU oracle.  Marked gpu: needs an sm_103a device and the built
library; every call goes through the C ABI.
"""
import os
import zlib

import numpy as np
import pytest

import gemm_decode_gb300 as q4
import oracle
import synth
from conftest import GOLDEN_FILES, golden_x, load_golden, pack_codes, pack_zeros
from gpu_util import assert_within_bound, dev, host, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    t = torch_cuda()
    q4.lib()
    return t


def run_gemv(torch, w, x, guard=64):
    """q4gemv_run on device copies; y has guard words on both sides."""
    M, K = x.shape
    buf = torch.full((M * w.N + 2 * guard,), 12345.0, dtype=torch.float32, device="cuda")
    y = buf[guard:guard + M * w.N]
    q4.q4gemv_run(dev(w.codes, torch), dev(w.scales, torch), dev(w.zeros, torch), dev(x, torch), y,
                  M, w.N, K, w.group)
    torch.cuda.synchronize()
    b = host(buf)
    assert np.all(b[:guard] == 12345.0) and np.all(b[guard + M * w.N:] == 12345.0), "guard words written"
    return b[guard:guard + M * w.N].reshape(M, w.N)


@pytest.mark.parametrize("name", GOLDEN_FILES)
def test_hand_worked_examples_exact(torch, name):
    d = load_golden(name)
    w = synth.Q4Weights(d["codes"], d["scales"], d["zeros"], d["N"], d["K"], d["group"])
    for kind, y_expect in d["cases"]:
        y = run_gemv(torch, w, golden_x(kind, d["K"]))
        np.testing.assert_array_equal(y[0], y_expect)


@pytest.mark.parametrize("g", [32, 64, 128])
@pytest.mark.parametrize("symmetric", [False, True])
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8, 13, 16])
def test_small_shapes_against_oracle(torch, g, symmetric, M):
    for N, K in [(1, g), (7, 3 * g), (129, 896 if 896 % g == 0 else 1024), (300, 4864 if 4864 % g == 0 else 4608),
                 (1000, 2 * g), (64, 16384)]:
        if N * K * M > 40_000_000:
            continue
        seed = N * 7 + K + g + M
        w = synth.q4_weights(seed, N, K, g, symmetric=symmetric)
        x = synth.activations_f32(seed, M, K)
        y = run_gemv(torch, w, x)
        y_ref, bound = oracle.q4_gemv(w.codes, w.scales, w.zeros, x, g)
        assert_within_bound(y, y_ref, bound, f"N={N} K={K} M={M} g={g} sym={symmetric}")


@pytest.mark.parametrize("g", [32, 64, 128])
def test_codes_equal_to_zero_point_give_exact_zero(torch, g):
    r = np.random.default_rng(g)
    N, K = 333, 12 * g
    z = r.integers(0, 16, size=(N, K // g))
    q = np.repeat(z, g, axis=1)
    s = r.uniform(0.001, 0.5, size=(N, K // g)).astype(np.float16).view(np.uint16)
    w = synth.Q4Weights(pack_codes(q), s, pack_zeros(z), N, K, g)
    for M in (1, 4, 16):
        x = r.standard_normal((M, K)).astype(np.float32) * 100
        y = run_gemv(torch, w, x)
        assert np.all(y == 0.0)


@pytest.mark.parametrize("outlier", [10.0, 300.0])
def test_heavy_tailed_activations(torch, outlier):
    # activation outliers: a few channels far larger than the rest (every 32-wide
    # slice of x holds one), the case a per-slice shared exponent is most sensitive to
    N, K, g = 2048, 896, 32
    w = synth.q4_weights(31, N, K, g)
    r = np.random.default_rng(int(outlier))
    x = r.standard_normal((2, K)).astype(np.float32)
    x[:, 5::32] *= np.float32(outlier)
    for M in (1, 2):
        y = run_gemv(torch, w, x[:M])
        y_ref, bound = oracle.q4_gemv(w.codes, w.scales, w.zeros, x[:M], g)
        assert_within_bound(y, y_ref, bound, f"outlier {outlier} M={M}")


def test_deterministic_and_row_independent(torch):
    w = synth.q4_weights(5, 4864, 896, 32)
    x = synth.activations_f32(5, 8, 896)
    y1 = run_gemv(torch, w, x)
    y2 = run_gemv(torch, w, x)
    np.testing.assert_array_equal(y1, y2)
    for m in (0, 5):
        ym = run_gemv(torch, w, x[m:m + 1])
        y_ref, bound = oracle.q4_gemv_rows(w.codes, w.scales, w.zeros, x[m:m + 1], 32, range(0, 4864, 97))
        assert_within_bound(ym[:, ::97], y_ref, bound, "row subset")


@pytest.mark.parametrize("g", [32, 64, 128])
@pytest.mark.parametrize("symmetric", [False, True])
def test_dequant_exports_bit_exact(torch, g, symmetric):
    N, K = 77, 7 * 128
    w = synth.q4_weights(g + 1, N, K, g, symmetric=symmetric)
    wf = torch.empty((N, K), dtype=torch.float32, device="cuda")
    wb = torch.empty((N, K), dtype=torch.int16, device="cuda")
    q4.q4_dequant_f32_run(dev(w.codes, torch), dev(w.scales, torch), dev(w.zeros, torch), wf, N, K, g)
    q4.q4_dequant_bf16_run(dev(w.codes, torch), dev(w.scales, torch), dev(w.zeros, torch), wb, N, K, g)
    torch.cuda.synchronize()
    ref = oracle.q4_dequant(w.codes, w.scales, w.zeros, K, g)
    np.testing.assert_array_equal(host(wf).view(np.uint32), ref.view(np.uint32))
    refb = oracle.q4_dequant_bf16(w.codes, w.scales, w.zeros, K, g)
    np.testing.assert_array_equal(host(wb, np.uint16), refb)


def test_dense_equivalence_with_f32_control(torch):
    N, K, g = 2048, 1024, 64
    w = synth.q4_weights(9, N, K, g)
    x = synth.activations_f32(9, 2, K)
    wf = torch.empty((N, K), dtype=torch.float32, device="cuda")
    q4.q4_dequant_f32_run(dev(w.codes, torch), dev(w.scales, torch), dev(w.zeros, torch), wf, N, K, g)
    yd = torch.empty((2, N), dtype=torch.float32, device="cuda")
    q4.f32gemv_run(wf, dev(x, torch), yd)
    torch.cuda.synchronize()
    y = run_gemv(torch, w, x)
    _, bound = oracle.q4_gemv_rows(w.codes, w.scales, w.zeros, x, g, range(N))
    # both are within the tolerance of the same exact value, so within twice it
    err = np.abs(y.astype(np.float64) - host(yd).astype(np.float64))
    assert np.all(err <= 2 * (1e-3 * bound + 1e-6))


def test_empty_and_unsupported(torch):
    w = synth.q4_weights(1, 8, 64, 32)
    x = synth.activations_f32(1, 1, 64)
    y = torch.zeros((1, 8), dtype=torch.float32, device="cuda")
    assert q4.q4gemv_run(dev(w.codes, torch), dev(w.scales, torch), dev(w.zeros, torch), dev(x, torch), y,
                         0, 8, 64, 32) == q4.Q4_OK
    assert q4.q4gemv_run(dev(w.codes, torch), dev(w.scales, torch), dev(w.zeros, torch), dev(x, torch), y,
                         17, 8, 64, 32, check=False) == q4.Q4_ERR_UNSUPPORTED


# ----------------------------------------------------------------- full sizes

def _sample_rows(N, count, seed):
    r = np.random.default_rng(seed)
    rows = set(r.choice(N, size=min(N, count), replace=False).tolist())
    rows |= {0, N - 1}
    return sorted(rows)


def _full_size_check(torch, w, M, seed, count=96):
    x = synth.activations_f32(seed, M, w.K)
    y = run_gemv(torch, w, x)
    rows = _sample_rows(w.N, count, seed)
    y_ref, bound = oracle.q4_gemv_rows(w.codes, w.scales, w.zeros, x, w.group, rows)
    return assert_within_bound(y[:, rows], y_ref, bound, f"N={w.N} K={w.K} M={M}")


def _all_rows_check(torch, w, M, seed):
    """Every output against the oracle, run over the host cores in row slices."""
    x = synth.activations_f32(seed, M, w.K)
    y = run_gemv(torch, w, x)
    y_ref, bound = oracle.q4_gemv_threaded(w.codes, w.scales, w.zeros, x, w.group, os.cpu_count() or 1)
    return assert_within_bound(y, y_ref, bound, f"all rows N={w.N} K={w.K} M={M}")


@pytest.mark.parametrize("name,N,K", synth.DECODE_05B["shapes"])
def test_decode_05b_projection_set(torch, name, N, K):
    # every row of every projection, the LM head included
    w = synth.q4_weights(zlib.crc32(name.encode()) & 0xFFFF, N, K, 32, scale_range=synth.SCALE_05B, tag=name)
    _all_rows_check(torch, w, 1, 17)


def test_single_896(torch):
    w = synth.q4_weights(896, 896, 896, 32)
    x = synth.activations_f32(896, 1, 896)
    y = run_gemv(torch, w, x)
    y_ref, bound = oracle.q4_gemv(w.codes, w.scales, w.zeros, x, 32)
    assert_within_bound(y, y_ref, bound, "896x896")


@pytest.mark.parametrize("name,N,K", synth.DECODE_8B["shapes"])
def test_decode_8b_shapes(torch, name, N, K):
    # every row at every M (the LM head's 128256 rows included)
    w = synth.q4_weights(len(name) * 31, N, K, 128, scale_range=synth.SCALE_8B, tag=name)
    for M in synth.DECODE_8B["Ms"]:
        _all_rows_check(torch, w, M, 100 + M)


@pytest.mark.parametrize("K", synth.SWEEP["Ks"])
@pytest.mark.parametrize("g", synth.SWEEP["groups"])
def test_sweep_cells(torch, K, g):
    # every (N, symmetric, M) of the sweep at this (K, g): every row of the M = 1 cells
    # with at least 64 MB of packed weights (the bandwidth bar's cells), sampled rows of
    # the others
    for N in synth.SWEEP["Ns"]:
        for sym in synth.SWEEP["symmetric"]:
            w = synth.q4_weights(K + N + g, N, K, g, symmetric=sym, tag="sweep")
            for M in synth.SWEEP["Ms"]:
                if M == 1 and w.nbytes >= 64e6:
                    _all_rows_check(torch, w, M, K + M)
                else:
                    _full_size_check(torch, w, M, K + M, count=16)


def test_streamed_kernel_bounded_wait_reports_timeout_without_fault(torch):
    # the TMA-streamed GEMV (long-N shapes) bounds every mbarrier wait the same way
    # as the tensor-core path: with the bound at 0 it must stop, drain and report
    # the LM-head shape: about ten row blocks per CTA, so consumers must wait for
    # blocks the producer can only issue after a slot is released
    N = 151936
    w = synth.q4_weights(21, N, 896, 32)
    x = synth.activations_f32(21, 1, 896)
    y = torch.zeros((1, N), dtype=torch.float32, device="cuda")
    q4.q4gemv_run_ex(dev(w.codes, torch), dev(w.scales, torch), dev(w.zeros, torch), dev(x, torch), y,
                     1, N, 896, 32, wait_timeout_ns=0)
    st = q4.q4gemv_device_status()
    assert st == q4.Q4_ERR_TIMEOUT
    assert q4.q4gemv_device_status() == q4.Q4_OK
    y2 = run_gemv(torch, w, x)
    rows = _sample_rows(N, 64, 3)
    y_ref, bound = oracle.q4_gemv_rows(w.codes, w.scales, w.zeros, x, 32, rows)
    assert_within_bound(y2[:, rows], y_ref, bound, "after timeout")


@pytest.mark.parametrize("K,g,N", [(2048, 64, 9777), (4096, 128, 4899), (8192, 32, 4103), (16384, 128, 4099),
                                   (14336, 128, 4101), (4096, 32, 32771)])
@pytest.mark.parametrize("symmetric", [False, True])
def test_streamed_kernel_two_rows(torch, K, g, N, symmetric):
    # M = 2 on long matrices: the streamed kernel's two-row instances (both rows of x held
    # as planes, every block of codes serving both), partial last blocks; K = 14336 takes
    # the runtime-geometry instance.  Every row against the oracle.
    w = synth.q4_weights(N + 2 * K + g, N, K, g, symmetric=symmetric, tag="two-rows")
    x = synth.activations_f32(N + g + 2, 2, K)
    y = run_gemv(torch, w, x)
    y_ref, bound = oracle.q4_gemv_threaded(w.codes, w.scales, w.zeros, x, g, os.cpu_count() or 1)
    assert_within_bound(y, y_ref, bound, f"two rows N={N} K={K} g={g}")
    # and the call is deterministic
    np.testing.assert_array_equal(y, run_gemv(torch, w, x))


@pytest.mark.parametrize("K,g,N", [(4096, 128, 14336), (2048, 32, 12301), (14336, 64, 12289)])
@pytest.mark.parametrize("symmetric", [False, True])
def test_three_rows_as_two_streamed_launches(torch, K, g, N, symmetric):
    # M = 3 with N >= 12288 on long matrices: rows 0 and 1 of x on the two-row streamed
    # instances, row 2 on the one-row ones (x and y offset by two rows).  Every row of
    # every row of x against the oracle; rows of x are independent.
    w = synth.q4_weights(N + 3 * K + g, N, K, g, symmetric=symmetric, tag="three-rows")
    x = synth.activations_f32(N + g + 3, 3, K)
    y = run_gemv(torch, w, x)
    y_ref, bound = oracle.q4_gemv_threaded(w.codes, w.scales, w.zeros, x, g, os.cpu_count() or 1)
    assert_within_bound(y, y_ref, bound, f"three rows N={N} K={K} g={g}")
    np.testing.assert_array_equal(y[2:3], run_gemv(torch, w, x[2:3]))   # row 2 = the one-row launch alone


@pytest.mark.parametrize("K,g,N", [(896, 32, 9765), (896, 128, 9765), (2048, 64, 9777), (4096, 128, 4899),
                                   (4096, 64, 4899), (8192, 32, 4103), (16384, 32, 4099),
                                   (1152, 32, 9761), (14336, 128, 4101)])
@pytest.mark.parametrize("symmetric", [False, True])
def test_streamed_kernel_ragged_last_block(torch, K, g, N, symmetric):
    # M = 1 and many rows: the TMA-streamed kernel, with N not a multiple of its
    # rows per block, so the last block is partial (codes by bulk copy, scales and
    # zero points by plain copies); 1152 and 14336 take the runtime-geometry instance
    w = synth.q4_weights(N + K + g, N, K, g, symmetric=symmetric, tag="ragged")
    x = synth.activations_f32(N + g, 1, K)
    y = run_gemv(torch, w, x)
    y_ref, bound = oracle.q4_gemv(w.codes, w.scales, w.zeros, x, g)
    assert_within_bound(y, y_ref, bound, f"N={N} K={K} g={g}")
