"""GPU parity of the grouped decode GEMV (q4gemv_grouped_run) against the CPU oracle.

Several M = 1 GEMVs of one K, each with its own weights, x and y, issued as one call:
runs of matrices the streamed kernel serves go out as one launch in which every matrix
has CTAs of its own; the rest run one q4gemv_run each.  Every output is checked against
the oracle's binary64 reference within 1e-3 * sum_k |w x| + 1e-6 (sampled rows on the
LM-head-sized matrix, every row elsewhere), and guard words around each y must stay
untouched.  Marked gpu.
"""
import numpy as np
import pytest

import gemm_decode_gb300 as q4
import oracle
import synth
from gpu_util import assert_within_bound, dev, host, torch_cuda

pytestmark = pytest.mark.gpu

GUARD = 64


@pytest.fixture(scope="module")
def torch():
    t = torch_cuda()
    q4.lib()
    return t


def make(torch, specs, K, g, seed):
    """specs: (N, symmetric) per matrix -> host weights, host x, device tuples, y buffers."""
    hw, hx, segs, bufs = [], [], [], []
    for i, (N, symmetric) in enumerate(specs):
        w = synth.q4_weights(seed + 31 * i, N, K, g, symmetric=symmetric, tag="grouped")
        x = synth.activations_f32(seed + 31 * i + 1, 1, K)
        buf = torch.full((N + 2 * GUARD,), 12345.0, dtype=torch.float32, device="cuda")
        hw.append(w)
        hx.append(x)
        bufs.append(buf)
        segs.append((dev(w.codes, torch), dev(w.scales, torch), dev(w.zeros, torch), dev(x, torch),
                     buf[GUARD:GUARD + N], N))
    return hw, hx, segs, bufs


def check(hw, hx, bufs, K, g, what, sample_above=20000):
    for i, (w, x, buf) in enumerate(zip(hw, hx, bufs)):
        b = host(buf)
        assert np.all(b[:GUARD] == 12345.0) and np.all(b[GUARD + w.N:] == 12345.0), f"{what}[{i}]: guard words"
        y = b[GUARD:GUARD + w.N].reshape(1, w.N)
        if w.N > sample_above:
            rows = sorted(set(np.random.default_rng(i).choice(w.N, 256, replace=False).tolist()) | {0, w.N - 1})
            y_ref, bound = oracle.q4_gemv_rows(w.codes, w.scales, w.zeros, x, g, rows)
            assert_within_bound(y[:, rows], y_ref, bound, f"{what}[{i}] N={w.N}")
        else:
            y_ref, bound = oracle.q4_gemv(w.codes, w.scales, w.zeros, x, g)
            assert_within_bound(y, y_ref, bound, f"{what}[{i}] N={w.N}")


def test_decode_set_one_launch(torch):
    # the K = 896 projections of the 0.5B-class set, each with its own x: q, k, v, gate,
    # up and the LM head in one streamed launch
    specs = [(896, False), (128, False), (128, False), (4864, False), (4864, False), (151936, False)]
    hw, hx, segs, bufs = make(torch, specs, 896, 32, 5)
    q4.q4gemv_grouped_run(segs, 896, 32)
    torch.cuda.synchronize()
    check(hw, hx, bufs, 896, 32, "decode set")


@pytest.mark.parametrize("K,g", [(896, 128), (2048, 64), (4096, 128), (8192, 32)])
@pytest.mark.parametrize("symmetric", [False, True])
def test_ragged_matrices(torch, K, g, symmetric):
    # rows that end in partial blocks, a one-row matrix, and a matrix smaller than a block
    specs = [(4099, symmetric), (1, symmetric), (37, symmetric), (9000 if K < 2048 else 5003, symmetric)]
    hw, hx, segs, bufs = make(torch, specs, K, g, K + g)
    q4.q4gemv_grouped_run(segs, K, g)
    torch.cuda.synchronize()
    check(hw, hx, bufs, K, g, f"ragged K={K} g={g} sym={symmetric}")


def test_other_paths(torch):
    # K without a compile-time streamed geometry (one q4gemv_run per matrix), matrices with
    # and without zero points mixed (the same), eleven matrices (two grouped launches of
    # eight and three), and an empty entry: every matrix still right
    for K, specs in [(1024, [(4096, False), (300, False)]),
                     (896, [(5000, False), (700, True), (64, False)]),
                     # well over one block of rows per SM at K = 896, and K = 4096 (no block
                     # rule): only the mixed zero-point presence sends these down the fallback
                     (896, [(6000, False), (3000, True), (4864, False)]),
                     (4096, [(4096, True), (300, False), (1000, True)]),
                     (896, [(2000 + 97 * i, False) for i in range(11)])]:
        hw, hx, segs, bufs = make(torch, specs, K, 32, K + len(specs))
        segs.insert(1, (None, None, None, None, None, 0))
        q4.q4gemv_grouped_run(segs, K, 32)
        torch.cuda.synchronize()
        check(hw, hx, bufs, K, 32, f"K={K} n={len(specs)}")


def test_grouped_deterministic(torch):
    specs = [(4864, False), (896, False), (20000, False)]
    hw, hx, segs, bufs = make(torch, specs, 896, 32, 77)
    q4.q4gemv_grouped_run(segs, 896, 32)
    torch.cuda.synchronize()
    first = [host(b).copy() for b in bufs]
    q4.q4gemv_grouped_run(segs, 896, 32)
    torch.cuda.synchronize()
    for a, b in zip(first, bufs):
        np.testing.assert_array_equal(a, host(b))


def test_dependent_matrices_rejected_without_launch(torch):
    # a chain (the second matrix reads the first's output) is not one grouped launch: the
    # call is refused before anything runs
    w = synth.q4_weights(4, 4864, 896, 32)
    a = (dev(w.codes, torch), dev(w.scales, torch), dev(w.zeros, torch))
    x = torch.zeros((1, 896), dtype=torch.float32, device="cuda")
    y0 = torch.full((4864,), 7.0, dtype=torch.float32, device="cuda")
    y1 = torch.full((4864,), 7.0, dtype=torch.float32, device="cuda")
    st = q4.q4gemv_grouped_run([(*a, x, y0, 4864), (*a, y0[:896], y1, 4864)], 896, 32, check=False)
    assert st == q4.Q4_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert np.all(host(y0) == 7.0) and np.all(host(y1) == 7.0), "a rejected call launched work"


def test_empty_and_invalid(torch):
    assert q4.q4gemv_grouped_run([], 896, 32) == q4.Q4_OK
    w = synth.q4_weights(3, 64, 896, 32)
    x = torch.zeros((1, 896), dtype=torch.float32, device="cuda")
    y = torch.zeros((64,), dtype=torch.float32, device="cuda")
    ok = (dev(w.codes, torch), dev(w.scales, torch), dev(w.zeros, torch), x, y, 64)
    bad = (dev(w.codes, torch), dev(w.scales, torch), dev(w.zeros, torch), x[:, 1:], y, 64)   # x 4 bytes off
    y.fill_(7.0)
    assert q4.q4gemv_grouped_run([ok, bad], 896, 32, check=False) == q4.Q4_ERR_MISALIGNED
    torch.cuda.synchronize()
    assert np.all(host(y) == 7.0), "a rejected call launched work"
