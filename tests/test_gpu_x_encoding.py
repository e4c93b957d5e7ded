"""The x encoding of the dp4a GEMV kernels as a stated, tested contract.

The streamed (M = 1 and 2, long matrices; M = 3 as two launches on wide ones),
register-resident (M <= 2) and grouped
GEMV kernels hold each 32-element chunk c of a row of x as 24-bit integers
under one shared power of two 2^E_c, 2^(E_c-1) <= max_{k in c} |x_k| < 2^E_c
(E_c >= -100).  The library header states what that guarantees per output:

    |y - y_exact| <= B1 + (K/32 + 10) * 2^-24 * (sum_k |w_k x_k| + B1),
    B1 = (1 + 2^-7) * sum_c 2^(E_c - 23) * sum_{k in c} |w_k|

This file checks that bound, element by element against the oracle (binary64,
exact dequantised weights), on inputs built to stress it: chunks holding one
value 2^10 .. 2^20 times the rest at a position whose code equals its zero
point in every row (so the large value adds nothing to sum |w x| while it
coarsens its neighbours), rows of tiny, subnormal and huge values, and small K.
The same inputs through the CUDA-core float kernel (q4gemv_run_ex with
Q4_RUN_EXACT_X) must meet the stated tolerance 1e-3 * sum |w x| + 1e-6.
"""
import numpy as np
import pytest

import gemm_decode_gb300 as q4
import oracle
import synth
from conftest import pack_codes, pack_zeros
from gpu_util import assert_within_bound, dev, host, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    t = torch_cuda()
    q4.lib()
    return t


def unpack(w):
    """Integer codes q[N, K] and zero points z[N, K/g] of packed weights (test side)."""
    q = np.empty((w.N, w.K), np.int64)
    q[:, 0::2] = w.codes & 0xF
    q[:, 1::2] = w.codes >> 4
    nb = w.K // w.group
    if w.zeros is None:
        z = np.full((w.N, nb), 8, np.int64)
    else:
        z = np.empty((w.N, 2 * w.zeros.shape[1]), np.int64)
        z[:, 0::2] = w.zeros & 0xF
        z[:, 1::2] = w.zeros >> 4
        z = z[:, :nb]
    return q, z


def with_dead_columns(w, cols):
    """The same weights with the code of every column in `cols` set to its zero point
    in every row (those columns' weights are exactly 0)."""
    q, z = unpack(w)
    zk = np.repeat(z, w.group, axis=1)
    q[:, cols] = zk[:, cols]
    zeros = None if w.zeros is None else pack_zeros(z)
    return synth.Q4Weights(pack_codes(q), w.scales, zeros, w.N, w.K, w.group)


def encoding_bound(w, x):
    """The header's bound for the dp4a kernels, [M, N] in binary64."""
    wd = oracle.q4_dequant(w.codes, w.scales, w.zeros, w.K, w.group).astype(np.float64)
    aw = np.abs(wd)
    xa = np.abs(x.astype(np.float64))
    M, K = x.shape
    C = K // 32
    mu = xa.reshape(M, C, 32).max(axis=2)
    E = np.frexp(mu)[1]                         # mu = f * 2^E, 0.5 <= f < 1
    E = np.where(mu > 0, np.maximum(E, -100), -100)
    Wc = aw.reshape(w.N, C, 32).sum(axis=2)     # sum of |w| per chunk, [N, C]
    b1 = (1 + 2.0 ** -7) * (np.ldexp(1.0, E - 23) @ Wc.T)
    s = xa @ aw.T
    return b1 + (C + 10) * 2.0 ** -24 * (s + b1)


def check_bound(y, y_ref, w, x, what):
    lim = encoding_bound(w, x)
    err = np.abs(np.asarray(y, np.float64) - y_ref.astype(np.float64))
    bad = ~(err <= lim)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outputs outside the encoding bound; "
                             f"first {idx.tolist()}, err {err[bad][:5]}, bound {lim[bad][:5]}")
    return float(np.max(err / np.maximum(lim, 1e-300)))


def outlier_x(rng, M, K, cols, factor, base=1.0):
    x = (rng.standard_normal((M, K)) * base).astype(np.float32)
    x[:, cols] = np.float32(factor * base) * np.where(rng.random((M, len(cols))) < 0.5, -1, 1)
    return x


def adversarial_inputs(w, seed):
    """(name, weights, x[3, K]) cases for one weight matrix."""
    rng = np.random.default_rng(seed)
    K = w.K
    cols = np.arange(K // 32) * 32 + rng.integers(0, 32, K // 32)   # one column per chunk
    wd = with_dead_columns(w, cols)
    out = []
    for e in (10, 15, 20):
        out.append((f"outlier 2^{e} on dead columns", wd, outlier_x(rng, 3, K, cols, 2.0 ** e)))
    out.append(("outlier 2^20, live columns", w, outlier_x(rng, 3, K, cols, 2.0 ** 20)))
    out.append(("tiny rows 2^-40", w, (rng.standard_normal((3, K)) * 2.0 ** -40).astype(np.float32)))
    sub = (rng.standard_normal((3, K)) * 1e-39).astype(np.float32)      # subnormal binary32
    sub[:, ::7] = 0.0
    out.append(("subnormal rows", w, sub))
    out.append(("huge rows 2^60", w, (rng.standard_normal((3, K)) * 2.0 ** 60).astype(np.float32)))
    mixed = (rng.standard_normal((3, K)) * 2.0 ** -30).astype(np.float32)
    mixed[:, cols[::3]] = 1.0e3
    out.append(("tiny chunks beside unit outliers", w, mixed))
    return out


def gemv(torch, w, x, ex_flags=None):
    M, K = x.shape
    y = torch.full((M, w.N), float("nan"), dtype=torch.float32, device="cuda")
    args = (dev(w.codes, torch), dev(w.scales, torch), dev(w.zeros, torch), dev(x, torch), y, M, w.N, K, w.group)
    if ex_flags is None:
        q4.q4gemv_run(*args)
    else:
        q4.q4gemv_run_ex(*args, flags=ex_flags)
    torch.cuda.synchronize()
    return host(y)


# (N, K, g, symmetric, M): the streamed kernel (M = 1 and 2, long matrices), the register-
# resident kernel (M <= 2, short matrices and small K)
STREAMED = [(8192, 4096, 128, False, 1), (7680, 896, 32, False, 1), (4096, 2048, 64, True, 1),
            (8192, 4096, 128, False, 2), (4101, 14336, 32, True, 2), (12288, 4096, 128, False, 3)]
REGISTER_RESIDENT = [(1000, 896, 32, False, 1), (1000, 896, 32, False, 2), (300, 64, 32, False, 2),
                     (64, 4096, 128, True, 1), (777, 128, 64, False, 2)]


@pytest.mark.parametrize("N,K,g,symmetric,M", STREAMED + REGISTER_RESIDENT)
def test_encoding_bound_on_adversarial_activations(torch, N, K, g, symmetric, M):
    w = synth.q4_weights(N + K + g, N, K, g, symmetric=symmetric)
    worst = 0.0
    for name, wv, x in adversarial_inputs(w, N * 3 + K):
        x = x[:M]
        y = gemv(torch, wv, x)
        assert np.all(np.isfinite(y)), name
        y_ref, _ = oracle.q4_gemv(wv.codes, wv.scales, wv.zeros, x, g)
        worst = max(worst, check_bound(y, y_ref, wv, x, f"{name} N={N} K={K} g={g} M={M}"))
    assert worst <= 1.0


def test_encoding_bound_grouped(torch):
    # the six K = 896 matrices of a decode step in one grouped launch, each with its own
    # adversarial x (every matrix gets CTAs of its own; each must keep the bound)
    K, g = 896, 32
    shapes = [896, 128, 128, 4864, 4864, 2048]
    ws = [synth.q4_weights(70 + i, N, K, g, tag="grp") for i, N in enumerate(shapes)]
    cases = [adversarial_inputs(w, 90 + i) for i, w in enumerate(ws)]
    for j in range(len(cases[0])):
        wv = [cases[i][j][1] for i in range(len(ws))]
        xs = [cases[i][j][2][:1] for i in range(len(ws))]
        ys = [torch.full((1, w.N), float("nan"), dtype=torch.float32, device="cuda") for w in wv]
        keep = [(dev(w.codes, torch), dev(w.scales, torch), dev(w.zeros, torch), dev(x, torch)) for w, x in zip(wv, xs)]
        q4.q4gemv_grouped_run([(c, s, z, xd, y, w.N) for (c, s, z, xd), y, w in zip(keep, ys, wv)], K, g)
        torch.cuda.synchronize()
        for i, (w, x, y) in enumerate(zip(wv, xs, ys)):
            y_ref, _ = oracle.q4_gemv(w.codes, w.scales, w.zeros, x, g)
            check_bound(host(y), y_ref, w, x, f"grouped matrix {i}, {cases[0][j][0]}")


@pytest.mark.parametrize("N,K,g,symmetric,M", [(8192, 4096, 128, False, 1), (1000, 896, 32, False, 2),
                                              (7680, 896, 32, False, 1)])
def test_exact_x_flag_meets_stated_tolerance_on_adversarial_activations(torch, N, K, g, symmetric, M):
    # the CUDA-core float kernel: every product exact, rounded once, on every finite input
    w = synth.q4_weights(N + K + g, N, K, g, symmetric=symmetric)
    for name, wv, x in adversarial_inputs(w, N * 3 + K):
        x = x[:M]
        y = gemv(torch, wv, x, ex_flags=q4.Q4_RUN_EXACT_X)
        y_ref, bound = oracle.q4_gemv(wv.codes, wv.scales, wv.zeros, x, g)
        assert_within_bound(y, y_ref, bound, f"exact-x {name} N={N} K={K} M={M}")


def test_typical_activations_stay_far_inside_the_tolerance(torch):
    # on the workloads' N(0, 1) activations the encoding term is a tiny fraction of the
    # stated tolerance (the LM-head shape of the 0.5B set, streamed)
    N, K, g = 151936, 896, 32
    w = synth.q4_weights(3, N, K, g)
    x = synth.activations_f32(3, 1, K)
    y = gemv(torch, w, x)
    rows = np.arange(0, N, 37)
    y_ref, bound = oracle.q4_gemv_rows(w.codes, w.scales, w.zeros, x, g, rows)
    r = assert_within_bound(y[:, rows], y_ref, bound, "0.5B LM head")
    assert r < 0.05, r
