"""Pins for the CPU oracle, independent of the oracle itself (no GPU needed).

Each test fixes the oracle to something it does not compute itself: the
hand-worked fixtures under tests/golden/, numpy/torch library routines for the
number formats and for dense matmul, invariants that follow from the
definition (gerbil kernel reference, "3. MatMulInt4": value = (nibble - zero)
* scale, lowest nibble first), and brute force on tiny inputs written from
unpacked integer arrays.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from conftest import GOLDEN_FILES, golden_x, load_golden, load_golden_blocks, pack_codes, pack_zeros

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# -------------------------------------------------------------- golden values

@pytest.mark.parametrize("name", GOLDEN_FILES)
def test_hand_worked_examples(name):
    d = load_golden(name)
    for kind, y_expect in d["cases"]:
        x = golden_x(kind, d["K"])
        y, _ = oracle.q4_gemv(d["codes"], d["scales"], d["zeros"], x, d["group"])
        np.testing.assert_array_equal(y[0], y_expect)
    if "dequant" in d:
        w = oracle.q4_dequant(d["codes"], d["scales"], d["zeros"], d["K"], d["group"])
        np.testing.assert_array_equal(w[0], d["dequant"])


def test_hand_1x32_symmetric_is_zero8():
    d = load_golden("hand_1x32_g32.txt")
    for kind, y_expect in d["cases"]:
        x = golden_x(kind, d["K"])
        y, _ = oracle.q4_gemv(d["codes"], d["scales"], None, x, d["group"])
        np.testing.assert_array_equal(y[0], y_expect)


def test_hand_examples_through_bf16_matmul():
    # x = 1 and x = k (k < 256) are exact in bfloat16, so the matmul form of the
    # oracle must reproduce the same hand-worked values.
    for name in GOLDEN_FILES:
        d = load_golden(name)
        for kind, y_expect in d["cases"]:
            x = golden_x(kind, d["K"])
            a = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
            c, _ = oracle.q4_gemm(d["codes"], d["scales"], d["zeros"], a, d["group"])
            np.testing.assert_array_equal(c[0], y_expect)


# ------------------------------------------------------------- number formats

def test_fp16_decode_all_patterns_against_numpy():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = h.view(np.float16).astype(np.float32)
    got = np.array([oracle.f16_to_f32(v) for v in h], np.float32)
    finite = np.isfinite(ref)
    np.testing.assert_array_equal(got[finite].view(np.uint32), ref[finite].view(np.uint32))
    assert np.all(np.isnan(got[np.isnan(ref)]))
    assert np.all(got[np.isinf(ref)] == ref[np.isinf(ref)])


def test_bf16_rounding_against_torch():
    r = np.random.default_rng(7)
    vals = r.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** r.integers(-30, 30, 20000).astype(np.float32)
    # exact ties at both parities, the largest finite values and zero signs
    ties = np.array([0x3F808000, 0x3F818000, 0x3F80C000, 0x7F7FFFFF, 0x7F7F8000,
                     0x00008000, 0x80018000, 0x00000000, 0x80000000, 0x3F7FFFFF],
                    np.uint32).view(np.float32)
    vals = np.concatenate([vals[np.isfinite(vals)], ties])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.f32_to_bf16(v) for v in vals], np.uint16)
    np.testing.assert_array_equal(got, ref)
    back = np.array([oracle.bf16_to_f32(v) for v in ref[:500]], np.float32)
    np.testing.assert_array_equal(
        back, torch.from_numpy(ref[:500].view(np.int16)).view(torch.bfloat16).float().numpy())


def test_bf16_nan_stays_nan():
    # a NaN (signalling ones included: the bit patterns go to the routine unchanged) rounds
    # to a bfloat16 NaN, never to an infinity, as torch's conversion does
    import ctypes
    L = oracle.lib()
    for bits in (0x7F800001, 0x7FA00000, 0xFF800001, 0x7FC00000, 0x7FFFFFFF):
        f = ctypes.c_float.from_buffer_copy(np.uint32(bits).tobytes())
        out = L.orc_f32_to_bf16(f)
        assert (out & 0x7F80) == 0x7F80 and (out & 0x7F) != 0, hex(bits)
        ref = torch.from_numpy(np.array([bits], np.uint32).view(np.float32)).to(torch.bfloat16)
        assert torch.isnan(ref).all()


# ------------------------------------------------ definition via numpy routines

def _random_integer_problem(seed, N, K, g, symmetric):
    r = np.random.default_rng(seed)
    q = r.integers(0, 16, size=(N, K))
    nb = K // g
    z = np.full((N, nb), 8) if symmetric else r.integers(0, 16, size=(N, nb))
    s16 = r.uniform(-0.05, 0.05, size=(N, nb)).astype(np.float16)
    codes = pack_codes(q)
    zeros = None if symmetric else pack_zeros(z)
    scales = s16.view(np.uint16).copy()
    # definition, written in numpy on the unpacked integers (binary64)
    W = (q - np.repeat(z, g, axis=1)) * np.repeat(s16.astype(np.float64), g, axis=1)
    return codes, scales, zeros, W


@pytest.mark.parametrize("g", [32, 64, 128])
@pytest.mark.parametrize("symmetric", [False, True])
@pytest.mark.parametrize("N,K_groups", [(1, 1), (3, 3), (5, 7), (17, 2)])
def test_dequant_and_gemv_match_numpy_definition(g, symmetric, N, K_groups):
    K = g * K_groups
    codes, scales, zeros, W = _random_integer_problem(N * 1000 + K + g, N, K, g, symmetric)
    w = oracle.q4_dequant(codes, scales, zeros, K, g)
    # (q - z) * s is exact in binary32: the oracle's dequant must equal it bit for bit
    np.testing.assert_array_equal(w, W.astype(np.float32))
    assert np.all(W.astype(np.float32).astype(np.float64) == W)
    x = np.random.default_rng(K).standard_normal((3, K)).astype(np.float32)
    y, bound = oracle.q4_gemv(codes, scales, zeros, x, g)
    ref = x.astype(np.float64) @ W.T               # numpy binary64 matmul
    mag = np.abs(x.astype(np.float64)) @ np.abs(W.T)
    # both are binary64 sums of the same exact products; after one rounding to
    # binary32 they may differ by at most one unit in the last place
    assert np.all(np.abs(y - ref) <= np.spacing(np.abs(ref).astype(np.float32)) + 1e-30)
    np.testing.assert_allclose(bound, mag, rtol=1e-12, atol=0)


def test_bf16_dequant_matches_torch_rounding():
    codes, scales, zeros, W = _random_integer_problem(3, 4, 256, 64, False)
    wb = oracle.q4_dequant_bf16(codes, scales, zeros, 256, 64)
    ref = torch.from_numpy(W.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(wb, ref)


def test_f32_gemv_matches_numpy():
    W = synth.dense_f32(1, 37, 300)
    x = synth.activations_f32(1, 2, 300)
    y, bound = oracle.f32_gemv(W, x)
    ref = x.astype(np.float64) @ W.astype(np.float64).T
    assert np.all(np.abs(y - ref) <= np.spacing(np.abs(ref).astype(np.float32)) + 1e-30)
    np.testing.assert_allclose(bound, np.abs(x.astype(np.float64)) @ np.abs(W.astype(np.float64)).T,
                               rtol=1e-12)


def test_sum_matches_fsum():
    buf = synth.uniform_f32(3, 100003)
    assert oracle.sum_f32(buf) == math.fsum(buf.astype(np.float64))


# ---------------------------------------------------------------- invariants

@pytest.mark.parametrize("g", [32, 64, 128])
def test_codes_equal_to_zero_point_give_exact_zero(g):
    r = np.random.default_rng(g)
    N, K = 9, 5 * g
    z = r.integers(0, 16, size=(N, K // g))
    q = np.repeat(z, g, axis=1)
    scales = r.uniform(0.001, 0.5, size=(N, K // g)).astype(np.float16).view(np.uint16)
    x = r.standard_normal((2, K)).astype(np.float32) * 100
    y, bound = oracle.q4_gemv(pack_codes(q), scales, pack_zeros(z), x, g)
    assert np.all(y == 0.0) and np.all(bound == 0.0)


def test_symmetric_equals_explicit_zero_eight():
    w = synth.q4_weights(11, 19, 384, 64, symmetric=True)
    z8 = pack_zeros(np.full((19, 6), 8))
    x = synth.activations_f32(11, 2, 384)
    y0, _ = oracle.q4_gemv(w.codes, w.scales, None, x, 64)
    y1, _ = oracle.q4_gemv(w.codes, w.scales, z8, x, 64)
    np.testing.assert_array_equal(y0, y1)


def test_power_of_two_linearity():
    w = synth.q4_weights(12, 7, 256, 32)
    x = synth.activations_f32(12, 1, 256)
    y, _ = oracle.q4_gemv(w.codes, w.scales, w.zeros, x, 32)
    for j in (-3, 1, 5):
        yj, _ = oracle.q4_gemv(w.codes, w.scales, w.zeros, x * np.float32(2.0 ** j), 32)
        np.testing.assert_array_equal(yj, y * np.float32(2.0 ** j))


def test_one_hot_selects_a_column():
    w = synth.q4_weights(13, 6, 192, 64)
    W = oracle.q4_dequant(w.codes, w.scales, w.zeros, 192, 64)
    for k in (0, 1, 63, 64, 127, 191):
        x = np.zeros((1, 192), np.float32)
        x[0, k] = 1.0
        y, _ = oracle.q4_gemv(w.codes, w.scales, w.zeros, x, 64)
        np.testing.assert_array_equal(y[0], W[:, k])


def test_rows_of_x_are_independent():
    w = synth.q4_weights(14, 10, 256, 128)
    x = synth.activations_f32(14, 4, 256)
    y, _ = oracle.q4_gemv(w.codes, w.scales, w.zeros, x, 128)
    for m in range(4):
        ym, _ = oracle.q4_gemv(w.codes, w.scales, w.zeros, x[m:m + 1], 128)
        np.testing.assert_array_equal(ym[0], y[m])


def test_dense_equivalence_inside_the_oracle():
    w = synth.q4_weights(15, 33, 640, 32)
    x = synth.activations_f32(15, 3, 640)
    y, b = oracle.q4_gemv(w.codes, w.scales, w.zeros, x, 32)
    W = oracle.q4_dequant(w.codes, w.scales, w.zeros, 640, 32)
    y2, b2 = oracle.f32_gemv(W, x)
    np.testing.assert_array_equal(y, y2)
    np.testing.assert_array_equal(b, b2)


def test_gemm_equals_gemv_on_widened_activations():
    w = synth.q4_weights(16, 12, 256, 32)
    a = synth.activations_bf16(16, 5, 256)
    c, bc = oracle.q4_gemm(w.codes, w.scales, w.zeros, a, 32)
    xa = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).float().numpy()
    y, by = oracle.q4_gemv(w.codes, w.scales, w.zeros, xa, 32)
    np.testing.assert_array_equal(c, y)
    np.testing.assert_array_equal(bc, by)


def test_sampled_rows_match_full():
    w = synth.q4_weights(17, 50, 384, 128)
    x = synth.activations_f32(17, 2, 384)
    y, b = oracle.q4_gemv(w.codes, w.scales, w.zeros, x, 128)
    rows = [0, 7, 49]
    yr, br = oracle.q4_gemv_rows(w.codes, w.scales, w.zeros, x, 128, rows)
    np.testing.assert_array_equal(yr, y[:, rows])
    yt, bt = oracle.q4_gemv_threaded(w.codes, w.scales, w.zeros, x, 128, 3)
    np.testing.assert_array_equal(yt, y)
    np.testing.assert_array_equal(bt, b)
    np.testing.assert_array_equal(br, b[:, rows])


def test_sampled_matmul_and_control_elements_match_full():
    # the element-sampling forms used at full sizes agree with the whole computation
    w = synth.q4_weights(18, 40, 256, 64)
    a = synth.activations_bf16(18, 5, 256)
    c, cb = oracle.q4_gemm(w.codes, w.scales, w.zeros, a, 64)
    ms, ns = [4, 0, 2], [39, 0, 17]
    cs, csb = oracle.q4_gemm_rows(w.codes, w.scales, w.zeros, a, 64, ms, ns)
    np.testing.assert_array_equal(cs, c[np.ix_(ms, ns)])
    np.testing.assert_array_equal(csb, cb[np.ix_(ms, ns)])
    W = synth.dense_f32(19, 30, 200)
    x = synth.activations_f32(19, 3, 200)
    y, yb = oracle.f32_gemv(W, x)
    ys, ysb = oracle.f32_gemv_rows(W, x, [29, 3, 0])
    np.testing.assert_array_equal(ys, y[:, [29, 3, 0]])
    np.testing.assert_array_equal(ysb, yb[:, [29, 3, 0]])


# ---------------------------------------------------------------- brute force

def _naive_python(q, z, s, x, g):
    """Pure-Python loops over unpacked integers and scale values."""
    N, K = len(q), len(q[0])
    out = []
    for n in range(N):
        acc = 0.0
        for k in range(K):
            acc += (q[n][k] - z[n][k // g]) * s[n][k // g] * x[k]
        out.append(acc)
    return out


@pytest.mark.parametrize("g", [32, 64, 128])
def test_brute_force_every_code_and_zero(g):
    r = np.random.default_rng(100 + g)
    cases = [(N, mult) for N in (1, 2, 3) for mult in (1, 2, 3)] + [(1, 16)]
    seen_q, seen_z = set(), set()
    for N, mult in cases:
        K = g * mult
        q = (np.arange(N * K).reshape(N, K) * 7 + r.integers(0, 16)) % 16
        if mult == 16:
            z = np.arange(16).reshape(1, 16)          # every zero value once
        else:
            z = r.integers(0, 16, size=(N, mult))
        seen_q |= set(q.ravel().tolist())
        seen_z |= set(z.ravel().tolist())
        s16 = r.uniform(-1, 1, size=(N, mult)).astype(np.float16)
        x = r.integers(-4, 5, size=K).astype(np.float32)   # small integers
        ref = _naive_python(q.tolist(), z.tolist(), s16.astype(np.float64).tolist(),
                            x.astype(np.float64).tolist(), g)
        y, _ = oracle.q4_gemv(pack_codes(q), s16.view(np.uint16).copy(), pack_zeros(z),
                              x.reshape(1, K), g)
        # binary64 sums of at most 2048 terms of size < 2^15 * 2^-24 granularity
        # are exact, so both sides round the same real number once
        np.testing.assert_array_equal(y[0], np.array(ref, np.float32))
    assert seen_q == set(range(16)) and seen_z == set(range(16))


def test_code_accessor_nibble_order():
    codes = np.array([[0x21, 0x43]], np.uint8)
    assert [oracle.q4_code(codes, 4, 0, k) for k in range(4)] == [1, 2, 3, 4]


# ---------------------------------------------------------------------------
# The fused decode variants: RMSNorm prologue ("4. RMSNorm" of the kernel
# reference page), SiLU and the SwiGLU combine ("9. SiLU" and its notes).
# ---------------------------------------------------------------------------

SIGMOID_1 = 0.7310585786300049   # 1 / (1 + e^-1), the logistic function at 1


def test_rmsnorm_constant_rows_closed_form():
    # a row of equal values c: mean of squares c^2, so every element becomes
    # c / sqrt(c^2 + eps) * gamma[k]; a row of -c gives the negation
    K, c, eps = 96, 3.0, 0.25
    x = np.full((2, K), c, np.float32)
    x[1] = -c
    gamma = np.random.default_rng(7).uniform(0.5, 2.0, K).astype(np.float32)
    xn = oracle.rmsnorm(x, gamma, eps)
    expect = c / math.sqrt(c * c + eps) * gamma.astype(np.float64)
    np.testing.assert_allclose(xn[0], expect, rtol=1e-15, atol=0)
    np.testing.assert_allclose(xn[1], -expect, rtol=1e-15, atol=0)


def test_rmsnorm_unit_mean_square_and_scale_invariance():
    # with gamma = 1 and eps = 0 the output has mean square 1, and scaling a row by a
    # power of two leaves it unchanged (every step scales exactly)
    K = 640
    x = synth.activations_f32(31, 3, K)
    ones = np.ones(K, np.float32)
    xn = oracle.rmsnorm(x, ones, 0.0)
    np.testing.assert_allclose((xn * xn).mean(axis=1), 1.0, rtol=1e-13, atol=0)
    np.testing.assert_array_equal(oracle.rmsnorm(x * np.float32(4.0), ones, 0.0), xn)


def test_silu_values_and_odd_part():
    assert oracle.silu(0.0) == 0.0
    assert oracle.silu(1.0) == pytest.approx(SIGMOID_1, rel=1e-15)
    # silu(v) - silu(-v) = v (v sigma(v) + v (1 - sigma(v)))
    for v in (-3.0, -0.5, 0.7, 5.0, 20.0):
        assert oracle.silu(v) - oracle.silu(-v) == pytest.approx(v, rel=1e-14)
    assert oracle.silu(60.0) == pytest.approx(60.0, rel=1e-15)
    assert -1e-20 < oracle.silu(-60.0) < 0.0


def test_swiglu_is_silu_of_gate_times_up():
    gate = np.array([[0.0, 1.0, 1.0, -60.0]])
    up = np.array([[5.0, 2.0, -3.0, 7.0]])
    h = oracle.swiglu(gate, up)
    np.testing.assert_allclose(h[0, :3], [0.0, 2.0 * SIGMOID_1, -3.0 * SIGMOID_1], rtol=1e-15, atol=0)
    assert abs(h[0, 3]) < 1e-20


def test_fused_gemv_reduces_to_the_plain_gemv():
    N, K, g = 12, 256, 64
    w = synth.q4_weights(41, N, K, g)
    x = synth.activations_f32(42, 2, K)
    y32, _ = oracle.q4_gemv(w.codes, w.scales, w.zeros, x, g)
    # no normalisation: the binary64 result rounds to the plain oracle's value
    y64, tol = oracle.q4_gemv_fused(w.codes, w.scales, w.zeros, x, None, 0.0, g, False)
    np.testing.assert_array_equal(y64.astype(np.float32), y32)
    # a row of +-1 has root mean square 1: with gamma = 1 and eps = 0 nothing changes
    xs = np.where(x >= 0, 1.0, -1.0).astype(np.float32)
    ys32, _ = oracle.q4_gemv(w.codes, w.scales, w.zeros, xs, g)
    yn, _ = oracle.q4_gemv_fused(w.codes, w.scales, w.zeros, xs, np.ones(K, np.float32), 0.0, g, False)
    np.testing.assert_array_equal(yn.astype(np.float32), ys32)
    # gamma = 2 doubles the normalised input, hence the output, exactly
    y2, _ = oracle.q4_gemv_fused(w.codes, w.scales, w.zeros, xs, np.full(K, 2.0, np.float32), 0.0, g, False)
    np.testing.assert_array_equal(y2, 2.0 * yn)


def test_fused_swiglu_pairs_even_rows_with_odd_rows():
    # rows 2i (gate) and 2i+1 (up) of the weight feed output i
    N, K, g = 10, 128, 32
    w = synth.q4_weights(43, N, K, g)
    x = synth.activations_f32(44, 2, K)
    gamma = np.random.default_rng(9).uniform(0.5, 1.5, K).astype(np.float32)
    y, _ = oracle.q4_gemv_fused(w.codes, w.scales, w.zeros, x, gamma, 1e-5, g, False)
    h, tol = oracle.q4_gemv_fused(w.codes, w.scales, w.zeros, x, gamma, 1e-5, g, True)
    np.testing.assert_array_equal(h, oracle.swiglu(y[:, 0::2], y[:, 1::2]))
    assert h.shape == (2, N // 2) and np.all(tol > 0)
    # the selected-outputs form agrees with the full one
    hs, _ = oracle.q4_gemv_fused(w.codes, w.scales, w.zeros, x, gamma, 1e-5, g, True, outputs=[4, 1])
    np.testing.assert_array_equal(hs, h[:, [4, 1]])


def test_silu_slope_bound():
    # the constant the SwiGLU tolerance uses bounds |d silu / dv| everywhere and is
    # nearly attained (the maximum, about 1.0998, sits near v = 2.4)
    v = np.linspace(-40.0, 40.0, 80001)
    s = np.array([oracle.silu(t) for t in v])
    slope = np.abs(np.diff(s) / np.diff(v))
    assert slope.max() <= oracle.SILU_SLOPE_MAX
    assert slope.max() >= oracle.SILU_SLOPE_MAX - 0.005
    assert 2.3 < v[np.argmax(slope)] < 2.5


def test_swiglu_tolerance_covers_every_pair_within_its_bounds():
    # gate and up moved anywhere within their own GEMV bounds move silu(gate) * up by at
    # most the stated SwiGLU bound (the mean value theorem with the slope bound above);
    # the corners of the box are the extreme points of the product's second factor
    N, K, g = 128, 256, 32
    w = synth.q4_weights(47, N, K, g)
    x = synth.activations_f32(48, 2, K)
    gamma = np.random.default_rng(10).uniform(0.5, 1.5, K).astype(np.float32)
    y, b = oracle.q4_gemv_fused(w.codes, w.scales, w.zeros, x, gamma, 1e-6, g, False)
    h, bound = oracle.q4_gemv_fused(w.codes, w.scales, w.zeros, x, gamma, 1e-6, g, True)
    gate, up, bg, bu = y[:, 0::2], y[:, 1::2], b[:, 0::2], b[:, 1::2]
    worst = 0.0
    r = np.random.default_rng(11)
    for dg, du in [(-1, -1), (-1, 1), (1, -1), (1, 1), (0, 1), (1, 0)] + [tuple(t) for t in r.uniform(-1, 1, (8, 2))]:
        moved = oracle.swiglu(gate + dg * bg, up + du * bu)
        worst = max(worst, float(np.max(np.abs(moved - h) / bound)))
    assert worst <= 1.0
    assert worst >= 0.3    # the bound is not vacuous: some pair comes close to it


# ---------------------------------------------------------------------------
# The second format: Q4_0 blocks (32 elements in 18 bytes: binary16 scale, then
# 16 bytes of 4-bit codes, zero point 8).
# ---------------------------------------------------------------------------

def _q40_from_matmulnbits(codes, scales):
    """Repack symmetric g = 32 MatMulNBits weights into Q4_0 blocks (pure byte moves)."""
    N, half = codes.shape
    nblk = half // 16
    out = np.empty((N, nblk, 18), np.uint8)
    out[:, :, 0] = (scales & 0xFF).astype(np.uint8)
    out[:, :, 1] = (scales >> 8).astype(np.uint8)
    out[:, :, 2:] = codes.reshape(N, nblk, 16)
    return out


def test_q40_hand_worked_block():
    # the 1x32 example: codes q_k = k mod 16 (bytes 10 32 54 76 98 BA DC FE twice),
    # d = 0.5 (binary16 0x3800), zero point 8: x = 1 gives -8, x_k = k gives 216
    blk = np.zeros((1, 1, 18), np.uint8)
    blk[0, 0, 0], blk[0, 0, 1] = 0x00, 0x38
    blk[0, 0, 2:] = [0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE] * 2
    assert [oracle.q40_weight(blk, 32, 0, k) for k in (0, 1, 15, 16, 31)] == [-4.0, -3.5, 3.5, -4.0, 3.5]
    y, _ = oracle.q40_gemv(blk, np.ones((1, 32), np.float32))
    assert y[0, 0] == -8.0
    y, _ = oracle.q40_gemv(blk, np.arange(32, dtype=np.float32).reshape(1, 32))
    assert y[0, 0] == 216.0


def test_q40_equals_symmetric_g32_after_repacking():
    # Q4_0 is the symmetric g = 32 format with scale and codes interleaved per block:
    # the same numbers through the two oracles agree bit for bit
    N, K = 9, 320
    w = synth.q4_weights(51, N, K, 32, symmetric=True)
    blocks = _q40_from_matmulnbits(w.codes, w.scales)
    x = synth.activations_f32(52, 3, K)
    y1, b1 = oracle.q4_gemv(w.codes, w.scales, None, x, 32)
    y2, b2 = oracle.q40_gemv(blocks, x)
    np.testing.assert_array_equal(y1, y2)
    np.testing.assert_array_equal(b1, b2)
    y3, _ = oracle.q40_gemv_rows(blocks, x, [8, 0, 3])
    np.testing.assert_array_equal(y3, y2[:, [8, 0, 3]])


def test_q40_generator_layout():
    b = synth.q40_blocks(3, 4, 64)
    assert b.shape == (4, 2, 18) and b.dtype == np.uint8
    d = (b[:, :, 0].astype(np.uint16) | (b[:, :, 1].astype(np.uint16) << 8)).view(np.float16).astype(np.float32)
    assert np.all((d >= 0.004) & (d <= 0.021))


# ---------------------------------------------------------------------------
# The third format: Q8_0 blocks (32 elements in 34 bytes: binary16 scale, then
# 32 two's-complement int8 codes, no zero point).
# ---------------------------------------------------------------------------

def test_q80_hand_worked_blocks():
    d = load_golden_blocks("hand_q8_0_1x64.txt")
    blocks, K = d["blocks"], d["K"]
    assert blocks.shape == (1, 2, 34)
    w = np.array([oracle.q80_weight(blocks, K, 0, k) for k in range(K)], np.float32)
    np.testing.assert_array_equal(w, d["weights"])
    for kind, y_expect in d["cases"]:
        y, _ = oracle.q80_gemv(blocks, golden_x(kind, K))
        np.testing.assert_array_equal(y[0], y_expect)


def test_q80_equals_q40_on_the_int4_range():
    # Q8_0 codes restricted to -8..7 are Q4_0 codes q + 8 with the same scale: the two
    # oracles agree bit for bit, products, sums and bounds alike
    N, K = 7, 192
    r = np.random.default_rng(61)
    q = r.integers(-8, 8, size=(N, K))
    d = r.uniform(0.005, 0.02, size=(N, K // 32)).astype(np.float16).view(np.uint16)
    b8 = np.empty((N, K // 32, 34), np.uint8)
    b8[:, :, 0], b8[:, :, 1] = d & 0xFF, d >> 8
    b8[:, :, 2:] = (q.reshape(N, K // 32, 32) & 0xFF).astype(np.uint8)
    codes = pack_codes(q + 8).reshape(N, K // 32, 16)
    b4 = np.empty((N, K // 32, 18), np.uint8)
    b4[:, :, 0], b4[:, :, 1] = d & 0xFF, d >> 8
    b4[:, :, 2:] = codes
    x = synth.activations_f32(62, 3, K)
    y8, m8 = oracle.q80_gemv(b8, x)
    y4, m4 = oracle.q40_gemv(b4, x)
    np.testing.assert_array_equal(y8, y4)
    np.testing.assert_array_equal(m8, m4)


def test_q80_weights_against_numpy_views():
    # brute force: every weight of a small matrix decoded by numpy's own int8 and
    # little-endian binary16 views of the same bytes
    N, K = 3, 96
    blocks = synth.q80_blocks(63, N, K)
    d = blocks[:, :, :2].copy().view("<f2")[..., 0].astype(np.float64)
    q = blocks[:, :, 2:].view(np.int8).astype(np.float64)
    w = (q * d[:, :, None]).reshape(N, K)
    got = np.array([[oracle.q80_weight(blocks, K, n, k) for k in range(K)] for n in range(N)], np.float64)
    np.testing.assert_array_equal(got, w)
    assert q.min() < -100 and q.max() > 100      # both signs and the far ends exercised


def test_q80_gemv_against_exact_sums():
    # y is one rounding of the exact sum (math.fsum) up to the f64 accumulation error
    N, K, M = 5, 320, 2
    blocks = synth.q80_blocks(64, N, K)
    x = synth.activations_f32(65, M, K)
    d = blocks[:, :, :2].copy().view("<f2")[..., 0].astype(np.float64)
    w = (blocks[:, :, 2:].view(np.int8).astype(np.float64) * d[:, :, None]).reshape(N, K)
    y, bound = oracle.q80_gemv(blocks, x)
    for m in range(M):
        for n in range(N):
            p = [w[n, k] * float(x[m, k]) for k in range(K)]
            exact = math.fsum(p)
            mag = math.fsum(abs(v) for v in p)
            assert abs(float(y[m, n]) - exact) <= abs(exact) * 2.0 ** -23 + K * 2.0 ** -52 * mag
            assert abs(bound[m, n] - mag) <= K * 2.0 ** -52 * mag
    ys, bs = oracle.q80_gemv_rows(blocks, x, [4, 0, 2])
    np.testing.assert_array_equal(ys, y[:, [4, 0, 2]])
    np.testing.assert_array_equal(bs, bound[:, [4, 0, 2]])


def test_q80_one_hot_and_linearity():
    N, K = 4, 64
    blocks = synth.q80_blocks(66, N, K)
    for k in (0, 31, 32, 63):
        x = np.zeros((1, K), np.float32)
        x[0, k] = 1.0
        y, _ = oracle.q80_gemv(blocks, x)
        np.testing.assert_array_equal(y[0], [oracle.q80_weight(blocks, K, n, k) for n in range(N)])
    x = synth.activations_f32(67, 1, K)
    y1, _ = oracle.q80_gemv(blocks, x)
    y2, _ = oracle.q80_gemv(blocks, x * np.float32(8.0))
    np.testing.assert_array_equal(y2, y1 * np.float32(8.0))


def test_q80_generator_layout():
    b = synth.q80_blocks(3, 4, 64)
    assert b.shape == (4, 2, 34) and b.dtype == np.uint8
    d = (b[:, :, 0].astype(np.uint16) | (b[:, :, 1].astype(np.uint16) << 8)).view(np.float16).astype(np.float32)
    assert np.all((d >= 0.0003) & (d <= 0.00126))


# ---------------------------------------------------------------------------
# The read probe's reference: the binary64 sum of a binary32 buffer.
# ---------------------------------------------------------------------------

def test_probe_sum_closed_forms_and_exact_sum():
    # 1 + 2 + ... + n is exact in binary64 and equals n (n + 1) / 2
    for n in (1, 2, 5, 1000, 4097):
        assert oracle.sum_f32(np.arange(1, n + 1, dtype=np.float32)) == n * (n + 1) / 2
    assert oracle.sum_f32(np.zeros(0, np.float32)) == 0.0
    # against the exactly rounded sum (math.fsum) within the binary64 accumulation error
    buf = synth.uniform_f32(9, 100003)
    exact = math.fsum(float(v) for v in buf)
    assert abs(oracle.sum_f32(buf) - exact) <= len(buf) * 2.0 ** -52 * float(np.abs(buf).sum())
    # a single large element placed last must be counted
    buf = np.ones(64, np.float32)
    buf[-1] = 1024.0
    assert oracle.sum_f32(buf) == 63 + 1024
