"""GPU parity of the tensor-core GEMV against the CPU oracle.

It serves 3 <= M <= 16 from one whole 128-row tile on (tiles of 128 rows, or of 256 as
two MMAs per CTA where that still fills the GPU): for M >= 5 every matrix of at
least 2^20 weights, for M = 3..4 long rows (K >= 2048, N >= 768) and matrices of at
least 2^24 weights; the cases below pick M and N inside that region.  With few tiles
the K-blocks of each tile are split over a cluster of up to 8 CTAs whose partial sums
are added in rank order (the split cases below).  The kernel dequantises each weight
exactly and rounds it once to fp16 (relative error
<= 2^-11), splits x into fp16 hi + lo parts and accumulates in fp32 in tensor memory.
Every case is checked against the stated tolerance 1e-3*sum|w x| + 1e-6 and against
the tighter bound that follows from that arithmetic, (2^-11 + 2^-18)*sum|w x| + 1e-6.
Marked gpu.
"""
import numpy as np
import pytest

import gemm_decode_gb300 as q4
import oracle
import synth
from gpu_util import assert_within_bound, dev, host, torch_cuda

pytestmark = pytest.mark.gpu

FP16_REL = 2.0 ** -11 + 2.0 ** -18


@pytest.fixture(scope="module")
def torch():
    t = torch_cuda()
    q4.lib()
    return t


def run(torch, w, x):
    M, K = x.shape
    guard = 64
    buf = torch.full((M * w.N + 2 * guard,), 12345.0, dtype=torch.float32, device="cuda")
    y = buf[guard:guard + M * w.N]
    q4.q4gemv_run(dev(w.codes, torch), dev(w.scales, torch), dev(w.zeros, torch), dev(x, torch), y,
                  M, w.N, K, w.group)
    torch.cuda.synchronize()
    b = host(buf)
    assert np.all(b[:guard] == 12345.0) and np.all(b[guard + M * w.N:] == 12345.0), "guard words written"
    return b[guard:guard + M * w.N].reshape(M, w.N)


def check(torch, w, x, what, rows=None):
    y = run(torch, w, x)
    if rows is None:
        y_ref, bound = oracle.q4_gemv(w.codes, w.scales, w.zeros, x, w.group)
        yy = y
    else:
        y_ref, bound = oracle.q4_gemv_rows(w.codes, w.scales, w.zeros, x, w.group, rows)
        yy = y[:, rows]
    assert_within_bound(yy, y_ref, bound, what)
    err = np.abs(yy.astype(np.float64) - y_ref.astype(np.float64))
    lim = FP16_REL * bound + 1e-6
    assert np.all(err <= lim), f"{what}: outside the fp16-weight bound, worst {float(np.max(err / lim)):.3f}"
    return y


@pytest.mark.parametrize("N,K,g", [(8192, 896, 32), (8196, 2048, 64), (8323, 4096, 128), (8192, 4128, 32)])
@pytest.mark.parametrize("symmetric", [False, True])
def test_shapes_against_oracle(torch, N, K, g, symmetric):
    # N = 8196 / 8323: a partial last 128-row tile; K = 4128: a half-empty last K-block;
    # M = 5..8 use 8 rows of x per half (N = 16 MMA), M = 9..16 use 16 (N = 32)
    w = synth.q4_weights(N + K + g, N, K, g, symmetric=symmetric, tag="tc")
    for M in (5, 8, 9, 16):
        x = synth.activations_f32(M * 7 + K, M, K)
        check(torch, w, x, f"M={M} N={N} K={K} g={g} sym={symmetric}")


def _offset_copy(torch, a, offset_bytes):
    """A device copy of uint8/uint16 array `a` whose data starts `offset_bytes` past a
    256-byte boundary (a view into a larger buffer)."""
    raw = np.ascontiguousarray(a).view(np.uint8).reshape(-1)
    buf = torch.zeros(raw.size + 256, dtype=torch.uint8, device="cuda")
    buf[offset_bytes:offset_bytes + raw.size] = torch.from_numpy(raw).cuda()
    return buf[offset_bytes:offset_bytes + raw.size]


@pytest.mark.parametrize("K,g,scale_off,zero_off", [
    (896, 32, 2, 1),      # 28 groups: four-group loads possible, but scales 2 bytes past 8 and zeros odd
    (2048, 64, 6, 0),     # scales 6 bytes past an 8-byte boundary
    (896, 64, 0, 0),      # 14 groups per row: rows of scales only 4-byte aligned
    (896, 128, 0, 0),     # 7 groups per row (a partial last chunk, 4 zero-point bytes per row)
    (4128, 32, 0, 1),     # 129 groups, the last K-block half empty
])
def test_side_data_loaded_one_value_at_a_time(torch, K, g, scale_off, zero_off):
    # Scales and zero points come in chunks of four groups per row: one 8-byte and one
    # 2-byte load where the groups per row are a multiple of 4 and the arrays 8- and
    # 2-byte aligned, else one load per value.  These cases take the second form.
    N = 8192
    w = synth.q4_weights(K + g + scale_off, N, K, g, tag="tc-side")
    sc = _offset_copy(torch, w.scales, scale_off)
    zr = _offset_copy(torch, w.zeros, zero_off)
    for M in (5, 16):
        x = synth.activations_f32(M + K, M, K)
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        q4.q4gemv_run(dev(w.codes, torch), sc.data_ptr(), zr.data_ptr(), dev(x, torch), y, M, N, K, g)
        torch.cuda.synchronize()
        y_ref, bound = oracle.q4_gemv(w.codes, w.scales, w.zeros, x, g)
        assert_within_bound(host(y), y_ref, bound, f"side data one value at a time K={K} g={g} M={M}")
        err = np.abs(host(y).astype(np.float64) - y_ref.astype(np.float64))
        assert np.all(err <= FP16_REL * bound + 1e-6)


@pytest.mark.parametrize("N,K,g,Ms", [(32768, 8192, 32, (4, 16)), (32768, 4096, 128, (8,))])
def test_long_rows_on_256_row_tiles_split_over_clusters(torch, N, K, g, Ms):
    # 128 tiles of 256 rows, each tile's K-blocks split over a cluster of 2 (as many CTAs
    # as 256 tiles of 128 rows, at half the per-weight cost): sampled rows, both ends
    w = synth.q4_weights(N + K + g, N, K, g, tag="tc-256")
    rows = sorted(set(np.random.default_rng(N + K).choice(N, size=160, replace=False).tolist()) | {0, 255, 256, N - 1})
    for M in Ms:
        x = synth.activations_f32(M + K, M, K)
        check(torch, w, x, f"256-row tiles N={N} K={K} g={g} M={M}", rows=rows)


def test_few_rows_of_x_on_a_tall_matrix(torch):
    # M = 3 and 4 take the tensor cores only for N >= 65536
    N, K = 65600, 896
    w = synth.q4_weights(7, N, K, 32, tag="tc-tall")
    rng = np.random.default_rng(4)
    rows = sorted(set(rng.choice(N, size=64, replace=False).tolist()) | {0, 65535, 65536, N - 1})
    for M in (3, 4):
        x = synth.activations_f32(50 + M, M, K)
        check(torch, w, x, f"M={M} N={N}", rows=rows)


@pytest.mark.parametrize("outlier", [10.0, 300.0])
def test_heavy_tailed_activations(torch, outlier):
    N, K = 4096, 2048
    w = synth.q4_weights(5, N, K, 32, tag="tc-tail")
    x = synth.activations_f32(6, 12, K)
    r = np.random.default_rng(3)
    cols = r.choice(K, size=16, replace=False)
    x[:, cols] *= outlier
    check(torch, w, x, f"outlier x{outlier}")


def test_rows_of_x_are_independent(torch):
    # row m of an M-row call equals the call on x[m] alone (M = 1 takes another kernel)
    N, K = 8192, 1024
    w = synth.q4_weights(8, N, K, 64, tag="tc-rows")
    x = synth.activations_f32(9, 5, K)
    y5 = run(torch, w, x)
    for m in range(5):
        y_ref, bound = oracle.q4_gemv(w.codes, w.scales, w.zeros, x[m:m + 1], 64)
        assert_within_bound(y5[m:m + 1], y_ref, bound, f"row {m}")


def test_deterministic(torch):
    w = synth.q4_weights(11, 8192, 896, 32, tag="tc-det")
    x = synth.activations_f32(12, 16, 896)
    a = run(torch, w, x)
    b = run(torch, w, x)
    np.testing.assert_array_equal(a, b)


def test_codes_equal_to_zero_point_give_exact_zero(torch):
    N, K, g = 4096, 512, 32
    w = synth.q4_weights(13, N, K, g, tag="tc-zero")
    nb = K // g
    z = np.zeros((N, nb), np.uint8)
    for n in range(N):
        for b in range(nb):
            z[n, b] = (w.zeros[n, b // 2] >> (4 * (b % 2))) & 0xF
    q = np.repeat(z, g, axis=1)
    codes = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    w0 = synth.Q4Weights(codes, w.scales, w.zeros, N, K, g)
    x = synth.activations_f32(14, 10, K)
    y = run(torch, w0, x)
    assert np.all(y == 0.0)


def test_full_size_lm_head_sampled(torch):
    name, N, K = synth.DECODE_8B["shapes"][3]
    w = synth.q4_weights(31, N, K, 128, scale_range=synth.SCALE_8B, tag=name)
    rng = np.random.default_rng(2)
    rows = sorted(set(rng.choice(N, size=64, replace=False).tolist()) | {0, N - 1})
    for M in (3, 4, 8, 16):
        x = synth.activations_f32(40 + M, M, K)
        check(torch, w, x, f"8B LM head M={M}", rows=rows)


def test_bounded_wait_reports_timeout_without_fault(torch):
    N, K = 151936, 896
    w = synth.q4_weights(21, N, K, 32, tag="tc-timeout")
    x = synth.activations_f32(22, 4, K)
    y = torch.zeros((4, N), dtype=torch.float32, device="cuda")
    q4.q4gemv_run_ex(dev(w.codes, torch), dev(w.scales, torch), dev(w.zeros, torch), dev(x, torch), y,
                     4, N, K, 32, wait_timeout_ns=0)
    st = q4.q4gemv_device_status()
    assert st == q4.Q4_ERR_TIMEOUT
    assert q4.q4gemv_device_status() == q4.Q4_OK   # the flag was cleared
    rows = [0, 1, 4095, 77777, N - 1]
    check(torch, w, x, "after timeout", rows=rows)


@pytest.mark.parametrize("N,K,g,Ms", [
    (4096, 4096, 128, (3, 4, 5, 8, 9, 16)),     # 32 tiles of 128 rows: 8 CTAs per cluster, 8 K-blocks each
    (896, 4864, 32, (3, 8, 16)),                # 7 tiles, 76 K-blocks over 8 CTAs (uneven shares)
    (4099, 14336, 128, (4, 9)),                 # a 3-row last tile, 224 K-blocks
    (1024, 4128, 32, (5, 16)),                  # 65 K-blocks, the last one half empty
    (14336, 4096, 64, (4, 8)),                  # 56 tiles of 256 rows: 4 CTAs per cluster
    (8196, 2048, 32, (5, 16)),                  # 33 tiles of 256 rows, the last 4 rows; 8 CTAs per cluster
    (300, 4864, 64, (5, 13)),                   # 3 tiles, the last one 44 rows
])
@pytest.mark.parametrize("symmetric", [False, True])
def test_split_k_clusters_against_oracle(torch, N, K, g, Ms, symmetric):
    w = synth.q4_weights(N + 3 * K + g, N, K, g, symmetric=symmetric, tag="tc-split")
    rows = None if N <= 4096 else sorted(set(np.random.default_rng(5).choice(N, size=96, replace=False).tolist())
                                         | {0, N - 1})
    for M in Ms:
        x = synth.activations_f32(N + M, M, K)
        check(torch, w, x, f"split N={N} K={K} g={g} M={M} sym={symmetric}", rows=rows)


def test_split_k_deterministic(torch):
    # partial sums are added in rank order: repeated calls agree bit for bit
    w = synth.q4_weights(17, 4096, 14336, 128, tag="tc-split-det")
    x = synth.activations_f32(18, 8, 14336)
    np.testing.assert_array_equal(run(torch, w, x), run(torch, w, x))


def test_split_k_bounded_wait_reports_timeout_without_fault(torch):
    N, K = 4096, 4096
    w = synth.q4_weights(23, N, K, 128, tag="tc-split-timeout")
    x = synth.activations_f32(24, 8, K)
    y = torch.zeros((8, N), dtype=torch.float32, device="cuda")
    q4.q4gemv_run_ex(dev(w.codes, torch), dev(w.scales, torch), dev(w.zeros, torch), dev(x, torch), y, 8, N, K, 128,
                     wait_timeout_ns=0)
    st = q4.q4gemv_device_status()
    assert st == q4.Q4_ERR_TIMEOUT
    assert q4.q4gemv_device_status() == q4.Q4_OK
    check(torch, w, x, "after timeout (split)")
