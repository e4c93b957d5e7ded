"""Host-side checks of the C ABI (no GPU needed, no kernel launched).

The library must load, export every function include/q4gemv.h declares, size
packed matrices correctly and reject bad arguments before any launch.  The
rejected calls below fail a check that runs before the first CUDA call, so no
pointer here is ever dereferenced.
"""
import ctypes
import os
import subprocess

import pytest

import gemm_decode_gb300 as q4
from gemm_decode_gb300 import build as q4build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    q4build.build()
    return q4.lib()


def test_library_exports_every_declared_function(L):
    names = q4.exported_names()
    assert set(names) >= {"q4gemv_pack_info", "q4gemv_run", "q4gemm_run", "f32gemv_run",
                          "q4gemv_status_string"}
    for n in names:
        assert hasattr(L, n), f"{n} declared in q4gemv.h but not exported"


def test_only_declared_functions_are_exported(L):
    out = subprocess.run(["nm", "-D", "--defined-only", q4.library_path()],
                         capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert exported == set(q4.exported_names())


def test_library_links_no_oracle():
    out = subprocess.run(["nm", "-D", q4.library_path()], capture_output=True, text=True).stdout
    assert "orc_" not in out


def test_pack_info_sizes(L):
    info = q4.q4gemv_pack_info(151936, 896, 32)
    assert info["blocks_per_row"] == 28
    assert info["codes_bytes"] == 151936 * 448 == 68067328
    assert info["scales_bytes"] == 8508416
    assert info["zeros_row_bytes"] == 14 and info["zeros_bytes"] == 2127104
    assert info["base_alignment"] == 16
    odd = q4.q4gemv_pack_info(4096, 896, 128)       # 7 groups: a pad nibble
    assert odd["blocks_per_row"] == 7 and odd["zeros_row_bytes"] == 4
    big = q4.q4gemv_pack_info(128256, 4096, 128)
    assert big["codes_bytes"] + big["scales_bytes"] + big["zeros_bytes"] == 272928768


@pytest.mark.parametrize("N,K,g", [(-1, 64, 32), (4, 0, 32), (4, 96, 48), (4, 80, 32), (4, 64, 16)])
def test_pack_info_rejects(L, N, K, g):
    info = q4._PackInfo()
    assert L.q4gemv_pack_info(N, K, g, ctypes.byref(info)) == q4.Q4_ERR_INVALID_ARG
    assert L.q4gemv_pack_info(4, 64, 32, None) == q4.Q4_ERR_INVALID_ARG


A = 0x100000  # an aligned address that is never dereferenced (every call fails first)


def test_status_strings(L):
    for s in range(6):
        assert q4.q4gemv_status_string(s)
    assert q4.q4gemv_status_string(99) == "unknown status"


def test_gemv_argument_checks(L):
    r = L.q4gemv_run
    ok_shape = (4, 64, 64, 32)
    # bad scalars
    assert r(A, A, None, A, A, -1, 64, 64, 32, None) == q4.Q4_ERR_INVALID_ARG
    assert r(A, A, None, A, A, 1, 64, 0, 32, None) == q4.Q4_ERR_INVALID_ARG
    assert r(A, A, None, A, A, 1, 64, 96, 64, None) == q4.Q4_ERR_INVALID_ARG
    assert r(A, A, None, A, A, 1, 64, 64, 48, None) == q4.Q4_ERR_INVALID_ARG
    # empty problems are no-ops, whatever the pointers
    assert r(None, None, None, None, None, 0, 64, 64, 32, None) == q4.Q4_OK
    assert r(None, None, None, None, None, 3, 0, 64, 32, None) == q4.Q4_OK
    # M beyond the CUDA-core kernel
    assert r(A, A, None, A, A, 17, 64, 64, 32, None) == q4.Q4_ERR_UNSUPPORTED
    # null and misaligned pointers
    assert r(None, A, None, A, A, 1, 64, 64, 32, None) == q4.Q4_ERR_INVALID_ARG
    assert r(A, None, None, A, A, 1, 64, 64, 32, None) == q4.Q4_ERR_INVALID_ARG
    assert r(A, A, None, None, A, 1, 64, 64, 32, None) == q4.Q4_ERR_INVALID_ARG
    assert r(A, A, None, A, None, 1, 64, 64, 32, None) == q4.Q4_ERR_INVALID_ARG
    assert r(A + 8, A, None, A, A, 1, 64, 64, 32, None) == q4.Q4_ERR_MISALIGNED
    assert r(A, A + 1, None, A, A, 1, 64, 64, 32, None) == q4.Q4_ERR_MISALIGNED
    assert r(A, A, None, A + 4, A, 1, 64, 64, 32, None) == q4.Q4_ERR_MISALIGNED
    assert r(A, A, None, A, A + 2, 1, 64, 64, 32, None) == q4.Q4_ERR_MISALIGNED
    del ok_shape


def test_fused_gemv_argument_checks(L):
    r = L.q4gemv_fused_run
    NONE, SWIGLU = q4.Q4_EPILOGUE_NONE, q4.Q4_EPILOGUE_SWIGLU
    # unknown epilogue, odd N with SwiGLU, a negative or NaN eps with gamma
    assert r(A, A, None, A, A, 1e-6, A, 1, 64, 64, 32, 7, None) == q4.Q4_ERR_INVALID_ARG
    assert r(A, A, None, A, None, 0.0, A, 1, 63, 64, 32, SWIGLU, None) == q4.Q4_ERR_INVALID_ARG
    assert r(A, A, None, A, A, -1e-6, A, 1, 64, 64, 32, NONE, None) == q4.Q4_ERR_INVALID_ARG
    assert r(A, A, None, A, A, float("nan"), A, 1, 64, 64, 32, NONE, None) == q4.Q4_ERR_INVALID_ARG
    # the shape checks of q4gemv_run
    assert r(A, A, None, A, A, 1e-6, A, 1, 64, 96, 64, NONE, None) == q4.Q4_ERR_INVALID_ARG
    assert r(A, A, None, A, A, 1e-6, A, 17, 64, 64, 32, NONE, None) == q4.Q4_ERR_UNSUPPORTED
    # empty problems are no-ops
    assert r(None, None, None, None, None, 1e-6, None, 0, 64, 64, 32, SWIGLU, None) == q4.Q4_OK
    # null and misaligned pointers (gamma: 16-byte aligned)
    assert r(A, A, None, None, A, 1e-6, A, 1, 64, 64, 32, NONE, None) == q4.Q4_ERR_INVALID_ARG
    assert r(A, A, None, A, A, 1e-6, None, 1, 64, 64, 32, NONE, None) == q4.Q4_ERR_INVALID_ARG
    assert r(A, A, None, A, A + 4, 1e-6, A, 1, 64, 64, 32, NONE, None) == q4.Q4_ERR_MISALIGNED
    assert r(A, A, None, A + 4, A, 1e-6, A, 1, 64, 64, 32, NONE, None) == q4.Q4_ERR_MISALIGNED


def test_grouped_argument_checks(L):
    r = L.q4gemv_grouped_run
    S = q4._Segment
    assert r(None, 0, 896, 32, None) == q4.Q4_OK
    assert r(None, 2, 896, 32, None) == q4.Q4_ERR_INVALID_ARG
    assert r((S * 1)(S(A, A, None, A, A, 4)), -1, 896, 32, None) == q4.Q4_ERR_INVALID_ARG
    assert r((S * 1)(S(A, A, None, A, A, 4)), 1, 96, 64, None) == q4.Q4_ERR_INVALID_ARG     # K % g != 0
    assert r((S * 1)(S(A, A, None, A, A, -1)), 1, 896, 32, None) == q4.Q4_ERR_INVALID_ARG
    assert r((S * 1)(S(None, None, None, None, None, 0)), 1, 896, 32, None) == q4.Q4_OK    # empty entry
    assert r((S * 1)(S(A, A, None, None, A, 4)), 1, 896, 32, None) == q4.Q4_ERR_INVALID_ARG
    # a bad entry anywhere rejects the whole call before any launch
    assert r((S * 2)(S(A, A, None, A, A, 4), S(A, A, None, A + 4, A, 4)), 2, 896, 32, None) == q4.Q4_ERR_MISALIGNED
    assert r((S * 2)(S(A, A, None, A, A, 4), S(A + 8, A, None, A, A, 4)), 2, 896, 32, None) == q4.Q4_ERR_MISALIGNED


# disjoint aligned address ranges, 1 MiB apart, never dereferenced (every call below
# fails a host check before the first CUDA call)
B0, B1, B2, B3, B4, B5 = (0x10000000 + i * 0x100000 for i in range(6))


def test_outputs_must_not_overlap_inputs(L):
    r = L.q4gemv_run
    M, N, K, g = 1, 64, 64, 32
    # y on x, on the codes, on the scales, on the zero points; y ending where x starts is fine
    # (that call would launch, so it is not made here: the overlap rules are the checks)
    assert r(B0, B1, B2, B3, B3, M, N, K, g, None) == q4.Q4_ERR_INVALID_ARG
    assert r(B0, B1, B2, B3, B0 + 16, M, N, K, g, None) == q4.Q4_ERR_INVALID_ARG
    assert r(B0, B1, B2, B3, B1, M, N, K, g, None) == q4.Q4_ERR_INVALID_ARG
    assert r(B0, B1, B2, B3, B2, M, N, K, g, None) == q4.Q4_ERR_INVALID_ARG
    # the last byte of x (4 M K bytes from B3) overlapping the first of y
    assert r(B0, B1, B2, B3, B3 + 4 * K - 4, M, N, K, g, None) == q4.Q4_ERR_INVALID_ARG
    f = L.q4gemv_fused_run
    assert f(B0, B1, None, B3, B4, 1e-6, B4 + 64, 1, N, K, g, q4.Q4_EPILOGUE_NONE, None) == q4.Q4_ERR_INVALID_ARG
    assert L.q4_0_gemv_run(B0, B3, B0 + 32, 1, N, K, None) == q4.Q4_ERR_INVALID_ARG
    assert L.q4gemm_run(B0, B1, None, B3, B3 + 64, 128, N, K, g, None) == q4.Q4_ERR_INVALID_ARG
    assert L.f32gemv_run(B0, B3, B0 + 4 * N * K - 4, 1, N, K, None) == q4.Q4_ERR_INVALID_ARG


def test_grouped_matrices_must_be_independent(L):
    r = L.q4gemv_grouped_run
    S = q4._Segment
    K, g, N = 896, 32, 64
    # a chain: matrix 1 reads the output of matrix 0
    chain = (S * 2)(S(B0, B1, None, B2, B3, N), S(B4, B5, None, B3, B3 + 0x1000, N))
    assert r(chain, 2, K, g, None) == q4.Q4_ERR_INVALID_ARG
    # matrix 0 writes over matrix 1's codes, or over its output
    over_w = (S * 2)(S(B0, B1, None, B2, B4 + 64, N), S(B4, B5, None, B2, B3, N))
    assert r(over_w, 2, K, g, None) == q4.Q4_ERR_INVALID_ARG
    over_y = (S * 2)(S(B0, B1, None, B2, B3, N), S(B4, B5, None, B2, B3 + 128, N))
    assert r(over_y, 2, K, g, None) == q4.Q4_ERR_INVALID_ARG
    # an empty entry takes no part in the check
    empty = (S * 2)(S(B0, B1, None, B2, B3, 0), S(B4, B5, None, B2, B3, N))
    with_alias = (S * 2)(S(B0, B1, None, B2, B2, 0), S(B4, B5, None, B2, B2, N))
    assert r(with_alias, 2, K, g, None) == q4.Q4_ERR_INVALID_ARG
    del empty


def test_per_call_options_are_checked(L):
    O = q4._RunOptions
    ok = (B0, B1, None, B3, B4, 1, 64, 64, 32)
    # an unknown flag or a nonzero reserved field is rejected before anything else
    assert L.q4gemv_run_ex(*ok, ctypes.byref(O(0x80, 0, 0)), None) == q4.Q4_ERR_INVALID_ARG
    assert L.q4gemv_run_ex(*ok, ctypes.byref(O(0, 1, 0)), None) == q4.Q4_ERR_INVALID_ARG
    # the matmul takes the overlapped launch and the wait bound, not the exact-x kernel:
    # with the overlapped flag the options pass and the argument checks run (a misaligned A)
    gm = (B0, B1, None, B3, B4, 128, 64, 64, 32)
    assert L.q4gemm_run_ex(*gm, ctypes.byref(O(q4.Q4_RUN_EXACT_X, 0, 0)), None) == q4.Q4_ERR_INVALID_ARG
    assert L.q4gemm_run_ex(B0, B1, None, B3 + 2, B4, 128, 64, 64, 32,
                           ctypes.byref(O(q4.Q4_RUN_OVERLAPPED | q4.Q4_RUN_WAIT_TIMEOUT, 0, 5)), None) \
        == q4.Q4_ERR_MISALIGNED
    # valid options, then the usual argument checks
    good = ctypes.byref(O(q4.Q4_RUN_OVERLAPPED | q4.Q4_RUN_EXACT_X | q4.Q4_RUN_WAIT_TIMEOUT, 0, 5))
    assert L.q4gemv_run_ex(B0, B1, None, B3, B4, 17, 64, 64, 32, good, None) == q4.Q4_ERR_UNSUPPORTED
    assert L.q4gemv_run_ex(B0, B1, None, B3, B3, 1, 64, 64, 32, None, None) == q4.Q4_ERR_INVALID_ARG
    assert L.q4gemv_run_ex(None, None, None, None, None, 0, 64, 64, 32, good, None) == q4.Q4_OK
    assert L.q4gemv_fused_run_ex(B0, B1, None, B3, None, 0.0, B4, 1, 63, 64, 32, q4.Q4_EPILOGUE_SWIGLU, good,
                                 None) == q4.Q4_ERR_INVALID_ARG
    S = q4._Segment
    assert L.q4gemv_grouped_run_ex((S * 1)(S(B0, B1, None, B2, B3, 4)), 1, 96, 64, good, None) == \
        q4.Q4_ERR_INVALID_ARG
    assert L.q4gemm_run_ex(B0, B1, None, B3 + 2, B4, 128, 64, 64, 32, None, None) == q4.Q4_ERR_MISALIGNED
    # the binding's form
    with pytest.raises(q4.Q4Error):
        q4.q4gemv_run_ex(B0, B1, None, B3, B4, 1, 64, 64, 32, flags=0x100, stream=0)
    assert q4.q4gemv_run_ex(B0, B1, None, B3, B4, 1, 64, 64, 32, flags=0, _reserved=3, stream=0,
                            check=False) == q4.Q4_ERR_INVALID_ARG


def test_q40_argument_checks(L):
    r = L.q4_0_gemv_run
    assert r(A, A, A, 1, 64, 48, None) == q4.Q4_ERR_INVALID_ARG      # K not a multiple of 32
    assert r(A, A, A, -1, 64, 64, None) == q4.Q4_ERR_INVALID_ARG
    assert r(A, A, A, 17, 64, 64, None) == q4.Q4_ERR_UNSUPPORTED
    assert r(None, None, None, 0, 64, 64, None) == q4.Q4_OK
    assert r(None, A, A, 1, 64, 64, None) == q4.Q4_ERR_INVALID_ARG
    assert r(A + 1, A, A, 1, 64, 64, None) == q4.Q4_ERR_MISALIGNED    # blocks: 2-byte aligned
    assert r(A + 2, A + 4, A, 1, 64, 64, None) == q4.Q4_ERR_MISALIGNED  # x: 16-byte aligned


def test_q80_argument_checks(L):
    r = L.q8_0_gemv_run
    assert r(A, A, A, 1, 64, 48, None) == q4.Q4_ERR_INVALID_ARG      # K not a multiple of 32
    assert r(A, A, A, -1, 64, 64, None) == q4.Q4_ERR_INVALID_ARG
    assert r(A, A, A, 17, 64, 64, None) == q4.Q4_ERR_UNSUPPORTED
    assert r(None, None, None, 0, 64, 64, None) == q4.Q4_OK
    assert r(None, A, A, 1, 64, 64, None) == q4.Q4_ERR_INVALID_ARG
    assert r(A + 1, A, A, 1, 64, 64, None) == q4.Q4_ERR_MISALIGNED    # blocks: 2-byte aligned
    assert r(A + 2, A + 4, A, 1, 64, 64, None) == q4.Q4_ERR_MISALIGNED  # x: 16-byte aligned
    assert r(B0, B3, B0 + 64, 1, 64, 64, None) == q4.Q4_ERR_INVALID_ARG  # y inside the blocks


def test_gemm_and_control_argument_checks(L):
    g = L.q4gemm_run
    assert g(A, A, None, A, A, 1, 64, 100, 32, None) == q4.Q4_ERR_INVALID_ARG
    assert g(A, A, None, None, A, 128, 64, 64, 32, None) == q4.Q4_ERR_INVALID_ARG
    assert g(A, A, None, A + 2, A, 128, 64, 64, 32, None) == q4.Q4_ERR_MISALIGNED
    assert g(None, None, None, None, None, 0, 64, 64, 32, None) == q4.Q4_OK
    f = L.f32gemv_run
    assert f(A, A, A, 17, 64, 64, None) == q4.Q4_ERR_UNSUPPORTED
    assert f(A, A, A, 1, 64, 66, None) == q4.Q4_ERR_UNSUPPORTED
    assert f(None, A, A, 1, 64, 64, None) == q4.Q4_ERR_INVALID_ARG
    assert f(A + 4, A, A, 1, 64, 64, None) == q4.Q4_ERR_MISALIGNED
    assert f(None, None, None, 0, 64, 64, None) == q4.Q4_OK
    p = L.vec4_read_probe_run
    assert p(A, 24, A, 1, None, None) == q4.Q4_ERR_INVALID_ARG
    assert p(A + 8, 32, A, 1, None, None) == q4.Q4_ERR_MISALIGNED
    d = L.q4_dequant_f32_run
    assert d(A, A, None, A + 4, 4, 64, 32, None) == q4.Q4_ERR_MISALIGNED
    assert d(A, A, None, None, 4, 64, 32, None) == q4.Q4_ERR_INVALID_ARG


def test_binding_raises_without_library(tmp_path, monkeypatch):
    monkeypatch.setattr(q4, "_lib", None)
    monkeypatch.setattr(q4, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(OSError):
        q4.lib()


def test_overlapped_launch_setting_round_trips(L):
    # host-only state: the call launches nothing
    assert L.q4gemv_set_overlapped_launch(1) == 0
    assert L.q4gemv_set_overlapped_launch(7) == 1
    assert L.q4gemv_set_overlapped_launch(0) == 1
    assert L.q4gemv_set_overlapped_launch(0) == 0


def test_bounds_violations_query_without_checks(L):
    # the product library is built without -DQ4_BOUNDS_CHECK: the query answers -1 and
    # touches no device
    assert L.q4gemv_bounds_violations(None) == -1


def test_binding_rejects_strided_and_mistyped_tensors(L):
    # the binding's checks read tensor metadata only and raise before the library is
    # called, so CPU tensors serve here and nothing is launched
    torch = pytest.importorskip("torch")
    codes = torch.zeros((8, 32), dtype=torch.uint8)
    scales = torch.zeros((8, 2), dtype=torch.int16)
    x = torch.zeros((1, 64), dtype=torch.float32)
    y = torch.zeros((1, 8), dtype=torch.float32)
    strided_x = torch.zeros((1, 128), dtype=torch.float32)[:, ::2]
    with pytest.raises(ValueError, match="x: a contiguous tensor"):
        q4.q4gemv_run(codes, scales, None, strided_x, y, 1, 8, 64, 32)
    with pytest.raises(ValueError, match="y: 4-byte elements"):
        q4.q4gemv_run(codes, scales, None, x, y.to(torch.float64), 1, 8, 64, 32)
    with pytest.raises(ValueError, match="scales_f16: 2-byte elements"):
        q4.q4gemv_run(codes, scales.to(torch.float32), None, x, y, 1, 8, 64, 32)
    with pytest.raises(ValueError, match="codes: 1-byte elements"):
        q4.q4gemm_run(codes.to(torch.int16), scales, None, x.to(torch.bfloat16), y, 1, 8, 64, 32)
    with pytest.raises(ValueError, match="a_bf16: 2-byte elements"):
        q4.q4gemm_run(codes, scales, None, x, y, 1, 8, 64, 32)
    with pytest.raises(ValueError, match="gamma: a contiguous tensor"):
        q4.q4gemv_fused_run(codes, scales, None, x, strided_x[0], 1e-6, y, 1, 8, 64, 32)
    with pytest.raises(ValueError, match="blocks: 1-byte elements"):
        q4.q4_0_gemv_run(torch.zeros((8, 2, 9), dtype=torch.int16), x, y, 1, 8, 64)
    with pytest.raises(ValueError, match="W: a contiguous tensor"):
        q4.f32gemv_run(torch.zeros((64, 8), dtype=torch.float32).t(), x, y, 1, 8, 64)
    with pytest.raises(ValueError, match="wb: 2-byte elements"):
        q4.q4_dequant_bf16_run(codes, scales, None, torch.zeros((8, 64)), 8, 64, 32)


def test_plain_c_client_links_and_runs(L, tmp_path):
    # the header is plain C (and valid C++); a C99 program that includes nothing else
    # links the library and gets the documented results from the calls that need no GPU
    inc = os.path.join(ROOT, "include")
    libdir = os.path.dirname(q4.library_path())
    exe = str(tmp_path / "abi_client")
    subprocess.run(["gcc", "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror", "-I", inc,
                    os.path.join(ROOT, "tests", "abi_client.c"), "-o", exe, "-L", libdir, "-l:libq4gemv.so",
                    "-Wl,-rpath," + libdir], check=True, capture_output=True, text=True)
    subprocess.run(["g++", "-std=c++17", "-Wall", "-Wextra", "-Werror", "-fsyntax-only", "-x", "c++",
                    os.path.join(inc, "q4gemv.h")], check=True, capture_output=True, text=True)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0 and out.stdout.strip() == "ok", out.stdout + out.stderr


def test_grouped_cta_split(L):
    # the split the grouped launch makes, computed on the host by the library's own code:
    # every block of every matrix goes to exactly one CTA (the kernel's split of a matrix's
    # blocks over its CTAs), every CTA gets at least one block, all grid_max CTAs are used
    # when there are more blocks, and moving a CTA between matrices never lowers the
    # largest share
    import random
    rng = random.Random(5)
    rows = {896: 48, 4096: 32}
    for _ in range(400):
        K = rng.choice([896, 4096])
        count = rng.randint(1, 8)
        Ns = [rng.choice([1, 7, 48, 128, 896, 4864, rng.randint(1, 200000)]) for _ in range(count)]
        grid_max = rng.choice([152, 304, 456])
        grid, nb, cb = q4.q4gemv_grouped_split(Ns, K, 32, grid_max)
        assert nb == [-(-n // rows[K]) for n in Ns]
        ends = cb[1:] + [grid]
        c = [e - b for b, e in zip(cb, ends)]
        assert cb[0] == 0 and all(1 <= ci <= nbi for ci, nbi in zip(c, nb))
        assert grid == (sum(nb) if sum(nb) <= grid_max else grid_max)
        for i in range(count):
            covered = []
            for k in range(c[i]):
                b0, b1 = nb[i] * k // c[i], nb[i] * (k + 1) // c[i]
                assert b1 > b0
                covered += range(b0, b1)
            assert covered == list(range(nb[i]))
        worst = max(n / ci for n, ci in zip(nb, c))
        for i in range(count):
            for j in range(count):
                if i != j and c[i] > 1 and c[j] < nb[j]:
                    c2 = list(c)
                    c2[i] -= 1
                    c2[j] += 1
                    assert max(n / ci for n, ci in zip(nb, c2)) >= worst - 1e-12
    with pytest.raises(q4.Q4Error):
        q4.q4gemv_grouped_split([100], 1000, 32, 152)     # K % g != 0
    with pytest.raises(q4.Q4Error):
        q4.q4gemv_grouped_split([0], 896, 32, 152)
