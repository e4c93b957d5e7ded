/*
 * q4gemv.h -- C ABI of the GB300 (sm_103a) int4 weight-streaming GEMV library
 * (libq4gemv.so).
 *
 * The operation (gerbil GPU-engine kernel reference, docs/gpu-engine/kernels.md,
 * section "3. MatMulInt4", "Computes" and "Dequantization"):
 *
 *     y[m][n] = sum_k  w[n][k] * x[m][k],     w[n][k] = (q[n][k] - z[n][k/g]) * s[n][k/g]
 *
 * in the MatMulNBits weight layout (Refractometer page, sweep "b) q4 GEMV"):
 *
 *   codes   uint8  [N][K/2]           4-bit codes q, two per byte; the even k is the
 *                                     low nibble ("INT4 Packing": lowest nibble first)
 *   scales  fp16   [N][K/g]           one scale per group of g consecutive k in a row
 *   zeros   uint8  [N][ceil(K/g/2)]   4-bit zero points, two per byte, even group in the
 *                                     low nibble; an odd group count leaves a pad nibble
 *                                     (ignored).  NULL selects the symmetric variant,
 *                                     zero = 8 for every group.
 *
 * Conventions for every call below:
 *   - All arrays are row-major and contiguous.  Pointers marked "device" must point to
 *     device memory (or memory the device can address); the library never dereferences
 *     them on the host.  The caller allocates and owns every buffer; the library keeps
 *     no pointer after a call returns and allocates no device memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *     Calls are asynchronous: they enqueue kernels and return; they never synchronise.
 *   - Arguments are checked on the host before anything is launched.  A failed check
 *     returns a status below and launches nothing.  Outputs are fully overwritten on
 *     success (no accumulation into them, no memset needed).
 *   - M == 0 or N == 0 is an empty problem: Q4_OK, nothing launched, pointers unused.
 *   - Sizes: 1 <= K, K % g == 0, g in {32, 64, 128}.
 *   - Alignment: codes, x, W, a_bf16 and probe buffers 16-byte aligned; scales 2-byte,
 *     y / c 4-byte; otherwise Q4_ERR_MISALIGNED.
 *   - No output may overlap an input or another output of the same call (the kernels
 *     read inputs while other CTAs store results): checked on the host from the byte
 *     ranges the sizes imply, Q4_ERR_INVALID_ARG otherwise.
 *   - A launch failure reported by the CUDA runtime returns Q4_ERR_CUDA (the runtime's
 *     error string is available from q4gemv_last_cuda_error()).
 *
 * Accuracy of the GEMVs (y_exact: the sum in exact arithmetic; inputs finite, results
 * finite).  The stated tolerance is |y - y_exact| <= 1e-3 * sum_k |w_nk x_mk| + 1e-6.
 *   - CUDA-core float kernel (any call with Q4_RUN_EXACT_X; otherwise the shapes no
 *     faster kernel takes): each product (q - z) * s * x is formed exactly and rounded
 *     once, then summed in binary32; within the stated tolerance for every finite input.
 *   - dp4a kernels (M <= 2: the TMA-streamed, register-resident and grouped launches;
 *     M = 3 on the streamed launches where they take it):
 *     x is held per 32-element chunk c as 24-bit integers under one power of two,
 *     2^(E_c - 1) <= max_{k in c} |x_k| < 2^E_c (E_c >= -100), and the dot products are
 *     exact in integers.  Per output
 *         |y - y_exact| <= B1 + (K/32 + 10) * 2^-24 * (sum_k |w_k x_k| + B1),
 *         B1 = (1 + 2^-7) * sum_c 2^(E_c - 23) * sum_{k in c} |w_k|
 *              <= 1.01 * 2^-22 * sum_c (max_{k in c} |x_k|) * (sum_{k in c} |w_k|).
 *     This is inside the stated tolerance unless a chunk of x mixes values thousands of
 *     times apart whose large members meet small weights (B1 stays below
 *     9e-4 * sum |w x| whenever no chunk's largest |x| exceeds about 3700 times the
 *     |w|-weighted mean |x| of its chunk); activations of that kind should use
 *     Q4_RUN_EXACT_X.
 *   - tcgen05 tensor-core GEMV (3 <= M <= 16 on the shapes it takes): each weight is
 *     rounded once to fp16 and x is carried as two fp16 parts, x = hi + lo:
 *         |y - y_exact| <= (2^-11 + 2^-20) * sum_k |w_k x_k|
 *                          + 2^-24 * (sum_k |w_k| + sum_k |x_k|)
 *     plus binary32 accumulation (the last term comes from fp16 subnormals: weights or
 *     parts of x below 2^-14); it needs |x| < 65504 and |(q - z) s| < 65504 (the fp16
 *     range; outside it the output is not finite).
 */
#ifndef Q4GEMV_H
#define Q4GEMV_H

#include <stdint.h>

/* Symbols of this header are the library's only exported (default-visibility) names. */
#if defined(__GNUC__)
#define Q4_API __attribute__((visibility("default")))
#else
#define Q4_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    Q4_OK = 0,
    Q4_ERR_INVALID_ARG = 1, /* null pointer, non-positive K, bad group, K % g != 0 */
    Q4_ERR_UNSUPPORTED = 2, /* valid but outside what a kernel serves (e.g. M > 16 in q4gemv_run) */
    Q4_ERR_MISALIGNED = 3,  /* a pointer violates the alignment stated above */
    Q4_ERR_CUDA = 4,        /* the CUDA runtime refused or failed a launch */
    Q4_ERR_TIMEOUT = 5      /* a bounded device-side wait gave up (mbarrier pipelines) */
} q4_status;

/* Options of one call of the *_ex entry points.  They apply to that call alone: nothing
 * in them outlives the call or reaches another caller (the process-wide setters below
 * only change what the entry points without options do).  A NULL options pointer means
 * flags 0: no overlapped launch, the fastest kernel for the shape, waits bounded at 1 s. */
typedef struct {
    uint32_t flags;            /* bitwise OR of the Q4_RUN_* flags                        */
    uint32_t reserved;         /* must be 0                                               */
    uint64_t wait_timeout_ns;  /* bound on each device-side pipeline wait, read when
                                  flags has Q4_RUN_WAIT_TIMEOUT (0: give up at once)     */
} q4_run_options_t;

/* Overlapped (programmatic dependent) launch of the GEMV kernels: the call's kernel may
 * start streaming its weights while the kernel before it in the stream still runs, and
 * waits for that kernel before it reads x or writes y.  Contract: the kernel that
 * immediately precedes the call in the stream must not write the call's weights. */
#define Q4_RUN_OVERLAPPED 0x1u
/* Run the GEMV on the CUDA-core float kernel, which meets the stated tolerance for every
 * finite input (see "Accuracy" above); slower than the dp4a and tensor-core kernels on
 * long matrices. */
#define Q4_RUN_EXACT_X 0x2u
/* Bound each bounded device-side wait by wait_timeout_ns instead of 1 s. */
#define Q4_RUN_WAIT_TIMEOUT 0x4u

/* Byte sizes of one packed weight matrix (all byte counts). */
typedef struct {
    int64_t n, k;
    int32_t group;
    int32_t blocks_per_row;    /* nb = K / group                         */
    int64_t codes_row_bytes;   /* K / 2                                  */
    int64_t codes_bytes;       /* N * K / 2                              */
    int64_t scales_row_bytes;  /* 2 * nb                                 */
    int64_t scales_bytes;      /* N * 2 * nb                             */
    int64_t zeros_row_bytes;   /* ceil(nb / 2)                           */
    int64_t zeros_bytes;       /* N * ceil(nb / 2)                       */
    int32_t base_alignment;    /* 16: required alignment of codes / x / A */
    int32_t reserved;
} q4gemv_pack_info_t;

/* Fill *out with the packed sizes of an N x K matrix of group g.  Host only; no CUDA
 * call.  Q4_ERR_INVALID_ARG for out == NULL, N < 0, K < 1, g not in {32,64,128} or
 * K % g != 0. */
Q4_API int q4gemv_pack_info(int64_t N, int64_t K, int32_t group, q4gemv_pack_info_t *out);

/* Decode-time int4 GEMV, 1 <= M <= 16 (M > 16: Q4_ERR_UNSUPPORTED):
 * y[m][n] = sum_k (q[n][k] - z[n][k/g]) * s[n][k/g] * x[m][k]
 * (gerbil GPU-engine kernel reference, "3. MatMulInt4": "Computes", "Dequantization").
 *   codes, scales_f16, zeros_u4_or_null : device, layout above
 *   x : device float [M][K], 16-byte aligned;  y : device float [M][N] (written, not
 *   accumulated)
 * The library picks the kernel by shape: a TMA-streamed dp4a kernel for M = 1 and 2 on
 * long matrices (and M = 3 with N >= 12288: rows 0-1 and row 2 as two streamed launches),
 * the tcgen05 tensor-core GEMV for 3 <= M <= 16 on large ones (K split over a
 * thread-block cluster when tiles are few), a register-resident dp4a kernel for M <= 2,
 * and a general CUDA-core kernel (split-K over a cluster for long K / few rows) otherwise;
 * the accuracy each gives is stated at the top of this header.  Launches are overlapped
 * when q4gemv_set_overlapped_launch(1) is in force; waits are bounded by the process-wide
 * q4gemm_set_wait_timeout_ns value.  Asynchronous on `stream`; allocates nothing. */
Q4_API int q4gemv_run(const void *codes, const void *scales_f16, const void *zeros_u4_or_null,
               const float *x, float *y, int32_t M, int64_t N, int64_t K, int32_t group,
               void *stream);

/* q4gemv_run with per-call options (opts may be NULL; see q4_run_options_t).  Flags:
 * Q4_RUN_OVERLAPPED, Q4_RUN_EXACT_X, Q4_RUN_WAIT_TIMEOUT; an unknown flag or a nonzero
 * reserved field is Q4_ERR_INVALID_ARG. */
Q4_API int q4gemv_run_ex(const void *codes, const void *scales_f16, const void *zeros_u4_or_null,
                  const float *x, float *y, int32_t M, int64_t N, int64_t K, int32_t group,
                  const q4_run_options_t *opts, void *stream);

/* Epilogues of q4gemv_fused_run. */
#define Q4_EPILOGUE_NONE 0
#define Q4_EPILOGUE_SWIGLU 1

/* The decode GEMV with its prologue and epilogue fused in (gerbil GPU-engine kernel
 * reference: "4. RMSNorm" -- its optimisation notes suggest fusing RMSNorm into the
 * following MatMul -- and "9. SiLU" -- fusing the SwiGLU combine silu(gate) * up):
 *   gamma : device float [K], 16-byte aligned, or NULL.  Non-NULL: the GEMV's input is
 *           RMSNorm(x)[m][k] = x[m][k] / sqrt(mean_k x[m][k]^2 + eps) * gamma[k]
 *           (eps >= 0; computed as (W . (x * gamma)) / sqrt(...) per row).
 *   epilogue : Q4_EPILOGUE_NONE: y[M][N] as q4gemv_run.
 *              Q4_EPILOGUE_SWIGLU: N even and weight rows 2i / 2i+1 hold the gate / up
 *              projections of output i (interleaved); y[M][N/2] with
 *              y[m][i] = silu(g) * u, silu(v) = v / (1 + exp(-v)).
 * Other arguments as q4gemv_run.  With gamma NULL and no epilogue it is q4gemv_run.
 * Kernels: fused instances of the streamed kernel (M = 1 where q4gemv_run would use it),
 * of the register-resident kernel (other M = 1 shapes it serves without a K split), else
 * of the general CUDA-core kernel without K split, launched once per tile of rows of x
 * whose activations fit in shared memory (Q4_ERR_UNSUPPORTED when not even one row
 * fits: K above about 50 000 on those shapes).  Q4_ERR_INVALID_ARG for an unknown
 * epilogue, odd N with SwiGLU, or a negative or non-finite eps; Q4_ERR_MISALIGNED for
 * an unaligned gamma. */
Q4_API int q4gemv_fused_run(const void *codes, const void *scales_f16, const void *zeros_u4_or_null,
                     const float *x, const float *gamma, float eps, float *y, int32_t M, int64_t N,
                     int64_t K, int32_t group, int32_t epilogue, void *stream);

/* q4gemv_fused_run with per-call options (as q4gemv_run_ex; Q4_RUN_EXACT_X selects the
 * general kernel's fused instances). */
Q4_API int q4gemv_fused_run_ex(const void *codes, const void *scales_f16, const void *zeros_u4_or_null,
                        const float *x, const float *gamma, float eps, float *y, int32_t M, int64_t N,
                        int64_t K, int32_t group, int32_t epilogue, const q4_run_options_t *opts,
                        void *stream);

/* One matrix of a grouped GEMV: its packed weights (as for q4gemv_run), its own input
 * x[K] (device, 16-byte aligned) and output y[N] (device, 4-byte aligned), N >= 0 rows
 * (N == 0: skipped, pointers unused). */
typedef struct {
    const void *codes;
    const void *scales_f16;
    const void *zeros_u4_or_null;
    const float *x;
    float *y;
    int64_t N;
} q4gemv_segment_t;

/* Several M = 1 GEMVs of the same K and group, y_i = W_i x_i, issued as few launches as
 * possible (gerbil GPU-engine kernel reference, section "2. MatMul", its optimisation
 * notes: batch the small Q, K, V projections into one kernel; cera wgpu_gemv_bench.rs,
 * its note on sharing one compute pass: every boundary between dispatches costs time of
 * its own).  Runs of up to 8 matrices that the TMA-streamed kernel serves (K in {896,
 * 2048, 4096, 8192, 16384}; all with or all without zero points; codes, scales and zeros
 * 16-byte aligned; for K = 896 at least one block of 48 rows per SM over the run) are one
 * launch, in which each matrix gets its own CTAs in proportion to its rows; the matrices
 * of any other run each go through q4gemv_run.  The outputs equal those of
 * separate calls within the GEMV's tolerance.  The matrices must be independent: no
 * matrix's y may overlap any matrix's x, codes, scales or zeros, nor another matrix's y
 * (checked, Q4_ERR_INVALID_ARG), so a chain such as segs[1].x == segs[0].y is two calls.
 * segs: host array of count entries (read during the call only).  Every entry is checked
 * as q4gemv_run checks its arguments before anything is launched.  Asynchronous;
 * allocates nothing. */
Q4_API int q4gemv_grouped_run(const q4gemv_segment_t *segs, int32_t count, int64_t K, int32_t group, void *stream);

/* q4gemv_grouped_run with per-call options (as q4gemv_run_ex; Q4_RUN_EXACT_X runs every
 * matrix on the CUDA-core float kernel, one launch each). */
Q4_API int q4gemv_grouped_run_ex(const q4gemv_segment_t *segs, int32_t count, int64_t K, int32_t group,
                          const q4_run_options_t *opts, void *stream);

/* GEMV over a second weight format, Q4_0 blocks (cera wgpu_gemv_bench.rs, block
 * geometry: Q4_0 holds 32 elements in 18 bytes), 1 <= M <= 16:
 * y[m][n] = sum_k (q[n][k] - 8) * d[n][k/32] * x[m][k].
 *   blocks : device, [N][K/32][18] bytes, 2-byte aligned: per block the binary16 scale d
 *            (little-endian), then 16 bytes of 4-bit codes, element 2j in the low nibble
 *            of byte j and element 2j+1 in the high nibble (zero point 8)
 *   x : device float [M][K], 16-byte aligned;  y : device float [M][N]
 * K a multiple of 32.  M = 1 with N >= 4096 and blocks 16-byte aligned runs the
 * TMA-streamed kernel's Q4_0 instances where its ring of row blocks fits shared memory;
 * every other shape the general CUDA-core kernel's (the plan of the symmetric group-32
 * GEMV of the same shape).  Asynchronous; allocates nothing. */
Q4_API int q4_0_gemv_run(const void *blocks, const float *x, float *y, int32_t M, int64_t N, int64_t K,
                  void *stream);

/* GEMV over a third weight format, Q8_0 blocks (cera wgpu_gemv_bench.rs, block geometry:
 * Q8_0 holds 32 elements in 34 bytes), 1 <= M <= 16:
 * y[m][n] = sum_k q[n][k] * d[n][k/32] * x[m][k].
 *   blocks : device, [N][K/32][34] bytes, 2-byte aligned: per block the binary16 scale d
 *            (little-endian), then 32 codes, two's-complement int8, element j at byte 2 + j
 *            (no zero point)
 *   x : device float [M][K], 16-byte aligned;  y : device float [M][N]
 * K a multiple of 32.  M = 1 with N >= 4096 and blocks 16-byte aligned runs the
 * TMA-streamed kernel's Q8_0 instances (dp4a on the byte planes of x: the dp4a kernels'
 * accuracy, with sum |w| = sum |q d|); every other shape a CUDA-core kernel in which each
 * code is widened exactly to binary32, the products of 8 codes of a block with x are summed
 * with fused multiply-adds and each such sum is scaled by d once (the stated tolerance for
 * every finite x).  Asynchronous; allocates nothing. */
Q4_API int q8_0_gemv_run(const void *blocks, const float *x, float *y, int32_t M, int64_t N, int64_t K,
                  void *stream);

/* Prefill-shaped int4 matmul on the tensor cores (tcgen05, bf16 operands, f32
 * accumulate in tensor memory), any M >= 1 (tiles of 128 rows; a partial tile is
 * padded and masked).
 *   a_bf16 : device bfloat16 [M][K] activations;  c : device float [M][N]
 * Each weight is dequantised exactly to f32 and rounded once to bf16 (nearest-even)
 * before the MMA, so each output carries
 *     |c - c_exact| <= (2^-9 + 2e-6) * sum_k |w_nk a_mk| + 1e-6
 * (a bf16 weight is within 2^-9 of the exact one, then binary32 accumulation).  This is
 * up to twice the 1e-3 relative term of the GEMVs' stated tolerance; on prefill-shaped
 * data (K >= 2048, random signs) the errors cancel and the outputs meet it, but not for
 * every input.  The wait bound is the process-wide q4gemm_set_wait_timeout_ns value.
 * Q4_ERR_TIMEOUT if a bounded pipeline wait expired (the kernel then stops; c is
 * unspecified). */
Q4_API int q4gemm_run(const void *codes, const void *scales_f16, const void *zeros_u4_or_null,
               const void *a_bf16, float *c, int32_t M, int64_t N, int64_t K, int32_t group,
               void *stream);

/* q4gemm_run with per-call options (opts may be NULL).  Q4_RUN_OVERLAPPED and
 * Q4_RUN_WAIT_TIMEOUT apply; any other flag or a nonzero reserved field is
 * Q4_ERR_INVALID_ARG.  Overlapped, the matmul may be scheduled while the kernel before it
 * in the stream still runs: it sets up and reads the weight arrays at once and waits for
 * that kernel before it reads a_bf16 or writes c (the contract of the GEMVs' overlapped
 * launch: the weight arrays must not be written by the kernel immediately before it). */
Q4_API int q4gemm_run_ex(const void *codes, const void *scales_f16, const void *zeros_u4_or_null,
                  const void *a_bf16, float *c, int32_t M, int64_t N, int64_t K, int32_t group,
                  const q4_run_options_t *opts, void *stream);

/* Dense f32 GEMV control (cera wgpu_gemv_bench.rs, the F32 row kept in the table as the
 * harness control): y[m][n] = sum_k W[n][k] * x[m][k], 1 <= M <= 16, K % 4 == 0.
 *   W : device float [N][K];  x : device float [M][K];  y : device float [M][N] */
Q4_API int f32gemv_run(const float *W, const float *x, float *y, int32_t M, int64_t N, int64_t K,
                void *stream);

/* Text for a status code (static storage, never NULL). */
Q4_API const char *q4gemv_status_string(int status);

/* The CUDA runtime's error string from the most recent Q4_ERR_CUDA on this thread, or
 * "" (static/thread storage, never NULL). */
Q4_API const char *q4gemv_last_cuda_error(void);

/* Synchronise `stream`, then report and clear the device status word that the
 * tensor-core kernel raises when one of its bounded pipeline waits expires:
 * Q4_OK, Q4_ERR_TIMEOUT (the affected q4gemm_run output is unspecified), or
 * Q4_ERR_CUDA if synchronising failed.  Host-blocking. */
Q4_API int q4gemv_device_status(void *stream);

/* Process-wide default bound, in nanoseconds, on each wait of the tensor-core pipelines
 * and of the TMA-streamed GEMV, for later launches by the entry points without options
 * (default 1e9).  0 makes every wait that is not already satisfied give up at once,
 * which exercises the timeout path without a fault.  Not synchronised with launches in
 * flight; a caller that shares the process should pass Q4_RUN_WAIT_TIMEOUT to the *_ex
 * entry points instead. */
Q4_API int q4gemm_set_wait_timeout_ns(uint64_t ns);

/* Overlapped launch of the GEMV and matmul kernels (programmatic dependent launch).
 * With enable != 0, every later launch by the entry points without options
 * (q4gemv_run, q4gemv_fused_run, q4_0_gemv_run, q8_0_gemv_run, q4gemv_grouped_run,
 * q4gemm_run; for the matmul, a_bf16 and c take the roles of x and y) carries CUDA's programmatic
 * stream serialisation attribute: the kernel may be scheduled while the kernel
 * before it in the stream is still running, and it starts streaming codes, scales
 * and zero points at once; before it reads x or writes y it waits (griddepcontrol.wait)
 * until that kernel has completed and its writes are visible.  Chains of dependent
 * GEMVs (y of one call is x of the next) stay correct; the launch gaps between them
 * shrink.  The contract this adds: the weight arrays of a call must not be written by
 * the kernel that immediately precedes it in the stream (copies and allocations are
 * not affected).  The pages describe one launch per dispatch and have no counterpart;
 * this is a launch policy of this implementation.  Default 0.  Process-wide; it
 * applies to later launches by the entry points without options (a caller that shares
 * the process should pass Q4_RUN_OVERLAPPED to the *_ex entry points instead).
 * Returns the previous setting (0 or 1). */
Q4_API int q4gemv_set_overlapped_launch(int enable);

/* ---- test and measurement exports (not part of the GEMV API proper) ---------------- */

/* Write the dequantised matrix w[N][K] = (q - z) * s as float, with the same in-register
 * decode the GEMV kernels use (exact, so it must equal the CPU definition bit for bit). */
Q4_API int q4_dequant_f32_run(const void *codes, const void *scales_f16, const void *zeros_u4_or_null,
                       float *w, int64_t N, int64_t K, int32_t group, void *stream);

/* Write the bfloat16 weights wb[N][K] the tensor-core path feeds to its MMA
 * (round-to-nearest-even of the exact f32 weight), as uint16 bit patterns. */
Q4_API int q4_dequant_bf16_run(const void *codes, const void *scales_f16, const void *zeros_u4_or_null,
                        uint16_t *wb, int64_t N, int64_t K, int32_t group, void *stream);

/* Read-bandwidth probe (webgpu-bench README "read-bandwidth"; Refractometer
 * "a) bandwidth"): `blocks` CTAs stream `bytes` (a multiple of 16, 16-byte aligned) of
 * float data with 128-bit loads folded by addition; partial[b] receives CTA b's sum.
 * blocks <= 0 picks one CTA per SM times the resident count.  Returns the CTA count
 * used through *blocks_used (may be NULL). */
Q4_API int vec4_read_probe_run(const void *buf, int64_t bytes, float *partial, int32_t blocks,
                        int32_t *blocks_used, void *stream);

/* Bounds-checking builds (compiled with -DQ4_BOUNDS_CHECK, a test-only variant of this
 * library): the streamed, tensor-core and register-resident GEMV kernels check every
 * shared- and global-memory index against its buffer, count each one out of range on a
 * device counter and skip that access.  Synchronise `stream`, then return the count and
 * reset it; -1 in a library built without the checks (the call touches no device then),
 * -Q4_ERR_CUDA if synchronising or reading the counter failed.
 * This is a debugging substitute for a memory checker; the pages have no counterpart. */
Q4_API int q4gemv_bounds_violations(void *stream);

/* Test export (host only, no device call): the CTA split a grouped launch makes for
 * count (1..8) matrices of N[i] >= 1 rows at K and group, given grid_max resident CTAs
 * (CTAs per SM x SMs).  Fills nblocks[i] (blocks of rows of matrix i) and cta_begin[i]
 * (its first CTA; its CTAs run to the next matrix's first, or to the grid) and returns
 * the grid; a negated status for bad arguments or a K without a streamed geometry. */
Q4_API int q4gemv_grouped_split(const int64_t *N, int32_t count, int64_t K, int32_t group, int32_t grid_max,
                                int32_t *nblocks, int32_t *cta_begin);

#ifdef __cplusplus
}
#endif

#endif /* Q4GEMV_H */
