// q4gemm.cu -- prefill-shaped int4 matmul on the 5th-generation tensor cores.
//
// C[m][n] = sum_k A[m][k] * w[n][k],  w[n][k] = bf16((q[n][k] - z) * s)
// (gerbil GPU-engine kernel reference, "3. MatMulInt4", "Computes" /
// "Dequantization"; its optimisation note "pre-dequantize tiles ... then
// tiled multiply" is what this kernel does, on tcgen05).
//
// One CTA computes an (NH * 128) x 128 tile of C with UMMA (tcgen05.mma,
// kind::f16, bf16 inputs, f32 accumulators in tensor memory), K in blocks of 64.
// With NH = 2 the CTA holds two 128-row halves of A against one dequantised
// weight tile, so each weight tile is dequantised once per 256 rows of A:
//   warp 0      TMA producer: A tile [NH*128 m x 64 k] bf16 -> shared memory,
//               128-byte swizzled, completion counted on an mbarrier;
//   warp 1      allocates NH*128 TMEM columns; one lane issues NH*4 MMAs per
//               K-block (one accumulator per half) and commits them to the
//               stage's "empty" barrier;
//   warps 2..9  dequantisers: each thread turns 32 codes of one weight row
//               into exact binary32 (q - z) * s, rounds to bf16 (nearest
//               even) and stores them in the same swizzled K-major layout
//               the MMA reads; then fence.proxy.async and arrive;
//   warps 2..9  afterwards read the accumulators (tcgen05.ld, one TMEM lane
//               per thread; warp w reads lane quadrant w % 4 of half
//               (w - 2) / 4) and store C in binary32.
// A 4-stage ring of (A, B) tiles overlaps TMA, dequantisation and MMA.
// Every mbarrier wait is bounded by a %globaltimer deadline; on expiry the
// CTA raises a device status flag (read by q4gemv_device_status), stops
// issuing work, drains what it issued and returns, so a broken pipeline
// reports Q4_ERR_TIMEOUT instead of hanging the GPU.
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "q4_common.cuh"
#include "q4_tc.cuh"
#include "q4gemv_stream.cuh"

namespace q4 {

using namespace tc;

__device__ unsigned int g_gemm_status = 0;   // 1 = a bounded wait expired

namespace {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int BK = 64;
constexpr int kDequantWarps = 8;
constexpr int kThreads = (2 + kDequantWarps) * 32;
constexpr int kTileBytes = BM * BK * 2;   // 16 KB: one 128-row half of A, or B

struct GemmArgs {
    const uint8_t *codes;
    const uint16_t *scales;
    const uint8_t *zeros;
    float *c;
    int M, N, K, nb, zrow, gshift;
    int c_vec;   // C is 16-byte aligned and N % 4 == 0: float4 stores
    unsigned long long timeout_ns;
    unsigned int *bounds;   // out-of-range access counter (bounds-checking builds)
};

// Instruction descriptor: D f32, A/B bf16, both K-major, N = BN, M = BM.
constexpr uint32_t kIdesc = idesc_f16(true, BM, BN);

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t accumulate) {
    umma_f16(d_tmem, a_desc, b_desc, kIdesc, accumulate);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

}  // namespace

// NH: 128-row halves of A per CTA (1..4); STAGES: depth of the (A, B) ring.
template <int NH, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
q4gemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_a, const GemmArgs g) {
    // TMEM allocations are powers of two columns, at least 32
    constexpr int kTmemCols = NH * BN <= 128 ? 128 : (NH * BN <= 256 ? 256 : 512);
    constexpr int kATile = NH * kTileBytes;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte aligned tile area (swizzle atoms are address-based)
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char *tiles_a = smem;                               // STAGES x NH x 16 KB
    unsigned char *tiles_b = smem + STAGES * kATile;             // STAGES x 16 KB
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * (kATile + kTileBytes));
    // bars: full_a[S], full_b[S], empty[S], done
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 3 * STAGES + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BN;
    const int m0 = blockIdx.y * (NH * BM);
    const int kblocks = (g.K + BK - 1) / BK;

    const uint32_t bar0 = smem_addr(bars);
    auto full_a = [&](int s) { return bar0 + 8u * s; };
    auto full_b = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto empty = [&](int s) { return bar0 + 8u * (2 * STAGES + s); };
    const uint32_t done_bar = bar0 + 8u * (3 * STAGES);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_a(s), 1);
            mbar_init(full_b(s), kDequantWarps * 32);
            mbar_init(empty(s), 1);
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    allow_next_grid();   // (overlapped launch) the next kernel may be scheduled
    const unsigned long long limit = g.timeout_ns;
    auto ib = [&](bool ok) { return q4_in_bounds(ok, g.bounds); };   // bounds-checking builds

    auto fail = [&]() {
        *abort_flag = 1;
        atomicOr(&g_gemm_status, 1u);
    };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer (A)
        if (lane == 0) {
            // (overlapped launch) A may be written by the kernel before this one in the
            // stream; the weights are read without waiting
            wait_prior_grid();
            int issued = 0;
            for (int kb = 0; kb < kblocks && !*abort_flag; ++kb) {
                const int s = kb % STAGES;
                if (kb >= STAGES && !mbar_wait(empty(s), ((kb / STAGES) - 1) & 1, limit)) {
                    fail();
                    break;
                }
                mbar_expect_tx(full_a(s), kATile);
#pragma unroll
                for (int h = 0; h < NH; ++h)   // one 128-row box per half
                    tma_load_2d(smem_addr(tiles_a + s * kATile + h * kTileBytes), &tmap_a, full_a(s), kb * BK,
                                m0 + h * BM);
                issued = kb + 1;
            }
            if (*abort_flag) {
                // drain (bounded): every issued tile lands before the CTA may exit
                for (int kb = issued - STAGES > 0 ? issued - STAGES : 0; kb < issued; ++kb)
                    mbar_wait(full_a(kb % STAGES), (kb / STAGES) & 1, 50ull * 1000 * 1000);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            for (int kb = 0; kb < kblocks && !*abort_flag; ++kb) {
                const int s = kb % STAGES;
                const uint32_t ph = (kb / STAGES) & 1;
                if (!mbar_wait(full_a(s), ph, limit) || !mbar_wait(full_b(s), ph, limit)) {
                    fail();
                    break;
                }
                tc_fence_after();
                const uint32_t a_base = smem_addr(tiles_a + s * kATile);
                const uint32_t b_base = smem_addr(tiles_b + s * kTileBytes);
#pragma unroll
                for (int h = 0; h < NH; ++h) {
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        // advancing 16 bf16 = 32 bytes inside the 128-byte swizzle span; half h
                        // of A starts 16 KB (16 swizzle atoms) further, its accumulator 128
                        // TMEM columns further
                        umma_bf16(tmem + h * BN, umma_desc(a_base + h * kTileBytes + kk * 32),
                                  umma_desc(b_base + kk * 32), (kb > 0 || kk > 0) ? 1u : 0u);
                    }
                }
                umma_commit(empty(s));
            }
            // all issued MMAs complete -> accumulator ready (also the drain on abort)
            umma_commit(done_bar);
        }
    } else {
        // ------------------------------------------------------------ dequantisers
        const int t = threadIdx.x - 64;            // 0..255
        const int row = t >> 1;                    // B-tile row (weight row n0 + row)
        const int half = t & 1;                    // which 32 codes of the 64-wide K-block
        const int n = n0 + row < g.N ? n0 + row : g.N - 1;
        const uint8_t *crow = g.codes + static_cast<int64_t>(n) * (g.K / 2);
        const uint16_t *srow = g.scales + static_cast<int64_t>(n) * g.nb;
        const uint8_t *zrow = g.zeros ? g.zeros + static_cast<int64_t>(n) * g.zrow : nullptr;
        // codes / scale / zero point of K-block kb, fetched PF blocks ahead
        constexpr int PF = 3;
        struct Fetch {
            uint4 cw;
            uint32_t sc, zb;
        };
        auto fetch = [&](Fetch &f, int kb) {
            const int k = kb * BK + half * 32;
            if (kb < kblocks && k < g.K) {
                const int grp = k >> (5 + g.gshift);
                if (ib(k / 2 + 16 <= g.K / 2)) f.cw = ldg_stream(crow + k / 2);
                if (ib(grp < g.nb)) f.sc = ldg_u16(srow + grp);
                f.zb = (zrow && ib((grp >> 1) < g.zrow)) ? ldg_u8(zrow + (grp >> 1)) : 0u;
            }
        };
        static_assert(PF == 3, "the fetch ring below rotates three registers sets");
        Fetch f0, f1, f2;
        fetch(f0, 0);
        fetch(f1, 1);
        fetch(f2, 2);
        for (int kb = 0; kb < kblocks && !*abort_flag; ++kb) {
            const int s = kb % STAGES;
            const Fetch cur = f0;   // rotate without dynamic indexing (stays in registers)
            f0 = f1;
            f1 = f2;
            fetch(f2, kb + PF);
            if (kb >= STAGES && !mbar_wait(empty(s), ((kb / STAGES) - 1) & 1, limit)) {
                fail();
                break;
            }
            const int k = kb * BK + half * 32;     // first code of this thread's chunk
            uint32_t out[16];
            if (k < g.K) {
                const uint4 cw = cur.cw;
                const int grp = k >> (5 + g.gshift);
                const float sc = half_bits_to_float(cur.sc);
                uint32_t z = 8u;
                if (zrow) z = (grp & 1) ? (cur.zb >> 4) : (cur.zb & 0xFu);
                const ZeroTerms zt = zero_terms(z);
                // s / e_p for the eight positions (exact power-of-two scalings of s)
                const float2 f01 = make_float2(sc, sc * 0x1p-4f), f23 = make_float2(sc * 0x1p-8f, sc * 0x1p-12f);
                const float2 f45 = make_float2(sc * 0x1p-16f, sc * 0x1p-8f),
                             f67 = make_float2(sc * 0x1p-12f, sc * 0x1p-16f);
                const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const WordTerms d = decode_word(words[w], zt);
                    // (e_p (q - z)) * (s / e_p) = (q - z) * s exactly; then one bf16 rounding
                    const float2 v01 = __fmul2_rn(d.d01, f01), v23 = __fmul2_rn(d.d23, f23);
                    const float2 v45 = __fmul2_rn(d.d45, f45), v67 = __fmul2_rn(d.d67, f67);
                    out[4 * w + 0] = pack_bf16(v01.x, v01.y);
                    out[4 * w + 1] = pack_bf16(v23.x, v23.y);
                    out[4 * w + 2] = pack_bf16(v45.x, v45.y);
                    out[4 * w + 3] = pack_bf16(v67.x, v67.y);
                }
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) out[i] = 0u;   // K tail: zero weights
            }
            unsigned char *tb = tiles_b + s * kTileBytes;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const uint32_t off = sw128_offset(row, half * 4 + w);
                if (ib(off + 16 <= static_cast<uint32_t>(kTileBytes)))
                    *reinterpret_cast<uint4 *>(tb + off) =
                        make_uint4(out[4 * w], out[4 * w + 1], out[4 * w + 2], out[4 * w + 3]);
            }
            fence_proxy_async();      // generic-proxy stores -> visible to the tensor core
            mbar_arrive(full_b(s));
        }
        // ------------------------------------------------------------ epilogue
        // warps 2..5 read halves 0, 2, ..., warps 6..9 halves 1, 3, ...
        for (int eh = (warp - 2) >> 2; eh < NH; eh += 2) {
            const int quad = warp & 3;             // TMEM lane quadrant this warp may access
            const int r = quad * 32 + lane;        // accumulator row = TMEM lane
            const bool ok = mbar_wait(done_bar, 0, limit);
            if (!ok) fail();
            wait_prior_grid();   // (overlapped launch) c may be in use by the kernel before this one
            if (ok && !*abort_flag) {
                tc_fence_after();
                const int m = m0 + eh * BM + r;
#pragma unroll 1
                for (int cb = 0; cb < BN / 32; ++cb) {
                    uint32_t v[32];
                    const uint32_t taddr = tmem + (static_cast<uint32_t>(quad * 32) << 16) + eh * BN + cb * 32;
                    asm volatile(
                        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
                          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
                          "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
                          "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
                          "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
                        : "r"(taddr));
                    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                    if (m < g.M) {
                        float *dst = g.c + static_cast<int64_t>(m) * g.N + n0 + cb * 32;
                        const int ncols = g.N - (n0 + cb * 32);
                        if (ncols >= 32 && g.c_vec) {
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                reinterpret_cast<float4 *>(dst)[q] =
                                    make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                                __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
                        } else {
#pragma unroll
                            for (int q = 0; q < 32; ++q)
                                if (q < ncols) dst[q] = __uint_as_float(v[q]);
                        }
                    }
                }
            }
        }
    }
    // ---- teardown: make sure every issued MMA finished before TMEM is released ----
    if (warp == 1 && lane == 0 && *abort_flag) {
        // drain (bounded): the commit on done_bar tracks all MMAs this thread issued
        mbar_wait(done_bar, 0, 50ull * 1000 * 1000);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
    }
}

// ------------------------------------------------------------------ host side

// Address of the tensor-core status word, for kernels in other translation units.
unsigned int *gemm_status_word() {
    static std::atomic<unsigned int *> addr[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    if (addr[dev] == nullptr) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_gemm_status);
        if (e != cudaSuccess) {
            set_cuda_error(e);
            return nullptr;
        }
        addr[dev] = static_cast<unsigned int *>(p);
    }
    return addr[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> fn{nullptr};
    if (fn == nullptr) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        cudaGetLastError();
    }
    return fn;
}

// The split launch (q4gemm_split.cu) for shapes whose 128 x 128 tiles leave most SMs idle.
bool gemm_split_plan(int M, int64_t N, int K, int64_t regular, int &bn, int &split);
int launch_q4gemm_split(const CUtensorMap &map_a, const uint8_t *codes, const uint16_t *scales, const uint8_t *zeros,
                        float *c, int M, int64_t N, int K, int group, int bn, int split, cudaStream_t stream);

// Halves of A per CTA for M rows: the fewest padded rows plus dequantisation, counting
// one dequantised weight tile as much work as 256 rows of MMA (the dequantiser warps,
// not the tensor core, set the pace at the prefill shapes).
static int gemm_halves(int M) {
    int best = 1;
    int64_t best_cost = -1;
    for (int nh = 4; nh >= 1; --nh) {
        const int64_t tiles = (M + nh * BM - 1) / (nh * BM);
        const int64_t cost = tiles * nh * BM + tiles * 2 * BM;
        if (best_cost < 0 || cost < best_cost) {
            best = nh;
            best_cost = cost;
        }
    }
    return best;
}

size_t gemm_smem_bytes(int nh, int stages) {
    return 1024 + static_cast<size_t>(stages) * (nh + 1) * kTileBytes + 8 * (3 * stages + 1) + 16;
}

template <int NH, int STAGES>
static int launch_tc(const CUtensorMap &map, const GemmArgs &g, int M, int64_t N, cudaStream_t stream) {
    static std::atomic<bool> configured[64];
    int dev = 0;
    cudaGetDevice(&dev);
    const size_t smem = gemm_smem_bytes(NH, STAGES);
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(q4gemm_tc_kernel<NH, STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) {
            set_cuda_error(e);
            return Q4_ERR_CUDA;
        }
        configured[dev] = true;
    }
    const dim3 grid(static_cast<unsigned>((N + BN - 1) / BN), static_cast<unsigned>((M + NH * BM - 1) / (NH * BM)));
    if (grid.y > 65535) return Q4_ERR_UNSUPPORTED;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    add_overlap_attr(cfg, attr);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, q4gemm_tc_kernel<NH, STAGES>, map, g);
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return Q4_ERR_CUDA;
    }
    return launch_status();
}

int launch_q4gemm(const uint8_t *codes, const uint16_t *scales, const uint8_t *zeros, const uint16_t *a, float *c,
                  int M, int64_t N, int K, int group, cudaStream_t stream) {
    if (K % 8 != 0) return Q4_ERR_UNSUPPORTED;   // TMA row pitch must be a multiple of 16 bytes
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (encode == nullptr) return Q4_ERR_CUDA;
    // 128-row halves of A per CTA: each dequantised weight tile then serves nh * 128 rows
    const int nh = gemm_halves(M);
    CUtensorMap map;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    const cuuint32_t box[2] = {BK, BM};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = encode(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(a), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return Q4_ERR_UNSUPPORTED;
    {   // few tiles (e.g. 128 tokens x 512 weight rows): narrower tiles with K split over a cluster
        const int64_t regular = ((N + BN - 1) / BN) * ((M + nh * BM - 1) / (nh * BM));
        int bn = 0, split = 1;
        if (gemm_split_plan(M, N, K, regular, bn, split))
            return launch_q4gemm_split(map, codes, scales, zeros, c, M, N, K, group, bn, split, stream);
    }
    GemmArgs g;
    g.codes = codes;
    g.scales = scales;
    g.zeros = zeros;
    g.c = c;
    g.M = M;
    g.N = static_cast<int>(N);
    g.K = K;
    g.nb = K / group;
    g.zrow = (g.nb + 1) / 2;
    g.gshift = group == 32 ? 0 : (group == 64 ? 1 : 2);
    g.c_vec = (aligned(c, 16) && (N % 4) == 0) ? 1 : 0;
    g.timeout_ns = call_options().wait_ns;
    g.bounds = bounds_counter();
    switch (nh) {
        case 4: return launch_tc<4, 2>(map, g, M, N, stream);
        case 3: return launch_tc<3, 3>(map, g, M, N, stream);
        case 2: return launch_tc<2, 4>(map, g, M, N, stream);
        default: return launch_tc<1, 4>(map, g, M, N, stream);
    }
}

int read_device_status(cudaStream_t stream) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return Q4_ERR_CUDA;
    }
    unsigned int v = 0, w = 0;
    e = cudaMemcpyFromSymbol(&v, g_gemm_status, sizeof v);
    if (e != cudaSuccess || read_and_clear_stream_status(&w) != Q4_OK) {
        set_cuda_error(e != cudaSuccess ? e : cudaGetLastError());
        return Q4_ERR_CUDA;
    }
    if (v != 0) {
        const unsigned int zero = 0;
        cudaMemcpyToSymbol(g_gemm_status, &zero, sizeof zero);
    }
    return (v != 0 || w != 0) ? Q4_ERR_TIMEOUT : Q4_OK;
}

}  // namespace q4
