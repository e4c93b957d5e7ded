// q4gemm_split.cu -- the prefill-shaped int4 matmul on the tensor cores for shapes
// whose 128 x 128 tiles are too few to occupy the GPU (such as 128 tokens against 512
// weight rows: four tiles on 152 SMs).
//
// C[m][n] = sum_k A[m][k] * w[n][k],  w[n][k] = bf16((q[n][k] - z) * s)
// (gerbil GPU-engine kernel reference, "3. MatMulInt4", "Computes" / "Dequantization";
// the Refractometer page's tiled-matmul sweep names this 128 x 2048 x 512 shape as the
// one where too few workgroups leave the device idle).
//
// Each tile is 128 rows of A by BN = 32 or 64 weight rows, and the K-blocks of a tile
// are split over a thread-block cluster of S CTAs (S = 1, 2, 4 or 8, grid x), each
// accumulating its own K range in its own tensor memory:
//   warp 0      TMA producer: the 128 x 64 bf16 A tile of each K-block -> shared
//               memory (128-byte swizzle), completion counted on an mbarrier;
//   warp 1      allocates the accumulator's TMEM columns; one lane issues 4 MMAs
//               (M = 128, N = BN, K = 16) per K-block and commits them to the stage's
//               "empty" barrier;
//   warps 2..5  dequantisers: each thread turns BN / 2 codes of one weight row into
//               exact binary32 (q - z) * s, rounds to bf16 (nearest even) and stores
//               them in the swizzled K-major layout the MMA reads; then one lane
//               quadrant each of the accumulator (tcgen05.ld), each row pushed by
//               16-byte stores into the shared memory of the cluster CTA that owns it.
// Row r of the tile belongs to CTA r / (128 / S) of the cluster, which receives the S
// partials of its rows in S slots (distributed shared memory); after one cluster
// barrier it adds them in rank order (deterministic; nothing but C goes to global
// memory).  A relaxed cluster arrive right after set-up, waited on before the first
// store into a peer, makes sure every CTA of the cluster has started before its shared
// memory is written.  Every mbarrier wait is bounded by %globaltimer; on expiry the CTA
// raises the device status word, drains what it issued and still meets both cluster
// barrier phases, so a broken pipeline reports Q4_ERR_TIMEOUT instead of hanging.
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include "q4_common.cuh"
#include "q4_tc.cuh"

namespace q4 {

using namespace tc;
namespace cg = cooperative_groups;

unsigned int *gemm_status_word();

namespace {

constexpr int SBM = 128;                    // rows of A per tile (the MMA's M)
constexpr int SBK = 64;                     // K per block: one 128-byte row of bf16
constexpr int kSplitStages = 4;             // depth of the (A, B) ring
constexpr int kSplitThreads = 6 * 32;       // producer, MMA issuer, 4 dequantiser warps
constexpr int kATileS = SBM * SBK * 2;      // 16 KB

struct SplitArgs {
    const uint8_t *codes;
    const uint16_t *scales;
    const uint8_t *zeros;
    float *c;
    int M, N, K, nb, zrow, gshift;
    int S;                           // CTAs per cluster: the K split
    unsigned long long timeout_ns;   // bound on every mbarrier wait
    unsigned int *status;            // device status word, set to 1 when a wait expires
    unsigned int *bounds;            // out-of-range access counter (bounds-checking builds)
};

// The two halves of a cluster barrier phase (every thread of every CTA of the cluster
// arrives once and waits once per phase).
__device__ __forceinline__ void cluster_arrive_relaxed() { asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// Floats per row of the partial-sum slots: BN plus 4 (rows stay 16-byte aligned for
// vector stores and start in different banks).
template <int BN>
constexpr int split_rld() {
    return BN + 4;
}

template <int BN>
constexpr size_t split_smem_bytes() {
    return 1024 + static_cast<size_t>(kSplitStages) * (kATileS + BN * SBK * 2) +
           static_cast<size_t>(SBM) * split_rld<BN>() * 4 + 8 * (3 * kSplitStages + 1) + 16;
}

}  // namespace

template <int BN>
__global__ void __launch_bounds__(kSplitThreads, 1)
q4gemm_split_kernel(const __grid_constant__ CUtensorMap tmap_a, const SplitArgs g) {
    static_assert(BN == 32 || BN == 64, "32 or 64 weight rows per tile");
    constexpr int kBTile = BN * SBK * 2;         // bf16 weights per K-block: 4 or 8 KB
    constexpr int kTmemCols = BN;                // f32 accumulator columns (a power of two >= 32)
    constexpr int RLD = split_rld<BN>();         // floats per row of the partial-sum slots
    constexpr int CPT = BN / 2;                  // codes per dequantiser thread and K-block
    constexpr int WPT = CPT / 8;                 // 32-bit code words per thread: 2 or 4
    constexpr int TPR = SBK / CPT;               // dequantiser threads per weight row: 4 or 2
    constexpr uint32_t kIdesc = idesc_f16(true, SBM, BN);
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char *tiles_a = smem;                                   // stages x 16 KB
    unsigned char *tiles_b = smem + kSplitStages * kATileS;          // stages x kBTile
    // partial-sum slots: [S][128 / S][RLD], slot q holding CTA q's partials of this CTA's rows
    float *red = reinterpret_cast<float *>(tiles_b + kSplitStages * kBTile);
    uint64_t *bars = reinterpret_cast<uint64_t *>(red + SBM * RLD);  // full_a[S], full_b[S], empty[S], done
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 3 * kSplitStages + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    cg::cluster_group cluster = cg::this_cluster();
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int split = g.S;
    const int rank = split > 1 ? static_cast<int>(cluster.block_rank()) : 0;
    const int n0 = static_cast<int>(blockIdx.y) * BN;
    const int m0 = static_cast<int>(blockIdx.z) * SBM;
    const int kblocks = (g.K + SBK - 1) / SBK;
    const int kb_begin = kblocks * rank / split, kb_end = kblocks * (rank + 1) / split;
    const int nkb = kb_end - kb_begin;
    const unsigned long long limit = g.timeout_ns;
    auto ib = [&](bool ok) { return q4_in_bounds(ok, g.bounds); };   // bounds-checking builds

    const uint32_t bar0 = smem_addr(bars);
    auto full_a = [&](int s) { return bar0 + 8u * s; };
    auto full_b = [&](int s) { return bar0 + 8u * (kSplitStages + s); };
    auto empty = [&](int s) { return bar0 + 8u * (2 * kSplitStages + s); };
    const uint32_t done_bar = bar0 + 8u * (3 * kSplitStages);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kSplitStages; ++s) {
            mbar_init(full_a(s), 1);
            mbar_init(full_b(s), 4 * 32);
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
    if (split > 1) cluster_arrive_relaxed();   // phase 1: this CTA has started (waited on before any push)

    auto fail = [&]() {
        *abort_flag = 1;
        atomicOr(g.status, 1u);
    };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer (A)
        if (lane == 0) {
            // (overlapped launch) A may be written by the kernel before this one in the
            // stream; the weights are read without waiting
            wait_prior_grid();
            int issued = 0;
            for (int j = 0; j < nkb && !*abort_flag; ++j) {
                const int s = j % kSplitStages;
                if (j >= kSplitStages && !mbar_wait(empty(s), ((j / kSplitStages) - 1) & 1, limit)) {
                    fail();
                    break;
                }
                mbar_expect_tx(full_a(s), kATileS);
                tma_load_2d(smem_addr(tiles_a + s * kATileS), &tmap_a, full_a(s), (kb_begin + j) * SBK, m0);
                issued = j + 1;
            }
            if (*abort_flag) {
                // drain (bounded): every issued tile lands before the CTA may exit
                for (int j = issued - kSplitStages > 0 ? issued - kSplitStages : 0; j < issued; ++j)
                    mbar_wait(full_a(j % kSplitStages), (j / kSplitStages) & 1, 50ull * 1000 * 1000);
            }
        }
        __syncwarp();
        if (split > 1) cluster_wait();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            for (int j = 0; j < nkb && !*abort_flag; ++j) {
                const int s = j % kSplitStages;
                const uint32_t ph = (j / kSplitStages) & 1;
                if (!mbar_wait(full_a(s), ph, limit) || !mbar_wait(full_b(s), ph, limit)) {
                    fail();
                    break;
                }
                tc_fence_after();
                const uint32_t a_base = smem_addr(tiles_a + s * kATileS);
                const uint32_t b_base = smem_addr(tiles_b + s * kBTile);
#pragma unroll
                for (int kk = 0; kk < SBK / 16; ++kk)   // 16 bf16 = 32 bytes inside the swizzle span
                    umma_f16(tmem, umma_desc(a_base + kk * 32), umma_desc(b_base + kk * 32), kIdesc,
                             (j > 0 || kk > 0) ? 1u : 0u);
                umma_commit(empty(s));
            }
            umma_commit(done_bar);   // all issued MMAs complete (also the drain on abort)
        }
        __syncwarp();
        if (split > 1) cluster_wait();
    } else {
        // ------------------------------------------------------------ dequantisers
        const int t = threadIdx.x - 64;              // 0..127
        const int row = t / TPR;                     // B-tile row (weight row n0 + row)
        const int part = t - row * TPR;              // which CPT codes of the 64-wide K-block
        const int n = n0 + row < g.N ? n0 + row : g.N - 1;
        const uint8_t *crow = g.codes + static_cast<int64_t>(n) * (g.K / 2);
        const uint16_t *srow = g.scales + static_cast<int64_t>(n) * g.nb;
        const uint8_t *zrow = g.zeros ? g.zeros + static_cast<int64_t>(n) * g.zrow : nullptr;
        struct Fetch {
            uint32_t w[WPT];
            uint32_t sc, zb;
        };
        // codes / scale / zero-point byte of K-block kb (CPT codes lie inside one group)
        auto fetch = [&](Fetch &f, int kb) {
            const int k = kb * SBK + part * CPT;
            if (kb < kb_end && k < g.K) {
                const int grp = k >> (5 + g.gshift);
                if constexpr (WPT == 2) {
                    const uint2 v = *reinterpret_cast<const uint2 *>(crow + k / 2);
                    f.w[0] = v.x;
                    f.w[1] = v.y;
                } else {
                    const uint4 v = ldg_stream(crow + k / 2);
                    f.w[0] = v.x;
                    f.w[1] = v.y;
                    f.w[2] = v.z;
                    f.w[3] = v.w;
                }
                f.sc = ldg_u16(srow + grp);
                f.zb = zrow ? ldg_u8(zrow + (grp >> 1)) : 0u;
            }
        };
        Fetch f0{}, f1{};
        fetch(f0, kb_begin);
        fetch(f1, kb_begin + 1);
        for (int j = 0; j < nkb && !*abort_flag; ++j) {
            const int kb = kb_begin + j;
            const int s = j % kSplitStages;
            const Fetch cur = f0;   // rotate without dynamic indexing (stays in registers)
            f0 = f1;
            fetch(f1, kb + 2);
            if (j >= kSplitStages && !mbar_wait(empty(s), ((j / kSplitStages) - 1) & 1, limit)) {
                fail();
                break;
            }
            const int k = kb * SBK + part * CPT;     // first code of this thread's share
            uint32_t out[4 * WPT];
            if (k < g.K) {
                const int grp = k >> (5 + g.gshift);
                const float sc = half_bits_to_float(cur.sc);
                uint32_t z = 8u;
                if (zrow) z = (grp & 1) ? (cur.zb >> 4) : (cur.zb & 0xFu);
                const ZeroTerms zt = zero_terms(z);
                // s / e_p for the eight positions (exact power-of-two scalings of s)
                const float2 f01 = make_float2(sc, sc * 0x1p-4f), f23 = make_float2(sc * 0x1p-8f, sc * 0x1p-12f);
                const float2 f45 = make_float2(sc * 0x1p-16f, sc * 0x1p-8f),
                             f67 = make_float2(sc * 0x1p-12f, sc * 0x1p-16f);
#pragma unroll
                for (int w = 0; w < WPT; ++w) {
                    const WordTerms d = decode_word(cur.w[w], zt);
                    // (e_p (q - z)) * (s / e_p) = (q - z) * s exactly; then one bf16 rounding
                    const float2 v01 = __fmul2_rn(d.d01, f01), v23 = __fmul2_rn(d.d23, f23);
                    const float2 v45 = __fmul2_rn(d.d45, f45), v67 = __fmul2_rn(d.d67, f67);
                    out[4 * w + 0] = pack_bf16x2(v01.x, v01.y);
                    out[4 * w + 1] = pack_bf16x2(v23.x, v23.y);
                    out[4 * w + 2] = pack_bf16x2(v45.x, v45.y);
                    out[4 * w + 3] = pack_bf16x2(v67.x, v67.y);
                }
            } else {
#pragma unroll
                for (int i = 0; i < 4 * WPT; ++i) out[i] = 0u;   // K tail: zero weights
            }
            unsigned char *tb = tiles_b + s * kBTile;
#pragma unroll
            for (int w = 0; w < WPT; ++w) {   // word w of the share is 16-byte chunk part * WPT + w of the row
                const uint32_t off = sw128_offset(row, part * WPT + w);
                if (ib(off + 16 <= static_cast<uint32_t>(kBTile)))
                    *reinterpret_cast<uint4 *>(tb + off) = make_uint4(out[4 * w], out[4 * w + 1], out[4 * w + 2],
                                                                      out[4 * w + 3]);
            }
            fence_proxy_async();      // generic-proxy stores -> visible to the tensor core
            mbar_arrive(full_b(s));
        }
        // ------------------------------------------------------------ accumulator -> partial tile
        const int quad = warp & 3;                   // TMEM lane quadrant this warp may access
        const int r = quad * 32 + lane;              // accumulator row = TMEM lane = row of A
        const bool ok = mbar_wait(done_bar, 0, limit);
        if (!ok) fail();
        wait_prior_grid();   // (overlapped launch) c may be in use by the kernel before this one
        __syncwarp();
        if (split > 1) cluster_wait();   // every peer has started: its shared memory may be written
        if (ok && !*abort_flag) {
            tc_fence_after();
#pragma unroll
            for (int cb = 0; cb < BN / 32; ++cb) {
                uint32_t v[32];
                const uint32_t taddr = tmem + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(cb * 32);
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
                if (split == 1) {
                    // no K split: this CTA's accumulator is the result
                    const int m = m0 + r;
                    if (m < g.M) {
                        float *dst = g.c + static_cast<int64_t>(m) * g.N;
#pragma unroll
                        for (int q = 0; q < 32; ++q)
                            if (n0 + cb * 32 + q < g.N) dst[n0 + cb * 32 + q] = __uint_as_float(v[q]);
                    }
                } else {
                    // this CTA's partial of row r (0 when its K range is empty: no MMA ran),
                    // into slot `rank` of the CTA that owns the row
                    const int rows_per = SBM / split;
                    const int owner = r / rows_per, rr = r - owner * rows_per;
                    const int idx = (rank * rows_per + rr) * RLD + cb * 32;
                    float *dst = cluster.map_shared_rank(red, owner) + idx;
                    if (ib(idx + 32 <= SBM * RLD)) {
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            reinterpret_cast<float4 *>(dst)[q] =
                                nkb > 0 ? make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                                      __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]))
                                        : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    }
                }
            }
        }
    }
    if (split > 1) {
        // every partial has been pushed to its owner once all CTAs pass this barrier; each
        // CTA then finishes its rows [rank * 128 / S, (rank + 1) * 128 / S) of the tile by
        // adding its S slots in rank order (local reads only, so no second barrier)
        __syncwarp();     // (the producer and MMA lanes rejoin their warps first)
        cluster.sync();
        if (warp >= 2 && !*abort_flag) {
            const int rows_per = SBM / split;
#pragma unroll 4
            for (int i = (warp - 2) * 32 + lane; i < rows_per * BN; i += 4 * 32) {
                const int rr = i / BN, col = i % BN;
                const int m = m0 + rank * rows_per + rr, nn = n0 + col;
                if (m < g.M && nn < g.N) {
                    float acc = 0.0f;
                    for (int q = 0; q < split; ++q)
                        if (ib((q * rows_per + rr) * RLD + col < SBM * RLD)) acc += red[(q * rows_per + rr) * RLD + col];
                    g.c[static_cast<int64_t>(m) * g.N + nn] = acc;
                }
            }
        }
    }
    // ---- teardown: every issued MMA finished before TMEM is released ----
    if (warp == 1 && lane == 0 && *abort_flag) mbar_wait(done_bar, 0, 50ull * 1000 * 1000);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
    }
}

// ------------------------------------------------------------------ host side

// The split launch for M x N x K: tile width BN (32 or 64 weight rows) and K split S
// (1, 2, 4 or 8 CTAs per cluster), chosen for the most CTAs up to one per SM with at
// least two K-blocks per CTA (ties: the wider tile, fewer re-reads of A).  Returns false
// when even that leaves the GPU no better occupied than the 128 x 128 tiles would
// (regular: the CTAs the 128 x 128 kernel launches).
bool gemm_split_plan(int M, int64_t N, int K, int64_t regular, int &bn, int &split) {
    const int64_t sms = device_info().sms;
    if (regular * 2 > sms) return false;   // the regular kernel already fills half the SMs
    const int kblocks = (K + SBK - 1) / SBK;
    const int64_t mtiles = (M + SBM - 1) / SBM;
    if (mtiles > 65535) return false;
    int64_t best = 0;
    for (int cand : {64, 32}) {
        const int64_t ntiles = (N + cand - 1) / cand;
        if (ntiles > 65535) continue;
        int s = 1;
        while (s < 8 && mtiles * ntiles * s * 2 <= sms && kblocks / (2 * s) >= 2) s *= 2;
        const int64_t ctas = mtiles * ntiles * s;
        if (ctas > best) {
            best = ctas;
            bn = cand;
            split = s;
        }
    }
    return best > regular;
}

template <int BN>
static int launch_split(const CUtensorMap &map, const SplitArgs &g, cudaStream_t stream) {
    auto kern = q4gemm_split_kernel<BN>;
    constexpr size_t smem = split_smem_bytes<BN>();
    static std::atomic<bool> configured[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) {
            set_cuda_error(e);
            return Q4_ERR_CUDA;
        }
        configured[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(g.S), static_cast<unsigned>((g.N + BN - 1) / BN),
                       static_cast<unsigned>((g.M + SBM - 1) / SBM));
    cfg.blockDim = dim3(kSplitThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(g.S);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    add_overlap_attr(cfg, attr);
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, map, g);
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return Q4_ERR_CUDA;
    }
    return launch_status();
}

int launch_q4gemm_split(const CUtensorMap &map_a, const uint8_t *codes, const uint16_t *scales, const uint8_t *zeros,
                        float *c, int M, int64_t N, int K, int group, int bn, int split, cudaStream_t stream) {
    SplitArgs g;
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
    g.S = split;
    g.timeout_ns = call_options().wait_ns;
    g.status = gemm_status_word();
    if (g.status == nullptr) return Q4_ERR_CUDA;
    g.bounds = bounds_counter();
    return bn == 64 ? launch_split<64>(map_a, g, stream) : launch_split<32>(map_a, g, stream);
}

}  // namespace q4
