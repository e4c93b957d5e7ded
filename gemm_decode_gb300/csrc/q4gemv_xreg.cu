// q4gemv_xreg.cu -- the streaming int4 GEMV for 1 <= M <= 2 on CUDA cores.
//
// Computes y[m][n] = sum_k (q[n][k] - z[n][k/g]) * s[n][k/g] * x[m][k]
// (gerbil GPU-engine kernel reference, "3. MatMulInt4": "Computes",
// "Dequantization"; MatMulNBits layout per the Refractometer page's
// "b) q4 GEMV" sweep).
//
// Work decomposition.  A row of codes is C = K/32 chunks of 16 bytes (32
// codes, inside one group).  Every thread owns ONE chunk position c for the
// whole launch and keeps the matching 32 values of x in registers; rows stream
// past it.  A CTA has CTp threads per row (CTp = the chunk positions of this
// CTA's K-slice, rounded up to a warp multiple when at least 32) times RG rows,
// so one "row group" of RG rows is covered by one pass of all threads, and an
// iteration covers U row groups.  Each thread copies its own 16-byte code
// chunk, scale word and zero-point word of future iterations into a private
// shared-memory ring with cp.async (D slots), so loads run far ahead of the
// arithmetic without holding registers and without CTA-wide barriers.  The
// per-row partial sums go to shared memory and are reduced every RB
// iterations.  Long rows are split over S CTAs of a thread-block cluster whose
// partials are added in rank order through distributed shared memory.
//
// Arithmetic.  x is represented per 32-element chunk as 24-bit integers
// m_k = round(x_k * 2^(22-E)) with E the exponent of the chunk's largest |x|
// (|m_k| <= 2^22), split into three byte planes.  With the codes unpacked to
// bytes (even k, odd k), dp4a forms sum_k q_k * plane_b(k) exactly in int32 for
// each plane b; the zero point enters exactly as - z * sum_k plane_b(k).  The
// three plane sums are combined in binary32 and scaled once by s * 2^(E-22).
// Every integer step is exact; the only approximations are x's 24-bit chunk
// representation (absolute error <= 2^-23 * 2^E per element) and binary32
// rounding of the per-chunk and per-row sums.  Codes equal to their zero point
// contribute exactly 0.
#include <cooperative_groups.h>
#include <type_traits>

#include "q4_common.cuh"
#include "q4gemv_xreg.cuh"
#include "q4gemv_xplanes.cuh"

namespace q4 {

namespace cg = cooperative_groups;
using namespace xp;


// Compile-time geometry: KC = chunks per row and G = group size when known at
// compile time (0 = read from the arguments); U rows groups per ring iteration
// and D ring slots.
// FUSED (M = 1, no K split): x is encoded multiplied by a.gamma and every output
// multiplied by 1 / sqrt(mean(x^2) + eps) when a.gamma is set (the RMSNorm prologue);
// with a.swiglu the gate / up row pairs leave silu(gate) * up.
template <bool FUSED>
using XregArgsOf = std::conditional_t<FUSED, XregFusedArgs, XregArgs>;

template <int MT, bool ASYM, int CTP, int RG, int KC, int G, int U, int D, bool FUSED = false>
__global__ void __launch_bounds__(CTP * RG)
q4gemv_xreg_kernel(const XregArgsOf<FUSED> a) {
    static_assert(!FUSED || MT == 1, "the fused variant serves one row of x");
    constexpr int T = CTP * RG;
    constexpr bool WARPRED = CTP >= 32;
    constexpr int RED_LD = WARPRED ? CTP / 32 : CTP + 1;
    constexpr int ROWS_IT = U * RG;                     // rows per ring iteration
    constexpr int RB = (64 / ROWS_IT) > 0 ? (64 / ROWS_IT) : 1;     // iterations per reduction batch
    constexpr int ROWS_B = RB * ROWS_IT;
    constexpr int RED_FLOATS = ROWS_B * MT * RED_LD;
    constexpr uint32_t SLOT = U * T * (ASYM ? 24 : 20);  // ring bytes per iteration
    extern __shared__ __align__(16) unsigned char smem[];
    const int tid = threadIdx.x;
    const int r = tid / CTP;            // row within a row group
    const int cl = tid - r * CTP;       // chunk position within this CTA's K-slice
    const int split = KC ? 0 : static_cast<int>(blockIdx.y);
    const int C = KC ? KC : a.C;
    const int K = C * 32;
    const int CT = KC ? KC : a.CT;
    const int nb = G ? K / G : a.nb;
    const int zrow = (nb + 1) / 2;
    const int gshift = G ? (G == 32 ? 0 : (G == 64 ? 1 : 2)) : a.gshift;
    const int c = split * CT + cl;      // chunk position in the row
    // with compile-time geometry every thread holds a real chunk (KC == CTP)
    const bool active = (KC == CTP) || ((cl < CT) && (c < C));

    // shared memory: planes [MT][CTP][28] | red [2][ROWS_B][MT][RED_LD] | ring [D][SLOT] | ysum [ROWS_B][MT]
    uint32_t *planes = reinterpret_cast<uint32_t *>(smem);
    float *red0 = reinterpret_cast<float *>(smem + a.off_red);
    unsigned char *ring = smem + a.off_ring;
    float *ysum = reinterpret_cast<float *>(smem + a.off_ysum);

    const int gsz = static_cast<int>(gridDim.x);
    const int g_begin = static_cast<int>(static_cast<int64_t>(a.nsuper) * blockIdx.x / gsz);
    const int g_end = static_cast<int>(static_cast<int64_t>(a.nsuper) * (blockIdx.x + 1) / gsz);
    const int ng = g_end - g_begin;

    // ---- per-thread streams (loop-carried pointers; per-thread constant shifts) ----
    const int grp = c >> gshift;
    const int64_t row0 = static_cast<int64_t>(g_begin) * ROWS_IT + r;
    const int64_t pitch = K / 2;
    const unsigned char *gc = a.codes + row0 * pitch + static_cast<int64_t>(c) * 16;
    const int64_t se = row0 * nb + grp;                         // scale element index
    const unsigned char *gs = reinterpret_cast<const unsigned char *>(a.scales) + (se & ~1LL) * 2;
    const int ssh = static_cast<int>(se & 1) * 16;
    const int64_t ze = row0 * zrow + (grp >> 1);                // zero-point byte index
    const unsigned char *gz = ASYM ? a.zeros + (ze & ~3LL) : nullptr;
    const int zsh = static_cast<int>(ze & 3) * 8 + (grp & 1) * 4;
    const int64_t rg_c = static_cast<int64_t>(RG) * pitch, rg_s = static_cast<int64_t>(RG) * nb * 2,
                  rg_z = static_cast<int64_t>(RG) * zrow;
    const uint32_t ring_s = static_cast<uint32_t>(__cvta_generic_to_shared(ring));
    const uint32_t my_c = ring_s + tid * 16;
    const uint32_t my_s = ring_s + U * T * 16 + tid * 4;
    const uint32_t my_z = my_s + U * T * 4;

    // bounds-checking builds: every global source lies inside its array (codes 16 bytes,
    // scale and zero-point words 4 bytes), else the copy is counted and skipped
    const int64_t codes_b = static_cast<int64_t>(a.N) * pitch, scales_b = static_cast<int64_t>(a.N) * nb * 2,
                  zeros_b = static_cast<int64_t>(a.N) * zrow;
    auto src_ok = [&](const void *p, const void *base, int64_t size, int bytes) {
        const int64_t off = reinterpret_cast<const unsigned char *>(p) - reinterpret_cast<const unsigned char *>(base);
        return q4_in_bounds(off >= 0 && off + bytes <= size, a.bounds);
    };
    int issued = 0;
    auto issue_next = [&]() {
        if (active) {
            const uint32_t so = static_cast<uint32_t>(issued % D) * SLOT;
            const int64_t rb = static_cast<int64_t>(g_begin + issued) * ROWS_IT;   // first row of the iteration
            if (rb + ROWS_IT <= a.N) {
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    if (src_ok(gc + u * rg_c, a.codes, codes_b, 16)) cp_async16(my_c + so + u * T * 16, gc + u * rg_c);
                    if (src_ok(gs + u * rg_s, a.scales, scales_b, 4)) cp_async4(my_s + so + u * T * 4, gs + u * rg_s);
                    if (ASYM && src_ok(gz + u * rg_z, a.zeros, zeros_b, 4))
                        cp_async4(my_z + so + u * T * 4, gz + u * rg_z);
                }
            } else {
                // Tail: a row past N reads row n - RG*k <= N-1 instead (same alignment
                // class, so the per-thread shifts stay valid); its result is discarded.
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t n = rb + u * RG + r;
                    int64_t back = 0;
                    if (n >= a.N) back = (n - (a.N - 1) + RG - 1) / RG;
                    const int64_t j = u - back;
                    if (src_ok(gc + j * rg_c, a.codes, codes_b, 16)) cp_async16(my_c + so + u * T * 16, gc + j * rg_c);
                    if (src_ok(gs + j * rg_s, a.scales, scales_b, 4)) cp_async4(my_s + so + u * T * 4, gs + j * rg_s);
                    if (ASYM && src_ok(gz + j * rg_z, a.zeros, zeros_b, 4))
                        cp_async4(my_z + so + u * T * 4, gz + j * rg_z);
                }
            }
        }
        gc += U * rg_c;
        gs += U * rg_s;
        if (ASYM) gz += U * rg_z;
        ++issued;
    };

#pragma unroll 1
    for (int p = 0; p < D - 1; ++p) {
        if (p < ng) issue_next();
        cp_commit();
    }
    // The weights are already on their way; x (and the y this grid writes) may belong
    // to the kernel before this one in the stream.
    allow_next_grid();
    wait_prior_grid();

    // ---- encode this CTA's x slice into planes (four threads per chunk and row of x) ----
    // (the round count is the same for every thread, so every lane reaches the shuffles)
    [[maybe_unused]] float ssq = 0.0f;   // (fused RMSNorm) this thread's sum of x^2
    for (int base = 0; base < MT * CTP; base += T / 4) {
        const int i = base + (tid >> 2);
        const bool in_range = i < MT * CTP;
        const int ii = in_range ? i : 0;
        const int m = ii / CTP, ci = ii - m * CTP;
        const int cc = split * CT + ci;
        const bool valid = in_range && m < a.M && ci < CT && cc < C;
        bool done = false;
        if constexpr (FUSED) {
            if (a.gamma != nullptr) {
                encode_chunk4_gamma(a.x + static_cast<int64_t>(valid ? m : 0) * K + (valid ? cc : 0) * 32,
                                    a.gamma + (valid ? cc : 0) * 32, valid, in_range,
                                    planes + (m * CTP + ci) * kPlaneWords, tid & 3, ssq);
                done = true;
            }
        }
        if (!done)
            encode_chunk4(a.x + static_cast<int64_t>(valid ? m : 0) * K + (valid ? cc : 0) * 32, valid, in_range,
                          planes + (m * CTP + ci) * kPlaneWords, tid & 3);
    }
    if constexpr (FUSED) {
        if (a.gamma != nullptr) {   // per-warp sums of x^2 -> shared memory
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) ssq += __shfl_xor_sync(0xffffffffu, ssq, o);
            if ((tid & 31) == 0) reinterpret_cast<float *>(smem + a.off_norm)[tid >> 5] = ssq;
        }
    }
    __syncthreads();
    // Load this thread's planes once.  The loads are volatile asm so the compiler
    // keeps the values in registers instead of re-reading shared memory at each use.
    Planes P[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        const uint32_t pa = static_cast<uint32_t>(__cvta_generic_to_shared(planes + (m * CTP + cl) * kPlaneWords));
        uint32_t w[28];
#pragma unroll
        for (int i = 0; i < 7; ++i)
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w[4 * i]), "=r"(w[4 * i + 1]), "=r"(w[4 * i + 2]), "=r"(w[4 * i + 3])
                         : "r"(pa + 16 * i));
#pragma unroll
        for (int i = 0; i < 24; ++i) P[m].p[i] = w[i];
        P[m].s_lo = static_cast<int>(w[24]);
        P[m].s_hi = static_cast<int>(w[25]);
        P[m].f = __uint_as_float(w[27]);
    }

    const uint4 *rc_t = reinterpret_cast<const uint4 *>(ring) + tid;
    const uint32_t *rs_t = reinterpret_cast<const uint32_t *>(ring + U * T * 16) + tid;
    const uint32_t *rz_t = rs_t + U * T;
    cg::cluster_group cluster = cg::this_cluster();
    const int nsplit = static_cast<int>(gridDim.y);
    // this thread's slot in a partial-sum buffer (row r of iteration bi, sub-row u)
    const int red_col = WARPRED ? (cl >> 5) : cl;

    int pp = 0;
    for (int b0 = 0; b0 < ng; b0 += RB, pp ^= 1) {
        const int nbat = min(RB, ng - b0);
        float *red = red0 + pp * RED_FLOATS;
#pragma unroll 1
        for (int bi = 0; bi < nbat; ++bi) {
            if (issued < ng) issue_next();
            cp_commit();
            cp_wait<D - 1>();
            const uint32_t so = static_cast<uint32_t>((b0 + bi) % D) * SLOT;
            const uint4 *rc = reinterpret_cast<const uint4 *>(reinterpret_cast<const unsigned char *>(rc_t) + so);
            const uint32_t *rs = reinterpret_cast<const uint32_t *>(reinterpret_cast<const unsigned char *>(rs_t) + so);
            const uint32_t *rz = reinterpret_cast<const uint32_t *>(reinterpret_cast<const unsigned char *>(rz_t) + so);
            float *rd = red + ((bi * U) * RG + r) * MT * RED_LD + red_col;
            float part[U][MT];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (active) {
                    const uint4 cw = rc[u * T];
                    const uint32_t sw = rs[u * T];
                    const int z = ASYM ? static_cast<int>((rz[u * T] >> zsh) & 0xFu) : 8;
                    const float s = __half2float(__ushort_as_half(static_cast<unsigned short>(sw >> ssh)));
#pragma unroll
                    for (int m = 0; m < MT; ++m) part[u][m] = (s * P[m].f) * chunk_dot(cw, z, P[m]);
                } else {
#pragma unroll
                    for (int m = 0; m < MT; ++m) part[u][m] = 0.0f;
                }
            }
            if (WARPRED) {
                // Sum the U*MT values over the warp's 32 lanes by recursive halving: each
                // round halves the number of values a lane carries while doubling the lanes
                // it covers, then plain butterflies finish (U*MT - 1 + log2 of the rest
                // shuffles instead of 5 per value).  Lane l ends with value index
                // (l >> (5 - log2(U*MT))) summed over all 32 lanes.
                constexpr int NV = U * MT;
                float v[NV];
#pragma unroll
                for (int u = 0; u < U; ++u)
#pragma unroll
                    for (int m = 0; m < MT; ++m) v[u * MT + m] = part[u][m];
                const int lane = tid & 31;
                int width = NV;
                int off = 16;
#pragma unroll
                for (int round = 0; (NV >> round) > 1; ++round) {
                    const int half = (NV >> round) / 2;
                    const bool upper = (lane & off) != 0;
#pragma unroll
                    for (int i = 0; i < half; ++i) {
                        // keep the upper half of the values on lanes with the bit set
                        const float send = upper ? v[i] : v[i + half];
                        const float keep = upper ? v[i + half] : v[i];
                        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                    }
                    off >>= 1;
                    width >>= 1;
                }
                float t = v[0];
#pragma unroll
                for (int o = off; o >= 1; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
                (void)width;
                // lanes whose low bits are 0 write: value index = lane >> (log2(32/NV))
                constexpr int SHIFT = (NV >= 32) ? 0 : (NV == 1 ? 5 : (NV == 2 ? 4 : (NV == 4 ? 3 : (NV == 8 ? 2 : 1))));
                if ((lane & ((1 << SHIFT) - 1)) == 0) {
                    const int idx = lane >> SHIFT;      // = u * MT + m
                    const int u = idx / MT, m = idx - u * MT;
                    rd[(u * RG * MT + m) * RED_LD] = t;
                }
            } else {
#pragma unroll
                for (int u = 0; u < U; ++u)
#pragma unroll
                    for (int m = 0; m < MT; ++m) rd[(u * RG * MT + m) * RED_LD] = part[u][m];
            }
        }
        // One barrier per batch: the partial buffers alternate, and the next batch's
        // barrier orders this batch's reads before the buffer is written again.
        __syncthreads();
        const int nrows = nbat * ROWS_IT;
        constexpr int NTERMS = WARPRED ? CTP / 32 : CTP;
        const int64_t first_row = static_cast<int64_t>(g_begin + b0) * ROWS_IT;
        if constexpr (FUSED) {
            // the row's 1 / sqrt(mean(x^2) + eps) from the warp sums, in order
            float rn = 1.0f;
            if (a.gamma != nullptr) {
                const float *nrm = reinterpret_cast<const float *>(smem + a.off_norm);
                float t = 0.0f;
                for (int w = 0; w < T / 32; ++w) t += nrm[w];
                rn = rsqrtf(t / static_cast<float>(K) + a.eps);
            }
            if (a.swiglu) {   // rows 2i, 2i + 1 of the batch (first_row is even)
                for (int i = tid; i < nrows / 2; i += T) {
                    const float *sg = red + (2 * i) * RED_LD, *su = red + (2 * i + 1) * RED_LD;
                    float gv = 0.0f, uv = 0.0f;
#pragma unroll
                    for (int q = 0; q < NTERMS; ++q) {
                        gv += sg[q];
                        uv += su[q];
                    }
                    gv *= rn;
                    uv *= rn;
                    const int64_t n = first_row + 2 * i;
                    if (n + 1 < a.N) a.y[n >> 1] = gv / (1.0f + expf(-gv)) * uv;
                }
            } else {
                for (int i = tid; i < nrows; i += T) {
                    const float *src = red + i * RED_LD;
                    float v = 0.0f;
#pragma unroll
                    for (int q = 0; q < NTERMS; ++q) v += src[q];
                    const int64_t n = first_row + i;
                    if (n < a.N) a.y[n] = v * rn;
                }
            }
        } else if (nsplit == 1) {
            for (int i = tid; i < nrows * MT; i += T) {
                const float *src = red + i * RED_LD;
                float v = 0.0f;
#pragma unroll
                for (int q = 0; q < NTERMS; ++q) v += src[q];
                const int rr = i / MT, m = i - rr * MT;
                const int64_t n = first_row + rr;
                if (n < a.N && m < a.M) a.y[static_cast<int64_t>(m) * a.N + n] = v;
            }
        } else {
            for (int i = tid; i < nrows * MT; i += T) {
                const float *src = red + i * RED_LD;
                float v = 0.0f;
#pragma unroll
                for (int q = 0; q < NTERMS; ++q) v += src[q];
                ysum[i] = v;
            }
            // add the K-slices of the cluster in rank order
            cluster.sync();
            const int rank = static_cast<int>(cluster.block_rank());
            for (int i = rank * T + tid; i < nrows * MT; i += nsplit * T) {
                float v = 0.0f;
                for (int q = 0; q < nsplit; ++q) v += cluster.map_shared_rank(ysum, q)[i];
                const int rr = i / MT, m = i - rr * MT;
                const int64_t n = first_row + rr;
                if (n < a.N && m < a.M) a.y[static_cast<int64_t>(m) * a.N + n] = v;
            }
            cluster.sync();
        }
    }
    cp_wait<0>();
}

// ------------------------------------------------------------------ host side

// Supported (threads per row, rows per group) pairs.
#define Q4_XREG_SHAPES(X) X(28, 8) X(32, 4) X(64, 4) X(96, 4) X(128, 4) X(160, 2) X(192, 2) X(224, 2) X(256, 2)

static int rows_per_group(int ctp) {
#define Q4_RG(C, R) if (ctp == C) return R;
    Q4_XREG_SHAPES(Q4_RG)
#undef Q4_RG
    return 0;
}

template <int MT, bool ASYM, int CTP, int RG, int KC = 0, int G = 0, int U = kXregU, int D = kXregD,
          bool FUSED = false>
static int launch_one(const XregPlan &p, const XregArgsOf<FUSED> &a, cudaStream_t stream) {
    auto kern = q4gemv_xreg_kernel<MT, ASYM, CTP, RG, KC, G, U, D, FUSED>;
    constexpr int T = CTP * RG;
    static std::atomic<bool> configured[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             device_info().smem_optin);
        if (e != cudaSuccess) {
            set_cuda_error(e);
            return Q4_ERR_CUDA;
        }
        configured[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(T, 1, 1);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    if (p.S > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = static_cast<unsigned>(p.S);
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    // Persistent grid: as many CTAs (clusters) as can be resident at once.
    int resident = 0;
    if (p.S > 1) {
        cfg.gridDim = dim3(1, static_cast<unsigned>(p.S), 1);
        cudaError_t e = cudaOccupancyMaxActiveClusters(&resident, kern, &cfg);
        if (e != cudaSuccess) {
            set_cuda_error(e);
            return Q4_ERR_CUDA;
        }
    } else {
        int per_sm = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, T, p.smem);
        if (e != cudaSuccess) {
            set_cuda_error(e);
            return Q4_ERR_CUDA;
        }
        resident = per_sm * device_info().sms;
    }
    if (resident < 1) return Q4_ERR_UNSUPPORTED;
    const int nsuper = static_cast<int>((a.N + U * RG - 1) / (U * RG));
    XregArgsOf<FUSED> aa = a;
    aa.nsuper = nsuper;
    const int grid_x = resident < nsuper ? resident : nsuper;
    cfg.gridDim = dim3(static_cast<unsigned>(grid_x), static_cast<unsigned>(p.S), 1);
    add_overlap_attr(cfg, attr);
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, aa);
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return Q4_ERR_CUDA;
    }
    return launch_status();
}

template <int MT, bool ASYM>
static int launch_shape(const XregPlan &p, const XregArgs &a, cudaStream_t s) {
    // compile-time geometry for the long-N decode shapes (LM heads)
    if (p.special) {
        if (a.C == 28 && a.nb == 28) return launch_one<MT, ASYM, 28, 8, 28, 32, kXregUSpecial, kXregDSpecial>(p, a, s);
        if (a.C == 128 && a.nb == 32) return launch_one<MT, ASYM, 128, 4, 128, 128, kXregUSpecial, kXregDSpecial>(p, a, s);
    }
#define Q4_CASE(C, R) \
    if (a.CTp == C) return launch_one<MT, ASYM, C, R>(p, a, s);
    Q4_XREG_SHAPES(Q4_CASE)
#undef Q4_CASE
    return Q4_ERR_UNSUPPORTED;
}

template <bool ASYM>
static int launch_shape_fused(const XregPlan &p, const XregFusedArgs &a, cudaStream_t s) {
#define Q4_CASE(C, R) \
    if (a.CTp == C) return launch_one<1, ASYM, C, R, 0, 0, kXregU, kXregD, true>(p, a, s);
    Q4_XREG_SHAPES(Q4_CASE)
#undef Q4_CASE
    return Q4_ERR_UNSUPPORTED;
}

int launch_q4gemv_xreg_fused(const XregPlan &p, const XregFusedArgs &a, cudaStream_t stream) {
    if (!p.fused || p.MT != 1 || p.S != 1 || p.special) return Q4_ERR_UNSUPPORTED;
    XregFusedArgs aa = a;
    aa.off_norm = p.off_norm;
    return p.asym ? launch_shape_fused<true>(p, aa, stream) : launch_shape_fused<false>(p, aa, stream);
}

int launch_q4gemv_xreg(const XregPlan &p, const XregArgs &a, cudaStream_t stream) {
    if (p.fused) return Q4_ERR_UNSUPPORTED;
    if (p.MT == 1) return p.asym ? launch_shape<1, true>(p, a, stream) : launch_shape<1, false>(p, a, stream);
    if (p.MT == 2) return p.asym ? launch_shape<2, true>(p, a, stream) : launch_shape<2, false>(p, a, stream);
    return Q4_ERR_UNSUPPORTED;
}

// Shared-memory layout of one instance (must match the carve-up in the kernel).
static size_t xreg_smem(int MT, int CTp, int RG, int U, int D, int S, bool asym, XregArgs &a, bool fused,
                        int *off_norm_out) {
    const int T = CTp * RG;
    const int rows_it = U * RG;
    const bool warpred = CTp >= 32;
    const int red_ld = warpred ? CTp / 32 : CTp + 1;
    const int RB = (64 / rows_it) > 0 ? (64 / rows_it) : 1;
    const size_t planes_b = static_cast<size_t>(MT) * CTp * kPlaneWords * 4;
    const size_t off_red = (planes_b + 15) / 16 * 16;
    const size_t red_b = 2 * static_cast<size_t>(RB) * rows_it * MT * red_ld * 4;
    const size_t off_ring = (off_red + red_b + 15) / 16 * 16;
    const size_t ring_b = static_cast<size_t>(D) * U * T * (asym ? 24 : 20);
    const size_t off_ysum = off_ring + ring_b;
    const size_t ysum_b = S > 1 ? static_cast<size_t>(RB) * rows_it * MT * 4 : 0;
    a.red_ld = red_ld;
    a.RB = RB;
    a.off_red = static_cast<int>(off_red);
    a.off_ring = static_cast<int>(off_ring);
    a.off_ysum = static_cast<int>(off_ysum);
    const size_t off_norm = (off_ysum + ysum_b + 15) / 16 * 16;
    *off_norm_out = static_cast<int>(off_norm);
    return fused ? off_norm + static_cast<size_t>((T + 31) / 32) * 4 : off_ysum + ysum_b;
}

// Plan: K-slices S, threads per row CTp, rows per group RG.  Returns false when the
// shape does not suit this kernel (the caller then uses the general kernel).
bool plan_q4gemv_xreg(int M, int64_t N, int K, int group, const void *scales, const void *zeros,
                      XregPlan &p, XregArgs &a, bool fused) {
    if (M < 1 || M > 2) return false;
    if (fused && M != 1) return false;
    const int C = K / 32;
    const int nb = K / group;
    const int zrow = (nb + 1) / 2;
    const bool asym = zeros != nullptr;
    // word-granular scale / zero-point reads: 4-byte aligned bases, no word past the end
    if (!aligned(scales, 4) || (asym && !aligned(zeros, 4))) return false;
    if ((N * nb) % 2 != 0) return false;
    if (asym && (N * zrow) % 4 != 0) return false;
    const DeviceInfo &d = device_info();
    const int MT = M;
    int S = (C + 255) / 256;
    if (S > 8 || (fused && S != 1)) return false;
    const int CT = (C + S - 1) / S;
    const int CTp = CT >= 32 ? (CT + 31) / 32 * 32 : CT;
    const int RG = rows_per_group(CTp);
    if (RG == 0) return false;
    // the per-thread shift constants need RG rows to advance whole words
    if (asym && (static_cast<int64_t>(RG) * zrow) % 4 != 0) return false;
    if ((static_cast<int64_t>(RG) * nb) % 2 != 0) return false;
    // compile-time-geometry instances serve the long-N shapes they were built for
    const bool special = !fused && S == 1 && ((C == 28 && group == 32) || (C == 128 && group == 128)) &&
                         N >= 64 * kXregUSpecial * RG;
    const int U = special ? kXregUSpecial : kXregU;
    const int D = special ? kXregDSpecial : kXregD;
    const int T = CTp * RG;
    if (N < 4 * U * RG) return false;
    int off_norm = 0;
    const size_t smem = xreg_smem(MT, CTp, RG, U, D, S, asym, a, fused, &off_norm);
    if (smem > static_cast<size_t>(d.smem_optin) - 1024) return false;
    p.MT = MT;
    p.S = S;
    p.threads = T;
    p.grid_x = 0;
    p.smem = smem;
    p.asym = asym;
    p.warpred = CTp >= 32;
    p.special = special;
    p.fused = fused;
    p.off_norm = off_norm;
    a.M = M;
    a.N = static_cast<int>(N);
    a.K = K;
    a.C = C;
    a.nb = nb;
    a.zrow = zrow;
    a.gshift = group == 32 ? 0 : (group == 64 ? 1 : 2);
    a.CT = CT;
    a.CTp = CTp;
    a.RG = RG;
    a.nsuper = static_cast<int>((N + U * RG - 1) / (U * RG));
    return true;
}

}  // namespace q4
