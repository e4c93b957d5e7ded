// q4gemv_stream.cu -- the M = 1 int4 GEMV for long-N shapes whose rows are short
// enough that a block of rows is one contiguous stretch of memory (LM heads).
//
// Computes y[n] = sum_k (q[n][k] - z[n][k/g]) * s[n][k/g] * x[k]
// (gerbil GPU-engine kernel reference, "3. MatMulInt4": "Computes",
// "Dequantization"; MatMulNBits layout per the Refractometer page's
// "b) q4 GEMV" sweep).
//
// One warp of each CTA is a producer: one of its threads streams each block of
// ROWS consecutive rows -- their codes, scales and zero points, three
// contiguous stretches -- into a ring of shared-memory slots with the TMA bulk
// copy engine (cp.async.bulk), completion counted on the slot's mbarrier.  The
// other warps are consumers: thread (r, c) owns chunk position c (32 codes) of
// row r of every block and keeps the matching 32 values of x in registers as
// 24-bit byte planes (see q4gemv_xplanes.cuh); it unpacks its chunk to bytes,
// forms the exact integer dot product with dp4a, subtracts the zero-point
// term exactly, and scales once.  Per-row partial sums go to one of three
// shared buffers; the reduction of block b is done by one consumer warp
// (rotating) while the others already compute block b+1, ordered by
// mbarriers rather than CTA barriers.  Every wait is bounded by a
// %globaltimer deadline (device status word on expiry).
#include "q4_common.cuh"
#include "q4gemv_xplanes.cuh"
#include "q4gemv_stream.cuh"

namespace q4 {

using namespace xp;

__device__ unsigned int g_stream_status = 0;   // 1 = a bounded wait expired

namespace {

template <int C, int RG, int G, int U, int D>
struct StreamGeom {
    static constexpr int K = C * 32;
    static constexpr int NB = K / G;                  // groups per row
    static constexpr int ZROW = (NB + 1) / 2;          // zero-point bytes per row
    static constexpr int GSHIFT = G == 32 ? 0 : (G == 64 ? 1 : 2);
    static constexpr int ROWS = U * RG;                // rows per block (one ring slot)
    static constexpr int CODE_B = ROWS * C * 16;
    static constexpr int SC_B = ROWS * NB * 2;
    static constexpr int Z_B = ROWS * ZROW;
    static constexpr int SLOT_B = (CODE_B + SC_B + Z_B + 127) / 128 * 128;
    static constexpr int TC = C * RG;                  // consumer threads
    static constexpr int NWC = TC / 32;                // consumer warps
    static constexpr int T = TC + 32;                  // + one producer warp
    static constexpr int RED_LD = C + 1;
    static constexpr int RED_B = ROWS * RED_LD * 4;    // one partial-sum buffer
    // shared memory: planes | red[3] | ring[D] | barriers
    static constexpr int OFF_RED = (C * 28 * 4 + 127) / 128 * 128;
    static constexpr int OFF_RING = (OFF_RED + 3 * RED_B + 127) / 128 * 128;
    static constexpr int OFF_BAR = OFF_RING + D * SLOT_B;
    static constexpr int SMEM = OFF_BAR + 8 * (2 * D + 6) + 16;
    static_assert(TC % 32 == 0, "consumer threads must fill whole warps");
    static_assert(CODE_B % 16 == 0 && SC_B % 16 == 0 && Z_B % 16 == 0, "bulk copies move 16-byte multiples");
};

}  // namespace

template <int C, int RG, int G, bool ASYM, int U, int D>
__global__ void __launch_bounds__(C * RG + 32)
q4gemv_stream_kernel(const StreamArgs a) {
    using Gm = StreamGeom<C, RG, G, U, D>;
    extern __shared__ __align__(128) unsigned char smem[];
    uint32_t *planes = reinterpret_cast<uint32_t *>(smem);
    float *red = reinterpret_cast<float *>(smem + Gm::OFF_RED);
    unsigned char *ring = smem + Gm::OFF_RING;
    const uint32_t bar0 = static_cast<uint32_t>(__cvta_generic_to_shared(smem + Gm::OFF_BAR));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Gm::OFF_BAR + 8 * (2 * D + 6));
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (D + s); };
    auto redfull = [&](int b) { return bar0 + 8u * (2 * D + b); };
    auto reddone = [&](int b) { return bar0 + 8u * (2 * D + 3 + b); };

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const unsigned long long limit = a.timeout_ns;

    // blocks of this CTA (contiguous range)
    const int gsz = static_cast<int>(gridDim.x);
    const int b_begin = static_cast<int>(static_cast<int64_t>(a.nblocks) * blockIdx.x / gsz);
    const int b_end = static_cast<int>(static_cast<int64_t>(a.nblocks) * (blockIdx.x + 1) / gsz);
    const int nbk = b_end - b_begin;

    if (tid == 0) {
        for (int s = 0; s < D; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), Gm::NWC);
        }
        for (int b = 0; b < 3; ++b) {
            mbar_init(redfull(b), Gm::NWC);
            mbar_init(reddone(b), 1);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    allow_next_grid();

    auto fail = [&]() {
        *abort_flag = 1;
        atomicOr(&g_stream_status, 1u);
    };

    if (warp == Gm::NWC) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int issued = 0;
            for (int i = 0; i < nbk && !*abort_flag; ++i) {
                const int s = i % D;
                if (i >= D && !mbar_wait(empty(s), ((i / D) - 1) & 1, limit)) {
                    fail();
                    break;
                }
                const int64_t row0 = static_cast<int64_t>(b_begin + i) * Gm::ROWS;
                const int rows = static_cast<int>(a.N - row0 < Gm::ROWS ? a.N - row0 : Gm::ROWS);
                const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(ring + s * Gm::SLOT_B));
                const unsigned char *src_c = a.codes + row0 * (C * 16);
                const unsigned char *src_s = reinterpret_cast<const unsigned char *>(a.scales) + row0 * (Gm::NB * 2);
                const unsigned char *src_z = ASYM ? a.zeros + row0 * Gm::ZROW : nullptr;
                if (rows == Gm::ROWS) {
                    mbar_expect_tx(full(s), Gm::CODE_B + Gm::SC_B + (ASYM ? Gm::Z_B : 0));
                    bulk_copy(dst, src_c, Gm::CODE_B, full(s));
                    bulk_copy(dst + Gm::CODE_B, src_s, Gm::SC_B, full(s));
                    if (ASYM) bulk_copy(dst + Gm::CODE_B + Gm::SC_B, src_z, Gm::Z_B, full(s));
                } else {
                    // last, partial block: codes by bulk copy (rows * C * 16 bytes), the
                    // scale and zero-point bytes by plain copies (their size need not be a
                    // multiple of 16); the arrive below publishes the plain stores
                    const int sb = rows * Gm::NB * 2, zb = rows * Gm::ZROW;
                    unsigned char *sl = ring + s * Gm::SLOT_B;
                    for (int j = 0; j < sb; ++j) sl[Gm::CODE_B + j] = src_s[j];
                    if (ASYM)
                        for (int j = 0; j < zb; ++j) sl[Gm::CODE_B + Gm::SC_B + j] = src_z[j];
                    mbar_expect_tx(full(s), rows * C * 16);
                    bulk_copy(dst, src_c, rows * C * 16, full(s));
                }
                issued = i + 1;
            }
            if (*abort_flag) {
                // drain (bounded): every issued copy lands before the CTA may exit
                for (int i = issued - D > 0 ? issued - D : 0; i < issued; ++i)
                    mbar_wait(full(i % D), (i / D) & 1, 50ull * 1000 * 1000);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    // x and y may belong to the kernel before this one in the stream; the producer
    // streams only weights and needs no such wait.
    wait_prior_grid();
    const int r = tid / C, c = tid - r * C;
    // encode x into planes (four consumer threads per chunk), then a consumer-only barrier
    for (int base = 0; base < C; base += Gm::TC / 4) {
        const int i = base + (tid >> 2);
        const bool in_range = i < C;
        encode_chunk4(a.x + (in_range ? i : 0) * 32, in_range, in_range, planes + (in_range ? i : 0) * kPlaneWords,
                      tid & 3);
    }
    asm volatile("bar.sync 1, %0;" ::"r"(Gm::TC) : "memory");
    Planes P;
    {
        const uint32_t pa = static_cast<uint32_t>(__cvta_generic_to_shared(planes + c * kPlaneWords));
        uint32_t w[28];
#pragma unroll
        for (int i = 0; i < 7; ++i)
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w[4 * i]), "=r"(w[4 * i + 1]), "=r"(w[4 * i + 2]), "=r"(w[4 * i + 3])
                         : "r"(pa + 16 * i));
#pragma unroll
        for (int i = 0; i < 24; ++i) P.p[i] = w[i];
        P.s_lo = static_cast<int>(w[24]);
        P.s_hi = static_cast<int>(w[25]);
        P.f = __uint_as_float(w[27]);
    }
    const int grp = c >> Gm::GSHIFT;
    // byte offsets of this thread's data inside a slot, for sub-row u = 0
    const int off_c = (r * C + c) * 16;
    const int off_s = Gm::CODE_B + (r * Gm::NB + grp) * 2;
    const int off_z = Gm::CODE_B + Gm::SC_B + r * Gm::ZROW + (grp >> 1);
    const int zsh = (grp & 1) * 4;

    for (int i = 0; i < nbk; ++i) {
        if (*abort_flag) break;
        const int s = i % D;
        const int rb = i % 3;
        if (!mbar_wait(full(s), (i / D) & 1, limit)) {
            fail();
            break;
        }
        if (i >= 3 && !mbar_wait(reddone(rb), ((i / 3) - 1) & 1, limit)) {
            fail();
            break;
        }
        const unsigned char *sl = ring + s * Gm::SLOT_B;
        float *rd = red + rb * (Gm::RED_B / 4) + r * Gm::RED_LD + c;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint4 cw = *reinterpret_cast<const uint4 *>(sl + off_c + u * RG * C * 16);
            const uint32_t sh = *reinterpret_cast<const uint16_t *>(sl + off_s + u * RG * Gm::NB * 2);
            const int z = ASYM ? static_cast<int>((sl[off_z + u * RG * Gm::ZROW] >> zsh) & 0xFu) : 8;
            const float sc = __half2float(__ushort_as_half(static_cast<unsigned short>(sh)));
            rd[u * RG * Gm::RED_LD] = (sc * P.f) * chunk_dot(cw, z, P);
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(empty(s));      // slot s may be refilled
            mbar_arrive(redfull(rb));   // this warp's partials of block i are written
        }
        // deferred reduction of block i-1 by one (rotating) consumer warp
        if (i >= 1 && warp == (i - 1) % Gm::NWC) {
            const int pb = (i - 1) % 3;
            if (!mbar_wait(redfull(pb), ((i - 1) / 3) & 1, limit)) {
                fail();
                break;
            }
            const float *src = red + pb * (Gm::RED_B / 4);
            const int64_t row0 = static_cast<int64_t>(b_begin + i - 1) * Gm::ROWS;
            for (int rho = lane; rho < Gm::ROWS; rho += 32) {
                float v = 0.0f;
#pragma unroll
                for (int q = 0; q < C; ++q) v += src[rho * Gm::RED_LD + q];
                if (row0 + rho < a.N) a.y[row0 + rho] = v;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(reddone(pb));
        }
    }
    // the last block's reduction
    if (nbk > 0 && !*abort_flag && warp == (nbk - 1) % Gm::NWC) {
        const int pb = (nbk - 1) % 3;
        if (!mbar_wait(redfull(pb), ((nbk - 1) / 3) & 1, limit)) {
            fail();
        } else {
            const float *src = red + pb * (Gm::RED_B / 4);
            const int64_t row0 = static_cast<int64_t>(b_end - 1) * Gm::ROWS;
            for (int rho = lane; rho < Gm::ROWS; rho += 32) {
                float v = 0.0f;
#pragma unroll
                for (int q = 0; q < C; ++q) v += src[rho * Gm::RED_LD + q];
                if (row0 + rho < a.N) a.y[row0 + rho] = v;
            }
        }
    }
}

// ------------------------------------------------------------------ host side

template <int C, int RG, int G, bool ASYM, int U, int D>
static int launch_stream(const StreamArgs &a0, cudaStream_t stream) {
    using Gm = StreamGeom<C, RG, G, U, D>;
    auto kern = q4gemv_stream_kernel<C, RG, G, ASYM, U, D>;
    static bool configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Gm::SMEM);
        if (e != cudaSuccess) {
            set_cuda_error(e);
            return Q4_ERR_CUDA;
        }
        configured[dev] = true;
    }
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, Gm::T, Gm::SMEM);
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return Q4_ERR_CUDA;
    }
    if (per_sm < 1) return Q4_ERR_UNSUPPORTED;
    StreamArgs a = a0;
    a.nblocks = static_cast<int>((a.N + Gm::ROWS - 1) / Gm::ROWS);
    int grid = per_sm * device_info().sms;
    if (grid > a.nblocks) grid = a.nblocks;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(Gm::T, 1, 1);
    cfg.dynamicSmemBytes = Gm::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    add_overlap_attr(cfg, attr);
    e = cudaLaunchKernelEx(&cfg, kern, a);
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return Q4_ERR_CUDA;
    }
    return launch_status();
}

bool stream_applies(int M, int64_t N, int K, int group, const void *codes, const void *scales, const void *zeros) {
    if (M != 1) return false;
    const bool shape = (K == 896 && group == 32) || (K == 4096 && group == 128);
    if (!shape) return false;
    if (!aligned(codes, 16) || !aligned(scales, 16) || (zeros && !aligned(zeros, 16))) return false;
    return N >= 4096;
}

static unsigned long long g_stream_timeout_ns = 1000ull * 1000 * 1000;
void set_stream_wait_timeout_ns(unsigned long long ns) { g_stream_timeout_ns = ns; }

int launch_q4gemv_stream(const uint8_t *codes, const uint16_t *scales, const uint8_t *zeros, const float *x,
                         float *y, int64_t N, int K, int group, cudaStream_t stream) {
    StreamArgs a;
    a.codes = codes;
    a.scales = scales;
    a.zeros = zeros;
    a.x = x;
    a.y = y;
    a.N = N;
    a.nblocks = 0;
    a.timeout_ns = g_stream_timeout_ns;
    const bool asym = zeros != nullptr;
    if (K == 896 && group == 32)
        return asym ? launch_stream<28, 8, 32, true, 4, 3>(a, stream) : launch_stream<28, 8, 32, false, 4, 3>(a, stream);
    if (K == 4096 && group == 128)
        return asym ? launch_stream<128, 4, 128, true, 2, 4>(a, stream)
                    : launch_stream<128, 4, 128, false, 2, 4>(a, stream);
    return Q4_ERR_UNSUPPORTED;
}

int read_and_clear_stream_status(unsigned int *v) {
    cudaError_t e = cudaMemcpyFromSymbol(v, g_stream_status, sizeof *v);
    if (e != cudaSuccess) return Q4_ERR_CUDA;
    if (*v) {
        const unsigned int zero = 0;
        cudaMemcpyToSymbol(g_stream_status, &zero, sizeof zero);
    }
    return Q4_OK;
}

}  // namespace q4
