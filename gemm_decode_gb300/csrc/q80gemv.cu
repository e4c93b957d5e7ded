// q80gemv.cu -- the GEMV over Q8_0 blocks (q8_0_gemv_run), 1 <= M <= 16.
//
// y[m][n] = sum_k q[n][k] * d[n][k/32] * x[m][k], where each row of weights is K/32
// blocks of 34 bytes: the binary16 scale d (little-endian), then 32 two's-complement
// 8-bit codes, element j of the block at byte 2 + j, no zero point (cera's
// wgpu_gemv_bench.rs, block geometry "Q8_0 (32, 34)").
//
// M = 1 on long matrices runs the TMA-streamed kernel's Q8_0 instances (a block of rows
// is one stretch of 34-byte blocks, dp4a on the byte planes of x; q4gemv_stream.cu).
// Every other shape runs the kernel below on CUDA cores.  A warp takes two blocks of a
// row at a time, lanes 0-15 the first and 16-31 the second, each lane two neighbouring
// elements (one 16-bit load of codes: blocks are only 2-byte aligned), so that a warp's
// read of a row of x is 256 contiguous bytes.  Each weight q * d is formed exactly in
// binary32 (an 8-bit integer times an 11-bit significand) and accumulated with fused
// multiply-adds.  A warp carries R rows of weights, so that each load of x serves R rows;
// when the rows alone would give too few CTAs, the warps of a CTA split the blocks of
// their rows and add their partial sums in shared memory in warp order.
#include "q4_common.cuh"
#include "q4gemv_stream.cuh"

namespace q4 {

namespace {

constexpr int kQ80Threads = 256;
constexpr int kQ80Warps = kQ80Threads / 32;

// Sums each of v[0 .. V-1] over the 32 lanes of the warp (V a power of two, <= 32):
// halving exchanges leave lane l holding, in v[0], the whole sum of entry l / (32 / V).
template <int V>
__device__ __forceinline__ void warp_sum_scatter(float (&v)[V], int lane) {
#pragma unroll
    for (int s = 0; s < 5; ++s) {
        const int o = 16 >> s;
        const int c = V >> s;   // entries still held by each lane
        if (c >= 2) {
            const bool upper = (lane & o) != 0;
#pragma unroll
            for (int i = 0; i < c / 2; ++i) {
                const float send = upper ? v[i] : v[i + c / 2];
                const float keep = upper ? v[i + c / 2] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
            }
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
        }
    }
}

// MT rows of x at most (M <= MT at run time), R weight rows per warp, ksplit warps per
// group of rows (a divisor of 8).  Lane l takes codes 8p .. 8p + 7 (p = l % 4) of block
// b0 + l / 4, so a warp covers 8 blocks of each of its rows per step: three aligned loads
// (32, 32 and 16 bits) hold the 8 codes, which start 2 bytes into the block, after a shift
// by 0 or 16 bits; the block's scale is one 16-bit load.  Each code is widened exactly, the
// 8 products of a row of x are summed with fused multiply-adds and that sum is scaled by d
// once.  Rows of x are taken four at a time (their 8 x values each in registers).  Entry
// e = m * R + r of a lane's sums is y[m][n0 + r].
template <int MT, int R>
__global__ void __launch_bounds__(kQ80Threads)
q80_gemv_kernel(const uint8_t *__restrict__ blocks, const float *__restrict__ x, float *__restrict__ y, int M,
                int64_t N, int K, int ksplit, unsigned int *bounds) {
    constexpr int V = MT * R;
    constexpr int MG = MT < 4 ? MT : 4;   // rows of x per pass
    static_assert(V <= 32 && (V & (V - 1)) == 0, "entries per lane");
    __shared__ float part[kQ80Warps][V];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int group = warp / ksplit, kw = warp - group * ksplit;
    const int64_t n0 = (static_cast<int64_t>(blockIdx.x) * (kQ80Warps / ksplit) + group) * R;
    const int nblk = K >> 5, nstep = (nblk + 7) >> 3;
    const int bs = lane >> 2, p = lane & 3;
    // rows past N read row N - 1; their sums are not stored
    const uint8_t *row[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t n = n0 + r < N ? n0 + r : N - 1;
        row[r] = blocks + n * nblk * 34;
    }
    // (bounds-checking builds) a load of sz bytes at p lies inside the blocks and is
    // naturally aligned
    const uint8_t *const blocks_end = blocks + N * nblk * 34;
    auto ok_w = [&](const void *p, int sz) {
        const uint8_t *b = static_cast<const uint8_t *>(p);
        return q4_in_bounds(b >= blocks && b + sz <= blocks_end && (reinterpret_cast<uintptr_t>(b) % sz) == 0,
                            bounds);
    };
    float acc[V];
#pragma unroll
    for (int e = 0; e < V; ++e) acc[e] = 0.0f;
    wait_prior_grid();   // x may belong to the kernel before this one in the stream
    for (int st = kw; st < nstep; st += ksplit) {
        const int bl = 8 * st + bs;
        const bool live = bl < nblk;   // false only for lanes past an incomplete last step
        const int b = live ? bl : nblk - 1;
        // codes 8p .. 8p + 7 start at byte 34 b + 2 + 8p of the row, an address that is only
        // 2-byte aligned (rows and blocks start on even bytes): two 32-bit words from the
        // 4-byte boundary at or below it, shifted by 0 or 16 bits, and after a shift a 16-bit
        // load for the last two codes (so every load ends on the block's last code byte)
        const uint32_t off = static_cast<uint32_t>(b) * 34u + 2u + 8u * p;
        float q[R][8], d[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint8_t *cp = row[r] + off;
            const uint32_t shift = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(cp) & 2u) * 8u;   // 0 or 16
            const uint32_t *wp = reinterpret_cast<const uint32_t *>(cp - (shift >> 3));
            const uint32_t a0 = ok_w(wp, 4) ? __ldg(wp) : 0u, a1 = ok_w(wp + 1, 4) ? __ldg(wp + 1) : 0u;
            const uint32_t a2 =
                shift && ok_w(cp + 6, 2) ? ldg_u16(reinterpret_cast<const uint16_t *>(cp + 6)) : 0u;
            const uint32_t w0 = __funnelshift_r(a0, a1, shift), w1 = __funnelshift_r(a1, a2, shift);
            d[r] = live && ok_w(row[r] + 34u * b, 2)
                       ? half_bits_to_float(ldg_u16(reinterpret_cast<const uint16_t *>(row[r] + 34u * b)))
                       : 0.0f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                q[r][i] = static_cast<float>(static_cast<int32_t>(w0 << (24 - 8 * i)) >> 24);
                q[r][4 + i] = static_cast<float>(static_cast<int32_t>(w1 << (24 - 8 * i)) >> 24);
            }
        }
        const float *xb = x + 32 * b + 8 * p;
#pragma unroll
        for (int m0 = 0; m0 < MT; m0 += MG) {
            float xv[MG][8];
#pragma unroll
            for (int mm = 0; mm < MG; ++mm) {
                const int m = m0 + mm;
                const float *xp = xb + static_cast<int64_t>(m) * K;
                if (m < M && q4_in_bounds(xp >= x && xp + 8 <= x + static_cast<int64_t>(M) * K &&
                                              (reinterpret_cast<uintptr_t>(xp) & 15u) == 0,
                                          bounds)) {
                    const float4 lo = __ldg(reinterpret_cast<const float4 *>(xb + static_cast<int64_t>(m) * K));
                    const float4 hi = __ldg(reinterpret_cast<const float4 *>(xb + static_cast<int64_t>(m) * K) + 1);
                    xv[mm][0] = lo.x; xv[mm][1] = lo.y; xv[mm][2] = lo.z; xv[mm][3] = lo.w;
                    xv[mm][4] = hi.x; xv[mm][5] = hi.y; xv[mm][6] = hi.z; xv[mm][7] = hi.w;
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) xv[mm][i] = 0.0f;
                }
            }
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int mm = 0; mm < MG; ++mm) {
                    float sum = q[r][0] * xv[mm][0];
#pragma unroll
                    for (int i = 1; i < 8; ++i) sum = fmaf(q[r][i], xv[mm][i], sum);
                    acc[(m0 + mm) * R + r] = fmaf(d[r], sum, acc[(m0 + mm) * R + r]);
                }
        }
    }
    allow_next_grid();
    warp_sum_scatter<V>(acc, lane);
    constexpr int kCopies = 32 / V;   // lanes holding the same entry
    const int e = lane / kCopies;
    const bool writer = (lane % kCopies) == 0;
    if (ksplit == 1) {
        const int m = e / R, r = e - (e / R) * R;
        if (writer && m < M && n0 + r < N) y[static_cast<int64_t>(m) * N + n0 + r] = acc[0];
        return;
    }
    if (writer) part[warp][e] = acc[0];
    __syncthreads();
    if (kw == 0 && lane < V) {
        float s = part[warp][lane];
        for (int w = 1; w < ksplit; ++w) s += part[warp + w][lane];
        const int m = lane / R, r = lane - (lane / R) * R;
        if (m < M && n0 + r < N) y[static_cast<int64_t>(m) * N + n0 + r] = s;
    }
}

template <int MT, int R>
int launch_q80(const uint8_t *blocks, const float *x, float *y, int M, int64_t N, int K, int ksplit,
               cudaStream_t stream) {
    const int64_t rows_per_cta = static_cast<int64_t>(kQ80Warps / ksplit) * R;
    const int64_t grid = (N + rows_per_cta - 1) / rows_per_cta;
    if (grid > 0x7fffffffLL) return Q4_ERR_UNSUPPORTED;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(kQ80Threads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    add_overlap_attr(cfg, attr);
    cudaError_t e = cudaLaunchKernelEx(&cfg, q80_gemv_kernel<MT, R>, blocks, x, y, M, N, K, ksplit, bounds_counter());
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return Q4_ERR_CUDA;
    }
    return launch_status();
}

// The smallest split of the blocks over the warps of a CTA (1, 2, 4 or 8, at most the
// steps of 8 blocks in a row) that gives at least `want` CTAs, or the largest allowed.
int q80_split(int64_t N, int R, int nstep, int64_t want) {
    int ks = 1;
    while (ks < kQ80Warps && 2 * ks <= nstep) {
        const int64_t rows = static_cast<int64_t>(kQ80Warps / ks) * R;
        if ((N + rows - 1) / rows >= want) break;
        ks *= 2;
    }
    return ks;
}

// R = RW (2 to 4 weight rows per warp) where that still gives `want` CTAs, else one row
// per warp.
template <int MT, int RW>
int launch_q80_m(const uint8_t *blocks, const float *x, float *y, int M, int64_t N, int K, cudaStream_t stream) {
    const int nstep = (K / 32 + 7) / 8;
    const int64_t want = 4LL * device_info().sms;
    const int ks = q80_split(N, RW, nstep, want);
    const int64_t rows = static_cast<int64_t>(kQ80Warps / ks) * RW;
    if ((N + rows - 1) / rows >= want) return launch_q80<MT, RW>(blocks, x, y, M, N, K, ks, stream);
    return launch_q80<MT, 1>(blocks, x, y, M, N, K, q80_split(N, 1, nstep, want), stream);
}

}  // namespace

int launch_q80gemv(const uint8_t *blocks, const float *x, float *y, int M, int64_t N, int K, cudaStream_t stream) {
    if (!call_options().exact_x && stream_q80_applies(M, N, K, blocks))
        return launch_q4gemv_stream_q80(blocks, x, y, N, K, stream);
    if (M <= 1) return launch_q80_m<1, 4>(blocks, x, y, M, N, K, stream);
    if (M <= 2) return launch_q80_m<2, 4>(blocks, x, y, M, N, K, stream);
    if (M <= 4) return launch_q80_m<4, 4>(blocks, x, y, M, N, K, stream);
    if (M <= 8) return launch_q80_m<8, 2>(blocks, x, y, M, N, K, stream);
    return launch_q80_m<16, 2>(blocks, x, y, M, N, K, stream);
}

}  // namespace q4
