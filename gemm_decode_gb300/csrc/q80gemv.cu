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
// group of rows (a divisor of 8).  Entry e = m * R + r of a lane's sums is y[m][n0 + r].
template <int MT, int R>
__global__ void __launch_bounds__(kQ80Threads)
q80_gemv_kernel(const uint8_t *__restrict__ blocks, const float *__restrict__ x, float *__restrict__ y, int M,
                int64_t N, int K, int ksplit) {
    constexpr int V = MT * R;
    static_assert(V <= 32 && (V & (V - 1)) == 0, "entries per lane");
    __shared__ float part[kQ80Warps][V];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int group = warp / ksplit, kw = warp - group * ksplit;
    const int64_t n0 = (static_cast<int64_t>(blockIdx.x) * (kQ80Warps / ksplit) + group) * R;
    const int nblk = K >> 5, npair = (nblk + 1) >> 1;
    const int half = lane >> 4, j = lane & 15;
    // rows past N read row N - 1; their sums are not stored
    const uint16_t *row[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t n = n0 + r < N ? n0 + r : N - 1;
        row[r] = reinterpret_cast<const uint16_t *>(blocks) + n * nblk * 17;
    }
    float acc[V];
#pragma unroll
    for (int e = 0; e < V; ++e) acc[e] = 0.0f;
    wait_prior_grid();   // x may belong to the kernel before this one in the stream
#pragma unroll 2
    for (int p = kw; p < npair; p += ksplit) {
        const int bl = 2 * p + half;
        const bool live = bl < nblk;           // false only for lanes 16-31 past an odd last block
        const int b = live ? bl : nblk - 1;
        float t0[R], t1[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint32_t c = ldg_u16(row[r] + b * 17 + 1 + j);   // elements 2j (low byte), 2j + 1
            const float d = live ? half_bits_to_float(ldg_u16(row[r] + b * 17)) : 0.0f;
            t0[r] = static_cast<float>(static_cast<int32_t>(c << 24) >> 24) * d;
            t1[r] = static_cast<float>(static_cast<int32_t>(c << 16) >> 24) * d;
        }
        const float *xb = x + b * 32 + 2 * j;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m < M) {
                const float2 xv = __ldg(reinterpret_cast<const float2 *>(xb + static_cast<int64_t>(m) * K));
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    acc[m * R + r] = fmaf(t0[r], xv.x, acc[m * R + r]);
                    acc[m * R + r] = fmaf(t1[r], xv.y, acc[m * R + r]);
                }
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
    cudaError_t e = cudaLaunchKernelEx(&cfg, q80_gemv_kernel<MT, R>, blocks, x, y, M, N, K, ksplit);
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return Q4_ERR_CUDA;
    }
    return launch_status();
}

// The smallest split of the blocks over the warps of a CTA (1, 2, 4 or 8, at most the
// pairs of blocks in a row) that gives at least `want` CTAs, or the largest allowed.
int q80_split(int64_t N, int R, int npair, int64_t want) {
    int ks = 1;
    while (ks < kQ80Warps && 2 * ks <= npair) {
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
    const int npair = (K / 32 + 1) / 2;
    const int64_t want = 4LL * device_info().sms;
    const int ks = q80_split(N, RW, npair, want);
    const int64_t rows = static_cast<int64_t>(kQ80Warps / ks) * RW;
    if ((N + rows - 1) / rows >= want) return launch_q80<MT, RW>(blocks, x, y, M, N, K, ks, stream);
    return launch_q80<MT, 1>(blocks, x, y, M, N, K, q80_split(N, 1, npair, want), stream);
}

}  // namespace

int launch_q80gemv(const uint8_t *blocks, const float *x, float *y, int M, int64_t N, int K, cudaStream_t stream) {
    if (!call_options().exact_x && stream_q80_applies(M, N, K, blocks))
        return launch_q4gemv_stream_q80(blocks, x, y, N, K, stream);
    if (M <= 1) return launch_q80_m<1, 4>(blocks, x, y, M, N, K, stream);
    if (M <= 2) return launch_q80_m<2, 4>(blocks, x, y, M, N, K, stream);
    if (M <= 4) return launch_q80_m<4, 4>(blocks, x, y, M, N, K, stream);
    if (M <= 8) return launch_q80_m<8, 4>(blocks, x, y, M, N, K, stream);
    return launch_q80_m<16, 2>(blocks, x, y, M, N, K, stream);
}

}  // namespace q4
