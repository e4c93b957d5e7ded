// q80gemv.cu -- the GEMV over Q8_0 blocks (q8_0_gemv_run), 1 <= M <= 16.
//
// y[m][n] = sum_k q[n][k] * d[n][k/32] * x[m][k], where each row of weights is K/32
// blocks of 34 bytes: the binary16 scale d (little-endian), then 32 two's-complement
// 8-bit codes, element j of the block at byte 2 + j, no zero point (cera's
// wgpu_gemv_bench.rs, block geometry "Q8_0 (32, 34)").
//
// M = 1 on long matrices runs the TMA-streamed kernel's Q8_0 instances (a block of rows
// is one stretch of 34-byte blocks, dp4a on the byte planes of x; q4gemv_stream.cu).
// Every other shape runs the kernel below on CUDA cores: one warp per weight row, its
// lanes striding over the row's blocks; each code is widened exactly to binary32, the 32
// products of a block summed with fused multiply-adds and scaled once by d, the blocks
// summed over the lanes by shuffles.  Blocks are only 2-byte aligned, so a block is read
// as 17 16-bit loads; x is read through the read-only cache as 16-byte vectors.
#include "q4_common.cuh"
#include "q4gemv_stream.cuh"

namespace q4 {

namespace {

constexpr int kQ80Threads = 256;
constexpr int kQ80RowsPerCta = kQ80Threads / 32;

template <int MT>
__global__ void __launch_bounds__(kQ80Threads)
q80_gemv_kernel(const uint8_t *__restrict__ blocks, const float *__restrict__ x, float *__restrict__ y, int M,
                int64_t N, int K) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t n = static_cast<int64_t>(blockIdx.x) * kQ80RowsPerCta + warp;
    if (n >= N) return;   // (warp-uniform)
    wait_prior_grid();    // x may belong to the kernel before this one in the stream
    const int nblk = K / 32;
    const uint16_t *row = reinterpret_cast<const uint16_t *>(blocks + n * static_cast<int64_t>(nblk) * 34);
    float acc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = 0.0f;
    for (int b = lane; b < nblk; b += 32) {
        const uint16_t *h = row + b * 17;           // block b: 17 half-words
        const float d = half_bits_to_float(ldg_u16(h));
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = ldg_u16(h + 1 + 2 * i) | (ldg_u16(h + 2 + 2 * i) << 16);
        float s[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) s[m] = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            // codes 4i .. 4i + 3 of the block, sign-extended and widened exactly
            float q[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) q[e] = static_cast<float>(static_cast<int32_t>(w[i] << (24 - 8 * e)) >> 24);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (m < M) {
                    const float4 xv = __ldg(reinterpret_cast<const float4 *>(x + static_cast<int64_t>(m) * K + b * 32) + i);
                    s[m] = fmaf(q[0], xv.x, s[m]);
                    s[m] = fmaf(q[1], xv.y, s[m]);
                    s[m] = fmaf(q[2], xv.z, s[m]);
                    s[m] = fmaf(q[3], xv.w, s[m]);
                }
            }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = fmaf(d, s[m], acc[m]);
    }
    allow_next_grid();
#pragma unroll
    for (int m = 0; m < MT; ++m) {
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], o);
        if (lane == m && m < M) y[static_cast<int64_t>(m) * N + n] = acc[m];
    }
}

template <int MT>
int launch_q80_mt(const uint8_t *blocks, const float *x, float *y, int M, int64_t N, int K, cudaStream_t stream) {
    const int64_t grid = (N + kQ80RowsPerCta - 1) / kQ80RowsPerCta;
    if (grid > 0x7fffffffLL) return Q4_ERR_UNSUPPORTED;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(kQ80Threads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    add_overlap_attr(cfg, attr);
    cudaError_t e = cudaLaunchKernelEx(&cfg, q80_gemv_kernel<MT>, blocks, x, y, M, N, K);
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return Q4_ERR_CUDA;
    }
    return launch_status();
}

}  // namespace

int launch_q80gemv(const uint8_t *blocks, const float *x, float *y, int M, int64_t N, int K, cudaStream_t stream) {
    if (!call_options().exact_x && stream_q80_applies(M, N, K, blocks))
        return launch_q4gemv_stream_q80(blocks, x, y, N, K, stream);
    if (M <= 1) return launch_q80_mt<1>(blocks, x, y, M, N, K, stream);
    if (M <= 2) return launch_q80_mt<2>(blocks, x, y, M, N, K, stream);
    if (M <= 4) return launch_q80_mt<4>(blocks, x, y, M, N, K, stream);
    if (M <= 8) return launch_q80_mt<8>(blocks, x, y, M, N, K, stream);
    return launch_q80_mt<16>(blocks, x, y, M, N, K, stream);
}

}  // namespace q4
