// aux_kernels.cu -- test and measurement kernels: the dequantised weight
// matrix written out with the GEMV's own decode (for bit-exact checks), and a
// 128-bit read-bandwidth probe.
#include "q4_common.cuh"

#include <cuda_bf16.h>

namespace q4 {

namespace {

// One thread per 16-byte chunk (32 codes of one row, inside one group).
template <bool BF16>
__global__ void __launch_bounds__(256)
dequant_kernel(const uint8_t *codes, const uint16_t *scales, const uint8_t *zeros, void *out,
               int64_t N, int K, int nb, int zrow, int gshift) {
    const int C = K / 32;
    const int64_t total = N * C;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t n = i / C;
        const int c = static_cast<int>(i - n * C);
        const int grp = c >> gshift;
        const uint4 cw = ldg_stream(codes + n * (K / 2) + static_cast<int64_t>(c) * 16);
        const float s = half_bits_to_float(ldg_u16(scales + n * nb + grp));
        uint32_t z = 8u;
        if (zeros != nullptr) {
            const uint32_t zb = ldg_u8(zeros + n * zrow + (grp >> 1));
            z = (grp & 1) ? (zb >> 4) : (zb & 0xFu);
        }
        const ZeroTerms zt = zero_terms(z);
        const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
        float v[32];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const WordTerms d = decode_word(words[w], zt);
            const float e[8] = {d.d01.x, d.d01.y, d.d23.x, d.d23.y, d.d45.x, d.d45.y, d.d67.x, d.d67.y};
#pragma unroll
            for (int p = 0; p < 8; ++p) v[8 * w + p] = (e[p] * inv_e(p)) * s;  // both products exact
        }
        const int64_t base = n * K + static_cast<int64_t>(c) * 32;
        if constexpr (BF16) {
            uint4 *o = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(out) + base);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t pk[4];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[8 * q + 2 * h], v[8 * q + 2 * h + 1]);
                    pk[h] = *reinterpret_cast<const uint32_t *>(&b2);
                }
                o[q] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
        } else {
            float4 *o = reinterpret_cast<float4 *>(static_cast<float *>(out) + base);
#pragma unroll
            for (int q = 0; q < 8; ++q) o[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
    }
}

// 128-bit loads folded by addition; each CTA writes one partial sum.
__global__ void __launch_bounds__(256)
read_probe_kernel(const float4 *buf, int64_t n16, float *partial) {
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    for (; i + 3 * stride < n16; i += 4 * stride) {
        const uint4 v0 = ldg_stream(buf + i);
        const uint4 v1 = ldg_stream(buf + i + stride);
        const uint4 v2 = ldg_stream(buf + i + 2 * stride);
        const uint4 v3 = ldg_stream(buf + i + 3 * stride);
        a0 += (__uint_as_float(v0.x) + __uint_as_float(v0.y)) + (__uint_as_float(v0.z) + __uint_as_float(v0.w));
        a1 += (__uint_as_float(v1.x) + __uint_as_float(v1.y)) + (__uint_as_float(v1.z) + __uint_as_float(v1.w));
        a2 += (__uint_as_float(v2.x) + __uint_as_float(v2.y)) + (__uint_as_float(v2.z) + __uint_as_float(v2.w));
        a3 += (__uint_as_float(v3.x) + __uint_as_float(v3.y)) + (__uint_as_float(v3.z) + __uint_as_float(v3.w));
    }
    for (; i < n16; i += stride) {
        const uint4 v0 = ldg_stream(buf + i);
        a0 += (__uint_as_float(v0.x) + __uint_as_float(v0.y)) + (__uint_as_float(v0.z) + __uint_as_float(v0.w));
    }
    float s = (a0 + a1) + (a2 + a3);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    __shared__ float ws[8];
    if ((threadIdx.x & 31) == 0) ws[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) t += ws[w];
        partial[blockIdx.x] = t;
    }
}

}  // namespace

int launch_dequant(const uint8_t *codes, const uint16_t *scales, const uint8_t *zeros, void *w,
                   bool bf16, int64_t N, int K, int group, cudaStream_t stream) {
    const int nb = K / group;
    const int zrow = (nb + 1) / 2;
    const int gshift = group == 32 ? 0 : (group == 64 ? 1 : 2);
    const int64_t total = N * (K / 32);
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = static_cast<int64_t>(device_info().sms) * 8;
    if (blocks > cap) blocks = cap;
    if (bf16)
        dequant_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(codes, scales, zeros, w, N, K,
                                                                               nb, zrow, gshift);
    else
        dequant_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(codes, scales, zeros, w, N, K,
                                                                                nb, zrow, gshift);
    return launch_status();
}

int launch_read_probe(const float4 *buf, int64_t n16, float *partial, int blocks, cudaStream_t stream) {
    read_probe_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(buf, n16, partial);
    return launch_status();
}

}  // namespace q4
