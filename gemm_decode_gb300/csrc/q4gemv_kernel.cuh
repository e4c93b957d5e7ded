// q4gemv_kernel.cuh -- the decode-time int4 GEMV kernel (1 <= M <= 16) on CUDA cores.
//
// Computes y[m][n] = sum_k (q[n][k] - z[n][k/g]) * s[n][k/g] * x[m][k]
// (gerbil GPU-engine kernel reference, "3. MatMulInt4": "Computes",
// "Dequantization"; weights in the MatMulNBits layout of the Refractometer
// page's "b) q4 GEMV" sweep).
//
// Work decomposition.  A row of codes is K/2 bytes = C = K/32 "chunks" of 16
// bytes; one chunk holds 32 consecutive codes and lies inside one group (the
// group size is a multiple of 32).  Each row is served by L consecutive lanes
// of a warp (a "slot"); lane j of the slot takes chunks j, j+L, j+2L, ... so
// that the L lanes of a slot read L*16 contiguous bytes per load.  A thread
// owns R rows (the same chunk positions in each), so every x value it reads
// from shared memory feeds R rows.  A CTA of 8 warps covers 8 * R * 32/L rows.
// For long K and few rows the chunk range is split over S CTAs of one
// thread-block cluster; their partial sums are added in a fixed order through
// distributed shared memory (no workspace, no atomics, deterministic).
//
// Exact in-register decode.  For a 32-bit word of 8 codes (nibble p holds
// k = 8w + p), OR-ing the masked nibble into the fraction of 2^23 gives the
// float 2^23 + e_p * q exactly, with e_p = 16^p for p <= 4 and, after one
// shift of the word by 12 bits, e_p = 16^(p-3) for p = 5, 6, 7.  The zero
// point is formed the same way from z replicated into every nibble, so one
// packed add of -(2^23 + e_p * z) gives e_p * (q - z) exactly.  x is stored
// in shared memory pre-multiplied by 1/e_p (a power of two, exact), so each
// product e_p (q - z) * x_k / e_p is the exact real (q - z) * x_k, rounded
// once by the fused multiply-add; accumulation is binary32.  The group scale
// multiplies the per-chunk sum once.  (q - z) is never rounded, so codes equal
// to their zero point contribute exactly 0.
#pragma once

#include <cooperative_groups.h>

#include "q4_common.cuh"

namespace q4 {

namespace cg = cooperative_groups;

constexpr int kGemvThreads = 256;
constexpr int kGemvWarps = kGemvThreads / 32;
// 32 pre-scaled x values of one chunk + 4 floats of padding: a chunk is 144
// bytes, so the chunks read by the L <= 8 lanes of a slot start on distinct
// 16-byte bank groups.
constexpr int kChunkFloats = 36;
constexpr int kGemvU = 4;   // chunks per row in flight per thread

struct GemvArgs {
    const uint8_t *codes;
    const uint16_t *scales;
    const uint8_t *zeros;
    const float *x;
    float *y;
    int M;
    int N;
    int K;
    int C;       // chunks per row, K / 32
    int nb;      // groups per row, K / g
    int zrow;    // zero-point bytes per row, ceil(nb / 2)
    int gshift;  // log2(g / 32): chunk index >> gshift = group index
    int CS;      // chunks per split
    // fused variant only: gamma[K] (non-null: RMSNorm prologue, eps); swiglu != 0:
    // rows 2i / 2i+1 are a gate / up pair and y[m][i] = silu(gate) * up (y has N / 2 columns)
    const float *gamma;
    float eps;
    int swiglu;
};

template <int MT, int L>
struct GemvShape {
    static constexpr int R = (MT <= 2) ? 2 : 1;
    static constexpr int SLOTS = 32 / L;
    static constexpr int ROWS_PER_WARP = SLOTS * R;
    static constexpr int ROWS_PER_CTA = ROWS_PER_WARP * kGemvWarps;
};

// FUSED (unsplit instances only): x is staged multiplied by a.gamma and every output
// multiplied by 1 / sqrt(mean(x^2) + eps) when a.gamma is set (the RMSNorm prologue),
// and with a.swiglu the gate / up row pairs (slots 2s, 2s + 1: lanes L apart) leave
// silu(gate) * up.
// Q40: the weights are Q4_0 blocks (cera wgpu_gemv_bench.rs block geometry: 32
// elements in 18 bytes), read as a binary16 scale followed by the 16 code bytes of one
// chunk in the packing above, zero point 8; a.codes points at the blocks [N][K/32][18]
// (2-byte aligned), a.scales is unused.  Scale and codes come in as nine 16-bit loads.
template <int MT, int L, bool ASYM, bool SPLIT, bool FUSED = false, bool Q40 = false>
__global__ void __launch_bounds__(kGemvThreads)
q4gemv_kernel(const GemvArgs a) {
    static_assert(!(FUSED && SPLIT), "the fused variant is unsplit");
    static_assert(!(Q40 && (ASYM || FUSED)), "Q4_0 blocks are symmetric and not fused");
    using S = GemvShape<MT, L>;
    constexpr int R = S::R;
    constexpr int SLOTS = S::SLOTS;
    constexpr int U = kGemvU;

    extern __shared__ __align__(16) float smem[];
    float *xs = smem;  // [MT][CS][kChunkFloats]

    const int split = SPLIT ? static_cast<int>(blockIdx.y) : 0;
    const int c_begin = split * a.CS;
    const int nchunks = min(a.C - c_begin, a.CS);
    const int tid = threadIdx.x;
    allow_next_grid();
    wait_prior_grid();   // x and y may belong to the kernel before this one in the stream

    // ---- stage x' = x / e_p for this CTA's chunk range (rows m >= M are zero) ----
    {
        const int per_m = a.CS * 8;  // float4 slots per m
        for (int i = tid; i < MT * per_m; i += kGemvThreads) {
            const int m = i / per_m;
            const int rem = i - m * per_m;
            const int cl = rem >> 3;
            const int f = rem & 7;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (m < a.M && cl < nchunks) {
                v = *reinterpret_cast<const float4 *>(a.x + static_cast<int64_t>(m) * a.K +
                                                      static_cast<int64_t>(c_begin + cl) * 32 + f * 4);
                if (FUSED && a.gamma != nullptr) {
                    const float4 gv = *reinterpret_cast<const float4 *>(a.gamma + static_cast<int64_t>(c_begin + cl) * 32 + f * 4);
                    v.x *= gv.x; v.y *= gv.y; v.z *= gv.z; v.w *= gv.w;
                }
            }
            if (f & 1) {  // positions 4..7 of a word
                v.x *= 0x1p-16f; v.y *= 0x1p-8f; v.z *= 0x1p-12f; v.w *= 0x1p-16f;
            } else {      // positions 0..3
                v.y *= 0x1p-4f; v.z *= 0x1p-8f; v.w *= 0x1p-12f;
            }
            *reinterpret_cast<float4 *>(xs + (m * a.CS + cl) * kChunkFloats + f * 4) = v;
        }
    }
    // (fused RMSNorm) per-warp sums of x^2 of every row of x, after the staged tile
    [[maybe_unused]] float *nrm = smem + MT * a.CS * kChunkFloats;   // [kGemvWarps][MT]
    if constexpr (FUSED) {
        if (a.gamma != nullptr) {
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                float t = 0.f;
                if (m < a.M)
                    for (int k = tid; k < a.K; k += kGemvThreads) {
                        const float v = a.x[static_cast<int64_t>(m) * a.K + k];
                        t = fmaf(v, v, t);
                    }
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
                if ((tid & 31) == 0) nrm[(tid >> 5) * MT + m] = t;
            }
        }
    }
    __syncthreads();

    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int slot = lane / L;
    const int j = lane % L;
    const int64_t row0 = static_cast<int64_t>(blockIdx.x) * S::ROWS_PER_CTA +
                         warp * S::ROWS_PER_WARP + slot;

    int64_t rowc[R];
    bool rvalid[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t n = row0 + r * SLOTS;
        rvalid[r] = n < a.N;
        rowc[r] = rvalid[r] ? n : (a.N - 1);  // clamped: loads stay in bounds
    }
    const int64_t pitch = a.K / 2;

    float acc[R][MT];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[r][m] = 0.f;

    for (int cb = j; cb < nchunks; cb += L * U) {
        uint4 cw[R][U];
        uint32_t sc[R][U];
        uint32_t zq[R][U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int cl = cb + u * L;
            const int c = c_begin + cl;
            const int grp = c >> a.gshift;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (Q40 && cl < nchunks) {
                    const uint16_t *hw = reinterpret_cast<const uint16_t *>(
                        a.codes + (rowc[r] * a.C + c) * 18);   // block c of row rowc[r]
                    sc[r][u] = ldg_u16(hw);
                    uint32_t h[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) h[i] = ldg_u16(hw + 1 + i);
                    cw[r][u] = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16),
                                          h[6] | (h[7] << 16));
                    zq[r][u] = 8u;
                } else if (cl < nchunks) {
                    cw[r][u] = ldg_stream(a.codes + rowc[r] * pitch + static_cast<int64_t>(c) * 16);
                    sc[r][u] = ldg_u16(a.scales + rowc[r] * a.nb + grp);
                    if (ASYM) {
                        const uint32_t zb = ldg_u8(a.zeros + rowc[r] * a.zrow + (grp >> 1));
                        zq[r][u] = (grp & 1) ? (zb >> 4) : (zb & 0xFu);
                    } else {
                        zq[r][u] = 8u;
                    }
                } else {
                    cw[r][u] = make_uint4(0u, 0u, 0u, 0u);
                    sc[r][u] = 0u;
                    zq[r][u] = 0u;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int cl = cb + u * L;
            if (cl >= nchunks) continue;
            const float4 *xc = reinterpret_cast<const float4 *>(xs + cl * kChunkFloats);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const ZeroTerms zt = zero_terms(zq[r][u]);
                float2 pa[MT], pb[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    pa[m] = make_float2(0.f, 0.f);
                    pb[m] = make_float2(0.f, 0.f);
                }
                const uint32_t words[4] = {cw[r][u].x, cw[r][u].y, cw[r][u].z, cw[r][u].w};
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const WordTerms d = decode_word(words[w], zt);
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        const float4 *xm = xc + m * a.CS * (kChunkFloats / 4);
                        const float4 xa = xm[2 * w];
                        const float4 xb = xm[2 * w + 1];
                        pa[m] = __ffma2_rn(d.d01, make_float2(xa.x, xa.y), pa[m]);
                        pb[m] = __ffma2_rn(d.d23, make_float2(xa.z, xa.w), pb[m]);
                        pa[m] = __ffma2_rn(d.d45, make_float2(xb.x, xb.y), pa[m]);
                        pb[m] = __ffma2_rn(d.d67, make_float2(xb.z, xb.w), pb[m]);
                    }
                }
                const float s = half_bits_to_float(sc[r][u]);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const float2 p = __fadd2_rn(pa[m], pb[m]);
                    acc[r][m] = fmaf(s, p.x + p.y, acc[r][m]);
                }
            }
        }
    }

    // ---- reduce over the L lanes of a slot (every lane ends with the sum) ----
#pragma unroll
    for (int off = L / 2; off >= 1; off >>= 1)
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m)
                acc[r][m] += __shfl_xor_sync(0xffffffffu, acc[r][m], off);

    if constexpr (FUSED) {
        float rn[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            rn[m] = 1.f;
            if (a.gamma != nullptr) {
                float t = 0.f;
                for (int w = 0; w < kGemvWarps; ++w) t += nrm[w * MT + m];
                rn[m] = rsqrtf(t / static_cast<float>(a.K) + a.eps);
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const float v = acc[r][m] * rn[m];
                const int64_t n = row0 + r * SLOTS;
                const bool mine = ((r * MT + m) % L) == j && rvalid[r] && m < a.M;
                if (a.swiglu) {
                    const float up = __shfl_xor_sync(0xffffffffu, v, L);   // row n + 1: the next slot
                    if (mine && (n & 1) == 0)
                        a.y[static_cast<int64_t>(m) * (a.N / 2) + (n >> 1)] = v / (1.0f + expf(-v)) * up;
                } else if (mine) {
                    a.y[static_cast<int64_t>(m) * a.N + n] = v;
                }
            }
    } else if constexpr (!SPLIT) {
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m)
                if (((r * MT + m) % L) == j && rvalid[r] && m < a.M)
                    a.y[static_cast<int64_t>(m) * a.N + row0 + r * SLOTS] = acc[r][m];
    } else {
        // Partials of this CTA's chunk range -> shared memory, then the cluster's
        // CTAs each finish a share of the rows by adding all ranks in rank order.
        float *red = smem + MT * a.CS * kChunkFloats;  // [ROWS_PER_CTA][MT]
        const int local0 = warp * S::ROWS_PER_WARP + slot;
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m)
                if (((r * MT + m) % L) == j)
                    red[(local0 + r * SLOTS) * MT + m] = acc[r][m];
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        const int nsplit = static_cast<int>(cluster.num_blocks());
        const int rank = static_cast<int>(cluster.block_rank());
        for (int i = rank * kGemvThreads + tid; i < S::ROWS_PER_CTA * MT; i += nsplit * kGemvThreads) {
            float v = 0.f;
            for (int q = 0; q < nsplit; ++q) v += cluster.map_shared_rank(red, q)[i];
            const int local = i / MT;
            const int m = i - local * MT;
            const int64_t n = static_cast<int64_t>(blockIdx.x) * S::ROWS_PER_CTA + local;
            if (n < a.N && m < a.M) a.y[static_cast<int64_t>(m) * a.N + n] = v;
        }
        cluster.sync();  // peers' shared memory stays valid until every read is done
    }
}

// Host side: launch one instantiation (defined per MT in q4gemv_mt*.cu).
struct GemvPlan {
    int MT, L, S, CS;
    bool asym;
    size_t smem;
    int row_blocks;
};
template <int MT>
int launch_q4gemv_mt(const GemvPlan &p, const GemvArgs &a, cudaStream_t stream);

}  // namespace q4
