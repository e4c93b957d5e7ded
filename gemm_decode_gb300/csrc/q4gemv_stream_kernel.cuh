// q4gemv_stream_kernel.cuh -- the TMA-streamed M = 1 int4 GEMV kernel template and
// its launcher template.  Each q4gemv_stream_k*.cu instantiates the compile-time
// row geometries of one K (in parallel translation units); q4gemv_stream.cu holds
// the runtime-geometry instance and the dispatch.
#pragma once

#include "q4_common.cuh"
#include "q4gemv_xplanes.cuh"
#include "q4gemv_stream.cuh"

namespace q4 {

using namespace xp;

namespace {

// The geometry an instance works with: compile-time when the instance fixes K, g
// and RG (the tuned decode shapes), else the launcher's.
template <int KC, int GC, int RGC, int UC, bool ASYM, bool FUSED, bool Q40 = false, int MXC = 1, bool Q80 = false>
__device__ __forceinline__ StreamGeo geo_of(const StreamGeo &rt) {
    if constexpr (KC != 0) {
        constexpr StreamGeo g = make_stream_geo(KC, GC, RGC, UC, stream_slots(KC, GC, RGC, UC, ASYM, Q40, MXC, Q80),
                                                ASYM, FUSED, Q40, MXC, Q80);
        return g;
    } else {
        return rt;
    }
}

}  // namespace

// UC: rows per consumer thread and block (compile-time in every instance; the host
// geometry carries the same value).  FUSE (the fused variant, q4gemv_fused_run): bit 0,
// the RMSNorm prologue when a.gamma is set -- a first pass sums x^2 over the row, then
// x is encoded as x * gamma / sqrt(mean(x^2) + eps), so the dot products and the
// reduction are those of the plain kernel; bit 1, the SwiGLU epilogue when a.swiglu is
// set -- the gate / up row pairs leave silu(gate) * up.  FUSE = 4: the weights are Q4_0
// blocks (a.codes; 18 bytes per 32 codes: binary16 scale, then the codes; zero point 8).
// FUSE = 8: a grouped launch (a.seg: several matrices, each served by its own CTAs).
// FUSE = 16: two rows of x (M = 2): x[2][K], y[2][N], every block of codes serving both.
// FUSE = 32: the weights are Q8_0 blocks (a.codes; 34 bytes per 32 codes: binary16 scale,
// then 32 two's-complement 8-bit codes; no zero point).
template <int KC, int GC, int RGC, int UC, bool ASYM, int FUSE>
__global__ void __launch_bounds__(KC ? KC / 32 * RGC + 32 : kStreamMaxTC + 32, 1)
q4gemv_stream_kernel(const StreamArgsOf<FUSE> a) {
    constexpr int U = UC, NRED = kStreamNRed;
    constexpr bool U_POW2 = (U & (U - 1)) == 0;
    constexpr bool NORM = (FUSE & 1) != 0, SWIG = (FUSE & 2) != 0, Q40 = (FUSE & 4) != 0, GROUPED = (FUSE & 8) != 0;
    constexpr int MX = (FUSE & 16) != 0 ? 2 : 1;   // rows of x
    constexpr bool Q80 = (FUSE & 32) != 0;
    static_assert(!Q80 || (!ASYM && (KC == 0 || GC == 32) && FUSE == 32), "Q8_0: group 32, no zero points, plain");
    static_assert(!Q40 || (!ASYM && (KC == 0 || GC == 32) && FUSE == 4), "Q4_0: group 32, symmetric, not fused");
    static_assert(!GROUPED || FUSE == 8, "grouped launches are plain");
    static_assert(MX == 1 || FUSE == 16, "two rows of x: plain launches only");
    const StreamGeo G = geo_of<KC, GC, RGC, UC, ASYM, (FUSE & 3) != 0, Q40, MX, Q80>(a.geo);
    const int D = G.D;
    const int C = G.C;
    extern __shared__ __align__(128) unsigned char smem[];
    const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    const uint32_t s_planes = sbase;
    const uint32_t s_red = sbase + G.OFF_RED;
    const uint32_t s_ring = sbase + G.OFF_RING;
    const uint32_t bar0 = sbase + G.OFF_BAR;
    const uint32_t s_flag = sbase + G.OFF_FLAG;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (D + s); };
    auto redfull = [&](int b) { return bar0 + 8u * (2 * D + b); };
    auto reddone = [&](int b) { return bar0 + 8u * (2 * D + NRED + b); };

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const unsigned long long limit = a.timeout_ns;

    // the matrix this CTA serves (a grouped launch: the segment whose CTA range holds it)
    const uint8_t *w_codes = a.codes;
    const uint16_t *w_scales = a.scales;
    const uint8_t *w_zeros = a.zeros;
    const float *w_x = a.x;
    float *w_y = a.y;
    int64_t w_N = a.N;
    int w_nblocks = a.nblocks;
    int cta = static_cast<int>(blockIdx.x), gsz = static_cast<int>(gridDim.x);
    if constexpr (GROUPED) {
        int first = 0, last = gsz;
#pragma unroll
        for (int g = 0; g < kStreamMaxSeg; ++g) {
            if (g < a.nseg && a.seg[g].cta_begin <= cta) {
                w_codes = a.seg[g].codes;
                w_scales = a.seg[g].scales;
                w_zeros = a.seg[g].zeros;
                w_x = a.seg[g].x;
                w_y = a.seg[g].y;
                w_N = a.seg[g].N;
                w_nblocks = a.seg[g].nblocks;
                first = a.seg[g].cta_begin;
                last = g + 1 < a.nseg ? a.seg[g + 1].cta_begin : gsz;
            }
        }
        cta -= first;
        gsz = last - first;
    }
    // blocks of this CTA (contiguous range)
    const int b_begin = static_cast<int>(static_cast<int64_t>(w_nblocks) * cta / gsz);
    const int b_end = static_cast<int>(static_cast<int64_t>(w_nblocks) * (cta + 1) / gsz);
    const int nbk = b_end - b_begin;

    if (tid == 0) {
        for (int s = 0; s < D; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), G.NWC);
        }
        for (int b = 0; b < NRED; ++b) {
            mbar_init(redfull(b), G.NWC);
            mbar_init(reddone(b), 1);
        }
        sts_volatile_u32(s_flag, 0u);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    allow_next_grid();

    auto aborted = [&]() { return lds_volatile_u32(s_flag) != 0u; };
    auto ib = [&](bool ok) { return q4_in_bounds(ok, a.bounds); };   // bounds-checking builds
    auto fail = [&]() {
        sts_volatile_u32(s_flag, 1u);
        atomicOr(a.status, 1u);
    };

    if (warp == G.NWC) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int issued = 0;
            int s = 0, ph = 0;   // slot and its wrap parity
            for (int i = 0; i < nbk && !aborted(); ++i) {
                if (i >= D && !mbar_wait(empty(s), ph ^ 1, limit)) {
                    fail();
                    break;
                }
                const int64_t row0 = static_cast<int64_t>(b_begin + i) * G.ROWS;
                const int rows = static_cast<int>(w_N - row0 < G.ROWS ? w_N - row0 : G.ROWS);
                const uint32_t dst = s_ring + s * G.SLOT_B;
                const unsigned char *src_c = w_codes + row0 * (C * 16);
                const unsigned char *src_s = reinterpret_cast<const unsigned char *>(w_scales) + row0 * (G.NB * 2);
                const unsigned char *src_z = ASYM ? w_zeros + row0 * G.ZROW : nullptr;
                if (!ib(row0 >= 0 && rows >= 1 && row0 + rows <= w_N && s < D)) {
                    mbar_arrive(full(s));   // (checking builds) keep the ring moving, copy nothing
                } else if constexpr (Q40 || Q80) {
                    // Q4_0 / Q8_0: one stretch of rows * C * 18 (34) bytes (a 16-byte multiple
                    // for a whole block of rows); its largest 16-byte multiple by bulk copy, the
                    // at most 15 bytes left by plain copies, published by the arrive below
                    constexpr int QB = Q40 ? 18 : 34;
                    const unsigned char *src = w_codes + row0 * (C * QB);
                    const int cb = rows * C * QB, cb16 = cb & ~15;
                    unsigned char *sl = smem + G.OFF_RING + s * G.SLOT_B;
                    for (int j = cb16; j < cb; ++j) sl[j] = src[j];
                    mbar_expect_tx(full(s), cb16);
                    bulk_copy(dst, src, cb16, full(s));
                } else if (rows == G.ROWS) {
                    mbar_expect_tx(full(s), G.CODE_B + G.SC_B + G.Z_B);
                    bulk_copy(dst, src_c, G.CODE_B, full(s));
                    bulk_copy(dst + G.CODE_B, src_s, G.SC_B, full(s));
                    if (ASYM) bulk_copy(dst + G.CODE_B + G.SC_B, src_z, G.Z_B, full(s));
                } else {
                    // last, partial block: the codes (rows * C * 16 bytes) and the largest
                    // 16-byte multiples of the scale and zero-point stretches by bulk copy,
                    // the at most 15 bytes left of each by plain copies, which the arrive
                    // below publishes (the stretches start 16-byte aligned: a whole block's
                    // scale and zero bytes are multiples of 16)
                    const int sb = rows * G.NB * 2, zb = ASYM ? rows * G.ZROW : 0;
                    const int sb16 = sb & ~15, zb16 = zb & ~15;
                    unsigned char *sl = smem + G.OFF_RING + s * G.SLOT_B;
                    for (int j = sb16; j < sb; ++j) sl[G.CODE_B + j] = src_s[j];
                    for (int j = zb16; j < zb; ++j) sl[G.CODE_B + G.SC_B + j] = src_z[j];
                    mbar_expect_tx(full(s), rows * C * 16 + sb16 + zb16);
                    bulk_copy(dst, src_c, rows * C * 16, full(s));
                    if (sb16 > 0) bulk_copy(dst + G.CODE_B, src_s, sb16, full(s));
                    if (zb16 > 0) bulk_copy(dst + G.CODE_B + G.SC_B, src_z, zb16, full(s));
                }
                issued = i + 1;
                if (++s == D) {
                    s = 0;
                    ph ^= 1;
                }
            }
            if (aborted()) {
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
    uint32_t *planes = reinterpret_cast<uint32_t *>(smem);
    if constexpr (NORM) {
        if (a.gamma != nullptr) {
            // first pass: this thread's x^2 (the elements it encodes), warp sums in shared
            // memory, a consumer barrier, the row's 1 / sqrt(mean(x^2) + eps)
            float ssq = 0.0f;
            for (int base = 0; base < C; base += G.TC / 4) {
                const int i = base + (tid >> 2);
                if (i < C && ib((i + 1) * 32 <= C * 32)) {
                    const float4 *xc = reinterpret_cast<const float4 *>(w_x + i * 32) + 2 * (tid & 3);
                    const float4 u = xc[0], v = xc[1];
                    ssq = fmaf(u.x, u.x, fmaf(u.y, u.y, fmaf(u.z, u.z, fmaf(u.w, u.w, ssq))));
                    ssq = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ssq))));
                }
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) ssq += __shfl_xor_sync(0xffffffffu, ssq, o);
            if (lane == 0 && ib(warp < 32)) sts_f32(sbase + G.OFF_NORM + 4 * warp, ssq);
            asm volatile("bar.sync 1, %0;" ::"r"(G.TC) : "memory");
            float t = 0.0f;
            for (int w = 0; w < G.NWC; ++w)
                if (ib(w < 32)) t += lds_f32(sbase + G.OFF_NORM + 4 * w);
            const float rnorm = rsqrtf(t / static_cast<float>(C * 32) + a.eps);
            for (int base = 0; base < C; base += G.TC / 4) {
                const int i = base + (tid >> 2);
                const bool in_range = i < C;
                const bool x_ok = ib(!in_range || (i + 1) * 32 <= C * 32);
                encode_chunk4_gamma_scaled(w_x + (in_range ? i : 0) * 32, a.gamma + (in_range ? i : 0) * 32, rnorm,
                                           in_range && x_ok, in_range, planes + (in_range ? i : 0) * kPlaneWords,
                                           tid & 3);
            }
        } else {
            for (int base = 0; base < C; base += G.TC / 4) {
                const int i = base + (tid >> 2);
                const bool in_range = i < C;
                const bool x_ok = ib(!in_range || (i + 1) * 32 <= C * 32);
                encode_chunk4(w_x + (in_range ? i : 0) * 32, in_range && x_ok, in_range,
                              planes + (in_range ? i : 0) * kPlaneWords, tid & 3);
            }
        }
    } else {
#pragma unroll
        for (int m = 0; m < MX; ++m) {   // row m of x: planes [m][C]
            for (int base = 0; base < C; base += G.TC / 4) {
                const int i = base + (tid >> 2);
                const bool in_range = i < C;
                const bool x_ok = ib(!in_range || (i + 1) * 32 <= C * 32);
                encode_chunk4(w_x + m * C * 32 + (in_range ? i : 0) * 32, in_range && x_ok, in_range,
                              planes + (m * C + (in_range ? i : 0)) * kPlaneWords, tid & 3);
            }
        }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(G.TC) : "memory");
    Planes P[MX];
#pragma unroll
    for (int m = 0; m < MX; ++m) {
        const uint32_t pa = s_planes + (m * C + c) * kPlaneWords * 4;
        uint32_t w[28];
#pragma unroll
        for (int i = 0; i < 7; ++i) {
            const uint4 v = lds128(pa + 16 * i);
            w[4 * i] = v.x;
            w[4 * i + 1] = v.y;
            w[4 * i + 2] = v.z;
            w[4 * i + 3] = v.w;
        }
#pragma unroll
        for (int i = 0; i < 24; ++i) P[m].p[i] = w[i];
        P[m].s_lo = static_cast<int>(w[24]);
        P[m].s_hi = static_cast<int>(w[25]);
        P[m].f = __uint_as_float(w[27]);
    }
    const int grp = c >> G.GSHIFT;
    // byte offsets of this thread's data inside a slot for sub-row u = 0, and the
    // distance between sub-rows u and u + 1 (RG rows)
    const uint32_t off_c = (r * C + c) * 16, str_c = G.RG * C * 16;
    const uint32_t off_s = G.CODE_B + (r * G.NB + grp) * 2, str_s = G.RG * G.NB * 2;
    const uint32_t off_z = G.CODE_B + G.SC_B + r * G.ZROW + (grp >> 1), str_z = G.RG * G.ZROW;
    const int zsh = (grp & 1) * 4;
    // where this thread's partial of sub-row u = 0 goes in a partial-sum buffer: with
    // whole-warp rows, lane l of the warp holds the warp total of sub-row l >> NSH
    constexpr int NSH = U == 1 ? 5 : (U == 2 ? 4 : (U == 4 ? 3 : (U == 8 ? 2 : (U == 16 ? 1 : 0))));
    const bool red_writer = !G.WRED || (lane & ((1 << NSH) - 1)) == 0;
    const int red_u = G.WRED ? (lane >> NSH) : 0;
    const uint32_t red_off = G.WRED ? ((red_u * G.RG + r) * G.RED_LD + (c >> 5)) * 4 : (r * G.RED_LD + c) * 4;
    const uint32_t str_red = G.RG * G.RED_LD * 4;
    const uint32_t red_m = G.ROWS * G.RED_LD * 4;   // bytes of one row of x's partials in a buffer

    // Sum the partials of rows [lo, hi) of a block and store them: ql lanes per row
    // (a power of two), each adding every ql-th partial, combined by shuffles.
    // ql = 1 is a lane per row, partials in order.
    auto reduce_rows = [&](int buf, int64_t row0, int lo, int hi, int ql) {
      const int q = lane & (ql - 1);
#pragma unroll
      for (int mr = 0; mr < MX; ++mr) {   // each row of x: its partials, its row of y
        const uint32_t src = s_red + buf * G.RED_B + mr * red_m;
        float *yrow = w_y + mr * w_N;
        for (int base = lo; base < hi; base += 32 / ql) {   // warp-uniform trip count
            const int rho = base + lane / ql;
            const bool mine = rho < hi;
            float acc = 0.0f;
            if (mine) {
#pragma unroll 4
                for (int p = q; p < G.PARTS; p += ql)
                    if (ib(rho * G.RED_LD + p < G.ROWS * G.RED_LD)) acc += lds_f32(src + (rho * G.RED_LD + p) * 4);
            }
            for (int o = ql >> 1; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if constexpr (SWIG) {
                if (a.swiglu) {
                    // row rho + 1 (the up row of the pair) sits ql lanes further on
                    const float up = __shfl_xor_sync(0xffffffffu, acc, ql);
                    if (mine && q == 0 && (rho & 1) == 0 && row0 + rho + 1 < w_N)
                        w_y[(row0 + rho) >> 1] = acc / (1.0f + expf(-acc)) * up;
                    continue;
                }
            }
            if (mine && q == 0 && row0 + rho < w_N) yrow[row0 + rho] = acc;
        }
      }
    };

    int s = 0, ph = 0;       // ring slot of block i and its wrap parity
    int rb = 0, rph = 0;     // partial-sum buffer of block i and its wrap parity
    int pb = 0, pph = 0;     // the same for block i - 1 (set at the end of each iteration)
    int rw = 0;              // the warp that reduces block i - 1: (i - 1) mod NWC
    for (int i = 0; i < nbk; ++i) {
        if (aborted()) break;
        if (!mbar_wait(full(s), ph, limit)) {
            fail();
            break;
        }
        if (i >= NRED && !mbar_wait(reddone(rb), rph ^ 1, limit)) {
            fail();
            break;
        }
        const uint32_t sl = s_ring + s * G.SLOT_B;
        const uint32_t rd = s_red + rb * G.RED_B;
        float v[MX][U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            uint4 cw;
            uint32_t sh;
            if constexpr (Q80) {
                // block (r + RG u) * C + c: its scale at 34 * block, its 32 code bytes from
                // 34 * block + 2 (2-byte aligned): nine words from the 4-byte boundary below,
                // shifted by 0 or 16 bits (the ninth may reach 4 bytes past the block, inside
                // the slot's 16 bytes of slack after its last block)
                const uint32_t boff = static_cast<uint32_t>((r * C + c) * 34) + u * static_cast<uint32_t>(G.RG * C * 34);
                const bool b_ok = ib(boff + 34 <= static_cast<uint32_t>(G.CODE_B));
                const uint32_t cstart = boff + 2, base = cstart & ~3u, shift = (cstart & 3u) * 8u;
                uint32_t w[9];
#pragma unroll
                for (int i = 0; i < 9; ++i) w[i] = b_ok ? lds_u32(sl + base + 4 * i) : 0u;
                uint32_t c8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) c8[i] = __funnelshift_r(w[i], w[i + 1], shift);
                const uint32_t dh = b_ok ? lds_u16(sl + boff) : 0u;
                const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(dh)));
                v[0][u] = (d * P[0].f) * chunk_dot_q8(c8, P[0]);
                continue;
            }
            if constexpr (Q40) {
                // block (r + RG u) * C + c: its scale at 18 * block, its 16 code bytes from
                // 18 * block + 2 (2-byte aligned): five words from the 4-byte boundary below,
                // shifted by 0 or 16 bits (the fifth word may reach 4 bytes past the block,
                // inside the slot's 16 bytes of slack after its last block)
                const uint32_t boff = static_cast<uint32_t>((r * C + c) * 18) + u * static_cast<uint32_t>(G.RG * C * 18);
                const bool b_ok = ib(boff + 18 <= static_cast<uint32_t>(G.CODE_B));
                const uint32_t cstart = boff + 2, base = cstart & ~3u, shift = (cstart & 3u) * 8u;
                uint32_t w[5] = {0u, 0u, 0u, 0u, 0u};
                if (b_ok) {
#pragma unroll
                    for (int i = 0; i < 5; ++i) w[i] = lds_u32(sl + base + 4 * i);
                }
                cw = make_uint4(__funnelshift_r(w[0], w[1], shift), __funnelshift_r(w[1], w[2], shift),
                                __funnelshift_r(w[2], w[3], shift), __funnelshift_r(w[3], w[4], shift));
                sh = b_ok ? lds_u16(sl + boff) : 0u;
            } else {
                const bool c_ok = ib(off_c + u * str_c + 16 <= static_cast<uint32_t>(G.CODE_B));
                const bool s_ok = ib(off_s + u * str_s + 2 <= static_cast<uint32_t>(G.CODE_B + G.SC_B));
                cw = c_ok ? lds128(sl + off_c + u * str_c) : make_uint4(0u, 0u, 0u, 0u);
                sh = s_ok ? lds_u16(sl + off_s + u * str_s) : 0u;
            }
            const bool z_ok = !ASYM || ib(off_z + u * str_z + 1 <= static_cast<uint32_t>(G.CODE_B + G.SC_B + G.Z_B));
            const int z = ASYM ? (z_ok ? static_cast<int>((lds_u8(sl + off_z + u * str_z) >> zsh) & 0xFu) : 8) : 8;
            const float sc = __half2float(__ushort_as_half(static_cast<unsigned short>(sh)));
            if constexpr (MX == 1) {
                v[0][u] = (sc * P[0].f) * chunk_dot(cw, z, P[0]);
            } else {
                float d0, d1;
                chunk_dot2(cw, z, P[0], P[1], d0, d1);
                v[0][u] = (sc * P[0].f) * d0;
                v[1][u] = (sc * P[1].f) * d1;
            }
        }
        bool summed = false;
        if constexpr (U_POW2) {
            if (G.WRED) {   // (the host pairs whole-warp rows with a power-of-two U only)
#pragma unroll
                for (int m = 0; m < MX; ++m) {
                    const float t = warp_sum_many<U>(v[m], lane);
                    if (red_writer &&
                        ib(rb * G.RED_B + m * red_m + red_off + 4 <= static_cast<uint32_t>(kStreamNRed * G.RED_B)))
                        sts_f32(rd + m * red_m + red_off, t);
                }
                summed = true;
            }
        }
        if (!summed) {
#pragma unroll
            for (int m = 0; m < MX; ++m)
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (ib(rb * G.RED_B + m * red_m + red_off + u * str_red + 4 <=
                           static_cast<uint32_t>(kStreamNRed * G.RED_B)))
                        sts_f32(rd + m * red_m + red_off + u * str_red, v[m][u]);
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(empty(s));      // slot s may be refilled
            mbar_arrive(redfull(rb));   // this warp's partials of block i are written
        }
        // deferred reduction of block i-1 by one (rotating) consumer warp
        if (i >= 1 && warp == rw) {
            if (!mbar_wait(redfull(pb), pph, limit)) {
                fail();
                break;
            }
            reduce_rows(pb, static_cast<int64_t>(b_begin + i - 1) * G.ROWS, 0, G.ROWS, 1);
            __syncwarp();
            if (lane == 0) mbar_arrive(reddone(pb));
        }
        if (i >= 1 && ++rw == G.NWC) rw = 0;
        pb = rb;
        pph = rph;
        if (++rb == NRED) {
            rb = 0;
            rph ^= 1;
        }
        if (++s == D) {
            s = 0;
            ph ^= 1;
        }
    }
    // the last block's reduction.  With per-thread partials (many per row) and a
    // compile-time geometry it is shared by all consumer warps, none of which has a
    // block left: warp w sums rows [w * rpw, (w + 1) * rpw), ql lanes per row.
    // Otherwise the next warp of the rotation does all of it, as for the other
    // blocks (measured faster with per-warp partials, and it keeps the registers of
    // the runtime-geometry instance down).
    if (nbk > 0 && !aborted()) {
        int lo = 0, hi = G.ROWS, ql = 1;
        if (KC == 0 || G.WRED) {
            if (warp != (nbk - 1) % G.NWC) hi = 0;
        } else {
            int rpw = (G.ROWS + G.NWC - 1) / G.NWC;
            if (SWIG && a.swiglu) rpw = (rpw + 1) & ~1;   // gate / up pairs stay in one warp
            lo = warp * rpw < G.ROWS ? warp * rpw : G.ROWS;
            hi = lo + rpw < G.ROWS ? lo + rpw : G.ROWS;
            while (ql * 2 * rpw <= 32 && ql < G.PARTS) ql *= 2;
        }
        const int lb = (nbk - 1) % NRED;
        if (lo < hi) {
            if (!mbar_wait(redfull(lb), ((nbk - 1) / NRED) & 1, limit))
                fail();
            else
                reduce_rows(lb, static_cast<int64_t>(b_end - 1) * G.ROWS, lo, hi, ql);
        }
    }
}

template <int KC, int GC, int RGC, int UC, bool ASYM, int FUSE = 0>
int launch_stream(const StreamArgs &a0, cudaStream_t stream) {
    auto kern = q4gemv_stream_kernel<KC, GC, RGC, UC, ASYM, FUSE>;
    const StreamGeo &g = a0.geo;
    const int T = g.TC + 32;
    static std::atomic<int> configured[64];   // largest dynamic shared memory set so far, per device
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && configured[dev] < g.SMEM) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             device_info().smem_optin);
        if (e != cudaSuccess) {
            set_cuda_error(e);
            return Q4_ERR_CUDA;
        }
        configured[dev] = device_info().smem_optin;
    }
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, T, g.SMEM);
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return Q4_ERR_CUDA;
    }
    if (per_sm < 1) return Q4_ERR_UNSUPPORTED;
    StreamArgs a = a0;
    a.nblocks = static_cast<int>((a.N + g.ROWS - 1) / g.ROWS);
    int grid = per_sm * device_info().sms;
    if (grid > a.nblocks) grid = a.nblocks;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(T), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(g.SMEM);
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


// A grouped launch: the CTAs a full grid holds (resident CTAs per SM x SMs) are shared out
// over the matrices (stream_assign_ctas), then one launch serves them all.
template <int KC, int GC, int RGC, int UC, bool ASYM>
int launch_stream_grouped(StreamGroupArgs &a, cudaStream_t stream) {
    auto kern = q4gemv_stream_kernel<KC, GC, RGC, UC, ASYM, 8>;
    const StreamGeo &g = a.geo;
    const int T = g.TC + 32;
    static std::atomic<int> configured[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && configured[dev] < g.SMEM) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             device_info().smem_optin);
        if (e != cudaSuccess) {
            set_cuda_error(e);
            return Q4_ERR_CUDA;
        }
        configured[dev] = device_info().smem_optin;
    }
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, T, g.SMEM);
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return Q4_ERR_CUDA;
    }
    if (per_sm < 1) return Q4_ERR_UNSUPPORTED;
    const int grid = stream_assign_ctas(a, per_sm * device_info().sms);
    if (grid < 1) return Q4_ERR_UNSUPPORTED;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(T), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(g.SMEM);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    add_overlap_attr(cfg, attr);
    e = cudaLaunchKernelEx(&cfg, kern, static_cast<const StreamGroupArgs &>(a));
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return Q4_ERR_CUDA;
    }
    return launch_status();
}

template <int KV, int GV, int RGV>
int launch_stream_grouped_kg(StreamGroupArgs &a, bool asym, cudaStream_t s) {
    constexpr int UV = stream_u(KV);
    return asym ? launch_stream_grouped<KV, GV, RGV, UV, true>(a, s) : launch_stream_grouped<KV, GV, RGV, UV, false>(a, s);
}

template <int KV, int GV, int RGV>
int launch_stream_kg(const StreamArgs &a, bool asym, int fuse, cudaStream_t s) {
    constexpr int UV = stream_u(KV);
    if (fuse == 4) {   // Q4_0 blocks: group 32, symmetric
        if constexpr (GV == 32) return asym ? Q4_ERR_UNSUPPORTED : launch_stream<KV, 32, RGV, UV, false, 4>(a, s);
        return Q4_ERR_UNSUPPORTED;
    }
    if (fuse == 32) {   // Q8_0 blocks: group 32, no zero points
        constexpr int UQ = stream_q80_u(KV);
        if constexpr (GV == 32) return asym ? Q4_ERR_UNSUPPORTED : launch_stream<KV, 32, RGV, UQ, false, 32>(a, s);
        return Q4_ERR_UNSUPPORTED;
    }
    if (fuse == 16) {   // two rows of x: the one-CTA-per-SM geometries (K >= 2048)
        if constexpr (KV >= 2048)
            return asym ? launch_stream<KV, GV, RGV, UV, true, 16>(a, s) : launch_stream<KV, GV, RGV, UV, false, 16>(a, s);
        return Q4_ERR_UNSUPPORTED;
    }
    switch (fuse) {
        case 0: return asym ? launch_stream<KV, GV, RGV, UV, true, 0>(a, s) : launch_stream<KV, GV, RGV, UV, false, 0>(a, s);
        case 1: return asym ? launch_stream<KV, GV, RGV, UV, true, 1>(a, s) : launch_stream<KV, GV, RGV, UV, false, 1>(a, s);
        case 3: return asym ? launch_stream<KV, GV, RGV, UV, true, 3>(a, s) : launch_stream<KV, GV, RGV, UV, false, 3>(a, s);
        default: return Q4_ERR_UNSUPPORTED;
    }
}

// One translation unit per K instantiates the compile-time geometries of that K (plain,
// RMSNorm, RMSNorm + SwiGLU, Q4_0, Q8_0, grouped, and for K >= 2048 two rows of x).
#define Q4_STREAM_K_LAUNCHER(KV, RGV)                                                                    \
    int launch_stream_k##KV(const StreamArgs &a, int group, bool asym, int fuse, cudaStream_t s) {    \
        switch (group) {                                                                              \
            case 32: return launch_stream_kg<KV, 32, RGV>(a, asym, fuse, s);                          \
            case 64: return launch_stream_kg<KV, 64, RGV>(a, asym, fuse, s);                          \
            case 128: return launch_stream_kg<KV, 128, RGV>(a, asym, fuse, s);                        \
            default: return Q4_ERR_UNSUPPORTED;                                                       \
        }                                                                                             \
    }                                                                                                 \
    int launch_stream_grouped_k##KV(StreamGroupArgs &a, int group, bool asym, cudaStream_t s) {       \
        switch (group) {                                                                              \
            case 32: return launch_stream_grouped_kg<KV, 32, RGV>(a, asym, s);                        \
            case 64: return launch_stream_grouped_kg<KV, 64, RGV>(a, asym, s);                        \
            case 128: return launch_stream_grouped_kg<KV, 128, RGV>(a, asym, s);                      \
            default: return Q4_ERR_UNSUPPORTED;                                                       \
        }                                                                                             \
    }

}  // namespace q4
