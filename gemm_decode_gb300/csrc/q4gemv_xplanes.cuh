// q4gemv_xplanes.cuh -- device helpers shared by the dp4a GEMV kernels: the
// 24-bit block-scaled byte-plane encoding of x, the exact integer chunk dot
// product, cp.async and mbarrier primitives.
#pragma once

#include "q4_common.cuh"

namespace q4 {
namespace xp {

constexpr int kPlaneWords = 28;  // 24 plane words + S_lo + S_hi + (unused) + chunk scale 2^(E-22)

__device__ __forceinline__ int dp4a_uu(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_su(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src));
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N));
}

// Encode one 32-element chunk of x into the plane layout, four threads per chunk
// (the four consecutive lanes 4j..4j+3 of a warp; thread q owns elements
// 8q..8q+7, i.e. code word q).  With 2^(E-1) <= max |x| < 2^E over the chunk,
// every element k is held as the 24-bit integer m_k = rint(x_k 2^(22-E))
// (|m_k| <= 2^22), i.e. to within 2^(E-23) <= 2^-22 max |x|.  For word w
// (elements 8w..8w+7) and plane b, word 6w+2b holds the b-th byte of m for the
// even elements 8w, 8w+2, 8w+4, 8w+6 and word 6w+2b+1 that of the odd
// elements; plane 2 is the signed top byte.  Words 24/25 hold the plane sums
// over the chunk (planes 0+1 combined as the sum of byte0 + 256 byte1, and
// plane 2), word 27 the chunk scale 2^(E-22).
// `valid` false encodes zeros; `store` false skips the stores (the shuffles
// still run: all lanes take part).
__device__ __forceinline__ void encode_values8(const float (&v)[8], bool store, uint32_t *pw, int q);

__device__ __forceinline__ void encode_chunk4(const float *xc, bool valid, bool store, uint32_t *pw, int q) {
    float v[8];
    if (valid) {
        const float4 a = reinterpret_cast<const float4 *>(xc)[2 * q];
        const float4 b = reinterpret_cast<const float4 *>(xc)[2 * q + 1];
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = 0.0f;
    }
    encode_values8(v, store, pw, q);
}

// The same for the fused RMSNorm prologue: encodes x[k] * gamma[k] (gc: the chunk's
// 32 gamma values) and adds this thread's sum of x[k]^2 to ssq.
__device__ __forceinline__ void encode_chunk4_gamma(const float *xc, const float *gc, bool valid, bool store,
                                                    uint32_t *pw, int q, float &ssq) {
    float v[8];
    if (valid) {
        const float4 a = reinterpret_cast<const float4 *>(xc)[2 * q];
        const float4 b = reinterpret_cast<const float4 *>(xc)[2 * q + 1];
        const float4 ga = reinterpret_cast<const float4 *>(gc)[2 * q];
        const float4 gb = reinterpret_cast<const float4 *>(gc)[2 * q + 1];
        const float xv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        const float gv[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            ssq = fmaf(xv[i], xv[i], ssq);
            v[i] = xv[i] * gv[i];
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = 0.0f;
    }
    encode_values8(v, store, pw, q);
}

// The same with the RMSNorm factor folded in: encodes x[k] * gamma[k] * r.
__device__ __forceinline__ void encode_chunk4_gamma_scaled(const float *xc, const float *gc, float r, bool valid,
                                                           bool store, uint32_t *pw, int q) {
    float v[8];
    if (valid) {
        const float4 a = reinterpret_cast<const float4 *>(xc)[2 * q];
        const float4 b = reinterpret_cast<const float4 *>(xc)[2 * q + 1];
        const float4 ga = reinterpret_cast<const float4 *>(gc)[2 * q];
        const float4 gb = reinterpret_cast<const float4 *>(gc)[2 * q + 1];
        const float xv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        const float gv[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = xv[i] * gv[i] * r;
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = 0.0f;
    }
    encode_values8(v, store, pw, q);
}

__device__ __forceinline__ void encode_values8(const float (&v)[8], bool store, uint32_t *pw, int q) {
    float mx = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) mx = fmaxf(mx, fabsf(v[i]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    // mx in [2^(E-1), 2^E): E from the binary32 exponent field; tiny chunks clamp.
    int E = static_cast<int>((__float_as_uint(mx) >> 23) & 0xFF) - 126;
    if (E < -100) E = -100;
    const float up = __uint_as_float(static_cast<uint32_t>(127 + 22 - E) << 23);   // 2^(22-E)
    int m[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) m[i] = __float2int_rn(v[i] * up);  // |m| <= 2^22
    // byte b of the four even (odd) elements -> one word, via byte permutes
#pragma unroll
    for (int par = 0; par < 2; ++par) {
#pragma unroll
        for (int b = 0; b < 3; ++b) {
            const uint32_t sel_lo = 0x0040u | (b) | ((4 + b) << 4);   // {m[i].byte b, m[i+2].byte b}
            const uint32_t t01 = __byte_perm(m[par], m[par + 2], sel_lo);
            const uint32_t t23 = __byte_perm(m[par + 4], m[par + 6], sel_lo);
            if (store) pw[6 * q + 2 * b + par] = __byte_perm(t01, t23, 0x5410u);
        }
    }
    // plane sums
    int s01 = 0, s2 = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        s01 += m[i] & 0xFFFF;   // byte0 + 256 byte1
        s2 += m[i] >> 16;       // arithmetic shift: the signed top byte
    }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
        s01 += __shfl_xor_sync(0xffffffffu, s01, o);
        s2 += __shfl_xor_sync(0xffffffffu, s2, o);
    }
    if (store && q == 0) {
        pw[24] = static_cast<uint32_t>(s01);
        pw[25] = static_cast<uint32_t>(s2);
        pw[26] = 0u;
        pw[27] = __float_as_uint(__uint_as_float(static_cast<uint32_t>(127 + E - 22) << 23));  // 2^(E-22)
    }
}

struct Planes {
    uint32_t p[24];
    int s_lo, s_hi;
    float f;
};

// Integer dot product of one 16-byte chunk with one x chunk, minus the
// zero-point term: sum_k (q_k - z) m_k, exact in int32 and returned as binary32
// (the conversion of the planes-0/1 part, |lo| < 2^26, may round once, by at
// most 2^-24 of it).
__device__ __forceinline__ float chunk_dot(const uint4 &cw, int z, const Planes &P) {
    const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
    int a0 = 0, a1 = 0, a2 = 0;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const uint32_t lo = words[w] & 0x0F0F0F0Fu;          // codes of even k, one per byte
        const uint32_t hi = (words[w] >> 4) & 0x0F0F0F0Fu;   // codes of odd k, one per byte
        a0 = dp4a_uu(lo, P.p[6 * w + 0], a0);
        a0 = dp4a_uu(hi, P.p[6 * w + 1], a0);
        a1 = dp4a_uu(lo, P.p[6 * w + 2], a1);
        a1 = dp4a_uu(hi, P.p[6 * w + 3], a1);
        a2 = dp4a_us(lo, P.p[6 * w + 4], a2);
        a2 = dp4a_us(hi, P.p[6 * w + 5], a2);
    }
    const int lo = a1 * 256 + a0 - z * P.s_lo;   // planes 0 and 1
    const int hi = a2 - z * P.s_hi;               // plane 2
    return fmaf(static_cast<float>(hi), 65536.0f, static_cast<float>(lo));
}

// Integer dot product of one Q8_0 block's 32 signed 8-bit codes (cw[j]: elements 4j ..
// 4j + 3, one per byte) with one x chunk: sum_k q_k m_k, exact in int32 (|lo| < 2^30),
// returned as binary32.  Two byte permutes per 8 codes regroup them into the even and
// odd elements the planes hold; no zero point.
__device__ __forceinline__ float chunk_dot_q8(const uint32_t (&cw)[8], const Planes &P) {
    int a0 = 0, a1 = 0, a2 = 0;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const uint32_t ev = __byte_perm(cw[2 * w], cw[2 * w + 1], 0x6420u);   // elements 8w, 8w+2, 8w+4, 8w+6
        const uint32_t od = __byte_perm(cw[2 * w], cw[2 * w + 1], 0x7531u);   // elements 8w+1, 8w+3, 8w+5, 8w+7
        a0 = dp4a_su(ev, P.p[6 * w + 0], a0);
        a0 = dp4a_su(od, P.p[6 * w + 1], a0);
        a1 = dp4a_su(ev, P.p[6 * w + 2], a1);
        a1 = dp4a_su(od, P.p[6 * w + 3], a1);
        a2 = dp4a_ss(ev, P.p[6 * w + 4], a2);
        a2 = dp4a_ss(od, P.p[6 * w + 5], a2);
    }
    return fmaf(static_cast<float>(a2), 65536.0f, static_cast<float>(a1 * 256 + a0));
}

// The same for two rows of x at once: the codes are unpacked once and serve both rows'
// planes (d0: row 0, d1: row 1).
__device__ __forceinline__ void chunk_dot2(const uint4 &cw, int z, const Planes &P0, const Planes &P1, float &d0,
                                           float &d1) {
    const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
    int a0 = 0, a1 = 0, a2 = 0, b0 = 0, b1 = 0, b2 = 0;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const uint32_t lo = words[w] & 0x0F0F0F0Fu;          // codes of even k, one per byte
        const uint32_t hi = (words[w] >> 4) & 0x0F0F0F0Fu;   // codes of odd k, one per byte
        a0 = dp4a_uu(lo, P0.p[6 * w + 0], a0);
        a0 = dp4a_uu(hi, P0.p[6 * w + 1], a0);
        a1 = dp4a_uu(lo, P0.p[6 * w + 2], a1);
        a1 = dp4a_uu(hi, P0.p[6 * w + 3], a1);
        a2 = dp4a_us(lo, P0.p[6 * w + 4], a2);
        a2 = dp4a_us(hi, P0.p[6 * w + 5], a2);
        b0 = dp4a_uu(lo, P1.p[6 * w + 0], b0);
        b0 = dp4a_uu(hi, P1.p[6 * w + 1], b0);
        b1 = dp4a_uu(lo, P1.p[6 * w + 2], b1);
        b1 = dp4a_uu(hi, P1.p[6 * w + 3], b1);
        b2 = dp4a_us(lo, P1.p[6 * w + 4], b2);
        b2 = dp4a_us(hi, P1.p[6 * w + 5], b2);
    }
    d0 = fmaf(static_cast<float>(a2 - z * P0.s_hi), 65536.0f, static_cast<float>(a1 * 256 + a0 - z * P0.s_lo));
    d1 = fmaf(static_cast<float>(b2 - z * P1.s_hi), 65536.0f, static_cast<float>(b1 * 256 + b0 - z * P1.s_lo));
}

// ---- mbarrier primitives with bounded waits ----
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Non-blocking test of the phase with the given parity (try_wait may suspend the
// thread for a while before it reports failure; test_wait returns at once).
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Wait for the phase with the given parity to complete, for at most limit_ns
// (checked between potentially blocking tries, each suspended for at most the
// system's own time limit; measured slightly faster than a 20 us suspend hint
// and than spinning on test_wait in the streamed GEMV).
// A zero bound means one non-blocking test (the timer is too coarse to mean less).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
    if (limit_ns == 0) return mbar_test(bar, parity);
    if (mbar_test(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (;;) {
        if (mbar_try(bar, parity)) return true;
        if (global_ns() - t0 > limit_ns) return false;
    }
}

// Explicit shared-memory accesses (32-bit shared-window addresses).
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t a) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds_u8(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ float lds_f32(uint32_t a) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ void sts_f32(uint32_t a, float v) {
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}
__device__ __forceinline__ uint32_t lds_volatile_u32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ void sts_volatile_u32(uint32_t a, uint32_t v) {
    asm volatile("st.volatile.shared.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

// Sum NV values per lane over the 32 lanes of a warp by recursive halving: each round
// halves the values a lane carries while doubling the lanes it covers; butterflies
// finish.  Returns the total of value index (lane >> (5 - log2 NV)) on every lane.
template <int NV>
__device__ __forceinline__ float warp_sum_many(float (&v)[NV], int lane) {
    static_assert(NV == 1 || NV == 2 || NV == 4 || NV == 8 || NV == 16 || NV == 32, "NV must be a power of two <= 32");
    int off = 16;
#pragma unroll
    for (int n = NV; n > 1; n >>= 1) {
        const int half = n / 2;
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? v[i] : v[i + half];
            const float keep = upper ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
        off >>= 1;
    }
    float t = v[0];
#pragma unroll
    for (int o = off; o >= 1; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    return t;
}
// 1-D bulk copy global -> shared (TMA engine), completion counted on an mbarrier.
__device__ __forceinline__ void bulk_copy(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

}  // namespace xp
}  // namespace q4
