// q4gemv.cu -- host planner for the decode GEMV: picks the M tile, lanes per
// row, split-K factor and shared-memory size, then launches one kernel.
#include "q4gemv_kernel.cuh"
#include "q4gemv_xreg.cuh"
#include "q4gemv_stream.cuh"

namespace q4 {

template <int MT>
int launch_q4gemv_mt(const GemvPlan &p, const GemvArgs &a, cudaStream_t s);
extern template int launch_q4gemv_mt<1>(const GemvPlan &, const GemvArgs &, cudaStream_t);
extern template int launch_q4gemv_mt<2>(const GemvPlan &, const GemvArgs &, cudaStream_t);
extern template int launch_q4gemv_mt<4>(const GemvPlan &, const GemvArgs &, cudaStream_t);
extern template int launch_q4gemv_mt<8>(const GemvPlan &, const GemvArgs &, cudaStream_t);
extern template int launch_q4gemv_mt<16>(const GemvPlan &, const GemvArgs &, cudaStream_t);
template <int MT>
int launch_q4gemv_fused_mt(const GemvPlan &p, const GemvArgs &a, cudaStream_t s);
extern template int launch_q4gemv_fused_mt<1>(const GemvPlan &, const GemvArgs &, cudaStream_t);
extern template int launch_q4gemv_fused_mt<2>(const GemvPlan &, const GemvArgs &, cudaStream_t);
extern template int launch_q4gemv_fused_mt<4>(const GemvPlan &, const GemvArgs &, cudaStream_t);
extern template int launch_q4gemv_fused_mt<8>(const GemvPlan &, const GemvArgs &, cudaStream_t);
extern template int launch_q4gemv_fused_mt<16>(const GemvPlan &, const GemvArgs &, cudaStream_t);
template <int MT>
int launch_q40_mt(const GemvPlan &p, const GemvArgs &a, cudaStream_t s);
extern template int launch_q40_mt<1>(const GemvPlan &, const GemvArgs &, cudaStream_t);
extern template int launch_q40_mt<2>(const GemvPlan &, const GemvArgs &, cudaStream_t);
extern template int launch_q40_mt<4>(const GemvPlan &, const GemvArgs &, cudaStream_t);
extern template int launch_q40_mt<8>(const GemvPlan &, const GemvArgs &, cudaStream_t);
extern template int launch_q40_mt<16>(const GemvPlan &, const GemvArgs &, cudaStream_t);

static int rows_per_cta(int MT, int L) {
    const int R = (MT <= 2) ? 2 : 1;
    return kGemvWarps * R * (32 / L);
}

// Plan a launch.  Returns Q4_OK or Q4_ERR_UNSUPPORTED (x slice does not fit).
//  - M tile MT: M rounded up to a power of two (rows of x beyond M are zero).
//  - L (lanes per row): as few as keep >= 16 warps per SM busy, since a slot's
//    lanes broadcast-share each x value read from shared memory.
//  - S (split-K over a cluster): when even L = 32 leaves fewer than 8 warps
//    per SM, or when the x slice of the whole row would not fit in shared
//    memory (large M x K).
static int plan_gemv(int M, int64_t N, int K, bool asym, GemvPlan &p) {
    const DeviceInfo &d = device_info();
    int MT = 1;
    while (MT < M) MT <<= 1;
    const int R = (MT <= 2) ? 2 : 1;
    const int C = K / 32;
    const int64_t target = static_cast<int64_t>(d.sms) * 16;
    int L = 4;
    while (L < 32 && (N * L) / (32 * R) < target) L <<= 1;
    const int64_t warps = (N * L + 32 * R - 1) / (32 * R);
    int S = 1;
    if (warps < target / 2) {
        int64_t want = (target + warps - 1) / warps;
        S = static_cast<int>(want < 8 ? want : 8);
        const int by_len = C / L;  // every split keeps at least L chunks
        if (S > by_len) S = by_len > 1 ? by_len : 1;
    }
    const size_t budget = static_cast<size_t>(d.smem_optin) - 1024;
    const int rpc = rows_per_cta(MT, L);
    int CS = 0;
    size_t smem = 0;
    for (;;) {
        CS = (C + S - 1) / S;
        smem = static_cast<size_t>(MT) * CS * kChunkFloats * sizeof(float) +
               (S > 1 ? static_cast<size_t>(rpc) * MT * sizeof(float) : 0);
        if (smem <= budget) break;
        if (S >= 8) return Q4_ERR_UNSUPPORTED;
        ++S;
    }
    S = (C + CS - 1) / CS;  // drop empty trailing splits
    smem = static_cast<size_t>(MT) * CS * kChunkFloats * sizeof(float) +
           (S > 1 ? static_cast<size_t>(rpc) * MT * sizeof(float) : 0);
    p.MT = MT;
    p.L = L;
    p.S = S;
    p.CS = CS;
    p.asym = asym;
    p.smem = smem;
    p.row_blocks = static_cast<int>((N + rpc - 1) / rpc);
    return Q4_OK;
}

int launch_q4gemv(const uint8_t *codes, const uint16_t *scales, const uint8_t *zeros,
                  const float *x, float *y, int M, int64_t N, int K, int group,
                  cudaStream_t stream) {
    // (a call with the exact-x option takes the general kernel for every shape: its
    // products are exact before one rounding, for any finite x)
    const bool exact = call_options().exact_x;
    if (!exact && stream_applies(M, N, K, group, codes, scales, zeros))
        return launch_q4gemv_stream(codes, scales, zeros, x, y, N, K, group, stream);
    if (!exact && stream2_applies(M, N, K, group, codes, scales, zeros))
        return launch_q4gemv_stream2(codes, scales, zeros, x, y, N, K, group, stream);
    // M = 3 on wide, long matrices: rows 0 and 1 of x on the two-row streamed instances and
    // row 2 on the one-row ones, two launches (8B LM head 109 us against 134 on the tensor
    // cores, 14336 x 4096 17.8 against 20.5, 32768 x 8192 68 against 90; at about 8192 rows
    // the two break even, and narrower matrices stay on the tensor cores)
    if (!exact && M == 3 && N >= 12288 && stream2_applies(2, N, K, group, codes, scales, zeros) &&
        stream_applies(1, N, K, group, codes, scales, zeros)) {
        const int st = launch_q4gemv_stream2(codes, scales, zeros, x, y, N, K, group, stream);
        if (st != Q4_OK) return st;
        return launch_q4gemv_stream(codes, scales, zeros, x + 2 * static_cast<int64_t>(K), y + 2 * N, N, K, group,
                                    stream);
    }
    if (!exact && tc_gemv_applies(M, N, K, codes))
        return launch_q4gemv_tc(codes, scales, zeros, x, y, M, N, K, group, stream);
    if (!exact) {
        XregPlan xp;
        XregArgs xa;
        if (plan_q4gemv_xreg(M, N, K, group, scales, zeros, xp, xa)) {
            xa.codes = codes;
            xa.scales = scales;
            xa.zeros = zeros;
            xa.x = x;
            xa.y = y;
            xa.bounds = bounds_counter();
            return launch_q4gemv_xreg(xp, xa, stream);
        }
    }
    GemvPlan p;
    int st = plan_gemv(M, N, K, zeros != nullptr, p);
    if (st != Q4_OK) return st;
    GemvArgs a;
    a.codes = codes;
    a.scales = scales;
    a.zeros = zeros;
    a.x = x;
    a.y = y;
    a.M = M;
    a.N = static_cast<int>(N);
    a.K = K;
    a.C = K / 32;
    a.nb = K / group;
    a.zrow = (a.nb + 1) / 2;
    a.gshift = group == 32 ? 0 : (group == 64 ? 1 : 2);
    a.CS = p.CS;
    a.gamma = nullptr;
    a.eps = 0.0f;
    a.swiglu = 0;
    switch (p.MT) {
        case 1: return launch_q4gemv_mt<1>(p, a, stream);
        case 2: return launch_q4gemv_mt<2>(p, a, stream);
        case 4: return launch_q4gemv_mt<4>(p, a, stream);
        case 8: return launch_q4gemv_mt<8>(p, a, stream);
        case 16: return launch_q4gemv_mt<16>(p, a, stream);
        default: return Q4_ERR_UNSUPPORTED;
    }
}

// The fused variant (q4gemv_fused_run): the streamed kernel for M = 1 where it applies,
// the register-resident kernel's fused instances for other M = 1 shapes it serves
// without a K split, else the general kernel's fused instance (16 lanes per row, no K split) over tiles of
// rows of x as large as the shared memory holds (x of every row of the tile for all of
// K, plus the RMSNorm sums), one launch per tile.
int launch_q4gemv_fused(const uint8_t *codes, const uint16_t *scales, const uint8_t *zeros, const float *x,
                        const float *gamma, float eps, int swiglu, float *y, int M, int64_t N, int K, int group,
                        cudaStream_t stream) {
    const bool exact = call_options().exact_x;   // (the general kernel only, as for launch_q4gemv)
    if (!exact && stream_applies(M, N, K, group, codes, scales, zeros)) {
        const int st = launch_q4gemv_stream_fused(codes, scales, zeros, x, gamma, eps, swiglu, y, N, K, group, stream);
        if (st != Q4_ERR_UNSUPPORTED) return st;   // (the fused carve-up is 128 bytes larger)
    }
    if (!exact) {   // M = 1 on shorter matrices: the register-resident kernel's fused instances
        XregPlan xp;
        XregFusedArgs xa;
        if (plan_q4gemv_xreg(M, N, K, group, scales, zeros, xp, xa, true)) {
            xa.codes = codes;
            xa.scales = scales;
            xa.zeros = zeros;
            xa.x = x;
            xa.y = y;
            xa.bounds = bounds_counter();
            xa.gamma = gamma;
            xa.eps = eps;
            xa.swiglu = swiglu;
            const int st = launch_q4gemv_xreg_fused(xp, xa, stream);
            if (st != Q4_ERR_UNSUPPORTED) return st;
        }
    }
    const int C = K / 32;
    const size_t budget = static_cast<size_t>(device_info().smem_optin) - 1024;
    auto smem_for = [&](int mt) {
        return static_cast<size_t>(mt) * C * kChunkFloats * sizeof(float) +
               static_cast<size_t>(kGemvWarps) * mt * sizeof(float);
    };
    int MT = 1;
    while (MT < M && MT < 16) MT <<= 1;
    while (MT > 1 && smem_for(MT) > budget) MT >>= 1;
    if (smem_for(MT) > budget) return Q4_ERR_UNSUPPORTED;
    GemvPlan p;
    p.MT = MT;
    p.L = 16;
    p.S = 1;
    p.CS = C;
    p.asym = zeros != nullptr;
    p.smem = smem_for(MT);
    p.row_blocks = static_cast<int>((N + rows_per_cta(MT, 16) - 1) / rows_per_cta(MT, 16));
    const int64_t ycols = swiglu ? N / 2 : N;
    for (int m0 = 0; m0 < M; m0 += MT) {
        GemvArgs a;
        a.codes = codes;
        a.scales = scales;
        a.zeros = zeros;
        a.x = x + static_cast<int64_t>(m0) * K;
        a.y = y + static_cast<int64_t>(m0) * ycols;
        a.M = M - m0 < MT ? M - m0 : MT;
        a.N = static_cast<int>(N);
        a.K = K;
        a.C = C;
        a.nb = K / group;
        a.zrow = (a.nb + 1) / 2;
        a.gshift = group == 32 ? 0 : (group == 64 ? 1 : 2);
        a.CS = C;
        a.gamma = gamma;
        a.eps = eps;
        a.swiglu = swiglu;
        int st = Q4_ERR_UNSUPPORTED;
        switch (MT) {
            case 1: st = launch_q4gemv_fused_mt<1>(p, a, stream); break;
            case 2: st = launch_q4gemv_fused_mt<2>(p, a, stream); break;
            case 4: st = launch_q4gemv_fused_mt<4>(p, a, stream); break;
            case 8: st = launch_q4gemv_fused_mt<8>(p, a, stream); break;
            case 16: st = launch_q4gemv_fused_mt<16>(p, a, stream); break;
        }
        if (st != Q4_OK) return st;
    }
    return Q4_OK;
}

// The Q4_0 GEMV (q4_0_gemv_run): the streamed kernel's Q4_0 instances for M = 1 on long
// matrices, else the general kernel's Q4_0 instances with the plan of a symmetric g = 32
// GEMV of the same shape.
int launch_q40gemv(const uint8_t *blocks, const float *x, float *y, int M, int64_t N, int K, cudaStream_t stream) {
    if (stream_q40_applies(M, N, K, blocks)) return launch_q4gemv_stream_q40(blocks, x, y, N, K, stream);
    GemvPlan p;
    int st = plan_gemv(M, N, K, false, p);
    if (st != Q4_OK) return st;
    GemvArgs a;
    a.codes = blocks;
    a.scales = nullptr;
    a.zeros = nullptr;
    a.x = x;
    a.y = y;
    a.M = M;
    a.N = static_cast<int>(N);
    a.K = K;
    a.C = K / 32;
    a.nb = K / 32;
    a.zrow = (a.nb + 1) / 2;
    a.gshift = 0;
    a.CS = p.CS;
    a.gamma = nullptr;
    a.eps = 0.0f;
    a.swiglu = 0;
    switch (p.MT) {
        case 1: return launch_q40_mt<1>(p, a, stream);
        case 2: return launch_q40_mt<2>(p, a, stream);
        case 4: return launch_q40_mt<4>(p, a, stream);
        case 8: return launch_q40_mt<8>(p, a, stream);
        case 16: return launch_q40_mt<16>(p, a, stream);
        default: return Q4_ERR_UNSUPPORTED;
    }
}

}  // namespace q4
