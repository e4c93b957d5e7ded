// q4gemv_tc.cu -- the 3 <= M <= 16 int4 GEMV on the 5th-generation tensor cores.
//
// Computes y[m][n] = sum_k w[n][k] * x[m][k], w[n][k] = (q[n][k] - z[n][k/g]) * s[n][k/g]
// (gerbil GPU-engine kernel reference, "3. MatMulInt4": "Computes", "Dequantization";
// MatMulNBits layout).  With a few rows of x the work is still a stream of weights, but
// the CUDA-core GEMV pays its multiply-adds once per row of x; here one dequantisation
// of each weight serves every row through the tensor core.
//
// Roles: the weights are the MMA's A operand (256 weight rows per CTA, two MMAs of
// M = 128 sharing each x tile), x the B operand.  x is split into two fp16 parts,
// x = hi + lo with hi = fp16(x) and lo = fp16(x - hi), stored as 2*MP rows of B (hi rows
// 0..MP-1, lo rows MP..2MP-1, rows past M zero), so the MMA's N is 16 or 32 and each
// D = [W x_hi^T | W x_lo^T] sits in 16 or 32 TMEM columns; the epilogue adds the two
// halves.  Each weight is dequantised exactly in binary32 ((q - z) * s) and rounded once
// to fp16 (relative error at most 2^-11, inside the 1e-3 tolerance); hi + lo carries x to
// about 2^-22.
//
//   warp 0      TMA producer: the 256 rows x 32 bytes of codes of each 64-wide K-block
//               (2D tensor map over codes[N][K/2]) into a 4-stage ring, completion
//               counted on the slot's mbarrier;
//   warp 1      allocates 64 TMEM columns (two accumulators); one lane issues 2 x 4 MMAs
//               (K = 16 each) per K-block and commits them to the weight/x stage's
//               "empty" barrier;
//   warps 2..9  dequantisers: each thread turns the 64 codes of one weight row in a
//               K-block (read from the code ring) into fp16 in the UMMA K-major
//               128-byte-swizzled layout (k permuted within each group of 8 to the
//               decode's nibble-pair order), and converts its share of x for the same
//               K-block into the hi/lo rows with the same permutation; scales, zero
//               points and x are prefetched into registers 4 blocks ahead; afterwards
//               each warp reads one TMEM lane quadrant of one accumulator (one lane per
//               weight row) and stores y.
// Few weight rows (N / 256 tiles below one per SM): the K-blocks of a tile are split
// over a cluster of S CTAs (grid y), each accumulating its own range in its own TMEM;
// the epilogue leaves each CTA's partial rows in shared memory and every CTA of the
// cluster finishes a share of the rows by adding the S partials in rank order through
// distributed shared memory (deterministic, nothing written to global memory but y).
// Every mbarrier wait is bounded by %globaltimer; on expiry the CTA raises the device
// status word (read by q4gemv_device_status), drains what it issued and returns.
#include <cooperative_groups.h>
#include <cuda_fp16.h>

#include "q4_common.cuh"
#include "q4_tc.cuh"

namespace q4 {

using namespace tc;
namespace cg = cooperative_groups;

unsigned int *gemm_status_word();

namespace {

constexpr int TMH = 128;                   // MMA M
constexpr int TK = 64;                     // K per block: one 128-byte row of fp16
constexpr int WST = 2;                     // weight/x tile stages (a power of two)
constexpr int PF = 4;                      // scale / zero-point / x prefetch distance (blocks)
constexpr int kDeqWarps = 8;
constexpr int kThreads = (2 + kDeqWarps) * 32;

// Tile geometry: TM weight rows per CTA, 128 (one MMA, two dequantiser threads per row)
// or 256 (two MMAs sharing each x tile, one dequantiser thread per row: half the
// per-weight cost of the waits, side data and x conversion, half the tiles).
template <int TM_>
struct TcGeo {
    static constexpr int TM = TM_;
    static constexpr int NACC = TM / TMH;              // accumulators: MMAs per K step
    static constexpr int NH = TM / TMH;                // 32-code halves per dequantiser thread and block
    static constexpr int CST = TM == 256 ? 4 : 16;     // code-ring stages (a power of two: cheap slot and parity)
    static constexpr int kCodeStage = TM * TK / 2;     // codes per block: 4 or 8 KB
    static constexpr int kWTile = TM * TK * 2;         // fp16 weights per block: 16 or 32 KB
    static constexpr int kTmemCols = 32 * NACC;        // accumulators of up to 32 columns
};

struct TcArgs {
    const uint16_t *scales;
    const uint8_t *zeros;
    const float *x;
    float *y;
    int64_t N;
    int M, K, nb, zrow, gshift;
    int S;                  // K split: CTAs per cluster (grid y), 1 = no cluster
    int side_vec;           // nb % 4 == 0, scales 8-byte and zeros 2-byte aligned: a chunk of
                            // four groups' side data is one 8-byte and one 2-byte load
    unsigned long long timeout_ns;
    unsigned int *status;
    unsigned int *bounds;   // out-of-range access counter (bounds-checking builds)
};

// (a & mask) | bits, one LOP3
__device__ __forceinline__ uint32_t lop3_or_and(uint32_t a, uint32_t mask, uint32_t bits) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(bits));
    return d;
}
// (m - zz) * ss on f16x2 pairs held in 32-bit registers: the subtraction is exact for the
// decoded nibbles, the multiply rounds once.
__device__ __forceinline__ uint32_t f16x2_sub_mul(uint32_t m, uint32_t zz, uint32_t ss) {
    uint32_t d;
    asm("{\n\t.reg .b32 t;\n\tsub.rn.f16x2 t, %1, %2;\n\tmul.rn.f16x2 %0, t, %3;\n\t}"
        : "=r"(d)
        : "r"(m), "r"(zz), "r"(ss));
    return d;
}
// Two floats to fp16 hi + lo pairs: hi = fp16(a), fp16(b); lo = fp16(a - hi_a), fp16(b - hi_b).
__device__ __forceinline__ void f16x2_split(float a, float b, uint32_t &hi, uint32_t &lo) {
    asm("{\n\t.reg .b16 ha, hb;\n\t.reg .f32 fa, fb;\n\t"
        "cvt.rn.f16x2.f32 %0, %3, %2;\n\t"
        "mov.b32 {ha, hb}, %0;\n\t"
        "cvt.f32.f16 fa, ha;\n\tcvt.f32.f16 fb, hb;\n\t"
        "sub.rn.f32 fa, %2, fa;\n\tsub.rn.f32 fb, %3, fb;\n\t"
        "cvt.rn.f16x2.f32 %1, fb, fa;\n\t}"
        : "=r"(hi), "=r"(lo)
        : "f"(a), "f"(b));
}
// Slot j of an 8-code group in the stored tiles holds code k = perm(j): the nibble-pair
// order (0,4), (1,5), (2,6), (3,7) of the decode.
__device__ __forceinline__ int slot_k(int j) { return (j >> 1) + 4 * (j & 1); }

}  // namespace

template <int MP, int TMV>
constexpr size_t tc_smem_bytes() {
    using Gm = TcGeo<TMV>;
    return 1024 + static_cast<size_t>(WST) * (Gm::kWTile + 2 * MP * TK * 2) +
           static_cast<size_t>(Gm::CST) * Gm::kCodeStage + 8 * (2 * Gm::CST + 2 * WST + 1) + 16;
}

// SPLIT: the launch is a cluster of g.S CTAs along grid y sharing each tile's K-blocks
// (compiled separately so the unsplit kernel carries none of it).
template <int MP, bool SPLIT, int TMV>
__global__ void __launch_bounds__(kThreads, 2)
q4gemv_tc_kernel(const __grid_constant__ CUtensorMap tmap_codes, const TcArgs g) {
    using Gm = TcGeo<TMV>;
    constexpr int TM = Gm::TM, NACC = Gm::NACC, NH = Gm::NH, CST = Gm::CST;
    constexpr int kCodeStage = Gm::kCodeStage, kWTile = Gm::kWTile, kTmemCols = Gm::kTmemCols;
    constexpr int NX = 2 * MP;                   // MMA N: MP hi rows then MP lo rows
    constexpr int kXTile = NX * TK * 2;          // 2 or 4 KB
    constexpr uint32_t kIdescTc = idesc_f16(false, TMH, NX);
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char *wtiles = smem;                                  // WST x 16 KB
    unsigned char *xtiles = wtiles + WST * kWTile;                 // WST x kXTile
    unsigned char *ctiles = xtiles + WST * kXTile;                 // CST x 4 KB
    uint64_t *bars = reinterpret_cast<uint64_t *>(ctiles + CST * kCodeStage);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * CST + 2 * WST + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * TM;
    // this CTA's K-blocks: [kb_begin, kb_end) of the tile's kblocks_all (its share of the
    // cluster's split); ring slots and parities count from kb_begin
    const int kblocks_all = (g.K + TK - 1) / TK;
    const int split = SPLIT ? g.S : 1;
    const int rank = SPLIT ? static_cast<int>(blockIdx.y) : 0;
    const int kb_begin = static_cast<int>(static_cast<int64_t>(kblocks_all) * rank / split);
    const int kb_end = static_cast<int>(static_cast<int64_t>(kblocks_all) * (rank + 1) / split);
    const int nkb = kb_end - kb_begin;
    const unsigned long long limit = g.timeout_ns;

    const uint32_t bar0 = smem_addr(bars);
    auto cfull = [&](int s) { return bar0 + 8u * s; };
    auto cempty = [&](int s) { return bar0 + 8u * (CST + s); };
    auto wfull = [&](int s) { return bar0 + 8u * (2 * CST + s); };
    auto wempty = [&](int s) { return bar0 + 8u * (2 * CST + WST + s); };
    const uint32_t done_bar = bar0 + 8u * (2 * CST + 2 * WST);

    if (threadIdx.x == 0) {
        for (int s = 0; s < CST; ++s) {
            mbar_init(cfull(s), 1);
            mbar_init(cempty(s), kDeqWarps * 32);
        }
        for (int s = 0; s < WST; ++s) {
            mbar_init(wfull(s), kDeqWarps * 32);
            mbar_init(wempty(s), 1);
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    allow_next_grid();
    const uint32_t tmem = *tmem_slot;

    auto fail = [&]() {
        *abort_flag = 1;
        atomicOr(g.status, 1u);
    };
    auto ib = [&](bool ok) { return q4_in_bounds(ok, g.bounds); };   // bounds-checking builds

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer (codes)
        if (lane == 0) {
            int issued = 0;
            for (int j = 0; j < nkb && !*abort_flag; ++j) {
                const int kb = kb_begin + j;
                const int s = j % CST;
                if (j >= CST && !mbar_wait(cempty(s), ((j / CST) - 1) & 1, limit)) {
                    fail();
                    break;
                }
                if (!ib(kb * (TK / 2) < (g.K + 1) / 2 && n0 < g.N)) {
                    mbar_arrive(cfull(s));   // (checking builds) keep the ring moving, load nothing
                } else {
                    mbar_expect_tx(cfull(s), kCodeStage);
                    tma_load_2d(smem_addr(ctiles + s * kCodeStage), &tmap_codes, cfull(s), kb * (TK / 2),
                                static_cast<int>(n0));
                }
                issued = j + 1;
            }
            if (*abort_flag) {
                // drain (bounded): every issued box lands before the CTA may exit
                for (int j = issued - CST > 0 ? issued - CST : 0; j < issued; ++j)
                    mbar_wait(cfull(j % CST), (j / CST) & 1, 50ull * 1000 * 1000);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            for (int j = 0; j < nkb && !*abort_flag; ++j) {
                const int s = j % WST;
                if (!mbar_wait(wfull(s), (j / WST) & 1, limit)) {
                    fail();
                    break;
                }
                tc_fence_after();
                const uint32_t a_base = smem_addr(wtiles + s * kWTile);
                const uint32_t b_base = smem_addr(xtiles + s * kXTile);
#pragma unroll
                for (int kk = 0; kk < TK / 16; ++kk)     // 16 fp16 = 32 bytes per step in the swizzle span
#pragma unroll
                    for (int a = 0; a < NACC; ++a)       // rows 128 a .. 128 a + 127 into columns 32 a ..
                        umma_f16(tmem + 32u * a, umma_desc(a_base + a * (kWTile / NACC) + kk * 32),
                                 umma_desc(b_base + kk * 32), kIdescTc, (j > 0 || kk > 0) ? 1u : 0u);
                umma_commit(wempty(s));
            }
            umma_commit(done_bar);   // all issued MMAs complete (also the drain on abort)
        }
    } else {
        // ------------------------------------------------------------ dequantisers
        const int t = threadIdx.x - 64;            // 0..255
        // weight row within the tile and the first of the NH 32-code halves of each block
        // this thread decodes (TM = 256: the whole row; TM = 128: one half)
        const int row = NH == 2 ? t : t >> 1;
        const int h0 = NH == 2 ? 0 : (t & 1);
        const int64_t n = n0 + row < g.N ? n0 + row : g.N - 1;
        const uint16_t *srow = g.scales + n * g.nb;
        const uint8_t *zrow = g.zeros ? g.zeros + n * g.zrow : nullptr;
        // x share: VPT consecutive slots (see slot_k) of one x row per K-block
        constexpr int VPT = MP / 4;                // 2 (MP = 8) or 4 (MP = 16)
        constexpr int TPR = TK / VPT;              // threads per x row
        const int xm = t / TPR;                    // x row (< MP)
        const int xk = (t - xm * TPR) * VPT;       // first slot of the share within the block

        // 256-row tiles (a whole 64-code row segment per thread and block): scales and zero
        // points come in chunks of four groups of this thread's row: the four binary16 scales
        // in two words and the four zero nibbles in 16 bits (8 each when symmetric), one
        // 8-byte and one 2-byte load per chunk where the layout allows (side_vec), else one
        // load per value.  The chunk in use and the next one (in flight) are held in
        // registers: a chunk spans 2 (g = 32) to 8 (g = 128) K-blocks, and the K-blocks'
        // groups never skip a chunk (at most two groups per block).  (Measured against one
        // 2-byte load per scale and one 1-byte load per zero-point pair and block, prefetched
        // four blocks ahead: 3-8 % faster with 256-row tiles, 2-13 % slower with 128-row
        // tiles, whose threads convert half a block each; those keep the per-block loads.)
        // (volatile: issued where written, a chunk ahead of its use)
        auto load_chunk = [&](int c, uint2 &sv, uint32_t &zv) {
            const int g0 = 4 * c;
            if (g.side_vec) {
                if (ib(g0 + 4 <= g.nb)) {
                    asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(sv.x), "=r"(sv.y) : "l"(srow + g0));
                }
                zv = 0x8888u;
                if (zrow && ib((g0 >> 1) + 2 <= g.zrow)) {
                    unsigned short h;
                    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(h) : "l"(zrow + (g0 >> 1)));
                    zv = h;
                }
            } else {
                uint32_t v[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) v[i] = g0 + i < g.nb ? ldg_u16(srow + g0 + i) : 0u;
                sv = make_uint2(v[0] | (v[1] << 16), v[2] | (v[3] << 16));
                zv = 0x8888u;
                if (zrow) {
                    const uint32_t z0 = ldg_u8(zrow + (g0 >> 1));
                    const uint32_t z1 = (g0 >> 1) + 1 < g.zrow ? ldg_u8(zrow + (g0 >> 1) + 1) : 0u;
                    zv = z0 | (z1 << 8);
                }
            }
        };
        // 128-row tiles: the scale of this thread's half of K-block kb and the zero-point byte
        // that holds its nibble; both tile heights: this thread's share of x for the block
        struct Side {
            uint32_t sc, zb;
            float xv[VPT];
        };
        auto fetch_w = [&](Side &f, int kb) {
            if constexpr (NH == 1) {
                const int k = kb * TK + h0 * 32;
                if (kb < kb_end && k < g.K) {
                    const int grp0 = k >> (5 + g.gshift);
                    if (ib(grp0 < g.nb)) f.sc = ldg_u16(srow + grp0);
                    if (zrow && ib((grp0 >> 1) < g.zrow)) f.zb = ldg_u8(zrow + (grp0 >> 1));
                }
            }
        };
        // slots xk .. xk + VPT - 1 of a block hold x at k = 8 * (slot / 8) + slot_k(slot % 8):
        // offsets fixed per thread; rows of x past M read as zero
        int xoff[VPT];
#pragma unroll
        for (int i = 0; i < VPT; ++i) xoff[i] = ((xk + i) & ~7) + slot_k((xk + i) & 7);
        const float *xrow = g.x + static_cast<int64_t>(xm < g.M ? xm : 0) * g.K;
        const bool xlive = xm < g.M;
        auto fetch_x = [&](Side &f, int kb) {
            const int k0 = kb * TK;
            if (xlive && kb < kb_end && k0 + TK <= g.K) {   // a whole block inside K
#pragma unroll
                for (int i = 0; i < VPT; ++i) f.xv[i] = __ldg(xrow + k0 + xoff[i]);
            } else {
#pragma unroll
                for (int i = 0; i < VPT; ++i)
                    f.xv[i] = (xlive && kb < kb_end && k0 + xoff[i] < g.K) ? __ldg(xrow + k0 + xoff[i]) : 0.0f;
            }
        };
        static_assert(PF == 4, "the K loop below is unrolled over four register sets");
        Side f0{}, f1{}, f2{}, f3{};
        // the chunk of the first K-block's groups, and the next one
        int cur_c = ((kb_begin * TK + h0 * 32) >> (5 + g.gshift)) >> 2;
        uint2 sc_cur = make_uint2(0u, 0u), sc_next = make_uint2(0u, 0u);
        uint32_t z_cur = 0x8888u, z_next = 0x8888u;
        if constexpr (NH == 2) {
            if (nkb > 0 && kb_begin * TK < g.K) {
                load_chunk(cur_c, sc_cur, z_cur);
                if (4 * (cur_c + 1) < g.nb) load_chunk(cur_c + 1, sc_next, z_next);
            }
        }
        fetch_w(f0, kb_begin);
        fetch_w(f1, kb_begin + 1);
        fetch_w(f2, kb_begin + 2);
        fetch_w(f3, kb_begin + 3);
        wait_prior_grid();   // x and y may belong to the kernel before this one in the stream
        fetch_x(f0, kb_begin);
        fetch_x(f1, kb_begin + 1);
        fetch_x(f2, kb_begin + 2);
        fetch_x(f3, kb_begin + 3);

        // loop-invariant shared-memory offsets of this thread: its 32 code bytes, and its
        // row in the weight tile (rows 128..255: the second operand).  Chunk w of the row
        // sits at w_row ^ (w << 4): the swizzle XORs the chunk index with row & 7, and the
        // row offset has those bits clear (a multiple of 128), as has the tile base.
        const uint32_t c_off = static_cast<uint32_t>(row * (TK / 2) + h0 * 16);
        const uint32_t w_row = (row >= TMH ? kWTile / 2 : 0) + sw128_offset(row & (TMH - 1), 0);
        const uint32_t within = static_cast<uint32_t>((xk & 7) * 2);   // byte offset inside the 16-byte chunk
        const uint32_t xhi_off = sw128_offset(xm, xk >> 3) + within;
        const uint32_t xlo_off = sw128_offset(MP + xm, xk >> 3) + within;

        // The j-th K-block of this CTA (block kb_begin + j) with the register set f that
        // holds its side data, which is then refilled for block kb + PF.  Returns false
        // when a bounded wait expired.
        auto step = [&](Side &f, int j) -> bool {
            const int kb = kb_begin + j;
            const int cs = j % CST, ws = j % WST;
            if (!mbar_wait(cfull(cs), (j / CST) & 1, limit)) return false;
            uint4 cw[NH];
#pragma unroll
            for (int i = 0; i < NH; ++i) cw[i] = make_uint4(0u, 0u, 0u, 0u);
            if (ib(c_off + 16 * NH <= static_cast<uint32_t>(kCodeStage))) {
                const uint32_t ca = smem_addr(ctiles + cs * kCodeStage) + c_off;
#pragma unroll
                for (int h = 0; h < NH; ++h)
                    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(cw[h].x), "=r"(cw[h].y), "=r"(cw[h].z), "=r"(cw[h].w)
                                 : "r"(ca + 16u * h));
            }
            if (j >= WST && !mbar_wait(wempty(ws), ((j / WST) - 1) & 1, limit)) return false;
            const uint32_t wrow_addr = smem_addr(wtiles + ws * kWTile) + w_row;
            // (256-row tiles) move to the next chunk of side data when this block's groups start it
            if constexpr (NH == 2) {
                if (kb * TK < g.K && (((kb * TK) >> (5 + g.gshift)) >> 2) != cur_c) {
                    sc_cur = sc_next;
                    z_cur = z_next;
                    ++cur_c;
                    if (4 * (cur_c + 1) < g.nb) load_chunk(cur_c + 1, sc_next, z_next);
                }
            }
            // this thread's 32-code halves of the row's block, one after the other
#pragma unroll
            for (int i = 0; i < NH; ++i) {
                const int h = h0 + i;              // which half of the 64-wide block
                const int k = kb * TK + h * 32;    // first code of this half
                uint32_t out[16];
                if (k < g.K) {
                    uint32_t z = 8u, ss;
                    if constexpr (NH == 2) {
                        const int gi = (k >> (5 + g.gshift)) & 3;   // the group's place in the chunk
                        z = (z_cur >> (4 * gi)) & 0xFu;
                        // the group's binary16 scale in both halves
                        ss = __byte_perm(gi & 2 ? sc_cur.y : sc_cur.x, 0u, gi & 1 ? 0x3232u : 0x1010u);
                    } else {
                        const int grp = k >> (5 + g.gshift);
                        if (zrow) z = (grp & 1) ? (f.zb >> 4) : (f.zb & 0xFu);
                        ss = f.sc * 0x00010001u;
                    }
                    // fp16 1024 + q from a nibble OR-ed into the fraction of 1024 (0x6400); the
                    // half2 subtraction of 1024 + z is exact, and one half2 multiply by s rounds the
                    // exact product (q - z) * s once -- the same value as rounding the binary32
                    // product.  Each word gives the nibble pairs (0,4), (1,5), (2,6), (3,7), stored
                    // in that order; x is stored with the same permutation of k.
                    const uint32_t zz = (0x6400u | z) * 0x00010001u;
                    const uint32_t words[4] = {cw[i].x, cw[i].y, cw[i].z, cw[i].w};
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
#pragma unroll
                        for (int p = 0; p < 4; ++p) {
                            const uint32_t m = lop3_or_and(words[w] >> (4 * p), 0x000F000Fu, 0x64006400u);
                            out[4 * w + p] = f16x2_sub_mul(m, zz, ss);
                        }
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) out[i] = 0u;   // K tail: zero weights
                }
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const uint32_t chunk = static_cast<uint32_t>(4 * h + w) << 4;
                    if (ib((w_row ^ chunk) + 16 <= static_cast<uint32_t>(kWTile)))
                        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(wrow_addr ^ chunk),
                                     "r"(out[4 * w]), "r"(out[4 * w + 1]), "r"(out[4 * w + 2]), "r"(out[4 * w + 3])
                                     : "memory");
                }
            }
            // x: hi part in row xm, lo part in row MP + xm (VPT fp16 at slot offset xk)
            {
                uint32_t hi[VPT / 2], lo[VPT / 2];
#pragma unroll
                for (int i = 0; i < VPT / 2; ++i) f16x2_split(f.xv[2 * i], f.xv[2 * i + 1], hi[i], lo[i]);
                unsigned char *xt = xtiles + ws * kXTile;
                const bool x_ok = ib(xhi_off + VPT * 2 <= static_cast<uint32_t>(kXTile) &&
                                     xlo_off + VPT * 2 <= static_cast<uint32_t>(kXTile));
                if (x_ok) {
                    if constexpr (VPT == 4) {
                        *reinterpret_cast<uint2 *>(xt + xhi_off) = make_uint2(hi[0], hi[1]);
                        *reinterpret_cast<uint2 *>(xt + xlo_off) = make_uint2(lo[0], lo[1]);
                    } else {
                        *reinterpret_cast<uint32_t *>(xt + xhi_off) = hi[0];
                        *reinterpret_cast<uint32_t *>(xt + xlo_off) = lo[0];
                    }
                }
            }
            fence_proxy_async();      // generic-proxy stores -> visible to the tensor core
            mbar_arrive(wfull(ws));
            // the code slot may be refilled only now, after the codes read from it have been
            // consumed: releasing it right after the shared-memory load let the TMA refill
            // overtake the load (measured: whole warps' rows wrong at random)
            mbar_arrive(cempty(cs));
            // this register set now serves block kb + PF (issued late: the old values are
            // consumed, so the loads land in the same registers without moves)
            fetch_w(f, kb + PF);
            fetch_x(f, kb + PF);
            return true;
        };

        for (int j0 = 0; j0 < nkb && !*abort_flag; j0 += PF) {
            bool ok = step(f0, j0);
            if (ok && j0 + 1 < nkb) ok = step(f1, j0 + 1);
            if (ok && j0 + 2 < nkb) ok = step(f2, j0 + 2);
            if (ok && j0 + 3 < nkb) ok = step(f3, j0 + 3);
            if (!ok) {
                fail();
                break;
            }
        }
        // ------------------------------------------------------------ epilogue (warps 2..9, or 2..5)
        if (NACC == 2 || warp < 6) {
            const int quad = warp & 3;             // TMEM lane quadrant this warp may access
            const int acc = NACC == 2 ? (warp - 2) >> 2 : 0;   // accumulator: rows 0..127 or 128..255
            const bool ok = mbar_wait(done_bar, 0, limit);
            if (!ok) fail();
            if (ok && !*abort_flag) {
                tc_fence_after();
                uint32_t v[32];
                const uint32_t taddr = tmem + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc * 32);
                if constexpr (NX == 32) {
                    asm volatile(
                        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
                          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
                          "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
                          "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
                          "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
                        : "r"(taddr));
                } else {
                    asm volatile(
                        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
                          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
                          "=r"(v[14]), "=r"(v[15])
                        : "r"(taddr));
                }
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                const int r = acc * TMH + quad * 32 + lane;   // weight row: accumulator, TMEM lane
                const int64_t nn = n0 + r;
                if constexpr (!SPLIT) {
                    if (nn < g.N) {
#pragma unroll
                        for (int m = 0; m < MP; ++m)
                            if (m < g.M)
                                g.y[static_cast<int64_t>(m) * g.N + nn] = __uint_as_float(v[m]) + __uint_as_float(v[MP + m]);
                    }
                } else {
                    // this CTA's partial of row r (no MMA ran if its K range is empty: the
                    // partial is 0), into the freed weight tiles
                    float *red = reinterpret_cast<float *>(wtiles);
#pragma unroll
                    for (int m = 0; m < MP; ++m)
                        if (ib((r * (MP + 1) + m + 1) * 4 <= WST * kWTile))
                            red[r * (MP + 1) + m] = nkb > 0 ? __uint_as_float(v[m]) + __uint_as_float(v[MP + m]) : 0.0f;
                }
            }
        }
    }
    if constexpr (SPLIT) {
        // every CTA of the cluster finishes rows [rank * TM / S, (rank + 1) * TM / S) of
        // the tile by adding the S partials in rank order
        cg::cluster_group cluster = cg::this_cluster();
        __syncwarp();     // (the producer and MMA lanes rejoin their warps first)
        cluster.sync();
        if (warp >= 2 && !*abort_flag) {
            const float *red = reinterpret_cast<const float *>(wtiles);
            const int r_lo = rank * TM / split, r_hi = (rank + 1) * TM / split;
            for (int i = (warp - 2) * 32 + lane; i < (r_hi - r_lo) * MP; i += kDeqWarps * 32) {
                const int r = r_lo + i / MP, m = i % MP;
                const int64_t nn = n0 + r;
                if (m < g.M && nn < g.N) {
                    float acc = 0.0f;
                    for (int q = 0; q < split; ++q)
                        if (ib((r * (MP + 1) + m + 1) * 4 <= WST * kWTile))
                            acc += cluster.map_shared_rank(red, q)[r * (MP + 1) + m];
                    g.y[static_cast<int64_t>(m) * g.N + nn] = acc;
                }
            }
        }
        cluster.sync();   // peers' shared memory stays valid until every read is done
    }
    // ---- teardown: every issued MMA finished before TMEM is released ----
    if (warp == 1 && lane == 0 && *abort_flag) mbar_wait(done_bar, 0, 50ull * 1000 * 1000);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
    }
}

// ------------------------------------------------------------------ host side

// K split (CTAs per cluster, a power of two up to the portable 8) for tiles of tm rows:
// the fewest that give a CTA per SM, keeping at least four K-blocks per CTA.  (Splitting
// further, to two CTAs per SM, measured slower: the extra CTAs run as a second wave.)
static int tc_gemv_split(int64_t N, int K, int tm) {
    const int64_t tiles = (N + tm - 1) / tm;
    const int kblocks = (K + TK - 1) / TK;
    const int64_t want = device_info().sms;
    int S = 1;
    while (S < 8 && tiles * S < want && kblocks / (2 * S) >= 4) S *= 2;
    return S;
}

// Tile height: 256 rows (cheaper per weight) when that still gives two tiles per SM; or
// when both heights need a K split and 256 rows launch at least as many CTAs; or when
// 128-row tiles would run unsplit and 256-row tiles split over clusters launch as many
// CTAs while keeping at least 32 K-blocks per CTA; otherwise 128 rows (twice the tiles).
// Measured on the decode and sweep shapes: 32768 x 8192 at M = 4..16 is 7-15 % faster
// as 128 tiles of 256 rows over clusters of 2 than as 256 unsplit 128-row tiles, while
// 32768 x 896 and x 2048 (7 and 16 K-blocks per CTA once split) are 5-25 % slower.
static int tc_gemv_tile_rows(int64_t N, int K) {
    const int64_t sms = device_info().sms;
    const int64_t t128 = (N + 127) / 128, t256 = (N + 255) / 256;
    const int s128 = tc_gemv_split(N, K, 128), s256 = tc_gemv_split(N, K, 256);
    const int kblocks = (K + TK - 1) / TK;
    if (t256 >= 2 * sms) return 256;
    if (s128 > 1 && t256 * s256 >= t128 * s128) return 256;
    if (s128 == 1 && t256 * s256 >= t128 && kblocks / s256 >= 32) return 256;
    return 128;
}

// Where the tensor-core GEMV beats the CUDA-core kernels (measured on the decode and
// sweep shapes at M = 3, 4, 5, 8, 9, 16): with the K split it wins from M = 5 on every
// matrix of at least 2^20 weights, and at M = 3 and 4 on long rows (K >= 2048, N >= 768)
// and on large matrices (2^24 weights and up); the CUDA-core kernels keep the small
// short-row shapes (896 x 896, 4864 x 896, 512 x 2048 at M <= 4), whose launches are
// latency-bound.
bool tc_gemv_applies(int M, int64_t N, int K, const void *codes) {
    if (M < 3 || M > 16) return false;
    if (K % 32 != 0 || !aligned(codes, 16)) return false;   // TMA: row pitch K/2 a multiple of 16 bytes
    if (N < TMH || N > (int64_t(1) << 31) - 256) return false;   // at least one whole 128-row tile
    const int64_t weights = N * static_cast<int64_t>(K);
    if (M >= 5) return weights >= (int64_t(1) << 20);
    return (K >= 2048 && N >= 768) || weights >= (int64_t(1) << 24);
}

template <int MP, bool SPLIT, int TMV>
static int launch_tc(const CUtensorMap &map, const TcArgs &g, cudaStream_t stream) {
    auto kern = q4gemv_tc_kernel<MP, SPLIT, TMV>;
    constexpr size_t smem = tc_smem_bytes<MP, TMV>();
    static std::atomic<bool> configured[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) {
            set_cuda_error(e);
            return Q4_ERR_CUDA;
        }
        configured[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((g.N + TMV - 1) / TMV), static_cast<unsigned>(g.S), 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    if (SPLIT) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = static_cast<unsigned>(g.S);
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    add_overlap_attr(cfg, attr);
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, map, g);
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return Q4_ERR_CUDA;
    }
    return launch_status();
}

template <int TMV>
static int launch_tc_rows(const CUtensorMap &map, const TcArgs &g, cudaStream_t stream) {
    if (g.S > 1)
        return g.M <= 8 ? launch_tc<8, true, TMV>(map, g, stream) : launch_tc<16, true, TMV>(map, g, stream);
    return g.M <= 8 ? launch_tc<8, false, TMV>(map, g, stream) : launch_tc<16, false, TMV>(map, g, stream);
}

int launch_q4gemv_tc(const uint8_t *codes, const uint16_t *scales, const uint8_t *zeros, const float *x, float *y,
                     int M, int64_t N, int K, int group, cudaStream_t stream) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (encode == nullptr) return Q4_ERR_CUDA;
    const int tm = tc_gemv_tile_rows(N, K);
    CUtensorMap map;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(N)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
    const cuuint32_t box[2] = {TK / 2, static_cast<cuuint32_t>(tm)};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = encode(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(codes), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return Q4_ERR_UNSUPPORTED;
    TcArgs g;
    g.scales = scales;
    g.zeros = zeros;
    g.x = x;
    g.y = y;
    g.N = N;
    g.M = M;
    g.K = K;
    g.nb = K / group;
    g.zrow = (g.nb + 1) / 2;
    g.gshift = group == 32 ? 0 : (group == 64 ? 1 : 2);
    g.timeout_ns = call_options().wait_ns;
    g.status = gemm_status_word();
    if (g.status == nullptr) return Q4_ERR_CUDA;
    g.bounds = bounds_counter();
    g.S = tc_gemv_split(N, K, tm);
    g.side_vec = (g.nb % 4 == 0 && aligned(scales, 8) && (zeros == nullptr || aligned(zeros, 2))) ? 1 : 0;
    return tm == 256 ? launch_tc_rows<256>(map, g, stream) : launch_tc_rows<128>(map, g, stream);
}

}  // namespace q4
