// q4gemv_stream.cuh -- launch interface of the TMA-streamed M = 1 int4 GEMV.
#pragma once

#include <type_traits>

#include "q4_common.cuh"

namespace q4 {

// Row-block geometry and shared-memory carve-up of one launch (all sizes in bytes).
// Block = ROWS = U * RG consecutive rows, one ring slot: codes | fp16 scales |
// zero-point bytes (asymmetric only), each a contiguous stretch of the arrays.
struct StreamGeo {
    int C;        // 32-code chunks per row (K / 32)
    int RG;       // row groups: consumer thread (r, c), r < RG, c < C
    int NB;       // groups per row
    int ZROW;     // zero-point bytes per row
    int GSHIFT;   // log2(g / 32): chunk >> GSHIFT = group
    int U;        // rows per consumer thread and block
    int ROWS;     // rows per block (U * RG)
    int TC;       // consumer threads (C * RG, whole warps)
    int NWC;      // consumer warps
    int CODE_B, SC_B, Z_B, SLOT_B;
    int WRED;     // 1: a row spans whole warps (C % 32 == 0), partials per warp
    int PARTS;    // partials per row
    int RED_LD;   // floats per row of a partial-sum buffer
    int RED_B;    // bytes of one partial-sum buffer
    int D;        // ring slots
    int OFF_RED, OFF_RING, OFF_BAR, OFF_FLAG, OFF_NORM, SMEM;
};

constexpr int kStreamNRed = 2;    // partial-sum buffers
constexpr int kStreamMaxTC = 608; // consumer threads per CTA, at most
constexpr int kStreamSmemBudget = 227 * 1024;   // opt-in shared memory per CTA on this GPU
constexpr int kStreamSmemPerSM = 228 * 1024;    // shared memory per SM (1 KB of it reserved per CTA)

__host__ __device__ constexpr int stream_round128(int v) { return (v + 127) / 128 * 128; }

// Rows per consumer thread and block: 6 for K = 896 (48-row blocks: three CTAs fit an
// SM), 8 otherwise.  Rows that span whole warps (K % 1024 == 0) need a power of two.
__host__ __device__ constexpr int stream_u(int K) { return K == 896 ? 6 : 8; }
// Q8_0 blocks carry 34 bytes per 32 codes: 4 rows per thread from K = 2048 on keep two
// ring slots inside the shared memory.
__host__ __device__ constexpr int stream_q80_u(int K) { return K == 896 ? 6 : 4; }

// fused: the fused-variant kernels also keep their RMSNorm sums (one float per consumer
// warp) in 128 bytes after the abort flag.  q40: the weights are Q4_0 blocks (32 codes and
// their binary16 scale in 18 bytes), so a block of rows is one stretch of ROWS * C * 18
// bytes (group 32, no zero points).  mx: rows of x (1, or 2 for the two-row instances),
// each with its own x planes and partial sums.  q80: Q8_0 blocks (32 int8 codes and their
// binary16 scale in 34 bytes), a block of rows one stretch of ROWS * C * 34 bytes.
__host__ __device__ constexpr StreamGeo make_stream_geo(int K, int G, int RG, int U, int D, bool asym,
                                                        bool fused = false, bool q40 = false, int mx = 1,
                                                        bool q80 = false) {
    StreamGeo g{};
    g.C = K / 32;
    g.RG = RG;
    g.NB = K / G;
    g.ZROW = (g.NB + 1) / 2;
    g.GSHIFT = G == 32 ? 0 : (G == 64 ? 1 : 2);
    g.U = U;
    g.ROWS = U * RG;
    g.TC = g.C * RG;
    g.NWC = g.TC / 32;
    const bool blocks = q40 || q80;   // scale and codes interleaved per 32-element block
    g.CODE_B = g.ROWS * g.C * (q40 ? 18 : (q80 ? 34 : 16));
    g.SC_B = blocks ? 0 : g.ROWS * g.NB * 2;
    g.Z_B = asym && !blocks ? g.ROWS * g.ZROW : 0;
    // (Q4_0 / Q8_0: 16 bytes of slack, as the 2-byte-aligned code reads fetch up to 2 or 4
    // bytes past a slot's last block)
    g.SLOT_B = stream_round128(g.CODE_B + g.SC_B + g.Z_B + (blocks ? 16 : 0));
    g.WRED = g.C % 32 == 0 ? 1 : 0;
    g.PARTS = g.WRED ? g.C / 32 : g.C;
    g.RED_LD = g.PARTS + 1;
    g.RED_B = g.ROWS * g.RED_LD * 4 * mx;   // [mx][ROWS][RED_LD]
    g.D = D;
    // shared memory: x planes | partial sums [kStreamNRed] | ring [D] | barriers | abort flag
    // | (fused) RMSNorm sums
    g.OFF_RED = stream_round128(g.C * 28 * 4 * mx);
    g.OFF_RING = stream_round128(g.OFF_RED + kStreamNRed * g.RED_B);
    g.OFF_BAR = g.OFF_RING + D * g.SLOT_B;
    g.OFF_FLAG = g.OFF_BAR + 8 * (2 * D + 2 * kStreamNRed);
    g.OFF_NORM = g.OFF_FLAG + 16;
    g.SMEM = g.OFF_NORM + (fused ? 128 : 0);
    return g;
}

// Ring slots: three (one more block in flight) when they fit the shared-memory
// budget without lowering the CTAs an SM holds, else two.
__host__ __device__ constexpr int stream_ctas_per_sm(int smem) { return kStreamSmemPerSM / (smem + 1024); }
__host__ __device__ constexpr int stream_slots(int K, int G, int RG, int U, bool asym, bool q40 = false, int mx = 1,
                                               bool q80 = false) {
    const int s2 = make_stream_geo(K, G, RG, U, 2, asym, false, q40, mx, q80).SMEM;
    const int s3 = make_stream_geo(K, G, RG, U, 3, asym, false, q40, mx, q80).SMEM;
    return (s3 <= kStreamSmemBudget && stream_ctas_per_sm(s3) >= stream_ctas_per_sm(s2)) ? 3 : 2;
}

struct StreamArgs {
    const uint8_t *codes;
    const uint16_t *scales;
    const uint8_t *zeros;
    const float *x;
    float *y;
    int64_t N;
    int nblocks;                     // blocks of rows (set by the launcher)
    unsigned long long timeout_ns;   // bound on every mbarrier wait
    unsigned int *status;            // device status word, set to 1 when a wait expires
    unsigned int *bounds;            // out-of-range access counter (bounds-checking builds)
    // fused variants only: gamma[K] (non-null: RMSNorm prologue, eps), swiglu != 0:
    // rows 2i / 2i+1 are a gate / up pair and y[i] = silu(gate) * up
    const float *gamma;
    float eps;
    int swiglu;
    StreamGeo geo;                   // used when the instance does not fix K and g
};

// Grouped launches: several matrices of the same K and group (each with its own x and y,
// M = 1) streamed by one launch.  Every CTA serves one matrix: matrix s owns the CTAs
// [cta_begin, next cta_begin) and splits its blocks of rows over them as a single
// launch would, so a CTA encodes one x and never switches.
constexpr int kStreamMaxSeg = 8;
struct StreamSeg {
    const uint8_t *codes;
    const uint16_t *scales;
    const uint8_t *zeros;
    const float *x;
    float *y;
    int64_t N;
    int nblocks;     // blocks of rows of this matrix
    int cta_begin;   // first CTA of this matrix
};
struct StreamGroupArgs : StreamArgs {
    StreamSeg seg[kStreamMaxSeg];
    int nseg;
};
// The kernel's argument type: the grouped instances (FUSE bit 3) take the segment table.
template <int FUSE>
using StreamArgsOf = std::conditional_t<(FUSE & 8) != 0, StreamGroupArgs, StreamArgs>;

// True when the streamed kernel serves this problem (M = 1, enough rows, a row
// geometry whose blocks are whole warps and 16-byte multiples, 16-byte aligned
// arrays, and a carve-up that fits the shared memory of one CTA).
bool stream_applies(int M, int64_t N, int K, int group, const void *codes, const void *scales, const void *zeros);
// Two rows of x (M = 2): the two-row instances, for K >= 2048 (one CTA per SM, so the second
// set of x planes has the registers it needs).
bool stream2_applies(int M, int64_t N, int K, int group, const void *codes, const void *scales, const void *zeros);
int launch_q4gemv_stream2(const uint8_t *codes, const uint16_t *scales, const uint8_t *zeros, const float *x,
                          float *y, int64_t N, int K, int group, cudaStream_t stream);
int launch_q4gemv_stream(const uint8_t *codes, const uint16_t *scales, const uint8_t *zeros, const float *x,
                         float *y, int64_t N, int K, int group, cudaStream_t stream);
// The fused variant (q4gemv_fused_run): gamma may be null (no RMSNorm), swiglu 0 or 1.
int launch_q4gemv_stream_fused(const uint8_t *codes, const uint16_t *scales, const uint8_t *zeros, const float *x,
                               const float *gamma, float eps, int swiglu, float *y, int64_t N, int K, int group,
                               cudaStream_t stream);
// Q4_0 blocks (q4_0_gemv_run): whether the streamed kernel serves the problem, and the launch.
bool stream_q40_applies(int M, int64_t N, int K, const void *blocks);
int launch_q4gemv_stream_q40(const uint8_t *blocks, const float *x, float *y, int64_t N, int K, cudaStream_t stream);
// Q8_0 blocks (q8_0_gemv_run): whether the streamed kernel serves the problem, and the launch.
bool stream_q80_applies(int M, int64_t N, int K, const void *blocks);
int launch_q4gemv_stream_q80(const uint8_t *blocks, const float *x, float *y, int64_t N, int K, cudaStream_t stream);
// Grouped: whether one streamed launch serves these matrices (same K and group, all with or
// all without zero points, every one streamable on its own alignment), and the launch.
bool stream_grouped_applies(const StreamSeg *segs, int nseg, int K, int group);
// Shares out at most grid_max CTAs over the matrices of a (sets every nblocks and
// cta_begin; each matrix gets at least one CTA and at most one per block of rows, the
// rest go where the blocks per CTA are highest) and returns the grid.
int stream_assign_ctas(StreamGroupArgs &a, int grid_max);
// The same split for matrices of N[i] rows at K (host only, for tests): fills nblocks and
// cta_begin, returns the grid; Q4_ERR_UNSUPPORTED (negated) when K has no streamed geometry.
int stream_grouped_split(const int64_t *N, int count, int K, int group, int grid_max, int *nblocks, int *cta_begin);
int launch_q4gemv_stream_grouped(const StreamSeg *segs, int nseg, int K, int group, cudaStream_t stream);
int read_and_clear_stream_status(unsigned int *v);

}  // namespace q4
