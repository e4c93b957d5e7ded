// q4gemv_stream.cu -- the M = 1 int4 GEMV for long-N shapes (LM heads and other
// tall matrices): a block of consecutive rows is three contiguous stretches of
// memory (codes, scales, zero points), streamed whole by the TMA bulk-copy engine.
//
// Computes y[n] = sum_k (q[n][k] - z[n][k/g]) * s[n][k/g] * x[k]
// (gerbil GPU-engine kernel reference, "3. MatMulInt4": "Computes",
// "Dequantization"; MatMulNBits layout per the Refractometer page's
// "b) q4 GEMV" sweep).
//
// One warp of each CTA is a producer: one of its threads streams each block of
// ROWS consecutive rows into a ring of shared-memory slots with cp.async.bulk,
// completion counted on the slot's mbarrier.  The other warps are consumers:
// thread (r, c) owns chunk position c (32 codes) of rows r, r + RG, ... of every
// block and keeps the matching 32 values of x in registers as byte planes (see
// q4gemv_xplanes.cuh); it unpacks each chunk to bytes, forms the integer dot
// product with dp4a, subtracts the zero-point term, and scales once.  Partial
// sums go to one of two shared buffers (summed over the warp first when a row
// spans whole warps); the reduction of block b is done by one consumer warp
// (rotating) while the others already compute block b+1, ordered by mbarriers
// rather than CTA barriers; all consumer warps share the last block's.  Every wait is bounded by a %globaltimer deadline
// (device status word on expiry).  The row geometry is fixed at compile time for
// the two decode LM-head shapes and read from the arguments otherwise.
#include "q4gemv_stream_kernel.cuh"

namespace q4 {

// Device status word of the streamed kernels: 1 = a bounded wait expired.  Its
// address is passed to every launch (the instances live in several translation units).
__device__ unsigned int g_stream_status = 0;

static unsigned int *stream_status_word() {
    static std::atomic<unsigned int *> addr[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    if (addr[dev] == nullptr) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_stream_status);
        if (e != cudaSuccess) {
            set_cuda_error(e);
            return nullptr;
        }
        addr[dev] = static_cast<unsigned int *>(p);
    }
    return addr[dev];
}

int launch_stream_k896(const StreamArgs &a, int group, bool asym, int fuse, cudaStream_t s);
int launch_stream_k2048(const StreamArgs &a, int group, bool asym, int fuse, cudaStream_t s);
int launch_stream_k4096(const StreamArgs &a, int group, bool asym, int fuse, cudaStream_t s);
int launch_stream_k8192(const StreamArgs &a, int group, bool asym, int fuse, cudaStream_t s);
int launch_stream_k14336(const StreamArgs &a, int group, bool asym, int fuse, cudaStream_t s);
int launch_stream_k16384(const StreamArgs &a, int group, bool asym, int fuse, cudaStream_t s);
int launch_stream_grouped_k896(StreamGroupArgs &a, int group, bool asym, cudaStream_t s);
int launch_stream_grouped_k2048(StreamGroupArgs &a, int group, bool asym, cudaStream_t s);
int launch_stream_grouped_k4096(StreamGroupArgs &a, int group, bool asym, cudaStream_t s);
int launch_stream_grouped_k8192(StreamGroupArgs &a, int group, bool asym, cudaStream_t s);
int launch_stream_grouped_k14336(StreamGroupArgs &a, int group, bool asym, cudaStream_t s);
int launch_stream_grouped_k16384(StreamGroupArgs &a, int group, bool asym, cudaStream_t s);

// ------------------------------------------------------------------ host side

// Row groups per block for K: the fewest that fill whole warps, then doubled while
// the CTA stays within 512 consumer threads and 8 row groups (64 rows per block).
// 0 when no choice fits.
static int stream_rg(int K) {
    const int C = K / 32;
    int r0 = 1;
    while ((C * r0) % 32 != 0) r0 *= 2;
    if (C * r0 > kStreamMaxTC) return 0;
    int rg = r0;
    while (C * rg * 2 <= 512 && rg * 2 <= 8) rg *= 2;
    return rg;
}

static bool stream_geo_ok(const StreamGeo &g, bool asym) {
    if (g.TC % 32 != 0 || g.TC > kStreamMaxTC) return false;
    if (g.WRED && (g.U & (g.U - 1)) != 0) return false;                  // warp sums need a power of two
    if (g.SC_B % 16 != 0 || (asym && g.Z_B % 16 != 0)) return false;   // bulk copies: 16-byte multiples
    if (g.CODE_B + g.SC_B + g.Z_B >= (1 << 20)) return false;            // mbarrier transaction count
    return g.SMEM <= device_info().smem_optin;
}

bool stream_applies(int M, int64_t N, int K, int group, const void *codes, const void *scales, const void *zeros) {
    if (M != 1 || N < 4096 || K % 32 != 0) return false;
    if (group != 32 && group != 64 && group != 128) return false;
    if (!aligned(codes, 16) || !aligned(scales, 16) || (zeros && !aligned(zeros, 16))) return false;
    const int rg = stream_rg(K);
    if (rg == 0) return false;
    const bool asym = zeros != nullptr;
    const int u = stream_u(K);
    const StreamGeo g = make_stream_geo(K, group, rg, u, stream_slots(K, group, rg, u, asym), asym);
    // short rows (K < 2048): at least one block of rows per SM, below which the
    // register-resident kernel's finer row split keeps more SMs busy
    if (K < 2048 && (N + g.ROWS - 1) / g.ROWS < device_info().sms) return false;
    return stream_geo_ok(g, asym);
}

bool stream2_applies(int M, int64_t N, int K, int group, const void *codes, const void *scales, const void *zeros) {
    if (M != 2 || N < 4096 || K < 2048 || K % 32 != 0) return false;
    if (group != 32 && group != 64 && group != 128) return false;
    if (!aligned(codes, 16) || !aligned(scales, 16) || (zeros && !aligned(zeros, 16))) return false;
    const int rg = stream_rg(K);
    if (rg == 0) return false;
    const bool asym = zeros != nullptr;
    const int u = stream_u(K);
    const StreamGeo g = make_stream_geo(K, group, rg, u, stream_slots(K, group, rg, u, asym, false, 2), asym, false,
                                        false, 2);
    return stream_geo_ok(g, asym);
}

// fuse: 0 plain, 1 RMSNorm, 3 RMSNorm and/or SwiGLU, 4 Q4_0 blocks (codes = the blocks),
// 16 two rows of x, 32 Q8_0 blocks (codes = the blocks)
static int launch_stream_any(const uint8_t *codes, const uint16_t *scales, const uint8_t *zeros, const float *x,
                             const float *gamma, float eps, int swiglu, int fuse, float *y, int64_t N, int K,
                             int group, cudaStream_t stream) {
    const bool asym = zeros != nullptr;
    const int rg = stream_rg(K);
    if (rg == 0) return Q4_ERR_UNSUPPORTED;
    StreamArgs a;
    a.codes = codes;
    a.scales = scales;
    a.zeros = zeros;
    a.x = x;
    a.y = y;
    a.N = N;
    a.nblocks = 0;
    a.timeout_ns = call_options().wait_ns;
    a.status = stream_status_word();
    a.bounds = bounds_counter();
    a.gamma = gamma;
    a.eps = eps;
    a.swiglu = swiglu;
    if (a.status == nullptr) return Q4_ERR_CUDA;
    const bool q40 = fuse == 4, q80 = fuse == 32;
    const int u = q80 ? stream_q80_u(K) : stream_u(K);
    const int mx = fuse == 16 ? 2 : 1;
    a.geo = make_stream_geo(K, group, rg, u, stream_slots(K, group, rg, u, asym, q40, mx, q80), asym,
                            fuse == 1 || fuse == 3, q40, mx, q80);
    if (!stream_geo_ok(a.geo, asym)) return Q4_ERR_UNSUPPORTED;
    // compile-time row geometry for the K of the decode and sweep shapes
    switch (K) {
        case 896: return launch_stream_k896(a, group, asym, fuse, stream);
        case 2048: return launch_stream_k2048(a, group, asym, fuse, stream);
        case 4096: return launch_stream_k4096(a, group, asym, fuse, stream);
        case 8192: return launch_stream_k8192(a, group, asym, fuse, stream);
        case 14336: return launch_stream_k14336(a, group, asym, fuse, stream);
        case 16384: return launch_stream_k16384(a, group, asym, fuse, stream);
        default:   // runtime geometry; stream_u(K) is 8 for every K without an instance
            if (fuse == 4) return launch_stream<0, 0, 0, 8, false, 4>(a, stream);
            if (fuse == 32) return launch_stream<0, 0, 0, stream_q80_u(0), false, 32>(a, stream);
            if (fuse == 16)
                return asym ? launch_stream<0, 0, 0, 8, true, 16>(a, stream) : launch_stream<0, 0, 0, 8, false, 16>(a, stream);
            if (fuse == 3)
                return asym ? launch_stream<0, 0, 0, 8, true, 3>(a, stream) : launch_stream<0, 0, 0, 8, false, 3>(a, stream);
            if (fuse == 1)
                return asym ? launch_stream<0, 0, 0, 8, true, 1>(a, stream) : launch_stream<0, 0, 0, 8, false, 1>(a, stream);
            return asym ? launch_stream<0, 0, 0, 8, true>(a, stream) : launch_stream<0, 0, 0, 8, false>(a, stream);
    }
}

int launch_q4gemv_stream(const uint8_t *codes, const uint16_t *scales, const uint8_t *zeros, const float *x,
                         float *y, int64_t N, int K, int group, cudaStream_t stream) {
    return launch_stream_any(codes, scales, zeros, x, nullptr, 0.0f, 0, 0, y, N, K, group, stream);
}

int launch_q4gemv_stream2(const uint8_t *codes, const uint16_t *scales, const uint8_t *zeros, const float *x,
                          float *y, int64_t N, int K, int group, cudaStream_t stream) {
    return launch_stream_any(codes, scales, zeros, x, nullptr, 0.0f, 0, 16, y, N, K, group, stream);
}

int launch_q4gemv_stream_fused(const uint8_t *codes, const uint16_t *scales, const uint8_t *zeros, const float *x,
                               const float *gamma, float eps, int swiglu, float *y, int64_t N, int K, int group,
                               cudaStream_t stream) {
    // fused instances: 1 = RMSNorm only, 3 = also SwiGLU (the norm stays a runtime choice)
    return launch_stream_any(codes, scales, zeros, x, gamma, eps, swiglu, swiglu ? 3 : 1, y, N, K, group, stream);
}

bool stream_q40_applies(int M, int64_t N, int K, const void *blocks) {
    if (M != 1 || N < 4096 || K % 32 != 0 || !aligned(blocks, 16)) return false;
    const int rg = stream_rg(K);
    if (rg == 0) return false;
    const int u = stream_u(K);
    const StreamGeo g = make_stream_geo(K, 32, rg, u, stream_slots(K, 32, rg, u, false, true), false, false, true);
    if (g.ROWS % 8 != 0) return false;   // every block of rows starts 16-byte aligned
    if (K < 2048 && (N + g.ROWS - 1) / g.ROWS < device_info().sms) return false;
    return stream_geo_ok(g, false);
}

int launch_q4gemv_stream_q40(const uint8_t *blocks, const float *x, float *y, int64_t N, int K, cudaStream_t stream) {
    return launch_stream_any(blocks, nullptr, nullptr, x, nullptr, 0.0f, 0, 4, y, N, K, 32, stream);
}

bool stream_q80_applies(int M, int64_t N, int K, const void *blocks) {
    if (M != 1 || N < 4096 || K % 32 != 0 || !aligned(blocks, 16)) return false;
    const int rg = stream_rg(K);
    if (rg == 0) return false;
    const int u = stream_q80_u(K);
    const StreamGeo g =
        make_stream_geo(K, 32, rg, u, stream_slots(K, 32, rg, u, false, false, 1, true), false, false, false, 1, true);
    if ((g.ROWS * g.C * 34) % 16 != 0) return false;   // every block of rows starts 16-byte aligned
    if (K < 2048 && (N + g.ROWS - 1) / g.ROWS < device_info().sms) return false;
    return stream_geo_ok(g, false);
}

int launch_q4gemv_stream_q80(const uint8_t *blocks, const float *x, float *y, int64_t N, int K, cudaStream_t stream) {
    return launch_stream_any(blocks, nullptr, nullptr, x, nullptr, 0.0f, 0, 32, y, N, K, 32, stream);
}

// ---- grouped launches (several matrices of the same K, one launch) ----

bool stream_grouped_applies(const StreamSeg *segs, int nseg, int K, int group) {
    if (nseg < 1 || nseg > kStreamMaxSeg) return false;
    if (group != 32 && group != 64 && group != 128) return false;
    if (K != 896 && K != 2048 && K != 4096 && K != 8192 && K != 14336 && K != 16384) return false;   // compile-time geometries
    const bool asym = segs[0].zeros != nullptr;
    const int rg = stream_rg(K);
    if (rg == 0) return false;
    const int u = stream_u(K);
    const StreamGeo g = make_stream_geo(K, group, rg, u, stream_slots(K, group, rg, u, asym), asym);
    if (!stream_geo_ok(g, asym)) return false;
    int64_t blocks = 0;
    for (int i = 0; i < nseg; ++i) {
        const StreamSeg &sg = segs[i];
        if (sg.N < 1 || (sg.zeros != nullptr) != asym) return false;
        if (!aligned(sg.codes, 16) || !aligned(sg.scales, 16) || (asym && !aligned(sg.zeros, 16))) return false;
        blocks += (sg.N + g.ROWS - 1) / g.ROWS;
    }
    // short rows: at least one block of rows per SM over the whole group, as for one matrix
    if (K < 2048 && blocks < device_info().sms) return false;
    return blocks < (int64_t(1) << 30);
}

int stream_assign_ctas(StreamGroupArgs &a, int grid_max) {
    const int rows = a.geo.ROWS;
    int64_t total = 0;
    for (int i = 0; i < a.nseg; ++i) {
        a.seg[i].nblocks = static_cast<int>((a.seg[i].N + rows - 1) / rows);
        total += a.seg[i].nblocks;
    }
    int c[kStreamMaxSeg] = {};
    int grid = 0;
    if (total <= grid_max) {   // a CTA per block of rows
        for (int i = 0; i < a.nseg; ++i) {
            c[i] = a.seg[i].nblocks;
            grid += c[i];
        }
    } else {
        // one CTA each, then one at a time to the matrix with the most blocks per CTA
        // (which minimises the largest share any CTA gets)
        for (int i = 0; i < a.nseg; ++i) c[i] = 1;
        grid = a.nseg;
        while (grid < grid_max) {
            int best = -1;
            for (int i = 0; i < a.nseg; ++i)
                if (c[i] < a.seg[i].nblocks &&
                    (best < 0 || static_cast<int64_t>(a.seg[i].nblocks) * c[best] >
                                     static_cast<int64_t>(a.seg[best].nblocks) * c[i]))
                    best = i;
            if (best < 0) break;
            ++c[best];
            ++grid;
        }
    }
    int begin = 0;
    for (int i = 0; i < a.nseg; ++i) {
        a.seg[i].cta_begin = begin;
        begin += c[i];
    }
    return grid;
}

int stream_grouped_split(const int64_t *N, int count, int K, int group, int grid_max, int *nblocks, int *cta_begin) {
    const int rg = stream_rg(K);
    if (rg == 0 || count < 1 || count > kStreamMaxSeg || grid_max < count) return -Q4_ERR_UNSUPPORTED;
    StreamGroupArgs a{};
    const int u = stream_u(K);
    a.geo = make_stream_geo(K, group, rg, u, stream_slots(K, group, rg, u, true), true);
    a.nseg = count;
    for (int i = 0; i < count; ++i) {
        if (N[i] < 1) return -Q4_ERR_INVALID_ARG;
        a.seg[i].N = N[i];
    }
    const int grid = stream_assign_ctas(a, grid_max);
    for (int i = 0; i < count; ++i) {
        nblocks[i] = a.seg[i].nblocks;
        cta_begin[i] = a.seg[i].cta_begin;
    }
    return grid;
}

int launch_q4gemv_stream_grouped(const StreamSeg *segs, int nseg, int K, int group, cudaStream_t stream) {
    if (!stream_grouped_applies(segs, nseg, K, group)) return Q4_ERR_UNSUPPORTED;
    const bool asym = segs[0].zeros != nullptr;
    StreamGroupArgs a{};
    a.codes = segs[0].codes;   // (the base fields are unused by the grouped instances)
    a.scales = segs[0].scales;
    a.zeros = segs[0].zeros;
    a.x = segs[0].x;
    a.y = segs[0].y;
    a.N = segs[0].N;
    a.nblocks = 0;
    a.timeout_ns = call_options().wait_ns;
    a.status = stream_status_word();
    a.bounds = bounds_counter();
    a.gamma = nullptr;
    a.eps = 0.0f;
    a.swiglu = 0;
    if (a.status == nullptr) return Q4_ERR_CUDA;
    const int rg = stream_rg(K), u = stream_u(K);
    a.geo = make_stream_geo(K, group, rg, u, stream_slots(K, group, rg, u, asym), asym);
    a.nseg = nseg;
    for (int i = 0; i < nseg; ++i) a.seg[i] = segs[i];
    switch (K) {
        case 896: return launch_stream_grouped_k896(a, group, asym, stream);
        case 2048: return launch_stream_grouped_k2048(a, group, asym, stream);
        case 4096: return launch_stream_grouped_k4096(a, group, asym, stream);
        case 8192: return launch_stream_grouped_k8192(a, group, asym, stream);
        case 14336: return launch_stream_grouped_k14336(a, group, asym, stream);
        case 16384: return launch_stream_grouped_k16384(a, group, asym, stream);
        default: return Q4_ERR_UNSUPPORTED;
    }
}

int read_and_clear_stream_status(unsigned int *v) {
    cudaError_t e = cudaMemcpyFromSymbol(v, g_stream_status, sizeof *v);
    if (e != cudaSuccess) return Q4_ERR_CUDA;
    if (*v) {
        const unsigned int zero = 0;
        cudaMemcpyToSymbol(g_stream_status, &zero, sizeof zero);
    }
    return Q4_OK;
}

}  // namespace q4
