// f32gemv.cu -- dense binary32 GEMV control, y[m][n] = sum_k W[n][k] x[m][k],
// 1 <= M <= 16 (cera wgpu_gemv_bench.rs keeps this F32 kernel in its table as
// the control that separates harness artefacts from kernel properties).
//
// Same decomposition as the int4 GEMV: L lanes per row read L consecutive
// 16-byte pieces of W per load, R rows per thread share each x value read from
// shared memory, a cluster of S CTAs splits K when rows are few, and partials
// are added in rank order through distributed shared memory.
#include <cooperative_groups.h>

#include "q4_common.cuh"

namespace q4 {

namespace cg = cooperative_groups;

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kU = 4;  // float4 per row in flight per thread

struct F32Args {
    const float *W;
    const float *x;
    float *y;
    int M;
    int N;
    int K;
    int C4;  // float4 per row, K / 4
    int CS;  // float4 per split
};

template <int MT, int L>
struct Shape {
    static constexpr int R = (MT <= 2) ? 2 : 1;
    static constexpr int SLOTS = 32 / L;
    static constexpr int ROWS_PER_WARP = SLOTS * R;
    static constexpr int ROWS_PER_CTA = ROWS_PER_WARP * kWarps;
};

template <int MT, int L, bool SPLIT>
__global__ void __launch_bounds__(kThreads) f32gemv_kernel(const F32Args a) {
    using S = Shape<MT, L>;
    constexpr int R = S::R;
    constexpr int SLOTS = S::SLOTS;
    extern __shared__ __align__(16) float4 smem4[];
    float4 *xs = smem4;  // [MT][CS]

    const int split = SPLIT ? static_cast<int>(blockIdx.y) : 0;
    const int c_begin = split * a.CS;
    const int n4 = min(a.C4 - c_begin, a.CS);
    const int tid = threadIdx.x;
    for (int i = tid; i < MT * a.CS; i += kThreads) {
        const int m = i / a.CS;
        const int cl = i - m * a.CS;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (m < a.M && cl < n4)
            v = reinterpret_cast<const float4 *>(a.x + static_cast<int64_t>(m) * a.K)[c_begin + cl];
        xs[i] = v;
    }
    __syncthreads();

    const int warp = tid >> 5, lane = tid & 31;
    const int slot = lane / L, j = lane % L;
    const int64_t row0 = static_cast<int64_t>(blockIdx.x) * S::ROWS_PER_CTA + warp * S::ROWS_PER_WARP + slot;
    const float4 *wrow[R];
    bool rvalid[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t n = row0 + r * SLOTS;
        rvalid[r] = n < a.N;
        wrow[r] = reinterpret_cast<const float4 *>(a.W + (rvalid[r] ? n : a.N - 1) * static_cast<int64_t>(a.K)) + c_begin;
    }
    float acc[R][MT];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[r][m] = 0.f;

    for (int cb = j; cb < n4; cb += L * kU) {
        float4 w[R][kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int cl = cb + u * L;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (cl < n4) {
                    uint4 v = ldg_stream(wrow[r] + cl);
                    w[r][u] = make_float4(__uint_as_float(v.x), __uint_as_float(v.y),
                                          __uint_as_float(v.z), __uint_as_float(v.w));
                } else {
                    w[r][u] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int cl = cb + u * L;
            if (cl >= n4) continue;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const float4 xv = xs[m * a.CS + cl];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    acc[r][m] = fmaf(w[r][u].x, xv.x, acc[r][m]);
                    acc[r][m] = fmaf(w[r][u].y, xv.y, acc[r][m]);
                    acc[r][m] = fmaf(w[r][u].z, xv.z, acc[r][m]);
                    acc[r][m] = fmaf(w[r][u].w, xv.w, acc[r][m]);
                }
            }
        }
    }
#pragma unroll
    for (int off = L / 2; off >= 1; off >>= 1)
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m) acc[r][m] += __shfl_xor_sync(0xffffffffu, acc[r][m], off);

    if constexpr (!SPLIT) {
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m)
                if (((r * MT + m) % L) == j && rvalid[r] && m < a.M)
                    a.y[static_cast<int64_t>(m) * a.N + row0 + r * SLOTS] = acc[r][m];
    } else {
        float *red = reinterpret_cast<float *>(smem4 + MT * a.CS);
        const int local0 = warp * S::ROWS_PER_WARP + slot;
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m)
                if (((r * MT + m) % L) == j) red[(local0 + r * SLOTS) * MT + m] = acc[r][m];
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        const int nsplit = static_cast<int>(cluster.num_blocks());
        const int rank = static_cast<int>(cluster.block_rank());
        for (int i = rank * kThreads + tid; i < S::ROWS_PER_CTA * MT; i += nsplit * kThreads) {
            float v = 0.f;
            for (int q = 0; q < nsplit; ++q) v += cluster.map_shared_rank(red, q)[i];
            const int local = i / MT;
            const int m = i - local * MT;
            const int64_t n = static_cast<int64_t>(blockIdx.x) * S::ROWS_PER_CTA + local;
            if (n < a.N && m < a.M) a.y[static_cast<int64_t>(m) * a.N + n] = v;
        }
        cluster.sync();
    }
}

struct Plan {
    int MT, L, S, CS, row_blocks;
    size_t smem;
};

template <int MT, int L, bool SPLIT>
int launch_one(const Plan &p, const F32Args &a, cudaStream_t stream) {
    auto kern = f32gemv_kernel<MT, L, SPLIT>;
    static std::atomic<bool> configured[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             device_info().smem_optin);
        if (e != cudaSuccess) {
            set_cuda_error(e);
            return Q4_ERR_CUDA;
        }
        configured[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.row_blocks), SPLIT ? p.S : 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (SPLIT) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = static_cast<unsigned>(p.S);
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return Q4_ERR_CUDA;
    }
    return launch_status();
}

template <int MT, int L>
int launch_l(const Plan &p, const F32Args &a, cudaStream_t s) {
    return p.S > 1 ? launch_one<MT, L, true>(p, a, s) : launch_one<MT, L, false>(p, a, s);
}

template <int MT>
int launch_mt(const Plan &p, const F32Args &a, cudaStream_t s) {
    switch (p.L) {
        case 4: return launch_l<MT, 4>(p, a, s);
        case 8: return launch_l<MT, 8>(p, a, s);
        case 16: return launch_l<MT, 16>(p, a, s);
        case 32: return launch_l<MT, 32>(p, a, s);
        default: return Q4_ERR_UNSUPPORTED;
    }
}

}  // namespace

int launch_f32gemv(const float *W, const float *x, float *y, int M, int64_t N, int K,
                   cudaStream_t stream) {
    const DeviceInfo &d = device_info();
    int MT = 1;
    while (MT < M) MT <<= 1;
    const int R = (MT <= 2) ? 2 : 1;
    const int C4 = K / 4;
    const int64_t target = static_cast<int64_t>(d.sms) * 16;
    int L = 4;
    while (L < 32 && (N * L) / (32 * R) < target) L <<= 1;
    const int64_t warps = (N * L + 32 * R - 1) / (32 * R);
    int S = 1;
    if (warps < target / 2) {
        int64_t want = (target + warps - 1) / warps;
        S = static_cast<int>(want < 8 ? want : 8);
        const int by_len = C4 / L;
        if (S > by_len) S = by_len > 1 ? by_len : 1;
    }
    const int rpc = kWarps * R * (32 / L);
    const size_t budget = static_cast<size_t>(d.smem_optin) - 1024;
    int CS = 0;
    size_t smem = 0;
    for (;;) {
        CS = (C4 + S - 1) / S;
        smem = static_cast<size_t>(MT) * CS * 16 + (S > 1 ? static_cast<size_t>(rpc) * MT * 4 : 0);
        if (smem <= budget) break;
        if (S >= 8) return Q4_ERR_UNSUPPORTED;
        ++S;
    }
    S = (C4 + CS - 1) / CS;
    smem = static_cast<size_t>(MT) * CS * 16 + (S > 1 ? static_cast<size_t>(rpc) * MT * 4 : 0);
    Plan p{MT, L, S, CS, static_cast<int>((N + rpc - 1) / rpc), smem};
    F32Args a{W, x, y, M, static_cast<int>(N), K, C4, CS};
    switch (MT) {
        case 1: return launch_mt<1>(p, a, stream);
        case 2: return launch_mt<2>(p, a, stream);
        case 4: return launch_mt<4>(p, a, stream);
        case 8: return launch_mt<8>(p, a, stream);
        case 16: return launch_mt<16>(p, a, stream);
        default: return Q4_ERR_UNSUPPORTED;
    }
}

}  // namespace q4
