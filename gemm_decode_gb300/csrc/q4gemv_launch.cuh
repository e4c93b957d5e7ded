// q4gemv_launch.cuh -- launches one instantiation of the GEMV kernel.  Each
// q4gemv_mt*.cu includes this file and instantiates one M tile, so the
// instantiations compile in parallel.
#pragma once

#include "q4gemv_kernel.cuh"

namespace q4 {

template <int MT, int L, bool ASYM, bool SPLIT, bool FUSED = false, bool Q40 = false>
static int launch_gemv_one(const GemvPlan &p, const GemvArgs &a, cudaStream_t stream) {
    auto kern = q4gemv_kernel<MT, L, ASYM, SPLIT, FUSED, Q40>;
    // Opt into the large shared-memory carve-out once per device.
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
    cfg.blockDim = dim3(kGemvThreads, 1, 1);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    if (SPLIT) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = static_cast<unsigned>(p.S);
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    add_overlap_attr(cfg, attr);
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return Q4_ERR_CUDA;
    }
    return launch_status();
}

template <int MT, int L>
static int launch_gemv_l(const GemvPlan &p, const GemvArgs &a, cudaStream_t s) {
    if (p.asym)
        return p.S > 1 ? launch_gemv_one<MT, L, true, true>(p, a, s)
                       : launch_gemv_one<MT, L, true, false>(p, a, s);
    return p.S > 1 ? launch_gemv_one<MT, L, false, true>(p, a, s)
                   : launch_gemv_one<MT, L, false, false>(p, a, s);
}

template <int MT>
int launch_q4gemv_mt(const GemvPlan &p, const GemvArgs &a, cudaStream_t s) {
    switch (p.L) {
        case 4: return launch_gemv_l<MT, 4>(p, a, s);
        case 8: return launch_gemv_l<MT, 8>(p, a, s);
        case 16: return launch_gemv_l<MT, 16>(p, a, s);
        case 32: return launch_gemv_l<MT, 32>(p, a, s);
        default: return Q4_ERR_UNSUPPORTED;
    }
}

// The fused variant: lanes per row 16 (gate / up pairs in neighbouring slots), no split.
template <int MT>
int launch_q4gemv_fused_mt(const GemvPlan &p, const GemvArgs &a, cudaStream_t s) {
    return p.asym ? launch_gemv_one<MT, 16, true, false, true>(p, a, s)
                  : launch_gemv_one<MT, 16, false, false, true>(p, a, s);
}

// Q4_0 blocks: the plan's lanes per row and split, symmetric.
template <int MT, int L>
static int launch_q40_l(const GemvPlan &p, const GemvArgs &a, cudaStream_t s) {
    return p.S > 1 ? launch_gemv_one<MT, L, false, true, false, true>(p, a, s)
                   : launch_gemv_one<MT, L, false, false, false, true>(p, a, s);
}

template <int MT>
int launch_q40_mt(const GemvPlan &p, const GemvArgs &a, cudaStream_t s) {
    switch (p.L) {
        case 4: return launch_q40_l<MT, 4>(p, a, s);
        case 8: return launch_q40_l<MT, 8>(p, a, s);
        case 16: return launch_q40_l<MT, 16>(p, a, s);
        case 32: return launch_q40_l<MT, 32>(p, a, s);
        default: return Q4_ERR_UNSUPPORTED;
    }
}

}  // namespace q4
