// q4gemv_xreg.cuh -- launch interface of the register-resident-x int4 GEMV (M <= 2).
#pragma once

#include "q4_common.cuh"

namespace q4 {

constexpr int kXregU = 2;   // row groups per ring iteration
constexpr int kXregD = 4;   // cp.async ring slots (iterations in flight + 1)
// compile-time-geometry instances (K = 896 with groups of 32, K = 4096 with groups of 128)
constexpr int kXregUSpecial = 4;
constexpr int kXregDSpecial = 2;

struct XregArgs {
    const uint8_t *codes;
    const uint16_t *scales;
    const uint8_t *zeros;
    const float *x;
    float *y;
    int M, N, K;
    int C;        // chunks per row (K / 32)
    int nb;       // groups per row
    int zrow;     // zero-point bytes per row
    int gshift;   // log2(group / 32)
    int CT;       // chunk positions per CTA (K-slice width)
    int CTp;      // threads per row (CT, or CT rounded up to a warp multiple)
    int RG;       // rows per row group
    int RB;       // iterations per reduction batch
    int red_ld;   // leading dimension of the partial-sum buffer
    int nsuper;   // iterations over all rows (kXregU * RG rows each)
    int off_red, off_ring, off_ysum;   // shared-memory offsets (bytes)
    unsigned int *bounds;              // out-of-range access counter (bounds-checking builds)
};

// The fused variant's arguments (M = 1, no K split); the plain kernels keep their own
// parameter type unchanged.  gamma[K] non-null: RMSNorm prologue with eps; swiglu != 0:
// rows 2i / 2i+1 are a gate / up pair and y[i] = silu(gate) * up; off_norm: shared-memory
// offset of the RMSNorm sums (one float per warp).
struct XregFusedArgs : XregArgs {
    const float *gamma;
    float eps;
    int swiglu;
    int off_norm;
};

struct XregPlan {
    int MT, S, threads, grid_x;
    size_t smem;
    bool asym, warpred;
    bool special;   // use the compile-time-geometry instance
    bool fused;     // the fused variant (q4gemv_fused_run)
    int off_norm;   // (fused) shared-memory offset of the RMSNorm sums
};

// fused: plan the fused variant, which serves M = 1 without a K split (false otherwise).
bool plan_q4gemv_xreg(int M, int64_t N, int K, int group, const void *scales, const void *zeros,
                      XregPlan &p, XregArgs &a, bool fused = false);
int launch_q4gemv_xreg(const XregPlan &p, const XregArgs &a, cudaStream_t stream);
int launch_q4gemv_xreg_fused(const XregPlan &p, const XregFusedArgs &a, cudaStream_t stream);

}  // namespace q4
