// q4_common.cuh -- internal helpers shared by the CUDA translation units of
// libq4gemv.so (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <atomic>

#include "q4gemv.h"

namespace q4 {

// ---------------------------------------------------------------- host side

// Remember the runtime's message for q4gemv_last_cuda_error().
void set_cuda_error(cudaError_t e);

// Device properties cached per device (SM count, opt-in shared memory).
struct DeviceInfo {
    int sms = 0;
    int smem_optin = 0;
    int cc_major = 0, cc_minor = 0;
};
const DeviceInfo &device_info();

inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Launch-result check: returns Q4_OK or Q4_ERR_CUDA (and records the message).
inline int launch_status() {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return Q4_ERR_CUDA;
    }
    return Q4_OK;
}

// Options of the API call in progress on the calling thread.  The entry points without
// an options argument take the process-wide defaults (q4gemv_set_overlapped_launch,
// q4gemm_set_wait_timeout_ns); the *_ex entry points install the caller's own for the
// duration of the call (CallScope), so nothing one caller chooses reaches another.
struct CallOptions {
    bool overlap = false;                        // programmatic dependent launch of the GEMVs
    bool exact_x = false;                        // GEMVs on the CUDA-core float kernel only
    unsigned long long wait_ns = 1000000000ull;  // bound on each bounded device-side wait
};
const CallOptions &call_options();
CallOptions default_call_options();
bool set_overlapped_launch(bool on);            // process default; returns the previous value
void set_default_wait_ns(unsigned long long ns);
class CallScope {
public:
    explicit CallScope(const CallOptions &o);
    ~CallScope();
    CallScope(const CallScope &) = delete;
    CallScope &operator=(const CallScope &) = delete;

private:
    CallOptions opts_;
    const CallOptions *prev_;
};

// add_overlap_attr appends the programmatic-stream-serialisation attribute to cfg when
// the call's options ask for an overlapped launch (attrs must have a free entry at
// cfg.numAttrs).
inline void add_overlap_attr(cudaLaunchConfig_t &cfg, cudaLaunchAttribute *attrs) {
    if (!call_options().overlap) return;
    cudaLaunchAttribute &at = attrs[cfg.numAttrs];
    at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attrs;
    ++cfg.numAttrs;
}

// Common validation of the packed-weight arguments (codes / scales / zeros, K, g).
int check_q4_args(const void *codes, const void *scales, int64_t N, int64_t K, int32_t group);

// Launchers implemented by the kernel translation units.
int launch_q4gemv(const uint8_t *codes, const uint16_t *scales, const uint8_t *zeros,
                  const float *x, float *y, int M, int64_t N, int K, int group,
                  cudaStream_t stream);
int launch_q4gemv_fused(const uint8_t *codes, const uint16_t *scales, const uint8_t *zeros, const float *x,
                        const float *gamma, float eps, int swiglu, float *y, int M, int64_t N, int K, int group,
                        cudaStream_t stream);
int launch_q40gemv(const uint8_t *blocks, const float *x, float *y, int M, int64_t N, int K, cudaStream_t stream);
int launch_q80gemv(const uint8_t *blocks, const float *x, float *y, int M, int64_t N, int K, cudaStream_t stream);
int launch_q4gemm(const uint8_t *codes, const uint16_t *scales, const uint8_t *zeros,
                  const uint16_t *a, float *c, int M, int64_t N, int K, int group,
                  cudaStream_t stream);
int launch_f32gemv(const float *W, const float *x, float *y, int M, int64_t N, int K,
                   cudaStream_t stream);
// 3 <= M <= 16 on the tensor cores (q4gemv_tc.cu): whether it serves the problem, and the launch.
bool tc_gemv_applies(int M, int64_t N, int K, const void *codes);
int launch_q4gemv_tc(const uint8_t *codes, const uint16_t *scales, const uint8_t *zeros, const float *x, float *y,
                     int M, int64_t N, int K, int group, cudaStream_t stream);
int read_device_status(cudaStream_t stream);
int launch_dequant(const uint8_t *codes, const uint16_t *scales, const uint8_t *zeros,
                   void *w, bool bf16, int64_t N, int K, int group, cudaStream_t stream);
int launch_read_probe(const float4 *buf, int64_t n16, float *partial, int blocks,
                      cudaStream_t stream);

// Device counter of out-of-range accesses in bounds-checking builds (nullptr when the
// library is built without -DQ4_BOUNDS_CHECK).  Kernels receive it in their arguments.
unsigned int *bounds_counter();

// ---------------------------------------------------------------- device side

// Bounds-checking builds: q4_in_bounds(cond, counter) counts a false condition and
// returns it, so the caller can skip the access; other builds compile it to true.
#ifdef Q4_BOUNDS_CHECK
__device__ __forceinline__ bool q4_in_bounds(bool ok, unsigned int *counter) {
    if (!ok && counter != nullptr) atomicAdd(counter, 1u);
    return ok;
}
#else
__device__ __forceinline__ bool q4_in_bounds(bool, unsigned int *) { return true; }
#endif

// Programmatic dependent launch.  wait_prior_grid: block until the grid this one
// depends on has completed and its memory writes are visible (a no-op when the
// launch carried no programmatic dependency).  allow_next_grid: let the next grid
// in the stream be scheduled once every CTA of this grid has executed it or exited.
__device__ __forceinline__ void wait_prior_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_next_grid() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// 2^23 as a binary32 bit pattern.  OR-ing an integer v < 2^23 into its fraction
// field gives the float 2^23 + v exactly; subtracting two such floats is exact.
constexpr uint32_t kMagic = 0x4B000000u;
constexpr uint32_t kNegMagic = 0xCB000000u;   // -(2^23 + v) for the same OR

// 128-bit streaming load of read-only data, not kept in L1.
__device__ __forceinline__ uint4 ldg_stream(const void *p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ldg_u16(const uint16_t *p) {
    unsigned short v;
    asm("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ldg_u8(const uint8_t *p) {
    uint32_t v;
    asm("ld.global.nc.u8 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ float half_bits_to_float(uint32_t h) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
}

__device__ __forceinline__ float2 f2(uint32_t a, uint32_t b) {
    return make_float2(__uint_as_float(a), __uint_as_float(b));
}

// Exact decode of one 32-bit word of eight 4-bit codes (nibble p = element
// 8w + p, lowest nibble first).  OR-ing a masked nibble into the fraction of
// 2^23 yields the float 2^23 + e_p * q exactly, where e_p = 16^p for p <= 4
// and, after shifting the word right by 12, e_p = 16^(p-3) for p = 5, 6, 7:
//     e = {1, 16, 256, 4096, 65536, 256, 4096, 65536}.
// The zero point z is replicated into nibbles 0..4 and decoded the same way
// with the sign bit set, giving -(2^23 + e_p * z); one packed add then leaves
// e_p * (q - z), an integer below 2^20 in magnitude, exactly.
struct ZeroTerms {
    float2 n01, n23, n45, n67;
};

__device__ __forceinline__ ZeroTerms zero_terms(uint32_t z) {
    const uint32_t zr = z * 0x11111u;
    ZeroTerms t;
    t.n01 = f2(kNegMagic | (zr & 0xFu), kNegMagic | (zr & 0xF0u));
    t.n23 = f2(kNegMagic | (zr & 0xF00u), kNegMagic | (zr & 0xF000u));
    t.n45 = f2(kNegMagic | (zr & 0xF0000u), kNegMagic | (zr & 0xF00u));
    t.n67 = f2(kNegMagic | (zr & 0xF000u), kNegMagic | (zr & 0xF0000u));
    return t;
}

struct WordTerms {
    float2 d01, d23, d45, d67;  // e_p * (q_p - z) for p = (0,1), (2,3), (4,5), (6,7)
};

__device__ __forceinline__ WordTerms decode_word(uint32_t wd, const ZeroTerms &zt) {
    const uint32_t t = wd >> 12;
    WordTerms d;
    d.d01 = __fadd2_rn(f2(kMagic | (wd & 0xFu), kMagic | (wd & 0xF0u)), zt.n01);
    d.d23 = __fadd2_rn(f2(kMagic | (wd & 0xF00u), kMagic | (wd & 0xF000u)), zt.n23);
    d.d45 = __fadd2_rn(f2(kMagic | (wd & 0xF0000u), kMagic | (t & 0xF00u)), zt.n45);
    d.d67 = __fadd2_rn(f2(kMagic | (t & 0xF000u), kMagic | (t & 0xF0000u)), zt.n67);
    return d;
}

// 1 / e_p for the eight positions of a word (powers of two: exact scaling).
__device__ __forceinline__ float inv_e(int p) {
    constexpr float v[8] = {1.0f, 0x1p-4f, 0x1p-8f, 0x1p-12f, 0x1p-16f, 0x1p-8f, 0x1p-12f, 0x1p-16f};
    return v[p];
}

}  // namespace q4
