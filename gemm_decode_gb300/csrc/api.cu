// api.cu -- the C ABI of libq4gemv.so: argument checks, status codes, device
// caches, and dispatch to the kernel launchers.  Every check runs on the host
// before any launch; a failed check launches nothing.
#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "q4_common.cuh"
#include "q4gemv_stream.cuh"

namespace q4 {

namespace {
thread_local char g_cuda_error[256] = "";
std::atomic<bool> g_overlapped_launch{false};
std::atomic<unsigned long long> g_default_wait_ns{1000ull * 1000 * 1000};   // 1 s per wait
thread_local const CallOptions *t_call_options = nullptr;
}

bool set_overlapped_launch(bool on) { return g_overlapped_launch.exchange(on); }
void set_default_wait_ns(unsigned long long ns) { g_default_wait_ns = ns; }

CallOptions default_call_options() {
    CallOptions o;
    o.overlap = g_overlapped_launch.load(std::memory_order_relaxed);
    o.wait_ns = g_default_wait_ns.load(std::memory_order_relaxed);
    return o;
}

const CallOptions &call_options() {
    if (t_call_options != nullptr) return *t_call_options;
    thread_local CallOptions d;
    d = default_call_options();
    return d;
}

CallScope::CallScope(const CallOptions &o) : opts_(o), prev_(t_call_options) { t_call_options = &opts_; }
CallScope::~CallScope() { t_call_options = prev_; }

void set_cuda_error(cudaError_t e) {
    std::snprintf(g_cuda_error, sizeof g_cuda_error, "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
}

const DeviceInfo &device_info() {
    static std::mutex mu;
    static DeviceInfo infos[64];
    static bool have[64] = {};
    static DeviceInfo fallback;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return fallback;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!have[dev]) {
        DeviceInfo d;
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
        cudaGetLastError();
        if (d.sms <= 0) d.sms = 1;
        if (d.smem_optin <= 0) d.smem_optin = 48 * 1024;
        infos[dev] = d;
        have[dev] = true;
    }
    return infos[dev];
}

static bool valid_group(int32_t g) { return g == 32 || g == 64 || g == 128; }

// Byte ranges [lo, hi) of the arrays of a call, for the check that no output overlaps
// an input or another output (the kernels read inputs while other CTAs store results).
struct Span {
    uintptr_t lo, hi;
};
static Span span(const void *p, int64_t bytes) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return Span{a, p == nullptr ? a : a + static_cast<uintptr_t>(bytes)};
}
static bool overlap(Span a, Span b) { return a.lo < b.hi && b.lo < a.hi; }
static bool overlaps_any(Span out, const Span *in, int n) {
    for (int i = 0; i < n; ++i)
        if (overlap(out, in[i])) return true;
    return false;
}
// The packed-weight arrays of an N x K matrix of group g (zeros may be null).
static int weight_spans(const void *codes, const void *scales, const void *zeros, int64_t N, int64_t K, int32_t g,
                        Span *out) {
    const int64_t nb = K / g;
    out[0] = span(codes, N * (K / 2));
    out[1] = span(scales, N * nb * 2);
    out[2] = span(zeros, N * ((nb + 1) / 2));
    return 3;
}

// Scalar checks shared by the packed-weight entry points.
static int check_shape(int64_t M, int64_t N, int64_t K, int32_t group) {
    if (M < 0 || N < 0 || K < 1 || !valid_group(group) || K % group != 0) return Q4_ERR_INVALID_ARG;
    if (N > 0x7fffffffLL || K > 0x7fffffffLL) return Q4_ERR_UNSUPPORTED;
    return Q4_OK;
}

int check_q4_args(const void *codes, const void *scales, int64_t N, int64_t K, int32_t group) {
    (void)N;
    (void)K;
    (void)group;
    if (codes == nullptr || scales == nullptr) return Q4_ERR_INVALID_ARG;
    if (!aligned(codes, 16) || !aligned(scales, 2)) return Q4_ERR_MISALIGNED;
    return Q4_OK;
}

#ifdef Q4_BOUNDS_CHECK
__device__ unsigned int g_bounds_violations = 0;

unsigned int *bounds_counter() {
    static std::atomic<unsigned int *> addr[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    if (addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_bounds_violations) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        addr[dev] = static_cast<unsigned int *>(p);
    }
    return addr[dev];
}
#else
unsigned int *bounds_counter() { return nullptr; }
#endif

}  // namespace q4

using namespace q4;

extern "C" {

const char *q4gemv_status_string(int status) {
    switch (status) {
        case Q4_OK: return "ok";
        case Q4_ERR_INVALID_ARG: return "invalid argument";
        case Q4_ERR_UNSUPPORTED: return "unsupported size";
        case Q4_ERR_MISALIGNED: return "misaligned pointer";
        case Q4_ERR_CUDA: return "CUDA runtime error";
        case Q4_ERR_TIMEOUT: return "device-side wait timed out";
        default: return "unknown status";
    }
}

const char *q4gemv_last_cuda_error(void) { return g_cuda_error; }

int q4gemv_pack_info(int64_t N, int64_t K, int32_t group, q4gemv_pack_info_t *out) {
    if (out == nullptr || N < 0 || K < 1 || !valid_group(group) || K % group != 0) return Q4_ERR_INVALID_ARG;
    const int64_t nb = K / group;
    std::memset(out, 0, sizeof *out);
    out->n = N;
    out->k = K;
    out->group = group;
    out->blocks_per_row = static_cast<int32_t>(nb);
    out->codes_row_bytes = K / 2;
    out->codes_bytes = N * (K / 2);
    out->scales_row_bytes = 2 * nb;
    out->scales_bytes = N * 2 * nb;
    out->zeros_row_bytes = (nb + 1) / 2;
    out->zeros_bytes = N * ((nb + 1) / 2);
    out->base_alignment = 16;
    return Q4_OK;
}

int q4gemv_run(const void *codes, const void *scales_f16, const void *zeros_u4_or_null, const float *x,
               float *y, int32_t M, int64_t N, int64_t K, int32_t group, void *stream) {
    int st = check_shape(M, N, K, group);
    if (st != Q4_OK) return st;
    if (M == 0 || N == 0) return Q4_OK;
    if (M > 16) return Q4_ERR_UNSUPPORTED;
    if ((st = check_q4_args(codes, scales_f16, N, K, group)) != Q4_OK) return st;
    if (x == nullptr || y == nullptr) return Q4_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(y, 4)) return Q4_ERR_MISALIGNED;
    {
        Span in[4];
        weight_spans(codes, scales_f16, zeros_u4_or_null, N, K, group, in);
        in[3] = span(x, 4 * M * K);
        if (overlaps_any(span(y, 4 * M * N), in, 4)) return Q4_ERR_INVALID_ARG;
    }
    return launch_q4gemv(static_cast<const uint8_t *>(codes), static_cast<const uint16_t *>(scales_f16),
                         static_cast<const uint8_t *>(zeros_u4_or_null), x, y, M, N, static_cast<int>(K), group,
                         static_cast<cudaStream_t>(stream));
}

int q4gemv_fused_run(const void *codes, const void *scales_f16, const void *zeros_u4_or_null, const float *x,
                     const float *gamma, float eps, float *y, int32_t M, int64_t N, int64_t K, int32_t group,
                     int32_t epilogue, void *stream) {
    int st = check_shape(M, N, K, group);
    if (st != Q4_OK) return st;
    if (epilogue != Q4_EPILOGUE_NONE && epilogue != Q4_EPILOGUE_SWIGLU) return Q4_ERR_INVALID_ARG;
    if (epilogue == Q4_EPILOGUE_SWIGLU && N % 2 != 0) return Q4_ERR_INVALID_ARG;
    if (gamma != nullptr && !(eps >= 0.0f && eps <= 3.0e38f)) return Q4_ERR_INVALID_ARG;   // NaN fails too
    if (M == 0 || N == 0) return Q4_OK;
    if (M > 16) return Q4_ERR_UNSUPPORTED;
    if ((st = check_q4_args(codes, scales_f16, N, K, group)) != Q4_OK) return st;
    if (x == nullptr || y == nullptr) return Q4_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(y, 4) || (gamma != nullptr && !aligned(gamma, 16))) return Q4_ERR_MISALIGNED;
    {
        Span in[5];
        weight_spans(codes, scales_f16, zeros_u4_or_null, N, K, group, in);
        in[3] = span(x, 4 * M * K);
        in[4] = span(gamma, 4 * K);
        const int64_t ycols = epilogue == Q4_EPILOGUE_SWIGLU ? N / 2 : N;
        if (overlaps_any(span(y, 4 * M * ycols), in, 5)) return Q4_ERR_INVALID_ARG;
    }
    if (gamma == nullptr && epilogue == Q4_EPILOGUE_NONE)
        return q4gemv_run(codes, scales_f16, zeros_u4_or_null, x, y, M, N, K, group, stream);
    return launch_q4gemv_fused(static_cast<const uint8_t *>(codes), static_cast<const uint16_t *>(scales_f16),
                               static_cast<const uint8_t *>(zeros_u4_or_null), x, gamma, eps,
                               epilogue == Q4_EPILOGUE_SWIGLU ? 1 : 0, y, M, N, static_cast<int>(K), group,
                               static_cast<cudaStream_t>(stream));
}

int q4gemv_grouped_run(const q4gemv_segment_t *segs, int32_t count, int64_t K, int32_t group, void *stream) {
    if (count < 0 || (count > 0 && segs == nullptr)) return Q4_ERR_INVALID_ARG;
    int st = check_shape(1, 1, K, group);
    if (st != Q4_OK) return st;
    // every check before any launch
    for (int32_t i = 0; i < count; ++i) {
        const q4gemv_segment_t &sg = segs[i];
        if (sg.N < 0) return Q4_ERR_INVALID_ARG;
        if (sg.N == 0) continue;
        if ((st = check_shape(1, sg.N, K, group)) != Q4_OK) return st;
        if ((st = check_q4_args(sg.codes, sg.scales_f16, sg.N, K, group)) != Q4_OK) return st;
        if (sg.x == nullptr || sg.y == nullptr) return Q4_ERR_INVALID_ARG;
        if (!aligned(sg.x, 16) || !aligned(sg.y, 4)) return Q4_ERR_MISALIGNED;
    }
    // the matrices must be independent: no output overlaps any matrix's inputs or another
    // output (one launch serves them all, with no order among its CTAs)
    for (int32_t i = 0; i < count; ++i) {
        const q4gemv_segment_t &si = segs[i];
        if (si.N == 0) continue;
        const Span yi = span(si.y, 4 * si.N);
        for (int32_t j = 0; j < count; ++j) {
            const q4gemv_segment_t &sj = segs[j];
            if (sj.N == 0) continue;
            Span in[5];
            weight_spans(sj.codes, sj.scales_f16, sj.zeros_u4_or_null, sj.N, K, group, in);
            in[3] = span(sj.x, 4 * K);
            in[4] = j != i ? span(sj.y, 4 * sj.N) : Span{0, 0};
            if (overlaps_any(yi, in, 5)) return Q4_ERR_INVALID_ARG;
        }
    }
    // runs of up to kStreamMaxSeg non-empty matrices: one streamed launch where it applies,
    // else one q4gemv_run per matrix
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t i = 0;
    while (i < count) {
        q4::StreamSeg run[q4::kStreamMaxSeg];
        int32_t idx[q4::kStreamMaxSeg];
        int n = 0;
        for (; i < count && n < q4::kStreamMaxSeg; ++i) {
            const q4gemv_segment_t &sg = segs[i];
            if (sg.N == 0) continue;
            run[n].codes = static_cast<const uint8_t *>(sg.codes);
            run[n].scales = static_cast<const uint16_t *>(sg.scales_f16);
            run[n].zeros = static_cast<const uint8_t *>(sg.zeros_u4_or_null);
            run[n].x = sg.x;
            run[n].y = sg.y;
            run[n].N = sg.N;
            run[n].nblocks = 0;
            run[n].cta_begin = 0;
            idx[n++] = i;
        }
        if (n == 0) break;
        if (!call_options().exact_x && q4::stream_grouped_applies(run, n, static_cast<int>(K), group)) {
            st = q4::launch_q4gemv_stream_grouped(run, n, static_cast<int>(K), group, s);
            if (st != Q4_OK) return st;
            continue;
        }
        for (int j = 0; j < n; ++j) {
            const q4gemv_segment_t &sg = segs[idx[j]];
            st = q4gemv_run(sg.codes, sg.scales_f16, sg.zeros_u4_or_null, sg.x, sg.y, 1, sg.N, K, group, stream);
            if (st != Q4_OK) return st;
        }
    }
    return Q4_OK;
}

int q4gemv_grouped_split(const int64_t *N, int32_t count, int64_t K, int32_t group, int32_t grid_max,
                         int32_t *nblocks, int32_t *cta_begin) {
    if (N == nullptr || nblocks == nullptr || cta_begin == nullptr || count < 1) return -Q4_ERR_INVALID_ARG;
    const int st = check_shape(1, 1, K, group);
    if (st != Q4_OK) return -st;
    return q4::stream_grouped_split(N, count, static_cast<int>(K), group, grid_max, nblocks, cta_begin);
}

int q4_0_gemv_run(const void *blocks, const float *x, float *y, int32_t M, int64_t N, int64_t K, void *stream) {
    if (M < 0 || N < 0 || K < 32 || K % 32 != 0) return Q4_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return Q4_OK;
    if (M > 16 || N > 0x7fffffffLL || K > 0x7fffffffLL) return Q4_ERR_UNSUPPORTED;
    if (blocks == nullptr || x == nullptr || y == nullptr) return Q4_ERR_INVALID_ARG;
    if (!aligned(blocks, 2) || !aligned(x, 16) || !aligned(y, 4)) return Q4_ERR_MISALIGNED;
    {
        const Span in[2] = {span(blocks, N * (K / 32) * 18), span(x, 4 * M * K)};
        if (overlaps_any(span(y, 4 * M * N), in, 2)) return Q4_ERR_INVALID_ARG;
    }
    return launch_q40gemv(static_cast<const uint8_t *>(blocks), x, y, M, N, static_cast<int>(K),
                          static_cast<cudaStream_t>(stream));
}

int q8_0_gemv_run(const void *blocks, const float *x, float *y, int32_t M, int64_t N, int64_t K, void *stream) {
    if (M < 0 || N < 0 || K < 32 || K % 32 != 0) return Q4_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return Q4_OK;
    if (M > 16 || N > 0x7fffffffLL || K > 0x7fffffffLL) return Q4_ERR_UNSUPPORTED;
    if (blocks == nullptr || x == nullptr || y == nullptr) return Q4_ERR_INVALID_ARG;
    if (!aligned(blocks, 2) || !aligned(x, 16) || !aligned(y, 4)) return Q4_ERR_MISALIGNED;
    {
        const Span in[2] = {span(blocks, N * (K / 32) * 34), span(x, 4 * M * K)};
        if (overlaps_any(span(y, 4 * M * N), in, 2)) return Q4_ERR_INVALID_ARG;
    }
    return launch_q80gemv(static_cast<const uint8_t *>(blocks), x, y, M, N, static_cast<int>(K),
                          static_cast<cudaStream_t>(stream));
}

int q4gemm_run(const void *codes, const void *scales_f16, const void *zeros_u4_or_null, const void *a_bf16,
               float *c, int32_t M, int64_t N, int64_t K, int32_t group, void *stream) {
    int st = check_shape(M, N, K, group);
    if (st != Q4_OK) return st;
    if (M == 0 || N == 0) return Q4_OK;
    if ((st = check_q4_args(codes, scales_f16, N, K, group)) != Q4_OK) return st;
    if (a_bf16 == nullptr || c == nullptr) return Q4_ERR_INVALID_ARG;
    if (!aligned(a_bf16, 16) || !aligned(c, 4)) return Q4_ERR_MISALIGNED;
    {
        Span in[4];
        weight_spans(codes, scales_f16, zeros_u4_or_null, N, K, group, in);
        in[3] = span(a_bf16, 2 * M * K);
        if (overlaps_any(span(c, 4 * M * N), in, 4)) return Q4_ERR_INVALID_ARG;
    }
    return launch_q4gemm(static_cast<const uint8_t *>(codes), static_cast<const uint16_t *>(scales_f16),
                         static_cast<const uint8_t *>(zeros_u4_or_null), static_cast<const uint16_t *>(a_bf16), c,
                         M, N, static_cast<int>(K), group, static_cast<cudaStream_t>(stream));
}

int f32gemv_run(const float *W, const float *x, float *y, int32_t M, int64_t N, int64_t K, void *stream) {
    if (M < 0 || N < 0 || K < 1) return Q4_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return Q4_OK;
    if (M > 16 || K % 4 != 0 || N > 0x7fffffffLL || K > 0x7fffffffLL) return Q4_ERR_UNSUPPORTED;
    if (W == nullptr || x == nullptr || y == nullptr) return Q4_ERR_INVALID_ARG;
    if (!aligned(W, 16) || !aligned(x, 16) || !aligned(y, 4)) return Q4_ERR_MISALIGNED;
    {
        const Span in[2] = {span(W, 4 * N * K), span(x, 4 * M * K)};
        if (overlaps_any(span(y, 4 * M * N), in, 2)) return Q4_ERR_INVALID_ARG;
    }
    return launch_f32gemv(W, x, y, M, N, static_cast<int>(K), static_cast<cudaStream_t>(stream));
}

int q4_dequant_f32_run(const void *codes, const void *scales_f16, const void *zeros_u4_or_null, float *w,
                       int64_t N, int64_t K, int32_t group, void *stream) {
    int st = check_shape(1, N, K, group);
    if (st != Q4_OK) return st;
    if (N == 0) return Q4_OK;
    if ((st = check_q4_args(codes, scales_f16, N, K, group)) != Q4_OK) return st;
    if (w == nullptr) return Q4_ERR_INVALID_ARG;
    if (!aligned(w, 16)) return Q4_ERR_MISALIGNED;
    return launch_dequant(static_cast<const uint8_t *>(codes), static_cast<const uint16_t *>(scales_f16),
                          static_cast<const uint8_t *>(zeros_u4_or_null), w, false, N, static_cast<int>(K), group,
                          static_cast<cudaStream_t>(stream));
}

int q4_dequant_bf16_run(const void *codes, const void *scales_f16, const void *zeros_u4_or_null, uint16_t *wb,
                        int64_t N, int64_t K, int32_t group, void *stream) {
    int st = check_shape(1, N, K, group);
    if (st != Q4_OK) return st;
    if (N == 0) return Q4_OK;
    if ((st = check_q4_args(codes, scales_f16, N, K, group)) != Q4_OK) return st;
    if (wb == nullptr) return Q4_ERR_INVALID_ARG;
    if (!aligned(wb, 16)) return Q4_ERR_MISALIGNED;
    return launch_dequant(static_cast<const uint8_t *>(codes), static_cast<const uint16_t *>(scales_f16),
                          static_cast<const uint8_t *>(zeros_u4_or_null), wb, true, N, static_cast<int>(K), group,
                          static_cast<cudaStream_t>(stream));
}

int q4gemv_device_status(void *stream) { return read_device_status(static_cast<cudaStream_t>(stream)); }

#ifdef Q4_BOUNDS_CHECK
int q4gemv_bounds_violations(void *stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    unsigned int v = 0;
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&v, q4::g_bounds_violations, sizeof v);
    if (e == cudaSuccess && v != 0) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(q4::g_bounds_violations, &zero, sizeof zero);
    }
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return -Q4_ERR_CUDA;
    }
    return static_cast<int>(v);
}
#else
int q4gemv_bounds_violations(void *) { return -1; }
#endif


int q4gemm_set_wait_timeout_ns(uint64_t ns) {
    set_default_wait_ns(ns);
    return Q4_OK;
}

int q4gemv_set_overlapped_launch(int enable) { return set_overlapped_launch(enable != 0) ? 1 : 0; }

int vec4_read_probe_run(const void *buf, int64_t bytes, float *partial, int32_t blocks, int32_t *blocks_used,
                        void *stream) {
    if (buf == nullptr || partial == nullptr || bytes <= 0 || bytes % 16 != 0) return Q4_ERR_INVALID_ARG;
    if (!aligned(buf, 16) || !aligned(partial, 4)) return Q4_ERR_MISALIGNED;
    if (blocks <= 0) blocks = device_info().sms * 8;
    if (blocks_used) *blocks_used = blocks;
    return launch_read_probe(static_cast<const float4 *>(buf), bytes / 16, partial, blocks,
                             static_cast<cudaStream_t>(stream));
}

// ---- entry points with per-call options ----

static int options_from(const q4_run_options_t *o, uint32_t allowed, CallOptions &out) {
    out = CallOptions{};   // built-in defaults, whatever the process-wide settings are
    if (o == nullptr) return Q4_OK;
    if (o->reserved != 0 || (o->flags & ~allowed) != 0) return Q4_ERR_INVALID_ARG;
    out.overlap = (o->flags & Q4_RUN_OVERLAPPED) != 0;
    out.exact_x = (o->flags & Q4_RUN_EXACT_X) != 0;
    if (o->flags & Q4_RUN_WAIT_TIMEOUT) out.wait_ns = o->wait_timeout_ns;
    return Q4_OK;
}

constexpr uint32_t kGemvFlags = Q4_RUN_OVERLAPPED | Q4_RUN_EXACT_X | Q4_RUN_WAIT_TIMEOUT;

int q4gemv_run_ex(const void *codes, const void *scales_f16, const void *zeros_u4_or_null, const float *x, float *y,
                  int32_t M, int64_t N, int64_t K, int32_t group, const q4_run_options_t *opts, void *stream) {
    CallOptions co;
    const int st = options_from(opts, kGemvFlags, co);
    if (st != Q4_OK) return st;
    CallScope scope(co);
    return q4gemv_run(codes, scales_f16, zeros_u4_or_null, x, y, M, N, K, group, stream);
}

int q4gemv_fused_run_ex(const void *codes, const void *scales_f16, const void *zeros_u4_or_null, const float *x,
                        const float *gamma, float eps, float *y, int32_t M, int64_t N, int64_t K, int32_t group,
                        int32_t epilogue, const q4_run_options_t *opts, void *stream) {
    CallOptions co;
    const int st = options_from(opts, kGemvFlags, co);
    if (st != Q4_OK) return st;
    CallScope scope(co);
    return q4gemv_fused_run(codes, scales_f16, zeros_u4_or_null, x, gamma, eps, y, M, N, K, group, epilogue, stream);
}

int q4gemv_grouped_run_ex(const q4gemv_segment_t *segs, int32_t count, int64_t K, int32_t group,
                          const q4_run_options_t *opts, void *stream) {
    CallOptions co;
    const int st = options_from(opts, kGemvFlags, co);
    if (st != Q4_OK) return st;
    CallScope scope(co);
    return q4gemv_grouped_run(segs, count, K, group, stream);
}

int q4gemm_run_ex(const void *codes, const void *scales_f16, const void *zeros_u4_or_null, const void *a_bf16,
                  float *c, int32_t M, int64_t N, int64_t K, int32_t group, const q4_run_options_t *opts,
                  void *stream) {
    CallOptions co;
    const int st = options_from(opts, Q4_RUN_OVERLAPPED | Q4_RUN_WAIT_TIMEOUT, co);
    if (st != Q4_OK) return st;
    CallScope scope(co);
    return q4gemm_run(codes, scales_f16, zeros_u4_or_null, a_bf16, c, M, N, K, group, stream);
}

}  // extern "C"
