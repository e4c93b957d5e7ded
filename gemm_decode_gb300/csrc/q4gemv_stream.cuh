// q4gemv_stream.cuh -- launch interface of the TMA-streamed M = 1 int4 GEMV.
#pragma once

#include "q4_common.cuh"

namespace q4 {

struct StreamArgs {
    const uint8_t *codes;
    const uint16_t *scales;
    const uint8_t *zeros;
    const float *x;
    float *y;
    int64_t N;
    int nblocks;                     // blocks of rows (set by the launcher)
    unsigned long long timeout_ns;   // bound on every mbarrier wait
};

// True when the streamed kernel serves this problem (M = 1, a compiled row
// geometry, 16-byte aligned side arrays, enough rows).
bool stream_applies(int M, int64_t N, int K, int group, const void *codes, const void *scales, const void *zeros);
int launch_q4gemv_stream(const uint8_t *codes, const uint16_t *scales, const uint8_t *zeros, const float *x,
                         float *y, int64_t N, int K, int group, cudaStream_t stream);
void set_stream_wait_timeout_ns(unsigned long long ns);
int read_and_clear_stream_status(unsigned int *v);

}  // namespace q4
