// q4gemv_stream_k16384.cu -- compile-time row geometry of the streamed M = 1 GEMV for
// K = 16384 (1 row group per block), groups 32, 64 and 128.
#include "q4gemv_stream_kernel.cuh"

namespace q4 {

Q4_STREAM_K_LAUNCHER(16384, 1)

}  // namespace q4
