// q4gemv_stream_k4096.cu -- compile-time row geometry of the streamed M = 1 GEMV for
// K = 4096 (4 row groups per block), groups 32, 64 and 128.
#include "q4gemv_stream_kernel.cuh"

namespace q4 {

Q4_STREAM_K_LAUNCHER(4096, 4)

}  // namespace q4
