// q4gemv_stream_k8192.cu -- compile-time row geometry of the streamed M = 1 GEMV for
// K = 8192 (2 row groups per block), groups 32, 64 and 128.
#include "q4gemv_stream_kernel.cuh"

namespace q4 {

Q4_STREAM_K_LAUNCHER(8192, 2)

}  // namespace q4
