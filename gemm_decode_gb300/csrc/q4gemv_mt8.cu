// GEMV kernel instantiations for an M tile of 8 row(s) of x.
#include "q4gemv_launch.cuh"

namespace q4 {
template int launch_q4gemv_mt<8>(const GemvPlan &, const GemvArgs &, cudaStream_t);
template int launch_q4gemv_fused_mt<8>(const GemvPlan &, const GemvArgs &, cudaStream_t);
template int launch_q40_mt<8>(const GemvPlan &, const GemvArgs &, cudaStream_t);
}  // namespace q4
