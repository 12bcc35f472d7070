// Backward kernels for head dimension 64 (fp16 / bf16, full / causal).
#include "fa_bwd_launch.cuh"

namespace fa {

cudaError_t launch_bwd_d64(bool bf16, bool causal, const CUtensorMap* maps, const BwdArgs& a,
                           const void* o, const void* dout, const float* lse, int grid,
                           cudaStream_t stream) {
  return bwd_detail::launch_d<64>(bf16, causal, maps, a, o, dout, lse, grid, stream);
}

}  // namespace fa
