// Instances of the attention forward kernel for head dimension 128
// (fp16 / bf16, full / causal) and their launch.
#include "fa_launch.cuh"

namespace fa {

int fwd_grid_d128(int n_units, int sm_count) {
  return launch_detail::fwd_grid(n_units, sm_count);
}

cudaError_t launch_fwd_d128(bool bf16, bool causal, const CUtensorMap* maps, const FwdArgs& a,
                            int grid, cudaStream_t stream) {
  return launch_detail::launch_fwd<128>(bf16, causal, maps, a, grid, stream);
}

}  // namespace fa
