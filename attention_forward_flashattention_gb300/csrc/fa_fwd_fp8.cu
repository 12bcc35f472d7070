// Instances of the attention forward kernel for 8-bit (e4m3) inputs, head
// dimension 128, bf16 output (full / causal), and their launch.
#include "fa_launch.cuh"

namespace fa {
namespace {

template <bool CAUSAL>
cudaError_t launch_one_fp8(const CUtensorMap* m, const FwdArgs& a, int grid, cudaStream_t st) {
  constexpr int kSmem = Layout<128, true>::kSmemBytes;
  auto kern = fa_fwd_kernel<128, true, CAUSAL, true>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kFwdThreads, kSmem, st>>>(m[0], m[1], m[2], m[3], a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_fp8(bool causal, const CUtensorMap* maps, const FwdArgs& a, int grid,
                           cudaStream_t stream) {
  if (grid <= 0) return cudaErrorInvalidValue;
  return causal ? launch_one_fp8<true>(maps, a, grid, stream)
                : launch_one_fp8<false>(maps, a, grid, stream);
}

int fwd_smem_bytes_fp8() { return Layout<128, true>::kSmemBytes; }

}  // namespace fa
