// Instances of the attention forward kernel for head dimension 128
// (fp16 / bf16, full / causal) and their launch.
#include "fa_kernel.cuh"

namespace fa {
namespace {

template <bool BF16, bool CAUSAL>
cudaError_t launch_one(const CUtensorMap* m, const FwdArgs& a, int grid, cudaStream_t st) {
  constexpr int kSmem = Layout<128>::kSmemBytes;
  auto kern = fa_fwd_kernel<128, BF16, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kFwdThreads, kSmem, st>>>(m[0], m[1], m[2], a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_d128(bool bf16, bool causal, const CUtensorMap* maps, const FwdArgs& a,
                           int grid, cudaStream_t stream) {
  if (bf16)
    return causal ? launch_one<true, true>(maps, a, grid, stream)
                  : launch_one<true, false>(maps, a, grid, stream);
  return causal ? launch_one<false, true>(maps, a, grid, stream)
                : launch_one<false, false>(maps, a, grid, stream);
}

}  // namespace fa
