// Instances of the CTA-pair attention forward (head dimension 128, fp16 /
// bf16 / e4m3, full / causal) and their launch.
#include "fa_pair.cuh"

namespace fa {
namespace {

template <bool BF16, bool CAUSAL, bool FP8 = false>
cudaError_t launch_one_pair(const CUtensorMap* m, const FwdArgs& a, int grid, cudaStream_t st) {
  constexpr int kSmem = PairLayout<FP8>::kSmemBytes;
  auto kern = fa_fwd_pair_kernel<BF16, CAUSAL, FP8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kFwdThreads, kSmem, st>>>(m[0], m[1], m[2], m[3], a);  // clusters of 2 CTAs
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_pair(bool bf16, bool causal, const CUtensorMap* maps, const FwdArgs& a,
                            int grid, cudaStream_t stream) {
  if (grid <= 0 || (grid & 1)) return cudaErrorInvalidValue;
  if (bf16)
    return causal ? launch_one_pair<true, true>(maps, a, grid, stream)
                  : launch_one_pair<true, false>(maps, a, grid, stream);
  return causal ? launch_one_pair<false, true>(maps, a, grid, stream)
                : launch_one_pair<false, false>(maps, a, grid, stream);
}

cudaError_t launch_fwd_pair_fp8(bool causal, const CUtensorMap* maps, const FwdArgs& a, int grid,
                                cudaStream_t stream) {
  if (grid <= 0 || (grid & 1)) return cudaErrorInvalidValue;
  return causal ? launch_one_pair<true, true, true>(maps, a, grid, stream)
                : launch_one_pair<true, false, true>(maps, a, grid, stream);
}

int fwd_smem_bytes_pair(bool fp8) {
  return fp8 ? PairLayout<true>::kSmemBytes : PairLayout<false>::kSmemBytes;
}

}  // namespace fa
