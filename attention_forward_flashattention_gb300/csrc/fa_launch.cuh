// Launch of the attention forward kernel instances of one head dimension
// (included by fa_fwd_d64.cu / fa_fwd_d128.cu, one translation unit each so
// the instances compile in parallel).
#pragma once

#include "fa_kernel.cuh"

namespace fa {
namespace launch_detail {

template <int D, bool BF16, bool CAUSAL>
cudaError_t launch_one(const CUtensorMap* m, const FwdArgs& a, int grid, cudaStream_t st) {
  constexpr int kSmem = Layout<D>::kSmemBytes;
  auto kern = fa_fwd_kernel<D, BF16, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kFwdThreads, kSmem, st>>>(m[0], m[1], m[2], m[3], a);
  return cudaGetLastError();
}

// One CTA per SM at most (each holds the SM's TMEM and most of its shared memory).
inline int fwd_grid(int n_units, int sm_count) { return n_units < sm_count ? n_units : sm_count; }

template <int D>
cudaError_t launch_fwd(bool bf16, bool causal, const CUtensorMap* maps, const FwdArgs& a,
                       int grid, cudaStream_t stream) {
  if (grid <= 0) return cudaErrorInvalidValue;
  if (bf16)
    return causal ? launch_one<D, true, true>(maps, a, grid, stream)
                  : launch_one<D, true, false>(maps, a, grid, stream);
  return causal ? launch_one<D, false, true>(maps, a, grid, stream)
                : launch_one<D, false, false>(maps, a, grid, stream);
}

}  // namespace launch_detail
}  // namespace fa
