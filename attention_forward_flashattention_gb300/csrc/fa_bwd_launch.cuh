// Launch of the backward kernels of one head dimension (included by
// fa_bwd_d64.cu / fa_bwd_d128.cu).
#pragma once

#include "fa_bwd.cuh"

namespace fa {
namespace bwd_detail {

template <int D, bool BF16, bool CAUSAL>
cudaError_t launch(const CUtensorMap* m, const BwdArgs& a, const void* o, const void* dout,
                   const float* lse, int grid, cudaStream_t st) {
  const long long rows = static_cast<long long>(a.BH) * a.n_t * 128;
  // eight threads per padded row, at most 2^20 blocks (the kernel strides)
  const long long blocks = (rows * 8 + 255) / 256;
  bwd_prep_kernel<D, BF16><<<static_cast<unsigned>(blocks < (1LL << 20) ? blocks : (1LL << 20)),
                             256, 0, st>>>(
      o, dout, lse, const_cast<float*>(a.lse2), const_cast<float*>(a.delta), a.N, a.n_t, rows);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  constexpr int kSmemKV = BwdLayout<D, true>::kSmemBytes;
  constexpr int kSmemQ = BwdLayout<D, false>::kSmemBytes;
  auto kv = fa_bwd_kernel<D, BF16, CAUSAL, true>;
  auto kq = fa_bwd_kernel<D, BF16, CAUSAL, false>;
  if ((e = cudaFuncSetAttribute(kv, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemKV)) !=
          cudaSuccess ||
      (e = cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemQ)) !=
          cudaSuccess)
    return e;
  kv<<<grid, kBwdThreads, kSmemKV, st>>>(m[0], m[1], m[2], m[3], a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  kq<<<grid, kBwdThreads, kSmemQ, st>>>(m[0], m[1], m[2], m[3], a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(bool bf16, bool causal, const CUtensorMap* m, const BwdArgs& a,
                     const void* o, const void* dout, const float* lse, int grid,
                     cudaStream_t st) {
  if (grid <= 0) return cudaErrorInvalidValue;
  if (bf16)
    return causal ? launch<D, true, true>(m, a, o, dout, lse, grid, st)
                  : launch<D, true, false>(m, a, o, dout, lse, grid, st);
  return causal ? launch<D, false, true>(m, a, o, dout, lse, grid, st)
                : launch<D, false, false>(m, a, o, dout, lse, grid, st);
}

}  // namespace bwd_detail
}  // namespace fa
