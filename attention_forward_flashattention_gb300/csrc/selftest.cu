// GPU unit tests of the building blocks of the attention kernel, exported as
// a separate library (libfa_selftest.so) that only the test suite loads.
//
//   fa_selftest_gemm_qk : C[128][128] = A[128][K] * B[128][K]^T (fp32), with A
//                         and B fetched by TMA into SW128 panels and multiplied
//                         by the same issue_qk sequence the attention kernel
//                         uses for S = Q K^T (covers the K-advance across the
//                         panel boundary at K = 128, the pitfall of the B300
//                         walkthrough, V14), read back by tcgen05.ld per warp
//                         lane quarter.
//   fa_selftest_gemm_pv : C[128][N] = A[128][128] * B[128][N], with A written
//                         by threads through store_row128_sw128 (the P path)
//                         and B fetched by TMA and used MN-major (the V path).
//                         `variant` swaps the two byte offsets of the B
//                         descriptor (both stay inside the B tile), so one run
//                         shows which assignment the hardware expects.
//   fa_selftest_gemm_ts : as gemm_pv, but A is stored by the threads into TMEM
//                         with tcgen05.st (packed pairs) and the MMA reads it
//                         from there (the P-in-TMEM path).
//   fa_selftest_gemm_qk_pair / _pv_pair : the same two products on a CTA pair
//                         (cta_group::2, M = 256): each CTA loads half of the
//                         B operand, the even CTA issues the MMAs, each CTA
//                         reads back its own 128 rows.
//   fa_selftest_wait_timeout : a wait on a barrier nothing completes, with a
//                         short limit; checks that the bounded wait gives up,
//                         records its status bit and lets the kernel exit.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fa_common.cuh"

namespace fa {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// rows x cols 16-bit row-major matrix, box = 64 columns x box_rows rows, SW128.
bool encode_2d(CUtensorMap* m, const void* ptr, bool bf16, int cols, int rows, int box_rows = 128) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows), 1u};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2u,
                                 static_cast<cuuint64_t>(cols) * rows * 2u};
  const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(box_rows), 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
             const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kSmemBytes = 4 * kPanelBytes + 1024 + 256;

struct Smem {
  uint32_t base;   // 1024-aligned: operand A panels at +0, B panels at +32 KB
  uint32_t bars;   // bar 0: TMA, bar 1: MMA done
  uint32_t* tmem_slot;
  volatile uint32_t* abort_flag;
};

__device__ Smem carve(uint8_t* raw) {
  const uint32_t r = ptx::smem_u32(raw);
  Smem s;
  s.base = (r + 1023u) & ~1023u;
  s.bars = s.base + 4 * kPanelBytes;
  uint8_t* g = raw + (s.base - r) + 4 * kPanelBytes;
  s.tmem_slot = reinterpret_cast<uint32_t*>(g + 64);
  s.abort_flag = reinterpret_cast<volatile uint32_t*>(g + 68);
  return s;
}

// Each warp copies its 32 TMEM lanes x ncols fp32 columns to C[row][col].
__device__ void read_back(uint32_t tmem, float* c, int ncols) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = warp * 32 + lane;
  for (int c0 = 0; c0 < ncols; c0 += 32) {
    uint32_t v[32];
    ptx::tmem_ld32(ptx::tmem_lane_base(tmem, warp) + c0, v);
    ptx::tmem_ld_wait(v);
    for (int e = 0; e < 32; ++e) c[row * ncols + c0 + e] = __uint_as_float(v[e]);
  }
}

template <int K, bool BF16>
__global__ void __launch_bounds__(128, 1)
    gemm_qk_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb,
                   float* c, uint32_t* status) {
  extern __shared__ __align__(1024) uint8_t raw[];
  const Smem s = carve(raw);
  const AbortCtx ab{s.abort_flag, status};
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    ptx::mbar_init(s.bars, 1);
    ptx::mbar_init(s.bars + 8, 1);
    *s.abort_flag = 0u;
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(ptx::smem_u32(s.tmem_slot), 128);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *s.tmem_slot;
  constexpr int kPanels = K / 64;
  bool ok = true;
  if (threadIdx.x == 0) {
    ptx::mbar_arrive_expect_tx(s.bars, 2 * kPanels * kPanelBytes);
    for (int p = 0; p < kPanels; ++p) {
      ptx::tma_load_3d(s.base + p * kPanelBytes, &ta, s.bars, 64 * p, 0, 0);
      ptx::tma_load_3d(s.base + 2 * kPanelBytes + p * kPanelBytes, &tb, s.bars, 64 * p, 0, 0);
    }
    ok = wait_bounded(s.bars, 0, ab, kStatusSelftest);
    if (ok) {
      ptx::tc_fence_after();
      issue_qk<K, BF16>(tmem, s.base, s.base + 2 * kPanelBytes);
    }
    ptx::umma_commit(s.bars + 8);
    if (!ok) wait_drain(s.bars, 0, ab, kStatusDrain);
  }
  __syncwarp();
  const bool done = wait_bounded_warp(s.bars + 8, 0, ab, kStatusSelftest);
  ptx::tc_fence_after();
  if (done && !*s.abort_flag) read_back(tmem, c, 128);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 0) ptx::tmem_dealloc(tmem, 128);
}

template <int N, bool BF16>
__global__ void __launch_bounds__(128, 1)
    gemm_pv_kernel(const uint16_t* a, const __grid_constant__ CUtensorMap tb, float* c,
                   int variant, uint32_t* status) {
  extern __shared__ __align__(1024) uint8_t raw[];
  const Smem s = carve(raw);
  const AbortCtx ab{s.abort_flag, status};
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    ptx::mbar_init(s.bars, 1);
    ptx::mbar_init(s.bars + 8, 1);
    *s.abort_flag = 0u;
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(ptx::smem_u32(s.tmem_slot), 128);
    ptx::tmem_relinquish();
  }
  // A: each thread writes its row of 128 elements the way softmax writes P.
  {
    const int r = threadIdx.x;
    uint32_t pk[64];
    const uint32_t* src = reinterpret_cast<const uint32_t*>(a + r * 128);
    for (int i = 0; i < 64; ++i) pk[i] = src[i];
    store_row128_sw128(s.base, r, pk);
    ptx::fence_proxy_async_smem();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *s.tmem_slot;
  constexpr int kPanels = N / 64;
  bool ok = true;
  if (threadIdx.x == 0) {
    ptx::mbar_arrive_expect_tx(s.bars, kPanels * kPanelBytes);
    for (int p = 0; p < kPanels; ++p)
      ptx::tma_load_3d(s.base + 2 * kPanelBytes + p * kPanelBytes, &tb, s.bars, 64 * p, 0, 0);
    ok = wait_bounded(s.bars, 0, ab, kStatusSelftest);
    if (ok) {
      ptx::tc_fence_after();
      const uint32_t lbo = variant == 0 ? kPanelBytes : 1024u;
      const uint32_t sbo = variant == 0 ? 1024u : kPanelBytes;
      issue_pv<N, BF16>(tmem, s.base, s.base + 2 * kPanelBytes, false, lbo, sbo);
    }
    ptx::umma_commit(s.bars + 8);
    if (!ok) wait_drain(s.bars, 0, ab, kStatusDrain);
  }
  __syncwarp();
  const bool done = wait_bounded_warp(s.bars + 8, 0, ab, kStatusSelftest);
  ptx::tc_fence_after();
  if (done && !*s.abort_flag) read_back(tmem, c, N);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 0) ptx::tmem_dealloc(tmem, 128);
}

// C[128][N] = A[128][128] * B[128][N] with A stored by the threads into TMEM
// (tcgen05.st, packed pairs, columns 128..191) and multiplied from there.
template <int N, bool BF16>
__global__ void __launch_bounds__(128, 1)
    gemm_ts_kernel(const uint16_t* a, const __grid_constant__ CUtensorMap tb, float* c,
                   uint32_t* status) {
  extern __shared__ __align__(1024) uint8_t raw[];
  const Smem s = carve(raw);
  const AbortCtx ab{s.abort_flag, status};
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    ptx::mbar_init(s.bars, 1);
    ptx::mbar_init(s.bars + 8, 1);
    *s.abort_flag = 0u;
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(ptx::smem_u32(s.tmem_slot), 256);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *s.tmem_slot;
  {
    const int r = threadIdx.x;
    uint32_t pk[2][32];
    const uint32_t* src = reinterpret_cast<const uint32_t*>(a + r * 128);
    for (int i = 0; i < 64; ++i) pk[i >> 5][i & 31] = src[i];
    const uint32_t t = ptx::tmem_lane_base(tmem, warp) + 128u;
    ptx::tmem_st32(t, pk[0]);
    ptx::tmem_st32(t + 32u, pk[1]);
    ptx::tmem_st_wait();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  constexpr int kPanels = N / 64;
  bool ok = true;
  if (threadIdx.x == 0) {
    ptx::mbar_arrive_expect_tx(s.bars, kPanels * kPanelBytes);
    for (int p = 0; p < kPanels; ++p)
      ptx::tma_load_3d(s.base + 2 * kPanelBytes + p * kPanelBytes, &tb, s.bars, 64 * p, 0, 0);
    ok = wait_bounded(s.bars, 0, ab, kStatusSelftest);
    if (ok) {
      ptx::tc_fence_after();
      issue_pv_ts<N, BF16>(tmem, tmem + 128u, s.base + 2 * kPanelBytes, false);
    }
    ptx::umma_commit(s.bars + 8);
    if (!ok) wait_drain(s.bars, 0, ab, kStatusDrain);
  }
  __syncwarp();
  const bool done = wait_bounded_warp(s.bars + 8, 0, ab, kStatusSelftest);
  ptx::tc_fence_after();
  if (done && !*s.abort_flag) read_back(tmem, c, N);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 0) ptx::tmem_dealloc(tmem, 256);
}

// Pair (cta_group::2) version of gemm_qk for K = 128: C[256][128] = A * B^T.
// CTA r loads A rows 128r..+128 and B rows (keys) 64r..+64, counting the bytes
// on the even CTA's barrier; the even CTA issues M = 256 MMAs; each CTA reads
// back its own 128 rows of C.
template <bool BF16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1)
    gemm_qk_pair_kernel(const __grid_constant__ CUtensorMap ta,
                        const __grid_constant__ CUtensorMap tb, float* c, uint32_t* status,
                        int variant) {
  extern __shared__ __align__(1024) uint8_t raw[];
  const Smem s = carve(raw);  // A at +0 (32 KB), B at +32 KB (16 KB)
  const AbortCtx ab{s.abort_flag, status};
  const int warp = threadIdx.x >> 5;
  const uint32_t rank = ptx::cluster_ctarank();
  if (threadIdx.x == 0) {
    ptx::mbar_init(s.bars, 1);
    ptx::mbar_init(s.bars + 8, 1);
    *s.abort_flag = 0u;
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc_pair(ptx::smem_u32(s.tmem_slot), 128);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();
  ptx::tc_fence_after();
  const uint32_t tmem = *s.tmem_slot;
  const uint32_t lead_load = ptx::mapa_shared(s.bars, 0);
  if (threadIdx.x == 0) {
    if (rank == 0) ptx::mbar_arrive_expect_tx(s.bars, 2 * (2 * kPanelBytes + kPanelBytes));
    for (int p = 0; p < 2; ++p) {
      ptx::tma_load_3d_pair(s.base + p * kPanelBytes, &ta, lead_load, 64 * p, 128 * rank, 0);
      ptx::tma_load_3d_pair(s.base + 2 * kPanelBytes + p * (kPanelBytes / 2), &tb, lead_load,
                            64 * p, 64 * rank, 0);
    }
    if (rank == 0) {
      const bool ok = wait_cluster<false>(s.bars, 0, ab, kStatusSelftest);
      if (ok) {
        ptx::tc_fence_after();
        issue_qk_pair<BF16>(tmem, desc_kmajor(s.base), desc_kmajor(s.base + 2 * kPanelBytes));
      }
      if (variant == 2) {
        ptx::umma_commit_pair(s.bars + 8, 2);  // the peer, multicast
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                s.bars + 8)
            : "memory");                       // this CTA
      } else {
        ptx::umma_commit_pair(s.bars + 8, 3);
      }
    }
  }
  __syncwarp();
  const bool done = wait_cluster<true>(s.bars + 8, 0, ab, kStatusSelftest);
  const bool all_done = __all_sync(0xffffffffu, done) != 0;
  if (variant == 1) {  // read back 1 ms later
    const uint64_t t0 = ptx::globaltimer_ns();
    while (ptx::globaltimer_ns() - t0 < 1000000ull) {
    }
  }
  ptx::tc_fence_after();
  if (all_done && !*s.abort_flag) read_back(tmem, c + rank * 128 * 128, 128);
  ptx::tc_fence_before();
  ptx::cluster_sync();
  ptx::tc_fence_after();
  if (warp == 0) ptx::tmem_dealloc_pair(tmem, 128);
}

// Pair version of the P V product: C[256][128] = P[256][128] * V[128][128] with
// each CTA storing its 128 rows of P into its TMEM (columns 128..191), loading
// its 64 columns of V, and signalling "P ready" on the even CTA's barrier.
template <bool BF16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1)
    gemm_pv_pair_kernel(const uint16_t* a, const __grid_constant__ CUtensorMap tv, float* c,
                        uint32_t* status) {
  extern __shared__ __align__(1024) uint8_t raw[];
  const Smem s = carve(raw);  // V half at +0 (16 KB)
  const AbortCtx ab{s.abort_flag, status};
  const int warp = threadIdx.x >> 5;
  const uint32_t rank = ptx::cluster_ctarank();
  if (threadIdx.x == 0) {
    ptx::mbar_init(s.bars, 1);         // V loaded (both halves)
    ptx::mbar_init(s.bars + 8, 256);   // P stored (both CTAs)
    ptx::mbar_init(s.bars + 16, 1);    // MMA done
    *s.abort_flag = 0u;
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc_pair(ptx::smem_u32(s.tmem_slot), 256);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();
  ptx::tc_fence_after();
  const uint32_t tmem = *s.tmem_slot;
  {
    const int r = threadIdx.x;
    uint32_t pk[2][32];
    const uint32_t* src = reinterpret_cast<const uint32_t*>(a + (128 * rank + r) * 128);
    for (int i = 0; i < 64; ++i) pk[i >> 5][i & 31] = src[i];
    const uint32_t t = ptx::tmem_lane_base(tmem, warp) + 128u;
    ptx::tmem_st32(t, pk[0]);
    ptx::tmem_st32(t + 32u, pk[1]);
    ptx::tmem_st_wait();
    ptx::tc_fence_before();
    ptx::mbar_arrive_cluster(ptx::mapa_shared(s.bars + 8, 0));
  }
  if (threadIdx.x == 0) {
    if (rank == 0) ptx::mbar_arrive_expect_tx(s.bars, 2 * kPanelBytes);
    ptx::tma_load_3d_pair(s.base, &tv, ptx::mapa_shared(s.bars, 0), 64 * rank, 0, 0);
    if (rank == 0) {
      const bool ok = wait_cluster<false>(s.bars, 0, ab, kStatusSelftest) &&
                      wait_cluster<false>(s.bars + 8, 0, ab, kStatusSelftest);
      if (ok) {
        ptx::tc_fence_after();
        issue_pv_ts_pair<BF16>(tmem, tmem + 128u, desc_v(s.base), false);
      }
      ptx::umma_commit_pair(s.bars + 16, 3);
    }
  }
  __syncwarp();
  const bool done = wait_cluster<true>(s.bars + 16, 0, ab, kStatusSelftest);
  const bool all_done = __all_sync(0xffffffffu, done) != 0;
  ptx::tc_fence_after();
  if (all_done && !*s.abort_flag) read_back(tmem, c + rank * 128 * 128, 128);
  ptx::tc_fence_before();
  ptx::cluster_sync();
  ptx::tc_fence_after();
  if (warp == 0) ptx::tmem_dealloc_pair(tmem, 256);
}

// rows x cols byte matrix (e4m3 codes), box = 128 x 128 bytes, SW128.
bool encode_2d_u8(CUtensorMap* m, const void* ptr, int cols, int rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows), 1u};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols),
                                 static_cast<cuuint64_t>(cols) * rows};
  const cuuint32_t box[3] = {128u, 128u, 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// e4m3: C[128][128] = A[128][128] * B[128][128]^T (fp32), A and B fetched by
// TMA as one 128-byte SW128 panel each (the S = Q K^T path of the 8-bit kernel).
__global__ void __launch_bounds__(128, 1)
    gemm_qk_fp8_kernel(const __grid_constant__ CUtensorMap ta,
                       const __grid_constant__ CUtensorMap tb, float* c, uint32_t* status) {
  extern __shared__ __align__(1024) uint8_t raw[];
  const Smem s = carve(raw);
  const AbortCtx ab{s.abort_flag, status};
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    ptx::mbar_init(s.bars, 1);
    ptx::mbar_init(s.bars + 8, 1);
    *s.abort_flag = 0u;
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(ptx::smem_u32(s.tmem_slot), 128);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *s.tmem_slot;
  if (threadIdx.x == 0) {
    ptx::mbar_arrive_expect_tx(s.bars, 2 * kPanelBytes);
    ptx::tma_load_3d(s.base, &ta, s.bars, 0, 0, 0);
    ptx::tma_load_3d(s.base + 2 * kPanelBytes, &tb, s.bars, 0, 0, 0);
    const bool ok = wait_bounded(s.bars, 0, ab, kStatusSelftest);
    if (ok) {
      ptx::tc_fence_after();
      issue_qk_fp8(tmem, desc_kmajor(s.base), desc_kmajor(s.base + 2 * kPanelBytes));
    }
    ptx::umma_commit(s.bars + 8);
    if (!ok) wait_drain(s.bars, 0, ab, kStatusDrain);
  }
  __syncwarp();
  const bool done = wait_bounded_warp(s.bars + 8, 0, ab, kStatusSelftest);
  ptx::tc_fence_after();
  if (done && !*s.abort_flag) read_back(tmem, c, 128);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 0) ptx::tmem_dealloc(tmem, 128);
}

// e4m3: C[128][128] = A[128][128] * Bt[128][128]^T with A (four codes per
// 32-bit word, row r = 32 words) stored by the threads into TMEM columns
// 128..159 and read from there, Bt fetched by TMA (the P V^T path).
__global__ void __launch_bounds__(128, 1)
    gemm_ts_fp8_kernel(const uint32_t* a, const __grid_constant__ CUtensorMap tb, float* c,
                       uint32_t* status) {
  extern __shared__ __align__(1024) uint8_t raw[];
  const Smem s = carve(raw);
  const AbortCtx ab{s.abort_flag, status};
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    ptx::mbar_init(s.bars, 1);
    ptx::mbar_init(s.bars + 8, 1);
    *s.abort_flag = 0u;
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(ptx::smem_u32(s.tmem_slot), 256);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *s.tmem_slot;
  {
    uint32_t pk[32];
    for (int i = 0; i < 32; ++i) pk[i] = a[threadIdx.x * 32 + i];
    ptx::tmem_st32(ptx::tmem_lane_base(tmem, warp) + 128u, pk);
    ptx::tmem_st_wait();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (threadIdx.x == 0) {
    ptx::mbar_arrive_expect_tx(s.bars, kPanelBytes);
    ptx::tma_load_3d(s.base + 2 * kPanelBytes, &tb, s.bars, 0, 0, 0);
    const bool ok = wait_bounded(s.bars, 0, ab, kStatusSelftest);
    if (ok) {
      ptx::tc_fence_after();
      issue_pv_fp8(tmem, tmem + 128u, desc_kmajor(s.base + 2 * kPanelBytes), false);
    }
    ptx::umma_commit(s.bars + 8);
    if (!ok) wait_drain(s.bars, 0, ab, kStatusDrain);
  }
  __syncwarp();
  const bool done = wait_bounded_warp(s.bars + 8, 0, ab, kStatusSelftest);
  ptx::tc_fence_after();
  if (done && !*s.abort_flag) read_back(tmem, c, 128);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 0) ptx::tmem_dealloc(tmem, 256);
}

// out[i] = pack4_e4m3(in[4i], in[4i+1], in[4i+2], in[4i+3]).
__global__ void pack_e4m3_kernel(const float* in, uint32_t* out, int n_words) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n_words) out[i] = ptx::pack4_e4m3(in[4 * i], in[4 * i + 1], in[4 * i + 2], in[4 * i + 3]);
}

// One warp waits on a barrier that never completes, with a 20 ms limit.
__global__ void wait_timeout_kernel(uint32_t* status, uint32_t* out) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t flag;
  const uint32_t b = ptx::smem_u32(&bar);
  if (threadIdx.x == 0) {
    ptx::mbar_init(b, 1);
    flag = 0u;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  const AbortCtx ab{&flag, status};
  const bool ok = wait_bounded(b, 0, ab, kStatusSelftest, 20000000ull);
  if (threadIdx.x == 0) out[0] = ok ? 1u : 0u;
}

}  // namespace
}  // namespace fa

extern "C" {

// Returns 0 on success, 1 on bad arguments, 3 on a CUDA error. `status` is a
// device word that receives status bits of failed waits.
int fa_selftest_gemm_qk(const void* a, const void* b, float* c, int K, int bf16,
                        uint32_t* status, void* stream) {
  if (!a || !b || !c || !status || (K != 64 && K != 128)) return 1;
  CUtensorMap ta, tb;
  if (!fa::encode_2d(&ta, a, bf16 != 0, K, 128) || !fa::encode_2d(&tb, b, bf16 != 0, K, 128)) return 3;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  (void)cudaGetLastError();
  auto launch = [&](auto kern) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, fa::kSmemBytes) !=
        cudaSuccess)
      return 3;
    kern<<<1, 128, fa::kSmemBytes, st>>>(ta, tb, c, status);
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
  };
  if (K == 64) return bf16 ? launch(fa::gemm_qk_kernel<64, true>) : launch(fa::gemm_qk_kernel<64, false>);
  return bf16 ? launch(fa::gemm_qk_kernel<128, true>) : launch(fa::gemm_qk_kernel<128, false>);
}

int fa_selftest_gemm_pv(const void* a, const void* b, float* c, int N, int bf16, int variant,
                        uint32_t* status, void* stream) {
  if (!a || !b || !c || !status || (N != 64 && N != 128) || (variant != 0 && variant != 1)) return 1;
  CUtensorMap tb;
  if (!fa::encode_2d(&tb, b, bf16 != 0, N, 128)) return 3;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  (void)cudaGetLastError();
  const uint16_t* a16 = static_cast<const uint16_t*>(a);
  auto launch = [&](auto kern) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, fa::kSmemBytes) !=
        cudaSuccess)
      return 3;
    kern<<<1, 128, fa::kSmemBytes, st>>>(a16, tb, c, variant, status);
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
  };
  if (N == 64) return bf16 ? launch(fa::gemm_pv_kernel<64, true>) : launch(fa::gemm_pv_kernel<64, false>);
  return bf16 ? launch(fa::gemm_pv_kernel<128, true>) : launch(fa::gemm_pv_kernel<128, false>);
}

int fa_selftest_gemm_ts(const void* a, const void* b, float* c, int N, int bf16,
                        uint32_t* status, void* stream) {
  if (!a || !b || !c || !status || (N != 64 && N != 128)) return 1;
  CUtensorMap tb;
  if (!fa::encode_2d(&tb, b, bf16 != 0, N, 128)) return 3;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  (void)cudaGetLastError();
  const uint16_t* a16 = static_cast<const uint16_t*>(a);
  auto launch = [&](auto kern) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, fa::kSmemBytes) !=
        cudaSuccess)
      return 3;
    kern<<<1, 128, fa::kSmemBytes, st>>>(a16, tb, c, status);
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
  };
  if (N == 64) return bf16 ? launch(fa::gemm_ts_kernel<64, true>) : launch(fa::gemm_ts_kernel<64, false>);
  return bf16 ? launch(fa::gemm_ts_kernel<128, true>) : launch(fa::gemm_ts_kernel<128, false>);
}

// C[256][128] = A[256][128] * B[128][128]^T on a CTA pair (cta_group::2).
int fa_selftest_gemm_qk_pair(const void* a, const void* b, float* c, int bf16, int variant,
                             uint32_t* status, void* stream) {
  if (!a || !b || !c || !status) return 1;
  CUtensorMap ta, tb;
  if (!fa::encode_2d(&ta, a, bf16 != 0, 128, 256) || !fa::encode_2d(&tb, b, bf16 != 0, 128, 128, 64))
    return 3;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  (void)cudaGetLastError();
  auto launch = [&](auto kern) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, fa::kSmemBytes) !=
        cudaSuccess)
      return 3;
    kern<<<2, 128, fa::kSmemBytes, st>>>(ta, tb, c, status, variant);
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
  };
  return bf16 ? launch(fa::gemm_qk_pair_kernel<true>) : launch(fa::gemm_qk_pair_kernel<false>);
}

// C[256][128] = P[256][128] * V[128][128] on a CTA pair, P from TMEM.
int fa_selftest_gemm_pv_pair(const void* p, const void* v, float* c, int bf16, uint32_t* status,
                             void* stream) {
  if (!p || !v || !c || !status) return 1;
  CUtensorMap tv;
  if (!fa::encode_2d(&tv, v, bf16 != 0, 128, 128)) return 3;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  (void)cudaGetLastError();
  const uint16_t* p16 = static_cast<const uint16_t*>(p);
  auto launch = [&](auto kern) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, fa::kSmemBytes) !=
        cudaSuccess)
      return 3;
    kern<<<2, 128, fa::kSmemBytes, st>>>(p16, tv, c, status);
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
  };
  return bf16 ? launch(fa::gemm_pv_pair_kernel<true>) : launch(fa::gemm_pv_pair_kernel<false>);
}

// out[0] = 1 if the wait completed (it must not), 0 if it gave up.
int fa_selftest_wait_timeout(uint32_t* status, uint32_t* out, void* stream) {
  if (!status || !out) return 1;
  (void)cudaGetLastError();
  fa::wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status, out);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

}  // extern "C"

extern "C" {

// e4m3 C[128][128] = A[128][128] * B[128][128]^T (row-major byte matrices).
int fa_selftest_gemm_qk_fp8(const void* a, const void* b, float* c, uint32_t* status,
                            void* stream) {
  if (!a || !b || !c || !status) return 1;
  CUtensorMap ta, tb;
  if (!fa::encode_2d_u8(&ta, a, 128, 128) || !fa::encode_2d_u8(&tb, b, 128, 128)) return 3;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  (void)cudaGetLastError();
  if (cudaFuncSetAttribute(fa::gemm_qk_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           fa::kSmemBytes) != cudaSuccess)
    return 3;
  fa::gemm_qk_fp8_kernel<<<1, 128, fa::kSmemBytes, st>>>(ta, tb, c, status);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

// e4m3 C[128][128] = A[128][128] * Bt[128][128]^T with A taken from TMEM.
int fa_selftest_gemm_ts_fp8(const void* a, const void* bt, float* c, uint32_t* status,
                            void* stream) {
  if (!a || !bt || !c || !status) return 1;
  CUtensorMap tb;
  if (!fa::encode_2d_u8(&tb, bt, 128, 128)) return 3;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  (void)cudaGetLastError();
  if (cudaFuncSetAttribute(fa::gemm_ts_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           fa::kSmemBytes) != cudaSuccess)
    return 3;
  fa::gemm_ts_fp8_kernel<<<1, 128, fa::kSmemBytes, st>>>(static_cast<const uint32_t*>(a), tb, c,
                                                          status);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

// Packs n_words groups of four floats into e4m3 codes with the kernel's packer.
int fa_selftest_pack_e4m3(const float* in, uint32_t* out, int n_words, void* stream) {
  if (!in || !out || n_words <= 0) return 1;
  (void)cudaGetLastError();
  fa::pack_e4m3_kernel<<<(n_words + 127) / 128, 128, 0, static_cast<cudaStream_t>(stream)>>>(
      in, out, n_words);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

}  // extern "C"
