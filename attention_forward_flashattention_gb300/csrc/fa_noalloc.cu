// fa_fwd_noalloc: the attention forward for callers that cannot allocate
// device memory. See include/fa.h for the contract.
//
// fa_fwd keeps its status word (the scratch its kernel writes when a bounded
// wait gives up) in device memory it allocates on its first call on a device.
// This entry point runs the one-CTA forward kernel (whose results fa_fwd's
// kernels all reproduce bit for bit) with that scratch taken from a
// statically sized device array of this library instead, so no call ever
// allocates: no cudaMalloc, no cudaFree, no allocating library routine.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "fa_kernel.cuh"

namespace {

// Scratch of the allocation-free entry point: word 0 is the status word of
// the launch in flight. Every device that loads this library holds these
// 256 bytes until the process exits; all calls share them.
constexpr int kNoAllocScratchWords = 64;
constexpr int kStatusWordsPerLaunch = 1;  // independent of B, H, N, d
static_assert(kStatusWordsPerLaunch <= kNoAllocScratchWords, "scratch maximum");
static __device__ __align__(256) uint32_t g_noalloc_scratch[kNoAllocScratchWords];

constexpr int kMaxDevices = 64;

struct NoAllocDevice {
  bool ready = false;
  bool arch_ok = false;
  int sm_count = 0;
  uint32_t* scratch = nullptr;  // device address of g_noalloc_scratch
};

std::mutex g_mu;
NoAllocDevice g_dev[kMaxDevices];

// Per-device set-up, done by the first call on each device with that device
// current: architecture check and the device address of the scratch array
// (the array's name is only a host-side stand-in in host code).
fa_status device_setup(NoAllocDevice** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  NoAllocDevice& st = g_dev[dev];
  if (!st.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return FA_ERR_CUDA;
    st.arch_ok = (major == 10 && minor == 3);
    st.sm_count = sms;
    if (st.arch_ok) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
        return FA_ERR_CUDA;
      st.scratch = static_cast<uint32_t*>(p);
    }
    st.ready = true;
  }
  if (!st.arch_ok) return FA_ERR_ARCH;
  *out = &st;
  return FA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

namespace fa {

// Called by fa_check after it synchronised its stream: reads word 0 of the
// scratch (the status word of the allocation-free launches) and clears it.
// With calls in flight on other streams the word may belong to any of them.
fa_status noalloc_take_status(int dev, bool* timed_out) {
  *timed_out = false;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  uint32_t* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    scratch = g_dev[dev].ready ? g_dev[dev].scratch : nullptr;
  }
  if (scratch == nullptr) return FA_OK;  // the entry point was not used on this device
  uint32_t word = 0;
  if (cudaMemcpy(&word, scratch, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return FA_ERR_CUDA;
  if (word != 0) {
    if (cudaMemset(scratch, 0, sizeof(word)) != cudaSuccess) return FA_ERR_CUDA;
    *timed_out = true;
  }
  return FA_OK;
}

}  // namespace fa

extern "C" fa_status fa_fwd_noalloc(const void* q, const void* k, const void* v, void* o,
                                    float* lse, int B, int H, int N, int d, int causal,
                                    float scale, fa_dtype dtype, void* stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_INVALID_ARG;
  if (!(std::isfinite(scale) && scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_FP16 && dtype != FA_DTYPE_BF16) return FA_ERR_INVALID_ARG;
  // Sizes: the scratch need is one status word whatever the problem, so the
  // limits are the kernel's own, checked by the same function as fa_fwd's.
  const fa_status sz = fa::check_sizes(B, H, N, d);
  if (sz != FA_OK) return sz;
  const long long BH = static_cast<long long>(B) * H;

  NoAllocDevice* st = nullptr;
  const fa_status ds = device_setup(&st);
  if (ds != FA_OK) return ds;

  const bool bf16 = dtype == FA_DTYPE_BF16;
  const fa_strides c = fa::contiguous_strides(H, N, d);
  const fa_strides strides[4] = {c, c, c, c};
  CUtensorMap maps[4];  // same tensor maps, unit plan and kernels as fa_fwd
  if (!fa::encode_fwd_maps(maps, q, k, v, o, strides, bf16, B, H, N, d)) return FA_ERR_CUDA;

  fa::FwdArgs a{};
  a.lse = lse;
  a.status = st->scratch;
  a.scale_log2 = scale * 1.4426950408889634f;
  int grid = 0;
  fa::plan_fwd(d, N, H, BH, st->sm_count, &a, &grid);

  (void)cudaGetLastError();
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The scratch keeps the previous call's contents: the status word must start
  // at zero for this launch.
  if (cudaMemsetAsync(st->scratch, 0, kStatusWordsPerLaunch * sizeof(uint32_t), s) != cudaSuccess)
    return FA_ERR_CUDA;
  const cudaError_t e = fa::launch_fwd(d, bf16, causal != 0, maps, a, grid, s);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
