// C ABI of the attention forward library (declared in include/fa.h):
// argument checks, per-device state, TMA descriptor encoding and launch.
//
// TMA descriptors follow the host-side construction of "TMA + Warp
// Specialization" (CUDA book ch. 17, section 17.3): cuTensorMapEncodeTiled on
// the host, passed by value as __grid_constant__ kernel parameters. Unlike
// that chapter's single {d, Bc} box, each tile here is fetched as 64-element
// (128-byte) wide panels, the layout fix of the B300 walkthrough (V14, second
// pitfall), so that what TMA writes is the tcgen05 K-major SW128 layout.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "fa_bwd.cuh"
#include "fa_kernel.cuh"
#include "fa_dispatch.h"
#include "fa_pair.cuh"

namespace fa {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  bool arch_ok = false;
  int sm_count = 0;
  // 256 bytes allocated on first use and kept until exit: word 0 is the status
  // word; bytes 64-87 the SM clock record (three uint64) of the launches since
  // the last fa_sm_clock_read
  uint32_t* status = nullptr;
};

constexpr int kClockRecordWord = 16;  // uint32 index of the clock record

unsigned long long* clock_record(const DeviceState& st) {
  return reinterpret_cast<unsigned long long*>(st.status + kClockRecordWord);
}

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
EncodeTiledFn g_encode = nullptr;

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  return g_encode;
}

// Device facts for the current device; allocates its status word on first use.
fa_status current_device(int* dev_out, DeviceState** st_out, bool need_status) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return FA_ERR_CUDA;
    st.arch_ok = (major == 10 && minor == 3);
    st.sm_count = sms;
    st.ready = true;
  }
  if (!st.arch_ok) return FA_ERR_ARCH;
  if (need_status && st.status == nullptr) {
    uint32_t* p = nullptr;
    if (cudaMalloc(&p, 256) != cudaSuccess) return FA_ERR_CUDA;
    if (cudaMemset(p, 0, 256) != cudaSuccess) {
      cudaFree(p);
      return FA_ERR_CUDA;
    }
    st.status = p;
  }
  *dev_out = dev;
  *st_out = &st;
  return FA_OK;
}

// One [B][H][N][d] 16-bit tensor with element strides `st` (d stride 1) as a
// 4-D map {d, N, H, B}; box = one 64-element x box_rows panel of one (b, h),
// 128-byte swizzle. Rows past N read as zero.
bool encode_qkv(CUtensorMap* m, const void* ptr, const fa_strides& st, bool bf16, int B, int H,
                int N, int d, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(st.n) * 2u,
                                 static_cast<cuuint64_t>(st.h) * 2u,
                                 static_cast<cuuint64_t>(st.b) * 2u};
  const cuuint32_t box[4] = {64u, static_cast<cuuint32_t>(box_rows), 1u, 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
             const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A 4-D byte tensor (e4m3 codes) {dims[0] (contiguous), dims[1], dims[2],
// dims[3]} with byte strides for dims 1..3; box = 128 x 128 x 1 x 1 bytes,
// 128-byte swizzle. Elements past dims[0] / dims[1] read as zero.
bool encode_bytes4(CUtensorMap* m, const void* ptr, const cuuint64_t (&dims)[4],
                   const cuuint64_t (&strides)[3], cuuint32_t box_rows = 128u) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint32_t box[4] = {128u, box_rows, 1u, 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

__global__ void clock_probe_kernel(uint64_t* out, long long cycles) {
  if (threadIdx.x != 0) return;
  const uint64_t g0 = ptx::globaltimer_ns();
  const long long c0 = clock64();
  long long c = c0;
  while (c - c0 < cycles) c = clock64();
  const uint64_t g1 = ptx::globaltimer_ns();
  out[0] = static_cast<uint64_t>(c - c0);
  out[1] = g1 - g0;
}

}  // namespace

fa_status check_sizes(int B, int H, int N, int d) {
  if (B <= 0 || H <= 0 || N <= 0) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const long long BH = static_cast<long long>(B) * H;
  if (BH > 0x7FFFFFFFLL) return FA_ERR_UNSUPPORTED;
  // unit count BH * ceil(N / 256) and row index bh * N + i stay in int range
  const long long units = BH * ((static_cast<long long>(N) + 255) / 256);
  if (units > 0x7FFFFFFFLL) return FA_ERR_UNSUPPORTED;
  if (N > (1 << 30)) return FA_ERR_UNSUPPORTED;  // tile row coordinates stay in int range
  return FA_OK;
}

int fwd_smem_bytes(int d) {
  return d == 64 ? Layout<64>::kSmemBytes : Layout<128>::kSmemBytes;
}

fa_strides contiguous_strides(int H, int N, int d) {
  fa_strides s;
  s.n = d;
  s.h = static_cast<long long>(N) * d;
  s.b = s.h * H;
  return s;
}

fa_status check_strides(const fa_strides* s, int d) {
  // Multiples of 8 elements (16 bytes: TMA rows and 16-byte output stores),
  // rows at least d apart; byte strides inside the tensor-map range.
  for (int t = 0; t < 4; ++t) {
    for (const long long v : {s[t].b, s[t].h, s[t].n})
      if (v <= 0 || (v & 7) != 0) return FA_ERR_INVALID_ARG;
    if (s[t].n < d) return FA_ERR_INVALID_ARG;
  }
  for (int t = 0; t < 4; ++t)
    for (const long long v : {s[t].b, s[t].h, s[t].n})
      if (v >= (1LL << 38)) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

bool encode_fwd_maps(CUtensorMap* maps, const void* q, const void* k, const void* v,
                     const void* o, const fa_strides* s, bool bf16, int B, int H, int N, int d,
                     int k_box_rows) {
  return encode_qkv(&maps[0], q, s[0], bf16, B, H, N, d, 128) &&
         encode_qkv(&maps[1], k, s[1], bf16, B, H, N, d,
                    k_box_rows > 0 ? k_box_rows : fwd_k_box_rows(d)) &&
         encode_qkv(&maps[2], v, s[2], bf16, B, H, N, d, 128) &&
         encode_qkv(&maps[3], o, s[3], bf16, B, H, N, d, kFwdOutBoxRows);
}

void plan_fwd(int d, int N, int H, long long BH, int sm_count, FwdArgs* a, int* grid) {
  const int rows = fwd_unit_rows(d);
  a->N = N;
  a->H = H;
  a->BH = static_cast<int>(BH);
  a->n_mblk = (N + rows - 1) / rows;
  a->n_units = static_cast<int>(BH * a->n_mblk);
  a->n_kv = (N + 127) / 128;
  *grid = d == 64 ? fwd_grid_d64(a->n_units, sm_count) : fwd_grid_d128(a->n_units, sm_count);
}

cudaError_t launch_fwd(int d, bool bf16, bool causal, const CUtensorMap* maps, const FwdArgs& a,
                       int grid, cudaStream_t stream) {
  return d == 64 ? launch_fwd_d64(bf16, causal, maps, a, grid, stream)
                 : launch_fwd_d128(bf16, causal, maps, a, grid, stream);
}

}  // namespace fa

extern "C" {

namespace {


// Which forward kernel a call runs: fa_fwd and fa_fwd_strided choose (kAuto),
// fa_fwd_pair asks for the CTA-pair kernel.
enum class FwdChoice { kAuto, kPair };

// fa_fwd, fa_fwd_strided and fa_fwd_pair: checks, tensor maps, plan, launch
// (the pair kernel takes head dimension 128 only).
fa_status fwd_call(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                   int N, int d, const fa_strides* s, int causal, float scale, fa_dtype dtype,
                   void* stream, FwdChoice choice = FwdChoice::kAuto) {
  const bool want_pair = choice == FwdChoice::kPair;
  if (!q || !k || !v || !o || !lse || !s) return FA_ERR_INVALID_ARG;
  if (!fa::aligned16(q) || !fa::aligned16(k) || !fa::aligned16(v) || !fa::aligned16(o) ||
      !fa::aligned16(lse))
    return FA_ERR_INVALID_ARG;
  if (!(std::isfinite(scale) && scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_FP16 && dtype != FA_DTYPE_BF16) return FA_ERR_INVALID_ARG;
  const fa_status sz = fa::check_sizes(B, H, N, d);
  if (sz != FA_OK) return sz;
  if (want_pair && d != 128) return FA_ERR_UNSUPPORTED;
  const fa_status ss = fa::check_strides(s, d);
  if (ss != FA_OK) return ss;

  int dev = 0;
  fa::DeviceState* st = nullptr;
  const fa_status ds = fa::current_device(&dev, &st, true);
  if (ds != FA_OK) return ds;

  const bool bf16 = dtype == FA_DTYPE_BF16;
  const long long BH = static_cast<long long>(B) * H;
  const bool pair = want_pair || fa::fwd_prefers_pair(d, causal != 0, BH, N, st->sm_count);
  CUtensorMap maps[4];
  if (!fa::encode_fwd_maps(maps, q, k, v, o, s, bf16, B, H, N, d, pair ? 64 : 0))
    return FA_ERR_CUDA;

  fa::FwdArgs a{};
  a.lse = lse;
  a.status = st->status;
  a.clk = fa::clock_record(*st);
  a.scale_log2 = scale * 1.4426950408889634f;
  int grid = 0;
  fa::plan_fwd(d, N, H, BH, st->sm_count, &a, &grid);
  if (pair) {  // units of 512 rows, two CTAs per unit
    a.n_mblk = (N + 511) / 512;
    a.n_units = static_cast<int>(BH * a.n_mblk);
    grid = fa::fwd_grid_pair(a.n_units, st->sm_count);
  }

  (void)cudaGetLastError();  // do not report an earlier, unrelated error as ours
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const cudaError_t e = pair ? fa::launch_fwd_pair(bf16, causal != 0, maps, a, grid, cs)
                             : fa::launch_fwd(d, bf16, causal != 0, maps, a, grid, cs);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int N, int d, int causal, float scale, fa_dtype dtype, void* stream) {
  if (B <= 0 || H <= 0 || N <= 0) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const fa_strides c = fa::contiguous_strides(H, N, d);
  const fa_strides s[4] = {c, c, c, c};
  return fwd_call(q, k, v, o, lse, B, H, N, d, s, causal, scale, dtype, stream);
}

fa_status fa_fwd_pair(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int H, int N, int d, int causal, float scale, fa_dtype dtype, void* stream) {
  if (B <= 0 || H <= 0 || N <= 0) return FA_ERR_INVALID_ARG;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  const fa_strides c = fa::contiguous_strides(H, N, d);
  const fa_strides s[4] = {c, c, c, c};
  return fwd_call(q, k, v, o, lse, B, H, N, d, s, causal, scale, dtype, stream,
                  FwdChoice::kPair);
}

fa_status fa_fwd_strided(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                         int H, int N, int d, const fa_strides* strides, int causal, float scale,
                         fa_dtype dtype, void* stream) {
  return fwd_call(q, k, v, o, lse, B, H, N, d, strides, causal, scale, dtype, stream);
}

namespace {

// The 8-bit forward of fa_fwd_fp8 (kAuto: the one-CTA kernel or, where it
// is faster, the CTA pair) and fa_fwd_fp8_pair (kPair).
fa_status fwd_fp8_call(const void* q, const void* k, const void* vt, void* o, float* lse, int B,
                       int H, int N, int d, int ldv, float q_scale, const float* k_scales,
                       float v_scale, int causal, float scale, void* stream, FwdChoice choice) {
  if (!q || !k || !vt || !o || !lse || !k_scales) return FA_ERR_INVALID_ARG;
  if (!fa::aligned16(q) || !fa::aligned16(k) || !fa::aligned16(vt) || !fa::aligned16(o) ||
      !fa::aligned16(lse) || (reinterpret_cast<uintptr_t>(k_scales) & 3u) != 0)
    return FA_ERR_INVALID_ARG;
  for (const float x : {scale, q_scale, v_scale})
    if (!(std::isfinite(x) && x > 0.f)) return FA_ERR_INVALID_ARG;
  const fa_status sz = fa::check_sizes(B, H, N, d);
  if (sz != FA_OK) return sz;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  if (ldv < N || (ldv & 15) != 0) return FA_ERR_INVALID_ARG;

  int dev = 0;
  fa::DeviceState* st = nullptr;
  const fa_status ds = fa::current_device(&dev, &st, true);
  if (ds != FA_OK) return ds;

  const long long BH = static_cast<long long>(B) * H;
  const bool pair = choice == FwdChoice::kPair ||
                    fa::fwd_fp8_prefers_pair(causal != 0, BH, N, st->sm_count);
  const cuuint64_t n = static_cast<cuuint64_t>(N), h = static_cast<cuuint64_t>(H),
                   b = static_cast<cuuint64_t>(B), lv = static_cast<cuuint64_t>(ldv);
  CUtensorMap maps[4];
  const cuuint64_t qk_dims[4] = {128u, n, h, b};
  const cuuint64_t qk_strides[3] = {128u, 128u * n, 128u * n * h};
  const cuuint64_t vt_dims[4] = {n, 128u, h, b};
  const cuuint64_t vt_strides[3] = {lv, 128u * lv, 128u * lv * h};
  const cuuint32_t half_rows = pair ? 64u : 128u;  // the pair loads K / V^T halves
  if (!fa::encode_bytes4(&maps[0], q, qk_dims, qk_strides) ||
      !fa::encode_bytes4(&maps[1], k, qk_dims, qk_strides, half_rows) ||
      !fa::encode_bytes4(&maps[2], vt, vt_dims, vt_strides, half_rows) ||
      !fa::encode_qkv(&maps[3], o, fa::contiguous_strides(H, N, d), true, B, H, N, d,
                      fa::kFwdOutBoxRows))
    return FA_ERR_CUDA;

  fa::FwdArgs a{};
  a.lse = lse;
  a.status = st->status;
  a.scale_log2 = scale * q_scale * 1.4426950408889634f;
  a.k_scales = k_scales;
  a.v_scale = v_scale;
  a.clk = fa::clock_record(*st);
  int grid = 0;
  fa::plan_fwd(d, N, H, BH, st->sm_count, &a, &grid);
  if (pair) {  // units of 512 rows, two CTAs per unit
    a.n_mblk = (N + 511) / 512;
    a.n_units = static_cast<int>(BH * a.n_mblk);
    grid = fa::fwd_grid_pair(a.n_units, st->sm_count);
  }

  (void)cudaGetLastError();
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const cudaError_t e = pair ? fa::launch_fwd_pair_fp8(causal != 0, maps, a, grid, cs)
                             : fa::launch_fwd_fp8(causal != 0, maps, a, grid, cs);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

fa_status fa_fwd_fp8(const void* q, const void* k, const void* vt, void* o, float* lse, int B,
                     int H, int N, int d, int ldv, float q_scale, const float* k_scales,
                     float v_scale, int causal, float scale, void* stream) {
  return fwd_fp8_call(q, k, vt, o, lse, B, H, N, d, ldv, q_scale, k_scales, v_scale, causal,
                      scale, stream, FwdChoice::kAuto);
}

fa_status fa_fwd_fp8_pair(const void* q, const void* k, const void* vt, void* o, float* lse,
                          int B, int H, int N, int d, int ldv, float q_scale,
                          const float* k_scales, float v_scale, int causal, float scale,
                          void* stream) {
  return fwd_fp8_call(q, k, vt, o, lse, B, H, N, d, ldv, q_scale, k_scales, v_scale, causal,
                      scale, stream, FwdChoice::kPair);
}

fa_status fa_bwd_workspace_size(int B, int H, int N, int d, size_t* bytes) {
  if (!bytes) return FA_ERR_INVALID_ARG;
  const fa_status sz = fa::check_sizes(B, H, N, d);
  if (sz != FA_OK) return sz;
  const long long n_t = (static_cast<long long>(N) + 127) / 128;
  *bytes = static_cast<size_t>(2LL * B * H * n_t * 128 * 4);
  return FA_OK;
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                 const float* lse, void* dq, void* dk, void* dv, void* workspace, int B, int H,
                 int N, int d, int causal, float scale, fa_dtype dtype, void* stream) {
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !workspace)
    return FA_ERR_INVALID_ARG;
  for (const void* p : {q, k, v, o, dout, static_cast<const void*>(lse),
                        static_cast<const void*>(dq), static_cast<const void*>(dk),
                        static_cast<const void*>(dv), static_cast<const void*>(workspace)})
    if (!fa::aligned16(p)) return FA_ERR_INVALID_ARG;
  if (!(std::isfinite(scale) && scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_FP16 && dtype != FA_DTYPE_BF16) return FA_ERR_INVALID_ARG;
  const fa_status sz = fa::check_sizes(B, H, N, d);
  if (sz != FA_OK) return sz;
  // the backward's units are 128-row tiles: their count must stay in int range
  if (static_cast<long long>(B) * H * ((static_cast<long long>(N) + 127) / 128) > 0x7FFFFFFFLL)
    return FA_ERR_UNSUPPORTED;

  int dev = 0;
  fa::DeviceState* st = nullptr;
  const fa_status ds = fa::current_device(&dev, &st, true);
  if (ds != FA_OK) return ds;

  const bool bf16 = dtype == FA_DTYPE_BF16;
  const fa_strides c = fa::contiguous_strides(H, N, d);
  CUtensorMap maps[4];
  if (!fa::encode_qkv(&maps[0], q, c, bf16, B, H, N, d, 128) ||
      !fa::encode_qkv(&maps[1], k, c, bf16, B, H, N, d, 128) ||
      !fa::encode_qkv(&maps[2], v, c, bf16, B, H, N, d, 128) ||
      !fa::encode_qkv(&maps[3], dout, c, bf16, B, H, N, d, 128))
    return FA_ERR_CUDA;

  fa::BwdArgs a{};
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.N = N;
  a.H = H;
  a.BH = B * H;
  a.n_t = (N + 127) / 128;
  a.n_units = a.BH * a.n_t;
  const size_t vec = static_cast<size_t>(a.BH) * a.n_t * 128;
  float* ws = static_cast<float*>(workspace);
  a.lse2 = ws;
  a.delta = ws + vec;
  a.status = st->status;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.scale = scale;
  a.clk = fa::clock_record(*st);
  const int grid = a.n_units < st->sm_count ? a.n_units : st->sm_count;

  (void)cudaGetLastError();
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = d == 64 ? fa::launch_bwd_d64(bf16, causal != 0, maps, a, o, dout, lse, grid, s)
                                : fa::launch_bwd_d128(bf16, causal != 0, maps, a, o, dout, lse, grid, s);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_check(void* stream) {
  int dev = 0;
  fa::DeviceState* st = nullptr;
  const fa_status ds = fa::current_device(&dev, &st, false);
  if (ds != FA_OK) return ds;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  // fa_fwd_noalloc keeps its status word in the library's static scratch
  bool noalloc_timeout = false;
  const fa_status ns = fa::noalloc_take_status(dev, &noalloc_timeout);
  if (ns != FA_OK) return ns;
  uint32_t word = 0;
  if (st->status != nullptr) {  // (null: nothing launched through fa_fwd & co. yet)
    if (cudaMemcpy(&word, st->status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
      return FA_ERR_CUDA;
    if (word != 0 && cudaMemset(st->status, 0, sizeof(word)) != cudaSuccess) return FA_ERR_CUDA;
  }
  return (word != 0 || noalloc_timeout) ? FA_ERR_TIMEOUT : FA_OK;
}

fa_status fa_sm_clock_read(void* stream, double* sm_mhz, unsigned long long* ctas) {
  if (!sm_mhz) return FA_ERR_INVALID_ARG;
  int dev = 0;
  fa::DeviceState* st = nullptr;
  const fa_status ds = fa::current_device(&dev, &st, false);
  if (ds != FA_OK) return ds;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  *sm_mhz = 0.0;
  if (ctas) *ctas = 0;
  if (st->status == nullptr) return FA_OK;  // nothing launched on this device yet
  unsigned long long rec[3] = {0, 0, 0};
  unsigned long long* dev_rec = fa::clock_record(*st);
  if (cudaMemcpy(rec, dev_rec, sizeof(rec), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(dev_rec, 0, sizeof(rec)) != cudaSuccess)
    return FA_ERR_CUDA;
  if (rec[1] > 0) *sm_mhz = 1000.0 * static_cast<double>(rec[0]) / static_cast<double>(rec[1]);
  if (ctas) *ctas = rec[2];
  return FA_OK;
}

fa_status fa_query_launch(int B, int H, int N, int d, int causal, int* grid, int* threads,
                          int* smem_bytes, int* units, int* cluster) {
  const fa_status sz = fa::check_sizes(B, H, N, d);
  if (sz != FA_OK) return sz;
  int dev = 0;
  fa::DeviceState* st = nullptr;
  const fa_status ds = fa::current_device(&dev, &st, false);
  if (ds != FA_OK) return ds;
  const long long BH = static_cast<long long>(B) * H;
  fa::FwdArgs a{};
  int g = 0;
  fa::plan_fwd(d, N, H, BH, st->sm_count, &a, &g);
  const bool pair = fa::fwd_prefers_pair(d, causal != 0, BH, N, st->sm_count);
  if (pair) {
    a.n_units = static_cast<int>(BH * ((N + 511) / 512));
    g = fa::fwd_grid_pair(a.n_units, st->sm_count);
  }
  if (grid) *grid = g;
  if (threads) *threads = fa::kFwdThreads;
  if (smem_bytes) *smem_bytes = pair ? fa::fwd_smem_bytes_pair() : fa::fwd_smem_bytes(d);
  if (units) *units = a.n_units;
  if (cluster) *cluster = pair ? 2 : 1;
  return FA_OK;
}

fa_status fa_sm_clock_probe(uint64_t* out, long long cycles, void* stream) {
  if (!out || cycles <= 0 || cycles > 8000000000LL) return FA_ERR_INVALID_ARG;
  int dev = 0;
  fa::DeviceState* st = nullptr;
  const fa_status ds = fa::current_device(&dev, &st, false);
  if (ds != FA_OK) return ds;
  (void)cudaGetLastError();
  fa::clock_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(out, cycles);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_ARCH: return "FA_ERR_ARCH";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
  }
  return "FA_ERR_UNKNOWN";
}

int fa_version(void) { return 100; }

}  // extern "C"
