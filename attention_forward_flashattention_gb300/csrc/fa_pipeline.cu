// fa_fwd_host: the attention forward on host buffers. The (b, h) slices are
// independent, so the heads are cut into chunks and each chunk's copy in,
// forward and copy out run on three streams: while chunk c computes, chunk
// c+1 is copied in and chunk c-1 copied out, and the call costs about the
// larger of the transfer and compute times instead of their sum.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxChunks = 9;

struct Streams {
  bool ready = false;
  cudaStream_t in = nullptr;    // host -> device copies
  cudaStream_t comp = nullptr;  // forward launches
  cudaStream_t out = nullptr;   // device -> host copies
};

std::mutex g_mu;
Streams g_streams[kMaxDevices];

// The device's three streams, created on first use and kept until exit.
fa_status device_streams(int dev, Streams** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  Streams& s = g_streams[dev];
  if (!s.ready) {
    cudaStream_t t[3] = {nullptr, nullptr, nullptr};
    for (int i = 0; i < 3; ++i) {
      if (cudaStreamCreateWithFlags(&t[i], cudaStreamNonBlocking) != cudaSuccess) {
        for (int j = 0; j < i; ++j) cudaStreamDestroy(t[j]);
        return FA_ERR_CUDA;
      }
    }
    s.in = t[0];
    s.comp = t[1];
    s.out = t[2];
    s.ready = true;
  }
  *out = &s;
  return FA_OK;
}

size_t align16(size_t x) { return (x + 15u) & ~static_cast<size_t>(15u); }

// Workspace: Q, K, V, O of the whole problem, then the per-chunk LSE blocks,
// each starting on a 16-byte boundary (fa_fwd's alignment rule).
fa_status workspace_bytes(long long BH, int N, int d, size_t* bytes) {
  const size_t elems = static_cast<size_t>(BH) * static_cast<size_t>(N) * static_cast<size_t>(d);
  *bytes = 4 * elems * 2 + static_cast<size_t>(BH) * static_cast<size_t>(N) * 4 + 16 * kMaxChunks;
  return FA_OK;
}

// Chunk count n: as many as keep one persistent wave of 256-row units busy
// in each, at most kMaxChunks - 1, at most one per head. The host link (about
// 200 GB/s each way) is about as slow as the forward or slower on every
// workload of interest, so a chunk's forward hides under the next chunk's
// copy; what is exposed is the first chunk's copy-in and the last chunk's
// forward and copy-out. So the call uses n + 1 chunks whose first and last
// are half the size of the others.
int pick_chunks(long long BH, int N, int sm_count) {
  const long long units = BH * ((static_cast<long long>(N) + 255) / 256);
  long long n = units / (sm_count > 0 ? sm_count : 1);
  if (n < 1) n = 1;
  if (n > kMaxChunks - 1) n = kMaxChunks - 1;
  if (n > BH) n = BH;
  return static_cast<int>(n);
}

// First head of chunk c of m: weights 1, 2, ..., 2, 1 (a single chunk when m
// is 1); edges are nondecreasing from 0 to BH, and a chunk may be empty.
long long chunk_edge(long long BH, int m, int c) {
  if (m == 1) return BH * c;
  const long long w = (c == 0) ? 0 : (c == m ? 2LL * (m - 1) : 2LL * c - 1);
  return BH * w / (2LL * (m - 1));
}

}  // namespace

extern "C" {

fa_status fa_fwd_host_workspace_size(int B, int H, int N, int d, size_t* bytes) {
  if (!bytes || B <= 0 || H <= 0 || N <= 0) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  return workspace_bytes(static_cast<long long>(B) * H, N, d, bytes);
}

fa_status fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int H, int N, int d, int causal, float scale, fa_dtype dtype,
                      void* workspace, size_t workspace_size, void* stream) {
  if (!q || !k || !v || !o || !lse || !workspace) return FA_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || N <= 0) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (dtype != FA_DTYPE_FP16 && dtype != FA_DTYPE_BF16) return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return FA_ERR_INVALID_ARG;
  if (!(std::isfinite(scale) && scale > 0.f)) return FA_ERR_INVALID_ARG;
  const long long BH = static_cast<long long>(B) * H;
  size_t need = 0;
  workspace_bytes(BH, N, d, &need);
  if (workspace_size < need) return FA_ERR_INVALID_ARG;
  // the per-chunk forwards see B = 1, H = heads of the chunk: check the whole
  // problem once here, with the forward's own rules, before enqueuing anything
  fa_status st = fa_query_launch(B, H, N, d, causal, nullptr, nullptr, nullptr, nullptr, nullptr);
  if (st != FA_OK) return st;

  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FA_ERR_CUDA;
  Streams* s = nullptr;
  if ((st = device_streams(dev, &s)) != FA_OK) return st;

  const int n = pick_chunks(BH, N, sms);
  const int m = n > 1 ? n + 1 : 1;
  const size_t head_elems = static_cast<size_t>(N) * static_cast<size_t>(d);
  const size_t total = static_cast<size_t>(BH) * head_elems;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint16_t* dev_t[4];
  for (int t = 0; t < 4; ++t) dev_t[t] = reinterpret_cast<uint16_t*>(ws) + t * total;
  uint8_t* lse_base = ws + 4 * total * 2;
  const uint16_t* host_in[3] = {static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(k),
                                static_cast<const uint16_t*>(v)};
  cudaStream_t caller = static_cast<cudaStream_t>(stream);

  // events: fork, two per chunk, three joins (destroyed at the end of the
  // call; CUDA releases each once it has completed)
  cudaEvent_t ev[1 + 2 * kMaxChunks + 3];
  int nev = 0;
  auto event = [&]() -> cudaEvent_t {
    cudaEvent_t e = nullptr;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    ev[nev++] = e;
    return e;
  };
  (void)cudaGetLastError();  // do not report an earlier, unrelated error as ours
  // fork: the three streams start after the caller's prior work
  cudaEvent_t fork = event();
  bool ok = fork && cudaEventRecord(fork, caller) == cudaSuccess &&
            cudaStreamWaitEvent(s->in, fork, 0) == cudaSuccess &&
            cudaStreamWaitEvent(s->comp, fork, 0) == cudaSuccess &&
            cudaStreamWaitEvent(s->out, fork, 0) == cudaSuccess;
  fa_status fwd_status = FA_OK;
  size_t lse_off = 0;
  for (int c = 0; ok && c < m; ++c) {
    const long long h0 = chunk_edge(BH, m, c), h1 = chunk_edge(BH, m, c + 1);
    const long long nh = h1 - h0;
    if (nh == 0) continue;
    const size_t off = static_cast<size_t>(h0) * head_elems;
    const size_t cnt = static_cast<size_t>(nh) * head_elems;
    const size_t lrows = static_cast<size_t>(nh) * static_cast<size_t>(N);
    float* dlse = reinterpret_cast<float*>(lse_base + lse_off);
    lse_off = align16(lse_off + lrows * 4);
    cudaEvent_t in_done = event(), fwd_done = event();
    ok = in_done && fwd_done;
    for (int t = 0; ok && t < 3; ++t)
      ok = cudaMemcpyAsync(dev_t[t] + off, host_in[t] + off, cnt * 2, cudaMemcpyHostToDevice,
                           s->in) == cudaSuccess;
    ok = ok && cudaEventRecord(in_done, s->in) == cudaSuccess &&
         cudaStreamWaitEvent(s->comp, in_done, 0) == cudaSuccess;
    if (ok) {
      fwd_status = fa_fwd(dev_t[0] + off, dev_t[1] + off, dev_t[2] + off, dev_t[3] + off, dlse, 1,
                          static_cast<int>(nh), N, d, causal, scale, dtype, s->comp);
      ok = fwd_status == FA_OK;
    }
    ok = ok && cudaEventRecord(fwd_done, s->comp) == cudaSuccess &&
         cudaStreamWaitEvent(s->out, fwd_done, 0) == cudaSuccess &&
         cudaMemcpyAsync(static_cast<uint16_t*>(o) + off, dev_t[3] + off, cnt * 2,
                         cudaMemcpyDeviceToHost, s->out) == cudaSuccess &&
         cudaMemcpyAsync(lse + static_cast<size_t>(h0) * N, dlse, lrows * 4,
                         cudaMemcpyDeviceToHost, s->out) == cudaSuccess;
  }
  // join: the caller's stream continues once all three streams are done
  // (also after an error, so that the workspace outlives whatever was enqueued)
  bool joined = true;
  for (cudaStream_t t : {s->in, s->comp, s->out}) {
    cudaEvent_t j = event();
    joined = joined && j && cudaEventRecord(j, t) == cudaSuccess &&
             cudaStreamWaitEvent(caller, j, 0) == cudaSuccess;
  }
  for (int i = 0; i < nev; ++i) cudaEventDestroy(ev[i]);
  if (!joined) return FA_ERR_CUDA;
  if (fwd_status != FA_OK) return fwd_status;
  return ok ? FA_OK : FA_ERR_CUDA;
}

}  // extern "C"
