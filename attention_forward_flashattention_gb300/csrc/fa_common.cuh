// Device-side building blocks shared by the attention kernel and the PTX
// self-test kernels: shared-memory tile layout, bounded mbarrier waits,
// swizzled row stores, and the two tcgen05.mma sequences (S = Q K^T and
// O += P V).
//
// Operand layout (the fix of the SW128 pitfall in "Flash Attention CUDA
// Kernel: 56 to 986 TFLOPS on B300, G4", V14 "pitfall two"): every 16-bit
// tile of 128 rows is held as panels of 128 rows x 128 bytes (64 elements);
// a d = 128 tile is two panels 16 KB apart. TMA writes each panel with
// 128-byte swizzling, which is the tcgen05 K-major SW128 canonical layout:
// 8-row x 128-byte atoms, stride 1024 bytes between 8-row groups. A K step of
// 16 elements advances the descriptor start by 32 bytes inside a panel and
// jumps to the next panel every 64 elements.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "ptx.cuh"

namespace fa {

// Rows of a Q / K / V / O tile and keys of a KV tile.
constexpr int kTileRows = 128;
// One swizzle panel: 128 rows x 128 bytes.
constexpr int kPanelBytes = 128 * 128;
// A wait that makes no progress for this long is treated as a deadlock.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// Status word bits (ORed into the device status word by a failed wait).
enum StatusBits : uint32_t {
  kStatusProducer = 1u,
  kStatusMma = 2u,
  kStatusSoftmax = 4u,
  kStatusEpilogue = 8u,
  kStatusDrain = 16u,
  kStatusSelftest = 32u,
};

struct AbortCtx {
  volatile uint32_t* flag;  // shared memory: set once any role gives up
  uint32_t* status;         // global memory: the device status word
};

// Waits for phase `parity` of `bar`. Returns false if the CTA is aborting, or
// after kWaitLimitNs without progress (then it raises the abort flag and
// records `code` in the status word).
// Each try_wait suspends the thread for at most this long (it wakes as soon as
// the phase completes); between attempts the abort flag and the limit are
// checked.
constexpr uint32_t kSleepHintNs = 100000u;

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const AbortCtx& ab,
                                             uint32_t code, uint64_t limit_ns = kWaitLimitNs) {
  if (ptx::mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (;;) {
    if (ptx::mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
    if (*ab.flag) return false;
    if (ptx::globaltimer_ns() - t0 > limit_ns) {
      *ab.flag = 1u;
      atomicOr(ab.status, code);
      return false;
    }
  }
}

// Spinning variant for the single-thread roles (TMA producer, MMA issuer):
// one poller costs little, and a test of a completed phase returns fastest.
__device__ __forceinline__ bool wait_spin(uint32_t bar, uint32_t parity, const AbortCtx& ab,
                                          uint32_t code) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0u) {
      if (*ab.flag) return false;
      if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
        *ab.flag = 1u;
        atomicOr(ab.status, code);
        return false;
      }
    }
  }
}

// Warp-uniform spinning wait for a role run by a whole warp (every lane
// polls; the warp leaves the loop together, so it stays converged).
__device__ __forceinline__ bool wait_spin_warp(uint32_t bar, uint32_t parity, const AbortCtx& ab,
                                               uint32_t code) {
  if (__all_sync(0xffffffffu, ptx::mbar_try_wait(bar, parity))) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (__all_sync(0xffffffffu, ptx::mbar_try_wait(bar, parity))) return true;
    if ((it & 63u) == 0u) {
      const bool late = ptx::globaltimer_ns() - t0 > kWaitLimitNs;
      const bool stop = *ab.flag != 0u || late;
      if (__any_sync(0xffffffffu, stop)) {
        if (__any_sync(0xffffffffu, late)) {
          *ab.flag = 1u;
          atomicOr(ab.status, code);
        }
        return false;
      }
    }
  }
}

// Same, ignoring the abort flag: used to drain work already in flight
// (TMA loads, MMAs) before a CTA exits.
__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity, const AbortCtx& ab,
                                           uint32_t code) {
  const uint64_t t0 = ptx::globaltimer_ns();
  for (;;) {
    if (ptx::mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
    if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
      *ab.flag = 1u;
      atomicOr(ab.status, code);
      return false;
    }
  }
}

// Cluster-scope variant for barriers that receive arrivals or transaction
// bytes from the peer CTA of a pair (sleeping, or spinning for the
// single-thread roles).
template <bool kSleep>
__device__ __forceinline__ bool wait_cluster(uint32_t bar, uint32_t parity, const AbortCtx& ab,
                                             uint32_t code) {
  auto test = [&] {
    return kSleep ? ptx::mbar_try_wait_cluster(bar, parity, kSleepHintNs)
                  : ptx::mbar_test_cluster(bar, parity);
  };
  if (test()) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (test()) return true;
    if (kSleep || (it & 63u) == 0u) {
      if (*ab.flag) return false;
      if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
        *ab.flag = 1u;
        atomicOr(ab.status, code);
        return false;
      }
    }
  }
}

// Warp-uniform cluster-scope wait (every lane polls, the warp leaves together).
__device__ __forceinline__ bool wait_cluster_warp(uint32_t bar, uint32_t parity,
                                                  const AbortCtx& ab, uint32_t code) {
  if (__all_sync(0xffffffffu, ptx::mbar_test_cluster(bar, parity))) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (__all_sync(0xffffffffu, ptx::mbar_test_cluster(bar, parity))) return true;
    if ((it & 63u) == 0u) {
      const bool late = ptx::globaltimer_ns() - t0 > kWaitLimitNs;
      const bool stop = *ab.flag != 0u || late;
      if (__any_sync(0xffffffffu, stop)) {
        if (__any_sync(0xffffffffu, late)) {
          *ab.flag = 1u;
          atomicOr(ab.status, code);
        }
        return false;
      }
    }
  }
}

// Warp-uniform variant: every lane polls; the warp proceeds only if all
// lanes saw the phase complete.
__device__ __forceinline__ bool wait_bounded_warp(uint32_t bar, uint32_t parity,
                                                  const AbortCtx& ab, uint32_t code) {
  const bool ok = wait_bounded(bar, parity, ab, code);
  return __all_sync(0xffffffffu, ok) != 0;
}

// SM clock of a launch, measured while it runs: thread 0 of each CTA takes
// clock64 (SM cycles) and %globaltimer (ns) when the CTA starts and adds the
// elapsed amounts, and a count of one, to clk[0], clk[1], clk[2] when it ends.
// The host's cycles / ns is then the clock the CTAs ran at, averaged over CTAs
// weighted by their run time (a power-capped board runs below its maximum).
// The start values wait in shared memory (`slot`, 16 bytes, 8-byte aligned),
// so no register stays live across the kernel's roles.
__device__ __forceinline__ void clock_begin(uint64_t* slot) {
  slot[0] = ptx::globaltimer_ns();
  slot[1] = static_cast<uint64_t>(clock64());
}

__device__ __forceinline__ void clock_end(unsigned long long* clk, const uint64_t* slot) {
  const long long c = clock64();
  const uint64_t g = ptx::globaltimer_ns();
  atomicAdd(clk + 0, static_cast<unsigned long long>(c - static_cast<long long>(slot[1])));
  atomicAdd(clk + 1, static_cast<unsigned long long>(g - slot[0]));
  atomicAdd(clk + 2, 1ull);
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  uint32_t u;
  if constexpr (BF16) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    __builtin_memcpy(&u, &h, 4);
  } else {
    const __half2 h = __floats2half2_rn(lo, hi);
    __builtin_memcpy(&u, &h, 4);
  }
  return u;
}

// Writes row r (64 packed 16-bit pairs = 128 elements) of a two-panel SW128
// tile: elements 0-63 go to panel 0, 64-127 to panel 1; 16-byte chunk q of a
// row lands at chunk q ^ (r % 8). Eight consecutive rows cover all 32 banks.
__device__ __forceinline__ void store_row128_sw128(uint32_t tile, int r, const uint32_t (&pk)[64]) {
  const uint32_t row = tile + static_cast<uint32_t>(r) * 128u;
  const uint32_t x = static_cast<uint32_t>(r & 7);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      ptx::st_shared_v4(row + h * kPanelBytes + ((static_cast<uint32_t>(q) ^ x) << 4),
                        pk[32 * h + 4 * q], pk[32 * h + 4 * q + 1], pk[32 * h + 4 * q + 2],
                        pk[32 * h + 4 * q + 3]);
    }
  }
}

// Writes one 128-byte row (32 words: 128 8-bit elements) as row r of a
// one-panel SW128 tile.
__device__ __forceinline__ void store_row_panel_sw128(uint32_t tile, int r,
                                                      const uint32_t (&pk)[32]) {
  const uint32_t row = tile + static_cast<uint32_t>(r) * 128u;
  const uint32_t x = static_cast<uint32_t>(r & 7);
#pragma unroll
  for (int q = 0; q < 8; ++q)
    ptx::st_shared_v4(row + ((static_cast<uint32_t>(q) ^ x) << 4), pk[4 * q], pk[4 * q + 1],
                      pk[4 * q + 2], pk[4 * q + 3]);
}

// Shared-memory descriptor of a K-major SW128 tile (8-row groups 1024 B apart).
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t saddr) {
  return ptx::sdesc_sw128(saddr, 16, 1024);
}
// Shared-memory descriptor of V as an MN-major B operand: 8-key groups 1024 B
// apart (SBO), 64-column panels 16 KB apart (LBO).
__device__ __forceinline__ uint64_t desc_v(uint32_t saddr) {
  return ptx::sdesc_sw128(saddr, kPanelBytes, 1024);
}
// A descriptor advanced by `bytes` (the start address field holds addr >> 4;
// shared addresses stay below 2^18, so the field never carries).
__device__ __forceinline__ uint64_t desc_add(uint64_t desc, uint32_t bytes) {
  return desc + static_cast<uint64_t>(bytes >> 4);
}

// S[tmem: 128 lanes x 128 cols] = Q[128 x D] * K[128 x D]^T, both K-major,
// from precomputed base descriptors (a K step of 16 is +32 B inside a panel,
// the next panel every 4 steps).
template <int D, bool BF16, bool kElect = false>
__device__ __forceinline__ void issue_qk_desc(uint32_t d_tmem, uint64_t dq, uint64_t dk) {
  constexpr uint32_t id = ptx::idesc_f16(BF16, false, 128, 128);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    if constexpr (kElect) ptx::umma_f16_ss_elect(d_tmem, dq, dk, id, kk > 0 ? 1u : 0u);
    else ptx::umma_f16_ss(d_tmem, dq, dk, id, kk > 0 ? 1u : 0u);
    // next K step: +32 B inside a panel, or on to the next panel
    const uint32_t step = ((kk & 3) == 3) ? static_cast<uint32_t>(kPanelBytes - 96) : 32u;
    dq = desc_add(dq, step);
    dk = desc_add(dk, step);
    asm volatile("" : "+l"(dq), "+l"(dk));  // advance in place: two live descriptors
  }
}

template <int D, bool BF16, bool kElect = false>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t sQ, uint32_t sK) {
  issue_qk_desc<D, BF16, kElect>(d_tmem, desc_kmajor(sQ), desc_kmajor(sK));
}

// O[tmem: 128 lanes x D cols] (+)= P[128 x 128] * V[128 x D]. P is K-major
// (two panels of 64 keys); V is stored as loaded, [key][d], i.e. MN-major for
// the B operand: 8-key groups 1024 bytes apart (SBO), 64-column panels
// 16 KB apart (LBO); a K step of 16 keys advances 2048 bytes.
template <int D, bool BF16>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t sP, uint32_t sV, bool accumulate,
                                         uint32_t lbo = kPanelBytes, uint32_t sbo = 1024) {
  constexpr uint32_t id = ptx::idesc_f16(BF16, true, 128, D);
#pragma unroll 1
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t aoff = static_cast<uint32_t>((kk >> 2) * kPanelBytes + (kk & 3) * 32);
    const uint32_t boff = static_cast<uint32_t>(kk * 2048);
    ptx::umma_f16_ss(d_tmem, ptx::sdesc_sw128(sP + aoff, 16, 1024),
                     ptx::sdesc_sw128(sV + boff, lbo, sbo), id,
                     (accumulate || kk > 0) ? 1u : 0u);
  }
}

// O[tmem] (+)= P[tmem] * V[smem]: the P operand comes from tensor memory
// (128 lanes x 64 columns holding 128 packed 16-bit keys), V as in issue_pv.
template <int D, bool BF16, bool kElect = false>
__device__ __forceinline__ void issue_pv_ts_desc(uint32_t d_tmem, uint32_t p_tmem, uint64_t dv,
                                                 bool accumulate) {
  constexpr uint32_t id = ptx::idesc_f16(BF16, true, 128, D);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t acc = (accumulate || kk > 0) ? 1u : 0u;
    if constexpr (kElect) ptx::umma_f16_ts_elect(d_tmem, p_tmem + 8u * kk, dv, id, acc);
    else ptx::umma_f16_ts(d_tmem, p_tmem + 8u * kk, dv, id, acc);
    dv = desc_add(dv, 2048u);
    asm volatile("" : "+l"(dv));
  }
}

template <int D, bool BF16>
__device__ __forceinline__ void issue_pv_ts(uint32_t d_tmem, uint32_t p_tmem, uint32_t sV,
                                            bool accumulate) {
  issue_pv_ts_desc<D, BF16>(d_tmem, p_tmem, desc_v(sV), accumulate);
}

// 8-bit (e4m3) products for head dimension 128: a 128-element row is one
// 128-byte SW128 panel, and one MMA covers K = 32 (+32 bytes per step).
// S[tmem] = Q[128 x 128] K[128 x 128]^T, both K-major in shared memory.
template <bool kElect = false>
__device__ __forceinline__ void issue_qk_fp8(uint32_t d_tmem, uint64_t dq, uint64_t dk) {
  constexpr uint32_t id = ptx::idesc_f8(128, 128);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    if constexpr (kElect) ptx::umma_f8_ss_elect(d_tmem, dq, dk, id, kk > 0 ? 1u : 0u);
    else ptx::umma_f8_ss(d_tmem, dq, dk, id, kk > 0 ? 1u : 0u);
    dq = desc_add(dq, 32u);
    dk = desc_add(dk, 32u);
    asm volatile("" : "+l"(dq), "+l"(dk));
  }
}
// O[tmem] (+)= P[tmem: 128 lanes x 32 columns, four keys per column] V with V
// given transposed, V^T[128 columns of O][128 keys], K-major in shared memory.
template <bool kElect = false>
__device__ __forceinline__ void issue_pv_fp8(uint32_t d_tmem, uint32_t p_tmem, uint64_t dvt,
                                             bool accumulate) {
  constexpr uint32_t id = ptx::idesc_f8(128, 128);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    const uint32_t acc = (accumulate || kk > 0) ? 1u : 0u;
    if constexpr (kElect) ptx::umma_f8_ts_elect(d_tmem, p_tmem + 8u * kk, dvt, id, acc);
    else ptx::umma_f8_ts(d_tmem, p_tmem + 8u * kk, dvt, id, acc);
    dvt = desc_add(dvt, 32u);
    asm volatile("" : "+l"(dvt));
  }
}

// O[tmem] (+)= P V with both operands in shared memory: P[128 x 128 keys]
// (e4m3, K-major SW128, one panel) and V^T[128 columns of O][128 keys].
template <bool kElect = false>
__device__ __forceinline__ void issue_pv_fp8_ss(uint32_t d_tmem, uint64_t dp, uint64_t dvt,
                                                bool accumulate) {
  constexpr uint32_t id = ptx::idesc_f8(128, 128);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    const uint32_t acc = (accumulate || kk > 0) ? 1u : 0u;
    if constexpr (kElect) ptx::umma_f8_ss_elect(d_tmem, dp, dvt, id, acc);
    else ptx::umma_f8_ss(d_tmem, dp, dvt, id, acc);
    dp = desc_add(dp, 32u);
    dvt = desc_add(dvt, 32u);
    asm volatile("" : "+l"(dp), "+l"(dvt));
  }
}

// Pair MMAs for head dimension 128 (M = 256: 128 query rows in each CTA).
// S = Q K^T: each CTA holds its 128 Q rows (two 16 KB panels) and 64 of the
// 128 keys (two 8 KB panels of 64 rows); the pair's S has all 128 keys.
template <bool BF16>
__device__ __forceinline__ void issue_qk_pair(uint32_t d_tmem, uint64_t dq, uint64_t dk) {
  constexpr uint32_t id = ptx::idesc_f16(BF16, false, 256, 128);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    ptx::umma_f16_ss_pair(d_tmem, dq, dk, id, kk > 0 ? 1u : 0u);
    const bool next_panel = (kk & 3) == 3;
    dq = desc_add(dq, next_panel ? static_cast<uint32_t>(kPanelBytes - 96) : 32u);
    dk = desc_add(dk, next_panel ? static_cast<uint32_t>(kPanelBytes / 2 - 96) : 32u);
    asm volatile("" : "+l"(dq), "+l"(dk));
  }
}

// O += P V: P (each CTA's 128 rows) from TMEM; each CTA holds 64 of the 128
// columns of V (one 128-key x 64-column panel, MN-major).
template <bool BF16>
__device__ __forceinline__ void issue_pv_ts_pair(uint32_t d_tmem, uint32_t p_tmem, uint64_t dv,
                                                 bool accumulate) {
  constexpr uint32_t id = ptx::idesc_f16(BF16, true, 256, 128);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    ptx::umma_f16_ts_pair(d_tmem, p_tmem + 8u * kk, dv, id, (accumulate || kk > 0) ? 1u : 0u);
    dv = desc_add(dv, 2048u);
    asm volatile("" : "+l"(dv));
  }
}

}  // namespace fa
