// Fused attention backward for sm_103a: dQ, dK, dV of the forward. The
// backward recomputes the scores instead of storing them ("TCA 51%, MFU below
// 8%", section "MFU is always a little below TCA"); the softmax weights come
// back from the forward's row logsumexp, which is why the forward emits it.
//
// With P_ij = exp(scale q_i.k_j - LSE_i), D_i = dO_i . O_i:
//   dV_j = sum_i P_ij dO_i            dP_ij = dO_i . v_j
//   dS_ij = P_ij (dP_ij - D_i)        dQ_i = scale sum_j dS_ij k_j
//   dK_j = scale sum_i dS_ij q_i
//
// Three launches, no atomics, deterministic:
//   1. bwd_prep_kernel: D_i and LSE_i * log2(e) into a workspace padded to
//      128-row tiles (padding rows: D = 0, lse2 = +inf, so their weights are 0).
//   2. dK/dV kernel: one unit = one 128-key tile of one head; it loops over
//      the 128-row query tiles that see it. Per query tile i (TMEM, lane = key):
//        S^T = K Q_i^T, dP^T = V dO_i^T           (both operands in smem)
//        P^T = 2^(c S^T - lse2_i)  -> 16 bit over the S^T columns
//        dV += P^T dO_i                           (A = P^T from TMEM)
//        dS^T = P^T (dP^T - D_i)   -> 16 bit over the dP^T columns
//        dK += dS^T Q_i                           (A = dS^T from TMEM)
//      dK and dV accumulate in TMEM; the epilogue scales dK and stores both.
//   3. dQ kernel: one unit = one 128-row query tile; it loops over the key
//      tiles it sees. Per key tile j (lane = query row):
//        S = Q K_j^T (into one of two S buffers), dP = dO V_j^T
//        P = 2^(c S - lse2), dS = P (dP - D)  -> 16 bit over the S columns
//        dQ += dS K_j                             (A = dS from TMEM)
//      dP is released as soon as it is read, so dP of tile j+1 is computed
//      while dS of tile j is formed. Two warps issue the MMAs: one S and dQ
//      (S(j+2) after dQ(j) has read its buffer), one dP.
//
// Roles (16 warps): warp 0 TMA producer (lane 0); warp 1 TMEM owner and, in
// the d = 128 dK/dV kernel, MMA issuer (the whole warp, one elected lane
// issuing); the dQ kernel and the d = 64 dK/dV kernel issue their MMAs as two
// chains on warps 2 and 3 instead; warpgroups 1 and 2 the
// element-wise softmax gradient (one thread per TMEM lane; warpgroup 1 takes
// columns 0-63 of each 128-column scratch tile, warpgroup 2 columns 64-127,
// and each packs its 16-bit result over the first 32 of its own columns);
// warpgroup 3 the epilogue. Every wait is bounded as in the forward (abort
// flag, status bits, drain before TMEM is freed).
#pragma once

#include <cuda.h>

#include <type_traits>

#include "fa.h"
#include "fa_common.cuh"

namespace fa {

struct BwdArgs {
  void* dq;               // [BH][N][D] outputs, 16-bit
  void* dk;
  void* dv;
  const float* lse2;      // workspace [BH][n_t * 128]: LSE * log2(e), +inf past N
  const float* delta;     // workspace [BH][n_t * 128]: D = dO . O, 0 past N
  uint32_t* status;
  int N;
  int H;
  int BH;
  int n_t;                // 128-row tiles per head: ceil(N / 128)
  int n_units;            // BH * n_t
  float scale_log2;       // scale * log2(e)
  float scale;
  unsigned long long* clk;  // optional [3]: SM clock record of the launch (clock_end), or null
};

constexpr int kBwdThreads = 512;
// setmaxnreg split: the 512-thread launch gives 128 registers per thread
// (65536 / 512); the four warpgroups move to 72 / 192 / 192 / 56, which sum
// to the same 4 x 128.
constexpr uint32_t kBwdRegsLaunch = 128;
constexpr uint32_t kBwdRegsWG0 = 72, kBwdRegsElem = 192, kBwdRegsEpi = 56;
static_assert(kBwdRegsWG0 + 2 * kBwdRegsElem + kBwdRegsEpi == 4 * kBwdRegsLaunch,
              "register split");
static_assert(kBwdRegsLaunch == (65536 / kBwdThreads) / 8 * 8, "launch allocation");

// Shared memory and TMEM of one kernel (KEYS: dK/dV, else dQ).
template <int D, bool KEYS>
struct BwdLayout {
  static constexpr int kPanels = D / 64;
  static constexpr int kTileBytes = kPanels * kPanelBytes;  // a 128-row tile of Q, K, V, dO
  static constexpr int kOffFix = 0;                         // two fixed tiles (K, V or Q, dO)
  static constexpr int kOffRing = 2 * kTileBytes;
  // dK/dV: one ring of stages, each a Q tile, a dO tile and their lse2 / D
  static constexpr int kStages = (D == 128) ? 2 : 4;
  static constexpr int kVecBytes = 2 * 128 * 4;
  static constexpr int kStageBytes = 2 * kTileBytes + kVecBytes;
  // dQ: a K ring (a K tile lives from S to dQ) and a V ring (read by dP only)
  static constexpr int kKSlots = (D == 128) ? 3 : 4;
  static constexpr int kVSlots = (D == 128) ? 2 : 3;
  static constexpr int kOffK = kOffRing;
  static constexpr int kOffV = kOffK + kKSlots * kTileBytes;
  static constexpr int kRingBytes =
      KEYS ? kStages * kStageBytes : (kKSlots + kVSlots) * kTileBytes;
  static constexpr int kOffBar = kOffRing + kRingBytes;
  static constexpr int kSmemBytes = kOffBar + 512 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kStageBytes % 1024 == 0, "stages keep tiles 1024-byte aligned");
  static_assert(kOffBar % 8 == 0, "barrier block alignment");
  // TMEM columns: 128-column fp32 scratch tiles and the accumulators. A
  // 16-bit operand written over a scratch tile sits in columns 0-31 (rows'
  // elements 0-63) and 64-95 (elements 64-127).
  static constexpr uint32_t kColA = 0;    // S^T, then 16-bit P^T (dkdv) / S, then dS (dq, even tiles)
  static constexpr uint32_t kColB = 128;  // dP^T, then 16-bit dS^T (dkdv) / dP (dq)
  static constexpr uint32_t kColAcc0 = 256;      // dV (dkdv) / dQ (dq)
  static constexpr uint32_t kColAcc1 = 256 + D;  // dK (dkdv)
  static constexpr uint32_t kColA1 = 384;        // S (dq) / S^T (dkdv, d=64), odd tiles
  // Two S buffers (tile c in A or A1 by parity): always in the dQ kernel; in
  // the dK/dV kernel where the accumulators leave room (d = 64).
  static constexpr bool kDblS = !KEYS || D == 64;
  static_assert(!kDblS || (KEYS ? kColAcc1 : kColAcc0) + D <= kColA1, "TMEM columns");
};

enum BwdBar : int {
  kBbFixFull = 0,    // the unit's two fixed tiles landed
  kBbFixEmpty = 1,   // MMA: the unit's last use of the fixed tiles done
  kBbAFull = 2,      // MMA: scratch A (S^T / S of even tiles) ready
  kBbBFull = 3,      // MMA: scratch B (dP^T / dP) ready
  kBbPFull = 4,      // element-wise (8 warps): P^T in TMEM (dkdv) / dP read (dq)
  kBbDsFull = 5,     // element-wise (8 warps): dS^T / dS in TMEM
  kBbAccFull = 6,    // MMA: the unit's accumulators final
  kBbAccFree = 7,    // epilogue (4 warps): accumulators read
  kBbDrain = 8,      // MMA: all tcgen05 ops done
  kBbA1Full = 9,     // MMA: S of odd tiles ready (dq)
  kBbRing = 10,      // dkdv: [stages] full, [stages] empty;
                     // dq: K [slots] full, K empty, V [slots] full, V empty
  kBbDrainB = 30,    // dkdv: chain B's MMAs all done
};
constexpr int kBwdSlotTmem = 480;
constexpr int kBwdSlotAbort = 484;
constexpr int kBwdSlotClock = 488;  // clock stamp (16 bytes)

// D_i and LSE_i * log2(e) into the tile-padded workspace. Eight lanes per
// padded row: lane p of a row reads its 16-byte chunks p, p + 8, ..., so a
// warp's loads cover four rows contiguously, and a shuffle sums the eight
// partial dot products. Grid-stride over rows * 8 threads (rows is a multiple
// of 128, so every warp runs the same iterations and all its lanes shuffle).
template <int D, bool BF16>
__global__ void bwd_prep_kernel(const void* o, const void* dout, const float* lse, float* lse2,
                                float* delta, int N, int n_t, long long rows) {
  constexpr int kLanes = 8, kChunks = D / 8;  // 16-byte chunks per row
  const long long total = rows * kLanes;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
       t += stride) {
    const long long g = t / kLanes;  // padded row
    const int part = static_cast<int>(t % kLanes);
    const long long bh = g / (static_cast<long long>(n_t) * 128);
    const int i = static_cast<int>(g - bh * n_t * 128);
    const size_t row = static_cast<size_t>(bh) * N + i;
    float acc = 0.f;
    if (i < N) {
      const uint4* po = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(o) + row * D);
      const uint4* pd =
          reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(dout) + row * D);
#pragma unroll
      for (int c = part; c < kChunks; c += kLanes) {
        const uint4 ua = po[c], ub = pd[c];
        const uint32_t wa[4] = {ua.x, ua.y, ua.z, ua.w}, wb[4] = {ub.x, ub.y, ub.z, ub.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float a0, a1, b0, b1;
          if constexpr (BF16) {
            a0 = __uint_as_float(wa[e] << 16);
            a1 = __uint_as_float(wa[e] & 0xFFFF0000u);
            b0 = __uint_as_float(wb[e] << 16);
            b1 = __uint_as_float(wb[e] & 0xFFFF0000u);
          } else {
            const __half2 ha = *reinterpret_cast<const __half2*>(&wa[e]);
            const __half2 hb = *reinterpret_cast<const __half2*>(&wb[e]);
            const float2 fa = __half22float2(ha), fb = __half22float2(hb);
            a0 = fa.x;
            a1 = fa.y;
            b0 = fb.x;
            b1 = fb.y;
          }
          acc = fmaf(a0, b0, acc);
          acc = fmaf(a1, b1, acc);
        }
      }
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    acc += __shfl_xor_sync(0xffffffffu, acc, 4);
    if (part == 0) {
      // padding rows: D = 0, lse2 = +inf, so their weights are exactly 0
      delta[g] = i < N ? acc : 0.f;
      lse2[g] = i < N ? lse[row] * 1.4426950408889634f : INFINITY;
    }
  }
}

// Unit order: causal problems longest first, odd rounds reversed (as the
// forward); otherwise head-major. A dkdv unit of key tile t sees the query
// tiles t.. n_t-1 (causal), a dq unit of query tile t the key tiles 0..t.
template <bool CAUSAL, bool KEYS>
__device__ __forceinline__ bool bwd_next_unit(int& round, const BwdArgs& a, int& bh, int& t) {
  const int G = static_cast<int>(gridDim.x);
  for (;;) {
    const long long base = static_cast<long long>(round) * G;
    if (base >= a.n_units) return false;
    int c = static_cast<int>(blockIdx.x);
    if (CAUSAL && (round & 1)) c = G - 1 - c;
    const long long u = base + c;
    ++round;
    if (u >= a.n_units) continue;
    if (CAUSAL) {
      const int lvl = static_cast<int>(u / a.BH);
      bh = static_cast<int>(u - static_cast<long long>(lvl) * a.BH);
      t = KEYS ? lvl : a.n_t - 1 - lvl;
    } else {
      bh = static_cast<int>(u / a.n_t);
      t = static_cast<int>(u - static_cast<long long>(bh) * a.n_t);
    }
    return true;
  }
}

// The streamed tiles of a unit: [first, last] (query tiles for dkdv, key tiles for dq).
template <bool CAUSAL, bool KEYS>
__device__ __forceinline__ void bwd_span(const BwdArgs& a, int t, int& first, int& last) {
  if (KEYS) {
    first = CAUSAL ? t : 0;
    last = a.n_t - 1;
  } else {
    first = 0;
    last = CAUSAL ? t : a.n_t - 1;
  }
}

// TMA producer (one thread). KEYS (dK/dV): fixed K, V; streamed Q, dO and the
// tile's lse2 / D vectors. Otherwise (dQ): fixed Q, dO; streamed K, V.
template <int D, bool CAUSAL, bool KEYS>
__device__ __forceinline__ void bwd_producer(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                             const CUtensorMap* tm_v, const CUtensorMap* tm_do,
                                             const BwdArgs& a, uint32_t sbase, uint32_t bars,
                                             const AbortCtx& ab) {
  using L = BwdLayout<D, KEYS>;
  constexpr int S = L::kStages;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  const CUtensorMap* fix0 = KEYS ? tm_k : tm_q;
  const CUtensorMap* fix1 = KEYS ? tm_v : tm_do;
  const CUtensorMap* str0 = KEYS ? tm_q : tm_k;
  const CUtensorMap* str1 = KEYS ? tm_do : tm_v;
  for (const CUtensorMap* m : {tm_q, tm_k, tm_v, tm_do}) ptx::prefetch_tmap(m);
  auto load_tile = [&](uint32_t dst, const CUtensorMap* tm, uint32_t b, int row, int hh, int bb) {
    for (int p = 0; p < L::kPanels; ++p)
      ptx::tma_load_4d(dst + p * kPanelBytes, tm, b, 64 * p, row, hh, bb);
  };
  constexpr int KS = L::kKSlots, VS = L::kVSlots;
  // dq rings: K full / empty, V full / empty barrier slots
  constexpr int kKFull = kBbRing, kKEmpty = kBbRing + KS;
  constexpr int kVFull = kBbRing + 2 * KS, kVEmpty = kBbRing + 2 * KS + VS;
  uint32_t ring = 0, kc = 0, vc = 0, units = 0;
  int round = 0, bh = 0, t = 0;
  bool ok = true;
  // one tile into ring slot `count % slots`, once its previous use is done
  auto ring_load = [&](int full, int empty, int slots, uint32_t count, uint32_t dst0,
                       const CUtensorMap* tm, int row, int hh, int bb) {
    const uint32_t sl = count % slots, ph = (count / slots) & 1u;
    if (!wait_spin(bar(empty + sl), ph ^ 1u, ab, kStatusProducer)) return false;
    ptx::mbar_arrive_expect_tx(bar(full + sl), L::kTileBytes);
    load_tile(dst0 + sl * L::kTileBytes, tm, bar(full + sl), row, hh, bb);
    return true;
  };
  while (ok && bwd_next_unit<CAUSAL, KEYS>(round, a, bh, t)) {
    int first, last;
    bwd_span<CAUSAL, KEYS>(a, t, first, last);
    const int hh = bh % a.H, bb = bh / a.H;
    if (!(ok = wait_spin(bar(kBbFixEmpty), (units & 1u) ^ 1u, ab, kStatusProducer))) break;
    ptx::mbar_arrive_expect_tx(bar(kBbFixFull), 2 * L::kTileBytes);
    load_tile(sbase + L::kOffFix, fix0, bar(kBbFixFull), 128 * t, hh, bb);
    load_tile(sbase + L::kOffFix + L::kTileBytes, fix1, bar(kBbFixFull), 128 * t, hh, bb);
    ++units;
    for (int st = first; st <= last && ok; ++st) {
      if constexpr (KEYS) {
        const uint32_t slot = ring % S, ph = (ring / S) & 1u;
        if (!(ok = wait_spin(bar(kBbRing + S + slot), ph ^ 1u, ab, kStatusProducer))) break;
        const uint32_t dst = sbase + L::kOffRing + slot * L::kStageBytes;
        ptx::mbar_arrive_expect_tx(bar(kBbRing + slot), 2 * L::kTileBytes + L::kVecBytes);
        load_tile(dst, str0, bar(kBbRing + slot), 128 * st, hh, bb);
        load_tile(dst + L::kTileBytes, str1, bar(kBbRing + slot), 128 * st, hh, bb);
        const size_t v0 = (static_cast<size_t>(bh) * a.n_t + st) * 128;
        ptx::bulk_load(dst + 2 * L::kTileBytes, a.lse2 + v0, 512, bar(kBbRing + slot));
        ptx::bulk_load(dst + 2 * L::kTileBytes + 512, a.delta + v0, 512, bar(kBbRing + slot));
        ++ring;
      } else {
        if (!(ok = ring_load(kKFull, kKEmpty, KS, kc, sbase + L::kOffK, str0, 128 * st, hh, bb)))
          break;
        ++kc;
        if (!(ok = ring_load(kVFull, kVEmpty, VS, vc, sbase + L::kOffV, str1, 128 * st, hh, bb)))
          break;
        ++vc;
      }
    }
  }
  if (!ok) {  // let the copies already issued land before the CTA exits
    auto drain = [&](int full, int slots, uint32_t count) {
      for (uint32_t sl = 0; sl < static_cast<uint32_t>(slots) && sl < count; ++sl) {
        const uint32_t lastp = count - 1 - ((count - 1 - sl) % slots);
        wait_drain(bar(full + sl), (lastp / slots) & 1u, ab, kStatusDrain);
      }
    };
    if constexpr (KEYS) {
      drain(kBbRing, S, ring);
    } else {
      drain(kKFull, KS, kc);
      drain(kVFull, VS, vc);
    }
    if (units > 0) wait_drain(bar(kBbFixFull), (units - 1) & 1u, ab, kStatusDrain);
  }
}

// C[tmem] (+)= A[tmem] B: A is a 16-bit operand written over a scratch tile
// (elements 0-63 in columns 0-31, 64-127 in columns 64-95, two per column),
// B a 128-row tile used MN-major (K = its rows).
template <int D, bool BF16>
__device__ __forceinline__ void bwd_issue_ts(uint32_t d_tmem, uint32_t a_tmem, uint32_t sB,
                                             bool accumulate) {
  constexpr uint32_t id = ptx::idesc_f16(BF16, true, 128, D);
  uint64_t db = desc_v(sB);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t acol = a_tmem + (kk < 4 ? 8u * kk : 64u + 8u * (kk - 4));
    ptx::umma_f16_ts_elect(d_tmem, acol, db, id, (accumulate || kk > 0) ? 1u : 0u);
    db = desc_add(db, 2048u);
    asm volatile("" : "+l"(db));
  }
}

// The MMA-issuing warp of the dK/dV kernel at d = 128 (order at the top of
// this file): one warp, so S^T(c+1) reaches the tensor core right after dV(c).
template <int D, bool BF16, bool CAUSAL, bool KEYS>
__device__ __forceinline__ void bwd_mma(const BwdArgs& a, uint32_t sbase, uint32_t bars,
                                        uint32_t tmem, const AbortCtx& ab) {
  using L = BwdLayout<D, KEYS>;
  constexpr int S = L::kStages;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  const uint32_t tA = tmem + L::kColA, tB = tmem + L::kColB;
  const uint32_t tAcc0 = tmem + L::kColAcc0, tAcc1 = tmem + L::kColAcc1;
  const uint32_t fix0 = sbase + L::kOffFix, fix1 = fix0 + L::kTileBytes;
  auto stage = [&](uint32_t r) { return sbase + L::kOffRing + (r % S) * L::kStageBytes; };
  auto ring_wait = [&](uint32_t r) {
    return wait_spin_warp(bar(kBbRing + r % S), (r / S) & 1u, ab, kStatusMma);
  };
  // The two scratch products of streamed tile r: S^T = K Q^T into tile c's S^T
  // buffer, dP^T = V dO^T into B (all operands K-major).
  constexpr bool kDbl = L::kDblS;
  auto sbuf = [&](uint32_t c) { return tmem + ((kDbl && (c & 1u)) ? L::kColA1 : L::kColA); };
  auto scratch_a = [&](uint32_t r, uint32_t c) {
    issue_qk<D, BF16, true>(sbuf(c), fix0, stage(r));
    ptx::umma_commit_elect(bar((kDbl && (c & 1u)) ? kBbA1Full : kBbAFull));
  };
  auto scratch_b = [&](uint32_t r) {
    issue_qk<D, BF16, true>(tB, fix1, stage(r) + L::kTileBytes);
    ptx::umma_commit_elect(bar(kBbBFull));
  };
  uint32_t ring = 0, units = 0, cnt = 0;
  int round = 0, bh = 0, t = 0;
  bool ok = true;
  while (ok && bwd_next_unit<CAUSAL, KEYS>(round, a, bh, t)) {
    int first, last;
    bwd_span<CAUSAL, KEYS>(a, t, first, last);
    const uint32_t n = static_cast<uint32_t>(last - first + 1);
    if (!(ok = wait_spin_warp(bar(kBbFixFull), units & 1u, ab, kStatusMma))) break;
    if (!(ok = ring_wait(ring))) break;
    ptx::tc_fence_after();
    scratch_a(ring, cnt);
    scratch_b(ring);
    if (kDbl && n > 1) {  // two S^T buffers: the next tile's S^T right away
      if (!(ok = ring_wait(ring + 1))) break;
      scratch_a(ring + 1, cnt + 1);
    }
    // ahead = how many tiles past the current one S^T is issued
    constexpr uint32_t ahead = kDbl ? 2u : 1u;
    for (uint32_t i = 0; i < n; ++i) {
      const uint32_t r = ring + i, c = cnt + i, ph = c & 1u;
      const bool acc = i > 0;
      // dV += P^T dO (P^T in TMEM over tile c's S^T columns; dO used MN-major)
      if (!(ok = wait_spin_warp(bar(kBbPFull), ph, ab, kStatusMma))) break;
      if (!acc && units > 0 &&
          !(ok = wait_spin_warp(bar(kBbAccFree), (units - 1) & 1u, ab, kStatusMma)))
        break;
      ptx::tc_fence_after();
      bwd_issue_ts<D, BF16>(tAcc0, sbuf(c), stage(r) + L::kTileBytes, acc);
      if (i + ahead < n) {  // S^T of a later tile into the buffer dV has just read
        if (!(ok = ring_wait(r + ahead))) break;
        scratch_a(r + ahead, c + ahead);
      }
      // dK += dS^T Q (dS^T in TMEM over the dP^T columns; Q used MN-major)
      if (!(ok = wait_spin_warp(bar(kBbDsFull), ph, ab, kStatusMma))) break;
      ptx::tc_fence_after();
      bwd_issue_ts<D, BF16>(tAcc1, tB, stage(r), acc);
      ptx::umma_commit_elect(bar(kBbRing + S + r % S));
      if (i + 1 < n) scratch_b(r + 1);  // stage r+1 was waited for with its S^T
    }
    if (!ok) break;
    ring += n;
    cnt += n;
    ptx::umma_commit_elect(bar(kBbAccFull));
    ptx::umma_commit_elect(bar(kBbFixEmpty));
    ++units;
  }
  ptx::umma_commit_elect(bar(kBbDrain));
  wait_drain(bar(kBbDrain), 0u, ab, kStatusDrain);
}

// At d = 64 (two S^T buffers) the dK/dV kernel's MMAs form two chains that
// share no TMEM columns, each issued in order by its own warp (on SM
// sub-partitions 2 and 3, away from the element-wise warps that share one
// with a busy issuer; at d = 128, where S^T(c+1) must follow dV(c) closely,
// a single issuer is faster):
//   chain A (warp 2): S^T(c) = K Q_c^T into tile c's S^T buffer, then
//                     dV += P^T(c) dO_c once P^T(c) is written over it;
//   chain B (warp 3): dP^T(c) = V dO_c^T into B, then dK += dS^T(c) Q_c
//                     once dS^T(c) is written over it.
// A streamed stage is free once both dV(c) and dK(c) are done, the fixed K, V
// once both chains' last products are, and the accumulators are final once
// both chains' last ones are: those barriers take one commit from each chain.
template <int D, bool BF16, bool CAUSAL, bool A>
__device__ __forceinline__ void bwd_mma_kv(const BwdArgs& a, uint32_t sbase, uint32_t bars,
                                           uint32_t tmem, const AbortCtx& ab) {
  using L = BwdLayout<D, true>;
  constexpr int S = L::kStages;
  constexpr bool kDbl = L::kDblS;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  const uint32_t tB = tmem + L::kColB;
  const uint32_t tAcc = tmem + (A ? L::kColAcc0 : L::kColAcc1);
  const uint32_t fix = sbase + L::kOffFix + (A ? 0 : L::kTileBytes);  // K (A) or V (B)
  auto stage = [&](uint32_t r) { return sbase + L::kOffRing + (r % S) * L::kStageBytes; };
  auto ring_wait = [&](uint32_t r) {
    return wait_spin_warp(bar(kBbRing + r % S), (r / S) & 1u, ab, kStatusMma);
  };
  auto sbuf = [&](uint32_t c) { return tmem + ((kDbl && (c & 1u)) ? L::kColA1 : L::kColA); };
  // the chain's scratch product of tile c (stage r): S^T = K Q^T or dP^T = V dO^T
  auto scratch = [&](uint32_t r, uint32_t c) {
    if constexpr (A) {
      issue_qk<D, BF16, true>(sbuf(c), fix, stage(r));
      ptx::umma_commit_elect(bar((kDbl && (c & 1u)) ? kBbA1Full : kBbAFull));
    } else {
      issue_qk<D, BF16, true>(tB, fix, stage(r) + L::kTileBytes);
      ptx::umma_commit_elect(bar(kBbBFull));
    }
  };
  // chain A issues S^T two tiles ahead where there are two S^T buffers
  constexpr uint32_t ahead = (A && kDbl) ? 2u : 1u;
  uint32_t ring = 0, units = 0, cnt = 0;
  int round = 0, bh = 0, t = 0;
  bool ok = true;
  while (ok && bwd_next_unit<CAUSAL, true>(round, a, bh, t)) {
    int first, last;
    bwd_span<CAUSAL, true>(a, t, first, last);
    const uint32_t n = static_cast<uint32_t>(last - first + 1);
    if (!(ok = wait_spin_warp(bar(kBbFixFull), units & 1u, ab, kStatusMma))) break;
    for (uint32_t k = 0; k < ahead && k < n && ok; ++k) {
      if (!(ok = ring_wait(ring + k))) break;
      ptx::tc_fence_after();
      scratch(ring + k, cnt + k);
    }
    for (uint32_t i = 0; i < n && ok; ++i) {
      const uint32_t r = ring + i, c = cnt + i, ph = c & 1u;
      // dV += P^T dO (chain A) or dK += dS^T Q (chain B), from TMEM over the
      // scratch columns; dO / Q used MN-major
      if (!(ok = wait_spin_warp(bar(A ? kBbPFull : kBbDsFull), ph, ab, kStatusMma))) break;
      if (i == 0 && units > 0 &&
          !(ok = wait_spin_warp(bar(kBbAccFree), (units - 1) & 1u, ab, kStatusMma)))
        break;
      ptx::tc_fence_after();
      if constexpr (A) bwd_issue_ts<D, BF16>(tAcc, sbuf(c), stage(r) + L::kTileBytes, i > 0);
      else bwd_issue_ts<D, BF16>(tAcc, tB, stage(r), i > 0);
      ptx::umma_commit_elect(bar(kBbRing + S + r % S));  // this chain's use of stage r done
      if (i + ahead < n) {  // the chain's next scratch product, after the one just read
        if (!(ok = ring_wait(r + ahead))) break;
        scratch(r + ahead, c + ahead);
      }
    }
    if (!ok) break;
    ring += n;
    cnt += n;
    ptx::umma_commit_elect(bar(kBbAccFull));
    ptx::umma_commit_elect(bar(kBbFixEmpty));
    ++units;
  }
  ptx::umma_commit_elect(bar(A ? kBbDrain : kBbDrainB));
  wait_drain(bar(A ? kBbDrain : kBbDrainB), 0u, ab, kStatusDrain);
}

// The dQ kernel's MMAs as two chains on their own warps (they share no TMEM
// columns): chain SQ (warp 2) issues S into the two S buffers and dQ += dS K
// from them (S(j+2) reuses a buffer after dQ(j) has read it, in order);
// chain P (warp 3) issues dP into B as soon as the element-wise role has read
// the previous one. Q, dO are released once both chains are done with them.
template <int D, bool BF16, bool CAUSAL, bool SQ>
__device__ __forceinline__ void bwd_mma_dq_chain(const BwdArgs& a, uint32_t sbase, uint32_t bars,
                                                 uint32_t tmem, const AbortCtx& ab) {
  using L = BwdLayout<D, false>;
  constexpr int KS = L::kKSlots, VS = L::kVSlots;
  constexpr int kKFull = kBbRing, kKEmpty = kBbRing + KS;
  constexpr int kVFull = kBbRing + 2 * KS, kVEmpty = kBbRing + 2 * KS + VS;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  const uint32_t tB = tmem + L::kColB, tAcc = tmem + L::kColAcc0;
  const uint32_t fixq = sbase + L::kOffFix, fixdo = fixq + L::kTileBytes;
  auto sbuf = [&](uint32_t c) { return tmem + ((c & 1u) ? L::kColA1 : L::kColA); };
  auto kslot = [&](uint32_t k) { return sbase + L::kOffK + (k % KS) * L::kTileBytes; };
  auto vslot = [&](uint32_t v) { return sbase + L::kOffV + (v % VS) * L::kTileBytes; };
  auto kwait = [&](uint32_t k) {
    return wait_spin_warp(bar(kKFull + k % KS), (k / KS) & 1u, ab, kStatusMma);
  };
  auto vwait = [&](uint32_t v) {
    return wait_spin_warp(bar(kVFull + v % VS), (v / VS) & 1u, ab, kStatusMma);
  };
  auto issue_s = [&](uint32_t c, uint32_t k) {
    issue_qk<D, BF16, true>(sbuf(c), fixq, kslot(k));
    ptx::umma_commit_elect(bar((c & 1u) ? kBbA1Full : kBbAFull));
  };
  auto issue_dp = [&](uint32_t v) {
    issue_qk<D, BF16, true>(tB, fixdo, vslot(v));
    ptx::umma_commit_elect(bar(kBbBFull));
    ptx::umma_commit_elect(bar(kVEmpty + v % VS));
  };
  uint32_t cnt = 0, kv = 0, units = 0;  // kv: K (chain SQ) or V (chain P) ring index
  int round = 0, bh = 0, t = 0;
  bool ok = true;
  while (ok && bwd_next_unit<CAUSAL, false>(round, a, bh, t)) {
    int first, last;
    bwd_span<CAUSAL, false>(a, t, first, last);
    const uint32_t n = static_cast<uint32_t>(last - first + 1);
    if (!(ok = wait_spin_warp(bar(kBbFixFull), units & 1u, ab, kStatusMma))) break;
    if constexpr (SQ) {
      for (uint32_t k = 0; k < 2 && k < n && ok; ++k) {
        if (!(ok = kwait(kv + k))) break;
        ptx::tc_fence_after();
        issue_s(cnt + k, kv + k);
      }
      for (uint32_t i = 0; i < n && ok; ++i) {
        const uint32_t c = cnt + i;
        // dQ += dS K (dS over the S columns of its buffer; K used MN-major)
        if (!(ok = wait_spin_warp(bar(kBbDsFull), c & 1u, ab, kStatusMma))) break;
        if (i == 0 && units > 0 &&
            !(ok = wait_spin_warp(bar(kBbAccFree), (units - 1) & 1u, ab, kStatusMma)))
          break;
        ptx::tc_fence_after();
        bwd_issue_ts<D, BF16>(tAcc, sbuf(c), kslot(kv + i), i > 0);
        ptx::umma_commit_elect(bar(kKEmpty + (kv + i) % KS));
        if (i + 2 < n) {  // in-order: after dQ(c) has read dS(c)
          if (!(ok = kwait(kv + i + 2))) break;
          issue_s(c + 2, kv + i + 2);
        }
      }
      if (!ok) break;
      ptx::umma_commit_elect(bar(kBbAccFull));
    } else {
      if (!(ok = vwait(kv))) break;
      ptx::tc_fence_after();
      issue_dp(kv);
      for (uint32_t i = 0; i < n && ok; ++i) {
        const uint32_t c = cnt + i;
        // dP(c) was read: the next dP into B
        if (!(ok = wait_spin_warp(bar(kBbPFull), c & 1u, ab, kStatusMma))) break;
        if (i + 1 < n) {
          if (!(ok = vwait(kv + i + 1))) break;
          ptx::tc_fence_after();
          issue_dp(kv + i + 1);
        }
      }
      if (!ok) break;
    }
    cnt += n;
    kv += n;
    ptx::umma_commit_elect(bar(kBbFixEmpty));
    ++units;
  }
  ptx::umma_commit_elect(bar(SQ ? kBbDrain : kBbDrainB));
  wait_drain(bar(SQ ? kBbDrain : kBbDrainB), 0u, ab, kStatusDrain);
}

// Element-wise softmax gradient, one thread per TMEM lane (row r of the
// 128-row scratch tiles) and 64 columns per warpgroup (half h). KEYS (dK/dV):
// the row is key k = 128 t + r, the columns are queries of the streamed tile,
// whose lse2 / D come from the stage's vectors. Otherwise (dQ): the row is
// query q = 128 t + r, the columns are keys, lse2 / D are the row's own.
// P stays in fp32 registers; only the MMA operands are rounded to 16 bits.
template <int D, bool BF16, bool CAUSAL, bool KEYS>
__device__ __forceinline__ void bwd_elementwise(const BwdArgs& a, const uint8_t* sgen,
                                                uint32_t bars, uint32_t tmem, const AbortCtx& ab,
                                                int warp, int lane) {
  using L = BwdLayout<D, KEYS>;
  constexpr int S = L::kStages;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  const int r = (warp & 3) * 32 + lane;
  const int h = (warp >> 2) - 1;  // column half of this warpgroup
  const int c0 = 64 * h;
  const uint32_t tl = ptx::tmem_lane_base(tmem, warp);
  const uint32_t tA0 = tl + L::kColA + static_cast<uint32_t>(c0);
  const uint32_t tA1 = tl + L::kColA1 + static_cast<uint32_t>(c0);
  const uint32_t tB = tl + L::kColB + static_cast<uint32_t>(c0);
  const float cl2 = a.scale_log2;
  const bool ragged = (a.N & 127) != 0;
  // Where the scores are issued ahead (dQ kernel; dK/dV at d = 64, two S^T
  // buffers) the waits are usually already satisfied: poll, which resumes
  // sooner; otherwise suspend and leave issue slots to the other warps.
  auto ew_wait = [&](uint32_t b, uint32_t parity) {
    return L::kDblS ? wait_spin_warp(b, parity, ab, kStatusSoftmax)
                    : wait_bounded_warp(b, parity, ab, kStatusSoftmax);
  };
  uint32_t ring = 0, cnt = 0;
  int round = 0, bh = 0, t = 0;
  bool ok = true;
  while (ok && bwd_next_unit<CAUSAL, KEYS>(round, a, bh, t)) {
    int first, last;
    bwd_span<CAUSAL, KEYS>(a, t, first, last);
    const int row = 128 * t + r;  // this thread's key (KEYS) or query
    float my_lse2 = 0.f, my_d = 0.f;
    if constexpr (!KEYS) {
      const size_t v0 = (static_cast<size_t>(bh) * a.n_t + t) * 128 + r;
      my_lse2 = a.lse2[v0];
      my_d = a.delta[v0];
    }
    for (int st = first; st <= last; ++st) {
      const uint32_t rr = ring++;
      const uint32_t c = cnt++;
      const uint32_t ph = c & 1u;
      // S (S^T) alternates between A and A1 where there are two buffers
      const bool odd = L::kDblS && (c & 1u);
      const uint32_t tA = odd ? tA1 : tA0;
      // the stage's lse2 / D vectors (TMA-written): observe their barrier too
      if (KEYS && !(ok = ew_wait(bar(kBbRing + rr % S), (rr / S) & 1u))) break;
      const float* vec = reinterpret_cast<const float*>(
          sgen + L::kOffRing + (rr % S) * L::kStageBytes + 2 * L::kTileBytes);
      // ---- P: scores of this tile against the row's reference
      if (!(ok = ew_wait(bar(odd ? kBbA1Full : kBbAFull), L::kDblS ? (c >> 1) & 1u : ph))) break;
      ptx::tc_fence_after();
      uint32_t sr[2][32];
      ptx::tmem_ld32(tA, sr[0]);
      ptx::tmem_ld32(tA + 32u, sr[1]);
      ptx::tmem_ld_wait(sr[0]);
      ptx::tmem_ld_wait(sr[1]);
      // masks only on the diagonal tile (causal) and the ragged last key tile
      const bool masked = KEYS ? (CAUSAL && st == t)
                               : ((CAUSAL && st == t) || (ragged && st == a.n_t - 1));
      auto weights = [&](auto mask_tag) {
        constexpr bool kMask = decltype(mask_tag)::value;
#pragma unroll
        for (int j = 0; j < 64; j += 4) {
          float ref[4];
          if constexpr (KEYS) {
            const float4 l4 = *reinterpret_cast<const float4*>(vec + c0 + j);
            ref[0] = l4.x; ref[1] = l4.y; ref[2] = l4.z; ref[3] = l4.w;
          } else {
            ref[0] = ref[1] = ref[2] = ref[3] = my_lse2;
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = j + e, col = 128 * st + c0 + c;
            uint32_t& x = sr[c >> 5][c & 31];
            bool keep = true;
            if constexpr (kMask) {
              if constexpr (KEYS) keep = col >= row;  // query col sees key row
              else keep = col < a.N && (!CAUSAL || col <= row);
            }
            // +inf lse2 (queries past N) gives weight 0 unmasked
            x = __float_as_uint(keep ? ptx::ex2(fmaf(__uint_as_float(x), cl2, -ref[e])) : 0.f);
          }
        }
      };
      if (masked) weights(std::true_type{});
      else weights(std::false_type{});
      if constexpr (KEYS) {
        // P^T (16 bit) over this half's first 32 S^T columns, for dV += P^T dO
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c)
          pk[c] = pack2<BF16>(__uint_as_float(sr[(2 * c) >> 5][(2 * c) & 31]),
                              __uint_as_float(sr[(2 * c + 1) >> 5][(2 * c + 1) & 31]));
        ptx::tmem_st32(tA, pk);
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar(kBbPFull));
      }
      // ---- dS = P (dP - D) (16 bit) over this half's first 32 dP^T columns
      // (dK/dV) or its first 32 S columns (dQ)
      if (!(ok = ew_wait(bar(kBbBFull), ph))) break;
      ptx::tc_fence_after();
      uint32_t dp[2][32];
      ptx::tmem_ld32(tB, dp[0]);
      ptx::tmem_ld32(tB + 32u, dp[1]);
      ptx::tmem_ld_wait(dp[0]);
      ptx::tmem_ld_wait(dp[1]);
      if constexpr (!KEYS) {  // dP is in registers: the MMA may overwrite B
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar(kBbPFull));
      }
      uint32_t ds[32];
#pragma unroll
      for (int j = 0; j < 64; j += 4) {
        float dd[4];
        if constexpr (KEYS) {
          const float4 d4 = *reinterpret_cast<const float4*>(vec + 128 + c0 + j);
          dd[0] = d4.x; dd[1] = d4.y; dd[2] = d4.z; dd[3] = d4.w;
        } else {
          dd[0] = dd[1] = dd[2] = dd[3] = my_d;
        }
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
          const int c = j + e;
          const float g0 = __uint_as_float(sr[c >> 5][c & 31]) *
                           (__uint_as_float(dp[c >> 5][c & 31]) - dd[e]);
          const float g1 = __uint_as_float(sr[(c + 1) >> 5][(c + 1) & 31]) *
                           (__uint_as_float(dp[(c + 1) >> 5][(c + 1) & 31]) - dd[e + 1]);
          ds[c >> 1] = pack2<BF16>(g0, g1);
        }
      }
      ptx::tmem_st32(KEYS ? tB : tA, ds);
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(kBbDsFull));
    }
  }
}

// Epilogue: the unit's accumulators (dV and dK, or dQ) from TMEM to global
// memory; dK and dQ carry the score scale.
template <int D, bool BF16, bool CAUSAL, bool KEYS>
__device__ __forceinline__ void bwd_epilogue(const BwdArgs& a, uint32_t bars, uint32_t tmem,
                                             const AbortCtx& ab, int warp, int lane) {
  using L = BwdLayout<D, KEYS>;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  const int r = (warp & 3) * 32 + lane;
  const uint32_t tl = ptx::tmem_lane_base(tmem, warp);
  uint32_t units = 0;
  int round = 0, bh = 0, t = 0;
  bool ok = true;
  // tcgen05.ld is warp-collective (.sync.aligned): every lane loads, only the
  // lanes of rows below N store.
  auto store = [&](uint32_t tcol, void* base, size_t row, bool valid, float mul) {
    uint4* orow = reinterpret_cast<uint4*>(static_cast<uint16_t*>(base) + row * D);
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
      uint32_t v[32];
      ptx::tmem_ld32(tcol + 32u * c, v);
      ptx::tmem_ld_wait(v);
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e)
        pk[e] = pack2<BF16>(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
      if (valid) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          __stcs(orow + 4 * c + q,
                 make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]));
      }
    }
  };
  while (ok && bwd_next_unit<CAUSAL, KEYS>(round, a, bh, t)) {
    if (!(ok = wait_bounded_warp(bar(kBbAccFull), units & 1u, ab, kStatusEpilogue))) break;
    ptx::tc_fence_after();
    const int row = 128 * t + r;
    const bool valid = row < a.N;
    const size_t grow = static_cast<size_t>(bh) * a.N + (valid ? row : 0);
    if constexpr (KEYS) {
      store(tl + L::kColAcc0, a.dv, grow, valid, 1.f);
      store(tl + L::kColAcc1, a.dk, grow, valid, a.scale);
    } else {
      store(tl + L::kColAcc0, a.dq, grow, valid, a.scale);
    }
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(bar(kBbAccFree));
    ++units;
  }
}

// One backward kernel: KEYS = dK / dV, otherwise dQ. Maps: Q, K, V, dO.
template <int D, bool BF16, bool CAUSAL, bool KEYS>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const BwdArgs a) {
  using L = BwdLayout<D, KEYS>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - raw);
  const uint32_t bars = sbase + L::kOffBar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sgen + L::kOffBar + kBwdSlotTmem);
  volatile uint32_t* abort_flag =
      reinterpret_cast<volatile uint32_t*>(sgen + L::kOffBar + kBwdSlotAbort);
  const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
  const AbortCtx ab{abort_flag, a.status};
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  uint64_t* clock_slot = reinterpret_cast<uint64_t*>(sgen + L::kOffBar + kBwdSlotClock);
  if (threadIdx.x == 0 && a.clk != nullptr) clock_begin(clock_slot);
  if (threadIdx.x == 0) {
    // two MMA chains (dK/dV at d = 64, dQ always) each commit the
    // shared-resource barriers
    constexpr uint32_t kChains = KEYS ? (L::kDblS ? 2u : 1u) : 2u;
    ptx::mbar_init(bar(kBbFixFull), 1);
    ptx::mbar_init(bar(kBbFixEmpty), kChains);
    ptx::mbar_init(bar(kBbAFull), 1);
    ptx::mbar_init(bar(kBbBFull), 1);
    ptx::mbar_init(bar(kBbPFull), 8);
    ptx::mbar_init(bar(kBbDsFull), 8);
    ptx::mbar_init(bar(kBbAccFull), KEYS ? kChains : 1u);  // dQ: chain SQ alone
    ptx::mbar_init(bar(kBbAccFree), 4);
    ptx::mbar_init(bar(kBbDrain), 1);
    ptx::mbar_init(bar(kBbA1Full), 1);
    ptx::mbar_init(bar(kBbDrainB), 1);
    if constexpr (KEYS) {  // stage full (TMA), stage empty (both chains)
      for (int s = 0; s < L::kStages; ++s) {
        ptx::mbar_init(bar(kBbRing + s), 1);
        ptx::mbar_init(bar(kBbRing + L::kStages + s), kChains);
      }
    } else {
      for (int s = 0; s < 2 * (L::kKSlots + L::kVSlots); ++s) ptx::mbar_init(bar(kBbRing + s), 1);
    }
    *abort_flag = 0u;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int wgrp = warp >> 2;
  if (wgrp == 0) {
    ptx::setmaxnreg_to<kBwdRegsWG0, kBwdRegsLaunch>();
    if (warp == 0) {
      if (lane == 0) bwd_producer<D, CAUSAL, KEYS>(&tm_q, &tm_k, &tm_v, &tm_do, a, sbase, bars, ab);
    } else if constexpr (KEYS && L::kDblS) {  // the two MMA chains, each a whole warp
      if (warp == 2) bwd_mma_kv<D, BF16, CAUSAL, true>(a, sbase, bars, tmem, ab);
      else if (warp == 3) bwd_mma_kv<D, BF16, CAUSAL, false>(a, sbase, bars, tmem, ab);
    } else if constexpr (!KEYS) {  // the dQ kernel's two MMA chains
      if (warp == 2) bwd_mma_dq_chain<D, BF16, CAUSAL, true>(a, sbase, bars, tmem, ab);
      else if (warp == 3) bwd_mma_dq_chain<D, BF16, CAUSAL, false>(a, sbase, bars, tmem, ab);
    } else if (warp == 1) {  // the whole warp
      bwd_mma<D, BF16, CAUSAL, true>(a, sbase, bars, tmem, ab);
    }
  } else if (wgrp <= 2) {
    ptx::setmaxnreg_to<kBwdRegsElem, kBwdRegsLaunch>();
    bwd_elementwise<D, BF16, CAUSAL, KEYS>(a, sgen, bars, tmem, ab, warp, lane);
  } else {
    ptx::setmaxnreg_to<kBwdRegsEpi, kBwdRegsLaunch>();
    bwd_epilogue<D, BF16, CAUSAL, KEYS>(a, bars, tmem, ab, warp, lane);
  }
  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, 512);
  if (threadIdx.x == 0 && a.clk != nullptr) clock_end(a.clk, clock_slot);
}

// Host side (fa_bwd_d64.cu / fa_bwd_d128.cu): the three launches of one call.
// maps: Q, K, V, dO ({d, N, H, B} 16-bit, 64 x 128 boxes); grid: persistent CTAs.
cudaError_t launch_bwd_d64(bool bf16, bool causal, const CUtensorMap* maps, const BwdArgs& a,
                           const void* o, const void* dout, const float* lse, int grid,
                           cudaStream_t stream);
cudaError_t launch_bwd_d128(bool bf16, bool causal, const CUtensorMap* maps, const BwdArgs& a,
                            const void* o, const void* dout, const float* lse, int grid,
                            cudaStream_t stream);

}  // namespace fa
