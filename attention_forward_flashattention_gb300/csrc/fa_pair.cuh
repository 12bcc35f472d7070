// Fused attention forward on CTA pairs (tcgen05.mma cta_group::2), head
// dimension 128, fp16 / bf16: the "CTA pair" of "TMA + Warp Specialization"
// (CUDA book ch. 17), section 17.9, item 3 -- two SMs share each tensor-core
// product, which makes the tile per product larger (M = 256 query rows).
//
// Work unit: 512 query rows of one (batch, head). Each CTA of the pair holds
// two 128-row Q tiles (tile i of CTA r: rows 512 m + 256 i + 128 r), and tile
// i of both CTAs forms one M = 256 product: each CTA supplies its own 128 rows
// of the A operand (Q, or P) and HALF of the B operand (64 of the 128 keys of
// a K tile, 64 of the 128 columns of a V tile), and receives its 128 rows of
// the result in its own tensor memory. So each SM loads and holds only half of
// every K / V tile (16 KB ring slots: a K ring and a V ring of their own, so a
// K half is refilled while the previous V half is still in use), and the two
// tiles ping-pong on the tensor core as in the one-CTA kernel: the softmax of
// one tile runs while the other's products run. Tensor memory holds S0, S1
// (columns 0-255) and O0, O1 (256-511); the softmax writes P_i as bf16/fp16 to
// shared memory in the layout the products read (128-byte swizzled, K-major),
// and the PV products take both operands from shared memory.
//
// Warp roles (16 warps), the same in both CTAs unless noted:
//   warp 0 (one lane): TMA producer: its two Q tiles, then per KV step its K
//           half of tile j and its V half of tile j-1, the bytes counted on the
//           EVEN CTA's barriers;
//   warps 1-3, even CTA only (whole warp, elected lane): the S products
//           (non-causal: warp 1 tile 0, warp 2 tile 1; causal: warp 2 both) and
//           the PV products (warp 3), with their commits; warp 1 also owns the
//           tensor memory in both CTAs;
//   warps 4-7 / 8-11: softmax of tile 0 / tile 1 of this CTA (one thread per
//           row; the one-CTA kernel's per-tile softmax);
//   warps 12-15: epilogue (O / l by TMA store of the CTA's rows).
// Barriers that collect arrivals from both CTAs (TMA bytes, S read, P written,
// O drained) live in the even CTA; products signal both CTAs by multicast
// commits. Every wait is bounded (1 s), as in the one-CTA kernel. The
// arithmetic of every output element is the one-CTA kernel's, so the two
// kernels' results are identical bit for bit.
#pragma once

#include <cuda.h>

#include "fa_kernel.cuh"

namespace fa {

constexpr int kPairSlotTmem = 480;
constexpr int kPairSlotAbort = 484;
constexpr int kPairSlotClock = 488;

// This pair's units: round k takes unit k * P + c (P pairs, c = this pair);
// causal units longest first, odd rounds in reverse pair order (as the
// one-CTA kernel's next_unit, with pairs in place of CTAs).
template <bool CAUSAL>
__device__ __forceinline__ bool next_pair_unit(int& round, const FwdArgs& a, int& bh, int& mblk) {
  const int G = static_cast<int>(gridDim.x >> 1);
  for (;;) {
    const long long base = static_cast<long long>(round) * G;
    if (base >= a.n_units) return false;
    int c = static_cast<int>(blockIdx.x >> 1);
    if (CAUSAL && (round & 1)) c = G - 1 - c;
    const long long u = base + c;
    ++round;
    if (u >= a.n_units) continue;
    if (CAUSAL) {
      const int lvl = static_cast<int>(u / a.BH);
      bh = static_cast<int>(u - static_cast<long long>(lvl) * a.BH);
      mblk = a.n_mblk - 1 - lvl;
    } else {
      bh = static_cast<int>(u / a.n_mblk);
      mblk = static_cast<int>(u - static_cast<long long>(bh) * a.n_mblk);
    }
    return true;
  }
}

// FP8: e4m3 Q, K and V^T, whose 128-element rows are one 128-byte panel, so
// every tile and ring slot is half as large (and the rings are deeper).
template <bool FP8 = false>
struct PairLayout {
  static constexpr int kTileBytes = (FP8 ? 1 : 2) * kPanelBytes;  // a Q or P tile (128 x 128)
  static constexpr int kSlotBytes = FP8 ? kPanelBytes / 2 : kPanelBytes;  // a K / V half
  static constexpr int kKSlots = FP8 ? 4 : 2;                   // K ring (K_j, K_{j+1}, ...)
  static constexpr int kVSlots = FP8 ? 4 : 3;                   // V ring
  static constexpr int kOffQ = 0;                               // Q0, Q1
  static constexpr int kOffP = 2 * kTileBytes;                  // P0, P1 (K-major SW128)
  static constexpr int kOffK = 4 * kTileBytes;
  static constexpr int kOffV = kOffK + kKSlots * kSlotBytes;
  static constexpr int kOffStats = kOffV + kVSlots * kSlotBytes;  // [2 tiles][128] row sums
  static constexpr int kOffOut = kOffStats + 1024;
  static constexpr int kOutSliceBytes = 32 * 128;
  static constexpr int kOffBar = kOffOut + 4 * kOutSliceBytes;
  static constexpr int kSmemBytes = kOffBar + 512 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kOffBar % 8 == 0 && kOffOut % 1024 == 0, "alignment");
  static constexpr uint32_t kColS = 0;    // S_i at 128 i
  static constexpr uint32_t kColO = 256;  // O_i at 256 + 128 i
  // barrier slots of the K and V rings (PairBar below)
  static constexpr int kBarKFull = 22;
  static constexpr int kBarKEmpty = kBarKFull + kKSlots;
  static constexpr int kBarVFull = kBarKEmpty + kKSlots;
  static constexpr int kBarVEmpty = kBarVFull + kVSlots;
  static_assert(8 * (kBarVEmpty + kVSlots) <= kPairSlotTmem, "barrier block");
};

enum PairBar : int {
  kQbQFull = 0,       // [2] even CTA: both CTAs' Q tile i landed
  kQbQEmpty = 2,      // both: the unit's last S products done (a commit per S warp)
  kQbSFull = 3,       // [2] both: S_i ready (multicast commit)
  kQbSFree = 5,       // [2] even CTA: S_i read by the 8 softmax warps of tile i (pair)
  kQbPFull = 7,       // [2] even CTA: P_i in shared memory, O_i rescaled (8 warps, pair)
  kQbPFree = 9,       // [2] both: PV_i done: P_i reusable, O_i updated (multicast commit)
  kQbOFull = 11,      // [2] both: the unit's last PV_i done (multicast commit)
  kQbOFree = 13,      // [2] even CTA: O_i read by the 8 epilogue warps of the pair
  kQbStatsFull = 15,  // [2] local: 128 softmax threads wrote tile i's row sums
  kQbStatsFree = 17,  // [2] local: 128 epilogue threads read them
  kQbDrain = 19,      // [2] even CTA: every product of S warp w completed
  kQbDrainPV = 21,    // even CTA: every PV product completed
  // then, from slot 22 (PairLayout::kBarKFull ...): [K slots] even CTA: both K
  // halves landed; [K slots] both: K slot free (a commit per S warp); [V slots]
  // even CTA: both V halves landed; [V slots] both: V slot free
};

// Units of 512 rows per pair (n_mblk = ceil(N / 512)): causal units visit KV
// tiles up to the diagonal of their last row.
template <bool CAUSAL>
__device__ __forceinline__ int pair_kv_tiles(const FwdArgs& a, int mblk) {
  return CAUSAL ? min(4 * mblk + 4, a.n_kv) : a.n_kv;
}

// Loads, per unit: both Q tiles, then K_0, then K_{j+1} before V_j (the S
// products of a tile need the next K while its softmax runs; V_j is needed
// only when P_j is written), from two rings that release slots independently.
template <bool CAUSAL, bool FP8>
__device__ __forceinline__ void pair_producer(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                              const CUtensorMap* tm_v, const FwdArgs& a,
                                              uint32_t sbase, uint32_t bars, uint32_t rank,
                                              const AbortCtx& ab) {
  using L = PairLayout<FP8>;
  constexpr int kQbKFull = L::kBarKFull, kQbKEmpty = L::kBarKEmpty;
  constexpr int kQbVFull = L::kBarVFull, kQbVEmpty = L::kBarVEmpty;
  constexpr int kPanels = FP8 ? 1 : 2;  // 128-byte panels per Q / K row
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  auto lead = [&](int i) { return ptx::mapa_shared(bar(i), 0); };
  ptx::prefetch_tmap(tm_q);
  ptx::prefetch_tmap(tm_k);
  ptx::prefetch_tmap(tm_v);
  uint32_t kcnt = 0, vcnt = 0, units = 0;
  int round = 0, bh = 0, mblk = 0;
  bool ok = true;
  while (ok && next_pair_unit<CAUSAL>(round, a, bh, mblk)) {
    const int nkv = pair_kv_tiles<CAUSAL>(a, mblk);
    if (!(ok = wait_cluster<false>(bar(kQbQEmpty), (units & 1u) ^ 1u, ab, kStatusProducer))) break;
    const int hh = bh % a.H, bb = bh / a.H;
    for (int i = 0; i < 2; ++i) {
      if (rank == 0) ptx::mbar_arrive_expect_tx(bar(kQbQFull + i), 2 * L::kTileBytes);
      for (int p = 0; p < kPanels; ++p)
        ptx::tma_load_4d_pair(sbase + L::kOffQ + i * L::kTileBytes + p * kPanelBytes, tm_q,
                              lead(kQbQFull + i), 64 * p,
                              mblk * 512 + 256 * i + 128 * static_cast<int>(rank), hh, bb);
    }
    ++units;
    for (int j = 0; j <= nkv && ok; ++j) {
      if (j < nkv) {  // K_j: keys 128 j + 64 rank .. +63
        const uint32_t s = kcnt % L::kKSlots, ph = (kcnt / L::kKSlots) & 1u;
        if (!(ok = wait_cluster<false>(bar(kQbKEmpty + s), ph ^ 1u, ab, kStatusProducer))) break;
        if (rank == 0) ptx::mbar_arrive_expect_tx(bar(kQbKFull + s), 2 * L::kSlotBytes);
        const uint32_t dst = sbase + L::kOffK + s * L::kSlotBytes;
        for (int p = 0; p < kPanels; ++p)
          ptx::tma_load_4d_pair(dst + p * (kPanelBytes / 2), tm_k, lead(kQbKFull + s), 64 * p,
                                128 * j + 64 * static_cast<int>(rank), hh, bb);
        ++kcnt;
      }
      if (j >= 1) {   // V_{j-1}: keys 128 (j - 1) .. +127, columns 64 rank .. +63
        const uint32_t s = vcnt % L::kVSlots, ph = (vcnt / L::kVSlots) & 1u;
        if (!(ok = wait_cluster<false>(bar(kQbVEmpty + s), ph ^ 1u, ab, kStatusProducer))) break;
        if (rank == 0) ptx::mbar_arrive_expect_tx(bar(kQbVFull + s), 2 * L::kSlotBytes);
        if constexpr (FP8)  // V^T {keys, d, h, b}: those keys of d rows 64 rank .. +63
          ptx::tma_load_4d_pair(sbase + L::kOffV + s * L::kSlotBytes, tm_v, lead(kQbVFull + s),
                                128 * (j - 1), 64 * static_cast<int>(rank), hh, bb);
        else
          ptx::tma_load_4d_pair(sbase + L::kOffV + s * L::kSlotBytes, tm_v, lead(kQbVFull + s),
                                64 * static_cast<int>(rank), 128 * (j - 1), hh, bb);
        ++vcnt;
      }
    }
  }
  if (!ok && rank == 0) {
    // let the copies already issued (both CTAs' halves) land before exit
    for (uint32_t s = 0; s < static_cast<uint32_t>(L::kKSlots) && s < kcnt; ++s) {
      const uint32_t last = kcnt - 1 - ((kcnt - 1 - s) % L::kKSlots);
      wait_drain(bar(kQbKFull + s), (last / L::kKSlots) & 1u, ab, kStatusDrain);
    }
    for (uint32_t s = 0; s < static_cast<uint32_t>(L::kVSlots) && s < vcnt; ++s) {
      const uint32_t last = vcnt - 1 - ((vcnt - 1 - s) % L::kVSlots);
      wait_drain(bar(kQbVFull + s), (last / L::kVSlots) & 1u, ab, kStatusDrain);
    }
    if (units > 0) {
      wait_drain(bar(kQbQFull + 0), (units - 1) & 1u, ab, kStatusDrain);
      wait_drain(bar(kQbQFull + 1), (units - 1) & 1u, ab, kStatusDrain);
    }
  }
}

// Even CTA: the products are issued by three warps (elected lane of each),
// which need no ordering between them: S products write S_i, PV products read
// P_i from shared memory and write O_i.
//   S warp(s): S_i(j) = Q_i K_j^T once the softmax has read S_i(j - 1).
//            Non-causal: one warp per tile, on different SM sub-partitions
//            (each MMA issue takes issue slots from the softmax warps beside
//            it, and the slowest softmax warp sets when P is complete);
//            causal: one warp for both tiles (measured faster there).
//   PV warp: O_i += P_i(j) V_j once P_i(j) is written (and the epilogue has
//            drained O_i, at a unit's first tile).
// K_j and V_j come from their own rings (global counters of the tiles loaded).
// S warps of a kernel instance (each issues the tiles i0 .. i1 - 1).
template <bool CAUSAL>
__host__ __device__ constexpr int pair_s_warps() { return CAUSAL ? 1 : 2; }

template <bool BF16, bool CAUSAL, bool FP8, int I0, int I1, int W>
__device__ __forceinline__ void pair_mma_s(const FwdArgs& a, uint32_t sbase, uint32_t bars,
                                           uint32_t tmem, const AbortCtx& ab) {
  using L = PairLayout<FP8>;
  constexpr int kQbKFull = L::kBarKFull, kQbKEmpty = L::kBarKEmpty;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  constexpr uint32_t kIdS = FP8 ? ptx::idesc_f8(256, 128) : ptx::idesc_f16(BF16, false, 256, 128);
  const uint64_t dQ0 = desc_kmajor(sbase + L::kOffQ);
  const uint64_t dK0 = desc_kmajor(sbase + L::kOffK);
  uint32_t units = 0, scnt = 0;  // scnt: K tiles used so far = S_i products issued (each tile)
  int round = 0, bh = 0, mblk = 0;
  bool ok = true;
  while (ok && next_pair_unit<CAUSAL>(round, a, bh, mblk)) {
    const int nkv = pair_kv_tiles<CAUSAL>(a, mblk);
#pragma unroll
    for (int i = I0; i < I1; ++i)
      ok = ok && wait_cluster_warp(bar(kQbQFull + i), units & 1u, ab, kStatusMma);
    for (int j = 0; j < nkv && ok; ++j, ++scnt) {
      const uint32_t ks = scnt % L::kKSlots;
      if (!(ok = wait_cluster_warp(bar(kQbKFull + ks), (scnt / L::kKSlots) & 1u, ab, kStatusMma)))
        break;
#pragma unroll
      for (int i = I0; i < I1; ++i) {
        if (!ok) break;
        // S_i(scnt) overwrites S_i(scnt - 1): read by the softmax?
        if (scnt > 0 &&
            !(ok = wait_cluster_warp(bar(kQbSFree + i), (scnt - 1) & 1u, ab, kStatusMma)))
          break;
        ptx::tc_fence_after();
        uint64_t q = desc_add(dQ0, static_cast<uint32_t>(i) * L::kTileBytes);
        uint64_t k = desc_add(dK0, ks * static_cast<uint32_t>(L::kSlotBytes));
        if constexpr (FP8) {  // K = 32 per product, one panel: +32 bytes per step
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            ptx::umma_f8_ss_pair_elect(tmem + L::kColS + 128u * i, q, k, kIdS, kk > 0 ? 1u : 0u);
            q = desc_add(q, 32u);
            k = desc_add(k, 32u);
            asm volatile("" : "+l"(q), "+l"(k));
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            ptx::umma_f16_ss_pair_elect(tmem + L::kColS + 128u * i, q, k, kIdS, kk > 0 ? 1u : 0u);
            const bool next_panel = (kk & 3) == 3;
            q = desc_add(q, next_panel ? static_cast<uint32_t>(kPanelBytes - 96) : 32u);
            k = desc_add(k, next_panel ? static_cast<uint32_t>(kPanelBytes / 2 - 96) : 32u);
            asm volatile("" : "+l"(q), "+l"(k));
          }
        }
        ptx::umma_commit_pair_elect(bar(kQbSFull + i), 3);
      }
      if (!ok) break;
      ptx::umma_commit_pair_elect(bar(kQbKEmpty + ks), 3);  // K_j consumed (by this warp's tiles)
      if (j + 1 == nkv) ptx::umma_commit_pair_elect(bar(kQbQEmpty), 3);
    }
    ++units;
  }
  ptx::umma_commit_pair_elect(bar(kQbDrain + W), 1);
  wait_drain(bar(kQbDrain + W), 0u, ab, kStatusDrain);
}

template <bool BF16, bool CAUSAL, bool FP8>
__device__ __forceinline__ void pair_mma_pv(const FwdArgs& a, uint32_t sbase, uint32_t bars,
                                            uint32_t tmem, const AbortCtx& ab) {
  using L = PairLayout<FP8>;
  constexpr int kQbVFull = L::kBarVFull, kQbVEmpty = L::kBarVEmpty;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  // 16-bit: V as stored ([key][d], MN-major B); FP8: V^T ([d][key], K-major B)
  constexpr uint32_t kIdPV = FP8 ? ptx::idesc_f8(256, 128) : ptx::idesc_f16(BF16, true, 256, 128);
  const uint64_t dP[2] = {desc_kmajor(sbase + L::kOffP),
                          desc_kmajor(sbase + L::kOffP + L::kTileBytes)};
  const uint64_t dV0 = FP8 ? desc_kmajor(sbase + L::kOffV) : desc_v(sbase + L::kOffV);
  uint32_t units = 0, pcnt = 0;  // pcnt: V tiles used so far = P_i tiles consumed (each tile)
  int round = 0, bh = 0, mblk = 0;
  bool ok = true;
  while (ok && next_pair_unit<CAUSAL>(round, a, bh, mblk)) {
    const int nkv = pair_kv_tiles<CAUSAL>(a, mblk);
    for (int j = 0; j < nkv && ok; ++j, ++pcnt) {
      const uint32_t vs = pcnt % L::kVSlots;
      if (!(ok = wait_cluster_warp(bar(kQbVFull + vs), (pcnt / L::kVSlots) & 1u, ab, kStatusMma)))
        break;
      for (int i = 0; i < 2 && ok; ++i) {
        if (!(ok = wait_cluster_warp(bar(kQbPFull + i), pcnt & 1u, ab, kStatusMma))) break;
        if (j == 0 && units > 0 &&
            !(ok = wait_cluster_warp(bar(kQbOFree + i), (units - 1) & 1u, ab, kStatusMma)))
          break;
        ptx::tc_fence_after();
        uint64_t pd = dP[i], v = desc_add(dV0, vs * static_cast<uint32_t>(L::kSlotBytes));
        if constexpr (FP8) {  // K = 32 keys per product: +32 bytes in P and V^T
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            ptx::umma_f8_ss_pair_elect(tmem + L::kColO + 128u * i, pd, v, kIdPV,
                                       (j > 0 || kk > 0) ? 1u : 0u);
            pd = desc_add(pd, 32u);
            v = desc_add(v, 32u);
            asm volatile("" : "+l"(pd), "+l"(v));
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            ptx::umma_f16_ss_pair_elect(tmem + L::kColO + 128u * i, pd, v, kIdPV,
                                        (j > 0 || kk > 0) ? 1u : 0u);
            pd = desc_add(pd, (kk & 3) == 3 ? static_cast<uint32_t>(kPanelBytes - 96) : 32u);
            v = desc_add(v, 2048u);
            asm volatile("" : "+l"(pd), "+l"(v));
          }
        }
        ptx::umma_commit_pair_elect(bar(kQbPFree + i), 3);
        if (j + 1 == nkv) ptx::umma_commit_pair_elect(bar(kQbOFull + i), 3);
      }
      if (!ok) break;
      ptx::umma_commit_pair_elect(bar(kQbVEmpty + vs), 3);  // V_j consumed
    }
    ++units;
  }
  ptx::umma_commit_pair_elect(bar(kQbDrainPV), 1);
  wait_drain(bar(kQbDrainPV), 0u, ab, kStatusDrain);
}

// Softmax of tile i (warpgroup 1 + i) of this CTA: the one-CTA kernel's
// per-tile softmax (d = 128, 16-bit), with S released as soon as it is in
// registers, P written to shared memory (K-major, 128-byte swizzle: the A
// operand of the PV product), and the S-read / P-written arrivals sent to the
// even CTA (one per warp).
template <bool BF16, bool CAUSAL, bool FP8>
__device__ __forceinline__ void pair_softmax(const FwdArgs& a, uint32_t sbase, uint32_t bars,
                                             uint32_t tmem, float* stats, uint32_t rank,
                                             const AbortCtx& ab, int warp, int lane) {
  using L = PairLayout<FP8>;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  const int wg = (warp >> 2) - 1;
  const int r = (warp & 3) * 32 + lane;
  const uint32_t tl = ptx::tmem_lane_base(tmem, warp);
  const uint32_t tS = tl + L::kColS + 128u * wg;
  const uint32_t tO = tl + L::kColO + 128u * wg;
  const uint32_t lead_pfull = ptx::mapa_shared(bar(kQbPFull + wg), 0);
  const uint32_t lead_sfree = ptx::mapa_shared(bar(kQbSFree + wg), 0);
  const uint32_t sP = sbase + L::kOffP + static_cast<uint32_t>(wg) * L::kTileBytes;
  const float cl2 = a.scale_log2;
  uint32_t scnt = 0, units = 0;
  int round = 0, bh = 0, mblk = 0;
  bool ok = true;
  while (ok && next_pair_unit<CAUSAL>(round, a, bh, mblk)) {
    const int nkv = pair_kv_tiles<CAUSAL>(a, mblk);
    const int tile_row0 = mblk * 512 + 256 * wg + 128 * static_cast<int>(rank);
    const int grow = tile_row0 + r;
    float m_ref = -INFINITY, l = 0.f, l_exp = 0.f;
    for (int j = 0; j < nkv; ++j) {
      if (!(ok = wait_cluster<true>(bar(kQbSFull + wg), scnt & 1u, ab, kStatusSoftmax))) break;
      if (!(ok = __all_sync(0xffffffffu, ok) != 0)) break;
      ++scnt;
      ptx::tc_fence_after();
      // S with its row maximum over each 64-column half formed by the loads
      uint32_t sr[2][2][32];
      float mx_lo, mx_hi;
      ptx::tmem_ld64_max(tS, sr[0], mx_lo);
      ptx::tmem_ld64_max(tS + 64u, sr[1], mx_hi);
      ptx::tmem_ld_wait64x2(sr[0], sr[1]);
      ptx::tmem_ld_wait_f2(mx_lo, mx_hi);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(lead_sfree);  // S_i may be overwritten
      // base-2 score scale of this tile (8-bit inputs: times its K block's scale)
      float cj = cl2;
      if constexpr (FP8) cj = cl2 * __ldg(a.k_scales + static_cast<size_t>(bh) * a.n_kv + j);
      const float2 c2 = make_float2(cj, cj);
      float s[128];
#pragma unroll
      for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c >> 6][(c >> 5) & 1][c & 31]);
      const int k0 = j * kTileRows;
      const bool need_mask = (k0 + kTileRows > a.N) || (CAUSAL && k0 + kTileRows - 1 > tile_row0);
      float m_raw = fmaxf(mx_lo, mx_hi);
      if (need_mask) {  // masked keys: the maximum over the visible ones only
        int lim = a.N - k0;
        if (CAUSAL) lim = min(lim, grow - k0 + 1);
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = (c < lim) ? s[c] : -INFINITY;
        float mx[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) mx[t] = fmaxf(s[2 * t], s[2 * t + 1]);
#pragma unroll
        for (int c = 16; c < 128; c += 16) {
#pragma unroll
          for (int t = 0; t < 8; ++t) mx[t] = ptx::fmax3(mx[t], s[c + 2 * t], s[c + 2 * t + 1]);
        }
        m_raw = fmaxf(ptx::fmax3(mx[0], mx[1], mx[2]),
                      ptx::fmax3(ptx::fmax3(mx[3], mx[4], mx[5]), mx[6], mx[7]));
      }
      const float m_tile = m_raw * cj;
      const float m_new = fmaxf(m_ref, m_tile);
      float alpha = 1.f;
      if (j == 0) {
        m_ref = m_new;
      } else if (m_new > m_ref + 8.f) {
        alpha = ptx::ex2(m_ref - m_new);
        m_ref = m_new;
      }
      const float2 neg2 = make_float2(-m_ref, -m_ref);
      float2 ls[4], lr[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) ls[t] = lr[t] = make_float2(0.f, 0.f);
      uint32_t pk[FP8 ? 32 : 64];
      if constexpr (FP8) {
        // P as e4m3, four keys per word (O is normalised by the unrounded sum)
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float2 t0 = ptx::ffma2(make_float2(s[4 * c], s[4 * c + 1]), c2, neg2);
          const float2 t1 = ptx::ffma2(make_float2(s[4 * c + 2], s[4 * c + 3]), c2, neg2);
          const float p0 = ptx::ex2(t0.x), p1 = ptx::ex2(t0.y);
          const float p2 = ptx::ex2(t1.x), p3 = ptx::ex2(t1.y);
          pk[c] = ptx::pack4_e4m3(p0, p1, p2, p3);
          ls[(2 * c) & 3] = ptx::fadd2(ls[(2 * c) & 3], make_float2(p0, p1));
          ls[(2 * c + 1) & 3] = ptx::fadd2(ls[(2 * c + 1) & 3], make_float2(p2, p3));
        }
      } else {
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float2 t = ptx::ffma2(make_float2(s[2 * c], s[2 * c + 1]), c2, neg2);
          const float p0 = ptx::ex2(t.x), p1 = ptx::ex2(t.y);
          const uint32_t w = pack2<BF16>(p0, p1);
          pk[c] = w;
          ls[c & 3] = ptx::fadd2(ls[c & 3], make_float2(p0, p1));
          if constexpr (BF16) {
            lr[c & 3].x = ptx::add_f32_bf16_lo(lr[c & 3].x, w);
            lr[c & 3].y = ptx::add_f32_bf16_hi(lr[c & 3].y, w);
          }
        }
      }
      // PV_i of the previous tile done: P_i reusable, O_i updated
      if (scnt > 1 &&
          !(ok = wait_cluster_warp(bar(kQbPFree + wg), (scnt - 2) & 1u, ab, kStatusSoftmax)))
        break;
      ptx::tc_fence_after();
      if constexpr (FP8) store_row_panel_sw128(sP, r, pk);
      else store_row128_sw128(sP, r, pk);
      const float2 s01 = ptx::fadd2(ptx::fadd2(ls[0], ls[1]), ptx::fadd2(ls[2], ls[3]));
      const float lsum = s01.x + s01.y;
      float lsum_p = lsum;
      if constexpr (BF16 && !FP8) {
        const float2 r01 = ptx::fadd2(ptx::fadd2(lr[0], lr[1]), ptx::fadd2(lr[2], lr[3]));
        lsum_p = r01.x + r01.y;
      }
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {  // O_i holds PV_i(j - 1) (P-free)
        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          ptx::tmem_ld32(tO + 32u * c, o);
          ptx::tmem_ld_wait(o);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 v =
                ptx::fmul2(make_float2(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), a2);
            o[e] = __float_as_uint(v.x);
            o[e + 1] = __float_as_uint(v.y);
          }
          ptx::tmem_st32(tO + 32u * c, o);
        }
      }
      ptx::fence_proxy_async_smem();  // P visible to the tensor core's reads
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(lead_pfull);
      l = l * alpha + lsum_p;
      l_exp = l_exp * alpha + lsum;
    }
    if (!ok) break;
    if (grow < a.N)
      a.lse[static_cast<size_t>(bh) * a.N + grow] = (m_ref + log2f(l_exp)) * 0.69314718055994531f;
    if (units > 0 &&
        !(ok = wait_bounded_warp(bar(kQbStatsFree + wg), (units - 1) & 1u, ab, kStatusSoftmax)))
      break;
    stats[wg * 128 + r] = l;
    ptx::mbar_arrive(bar(kQbStatsFull + wg));
    ++units;
  }
}

template <bool BF16, bool CAUSAL, bool FP8>
__device__ __forceinline__ void pair_epilogue(const CUtensorMap* tm_o, const FwdArgs& a,
                                               uint32_t sbase, uint32_t bars, uint32_t tmem,
                                               const float* stats, uint32_t rank,
                                               const AbortCtx& ab, int warp, int lane) {
  using L = PairLayout<FP8>;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  const int w = warp & 3;
  const int r = w * 32 + lane;
  const uint32_t tl = ptx::tmem_lane_base(tmem, warp);
  const uint32_t slice = sbase + L::kOffOut + static_cast<uint32_t>(w) * L::kOutSliceBytes;
  const uint32_t srow = slice + static_cast<uint32_t>(lane) * 128u;
  const uint32_t sx = static_cast<uint32_t>(lane & 7);
  if (lane == 0) ptx::prefetch_tmap(tm_o);
  bool pending = false;
  uint32_t units = 0;
  int round = 0, bh = 0, mblk = 0;
  bool ok = true;
  while (ok && next_pair_unit<CAUSAL>(round, a, bh, mblk)) {
    const int hh = bh % a.H, bb = bh / a.H;
    for (int i = 0; i < 2 && ok; ++i) {
      ok = wait_cluster<true>(bar(kQbOFull + i), units & 1u, ab, kStatusEpilogue);
      ok = __all_sync(0xffffffffu, ok) != 0 &&
           wait_bounded_warp(bar(kQbStatsFull + i), units & 1u, ab, kStatusEpilogue);
      if (!ok) break;
      ptx::tc_fence_after();
      const float inv_l = (FP8 ? a.v_scale : 1.f) / stats[i * 128 + r];
      ptx::mbar_arrive(bar(kQbStatsFree + i));
      const float2 il2 = make_float2(inv_l, inv_l);
      const int row0 = mblk * 512 + 256 * i + 128 * static_cast<int>(rank) + 32 * w;
#pragma unroll 1
      for (int p = 0; p < 2; ++p) {
        if (lane == 0 && pending) ptx::bulk_wait_read_all();
        __syncwarp();
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          uint32_t o[32];
          ptx::tmem_ld32(tl + L::kColO + static_cast<uint32_t>(128 * i + 64 * p + 32 * h), o);
          ptx::tmem_ld_wait(o);
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 v = ptx::fmul2(
                make_float2(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1])), il2);
            pk[e] = pack2<BF16>(v.x, v.y);
          }
#pragma unroll
          for (int t = 0; t < 4; ++t)
            ptx::st_shared_v4(srow + (((static_cast<uint32_t>(4 * h + t)) ^ sx) << 4), pk[4 * t],
                              pk[4 * t + 1], pk[4 * t + 2], pk[4 * t + 3]);
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && row0 < a.N) {
          ptx::tma_store_4d(tm_o, slice, 64 * p, row0, hh, bb);
          ptx::bulk_commit();
          pending = true;
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa_shared(bar(kQbOFree + i), 0));
    }
    ++units;
  }
  if (lane == 0 && pending) ptx::bulk_wait_all();
}

// FP8: e4m3 Q, K, V^T (instantiate with BF16 = true: bf16 O).
template <bool BF16, bool CAUSAL, bool FP8 = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kFwdThreads, 1)
    fa_fwd_pair_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_o, const FwdArgs a) {
  using L = PairLayout<FP8>;
  constexpr int kQbKFull = L::kBarKFull, kQbKEmpty = L::kBarKEmpty;
  constexpr int kQbVFull = L::kBarVFull, kQbVEmpty = L::kBarVEmpty;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - raw);
  const uint32_t bars = sbase + L::kOffBar;
  float* stats = reinterpret_cast<float*>(sgen + L::kOffStats);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sgen + L::kOffBar + kPairSlotTmem);
  volatile uint32_t* abort_flag =
      reinterpret_cast<volatile uint32_t*>(sgen + L::kOffBar + kPairSlotAbort);
  uint64_t* clock_slot = reinterpret_cast<uint64_t*>(sgen + L::kOffBar + kPairSlotClock);
  const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
  const uint32_t rank = ptx::cluster_ctarank();
  const AbortCtx ab{abort_flag, a.status};
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  if (threadIdx.x == 0 && a.clk != nullptr) clock_begin(clock_slot);
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(bar(kQbQFull + i), 1);
      ptx::mbar_init(bar(kQbSFull + i), 1);
      ptx::mbar_init(bar(kQbSFree + i), 8);      // 4 softmax warps of tile i in each CTA
      ptx::mbar_init(bar(kQbPFull + i), 8);
      ptx::mbar_init(bar(kQbPFree + i), 1);
      ptx::mbar_init(bar(kQbOFull + i), 1);
      ptx::mbar_init(bar(kQbOFree + i), 8);      // 4 epilogue warps in each CTA
      ptx::mbar_init(bar(kQbStatsFull + i), 128);
      ptx::mbar_init(bar(kQbStatsFree + i), 128);
    }
    ptx::mbar_init(bar(kQbQEmpty), pair_s_warps<CAUSAL>());
    ptx::mbar_init(bar(kQbDrain + 0), 1);
    ptx::mbar_init(bar(kQbDrain + 1), 1);
    ptx::mbar_init(bar(kQbDrainPV), 1);
    for (int s = 0; s < L::kKSlots; ++s) {
      ptx::mbar_init(bar(kQbKFull + s), 1);
      ptx::mbar_init(bar(kQbKEmpty + s), pair_s_warps<CAUSAL>());
    }
    for (int s = 0; s < L::kVSlots; ++s) {
      ptx::mbar_init(bar(kQbVFull + s), 1);
      ptx::mbar_init(bar(kQbVEmpty + s), 1);
    }
    *abort_flag = 0u;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), 512);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int wgrp = warp >> 2;
  if (wgrp == 0) {
    ptx::setmaxnreg_dec<kRegsWG0>();
    if (warp == 0) {
      if (lane == 0) pair_producer<CAUSAL, FP8>(&tm_q, &tm_k, &tm_v, a, sbase, bars, rank, ab);
    } else if (warp == 2 && rank == 0) {
      if constexpr (pair_s_warps<CAUSAL>() == 2)  // tile 1 (tile 0: warp 1)
        pair_mma_s<BF16, CAUSAL, FP8, 1, 2, 1>(a, sbase, bars, tmem, ab);
      else  // both tiles
        pair_mma_s<BF16, CAUSAL, FP8, 0, 2, 0>(a, sbase, bars, tmem, ab);
    } else if (warp == 1 && rank == 0 && pair_s_warps<CAUSAL>() == 2) {
      pair_mma_s<BF16, CAUSAL, FP8, 0, 1, 0>(a, sbase, bars, tmem, ab);
    } else if (warp == 3 && rank == 0) {
      pair_mma_pv<BF16, CAUSAL, FP8>(a, sbase, bars, tmem, ab);
    }
  } else if (wgrp < 3) {
    ptx::setmaxnreg_inc<kRegsSoftmax>();
    pair_softmax<BF16, CAUSAL, FP8>(a, sbase, bars, tmem, stats, rank, ab, warp, lane);
  } else {
    ptx::setmaxnreg_dec<kRegsEpilogue>();
    pair_epilogue<BF16, CAUSAL, FP8>(&tm_o, a, sbase, bars, tmem, stats, rank, ab, warp, lane);
  }
  __syncwarp();
  ptx::tc_fence_before();
  ptx::cluster_sync();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc_pair(tmem, 512);
  if (threadIdx.x == 0 && a.clk != nullptr) clock_end(a.clk, clock_slot);
}

// Host side (fa_fwd_pair.cu): maps = Q ({d, N, H, B}, 64 x 128 boxes), K (64 x 64
// boxes: a K half), V (64 x 128: a V half), O (64 x 32); units of 512 rows
// (a.n_mblk = ceil(N / 512)); grid = 2 x pairs.
cudaError_t launch_fwd_pair(bool bf16, bool causal, const CUtensorMap* maps, const FwdArgs& a,
                            int grid, cudaStream_t stream);
// 8-bit inputs: maps = Q, K ({128 bytes, N, H, B}: 128- / 64-row boxes), V^T
// ({keys, 128, H, B}: 128 keys x 64 rows), O as above.
cudaError_t launch_fwd_pair_fp8(bool causal, const CUtensorMap* maps, const FwdArgs& a, int grid,
                                cudaStream_t stream);
int fwd_smem_bytes_pair(bool fp8 = false);
// Grid of the pair kernel for n_units units: two CTAs per pair, one pair per
// two SMs at most.
inline int fwd_grid_pair(int n_units, int sm_count) {
  const int pairs = n_units < sm_count / 2 ? n_units : sm_count / 2;
  return 2 * (pairs > 0 ? pairs : 1);
}

}  // namespace fa
