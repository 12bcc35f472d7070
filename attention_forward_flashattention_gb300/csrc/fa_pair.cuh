// Fused attention forward on CTA pairs (tcgen05.mma cta_group::2), head
// dimension 128, fp16 / bf16: the "CTA pair" of "TMA + Warp Specialization"
// (CUDA book ch. 17), section 17.9, item 3 -- two SMs share each tensor-core
// product, which makes the tile per product larger (M = 256 query rows).
//
// Work unit: 256 query rows of one (batch, head); the even CTA of the pair
// holds rows 0-127 of the unit, the odd CTA rows 128-255. One M = 256 product
// covers both: each CTA supplies its own 128 rows of the A operand (Q, or P
// from its tensor memory) and HALF of the B operand (64 of the 128 keys of a
// K tile, 64 of the 128 columns of a V tile), and receives its own 128 rows
// of the result in its tensor memory. So each SM reads half of every K / V
// tile from L2 and holds half of it in shared memory, and its tensor memory
// holds only one 128-row tile's S and O, which leaves room for
//   S in two buffers (S(j+2) is computed while the softmax of S(j+1) runs),
//   P in two buffers of its own columns (P(j+1) is written while PV(j) runs),
// so no product waits for another to release columns; only the softmax sets
// the pace of a step.
//
// Warp roles (16 warps), the same in both CTAs unless noted:
//   warp 0 (one lane): TMA producer: its Q tile (two 128-row x 64-column
//           panels), then per KV tile its K half (64 keys) and V half (64
//           columns), counted on the EVEN CTA's barriers;
//   warp 1: TMEM owner; in the even CTA the MMA issuer (whole warp, elected
//           lane) of every pair product and commit;
//   warps 4-7 / 8-11: softmax of keys 0-63 / 64-127 of every KV tile for the
//           CTA's 128 rows (one thread per row and half); the two halves
//           exchange their partial row maxima through shared memory, so both
//           use the same reference maximum and the same lazy-rescale choice;
//   warps 12-15: epilogue (O / l, LSE, TMA store of the CTA's 128 rows).
// Barriers that collect arrivals from both CTAs (TMA bytes, S read, P
// written, O drained) live in the even CTA; products signal both CTAs by
// multicast commits. Every wait is bounded (1 s), as in the one-CTA kernel.
#pragma once

#include <cuda.h>

#include "fa_kernel.cuh"

namespace fa {

struct PairLayout {
  static constexpr int kQBytes = 2 * kPanelBytes;            // 128 rows x 128 columns
  static constexpr int kSlotBytes = kPanelBytes;             // a K half or a V half
  static constexpr int kStages = 8;                          // ring slots
  static constexpr int kOffQ = 0;                            // two Q buffers
  static constexpr int kOffKV = 2 * kQBytes;
  static constexpr int kOffStats = kOffKV + kStages * kSlotBytes;  // [2][128] l, [2][128] l_exp, [128] m
  static constexpr int kOffXMax = kOffStats + 5 * 128 * 4;         // [2 steps][2 halves][128]
  static constexpr int kOffOut = ((kOffXMax + 4 * 128 * 4 + 1023) / 1024) * 1024;
  static constexpr int kOutSliceBytes = 32 * 128;                  // per epilogue warp
  static constexpr int kOffBar = kOffOut + 4 * kOutSliceBytes;
  static constexpr int kSmemBytes = kOffBar + 512 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kOffBar % 8 == 0, "barrier block alignment");
  // TMEM columns (fp32, lane = row of this CTA's tile)
  static constexpr uint32_t kColS = 0;    // S buffer b at b * 128
  static constexpr uint32_t kColP = 256;  // P buffer b at 256 + b * 64 (two 16-bit keys per column)
  static constexpr uint32_t kColO = 384;  // O: 128 columns
};

enum PairBar : int {
  kPbQFull = 0,      // [2] even CTA: both CTAs' Q tiles landed (bytes)
  kPbQEmpty = 2,     // [2] both: the unit's last S product done (multicast commit)
  kPbSFull = 4,      // [2] both: S buffer b ready (multicast commit)
  kPbSFree = 6,      // [2] even CTA: S buffer b read by the 16 softmax warps of the pair
  kPbPFull = 8,      // [2] even CTA: P buffer b written by the 16 softmax warps
  kPbPFree = 10,     // [2] both: PV using P buffer b done, O updated (multicast commit)
  kPbOFull = 12,     // both: the unit's last PV done (multicast commit)
  kPbOFree = 13,     // even CTA: O read by the 8 epilogue warps of the pair
  kPbStatsFull = 14, // both, local: 256 softmax threads wrote the row sums
  kPbStatsFree = 15, // both, local: 128 epilogue threads read them
  kPbDrain = 16,     // even CTA: every product of the issuer completed
  kPbKVFull = 17,    // [stages] even CTA: both halves of a ring slot landed; then [stages] slot free (both)
  kPbXchg = 33,      // [2] both, local: the 8 softmax warps wrote their partial row maxima
};
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

// Waits for this CTA's barrier `bar` (which receives arrivals from the peer
// or multicast commits): every lane polls, the warp leaves together.
__device__ __forceinline__ bool pair_wait_warp(uint32_t bar, uint32_t parity, const AbortCtx& ab,
                                               uint32_t code) {
  return wait_cluster_warp(bar, parity, ab, code);
}

template <bool CAUSAL>
__device__ __forceinline__ void pair_producer(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                              const CUtensorMap* tm_v, const FwdArgs& a,
                                              uint32_t sbase, uint32_t bars, uint32_t rank,
                                              const AbortCtx& ab) {
  using L = PairLayout;
  constexpr int S = L::kStages;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  auto lead = [&](int i) { return ptx::mapa_shared(bar(i), 0); };  // the even CTA's barrier
  ptx::prefetch_tmap(tm_q);
  ptx::prefetch_tmap(tm_k);
  ptx::prefetch_tmap(tm_v);
  uint32_t ring = 0, units = 0;
  int round = 0, bh = 0, mblk = 0;
  bool ok = true;
  while (ok && next_pair_unit<CAUSAL>(round, a, bh, mblk)) {
    const int nkv = unit_kv_tiles<CAUSAL>(a, mblk);
    const uint32_t qb = units & 1u;
    if (!(ok = wait_cluster<false>(bar(kPbQEmpty + qb), ((units >> 1) & 1u) ^ 1u, ab,
                                   kStatusProducer)))
      break;
    const int hh = bh % a.H, bb = bh / a.H;
    if (rank == 0) ptx::mbar_arrive_expect_tx(bar(kPbQFull + qb), 2 * L::kQBytes);
    for (int p = 0; p < 2; ++p)
      ptx::tma_load_4d_pair(sbase + L::kOffQ + qb * L::kQBytes + p * kPanelBytes, tm_q,
                            lead(kPbQFull + qb), 64 * p,
                            mblk * 256 + 128 * static_cast<int>(rank), hh, bb);
    ++units;
    for (int j = 0; j < nkv && ok; ++j) {
      for (int t = 0; t < 2; ++t) {
        const uint32_t s = ring % S, ph = (ring / S) & 1u;
        if (!(ok = wait_cluster<false>(bar(kPbKVFull + S + s), ph ^ 1u, ab, kStatusProducer)))
          break;
        if (rank == 0) ptx::mbar_arrive_expect_tx(bar(kPbKVFull + s), 2 * L::kSlotBytes);
        const uint32_t dst = sbase + L::kOffKV + s * L::kSlotBytes;
        if (t == 0) {  // K: keys 128 j + 64 rank .. +63, two 64-row panels
          for (int p = 0; p < 2; ++p)
            ptx::tma_load_4d_pair(dst + p * (kPanelBytes / 2), tm_k, lead(kPbKVFull + s), 64 * p,
                                  128 * j + 64 * static_cast<int>(rank), hh, bb);
        } else {       // V: keys 128 j .. +127, columns 64 rank .. +63
          ptx::tma_load_4d_pair(dst, tm_v, lead(kPbKVFull + s), 64 * static_cast<int>(rank),
                                128 * j, hh, bb);
        }
        ++ring;
      }
    }
  }
  if (!ok && rank == 0) {
    // let the copies already issued (both CTAs' halves) land before exit
    for (uint32_t s = 0; s < static_cast<uint32_t>(S) && s < ring; ++s) {
      const uint32_t last = ring - 1 - ((ring - 1 - s) % S);
      wait_drain(bar(kPbKVFull + s), (last / S) & 1u, ab, kStatusDrain);
    }
    if (units > 0) {
      const uint32_t qb = (units - 1) & 1u;
      wait_drain(bar(kPbQFull + qb), ((units - 1) >> 1) & 1u, ab, kStatusDrain);
    }
  }
}

// Even CTA, whole warp: every pair product. Per unit: S(0), S(1), then for
// each KV tile j: S(j + 2) as soon as the softmax has read S(j) (its buffer)
// and K(j + 2) has landed, then PV(j) once P(j) is written. So the scores two
// tiles ahead are computed while the softmax of the current tile runs.
template <bool BF16, bool CAUSAL>
__device__ __forceinline__ void pair_mma(const FwdArgs& a, uint32_t sbase, uint32_t bars,
                                         uint32_t tmem, const AbortCtx& ab) {
  using L = PairLayout;
  constexpr int S = L::kStages;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  constexpr uint32_t kIdS = ptx::idesc_f16(BF16, false, 256, 128);
  constexpr uint32_t kIdPV = ptx::idesc_f16(BF16, true, 256, 128);
  const uint64_t dQ0 = desc_kmajor(sbase + L::kOffQ);
  const uint64_t dK0 = desc_kmajor(sbase + L::kOffKV);
  const uint64_t dV0 = desc_v(sbase + L::kOffKV);
  auto slot_off = [](uint32_t idx) { return (idx % S) * static_cast<uint32_t>(L::kSlotBytes); };
  auto kv_wait = [&](uint32_t idx) {
    return pair_wait_warp(bar(kPbKVFull + idx % S), (idx / S) & 1u, ab, kStatusMma);
  };
  // S(tt) = Q K^T into S buffer tt & 1 (K at ring index kidx)
  auto issue_s = [&](uint32_t tt, uint32_t kidx, uint64_t dq) -> bool {
    const uint32_t b = tt & 1u;
    if (!pair_wait_warp(bar(kPbSFree + b), ((tt >> 1) & 1u) ^ 1u, ab, kStatusMma)) return false;
    if (!kv_wait(kidx)) return false;
    ptx::tc_fence_after();
    uint64_t q = dq, k = desc_add(dK0, slot_off(kidx));
    const uint32_t d = tmem + L::kColS + 128u * b;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      ptx::umma_f16_ss_pair_elect(d, q, k, kIdS, kk > 0 ? 1u : 0u);
      const bool next_panel = (kk & 3) == 3;
      q = desc_add(q, next_panel ? static_cast<uint32_t>(kPanelBytes - 96) : 32u);
      k = desc_add(k, next_panel ? static_cast<uint32_t>(kPanelBytes / 2 - 96) : 32u);
      asm volatile("" : "+l"(q), "+l"(k));
    }
    ptx::umma_commit_pair_elect(bar(kPbSFull + b), 3);
    ptx::umma_commit_pair_elect(bar(kPbKVFull + S + kidx % S), 3);  // K half consumed
    return true;
  };
  uint32_t ring = 0, t = 0, units = 0;
  int round = 0, bh = 0, mblk = 0;
  bool ok = true;
  while (ok && next_pair_unit<CAUSAL>(round, a, bh, mblk)) {
    const int nkv = unit_kv_tiles<CAUSAL>(a, mblk);
    const uint32_t qb = units & 1u;
    if (!(ok = pair_wait_warp(bar(kPbQFull + qb), (units >> 1) & 1u, ab, kStatusMma))) break;
    const uint64_t dq = desc_add(dQ0, qb * static_cast<uint32_t>(L::kQBytes));
    for (int j = 0; j < 2 && j < nkv && ok; ++j) ok = issue_s(t + j, ring + 2u * j, dq);
    if (!ok) break;
    if (nkv <= 2) ptx::umma_commit_pair_elect(bar(kPbQEmpty + qb), 3);
    for (int j = 0; j < nkv; ++j) {
      const uint32_t tt = t + static_cast<uint32_t>(j), b = tt & 1u;
      const uint32_t vi = ring + 2u * static_cast<uint32_t>(j) + 1u;
      if (j + 2 < nkv) {
        if (!(ok = issue_s(tt + 2u, ring + 2u * static_cast<uint32_t>(j + 2), dq))) break;
        if (j + 3 == nkv) ptx::umma_commit_pair_elect(bar(kPbQEmpty + qb), 3);
      }
      if (!(ok = pair_wait_warp(bar(kPbPFull + b), (tt >> 1) & 1u, ab, kStatusMma))) break;
      if (j == 0 && units > 0 &&
          !(ok = pair_wait_warp(bar(kPbOFree), (units - 1) & 1u, ab, kStatusMma)))
        break;
      if (!(ok = kv_wait(vi))) break;
      ptx::tc_fence_after();
      {
        uint64_t v = desc_add(dV0, slot_off(vi));
        const uint32_t p = tmem + L::kColP + 64u * b;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          ptx::umma_f16_ts_pair_elect(tmem + L::kColO, p + 8u * kk, v, kIdPV,
                                      (j > 0 || kk > 0) ? 1u : 0u);
          v = desc_add(v, 2048u);
          asm volatile("" : "+l"(v));
        }
      }
      ptx::umma_commit_pair_elect(bar(kPbPFree + b), 3);
      ptx::umma_commit_pair_elect(bar(kPbKVFull + S + vi % S), 3);  // V half consumed
      if (j + 1 == nkv) ptx::umma_commit_pair_elect(bar(kPbOFull), 3);
    }
    ring += 2u * static_cast<uint32_t>(nkv);
    t += static_cast<uint32_t>(nkv);
    ++units;
  }
  // Every product this warp issued completes before TMEM is freed.
  ptx::umma_commit_pair_elect(bar(kPbDrain), 1);
  wait_drain(bar(kPbDrain), 0u, ab, kStatusDrain);
}

// Softmax of one half (h = 0: keys 0-63 of each KV tile, h = 1: keys 64-127)
// for the CTA's 128 rows, one thread per row.
template <bool BF16, bool CAUSAL>
__device__ __forceinline__ void pair_softmax(const FwdArgs& a, uint8_t* sgen, uint32_t bars,
                                             uint32_t tmem, uint32_t rank, const AbortCtx& ab,
                                             int warp, int lane) {
  using L = PairLayout;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  const int h = (warp >> 2) - 1;
  const int r = (warp & 3) * 32 + lane;
  const uint32_t tl = ptx::tmem_lane_base(tmem, warp);
  float* stats = reinterpret_cast<float*>(sgen + L::kOffStats);
  float* xmax = reinterpret_cast<float*>(sgen + L::kOffXMax);
  const float cl2 = a.scale_log2;
  const float2 c2 = make_float2(cl2, cl2);
  const uint32_t lead_sfree = ptx::mapa_shared(bar(kPbSFree), 0);
  const uint32_t lead_pfull = ptx::mapa_shared(bar(kPbPFull), 0);
  uint32_t t = 0, units = 0;
  int round = 0, bh = 0, mblk = 0;
  bool ok = true;
  while (ok && next_pair_unit<CAUSAL>(round, a, bh, mblk)) {
    const int nkv = unit_kv_tiles<CAUSAL>(a, mblk);
    const int tile_row0 = mblk * 256 + 128 * static_cast<int>(rank);
    const int grow = tile_row0 + r;
    float m_ref = -INFINITY, l = 0.f, l_exp = 0.f;
    for (int j = 0; j < nkv; ++j) {
      const uint32_t tt = t + static_cast<uint32_t>(j), b = tt & 1u;
      if (!(ok = wait_cluster<true>(bar(kPbSFull + b), (tt >> 1) & 1u, ab, kStatusSoftmax))) break;
      if (!(ok = __all_sync(0xffffffffu, ok) != 0)) break;
      ptx::tc_fence_after();
      uint32_t sr[2][32];
      ptx::tmem_ld64(tl + L::kColS + 128u * b + 64u * static_cast<uint32_t>(h), sr);
      ptx::tmem_ld_wait64(sr);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(lead_sfree + 8u * b);  // S buffer b read
      float s[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) s[c] = __uint_as_float(sr[c >> 5][c & 31]);
      const int k0 = j * kTileRows + 64 * h;
      const bool need_mask = (k0 + 64 > a.N) || (CAUSAL && k0 + 63 > tile_row0);
      if (need_mask) {
        int lim = a.N - k0;
        if (CAUSAL) lim = min(lim, grow - k0 + 1);
#pragma unroll
        for (int c = 0; c < 64; ++c) s[c] = (c < lim) ? s[c] : -INFINITY;
      }
      float mx[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) mx[q] = fmaxf(s[2 * q], s[2 * q + 1]);
#pragma unroll
      for (int c = 16; c < 64; c += 16) {
#pragma unroll
        for (int q = 0; q < 8; ++q) mx[q] = ptx::fmax3(mx[q], s[c + 2 * q], s[c + 2 * q + 1]);
      }
      const float mh = fmaxf(ptx::fmax3(mx[0], mx[1], mx[2]),
                             ptx::fmax3(ptx::fmax3(mx[3], mx[4], mx[5]), mx[6], mx[7]));
      // exchange the partial maxima of the two halves (buffer and barrier by
      // step parity, so a half one step ahead never overwrites a value the
      // other has yet to read; a bounded wait, so an aborting half never
      // strands the other)
      float* xm = xmax + b * 256;
      xm[h * 128 + r] = mh;
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(kPbXchg + b));
      if (!(ok = wait_bounded_warp(bar(kPbXchg + b), (tt >> 1) & 1u, ab, kStatusSoftmax))) break;
      const float m_tile = fmaxf(mh, xm[(1 - h) * 128 + r]) * cl2;
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
      for (int q = 0; q < 4; ++q) ls[q] = lr[q] = make_float2(0.f, 0.f);
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float2 x = ptx::ffma2(make_float2(s[2 * c], s[2 * c + 1]), c2, neg2);
        const float p0 = ptx::ex2(x.x), p1 = ptx::ex2(x.y);
        const uint32_t w = pack2<BF16>(p0, p1);
        pk[c] = w;
        ls[c & 3] = ptx::fadd2(ls[c & 3], make_float2(p0, p1));
        if constexpr (BF16) {  // normalise by the weights the product uses
          lr[c & 3].x = ptx::add_f32_bf16_lo(lr[c & 3].x, w);
          lr[c & 3].y = ptx::add_f32_bf16_hi(lr[c & 3].y, w);
        }
      }
      // P buffer b was read by PV(tt - 2)
      if (!(ok = wait_cluster_warp(bar(kPbPFree + b), ((tt >> 1) & 1u) ^ 1u, ab, kStatusSoftmax)))
        break;
      ptx::tc_fence_after();
      ptx::tmem_st32(tl + L::kColP + 64u * b + 32u * static_cast<uint32_t>(h), pk);
      const float2 s01 = ptx::fadd2(ptx::fadd2(ls[0], ls[1]), ptx::fadd2(ls[2], ls[3]));
      const float lsum = s01.x + s01.y;
      float lsum_p = lsum;
      if constexpr (BF16) {
        const float2 r01 = ptx::fadd2(ptx::fadd2(lr[0], lr[1]), ptx::fadd2(lr[2], lr[3]));
        lsum_p = r01.x + r01.y;
      }
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        // O must hold PV(tt - 1) before it is rescaled (and no later PV is
        // issued before this half's P-full arrival)
        const uint32_t pb = (tt - 1u) & 1u;
        if (!(ok = wait_cluster_warp(bar(kPbPFree + pb), ((tt - 1u) >> 1) & 1u, ab,
                                     kStatusSoftmax)))
          break;
        ptx::tc_fence_after();
        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t o[32];
          const uint32_t col = tl + L::kColO + 64u * static_cast<uint32_t>(h) + 32u * c;
          ptx::tmem_ld32(col, o);
          ptx::tmem_ld_wait(o);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 v =
                ptx::fmul2(make_float2(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), a2);
            o[e] = __float_as_uint(v.x);
            o[e + 1] = __float_as_uint(v.y);
          }
          ptx::tmem_st32(col, o);
        }
      }
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(lead_pfull + 8u * b);  // P buffer b written
      l = l * alpha + lsum_p;
      l_exp = l_exp * alpha + lsum;
    }
    if (!ok) break;
    // row sums of this half (and the reference maximum) for the epilogue
    if (units > 0 &&
        !(ok = wait_bounded_warp(bar(kPbStatsFree), (units - 1) & 1u, ab, kStatusSoftmax)))
      break;
    stats[h * 128 + r] = l;
    stats[256 + h * 128 + r] = l_exp;
    if (h == 0) stats[512 + r] = m_ref;
    ptx::mbar_arrive(bar(kPbStatsFull));
    t += static_cast<uint32_t>(nkv);
    ++units;
  }
}

// Epilogue: O / l in 16 bits by TMA store (per-warp 32-row staging slices, as
// the one-CTA kernel), the LSE from both halves' sums, then O-free to the
// even CTA.
template <bool BF16, bool CAUSAL>
__device__ __forceinline__ void pair_epilogue(const CUtensorMap* tm_o, const FwdArgs& a,
                                              uint8_t* sgen, uint32_t sbase, uint32_t bars,
                                              uint32_t tmem, uint32_t rank, const AbortCtx& ab,
                                              int warp, int lane) {
  using L = PairLayout;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  const int w = warp & 3;
  const int r = w * 32 + lane;
  const uint32_t tl = ptx::tmem_lane_base(tmem, warp);
  const float* stats = reinterpret_cast<const float*>(sgen + L::kOffStats);
  const uint32_t slice = sbase + L::kOffOut + static_cast<uint32_t>(w) * L::kOutSliceBytes;
  const uint32_t srow = slice + static_cast<uint32_t>(lane) * 128u;
  const uint32_t sx = static_cast<uint32_t>(lane & 7);
  const uint32_t lead_ofree = ptx::mapa_shared(bar(kPbOFree), 0);
  if (lane == 0) ptx::prefetch_tmap(tm_o);
  bool pending = false;
  uint32_t units = 0;
  int round = 0, bh = 0, mblk = 0;
  bool ok = true;
  while (ok && next_pair_unit<CAUSAL>(round, a, bh, mblk)) {
    const int hh = bh % a.H, bb = bh / a.H;
    ok = wait_cluster<true>(bar(kPbOFull), units & 1u, ab, kStatusEpilogue);
    ok = __all_sync(0xffffffffu, ok) != 0 &&
         wait_bounded_warp(bar(kPbStatsFull), units & 1u, ab, kStatusEpilogue);
    if (!ok) break;
    ptx::tc_fence_after();
    const float l = stats[r] + stats[128 + r];
    const float l_exp = stats[256 + r] + stats[384 + r];
    const float m = stats[512 + r];
    ptx::mbar_arrive(bar(kPbStatsFree));
    const int tile_row0 = mblk * 256 + 128 * static_cast<int>(rank);
    if (tile_row0 + r < a.N)
      a.lse[static_cast<size_t>(bh) * a.N + tile_row0 + r] = (m + log2f(l_exp)) * 0.69314718055994531f;
    const float inv_l = 1.f / l;
    const float2 il2 = make_float2(inv_l, inv_l);
    const int row0 = tile_row0 + 32 * w;
#pragma unroll 1
    for (int p = 0; p < 2; ++p) {
      if (lane == 0 && pending) ptx::bulk_wait_read_all();
      __syncwarp();
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        uint32_t o[32];
        ptx::tmem_ld32(tl + L::kColO + static_cast<uint32_t>(64 * p + 32 * half), o);
        ptx::tmem_ld_wait(o);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float2 v = ptx::fmul2(
              make_float2(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1])), il2);
          pk[e] = pack2<BF16>(v.x, v.y);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
          ptx::st_shared_v4(srow + ((static_cast<uint32_t>(4 * half + q) ^ sx) << 4), pk[4 * q],
                            pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
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
    if (lane == 0) ptx::mbar_arrive_cluster(lead_ofree);  // this warp's rows of O read
    ++units;
  }
  if (lane == 0 && pending) ptx::bulk_wait_all();
}

template <bool BF16, bool CAUSAL>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kFwdThreads, 1)
    fa_fwd_pair_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_o, const FwdArgs a) {
  using L = PairLayout;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - raw);
  const uint32_t bars = sbase + L::kOffBar;
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
      ptx::mbar_init(bar(kPbQFull + i), 1);
      ptx::mbar_init(bar(kPbQEmpty + i), 1);
      ptx::mbar_init(bar(kPbSFull + i), 1);
      ptx::mbar_init(bar(kPbSFree + i), 16);  // 8 softmax warps in each CTA
      ptx::mbar_init(bar(kPbPFull + i), 16);
      ptx::mbar_init(bar(kPbPFree + i), 1);
    }
    ptx::mbar_init(bar(kPbOFull), 1);
    ptx::mbar_init(bar(kPbOFree), 8);          // 4 epilogue warps in each CTA
    ptx::mbar_init(bar(kPbStatsFull), 256);
    ptx::mbar_init(bar(kPbStatsFree), 128);
    ptx::mbar_init(bar(kPbDrain), 1);
    ptx::mbar_init(bar(kPbXchg + 0), 8);      // 8 softmax warps of this CTA
    ptx::mbar_init(bar(kPbXchg + 1), 8);
    for (int s = 0; s < L::kStages; ++s) {
      ptx::mbar_init(bar(kPbKVFull + s), 1);
      ptx::mbar_init(bar(kPbKVFull + L::kStages + s), 1);
    }
    *abort_flag = 0u;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), 512);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();  // both CTAs' barriers exist before any peer arrival
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int wgrp = warp >> 2;
  if (wgrp == 0) {
    if (warp == 0) {
      if (lane == 0) pair_producer<CAUSAL>(&tm_q, &tm_k, &tm_v, a, sbase, bars, rank, ab);
    } else if (warp == 1 && rank == 0) {
      pair_mma<BF16, CAUSAL>(a, sbase, bars, tmem, ab);
    }
  } else if (wgrp < 3) {
    pair_softmax<BF16, CAUSAL>(a, sgen, bars, tmem, rank, ab, warp, lane);
  } else {
    pair_epilogue<BF16, CAUSAL>(&tm_o, a, sgen, sbase, bars, tmem, rank, ab, warp, lane);
  }
  __syncwarp();
  ptx::tc_fence_before();
  ptx::cluster_sync();  // no peer access to this CTA's shared memory or TMEM after this
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc_pair(tmem, 512);
  if (threadIdx.x == 0 && a.clk != nullptr) clock_end(a.clk, clock_slot);
}

// Host side (fa_fwd_pair.cu): maps = Q ({d, N, H, B}, 64 x 128 boxes), K (64 x 64
// boxes), V (64 x 128), O (64 x 32); grid = 2 x pairs.
cudaError_t launch_fwd_pair(bool bf16, bool causal, const CUtensorMap* maps, const FwdArgs& a,
                            int grid, cudaStream_t stream);
int fwd_smem_bytes_pair();
// Grid of the pair kernel for n_units units: two CTAs per pair, one pair per
// two SMs at most.
inline int fwd_grid_pair(int n_units, int sm_count) {
  const int pairs = n_units < sm_count / 2 ? n_units : sm_count / 2;
  return 2 * (pairs > 0 ? pairs : 1);
}

}  // namespace fa
