// Fused attention forward for sm_103a: TMA loads, tcgen05.mma with S and O
// accumulators in TMEM, online softmax in registers, TMA-store epilogue.
//
// Work unit: 256 query rows of one (batch, head), split into two 128-row
// Q tiles that share every K / V tile (ping-pong: while the softmax of one
// tile runs, the tensor core works on the other). A persistent grid of one
// CTA per SM walks the units.
//
// Warp roles (10 warps, 320 threads):
//   warp 0      TMA producer: Q tiles, then K_j, V_j into a ring of stages
//               (the producer loop of "TMA + Warp Specialization", 17.4).
//   warp 1      TMEM owner and single-thread MMA issuer (tcgen05.mma is
//               issued by one thread, "TCA 51%, MFU below 8%", B200 section).
//   warps 2-5   softmax for Q tile 0 (one thread per row = TMEM lane, as in
//               the B300 walkthrough, V14 item d).
//   warps 6-9   softmax for Q tile 1.
// A softmax warpgroup is four consecutive warps, so its warps cover the four
// TMEM lane quarters (warp w reaches lanes 32*(w%4)..+31).
//
// The MMA thread issues S0 = Q0 K_0^T, S1 = Q1 K_0^T, then per KV tile j, in order,
//   O0 += P0 V_j, S0 = Q0 K_{j+1}^T, O1 += P1 V_j, S1 = Q1 K_{j+1}^T
// Tensor-core ops of one thread execute in issue order, so S_i(j+1) may reuse
// the S_i columns right after the PV that consumed P_i(j).
//
// Online softmax in base 2 (c = scale * log2 e): m_new = max(m_ref, c * max s);
// the reference max m_ref is only moved (and O, l rescaled by
// 2^(m_ref - m_new)) when m_new exceeds it by more than 8, so most tiles skip
// the TMEM round trip of O that the B300 walkthrough names as an overhead
// (V17 discussion). Exact in real arithmetic: l and O share m_ref, and
// p <= 2^8 keeps fp16 / bf16 P and fp32 sums far from overflow.
#pragma once

#include <cuda.h>

#include "fa_common.cuh"

namespace fa {

struct FwdArgs {
  float* lse;        // [BH][N] fp32, natural-log logsumexp
  uint32_t* status;  // device status word (timeouts)
  int N;             // sequence length
  int BH;            // batch * heads
  int n_mblk;        // 256-row units per head: ceil(N / 256)
  int n_units;       // BH * n_mblk
  int n_kv;          // 128-key tiles per head: ceil(N / 128)
  float scale_log2;  // scale * log2(e)
};

template <int D>
struct Layout {
  static constexpr int kPanels = D / 64;                   // 128-byte panels per row
  static constexpr int kTileBytes = kPanels * kPanelBytes;  // a Q, K, V or O tile
  static constexpr int kPBytes = 2 * kPanelBytes;           // P tile: 128 x 128 16-bit
  static constexpr int kStages = (D == 128) ? 3 : 6;        // K / V ring slots
  static constexpr int kOffQ = 0;                           // Q0, Q1
  static constexpr int kOffP = 2 * kTileBytes;              // P0, P1 (also O staging)
  static constexpr int kOffKV = kOffP + 2 * kPBytes;        // ring
  static constexpr int kOffBar = kOffKV + kStages * kTileBytes;
  static constexpr int kSmemBytes = kOffBar + 256 + 1024;  // barriers + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;    // S_i at columns i*128
  static constexpr uint32_t kColO = 256;  // O_i at columns 256 + i*D
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// Barrier slots (8 bytes each) in the barrier block.
enum BarSlot : int {
  kBarQFull = 0,    // [2] TMA: Q_i landed
  kBarQEmpty = 2,   // MMA: all S MMAs of the unit done (Q tiles reusable)
  kBarSFull = 3,    // [2] MMA: S_i ready in TMEM
  kBarPFull = 5,    // [2] 128 softmax threads: P_i in smem, O_i rescaled
  kBarPVDone = 7,   // [2] MMA: O_i += P_i V done (P_i, O_i reusable)
  kBarEpiFull = 9,  // [2] 128 softmax threads: O_i staged in smem
  kBarEpiFree = 11, // [2] store thread: staged O_i read by the TMA store
  kBarDrain = 13,   // MMA: every tcgen05 op of the CTA completed
  kBarKVFull = 14,  // [stages] TMA: ring slot loaded
};
constexpr int kSlotTmem = 224;   // byte offset of the TMEM base address
constexpr int kSlotAbort = 228;  // byte offset of the abort flag

// Walks this CTA's units: round k takes unit k*G + c; for causal problems odd
// rounds go in reverse CTA order so per-CTA work evens out over the
// longest-first unit order.
template <bool CAUSAL>
__device__ __forceinline__ bool next_unit(int& round, const FwdArgs& a, int& bh, int& mblk) {
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
      // longest first: all heads of the last row block, then the one before
      const int lvl = static_cast<int>(u / a.BH);
      bh = static_cast<int>(u - static_cast<long long>(lvl) * a.BH);
      mblk = a.n_mblk - 1 - lvl;
    } else {
      // head-major, so concurrently running CTAs share K / V in L2
      bh = static_cast<int>(u / a.n_mblk);
      mblk = static_cast<int>(u - static_cast<long long>(bh) * a.n_mblk);
    }
    return true;
  }
}

// KV tiles a unit visits: all of them, or (causal) up to the diagonal of its
// second Q tile. Both Q tiles visit the same tiles; the first tile's last one
// is then fully masked.
template <bool CAUSAL>
__device__ __forceinline__ int unit_kv_tiles(const FwdArgs& a, int mblk) {
  return CAUSAL ? min(2 * mblk + 2, a.n_kv) : a.n_kv;
}

template <int D, bool BF16, bool CAUSAL>
__device__ __forceinline__ void producer_role(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                              const CUtensorMap* tm_v, const FwdArgs& a,
                                              uint32_t sbase, uint32_t bars, const AbortCtx& ab) {
  using L = Layout<D>;
  constexpr int S = L::kStages;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  ptx::prefetch_tmap(tm_q);
  ptx::prefetch_tmap(tm_k);
  ptx::prefetch_tmap(tm_v);
  uint32_t ring = 0, units = 0;
  int round = 0, bh = 0, mblk = 0;
  bool ok = true;
  while (ok && next_unit<CAUSAL>(round, a, bh, mblk)) {
    const int nkv = unit_kv_tiles<CAUSAL>(a, mblk);
    if (!wait_bounded(bar(kBarQEmpty), (units & 1u) ^ 1u, ab, kStatusProducer)) {
      ok = false;
      break;
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_arrive_expect_tx(bar(kBarQFull + i), L::kTileBytes);
      for (int p = 0; p < L::kPanels; ++p)
        ptx::tma_load_3d(sbase + L::kOffQ + i * L::kTileBytes + p * kPanelBytes, tm_q,
                         bar(kBarQFull + i), 64 * p, mblk * 256 + 128 * i, bh);
    }
    ++units;
    for (int j = 0; j < nkv && ok; ++j) {
      for (int t = 0; t < 2; ++t) {
        const uint32_t s = ring % S, ph = (ring / S) & 1u;
        if (!wait_bounded(bar(kBarKVFull + S + s), ph ^ 1u, ab, kStatusProducer)) {
          ok = false;
          break;
        }
        ptx::mbar_arrive_expect_tx(bar(kBarKVFull + s), L::kTileBytes);
        const CUtensorMap* tm = t ? tm_v : tm_k;
        for (int p = 0; p < L::kPanels; ++p)
          ptx::tma_load_3d(sbase + L::kOffKV + s * L::kTileBytes + p * kPanelBytes, tm,
                           bar(kBarKVFull + s), 64 * p, 128 * j, bh);
        ++ring;
      }
    }
  }
  if (!ok) {
    // Let the copies already issued land before the CTA exits.
    for (uint32_t s = 0; s < static_cast<uint32_t>(S) && s < ring; ++s) {
      const uint32_t last = ring - 1 - ((ring - 1 - s) % S);  // last load into slot s
      wait_drain(bar(kBarKVFull + s), (last / S) & 1u, ab, kStatusDrain);
    }
    if (units > 0) {
      wait_drain(bar(kBarQFull + 0), (units - 1) & 1u, ab, kStatusDrain);
      wait_drain(bar(kBarQFull + 1), (units - 1) & 1u, ab, kStatusDrain);
    }
  }
}

template <int D, bool BF16, bool CAUSAL>
__device__ __forceinline__ void mma_role(const FwdArgs& a, uint32_t sbase, uint32_t bars,
                                         uint32_t tmem, const AbortCtx& ab) {
  using L = Layout<D>;
  constexpr int S = L::kStages;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  const uint32_t sQ[2] = {sbase + L::kOffQ, sbase + L::kOffQ + L::kTileBytes};
  const uint32_t sP[2] = {sbase + L::kOffP, sbase + L::kOffP + L::kPBytes};
  const uint32_t tS[2] = {tmem + L::kColS, tmem + L::kColS + 128};
  const uint32_t tO[2] = {tmem + L::kColO, tmem + L::kColO + D};
  auto slot = [&](uint32_t idx) { return sbase + L::kOffKV + (idx % S) * L::kTileBytes; };
  uint32_t ring = 0, units = 0, pcnt[2] = {0u, 0u};
  int round = 0, bh = 0, mblk = 0;
  bool ok = true;
  while (ok && next_unit<CAUSAL>(round, a, bh, mblk)) {
    const int nkv = unit_kv_tiles<CAUSAL>(a, mblk);
    ok = wait_bounded(bar(kBarQFull + 0), units & 1u, ab, kStatusMma) &&
         wait_bounded(bar(kBarQFull + 1), units & 1u, ab, kStatusMma);
    if (!ok) break;
    ++units;
    // S_i(0) = Q_i K_0^T
    const uint32_t k0 = ring++;
    if (!(ok = wait_bounded(bar(kBarKVFull + k0 % S), (k0 / S) & 1u, ab, kStatusMma))) break;
    ptx::tc_fence_after();
    issue_qk<D, BF16>(tS[0], sQ[0], slot(k0));
    ptx::umma_commit(bar(kBarSFull + 0));
    issue_qk<D, BF16>(tS[1], sQ[1], slot(k0));
    ptx::umma_commit(bar(kBarSFull + 1));
    ptx::umma_commit(bar(kBarKVFull + S + k0 % S));
    if (nkv == 1) ptx::umma_commit(bar(kBarQEmpty));
    for (int j = 0; j < nkv; ++j) {
      const uint32_t vj = ring++;
      if (!(ok = wait_bounded(bar(kBarKVFull + vj % S), (vj / S) & 1u, ab, kStatusMma))) break;
      const bool more = j + 1 < nkv;
      const uint32_t kn = more ? ring : 0u;
      // Q tile 0: O0 += P0 V_j, then S0 = Q0 K_{j+1}^T
      if (!(ok = wait_bounded(bar(kBarPFull + 0), (pcnt[0]++) & 1u, ab, kStatusMma))) break;
      ptx::tc_fence_after();
      issue_pv<D, BF16>(tO[0], sP[0], slot(vj), j > 0);
      ptx::umma_commit(bar(kBarPVDone + 0));
      if (more) {
        ++ring;
        if (!(ok = wait_bounded(bar(kBarKVFull + kn % S), (kn / S) & 1u, ab, kStatusMma))) break;
        ptx::tc_fence_after();
        issue_qk<D, BF16>(tS[0], sQ[0], slot(kn));
        ptx::umma_commit(bar(kBarSFull + 0));
      }
      // Q tile 1: O1 += P1 V_j, then S1 = Q1 K_{j+1}^T
      if (!(ok = wait_bounded(bar(kBarPFull + 1), (pcnt[1]++) & 1u, ab, kStatusMma))) break;
      ptx::tc_fence_after();
      issue_pv<D, BF16>(tO[1], sP[1], slot(vj), j > 0);
      ptx::umma_commit(bar(kBarPVDone + 1));
      ptx::umma_commit(bar(kBarKVFull + S + vj % S));
      if (more) {
        issue_qk<D, BF16>(tS[1], sQ[1], slot(kn));
        ptx::umma_commit(bar(kBarSFull + 1));
        ptx::umma_commit(bar(kBarKVFull + S + kn % S));
        if (j + 2 == nkv) ptx::umma_commit(bar(kBarQEmpty));
      }
    }
  }
  // Every tcgen05 op this thread issued must finish before TMEM is freed.
  ptx::umma_commit(bar(kBarDrain));
  wait_drain(bar(kBarDrain), 0u, ab, kStatusDrain);
}

template <int D, bool BF16, bool CAUSAL>
__device__ __forceinline__ void softmax_role(const CUtensorMap* tm_o, const FwdArgs& a,
                                             uint32_t sbase, uint32_t bars, uint32_t tmem,
                                             const AbortCtx& ab, int warp, int lane) {
  using L = Layout<D>;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  const int wg = (warp - 2) >> 2;           // which Q tile
  const int r = (warp & 3) * 32 + lane;     // row in the tile = TMEM lane
  const uint32_t tl = ptx::tmem_lane_base(tmem, warp);
  const uint32_t tS = tl + L::kColS + 128u * wg;
  const uint32_t tO = tl + L::kColO + static_cast<uint32_t>(D) * wg;
  const uint32_t sP = sbase + L::kOffP + L::kPBytes * wg;  // P tile, then O staging
  const bool store_thread = (warp == 2 + 4 * wg) && lane == 0;
  const float cl2 = a.scale_log2;
  uint32_t scnt = 0, pvcnt = 0, units = 0;
  int round = 0, bh = 0, mblk = 0;
  bool ok = true;
  while (ok && next_unit<CAUSAL>(round, a, bh, mblk)) {
    const int nkv = unit_kv_tiles<CAUSAL>(a, mblk);
    const int tile_row0 = mblk * 256 + 128 * wg;
    const int grow = tile_row0 + r;
    // l: sum of the P weights that normalises O; l_exp: sum of the unrounded
    // exponentials, for the LSE. They differ only for bf16 (see below).
    float m_ref = -INFINITY, l = 0.f, l_exp = 0.f;
    for (int j = 0; j < nkv; ++j) {
      if (!(ok = wait_bounded_warp(bar(kBarSFull + wg), (scnt++) & 1u, ab, kStatusSoftmax))) break;
      ptx::tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) ptx::tmem_ld32(tS + 32u * c, sr[c]);
#pragma unroll
      for (int c = 0; c < 4; ++c) ptx::tmem_ld_wait(sr[c]);
      float s[128];
#pragma unroll
      for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c >> 5][c & 31]);
      // Mask keys past the end of the sequence and (causal) past the row.
      const int k0 = j * kTileRows;
      const bool need_mask = (k0 + kTileRows > a.N) || (CAUSAL && k0 + kTileRows - 1 > tile_row0);
      if (need_mask) {
        int lim = a.N - k0;
        if (CAUSAL) lim = min(lim, grow - k0 + 1);
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = (c < lim) ? s[c] : -INFINITY;
      }
      float mx[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
      for (int c = 4; c < 128; c += 4) {
        mx[0] = fmaxf(mx[0], s[c]);
        mx[1] = fmaxf(mx[1], s[c + 1]);
        mx[2] = fmaxf(mx[2], s[c + 2]);
        mx[3] = fmaxf(mx[3], s[c + 3]);
      }
      const float m_tile = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * cl2;
      const float m_new = fmaxf(m_ref, m_tile);
      float alpha = 1.f;
      if (j == 0) {
        m_ref = m_new;
      } else if (m_new > m_ref + 8.f) {
        alpha = ptx::ex2(m_ref - m_new);
        m_ref = m_new;
      }
      const float neg = -m_ref;
      uint32_t pk[64];
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
      float lr[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float p0 = ptx::ex2(fmaf(s[2 * c], cl2, neg));
        const float p1 = ptx::ex2(fmaf(s[2 * c + 1], cl2, neg));
        pk[c] = pack2<BF16>(p0, p1);
        ls[c & 3] += p0 + p1;
        if constexpr (BF16) {
          // bf16 P carries 8 significant bits: O is normalised by the sum of
          // the rounded weights the PV product actually uses (a row dominated
          // by one key then returns that V row exactly), while the LSE keeps
          // the unrounded sum.
          lr[c & 3] += __uint_as_float(pk[c] << 16) + __uint_as_float(pk[c] & 0xFFFF0000u);
        }
      }
      const float lsum = (ls[0] + ls[1]) + (ls[2] + ls[3]);
      const float lsum_p = BF16 ? (lr[0] + lr[1]) + (lr[2] + lr[3]) : lsum;
      if (j > 0) {
        // O_i must hold PV(j-1) before it is rescaled, and P_i must be free.
        if (!(ok = wait_bounded_warp(bar(kBarPVDone + wg), (pvcnt++) & 1u, ab, kStatusSoftmax)))
          break;
        ptx::tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            ptx::tmem_ld32(tO + 32u * c, o);
            ptx::tmem_ld_wait(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            ptx::tmem_st32(tO + 32u * c, o);
          }
          ptx::tmem_st_wait();
        }
      } else if (units > 0) {
        // P_i doubles as the previous unit's O staging: wait for its store.
        if (!(ok = wait_bounded_warp(bar(kBarEpiFree + wg), (units - 1) & 1u, ab, kStatusSoftmax)))
          break;
      }
      l = l * alpha + lsum_p;
      l_exp = l_exp * alpha + lsum;
      store_row128_sw128(sP, r, pk);
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(kBarPFull + wg));
    }
    if (!ok) break;
    // Epilogue: O_i / l -> 16-bit -> staging (SW128) -> TMA store; LSE.
    if (!(ok = wait_bounded_warp(bar(kBarPVDone + wg), (pvcnt++) & 1u, ab, kStatusSoftmax))) break;
    ptx::tc_fence_after();
    const float inv_l = 1.f / l;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      ptx::tmem_ld32(tO + 32u * c, o);
      ptx::tmem_ld_wait(o);
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e)
        pk[e] = pack2<BF16>(__uint_as_float(o[2 * e]) * inv_l, __uint_as_float(o[2 * e + 1]) * inv_l);
      store_row32_sw128(sP, r, 32 * c, pk);
    }
    if (grow < a.N)
      a.lse[static_cast<size_t>(bh) * a.N + grow] = (m_ref + log2f(l_exp)) * 0.69314718055994531f;
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    ptx::mbar_arrive(bar(kBarEpiFull + wg));
    if (store_thread) {
      if (wait_bounded(bar(kBarEpiFull + wg), units & 1u, ab, kStatusEpilogue)) {
        if (tile_row0 < a.N) {  // a tile wholly past N (odd tile count) has nothing to store
          for (int p = 0; p < L::kPanels; ++p)
            ptx::tma_store_3d(tm_o, sP + p * kPanelBytes, 64 * p, tile_row0, bh);
          ptx::bulk_commit();
          ptx::bulk_wait_read_all();
        }
        ptx::mbar_arrive(bar(kBarEpiFree + wg));
      } else {
        ok = false;
      }
    }
    __syncwarp();
    ++units;
  }
  if (store_thread) ptx::bulk_wait_all();
}

template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(320, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  const FwdArgs a) {
  using L = Layout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - raw);
  const uint32_t bars = sbase + L::kOffBar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sgen + L::kOffBar + kSlotTmem);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(sgen + L::kOffBar + kSlotAbort);
  const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
  const AbortCtx ab{abort_flag, a.status};
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(bar(kBarQFull + i), 1);
      ptx::mbar_init(bar(kBarSFull + i), 1);
      ptx::mbar_init(bar(kBarPFull + i), 128);
      ptx::mbar_init(bar(kBarPVDone + i), 1);
      ptx::mbar_init(bar(kBarEpiFull + i), 128);
      ptx::mbar_init(bar(kBarEpiFree + i), 1);
    }
    ptx::mbar_init(bar(kBarQEmpty), 1);
    ptx::mbar_init(bar(kBarDrain), 1);
    for (int s = 0; s < L::kStages; ++s) {
      ptx::mbar_init(bar(kBarKVFull + s), 1);
      ptx::mbar_init(bar(kBarKVFull + L::kStages + s), 1);
    }
    *abort_flag = 0u;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), L::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) producer_role<D, BF16, CAUSAL>(&tm_q, &tm_k, &tm_v, a, sbase, bars, ab);
  } else if (warp == 1) {
    if (lane == 0) mma_role<D, BF16, CAUSAL>(a, sbase, bars, tmem, ab);
  } else {
    softmax_role<D, BF16, CAUSAL>(&tm_o, a, sbase, bars, tmem, ab, warp, lane);
  }
  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, L::kTmemCols);
}

// Host-side launch of one instance (defined in the per-head-dim files).
cudaError_t launch_fwd_d64(bool bf16, bool causal, const CUtensorMap* maps, const FwdArgs& a,
                           int grid, cudaStream_t stream);
cudaError_t launch_fwd_d128(bool bf16, bool causal, const CUtensorMap* maps, const FwdArgs& a,
                            int grid, cudaStream_t stream);
int fwd_smem_bytes(int d);
constexpr int kFwdThreads = 320;

}  // namespace fa
