// Fused attention forward for sm_103a: TMA loads, tcgen05.mma with S, P and O
// in TMEM, online softmax in registers, TMA-store epilogue from TMEM.
//
// Work unit: 256 query rows of one (batch, head), split into two 128-row
// Q tiles that share every K / V tile (ping-pong: while the softmax of one
// tile runs, the tensor core works on the other). A persistent grid of one
// CTA per SM walks the units.
//
// Warp roles (16 warps = 4 warpgroups, 512 threads):
//   WG0  warp 0: TMA producer: Q tiles, then K_j, V_j into a ring of stages
//                (the producer loop of "TMA + Warp Specialization", 17.4).
//        warp 1: TMEM owner and MMA issuer: the whole warp runs the loop and
//                one elected lane issues each tcgen05 op (tcgen05.mma is
//                issued by one thread, "TCA 51%, MFU below 8%", B200 section).
//        warps 2-3 idle, except where P is kept apart from S (d = 64: TMEM
//                columns of its own; 8-bit inputs: shared memory): there
//                the S products come from warp 2 and the PV products from
//                warp 3 (d = 64: tile 0's from warp 3, tile 1's from
//                warp 1; see mma_s_role).
//   WG1  softmax of Q tile 0, one thread per row = TMEM lane (the B300
//        walkthrough, V14 item d);
//   WG2  softmax of Q tile 1;
//   WG3  epilogue of both tiles: O / l (the consumer's last step in "TMA +
//        Warp Specialization", 17.5) from TMEM through a per-warp shared
//        staging slice to global memory by TMA store.
// Each warpgroup's four warps cover the four TMEM lane quarters (warp w
// reaches lanes 32*(w%4)..+31). Registers are rebalanced with setmaxnreg
// (the register reallocation of "TMA + Warp Specialization", 17.4-17.5):
// 72 for WG0, 192 for each softmax WG, 56 for the epilogue, which sums to the
// 128 x 4 the CTA is launched with.
//
// TMEM (512 columns): S0 0-127, S1 128-255, O0 256.., O1 256+D..; at d = 128
// (16-bit) P_i is written by the softmax over the first 64 columns of S_i
// (two 16-bit values per column) and read from there by the O += P V MMA
// (A operand in TMEM). At d = 64, P_i sits in columns 384 + 64 i instead; for
// 8-bit inputs (no columns to spare) it goes through shared memory (see
// mma_s_role).
//
// MMA order at d = 128: S0 = Q0 K_0^T, S1 = Q1 K_0^T, then per KV tile j
//   O0 += P0 V_j, S0 = Q0 K_{j+1}^T, O1 += P1 V_j, S1 = Q1 K_{j+1}^T.
// Tensor-core ops of the issuer execute in issue order, so S_i(j+1) may
// overwrite the S_i / P_i columns right after the PV that consumed P_i(j),
// and the commit that signals S_i(j+1) also implies O_i holds PV_i(j).
//
// The row maximum of each S tile comes from the tensor-memory loads that read
// it (the .red form of tcgen05.ld returns each lane's maximum beside the
// loaded values); only tiles with masked keys take it by compare
// instructions.
//
// Online softmax in base 2 (c = scale * log2 e): m_new = max(m_ref, c * max s);
// the reference max m_ref is only moved (and O, l rescaled by
// 2^(m_ref - m_new)) when m_new exceeds it by more than 8, so most tiles skip
// the TMEM round trip of O that the B300 walkthrough names as an overhead
// (V17 discussion). Exact in real arithmetic: l and O share m_ref, and
// p <= 2^8 keeps fp16 / bf16 P and fp32 sums far from overflow.
#pragma once

#include <cuda.h>

#include "fa.h"
#include "fa_common.cuh"

namespace fa {

struct FwdArgs {
  float* lse;        // [BH][N] fp32, natural-log logsumexp (O goes through its tensor map)
  uint32_t* status;  // device status word (timeouts)
  int N;             // sequence length
  int H;             // heads
  int BH;            // batch * heads
  int n_mblk;        // 256-row units per head: ceil(N / 256)
  int n_units;       // BH * n_mblk
  int n_kv;          // 128-key tiles per head: ceil(N / 128)
  float scale_log2;  // scale * log2(e) (8-bit inputs: times the Q scale)
  const float* k_scales;  // 8-bit inputs: [BH][n_kv] scale of each 128-key block of K
  float v_scale;          // 8-bit inputs: scale of V
  unsigned long long* clk;  // optional [3]: SM clock record of the launch (clock_end), or null
};

constexpr int kFwdThreads = 512;
// setmaxnreg split per thread: WG0, each softmax WG, epilogue WG (sum 512 = 4 x 128).
constexpr uint32_t kRegsWG0 = 72, kRegsSoftmax = 192, kRegsEpilogue = 56;
static_assert(kRegsWG0 + 2 * kRegsSoftmax + kRegsEpilogue == 4 * (65536 / kFwdThreads),
              "register split must equal the launch allocation");

// FP8: e4m3 Q, K and V^T (d = 128 only): a 128-element row is one panel.
template <int D, bool FP8 = false>
struct Layout {
  static_assert(!FP8 || D == 128, "the 8-bit kernel is laid out for head dimension 128");
  static constexpr int kPanels = FP8 ? 1 : D / 64;         // 128-byte panels per row
  static constexpr int kTileBytes = kPanels * kPanelBytes;  // a Q, K or V (V^T) tile
  static constexpr int kStages = (D == 128 && !FP8) ? 4 : 8;  // K / V ring slots
  static constexpr int kOffQ = 0;                           // Q0, Q1
  static constexpr int kOffKV = 2 * kTileBytes;             // ring
  // 8-bit inputs: P_i goes through shared memory (one 128 x 128-byte panel
  // each; tensor memory holds S0, S1, O0, O1 and has no room for it), so
  // S_i(j+1) can be computed while softmax(j) runs and the PV products read
  // both operands from shared memory.
  static constexpr bool kPSmem = FP8;
  static constexpr int kOffP = kOffKV + kStages * kTileBytes;  // P0, P1 (kPSmem)
  static constexpr int kOffStats = kOffP + (kPSmem ? 2 * kTileBytes : 0);  // [2][128] row sums l
  // O staging for the TMA-store epilogue: one 32-row x 128-byte slice per
  // epilogue warp (1024-byte aligned, as the 128-byte swizzle requires)
  static constexpr int kOffOut = kOffStats + 1024;
  static constexpr int kOutSliceBytes = 32 * 128;
  static constexpr int kOffBar = kOffOut + 4 * kOutSliceBytes;
  static constexpr int kSmemBytes = kOffBar + 512 + 1024;  // barriers + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;    // S_i (and P_i unless kSepP) at columns i*128
  static constexpr uint32_t kColO = 256;  // O_i at columns 256 + i*D
  // d = 64 leaves room for P_i in columns of its own (64 each: two 16-bit
  // values per column), so S_i(j+1) can be computed while softmax(j) runs.
  static constexpr bool kSepP = D == 64 && !FP8;
  static constexpr uint32_t kColP = 256 + 2 * D;  // P_i at kColP + i*64 (kSepP)
  // P_i apart from S_i (TMEM columns of its own, or shared memory): S and PV
  // products are issued by separate warps, with S-free / P-free barriers
  static constexpr bool kSplit = kSepP || kPSmem;
  // PV products of the two tiles from two warps (d = 64) or from one (8-bit):
  // same-box A/B with the row maximum from the S loads, d = 64 1179 -> 1198
  // TFLOPS (causal 921 -> 989), 8-bit 1998 -> 1969 (causal 1713 -> 1671)
  static constexpr bool kPvPerTile = kSepP;
  static_assert(!kSplit || kStages % 2 == 0, "kSplit: K tiles in even ring slots, V in odd");
  static_assert(!kSepP || kColP + 128 <= kTmemCols, "TMEM columns");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kOffBar % 8 == 0, "barrier block alignment");
};

// Barrier slots (8 bytes each) in the barrier block.
enum BarSlot : int {
  kBarQFull = 0,      // [2] TMA: Q_i landed
  kBarQEmpty = 2,     // MMA: all S MMAs of the unit done (Q tiles reusable)
  kBarSFull = 3,      // [2] MMA: S_i ready in TMEM (and O_i holds every earlier PV)
  kBarPFull = 5,      // [2] 128 softmax threads: P_i in TMEM, O_i rescaled
  kBarOFull = 7,      // [2] MMA: the unit's last O_i += P_i V done
  kBarOFree = 9,      // [2] 128 epilogue threads: O_i read, may be overwritten
  kBarStatsFull = 11, // [2] 128 softmax threads: row sums l of tile i in smem
  kBarDrain = 13,     // MMA: every tcgen05 op of the CTA completed
  kBarStatsFree = 14, // [2] 128 epilogue threads: row sums of tile i read
  kBarSFree = 16,     // [2] 128 softmax threads: S_i read (kSepP)
  kBarPFree = 18,     // [2] MMA: O_i += P_i V done, P_i reusable (kSepP)
  kBarKVFull = 20,    // [stages] TMA: ring slot loaded; then [stages] ring slot free
  kBarDrainPV = 36,   // [2] PV-issuing warps (kSepP): every tcgen05 op each issued completed
};
constexpr int kSlotTmem = 480;   // byte offset of the TMEM base address
constexpr int kSlotAbort = 484;  // byte offset of the abort flag
constexpr int kSlotClock = 488;  // byte offset of the clock stamp (16 bytes)

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

template <int D, bool BF16, bool CAUSAL, bool FP8>
__device__ __forceinline__ void producer_role(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                              const CUtensorMap* tm_v, const FwdArgs& a,
                                              uint32_t sbase, uint32_t bars, const AbortCtx& ab) {
  using L = Layout<D, FP8>;
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
    if (!wait_spin(bar(kBarQEmpty), (units & 1u) ^ 1u, ab, kStatusProducer)) {
      ok = false;
      break;
    }
    const int hh = bh % a.H, bb = bh / a.H;  // tensor-map coordinates {d, n, h, b}
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_arrive_expect_tx(bar(kBarQFull + i), L::kTileBytes);
      for (int p = 0; p < L::kPanels; ++p)
        ptx::tma_load_4d(sbase + L::kOffQ + i * L::kTileBytes + p * kPanelBytes, tm_q,
                         bar(kBarQFull + i), 64 * p, mblk * 256 + 128 * i, hh, bb);
    }
    ++units;
    for (int j = 0; j < nkv && ok; ++j) {
      for (int t = 0; t < 2; ++t) {
        const uint32_t s = ring % S, ph = (ring / S) & 1u;
        if (!wait_spin(bar(kBarKVFull + S + s), ph ^ 1u, ab, kStatusProducer)) {
          ok = false;
          break;
        }
        ptx::mbar_arrive_expect_tx(bar(kBarKVFull + s), L::kTileBytes);
        const uint32_t dst = sbase + L::kOffKV + s * L::kTileBytes;
        if (FP8 && t) {
          // V^T {keys, d, h, b}: keys 128j.. of all d rows, one 128-byte panel
          ptx::tma_load_4d(dst, tm_v, bar(kBarKVFull + s), 128 * j, 0, hh, bb);
        } else {
          const CUtensorMap* tm = t ? tm_v : tm_k;
          for (int p = 0; p < L::kPanels; ++p)
            ptx::tma_load_4d(dst + p * kPanelBytes, tm, bar(kBarKVFull + s), 64 * p, 128 * j, hh,
                             bb);
        }
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

// One warp issues every tcgen05 instruction through an elected lane. An MMA
// of 128x128x16 keeps the tensor core busy ~64 cycles while its issue costs
// ~40-50, and the queue drains whenever the issuer waits, so the loop keeps
// everything else minimal: descriptors are built once and advanced in place,
// waits are warp-uniform try_waits, commits are elected (a few cycles each,
// against ~47 from a lone thread), and each step commits only what a waiter
// needs. (16-bit, P over S: head dimension 128; the other paths issue from
// mma_s_role / mma_pv_role.)
template <int D, bool BF16, bool CAUSAL>
__device__ __forceinline__ void mma_role(const FwdArgs& a, uint32_t sbase, uint32_t bars,
                                         uint32_t tmem, const AbortCtx& ab) {
  using L = Layout<D, false>;
  static_assert(!L::kSplit, "P over S only");
  constexpr int S = L::kStages;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  const uint64_t dQ[2] = {desc_kmajor(sbase + L::kOffQ),
                          desc_kmajor(sbase + L::kOffQ + L::kTileBytes)};
  const uint64_t dK0 = desc_kmajor(sbase + L::kOffKV);  // ring slot s: + s * kTileBytes
  const uint64_t dV0 = desc_v(sbase + L::kOffKV);  // V as stored ([key][d], MN-major B)
  const uint32_t tS[2] = {tmem + L::kColS, tmem + L::kColS + 128};
  const uint32_t tO[2] = {tmem + L::kColO, tmem + L::kColO + D};
  auto qk = [&](int i, uint64_t dk) { issue_qk_desc<D, BF16, true>(tS[i], dQ[i], dk); };
  auto slot_off = [](uint32_t idx) { return (idx % S) * static_cast<uint32_t>(L::kTileBytes); };
  auto kv_wait = [&](uint32_t idx) {
    return wait_spin_warp(bar(kBarKVFull + idx % S), (idx / S) & 1u, ab, kStatusMma);
  };
  uint32_t ring = 0, units = 0, pcnt[2] = {0u, 0u};
  int round = 0, bh = 0, mblk = 0;
  bool ok = true;
  while (ok && next_unit<CAUSAL>(round, a, bh, mblk)) {
    const int nkv = unit_kv_tiles<CAUSAL>(a, mblk);
    ok = wait_spin_warp(bar(kBarQFull + 0), units & 1u, ab, kStatusMma) &&
         wait_spin_warp(bar(kBarQFull + 1), units & 1u, ab, kStatusMma);
    if (!ok) break;
    // S_i(0) = Q_i K_0^T
    const uint32_t k0 = ring++;
    if (!(ok = kv_wait(k0))) break;
    ptx::tc_fence_after();
    {
      const uint64_t dk = desc_add(dK0, slot_off(k0));
      qk(0, dk);
      ptx::umma_commit_elect(bar(kBarSFull + 0));
      qk(1, dk);
      ptx::umma_commit_elect(bar(kBarSFull + 1));
      ptx::umma_commit_elect(bar(kBarKVFull + S + k0 % S));
      if (nkv == 1) ptx::umma_commit_elect(bar(kBarQEmpty));
    }
    // Slot releases of a step are committed after the next step's first PV is
    // queued, so the path from "P ready" to the tensor core stays short.
    uint32_t rel_v = 0, rel_k = 0;
    bool rel_pending = false;
    for (int j = 0; j < nkv; ++j) {
      const uint32_t vj = ring++;
      if (!(ok = kv_wait(vj))) break;
      const bool more = j + 1 < nkv;
      const uint32_t kn = ring;
      const uint64_t dv = desc_add(dV0, slot_off(vj));
      const uint64_t dk = desc_add(dK0, slot_off(kn));
      for (int i = 0; i < 2; ++i) {
        // O_i += P_i V_j (P_i read from TMEM), then S_i = Q_i K_{j+1}^T
        if (!(ok = wait_spin_warp(bar(kBarPFull + i), (pcnt[i]++) & 1u, ab, kStatusMma))) break;
        if (j == 0 && units > 0 &&
            !(ok = wait_spin_warp(bar(kBarOFree + i), (units - 1) & 1u, ab, kStatusMma)))
          break;
        ptx::tc_fence_after();
        issue_pv_ts_desc<D, BF16, true>(tO[i], tS[i], dv, j > 0);
        if (i == 0 && rel_pending) {
          ptx::umma_commit_elect(bar(kBarKVFull + S + rel_v % S));
          ptx::umma_commit_elect(bar(kBarKVFull + S + rel_k % S));
          rel_pending = false;
        }
        if (!more) {
          if (i == 1) ptx::umma_commit_elect(bar(kBarKVFull + S + vj % S));
          ptx::umma_commit_elect(bar(kBarOFull + i));
          continue;
        }
        if (i == 0 && !(ok = kv_wait(kn))) break;
        qk(i, dk);
        ptx::umma_commit_elect(bar(kBarSFull + i));
        if (i == 1) {
          // V_j and K_{j+1} are both consumed once S1(j+1) completes
          rel_v = vj;
          rel_k = kn;
          rel_pending = true;
          if (j + 2 == nkv) ptx::umma_commit_elect(bar(kBarQEmpty));
        }
      }
      if (!ok) break;
      if (more) ++ring;
    }
    if (rel_pending) {  // (only when the unit ended early on an abort)
      ptx::umma_commit_elect(bar(kBarKVFull + S + rel_v % S));
      ptx::umma_commit_elect(bar(kBarKVFull + S + rel_k % S));
    }
    ++units;
  }
  // Every tcgen05 op this warp issued must finish before TMEM is freed.
  ptx::umma_commit_elect(bar(kBarDrain));
  wait_drain(bar(kBarDrain), 0u, ab, kStatusDrain);
}

// MMA issue when P_i is kept apart from S_i (d = 64: TMEM columns of its
// own; 8-bit: shared memory), split over separate warps on separate SM
// sub-partitions: each tcgen05.mma takes issue cycles from the softmax warps
// sharing its sub-partition, and a softmax warp slowed that way delays its
// whole tile (P-full waits for all four). At d = 64 the S warp issues 8
// products per KV step and each of two PV warps (one per tile) 8; with one
// PV warp for both tiles (16 products) the two softmax warps beside it
// finished ~1700 cycles after their siblings on every step. The 8-bit kernel
// measured faster with one PV warp (kPvPerTile). S products never touch the
// P or O columns, so the warps need no ordering beyond the softmax's own
// barriers:
//   S warp:   S_i(j+1) = Q_i K_{j+1}^T once softmax i has read S_i(j);
//   PV warp(s): O_i += P_i(j) V_j once P_i(j) is written, then P-free (O_i
//             updated, P_i reusable), and O-full after a unit's last one.
// The softmax of tile j+1 never waits for PV(j): only its P store and O
// rescale do. All walk the same K, V ring: K_j at index 2j, V_j at 2j+1 of
// the unit's tiles (so with an even slot count K lands in even slots, V in
// odd ones, and at d = 64 a V slot is free once both PV warps have released
// it).
// (Both roles serve the Q tiles I0 .. I1-1 and drain on barrier DRAIN.)
template <int D, bool BF16, bool CAUSAL, bool FP8, int I0, int I1, int DRAIN>
__device__ __forceinline__ void mma_s_role(const FwdArgs& a, uint32_t sbase, uint32_t bars,
                                           uint32_t tmem, const AbortCtx& ab) {
  using L = Layout<D, FP8>;
  constexpr int S = L::kStages;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  const uint64_t dQ[2] = {desc_kmajor(sbase + L::kOffQ),
                          desc_kmajor(sbase + L::kOffQ + L::kTileBytes)};
  const uint64_t dK0 = desc_kmajor(sbase + L::kOffKV);
  const uint32_t tS[2] = {tmem + L::kColS, tmem + L::kColS + 128};
  auto slot_off = [](uint32_t idx) { return (idx % S) * static_cast<uint32_t>(L::kTileBytes); };
  auto kv_wait = [&](uint32_t idx) {
    return wait_spin_warp(bar(kBarKVFull + idx % S), (idx / S) & 1u, ab, kStatusMma);
  };
  uint32_t ring = 0, units = 0, scnt[2] = {0u, 0u};
  int round = 0, bh = 0, mblk = 0;
  bool ok = true;
  while (ok && next_unit<CAUSAL>(round, a, bh, mblk)) {
    const int nkv = unit_kv_tiles<CAUSAL>(a, mblk);
    ok = wait_spin_warp(bar(kBarQFull + 0), units & 1u, ab, kStatusMma) &&
         wait_spin_warp(bar(kBarQFull + 1), units & 1u, ab, kStatusMma);
    for (int j = -1; ok && j + 1 < nkv; ++j) {
      // S_i(j+1) = Q_i K_{j+1}^T (the first one of all waits for nothing)
      const uint32_t kn = ring + 2u * static_cast<uint32_t>(j + 1);
      if (!(ok = kv_wait(kn))) break;
#pragma unroll
      for (int i = I0; i < I1 && ok; ++i) {
        if (units > 0 || j >= 0)
          ok = wait_spin_warp(bar(kBarSFree + i), (scnt[i]++) & 1u, ab, kStatusMma);
        if (!ok) break;
        ptx::tc_fence_after();
        if constexpr (FP8) issue_qk_fp8<true>(tS[i], dQ[i], desc_add(dK0, slot_off(kn)));
        else issue_qk_desc<D, BF16, true>(tS[i], dQ[i], desc_add(dK0, slot_off(kn)));
        ptx::umma_commit_elect(bar(kBarSFull + i));
      }
      if (!ok) break;
      ptx::umma_commit_elect(bar(kBarKVFull + S + kn % S));  // K_{j+1} consumed
      if (j + 2 == nkv) ptx::umma_commit_elect(bar(kBarQEmpty));
    }
    ring += 2u * static_cast<uint32_t>(nkv);
    ++units;
  }
  // Every tcgen05 op this warp issued must finish before TMEM is freed.
  ptx::umma_commit_elect(bar(DRAIN));
  wait_drain(bar(DRAIN), 0u, ab, kStatusDrain);
}

template <int D, bool BF16, bool CAUSAL, bool FP8, int I0, int I1, int DRAIN>
__device__ __forceinline__ void mma_pv_role(const FwdArgs& a, uint32_t sbase, uint32_t bars,
                                            uint32_t tmem, const AbortCtx& ab) {
  using L = Layout<D, FP8>;
  constexpr int S = L::kStages;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  // V as stored ([key][d], MN-major B), or V^T for 8-bit (K-major)
  const uint64_t dV0 = FP8 ? desc_kmajor(sbase + L::kOffKV) : desc_v(sbase + L::kOffKV);
  const uint64_t dP[2] = {desc_kmajor(sbase + L::kOffP),  // (kPSmem)
                          desc_kmajor(sbase + L::kOffP + L::kTileBytes)};
  const uint32_t tO[2] = {tmem + L::kColO, tmem + L::kColO + D};
  const uint32_t tP[2] = {tmem + L::kColP, tmem + L::kColP + 64};
  auto slot_off = [](uint32_t idx) { return (idx % S) * static_cast<uint32_t>(L::kTileBytes); };
  auto kv_wait = [&](uint32_t idx) {
    return wait_spin_warp(bar(kBarKVFull + idx % S), (idx / S) & 1u, ab, kStatusMma);
  };
  uint32_t ring = 0, units = 0, pcnt[2] = {0u, 0u};
  int round = 0, bh = 0, mblk = 0;
  bool ok = true;
  while (ok && next_unit<CAUSAL>(round, a, bh, mblk)) {
    const int nkv = unit_kv_tiles<CAUSAL>(a, mblk);
    for (int j = 0; j < nkv && ok; ++j) {
      // O_i += P_i(j) V_j
      const uint32_t vj = ring + 2u * static_cast<uint32_t>(j) + 1u;
      if (!(ok = kv_wait(vj))) break;
#pragma unroll
      for (int i = I0; i < I1 && ok; ++i) {
        if (!(ok = wait_spin_warp(bar(kBarPFull + i), (pcnt[i]++) & 1u, ab, kStatusMma))) break;
        if (j == 0 && units > 0 &&
            !(ok = wait_spin_warp(bar(kBarOFree + i), (units - 1) & 1u, ab, kStatusMma)))
          break;
        ptx::tc_fence_after();
        if constexpr (FP8) issue_pv_fp8_ss<true>(tO[i], dP[i], desc_add(dV0, slot_off(vj)), j > 0);
        else issue_pv_ts_desc<D, BF16, true>(tO[i], tP[i], desc_add(dV0, slot_off(vj)), j > 0);
        ptx::umma_commit_elect(bar(kBarPFree + i));
        if (j + 1 == nkv) ptx::umma_commit_elect(bar(kBarOFull + i));
      }
      if (!ok) break;
      ptx::umma_commit_elect(bar(kBarKVFull + S + vj % S));  // V_j consumed by these tiles
    }
    ring += 2u * static_cast<uint32_t>(nkv);
    ++units;
  }
  ptx::umma_commit_elect(bar(DRAIN));
  wait_drain(bar(DRAIN), 0u, ab, kStatusDrain);
}

template <int D, bool BF16, bool CAUSAL, bool FP8>
__device__ __forceinline__ void softmax_role(const FwdArgs& a, uint32_t sbase, uint32_t bars,
                                             uint32_t tmem, float* stats, const AbortCtx& ab,
                                             int warp, int lane) {
  using L = Layout<D, FP8>;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  const int wg = (warp >> 2) - 1;           // which Q tile
  const int r = (warp & 3) * 32 + lane;     // row in the tile = TMEM lane
  const uint32_t tl = ptx::tmem_lane_base(tmem, warp);
  const uint32_t tS = tl + L::kColS + 128u * wg;  // S_i; P_i over its first 64 columns
  // or in columns of its own (kSepP)
  const uint32_t tP = L::kSepP ? tl + L::kColP + 64u * wg : tS;
  // or in shared memory (kPSmem: the A operand of the PV product, K-major)
  const uint32_t sP = sbase + L::kOffP + static_cast<uint32_t>(wg * L::kTileBytes);
  uint32_t pstores = 0;  // P_i stores so far (kSplit: each but the first waits for P-free)
  const uint32_t tO = tl + L::kColO + static_cast<uint32_t>(D) * wg;
  const float cl2 = a.scale_log2;
  uint32_t scnt = 0, units = 0;
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
      // with P apart from S, S_i(j+1) is computed during softmax(j), so S is
      // usually ready: poll (resumes sooner); otherwise suspend, leaving issue
      // slots to the other tile's softmax on the same sub-partition
      if (!(ok = L::kSplit
                     ? wait_spin_warp(bar(kBarSFull + wg), scnt & 1u, ab, kStatusSoftmax)
                     : wait_bounded_warp(bar(kBarSFull + wg), scnt & 1u, ab, kStatusSoftmax)))
        break;
      ++scnt;
      ptx::tc_fence_after();
      // base-2 score scale of this tile (8-bit inputs: times its K block's scale)
      float cj = cl2;
      if constexpr (FP8) cj = cl2 * __ldg(a.k_scales + static_cast<size_t>(bh) * a.n_kv + j);
      const float2 c2j = make_float2(cj, cj);
      // columns 0-63, 64-127, and the row maximum of each half formed by the loads
      uint32_t sr[2][2][32];
      float mx_lo, mx_hi;
      ptx::tmem_ld64_max(tS, sr[0], mx_lo);
      ptx::tmem_ld64_max(tS + 64u, sr[1], mx_hi);
      ptx::tmem_ld_wait64x2(sr[0], sr[1]);
      ptx::tmem_ld_wait_f2(mx_lo, mx_hi);
      if constexpr (L::kSplit) {  // S_i is in registers: S_i(j+1) may overwrite it
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(kBarSFree + wg));
      }
      float s[128];
#pragma unroll
      for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c >> 6][(c >> 5) & 1][c & 31]);
      // Mask keys past the end of the sequence and (causal) past the row.
      const int k0 = j * kTileRows;
      const bool need_mask = (k0 + kTileRows > a.N) || (CAUSAL && k0 + kTileRows - 1 > tile_row0);
      float m_raw = fmaxf(mx_lo, mx_hi);
      if (need_mask) {
        int lim = a.N - k0;
        if (CAUSAL) lim = min(lim, grow - k0 + 1);
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = (c < lim) ? s[c] : -INFINITY;
        // Row max over the visible keys: eight independent chains, elements
        // 2t and 2t + 1 of each 16-element group in chain t.
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
      if constexpr (FP8) {
        // P as e4m3, four keys per 32-bit word (O is normalised by the
        // unrounded sum), into shared memory.
        static_assert(L::kPSmem, "8-bit P goes through shared memory");
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float2 t0 = ptx::ffma2(make_float2(s[4 * c], s[4 * c + 1]), c2j, neg2);
          const float2 t1 = ptx::ffma2(make_float2(s[4 * c + 2], s[4 * c + 3]), c2j, neg2);
          const float p0 = ptx::ex2(t0.x), p1 = ptx::ex2(t0.y);
          const float p2 = ptx::ex2(t1.x), p3 = ptx::ex2(t1.y);
          pk[c] = ptx::pack4_e4m3(p0, p1, p2, p3);
          ls[(2 * c) & 3] = ptx::fadd2(ls[(2 * c) & 3], make_float2(p0, p1));
          ls[(2 * c + 1) & 3] = ptx::fadd2(ls[(2 * c + 1) & 3], make_float2(p2, p3));
        }
        // P_i(j-1) read and O_i updated by its PV before P_i is rewritten
        // (and before the O rescale below)
        if (pstores > 0 &&
            !(ok = wait_spin_warp(bar(kBarPFree + wg), (pstores - 1) & 1u, ab, kStatusSoftmax)))
          break;
        ptx::tc_fence_after();
        ++pstores;
        store_row_panel_sw128(sP, r, pk);
        ptx::fence_proxy_async_smem();  // visible to the tensor core's reads
      } else {
        uint32_t pk[2][32];
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float2 t = ptx::ffma2(make_float2(s[2 * c], s[2 * c + 1]), c2j, neg2);
          const float p0 = ptx::ex2(t.x), p1 = ptx::ex2(t.y);
          const uint32_t w = pack2<BF16>(p0, p1);
          pk[c >> 5][c & 31] = w;
          ls[c & 3] = ptx::fadd2(ls[c & 3], make_float2(p0, p1));
          if constexpr (BF16) {
            // bf16 P carries 8 significant bits: O is normalised by the sum of
            // the rounded weights the PV product actually uses (a row dominated
            // by one key then returns that V row exactly), while the LSE keeps
            // the unrounded sum.
            lr[c & 3].x = ptx::add_f32_bf16_lo(lr[c & 3].x, w);
            lr[c & 3].y = ptx::add_f32_bf16_hi(lr[c & 3].y, w);
          }
        }
        if constexpr (L::kSepP) {
          // P_i(j-1) read and O_i updated by its PV before P_i is rewritten
          // (and before the O rescale below)
          if (pstores > 0 &&
              !(ok = wait_spin_warp(bar(kBarPFree + wg), (pstores - 1) & 1u, ab,
                                    kStatusSoftmax)))
            break;
          ptx::tc_fence_after();
        }
        ++pstores;
        // P_i into TMEM: over the S_i columns this thread has already read, or
        // into its own columns (kSepP)
        ptx::tmem_st32(tP, pk[0]);
        ptx::tmem_st32(tP + 32u, pk[1]);
      }
      const float2 s01 = ptx::fadd2(ptx::fadd2(ls[0], ls[1]), ptx::fadd2(ls[2], ls[3]));
      const float lsum = s01.x + s01.y;
      float lsum_p = lsum;
      if constexpr (BF16 && !FP8) {
        const float2 r01 = ptx::fadd2(ptx::fadd2(lr[0], lr[1]), ptx::fadd2(lr[2], lr[3]));
        lsum_p = r01.x + r01.y;
      }
      // Rescale O_i (it holds PV_i(j-1): the S_i(j) commit came after it).
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
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
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(kBarPFull + wg));
      l = l * alpha + lsum_p;
      l_exp = l_exp * alpha + lsum;
    }
    if (!ok) break;
    if (grow < a.N)
      a.lse[static_cast<size_t>(bh) * a.N + grow] = (m_ref + log2f(l_exp)) * 0.69314718055994531f;
    // One slot per row, and at most one unit ahead of the epilogue: the
    // previous unit's sum must have been read (with a single KV tile per unit
    // this role could otherwise finish two units before the epilogue reads
    // the first, and the epilogue's parity wait would miss a phase).
    if (units > 0 &&
        !(ok = wait_bounded_warp(bar(kBarStatsFree + wg), (units - 1) & 1u, ab, kStatusSoftmax)))
      break;
    stats[wg * 128 + r] = l;
    ptx::mbar_arrive(bar(kBarStatsFull + wg));
    ++units;
  }
}

// Epilogue: O_i / l_i in 16 bits, written by TMA stores. Each warp owns the
// 32 rows of its TMEM lane quarter and a private 32-row staging slice (the
// store's box), so the four warps never wait for one another: per 64-column
// panel a warp reads its rows from TMEM, writes them to its slice in the
// 128-byte swizzled layout, and one lane stores the slice (rows past N are
// clipped by the tensor map). The slice is rewritten only after the
// previous store has read it.
template <int D, bool BF16, bool CAUSAL, bool FP8>
__device__ __forceinline__ void epilogue_role(const CUtensorMap* tm_o, const FwdArgs& a,
                                              uint32_t sbase, uint32_t bars, uint32_t tmem,
                                              const float* stats, const AbortCtx& ab, int warp,
                                              int lane) {
  using L = Layout<D, FP8>;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  const int w = warp & 3;
  const int r = w * 32 + lane;
  const uint32_t tl = ptx::tmem_lane_base(tmem, warp);
  const uint32_t slice = sbase + L::kOffOut + static_cast<uint32_t>(w) * L::kOutSliceBytes;
  const uint32_t srow = slice + static_cast<uint32_t>(lane) * 128u;  // this thread's row
  const uint32_t sx = static_cast<uint32_t>(lane & 7);               // its swizzle
  if (lane == 0) ptx::prefetch_tmap(tm_o);
  bool pending = false;  // (lane 0) a store of this warp may still be reading the slice
  uint32_t units = 0;
  int round = 0, bh = 0, mblk = 0;
  bool ok = true;
  while (ok && next_unit<CAUSAL>(round, a, bh, mblk)) {
    const int hh = bh % a.H, bb = bh / a.H;  // tensor-map coordinates {d, n, h, b}
    for (int i = 0; i < 2 && ok; ++i) {
      ok = wait_bounded_warp(bar(kBarOFull + i), units & 1u, ab, kStatusEpilogue) &&
           wait_bounded_warp(bar(kBarStatsFull + i), units & 1u, ab, kStatusEpilogue);
      if (!ok) break;
      ptx::tc_fence_after();
      const float inv_l = (FP8 ? a.v_scale : 1.f) / stats[i * 128 + r];
      ptx::mbar_arrive(bar(kBarStatsFree + i));
      const float2 il2 = make_float2(inv_l, inv_l);
      const int row0 = mblk * 256 + 128 * i + 32 * w;  // this warp's first row
#pragma unroll 1
      for (int p = 0; p < D / 64; ++p) {
        if (lane == 0 && pending) ptx::bulk_wait_read_all();
        __syncwarp();
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          uint32_t o[32];
          ptx::tmem_ld32(tl + L::kColO + static_cast<uint32_t>(D * i + 64 * p + 32 * h), o);
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
        ptx::fence_proxy_async_smem();  // the slice is visible to the TMA engine
        __syncwarp();
        if (lane == 0 && row0 < a.N) {
          ptx::tma_store_4d(tm_o, slice, 64 * p, row0, hh, bb);
          ptx::bulk_commit();
          pending = true;
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(kBarOFree + i));
    }
    ++units;
  }
  if (lane == 0 && pending) ptx::bulk_wait_all();  // before the CTA's shared memory goes
}

// FP8: e4m3 Q, K, V^T (d = 128), bf16 O (instantiate with BF16 = true).
template <int D, bool BF16, bool CAUSAL, bool FP8 = false>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  const FwdArgs a) {
  using L = Layout<D, FP8>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - raw);
  const uint32_t bars = sbase + L::kOffBar;
  float* stats = reinterpret_cast<float*>(sgen + L::kOffStats);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sgen + L::kOffBar + kSlotTmem);
  volatile uint32_t* abort_flag =
      reinterpret_cast<volatile uint32_t*>(sgen + L::kOffBar + kSlotAbort);
  const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
  const AbortCtx ab{abort_flag, a.status};
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  uint64_t* clock_slot = reinterpret_cast<uint64_t*>(sgen + L::kOffBar + kSlotClock);
  if (threadIdx.x == 0 && a.clk != nullptr) clock_begin(clock_slot);

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(bar(kBarQFull + i), 1);
      ptx::mbar_init(bar(kBarSFull + i), 1);
      ptx::mbar_init(bar(kBarPFull + i), 128);
      ptx::mbar_init(bar(kBarOFull + i), 1);
      ptx::mbar_init(bar(kBarOFree + i), 128);
      ptx::mbar_init(bar(kBarStatsFull + i), 128);
      ptx::mbar_init(bar(kBarStatsFree + i), 128);
      ptx::mbar_init(bar(kBarSFree + i), 128);
      ptx::mbar_init(bar(kBarPFree + i), 1);
    }
    ptx::mbar_init(bar(kBarQEmpty), 1);
    ptx::mbar_init(bar(kBarDrain), 1);
    ptx::mbar_init(bar(kBarDrainPV + 0), 1);
    ptx::mbar_init(bar(kBarDrainPV + 1), 1);
    for (int s = 0; s < L::kStages; ++s) {
      ptx::mbar_init(bar(kBarKVFull + s), 1);
      // kPvPerTile: a V slot (odd) is released by both PV warps, a K slot by the S warp
      ptx::mbar_init(bar(kBarKVFull + L::kStages + s), (L::kPvPerTile && (s & 1)) ? 2 : 1);
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

  const int wgrp = warp >> 2;
  if (wgrp == 0) {
    ptx::setmaxnreg_dec<kRegsWG0>();
    if (warp == 0) {
      if (lane == 0) producer_role<D, BF16, CAUSAL, FP8>(&tm_q, &tm_k, &tm_v, a, sbase, bars, ab);
    } else if constexpr (L::kSplit) {  // MMA issue split over warps 2, 3 (and 1)
      if (warp == 2) mma_s_role<D, BF16, CAUSAL, FP8, 0, 2, kBarDrain>(a, sbase, bars, tmem, ab);
      else if constexpr (L::kPvPerTile) {
        if (warp == 3)
          mma_pv_role<D, BF16, CAUSAL, FP8, 0, 1, kBarDrainPV>(a, sbase, bars, tmem, ab);
        else if (warp == 1)
          mma_pv_role<D, BF16, CAUSAL, FP8, 1, 2, kBarDrainPV + 1>(a, sbase, bars, tmem, ab);
      } else if (warp == 3) {
        mma_pv_role<D, BF16, CAUSAL, FP8, 0, 2, kBarDrainPV>(a, sbase, bars, tmem, ab);
      }
    } else if (warp == 1) {
      mma_role<D, BF16, CAUSAL>(a, sbase, bars, tmem, ab);  // the whole warp
    }
  } else if (wgrp < 3) {
    ptx::setmaxnreg_inc<kRegsSoftmax>();
    softmax_role<D, BF16, CAUSAL, FP8>(a, sbase, bars, tmem, stats, ab, warp, lane);
  } else {
    ptx::setmaxnreg_dec<kRegsEpilogue>();
    epilogue_role<D, BF16, CAUSAL, FP8>(&tm_o, a, sbase, bars, tmem, stats, ab, warp, lane);
  }
  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, L::kTmemCols);
  if (threadIdx.x == 0 && a.clk != nullptr) clock_end(a.clk, clock_slot);
}

// Host side (defined in the per-head-dimension files and fa_host.cu).
// Rows of Q per unit, and of K per TMA box.
constexpr int fwd_unit_rows(int) { return 256; }
constexpr int fwd_k_box_rows(int) { return 128; }
// Rows of O per TMA store: one epilogue warp's rows.
constexpr int kFwdOutBoxRows = 32;
// Persistent grid for n_units units on the current device.
int fwd_grid_d64(int n_units, int sm_count);
int fwd_grid_d128(int n_units, int sm_count);
// maps: Q, K, V (loads) and O (stores) tensor maps.
cudaError_t launch_fwd_d64(bool bf16, bool causal, const CUtensorMap* maps, const FwdArgs& a,
                           int grid, cudaStream_t stream);
cudaError_t launch_fwd_d128(bool bf16, bool causal, const CUtensorMap* maps, const FwdArgs& a,
                            int grid, cudaStream_t stream);
int fwd_smem_bytes(int d);
// Element strides of a contiguous [B][H][N][d] tensor, and the checks on a
// call's strides (fa_host.cu).
fa_strides contiguous_strides(int H, int N, int d);
fa_status check_strides(const fa_strides* s /* q, k, v, o */, int d);
// Size checks of every entry point (B, H, N >= 1; d in {64, 128}; unit and
// row counts in int range).
fa_status check_sizes(int B, int H, int N, int d);
// fa_fwd_noalloc's status word on device `dev` (fa_noalloc.cu): reads it and
// clears it; *timed_out is set when a launch recorded a timeout. FA_OK when
// that entry point has not been used on the device.
fa_status noalloc_take_status(int dev, bool* timed_out);
// Q, K, V, O tensor maps of a call (s: q, k, v, o strides); k_box_rows: keys
// per K box (0: the one-CTA kernel's 128; the CTA-pair kernel loads 64).
bool encode_fwd_maps(CUtensorMap* maps, const void* q, const void* k, const void* v,
                     const void* o, const fa_strides* s, bool bf16, int B, int H, int N, int d,
                     int k_box_rows = 0);
// Unit counts of a call into `a` (N, H, BH, n_mblk, n_units, n_kv) and its grid.
void plan_fwd(int d, int N, int H, long long BH, int sm_count, FwdArgs* a, int* grid);
cudaError_t launch_fwd(int d, bool bf16, bool causal, const CUtensorMap* maps, const FwdArgs& a,
                       int grid, cudaStream_t stream);
// 8-bit inputs (fa_fwd_fp8.cu): maps = Q, K ({128 bytes, N, H, B}) and V^T
// ({keys, 128, H, B}), all e4m3 bytes, and the bf16 O.
cudaError_t launch_fwd_fp8(bool causal, const CUtensorMap* maps, const FwdArgs& a, int grid,
                           cudaStream_t stream);
int fwd_smem_bytes_fp8();

}  // namespace fa
