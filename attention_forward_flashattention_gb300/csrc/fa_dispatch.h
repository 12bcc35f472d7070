// Which forward kernel the C entry points run: the measured policy between
// the one-CTA kernel and the CTA-pair kernel (host code only; the two give
// identical results, so the choice changes only the time).
#pragma once

namespace fa {

// Whether fa_fwd / fa_fwd_strided run the pair kernel: head dimension 128,
// enough 512-row units to give every SM pair one, and non-causal or long
// causal rows. Same-box measurements (row maximum from the S loads):
// non-causal B4 H16 N4096 ~5 % faster than the one-CTA kernel (~15 % in a
// power-capped sustained run); causal N = 4096 ~5 % slower (a 512-row unit
// visits up to two more wholly masked KV tiles than two 256-row units, a
// larger share of short rows' work), N = 8192 / 12288 even, N = 16384 and
// 32768 1-2 % faster. The two kernels' results are identical bit for bit.
inline bool fwd_prefers_pair(int d, bool causal, long long BH, int N, int sm_count) {
  return d == 128 && (!causal || N >= 16384) &&
         BH * ((static_cast<long long>(N) + 511) / 512) >= sm_count / 2;
}

// Whether fa_fwd_fp8 runs the pair kernel (8-bit inputs are always head
// dimension 128). Kept to the one-CTA kernel until measured otherwise.
inline bool fwd_fp8_prefers_pair(bool causal, long long BH, int N, int sm_count) {
  (void)causal;
  (void)BH;
  (void)N;
  (void)sm_count;
  return false;
}

}  // namespace fa
