// Attention forward oracle: plain, slow, fp64 CPU reference.
//
// TEST INFRASTRUCTURE ONLY. Nothing on the product path may call, link or
// load this file: only the test suite, the smoke check and the benchmark's
// CPU-baseline leg use it. It shares no code, header or constant with the
// CUDA library.
//
// What it computes (the plain definition that the fused, tiled kernel reaches
// up to rounding order):
//   for every batch b, head h and query row i
//     s_j    = scale * sum_t q_i[t] * k_j[t]        for j in J(i)
//     J(i)   = {0 .. N-1}, or {0 .. i} when causal (query i sees keys 0..i)
//     m      = max_j s_j
//     l      = sum_j exp(s_j - m)
//     O_i    = sum_j exp(s_j - m) * v_j / l
//     LSE_i  = m + ln(l)
// Sources:
//   - "TCA 51%, MFU below 8%" (zhihu), section on Flash Attention 2's online
//     softmax: attention is softmax of the scaled scores applied to V, and the
//     fused method only avoids materialising the score matrix.
//   - "TMA + Warp Specialization" (CUDA book ch. 17), section 17.5: the
//     consumer's per-tile steps (S = Q K^T, softmax, O += P V, final O / l).
//   The causal mask and the per-row logsumexp are not on those pages; they are
//   taken as the method's output specification (query i attends keys 0..i;
//   LSE in natural-log units).
//
// Inputs are the stored 16-bit values (IEEE binary16 or bfloat16 bit
// patterns), decoded exactly to double. Nothing is rounded back to 16 bits:
// O and LSE are returned in double.
//
// Parity pins (see tests/test_oracle_pins.py): closed forms for Q = 0
// (column mean / prefix mean of V, LSE = ln N / ln(i+1)), one-hot selection,
// V = const, linearity, permutation and shift invariances, exhaustive decoder
// checks against numpy/torch, and agreement with an explicit-softmax
// formulation built from scipy routines at N <= 64.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <thread>
#include <vector>

namespace {

// IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
double decode_binary16(uint16_t h) {
  const int sign = h >> 15;
  const int expo = (h >> 10) & 0x1F;
  const int frac = h & 0x3FF;
  double v;
  if (expo == 0) {
    v = std::ldexp(static_cast<double>(frac), -24);  // subnormal: frac * 2^-24
  } else if (expo == 31) {
    v = frac ? NAN : INFINITY;
  } else {
    // (1 + frac / 2^10) * 2^(expo - 15) = (2^10 + frac) * 2^(expo - 25)
    v = std::ldexp(static_cast<double>(frac | 0x400), expo - 25);
  }
  return sign ? -v : v;
}

// bfloat16: the upper half of an IEEE binary32 (8 exponent bits, bias 127,
// 7 fraction bits).
double decode_bfloat16(uint16_t b) {
  const int sign = b >> 15;
  const int expo = (b >> 7) & 0xFF;
  const int frac = b & 0x7F;
  double v;
  if (expo == 0) {
    v = std::ldexp(static_cast<double>(frac), -133);  // frac * 2^-126 / 2^7
  } else if (expo == 255) {
    v = frac ? NAN : INFINITY;
  } else {
    // (1 + frac / 2^7) * 2^(expo - 127) = (2^7 + frac) * 2^(expo - 134)
    v = std::ldexp(static_cast<double>(frac | 0x80), expo - 134);
  }
  return sign ? -v : v;
}

double decode(uint16_t x, int dtype) {
  return dtype == 0 ? decode_binary16(x) : decode_bfloat16(x);
}

void decode_block(const uint16_t* src, int64_t n, int dtype, double* dst) {
  for (int64_t t = 0; t < n; ++t) dst[t] = decode(src[t], dtype);
}

// One query row against the keys 0..nkeys-1 of one (batch, head).
// K and V are the decoded [N][d] matrices of that head.
void attend_row(const double* qi, const double* K, const double* V,
                int64_t d, int64_t nkeys, double scale,
                std::vector<double>& s, double* out_o, double* out_lse) {
  double m = -INFINITY;
  for (int64_t j = 0; j < nkeys; ++j) {
    double dot = 0.0;
    for (int64_t t = 0; t < d; ++t) dot += qi[t] * K[j * d + t];
    s[j] = scale * dot;
    m = std::max(m, s[j]);
  }
  double l = 0.0;
  for (int64_t j = 0; j < nkeys; ++j) {
    s[j] = std::exp(s[j] - m);
    l += s[j];
  }
  for (int64_t t = 0; t < d; ++t) out_o[t] = 0.0;
  for (int64_t j = 0; j < nkeys; ++j) {
    const double w = s[j];
    for (int64_t t = 0; t < d; ++t) out_o[t] += w * V[j * d + t];
  }
  for (int64_t t = 0; t < d; ++t) out_o[t] /= l;
  *out_lse = m + std::log(l);
}

// OCP 8-bit floating point E4M3 ("fn" variant): 1 sign bit, 4 exponent bits
// (bias 7), 3 fraction bits; no infinities; S.1111.111 is NaN; largest
// finite value 0x7E = 448; subnormals frac * 2^-9.
double decode_e4m3(uint8_t c) {
  const int sign = c >> 7;
  const int expo = (c >> 3) & 0xF;
  const int frac = c & 0x7;
  double v;
  if (expo == 0xF && frac == 0x7) {
    v = NAN;
  } else if (expo == 0) {
    v = std::ldexp(static_cast<double>(frac), -9);
  } else {
    // (1 + frac / 8) * 2^(expo - 7) = (8 + frac) * 2^(expo - 10)
    v = std::ldexp(static_cast<double>(frac | 0x8), expo - 10);
  }
  return sign ? -v : v;
}

// The 8-bit variant of attend_row: same definition, plus a bound on how far a
// kernel that rounds every softmax weight p to e4m3 before the P V product
// (and normalises by the sum of the unrounded weights) can land from O.
// Rounding p in [2^-6, 448] moves it by at most 2^-4 p (3 fraction bits),
// below 2^-6 by at most 2^-10 (subnormal spacing 2^-9), on the kernel's own
// weight scale, whose largest weight lies in [1, 2^8]; so on the scale where
// the largest weight is 1 each weight moves by at most 2^-4 p_j + 2^-10, and
//   |O_t - O'_t| <= sum_j (2^-4 p_j + 2^-10) |v_jt| / sum_j p_j.
void attend_row_bound(const double* qi, const double* K, const double* V,
                      int64_t d, int64_t nkeys, double scale, std::vector<double>& s,
                      double* out_o, double* out_lse, double* out_bound) {
  attend_row(qi, K, V, d, nkeys, scale, s, out_o, out_lse);  // s now holds p_j
  double l = 0.0;
  for (int64_t j = 0; j < nkeys; ++j) l += s[j];
  for (int64_t t = 0; t < d; ++t) out_bound[t] = 0.0;
  for (int64_t j = 0; j < nkeys; ++j) {
    const double w = 0.0625 * s[j] + 1.0 / 1024.0;
    for (int64_t t = 0; t < d; ++t) out_bound[t] += w * std::fabs(V[j * d + t]);
  }
  for (int64_t t = 0; t < d; ++t) out_bound[t] /= l;
}

int pick_threads(int requested) {
  if (requested > 0) return requested;
  const unsigned hc = std::thread::hardware_concurrency();
  return hc ? static_cast<int>(hc) : 1;
}

// Runs f(worker, count) on `nthreads` threads.
template <class F>
void run_parallel(int nthreads, F f) {
  std::vector<std::thread> pool;
  for (int w = 1; w < nthreads; ++w) pool.emplace_back(f, w, nthreads);
  f(0, nthreads);
  for (auto& t : pool) t.join();
}

}  // namespace

extern "C" {

// Number of worker threads the oracle uses for `requested` (0 = all cores).
int oracle_threads(int requested) { return pick_threads(requested); }

// Decodes n stored 16-bit values (dtype 0 = binary16, 1 = bfloat16).
void oracle_decode(const uint16_t* x, int dtype, int64_t n, double* out) {
  decode_block(x, n, dtype, out);
}

// Full forward: q, k, v are [B][H][N][d] stored 16-bit values; o is
// [B][H][N][d] double, lse is [B][H][N] double. Returns 0, or -1 on bad
// arguments.
int oracle_attn_fwd(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                    int dtype, int64_t B, int64_t H, int64_t N, int64_t d,
                    int causal, float scale, double* o, double* lse,
                    int nthreads) {
  if (!q || !k || !v || !o || !lse || B <= 0 || H <= 0 || N <= 0 || d <= 0 ||
      (dtype != 0 && dtype != 1))
    return -1;
  const int64_t BH = B * H;
  const double sc = static_cast<double>(scale);
  const int T = std::min<int64_t>(pick_threads(nthreads), BH);
  run_parallel(T, [&](int w, int nt) {
    std::vector<double> K(N * d), V(N * d), qi(d), s(N);
    for (int64_t bh = w; bh < BH; bh += nt) {
      const int64_t base = bh * N * d;
      decode_block(k + base, N * d, dtype, K.data());
      decode_block(v + base, N * d, dtype, V.data());
      for (int64_t i = 0; i < N; ++i) {
        decode_block(q + base + i * d, d, dtype, qi.data());
        const int64_t nkeys = causal ? i + 1 : N;
        attend_row(qi.data(), K.data(), V.data(), d, nkeys, sc, s,
                   o + base + i * d, lse + bh * N + i);
      }
    }
  });
  return 0;
}

// Selected rows only. rows[r] is a flat row index bh * N + i. Outputs are
// o[r][d] and lse[r]. Rows are split into contiguous chunks, one per thread;
// a thread re-decodes K and V whenever its (batch, head) changes, so callers
// should group rows by head.
int oracle_attn_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                     int dtype, int64_t B, int64_t H, int64_t N, int64_t d,
                     int causal, float scale, const int64_t* rows,
                     int64_t nrows, double* o, double* lse, int nthreads) {
  if (!q || !k || !v || !rows || !o || !lse || B <= 0 || H <= 0 || N <= 0 ||
      d <= 0 || nrows < 0 || (dtype != 0 && dtype != 1))
    return -1;
  const int64_t BH = B * H;
  for (int64_t r = 0; r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= BH * N) return -1;
  const double sc = static_cast<double>(scale);
  const int T = static_cast<int>(
      std::max<int64_t>(1, std::min<int64_t>(pick_threads(nthreads), nrows)));
  run_parallel(T, [&](int w, int nt) {
    const int64_t lo = nrows * w / nt, hi = nrows * (w + 1) / nt;
    std::vector<double> K(N * d), V(N * d), qi(d), s(N);
    int64_t cur = -1;
    for (int64_t r = lo; r < hi; ++r) {
      const int64_t bh = rows[r] / N, i = rows[r] % N;
      const int64_t base = bh * N * d;
      if (bh != cur) {
        decode_block(k + base, N * d, dtype, K.data());
        decode_block(v + base, N * d, dtype, V.data());
        cur = bh;
      }
      decode_block(q + base + i * d, d, dtype, qi.data());
      const int64_t nkeys = causal ? i + 1 : N;
      attend_row(qi.data(), K.data(), V.data(), d, nkeys, sc, s, o + r * d,
                 lse + r);
    }
  });
  return 0;
}

// Selected rows, as oracle_attn_rows, plus dev[r][d]: the weighted mean
// absolute deviation of V under the row's softmax weights,
//   dev_t = sum_j p_j |v_jt - O_t| / sum_j p_j.
// It bounds what rounding the weights costs: a kernel that rounds each weight
// p_j to r_j with |r_j - p_j| <= u p_j before the P V product and normalises
// by sum_j r_j gets O'_t - O_t = sum_j (r_j - p_j)(v_jt - O_t) / sum_j r_j,
// so |O'_t - O_t| <= u / (1 - u) * dev_t (before its own output rounding).
// The weights come from the same definition as attend_row.
int oracle_attn_rows_dev(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                         int dtype, int64_t B, int64_t H, int64_t N, int64_t d,
                         int causal, float scale, const int64_t* rows,
                         int64_t nrows, double* o, double* lse, double* dev, int nthreads) {
  if (!dev) return -1;
  const int rc = oracle_attn_rows(q, k, v, dtype, B, H, N, d, causal, scale, rows, nrows, o,
                                  lse, nthreads);
  if (rc != 0) return rc;
  const double sc = static_cast<double>(scale);
  const int T = static_cast<int>(
      std::max<int64_t>(1, std::min<int64_t>(pick_threads(nthreads), nrows)));
  run_parallel(T, [&](int w, int nt) {
    const int64_t lo = nrows * w / nt, hi = nrows * (w + 1) / nt;
    std::vector<double> K(N * d), V(N * d), qi(d), s(N), oi(d);
    int64_t cur = -1;
    for (int64_t r = lo; r < hi; ++r) {
      const int64_t bh = rows[r] / N, i = rows[r] % N;
      const int64_t base = bh * N * d;
      if (bh != cur) {
        decode_block(k + base, N * d, dtype, K.data());
        decode_block(v + base, N * d, dtype, V.data());
        cur = bh;
      }
      decode_block(q + base + i * d, d, dtype, qi.data());
      const int64_t nkeys = causal ? i + 1 : N;
      double li = 0.0;
      attend_row(qi.data(), K.data(), V.data(), d, nkeys, sc, s, oi.data(), &li);  // s = p_j
      double l = 0.0;
      for (int64_t j = 0; j < nkeys; ++j) l += s[j];
      double* out = dev + r * d;
      for (int64_t t = 0; t < d; ++t) out[t] = 0.0;
      for (int64_t j = 0; j < nkeys; ++j)
        for (int64_t t = 0; t < d; ++t) out[t] += s[j] * std::fabs(V[j * d + t] - oi[t]);
      for (int64_t t = 0; t < d; ++t) out[t] /= l;
    }
  });
  return 0;
}

// 8-bit forward. q8, k8: [B][H][N][d] e4m3 codes; vt8: [B][H][d][ldv] e4m3
// codes of V transposed (column n of row t is V[n][t]); the values are
//   q = q_scale * q8,  k_n = k_scales[b][h][n / 128] * k8_n,  v = v_scale * v8.
// rows: flat row indices bh * N + i (nrows of them), or all rows in order
// when rows is null. Outputs per row: o[r][d], lse[r] and bound[r][d], the
// e4m3-weight bound of attend_row_bound. Returns 0, or -1 on bad arguments.
int oracle_attn_fp8(const uint8_t* q8, const uint8_t* k8, const uint8_t* vt8, int64_t B,
                    int64_t H, int64_t N, int64_t d, int64_t ldv, float q_scale,
                    const float* k_scales, float v_scale, int causal, float scale,
                    const int64_t* rows, int64_t nrows, double* o, double* lse,
                    double* bound, int nthreads) {
  const int64_t BH = B * H;
  if (!q8 || !k8 || !vt8 || !k_scales || !o || !lse || !bound || B <= 0 || H <= 0 ||
      N <= 0 || d <= 0 || ldv < N)
    return -1;
  if (!rows) nrows = BH * N;
  if (nrows < 0) return -1;
  if (rows)
    for (int64_t r = 0; r < nrows; ++r)
      if (rows[r] < 0 || rows[r] >= BH * N) return -1;
  const int64_t ntiles = (N + 127) / 128;
  const double sc = static_cast<double>(scale);
  const int T = static_cast<int>(
      std::max<int64_t>(1, std::min<int64_t>(pick_threads(nthreads), nrows)));
  run_parallel(T, [&](int w, int nt) {
    const int64_t lo = nrows * w / nt, hi = nrows * (w + 1) / nt;
    std::vector<double> K(N * d), V(N * d), qi(d), s(N);
    int64_t cur = -1;
    for (int64_t r = lo; r < hi; ++r) {
      const int64_t row = rows ? rows[r] : r;
      const int64_t bh = row / N, i = row % N;
      if (bh != cur) {
        for (int64_t n = 0; n < N; ++n) {
          const double ks = static_cast<double>(k_scales[bh * ntiles + n / 128]);
          for (int64_t t = 0; t < d; ++t) {
            K[n * d + t] = ks * decode_e4m3(k8[(bh * N + n) * d + t]);
            V[n * d + t] = static_cast<double>(v_scale) * decode_e4m3(vt8[(bh * d + t) * ldv + n]);
          }
        }
        cur = bh;
      }
      for (int64_t t = 0; t < d; ++t)
        qi[t] = static_cast<double>(q_scale) * decode_e4m3(q8[(bh * N + i) * d + t]);
      const int64_t nkeys = causal ? i + 1 : N;
      attend_row_bound(qi.data(), K.data(), V.data(), d, nkeys, sc, s, o + r * d, lse + r,
                       bound + r * d);
    }
  });
  return 0;
}

// Decodes n e4m3 codes.
void oracle_decode_e4m3(const uint8_t* x, int64_t n, double* out) {
  for (int64_t t = 0; t < n; ++t) out[t] = decode_e4m3(x[t]);
}

// Backward pass of one (batch, head), from the definition. With
//   P_ij = exp(s_ij - LSE_i) (the softmax weights, j in J(i)),
//   O_i = sum_j P_ij v_j and a loss whose gradient at O is dO:
//   dV_j  = sum_i P_ij dO_i
//   dP_ij = dO_i . v_j
//   dS_ij = P_ij (dP_ij - D_i),   D_i = sum_j P_ij dP_ij = dO_i . O_i
//   dQ_i  = scale * sum_j dS_ij k_j
//   dK_j  = scale * sum_i dS_ij q_i
// (the chain rule through s = scale q.k and the softmax Jacobian
// diag(P) - P P^T. Source: "TCA 51%, MFU below 8%", section "MFU is always
// a little below TCA": the backward recomputes rather than storing the
// scores; recomputing P from the forward's logsumexp is this library's
// reading, and here P comes from the same definition as the forward's).
// Besides the gradients, mag_* hold the sums of the magnitudes of the terms
// of each element: sum_i |P_ij dO_it| for dV; for dQ and dK the sums
// scale * sum_j A_ij |k_jt| and scale * sum_i A_ij |q_it| with
//   A_ij = P_ij (sum_t |dO_it v_jt| + sum_t |dO_it| sum_j' P_ij' |v_j't|),
// the magnitudes of the terms of dP_ij and of D_i (through the terms of O_i).
// Rounding P, dS or O to a 16-bit format perturbs an element by a multiple
// of the unit roundoff times these sums, even where dP_ij - D_i cancels.
void bwd_head(const double* Q, const double* K, const double* V, const double* dO,
              int64_t N, int64_t d, bool causal, double scale, double* dq, double* dk,
              double* dv, double* mq, double* mk, double* mv, int nthreads) {
  std::vector<double> P(N * N, 0.0), dS(N * N, 0.0), DS(N * N, 0.0);
  // Rows i of P, dS and their magnitudes (rows are independent: split over
  // threads in interleaved order, which balances the causal triangle).
  run_parallel(nthreads, [&](int w, int nt) {
    std::vector<double> s(N), o(d), ao(d);
    for (int64_t i = w; i < N; i += nt) {
      const int64_t nk = causal ? i + 1 : N;
      double m = -INFINITY;
      for (int64_t j = 0; j < nk; ++j) {
        double dot = 0.0;
        for (int64_t t = 0; t < d; ++t) dot += Q[i * d + t] * K[j * d + t];
        s[j] = scale * dot;
        m = std::max(m, s[j]);
      }
      double l = 0.0;
      for (int64_t j = 0; j < nk; ++j) l += std::exp(s[j] - m);
      const double lse = m + std::log(l);
      for (int64_t t = 0; t < d; ++t) o[t] = ao[t] = 0.0;
      for (int64_t j = 0; j < nk; ++j) {
        P[i * N + j] = std::exp(s[j] - lse);
        for (int64_t t = 0; t < d; ++t) {
          o[t] += P[i * N + j] * V[j * d + t];
          ao[t] += P[i * N + j] * std::fabs(V[j * d + t]);
        }
      }
      // D_i = dO_i . O_i; its term magnitude sums |dO_it| over the terms of O_it
      double Di = 0.0, aDi = 0.0;
      for (int64_t t = 0; t < d; ++t) {
        Di += dO[i * d + t] * o[t];
        aDi += std::fabs(dO[i * d + t]) * ao[t];
      }
      for (int64_t j = 0; j < nk; ++j) {
        double dp = 0.0, adp = 0.0;
        for (int64_t t = 0; t < d; ++t) {
          dp += dO[i * d + t] * V[j * d + t];
          adp += std::fabs(dO[i * d + t] * V[j * d + t]);
        }
        dS[i * N + j] = P[i * N + j] * (dp - Di);
        DS[i * N + j] = P[i * N + j] * (adp + aDi);
      }
    }
  });
  // dQ_i = scale sum_j dS_ij k_j: one row per task.
  run_parallel(nthreads, [&](int w, int nt) {
    for (int64_t i = w; i < N; i += nt) {
      const int64_t nk = causal ? i + 1 : N;
      for (int64_t t = 0; t < d; ++t) dq[i * d + t] = mq[i * d + t] = 0.0;
      for (int64_t j = 0; j < nk; ++j) {
        const double ds = dS[i * N + j], ads = DS[i * N + j];
        for (int64_t t = 0; t < d; ++t) {
          dq[i * d + t] += scale * ds * K[j * d + t];
          mq[i * d + t] += scale * ads * std::fabs(K[j * d + t]);
        }
      }
    }
  });
  // dV_j = sum_i P_ij dO_i and dK_j = scale sum_i dS_ij q_i: blocks of 64 keys
  // per task, each summing over the rows i that see its keys in increasing i.
  constexpr int64_t kKeyBlock = 64;
  const int64_t nblk = (N + kKeyBlock - 1) / kKeyBlock;
  run_parallel(nthreads, [&](int w, int nt) {
    for (int64_t b = w; b < nblk; b += nt) {
      const int64_t j0 = b * kKeyBlock, j1 = std::min(N, j0 + kKeyBlock);
      for (int64_t x = j0 * d; x < j1 * d; ++x) dk[x] = dv[x] = mk[x] = mv[x] = 0.0;
      for (int64_t i = causal ? j0 : 0; i < N; ++i) {
        const int64_t jend = causal ? std::min(j1, i + 1) : j1;
        for (int64_t j = j0; j < jend; ++j) {
          const double p = P[i * N + j], ds = dS[i * N + j], ads = DS[i * N + j];
          for (int64_t t = 0; t < d; ++t) {
            dv[j * d + t] += p * dO[i * d + t];
            mv[j * d + t] += std::fabs(p * dO[i * d + t]);
            dk[j * d + t] += scale * ds * Q[i * d + t];
            mk[j * d + t] += scale * ads * std::fabs(Q[i * d + t]);
          }
        }
      }
    }
  });
}

// Backward for the heads listed in `heads` (flat bh indices): q, k, v, dout
// are [B][H][N][d] stored 16-bit values; outputs are [nheads][N][d] double
// (gradients and magnitude sums, see bwd_head). Returns 0, or -1 on bad
// arguments.
int oracle_attn_bwd(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* dout,
                    int dtype, int64_t B, int64_t H, int64_t N, int64_t d, int causal,
                    float scale, const int64_t* heads, int64_t nheads, double* dq, double* dk,
                    double* dv, double* mq, double* mk, double* mv, int nthreads) {
  if (!q || !k || !v || !dout || !heads || !dq || !dk || !dv || !mq || !mk || !mv || B <= 0 ||
      H <= 0 || N <= 0 || d <= 0 || nheads < 0 || (dtype != 0 && dtype != 1))
    return -1;
  for (int64_t r = 0; r < nheads; ++r)
    if (heads[r] < 0 || heads[r] >= B * H) return -1;
  const double sc = static_cast<double>(scale);
  // One thread per head when there are enough heads; otherwise the heads one
  // after another, each split over all the threads.
  const int T = pick_threads(nthreads);
  const int outer = nheads >= T ? T : 1;
  const int inner = nheads >= T ? 1 : T;
  run_parallel(outer, [&](int w, int nt) {
    std::vector<double> Q(N * d), K(N * d), V(N * d), dO(N * d);
    for (int64_t r = w; r < nheads; r += nt) {
      const int64_t base = heads[r] * N * d;
      decode_block(q + base, N * d, dtype, Q.data());
      decode_block(k + base, N * d, dtype, K.data());
      decode_block(v + base, N * d, dtype, V.data());
      decode_block(dout + base, N * d, dtype, dO.data());
      const int64_t off = r * N * d;
      bwd_head(Q.data(), K.data(), V.data(), dO.data(), N, d, causal != 0, sc, dq + off,
               dk + off, dv + off, mq + off, mk + off, mv + off, inner);
    }
  });
  return 0;
}

}  // extern "C"
