// Exact softmax attention, forward and backward, in fp64 on the host.
//
// TEST INFRASTRUCTURE ONLY. This file is the oracle that the CUDA path is
// checked against. Only the tests, the smoke check and the CPU-baseline leg of
// the benchmark load it. It shares no code, header, table or helper with the
// library under exact_attention_83_gb300/; neither side includes the other.
//
// What it computes is the plain definition of scaled-dot-product attention and
// its gradient, not the tiled algorithm (except oracle_*_tiled, which restates
// the tiled FlashAttention-2 recurrences only so that a test can show the
// result does not depend on the tile sizes).
//
// Sources, by page title and section:
//  * "FlashAttention-2 from PyTorch to Triton" (wpnews.pro), the section on the
//    three running quantities: the log-sum-exp L_i = m_i + log(l_i), which
//    equals log sum_k exp(S_ik), and the backward's recovery of the
//    probabilities as P = exp(S - L).  Its test harness: causal keeps key j for
//    query i iff j <= i (the `k_pos <= q_pos` predicate, top-left aligned), and
//    the scores are S = scale * Q K^T with scale = 1/sqrt(d).
//  * same page, defect list item 5: the backward needs D = rowsum(dO o O).
//  * "Triton FlashAttention" (architjain.me), project summary: the backward
//    rebuilds P from the saved log-sum-exp; rowsum(dO.O) is its own step.
//  * The gradient rows below are the standard softmax-attention derivative
//    (dV = P^T dO, dP = dO V^T, dS = P o (dP - Delta), dQ = scale dS K,
//    dK = scale dS^T Q).  The tutorial "Build a FlashAttention-2 Engine from
//    Scratch in Triton", step 5, prints a garbled version of these equations;
//    it is not followed.
//
// General problems.  The Triton page's test harness runs shapes whose query
// and key counts differ, with the causal mask the lower triangle of the
// Nq x Nk score matrix; the pages name grouped-query and multi-query
// attention, variable-length batches and dropout as branches they leave out,
// without defining them.  The oracle takes their plainest readings:
//  * grouped heads: Hq query heads and Hkv key/value heads, Hq % Hkv == 0;
//    query head h reads key/value head h / (Hq / Hkv); dK, dV of a key/value
//    head sum the contributions of every query head that reads it;
//  * variable lengths (Python wrapper): each packed sequence is its own
//    problem, positions counted from its first row;
//  * dropout: each weight P_ij is multiplied by Z_ij = keep_ij / (1 - p)
//    before the product with V (O = (P o Z) V); L stays the log-sum-exp of the
//    undropped scores; then dV = (P o Z)^T dO and dS = P o (Z o dP - Delta),
//    Delta = rowsum(dO o O) as before.  keep_ij is drawn from Philox4x32-10
//    (Salmon et al., SC 2011) at counter (j / 8, i, flat head, offset): the
//    16-bit half j mod 2 of word (j mod 8) / 2 is compared with
//    floor(p * 65536).
//
// Readings where the pages are open (each is also listed in the design notes):
//  * masked keys are excluded exactly (weight 0, never a finite sentinel);
//  * L is in natural-log units and always fp64 here; a row with no key at all
//    has L = -inf and O = 0 (the empty sum);
//  * Delta uses the oracle's own fp64 O.
//
// Layout: every tensor is a dense row-major array of doubles: Q, O, dO, dQ
// [B, Hq, Nq, D]; K, V, dK, dV [B, Hkv, Nk, D]; L and Delta [B, Hq, Nq].
// Inputs are the exact values of the rounded device inputs (fp16/bf16/fp32
// -> double is exact).
//
// Pins: softmax rows sum to 1; closed forms for constant V, causal row 0,
// Q = 0 and N = 1; finite differences of the forward; sum_j dK_j = 0;
// sum_j dV_j = sum_i dO_i; tile-size invariance; agreement with the dense
// N x N materialisation and with a library routine (tests/test_oracle_pins.py);
// Nq != Nk and grouped heads against the library routine, Philox known-answer
// vectors, dropout gradients against finite differences, packed against
// batched numbering (tests/test_oracle_pins_general.py).

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#include <algorithm>
#include <limits>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

inline double dot(const double* a, const double* b, int64_t D) {
  double s = 0.0;
  for (int64_t d = 0; d < D; ++d) s += a[d] * b[d];
  return s;
}

// Number of keys query row i may attend to: all Nk, or keys 0..i when causal
// (top-left aligned mask, "FlashAttention-2 from PyTorch to Triton", kernel's
// causal predicate and its test harness, which builds the mask as the lower
// triangle of the Nq x Nk score matrix).
inline int64_t keys_allowed(int64_t i, int64_t Nk, int causal) {
  return causal ? std::min(i + 1, Nk) : Nk;
}

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy
// as 1, 2, 3", SC 2011): ten rounds; a round multiplies counter words 0 and 2
// by the two round multipliers and mixes the high and low halves of the
// products with words 1 and 3 and the key; the key is advanced by the two
// Weyl increments between rounds.
void philox(const uint32_t ctr[4], uint32_t k0, uint32_t k1, uint32_t out[4]) {
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint64_t p0 = static_cast<uint64_t>(0xD2511F53u) * c0;
    const uint64_t p1 = static_cast<uint64_t>(0xCD9E8D57u) * c2;
    const uint32_t n0 = static_cast<uint32_t>(p1 >> 32) ^ c1 ^ k0;
    const uint32_t n1 = static_cast<uint32_t>(p1);
    const uint32_t n2 = static_cast<uint32_t>(p0 >> 32) ^ c3 ^ k1;
    const uint32_t n3 = static_cast<uint32_t>(p0);
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

}  // namespace

extern "C" {

// Dropout of the attention weights (none when on == 0): weight (i, j) of flat
// query head bh0 + (b * Hq + h) is kept iff the 16-bit half (j mod 2, 0 = low)
// of word ((j mod 8) / 2) of Philox4x32-10 at counter
// (j / 8, i, bh0 + b * Hq + h, offset) under key (key0, key1) is >= thr
// (= floor(p * 65536)); a kept weight is multiplied by rscale = 1 / (1 - p).
// i and j are positions within the sequence; bh0 lets a packed batch pass one
// sequence at a time with its own head numbering.
typedef struct {
  int on;
  uint32_t thr;
  double rscale;
  uint32_t key0, key1, offset;
  int64_t bh0;
} oracle_dropout;

}  // extern "C"

namespace {

// Z_ij of one weight, 1 without dropout.
inline double zfac(const oracle_dropout* dr, int64_t i, int64_t j, int64_t bh) {
  if (dr == nullptr || !dr->on) return 1.0;
  const uint32_t ctr[4] = {static_cast<uint32_t>(j / 8), static_cast<uint32_t>(i),
                           static_cast<uint32_t>(dr->bh0 + bh), dr->offset};
  uint32_t w[4];
  philox(ctr, dr->key0, dr->key1, w);
  const uint32_t word = w[(j % 8) / 2];
  const uint32_t half = (j % 2 == 0) ? (word & 0xFFFFu) : (word >> 16);
  return half >= dr->thr ? dr->rscale : 0.0;
}

// Forward for one query row (the plain definition).
//   s_j = scale * q_i . k_j          for allowed j
//   m   = max_j s_j
//   L   = m + log sum_j exp(s_j - m)           (= log sum_j exp(s_j); -inf
//                                               when no key is allowed)
//   p_j = exp(s_j - L)
//   o_i = sum_j z_j p_j v_j          (z_j = 1 without dropout)
// `s` is scratch of at least nk doubles; on return it holds p_j.  z is null
// (no dropout) or holds z_j.
void row_forward(const double* qi, const double* K, const double* V,
                 int64_t nk, int64_t D, double scale, const double* z,
                 double* s, double* oi, double* Li) {
  double m = -std::numeric_limits<double>::infinity();
  for (int64_t j = 0; j < nk; ++j) {
    s[j] = scale * dot(qi, K + j * D, D);
    m = std::max(m, s[j]);
  }
  for (int64_t d = 0; d < D; ++d) oi[d] = 0.0;
  if (nk == 0) {
    *Li = -std::numeric_limits<double>::infinity();
    return;
  }
  double sum = 0.0;
  for (int64_t j = 0; j < nk; ++j) sum += std::exp(s[j] - m);
  const double L = m + std::log(sum);
  for (int64_t j = 0; j < nk; ++j) {
    s[j] = std::exp(s[j] - L);
    const double w = z ? z[j] * s[j] : s[j];
    const double* vj = V + j * D;
    for (int64_t d = 0; d < D; ++d) oi[d] += w * vj[d];
  }
  *Li = L;
}

// Shapes of one call: Q, O, dO, dQ [B, Hq, Nq, D]; K, V, dK, dV [B, Hkv, Nk,
// D]; L, Delta [B, Hq, Nq].  Query head h reads key/value head h / (Hq / Hkv).
struct Dims {
  int64_t B, Hq, Hkv, Nq, Nk, D;
  int64_t G() const { return Hq / Hkv; }
  // base offsets of query head qh = b*Hq + h and of its key/value head
  int64_t qbase(int64_t qh) const { return qh * Nq * D; }
  int64_t kbase(int64_t qh) const { return ((qh / Hq) * Hkv + (qh % Hq) / G()) * Nk * D; }
};

// Pass 1 for one query row: O_i, L_i, Delta_i = dO_i . O_i and
//   dQ_i = scale * sum_j P_ij (Z_ij (dO_i . v_j) - Delta_i) k_j
// (dQ and Delta only when dO is non-null).  Optionally the magnitude sums
//   Oabs_i = sum_j Z_ij P_ij |v_j|,  dQabs_i = scale * sum_j |dS_ij| |k_j|.
void query_row(const Dims& dm, const double* Q, const double* K, const double* V,
               const double* dO, int causal, double scale, const oracle_dropout* dr,
               int64_t qh, int64_t i, std::vector<double>& p, std::vector<double>& z,
               double* oi, double* Li, double* Deltai, double* dqi, double* oabs,
               double* dqabs) {
  const int64_t D = dm.D;
  const int64_t qb = dm.qbase(qh), kb = dm.kbase(qh);
  const int64_t nk = keys_allowed(i, dm.Nk, causal);
  const bool drop = dr && dr->on;
  if (drop)
    for (int64_t j = 0; j < nk; ++j) z[j] = zfac(dr, i, j, qh);
  row_forward(Q + qb + i * D, K + kb, V + kb, nk, D, scale, drop ? z.data() : nullptr,
              p.data(), oi, Li);
  if (oabs) {
    for (int64_t d = 0; d < D; ++d) oabs[d] = 0.0;
    for (int64_t j = 0; j < nk; ++j) {
      const double w = (drop ? z[j] : 1.0) * p[j];
      const double* vj = V + kb + j * D;
      for (int64_t d = 0; d < D; ++d) oabs[d] += w * std::fabs(vj[d]);
    }
  }
  if (!dO) return;
  const double* doi = dO + qb + i * D;
  const double delta = dot(doi, oi, D);
  if (Deltai) *Deltai = delta;
  for (int64_t d = 0; d < D; ++d) dqi[d] = 0.0;
  if (dqabs)
    for (int64_t d = 0; d < D; ++d) dqabs[d] = 0.0;
  for (int64_t j = 0; j < nk; ++j) {
    const double* kj = K + kb + j * D;
    const double dpt = dot(doi, V + kb + j * D, D);
    const double ds = p[j] * ((drop ? z[j] : 1.0) * dpt - delta);
    for (int64_t d = 0; d < D; ++d) dqi[d] += ds * kj[d];
    if (dqabs)
      for (int64_t d = 0; d < D; ++d) dqabs[d] += std::fabs(ds) * std::fabs(kj[d]);
  }
  for (int64_t d = 0; d < D; ++d) dqi[d] *= scale;
  if (dqabs)
    for (int64_t d = 0; d < D; ++d) dqabs[d] *= scale;
}

// Pass 2 for one key row j of flat key/value head kh = b*Hkv + hk: over every
// query head h of its group and every query i that may attend to key j (all i,
// or i >= j when causal),
//   P_ij = exp(scale q_i . k_j - L_i),  Z_ij as above,  dP_ij = dO_i . v_j,
//   dS_ij = P_ij (Z_ij dP_ij - Delta_i),
//   dV_j = sum Z_ij P_ij dO_i,  dK_j = scale * sum dS_ij q_i.
// L and Delta are the full [B, Hq, Nq] arrays.  Optionally the magnitude sums
//   dVabs_j = sum Z_ij P_ij |dO_i|,  dKabs_j = scale * sum |dS_ij| |q_i|.
void key_row(const Dims& dm, const double* Q, const double* K, const double* V,
             const double* dO, const double* L, const double* Delta, int causal,
             double scale, const oracle_dropout* dr, int64_t kh, int64_t j, double* dkj,
             double* dvj, double* dkabs, double* dvabs) {
  const int64_t D = dm.D, G = dm.G();
  const int64_t b = kh / dm.Hkv, hk = kh % dm.Hkv;
  const double* kj = K + kh * dm.Nk * D + j * D;
  const double* vj = V + kh * dm.Nk * D + j * D;
  for (int64_t d = 0; d < D; ++d) { dkj[d] = 0.0; dvj[d] = 0.0; }
  if (dkabs)
    for (int64_t d = 0; d < D; ++d) { dkabs[d] = 0.0; dvabs[d] = 0.0; }
  for (int64_t g = 0; g < G; ++g) {
    const int64_t qh = b * dm.Hq + hk * G + g;
    const int64_t qb = dm.qbase(qh);
    for (int64_t i = causal ? j : 0; i < dm.Nq; ++i) {
      const double* qi = Q + qb + i * D;
      const double* doi = dO + qb + i * D;
      const double pij = std::exp(scale * dot(qi, kj, D) - L[qh * dm.Nq + i]);
      const double z = zfac(dr, i, j, qh);
      const double ds = pij * (z * dot(doi, vj, D) - Delta[qh * dm.Nq + i]);
      for (int64_t d = 0; d < D; ++d) {
        dvj[d] += z * pij * doi[d];
        dkj[d] += ds * qi[d];
      }
      if (dkabs)
        for (int64_t d = 0; d < D; ++d) {
          dvabs[d] += z * pij * std::fabs(doi[d]);
          dkabs[d] += std::fabs(ds) * std::fabs(qi[d]);
        }
    }
  }
  for (int64_t d = 0; d < D; ++d) dkj[d] *= scale;
  if (dkabs)
    for (int64_t d = 0; d < D; ++d) dkabs[d] *= scale;
}

// L and Delta of every query row of the listed flat query heads (pass 1
// without dQ), for pass 2.
void stats_for_heads(const Dims& dm, const double* Q, const double* K, const double* V,
                     const double* dO, int causal, double scale, const oracle_dropout* dr,
                     const std::vector<int64_t>& qheads, double* L, double* Delta) {
  for (const int64_t qh : qheads) {
#pragma omp parallel
    {
      std::vector<double> p(static_cast<size_t>(dm.Nk)), z(static_cast<size_t>(dm.Nk)),
          oi(static_cast<size_t>(dm.D));
#pragma omp for schedule(dynamic, 16)
      for (int64_t i = 0; i < dm.Nq; ++i) {
        query_row(dm, Q, K, V, nullptr, causal, scale, dr, qh, i, p, z, oi.data(),
                  &L[qh * dm.Nq + i], nullptr, nullptr, nullptr, nullptr);
        Delta[qh * dm.Nq + i] = dot(dO + dm.qbase(qh) + i * dm.D, oi.data(), dm.D);
      }
    }
  }
}

}  // namespace

extern "C" {

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

// Philox4x32-10 of one counter under one key (for the generator's pins).
void oracle_philox4x32_10(const uint32_t* ctr, const uint32_t* key, uint32_t* out) {
  philox(ctr, key[0], key[1], out);
}

// Z of the weights (i0 + r, j), r < nq, j < nk, of flat head bh (row-major
// [nq, nk]): keep / (1 - p), or 1 everywhere without dropout.
void oracle_dropout_z(const oracle_dropout* dr, int64_t bh, int64_t i0, int64_t nq, int64_t nk,
                      double* z) {
  for (int64_t r = 0; r < nq; ++r)
    for (int64_t j = 0; j < nk; ++j) z[r * nk + j] = zfac(dr, i0 + r, j, bh);
}

// Forward: O [B,Hq,Nq,D], L [B,Hq,Nq].
void oracle_fwd(const double* Q, const double* K, const double* V, int64_t B,
                int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t D, int causal,
                double scale, const oracle_dropout* dr, double* O, double* L) {
  const Dims dm{B, Hq, Hkv, Nq, Nk, D};
#pragma omp parallel
  {
    std::vector<double> p(static_cast<size_t>(Nk)), z(static_cast<size_t>(Nk));
#pragma omp for schedule(dynamic, 16)
    for (int64_t r = 0; r < B * Hq * Nq; ++r) {
      const int64_t qh = r / Nq, i = r % Nq;
      query_row(dm, Q, K, V, nullptr, causal, scale, dr, qh, i, p, z,
                O + dm.qbase(qh) + i * D, L + qh * Nq + i, nullptr, nullptr, nullptr,
                nullptr);
    }
  }
}

// Forward for a list of sampled rows.  rows[2*t] = flat query head b*Hq+h,
// rows[2*t+1] = query index i.  O_rows [n_rows, D], L_rows [n_rows].
void oracle_fwd_rows(const double* Q, const double* K, const double* V, int64_t B,
                     int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t D,
                     int causal, double scale, const oracle_dropout* dr, int64_t n_rows,
                     const int64_t* rows, double* O_rows, double* L_rows) {
  const Dims dm{B, Hq, Hkv, Nq, Nk, D};
#pragma omp parallel
  {
    std::vector<double> p(static_cast<size_t>(Nk)), z(static_cast<size_t>(Nk));
#pragma omp for schedule(dynamic, 1)
    for (int64_t t = 0; t < n_rows; ++t)
      query_row(dm, Q, K, V, nullptr, causal, scale, dr, rows[2 * t], rows[2 * t + 1], p, z,
                O_rows + t * D, L_rows + t, nullptr, nullptr, nullptr, nullptr);
  }
}

// Forward and backward.  Outputs O, L, Delta, dQ (query-shaped) and dK, dV
// (key-shaped): pass 1 over every query row, then pass 2 over every key row.
void oracle_fwd_bwd(const double* Q, const double* K, const double* V, const double* dO,
                    int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t D,
                    int causal, double scale, const oracle_dropout* dr, double* O,
                    double* L, double* Delta, double* dQ, double* dK, double* dV) {
  const Dims dm{B, Hq, Hkv, Nq, Nk, D};
#pragma omp parallel
  {
    std::vector<double> p(static_cast<size_t>(Nk)), z(static_cast<size_t>(Nk));
#pragma omp for schedule(dynamic, 16)
    for (int64_t r = 0; r < B * Hq * Nq; ++r) {
      const int64_t qh = r / Nq, i = r % Nq;
      const int64_t at = dm.qbase(qh) + i * D;
      query_row(dm, Q, K, V, dO, causal, scale, dr, qh, i, p, z, O + at, L + qh * Nq + i,
                Delta + qh * Nq + i, dQ + at, nullptr, nullptr);
    }
#pragma omp for schedule(dynamic, 16)
    for (int64_t r = 0; r < B * Hkv * Nk; ++r) {
      const int64_t kh = r / Nk, j = r % Nk;
      const int64_t at = kh * Nk * D + j * D;
      key_row(dm, Q, K, V, dO, L, Delta, causal, scale, dr, kh, j, dK + at, dV + at, nullptr,
              nullptr);
    }
  }
}

// Sampled query rows: O_i, L_i, Delta_i and dQ_i are row-local (they need
// only query row i and every key), so they are computed one row at a time
// with pass 1.  rows[2*t] = flat query head b*Hq+h, rows[2*t+1] = i.
// Oabs_rows / dQabs_rows: the magnitude sums of oracle_magnitudes, or null.
void oracle_query_rows(const double* Q, const double* K, const double* V, const double* dO,
                       int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk,
                       int64_t D, int causal, double scale, const oracle_dropout* dr,
                       int64_t n_rows, const int64_t* rows, double* O_rows, double* L_rows,
                       double* Delta_rows, double* dQ_rows, double* Oabs_rows,
                       double* dQabs_rows) {
  const Dims dm{B, Hq, Hkv, Nq, Nk, D};
#pragma omp parallel
  {
    std::vector<double> p(static_cast<size_t>(Nk)), z(static_cast<size_t>(Nk));
#pragma omp for schedule(dynamic, 1)
    for (int64_t t = 0; t < n_rows; ++t)
      query_row(dm, Q, K, V, dO, causal, scale, dr, rows[2 * t], rows[2 * t + 1], p, z,
                O_rows + t * D, L_rows + t, Delta_rows + t, dQ_rows + t * D,
                Oabs_rows ? Oabs_rows + t * D : nullptr,
                dQabs_rows ? dQabs_rows + t * D : nullptr);
  }
}

// Sampled key rows: dK_j and dV_j need L_i and Delta_i of every query of the
// query heads that read key/value head kh, so those are computed first (pass
// 1 without dQ), then pass 2 runs for the sampled keys only.
// rows[2*t] = flat key/value head b*Hkv+hk, rows[2*t+1] = key index j.
void oracle_key_rows(const double* Q, const double* K, const double* V, const double* dO,
                     int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t D,
                     int causal, double scale, const oracle_dropout* dr, int64_t n_rows,
                     const int64_t* rows, double* dK_rows, double* dV_rows,
                     double* dKabs_rows, double* dVabs_rows) {
  const Dims dm{B, Hq, Hkv, Nq, Nk, D};
  const int64_t G = dm.G();
  std::vector<int64_t> qheads;
  for (int64_t t = 0; t < n_rows; ++t) {
    const int64_t kh = rows[2 * t];
    for (int64_t g = 0; g < G; ++g) qheads.push_back((kh / Hkv) * Hq + (kh % Hkv) * G + g);
  }
  std::sort(qheads.begin(), qheads.end());
  qheads.erase(std::unique(qheads.begin(), qheads.end()), qheads.end());
  std::vector<double> L(static_cast<size_t>(B * Hq * Nq)), Delta(L.size());
  stats_for_heads(dm, Q, K, V, dO, causal, scale, dr, qheads, L.data(), Delta.data());
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t t = 0; t < n_rows; ++t)
    key_row(dm, Q, K, V, dO, L.data(), Delta.data(), causal, scale, dr, rows[2 * t],
            rows[2 * t + 1], dK_rows + t * D, dV_rows + t * D,
            dKabs_rows ? dKabs_rows + t * D : nullptr, dVabs_rows ? dVabs_rows + t * D : nullptr);
}

// Componentwise magnitude sums of the same products, for rounding-error
// bounds: a sum of products whose factors each carry a relative error of at
// most u deviates from the exact sum by at most u times the sum of the
// products' absolute values (the standard componentwise bound).
//   Oabs_id  = sum_j Z P_ij |V_jd|         dVabs_jd = sum_i Z P_ij |dO_id|
//   dQabs_id = scale sum_j |dS_ij| |K_jd|  dKabs_jd = scale sum_i |dS_ij| |Q_id|
// with P, Z, dS as in oracle_fwd_bwd (P, Z >= 0, so no absolute value is
// needed on them).
void oracle_magnitudes(const double* Q, const double* K, const double* V, const double* dO,
                       int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t D,
                       int causal, double scale, const oracle_dropout* dr, double* Oabs,
                       double* dQabs, double* dKabs, double* dVabs) {
  const Dims dm{B, Hq, Hkv, Nq, Nk, D};
  std::vector<double> L(static_cast<size_t>(B * Hq * Nq)), Delta(L.size());
#pragma omp parallel
  {
    std::vector<double> p(static_cast<size_t>(Nk)), z(static_cast<size_t>(Nk)),
        oi(static_cast<size_t>(D)), dqi(static_cast<size_t>(D));
#pragma omp for schedule(dynamic, 16)
    for (int64_t r = 0; r < B * Hq * Nq; ++r) {
      const int64_t qh = r / Nq, i = r % Nq;
      const int64_t at = dm.qbase(qh) + i * D;
      query_row(dm, Q, K, V, dO, causal, scale, dr, qh, i, p, z, oi.data(), &L[qh * Nq + i],
                &Delta[qh * Nq + i], dqi.data(), Oabs + at, dQabs + at);
    }
#pragma omp for schedule(dynamic, 16)
    for (int64_t r = 0; r < B * Hkv * Nk; ++r) {
      const int64_t kh = r / Nk, j = r % Nk;
      const int64_t at = kh * Nk * D + j * D;
      std::vector<double> dk(static_cast<size_t>(D)), dv(static_cast<size_t>(D));
      key_row(dm, Q, K, V, dO, L.data(), Delta.data(), causal, scale, dr, kh, j, dk.data(),
              dv.data(), dKabs + at, dVabs + at);
    }
  }
}

// Dense materialisation, for small N: the full N x N score and probability
// matrices are built per head, then every product is an explicit matrix loop.
// P is written to P_out [B,H,N,N] (masked entries exactly 0) when non-null.
// A second code path for the same definition; the tests cross-check it
// against oracle_fwd_bwd.
void oracle_dense(const double* Q, const double* K, const double* V,
                  const double* dO, int64_t B, int64_t H, int64_t N, int64_t D,
                  int causal, double scale, double* O, double* L, double* dQ,
                  double* dK, double* dV, double* P_out) {
  const int64_t BH = B * H;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bh = 0; bh < BH; ++bh) {
    const int64_t base = bh * N * D;
    const double* q = Q + base; const double* k = K + base;
    const double* v = V + base; const double* g = dO ? dO + base : nullptr;
    std::vector<double> S(N * N), P(N * N), dP(N * N), dS(N * N);
    std::vector<unsigned char> keep(N * N);
    for (int64_t i = 0; i < N; ++i)
      for (int64_t j = 0; j < N; ++j) {
        keep[i * N + j] = (!causal || j <= i) ? 1 : 0;
        double acc = 0.0;
        for (int64_t d = 0; d < D; ++d) acc += q[i * D + d] * k[j * D + d];
        S[i * N + j] = scale * acc;
      }
    for (int64_t i = 0; i < N; ++i) {
      double m = -std::numeric_limits<double>::infinity();
      for (int64_t j = 0; j < N; ++j) if (keep[i * N + j]) m = std::max(m, S[i * N + j]);
      double sum = 0.0;
      for (int64_t j = 0; j < N; ++j) if (keep[i * N + j]) sum += std::exp(S[i * N + j] - m);
      const double Li = m + std::log(sum);
      L[bh * N + i] = Li;
      for (int64_t j = 0; j < N; ++j)
        P[i * N + j] = keep[i * N + j] ? std::exp(S[i * N + j] - Li) : 0.0;
    }
    double* o = O + base;
    for (int64_t i = 0; i < N; ++i)
      for (int64_t d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int64_t j = 0; j < N; ++j) acc += P[i * N + j] * v[j * D + d];
        o[i * D + d] = acc;
      }
    if (P_out) std::memcpy(P_out + bh * N * N, P.data(), sizeof(double) * N * N);
    if (!g) continue;
    // dV = P^T dO ; dP = dO V^T ; Delta = rowsum(dO o O) ; dS = P o (dP - Delta)
    // dQ = scale dS K ; dK = scale dS^T Q
    std::vector<double> delta(N);
    for (int64_t i = 0; i < N; ++i) {
      double acc = 0.0;
      for (int64_t d = 0; d < D; ++d) acc += g[i * D + d] * o[i * D + d];
      delta[i] = acc;
    }
    for (int64_t i = 0; i < N; ++i)
      for (int64_t j = 0; j < N; ++j) {
        double acc = 0.0;
        for (int64_t d = 0; d < D; ++d) acc += g[i * D + d] * v[j * D + d];
        dP[i * N + j] = acc;
        dS[i * N + j] = P[i * N + j] * (acc - delta[i]);
      }
    for (int64_t j = 0; j < N; ++j)
      for (int64_t d = 0; d < D; ++d) {
        double av = 0.0, ak = 0.0;
        for (int64_t i = 0; i < N; ++i) {
          av += P[i * N + j] * g[i * D + d];
          ak += dS[i * N + j] * q[i * D + d];
        }
        dV[base + j * D + d] = av;
        dK[base + j * D + d] = scale * ak;
      }
    for (int64_t i = 0; i < N; ++i)
      for (int64_t d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int64_t j = 0; j < N; ++j) acc += dS[i * N + j] * k[j * D + d];
        dQ[base + i * D + d] = scale * acc;
      }
  }
}

// Tiled FlashAttention-2 forward in fp64, with query tiles of bq rows and key
// tiles of bk rows, restated from "FlashAttention-2 from PyTorch to Triton"
// (the PyTorch reference's double loop and the running quantities m, l, O):
//   for each query tile:  m = -inf, l = 0, O = 0
//     for each key tile (stopping after the tile holding the tile's last
//     allowed key when causal):
//       S = scale Q_i K_j^T with excluded keys at -inf
//       m_new = max(m, rowmax S);  P~ = exp(S - m_new);  a = exp(m - m_new)
//       l = a l + rowsum P~;        O = a O + P~ V_j;      m = m_new
//     O /= l;  L = m + log l
// Used only by the tile-invariance pin.
void oracle_fwd_tiled(const double* Q, const double* K, const double* V,
                      int64_t B, int64_t H, int64_t N, int64_t D, int causal,
                      double scale, int64_t bq, int64_t bk, double* O,
                      double* L) {
  const int64_t BH = B * H;
  const double ninf = -std::numeric_limits<double>::infinity();
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bh = 0; bh < BH; ++bh) {
    const int64_t base = bh * N * D;
    std::vector<double> m(bq), l(bq), acc(bq * D), S(bq * bk);
    for (int64_t q0 = 0; q0 < N; q0 += bq) {
      const int64_t nq = std::min(bq, N - q0);
      std::fill(m.begin(), m.end(), ninf);
      std::fill(l.begin(), l.end(), 0.0);
      std::fill(acc.begin(), acc.end(), 0.0);
      const int64_t kend = causal ? std::min(N, q0 + nq) : N;
      for (int64_t k0 = 0; k0 < kend; k0 += bk) {
        const int64_t nkt = std::min(bk, N - k0);
        for (int64_t a = 0; a < nq; ++a) {
          const int64_t i = q0 + a;
          double rowmax = ninf;
          for (int64_t b = 0; b < nkt; ++b) {
            const int64_t j = k0 + b;
            double s = ninf;
            if (!causal || j <= i) s = scale * dot(Q + base + i * D, K + base + j * D, D);
            S[a * bk + b] = s;
            rowmax = std::max(rowmax, s);
          }
          const double m_new = std::max(m[a], rowmax);
          const double alpha = (m[a] == ninf) ? 0.0 : std::exp(m[a] - m_new);
          double rowsum = 0.0;
          for (int64_t d = 0; d < D; ++d) acc[a * D + d] *= alpha;
          for (int64_t b = 0; b < nkt; ++b) {
            const double s = S[a * bk + b];
            const double pt = (s == ninf) ? 0.0 : std::exp(s - m_new);
            rowsum += pt;
            const double* vj = V + base + (k0 + b) * D;
            for (int64_t d = 0; d < D; ++d) acc[a * D + d] += pt * vj[d];
          }
          l[a] = alpha * l[a] + rowsum;
          m[a] = m_new;
        }
      }
      for (int64_t a = 0; a < nq; ++a) {
        const int64_t i = q0 + a;
        for (int64_t d = 0; d < D; ++d) O[base + i * D + d] = acc[a * D + d] / l[a];
        L[bh * N + i] = m[a] + std::log(l[a]);
      }
    }
  }
}

// Tiled FlashAttention-2 backward in fp64 ("Triton FlashAttention": P rebuilt
// from the saved log-sum-exp; "FlashAttention-2 from PyTorch to Triton",
// defect 5: an outer loop over key tiles, an inner loop over query tiles, with
// the precomputed Delta = rowsum(dO o O)).  dQ is accumulated directly.
// O and L come from oracle_fwd_tiled with the same tiles.
void oracle_bwd_tiled(const double* Q, const double* K, const double* V,
                      const double* O, const double* L, const double* dO,
                      int64_t B, int64_t H, int64_t N, int64_t D, int causal,
                      double scale, int64_t bq, int64_t bk, double* dQ,
                      double* dK, double* dV) {
  const int64_t BH = B * H;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bh = 0; bh < BH; ++bh) {
    const int64_t base = bh * N * D;
    std::vector<double> delta(N);
    for (int64_t i = 0; i < N; ++i)
      delta[i] = dot(dO + base + i * D, O + base + i * D, D);
    for (int64_t x = 0; x < N * D; ++x) { dQ[base + x] = 0.0; }
    std::vector<double> P(bq * bk), dS(bq * bk);
    for (int64_t k0 = 0; k0 < N; k0 += bk) {
      const int64_t nkt = std::min(bk, N - k0);
      std::vector<double> dk(nkt * D, 0.0), dv(nkt * D, 0.0);
      const int64_t qstart = causal ? (k0 / bq) * bq : 0;
      for (int64_t q0 = qstart; q0 < N; q0 += bq) {
        const int64_t nq = std::min(bq, N - q0);
        for (int64_t a = 0; a < nq; ++a) {
          const int64_t i = q0 + a;
          for (int64_t b = 0; b < nkt; ++b) {
            const int64_t j = k0 + b;
            double p = 0.0, ds = 0.0;
            if (!causal || j <= i) {
              p = std::exp(scale * dot(Q + base + i * D, K + base + j * D, D) - L[bh * N + i]);
              const double dp = dot(dO + base + i * D, V + base + j * D, D);
              ds = p * (dp - delta[i]);
            }
            P[a * bk + b] = p;
            dS[a * bk + b] = ds;
          }
        }
        for (int64_t b = 0; b < nkt; ++b)
          for (int64_t a = 0; a < nq; ++a) {
            const double p = P[a * bk + b], ds = dS[a * bk + b];
            const double* doi = dO + base + (q0 + a) * D;
            const double* qi = Q + base + (q0 + a) * D;
            for (int64_t d = 0; d < D; ++d) {
              dv[b * D + d] += p * doi[d];
              dk[b * D + d] += ds * qi[d];
            }
          }
        for (int64_t a = 0; a < nq; ++a)
          for (int64_t b = 0; b < nkt; ++b) {
            const double ds = dS[a * bk + b];
            const double* kj = K + base + (k0 + b) * D;
            double* dqi = dQ + base + (q0 + a) * D;
            for (int64_t d = 0; d < D; ++d) dqi[d] += scale * ds * kj[d];
          }
      }
      for (int64_t b = 0; b < nkt; ++b)
        for (int64_t d = 0; d < D; ++d) {
          dK[base + (k0 + b) * D + d] = scale * dk[b * D + d];
          dV[base + (k0 + b) * D + d] = dv[b * D + d];
        }
    }
  }
}

}  // extern "C"
