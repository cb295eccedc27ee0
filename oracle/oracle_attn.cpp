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
// Readings where the pages are open (each is also listed in the design notes):
//  * masked keys are excluded exactly (weight 0, never a finite sentinel);
//  * L is in natural-log units and always fp64 here;
//  * Delta uses the oracle's own fp64 O.
//
// Layout: every tensor is a dense row-major [B, H, N, D] array of doubles
// (L and Delta are [B, H, N]).  Inputs are the exact values of the rounded
// device inputs (fp16/bf16/fp32 -> double is exact).
//
// Pins: softmax rows sum to 1; closed forms for constant V, causal row 0,
// Q = 0 and N = 1; finite differences of the forward; sum_j dK_j = 0;
// sum_j dV_j = sum_i dO_i; tile-size invariance; agreement with the dense
// N x N materialisation and with a library routine.  See tests/test_oracle_pins.py.

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

// Number of keys query row i may attend to: all N, or keys 0..i when causal
// (top-left aligned mask, "FlashAttention-2 from PyTorch to Triton", kernel's
// causal predicate).
inline int64_t keys_allowed(int64_t i, int64_t N, int causal) {
  return causal ? (i + 1) : N;
}

// Forward for one query row (the plain definition).
//   s_j = scale * q_i . k_j          for allowed j
//   m   = max_j s_j
//   L   = m + log sum_j exp(s_j - m)           (= log sum_j exp(s_j))
//   p_j = exp(s_j - L)
//   o_i = sum_j p_j v_j
// `s` is scratch of at least N doubles; on return it holds p_j.
void row_forward(const double* qi, const double* K, const double* V,
                 int64_t nk, int64_t D, double scale,
                 double* s, double* oi, double* Li) {
  double m = -std::numeric_limits<double>::infinity();
  for (int64_t j = 0; j < nk; ++j) {
    s[j] = scale * dot(qi, K + j * D, D);
    m = std::max(m, s[j]);
  }
  double sum = 0.0;
  for (int64_t j = 0; j < nk; ++j) sum += std::exp(s[j] - m);
  const double L = m + std::log(sum);
  for (int64_t d = 0; d < D; ++d) oi[d] = 0.0;
  for (int64_t j = 0; j < nk; ++j) {
    s[j] = std::exp(s[j] - L);
    const double* vj = V + j * D;
    for (int64_t d = 0; d < D; ++d) oi[d] += s[j] * vj[d];
  }
  *Li = L;
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

// Forward: O [B,H,N,D], L [B,H,N].
void oracle_fwd(const double* Q, const double* K, const double* V,
                int64_t B, int64_t H, int64_t N, int64_t D,
                int causal, double scale, double* O, double* L) {
  const int64_t BH = B * H;
#pragma omp parallel
  {
    std::vector<double> s(static_cast<size_t>(N));
#pragma omp for schedule(dynamic, 16)
    for (int64_t r = 0; r < BH * N; ++r) {
      const int64_t bh = r / N, i = r % N;
      const int64_t base = bh * N * D;
      row_forward(Q + base + i * D, K + base, V + base,
                  keys_allowed(i, N, causal), D, scale, s.data(),
                  O + base + i * D, L + bh * N + i);
    }
  }
}

// Forward for a list of sampled rows.  rows[2*t] = flat head index b*H+h,
// rows[2*t+1] = query index i.  O_rows [n_rows, D], L_rows [n_rows].
void oracle_fwd_rows(const double* Q, const double* K, const double* V,
                     int64_t B, int64_t H, int64_t N, int64_t D,
                     int causal, double scale, int64_t n_rows,
                     const int64_t* rows, double* O_rows, double* L_rows) {
  (void)B; (void)H;
#pragma omp parallel
  {
    std::vector<double> s(static_cast<size_t>(N));
#pragma omp for schedule(dynamic, 1)
    for (int64_t t = 0; t < n_rows; ++t) {
      const int64_t bh = rows[2 * t], i = rows[2 * t + 1];
      const int64_t base = bh * N * D;
      row_forward(Q + base + i * D, K + base, V + base,
                  keys_allowed(i, N, causal), D, scale, s.data(),
                  O_rows + t * D, L_rows + t);
    }
  }
}

// Forward and backward.  Outputs O, L, Delta, dQ, dK, dV.
//
// Pass 1, one query row at a time (rows are independent):
//   O_i, L_i, P_i as in row_forward;
//   Delta_i = dO_i . O_i                         (rowsum(dO o O))
//   dP_ij   = dO_i . v_j
//   dS_ij   = P_ij (dP_ij - Delta_i)
//   dQ_i    = scale * sum_j dS_ij k_j
// Pass 2, one key row at a time (keys are independent):
//   for every query i that may attend to key j (all i, or i >= j if causal):
//     P_ij = exp(scale q_i.k_j - L_i),  dP_ij = dO_i . v_j,
//     dS_ij = P_ij (dP_ij - Delta_i)
//   dV_j = sum_i P_ij dO_i,   dK_j = scale * sum_i dS_ij q_i
void oracle_fwd_bwd(const double* Q, const double* K, const double* V,
                    const double* dO, int64_t B, int64_t H, int64_t N,
                    int64_t D, int causal, double scale, double* O, double* L,
                    double* Delta, double* dQ, double* dK, double* dV) {
  const int64_t BH = B * H;
#pragma omp parallel
  {
    std::vector<double> p(static_cast<size_t>(N));
#pragma omp for schedule(dynamic, 16)
    for (int64_t r = 0; r < BH * N; ++r) {
      const int64_t bh = r / N, i = r % N;
      const int64_t base = bh * N * D;
      const int64_t nk = keys_allowed(i, N, causal);
      const double* doi = dO + base + i * D;
      double* oi = O + base + i * D;
      row_forward(Q + base + i * D, K + base, V + base, nk, D, scale,
                  p.data(), oi, L + bh * N + i);
      const double delta = dot(doi, oi, D);
      Delta[bh * N + i] = delta;
      double* dqi = dQ + base + i * D;
      for (int64_t d = 0; d < D; ++d) dqi[d] = 0.0;
      for (int64_t j = 0; j < nk; ++j) {
        const double dp = dot(doi, V + base + j * D, D);
        const double ds = p[j] * (dp - delta);
        const double* kj = K + base + j * D;
        for (int64_t d = 0; d < D; ++d) dqi[d] += ds * kj[d];
      }
      for (int64_t d = 0; d < D; ++d) dqi[d] *= scale;
    }

#pragma omp for schedule(dynamic, 16)
    for (int64_t r = 0; r < BH * N; ++r) {
      const int64_t bh = r / N, j = r % N;
      const int64_t base = bh * N * D;
      const double* kj = K + base + j * D;
      const double* vj = V + base + j * D;
      double* dkj = dK + base + j * D;
      double* dvj = dV + base + j * D;
      for (int64_t d = 0; d < D; ++d) { dkj[d] = 0.0; dvj[d] = 0.0; }
      const int64_t i0 = causal ? j : 0;
      for (int64_t i = i0; i < N; ++i) {
        const double* qi = Q + base + i * D;
        const double* doi = dO + base + i * D;
        const double pij = std::exp(scale * dot(qi, kj, D) - L[bh * N + i]);
        const double dp = dot(doi, vj, D);
        const double ds = pij * (dp - Delta[bh * N + i]);
        for (int64_t d = 0; d < D; ++d) {
          dvj[d] += pij * doi[d];
          dkj[d] += ds * qi[d];
        }
      }
      for (int64_t d = 0; d < D; ++d) dkj[d] *= scale;
    }
  }
}

// Sampled query rows: O_i, L_i, Delta_i and dQ_i are row-local (they need
// only query row i and every key), so they are computed one row at a time
// with the same formulas as pass 1 of oracle_fwd_bwd.
// rows[2*t] = flat head index b*H+h, rows[2*t+1] = query index i.
void oracle_query_rows(const double* Q, const double* K, const double* V,
                       const double* dO, int64_t B, int64_t H, int64_t N,
                       int64_t D, int causal, double scale, int64_t n_rows,
                       const int64_t* rows, double* O_rows, double* L_rows,
                       double* Delta_rows, double* dQ_rows, double* Oabs_rows,
                       double* dQabs_rows) {
  (void)B; (void)H;
#pragma omp parallel
  {
    std::vector<double> p(static_cast<size_t>(N));
#pragma omp for schedule(dynamic, 1)
    for (int64_t t = 0; t < n_rows; ++t) {
      const int64_t bh = rows[2 * t], i = rows[2 * t + 1];
      const int64_t base = bh * N * D;
      const int64_t nk = keys_allowed(i, N, causal);
      const double* doi = dO + base + i * D;
      double* oi = O_rows + t * D;
      row_forward(Q + base + i * D, K + base, V + base, nk, D, scale, p.data(),
                  oi, L_rows + t);
      const double delta = dot(doi, oi, D);
      Delta_rows[t] = delta;
      double* dqi = dQ_rows + t * D;
      for (int64_t d = 0; d < D; ++d) dqi[d] = 0.0;
      for (int64_t j = 0; j < nk; ++j) {
        const double ds = p[j] * (dot(doi, V + base + j * D, D) - delta);
        const double* kj = K + base + j * D;
        for (int64_t d = 0; d < D; ++d) dqi[d] += ds * kj[d];
      }
      for (int64_t d = 0; d < D; ++d) dqi[d] *= scale;
      if (Oabs_rows == nullptr) continue;
      // magnitude sums, as in oracle_magnitudes
      double* oa = Oabs_rows + t * D;
      double* qa = dQabs_rows + t * D;
      for (int64_t d = 0; d < D; ++d) { oa[d] = 0.0; qa[d] = 0.0; }
      for (int64_t j = 0; j < nk; ++j) {
        const double* vj = V + base + j * D;
        const double* kj = K + base + j * D;
        const double ads = std::fabs(p[j] * (dot(doi, vj, D) - delta));
        for (int64_t d = 0; d < D; ++d) {
          oa[d] += p[j] * std::fabs(vj[d]);
          qa[d] += ads * std::fabs(kj[d]);
        }
      }
      for (int64_t d = 0; d < D; ++d) qa[d] *= scale;
    }
  }
}

// Sampled key rows: dK_j and dV_j need L_i and Delta_i of every query of the
// head, so those are computed first for each head that holds a sampled key
// (pass 1 of oracle_fwd_bwd without dQ), then pass 2 runs for the sampled
// keys only.  rows as in oracle_query_rows, with j in place of i.
void oracle_key_rows(const double* Q, const double* K, const double* V,
                     const double* dO, int64_t B, int64_t H, int64_t N,
                     int64_t D, int causal, double scale, int64_t n_rows,
                     const int64_t* rows, double* dK_rows, double* dV_rows,
                     double* dKabs_rows, double* dVabs_rows) {
  (void)B; (void)H;
  std::vector<int64_t> heads;
  for (int64_t t = 0; t < n_rows; ++t) heads.push_back(rows[2 * t]);
  std::sort(heads.begin(), heads.end());
  heads.erase(std::unique(heads.begin(), heads.end()), heads.end());
  std::vector<double> L(N), Delta(N);
  for (const int64_t bh : heads) {
    const int64_t base = bh * N * D;
#pragma omp parallel
    {
      std::vector<double> p(static_cast<size_t>(N)), oi(static_cast<size_t>(D));
#pragma omp for schedule(dynamic, 16)
      for (int64_t i = 0; i < N; ++i) {
        row_forward(Q + base + i * D, K + base, V + base,
                    keys_allowed(i, N, causal), D, scale, p.data(), oi.data(),
                    &L[i]);
        Delta[i] = dot(dO + base + i * D, oi.data(), D);
      }
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < n_rows; ++t) {
      if (rows[2 * t] != bh) continue;
      const int64_t j = rows[2 * t + 1];
      const double* kj = K + base + j * D;
      const double* vj = V + base + j * D;
      double* dkj = dK_rows + t * D;
      double* dvj = dV_rows + t * D;
      for (int64_t d = 0; d < D; ++d) { dkj[d] = 0.0; dvj[d] = 0.0; }
      if (dKabs_rows != nullptr)
        for (int64_t d = 0; d < D; ++d) {
          dKabs_rows[t * D + d] = 0.0;
          dVabs_rows[t * D + d] = 0.0;
        }
      for (int64_t i = causal ? j : 0; i < N; ++i) {
        const double* qi = Q + base + i * D;
        const double* doi = dO + base + i * D;
        const double pij = std::exp(scale * dot(qi, kj, D) - L[i]);
        const double ds = pij * (dot(doi, vj, D) - Delta[i]);
        for (int64_t d = 0; d < D; ++d) {
          dvj[d] += pij * doi[d];
          dkj[d] += ds * qi[d];
        }
        if (dKabs_rows == nullptr) continue;
        // magnitude sums, as in oracle_magnitudes
        double* ka = dKabs_rows + t * D;
        double* va = dVabs_rows + t * D;
        for (int64_t d = 0; d < D; ++d) {
          va[d] += pij * std::fabs(doi[d]);
          ka[d] += std::fabs(ds) * std::fabs(qi[d]);
        }
      }
      for (int64_t d = 0; d < D; ++d) dkj[d] *= scale;
      if (dKabs_rows != nullptr)
        for (int64_t d = 0; d < D; ++d) dKabs_rows[t * D + d] *= scale;
    }
  }
}

// Componentwise magnitude sums of the same products, for rounding-error
// bounds: a sum of products whose factors each carry a relative error of at
// most u deviates from the exact sum by at most u times the sum of the
// products' absolute values (the standard componentwise bound).
//   Oabs_id  = sum_j P_ij |V_jd|           dVabs_jd = sum_i P_ij |dO_id|
//   dQabs_id = scale sum_j |dS_ij| |K_jd|  dKabs_jd = scale sum_i |dS_ij| |Q_id|
// with P, dS as in oracle_fwd_bwd (P >= 0, so no absolute value is needed on it).
void oracle_magnitudes(const double* Q, const double* K, const double* V,
                       const double* dO, int64_t B, int64_t H, int64_t N,
                       int64_t D, int causal, double scale, double* Oabs,
                       double* dQabs, double* dKabs, double* dVabs) {
  const int64_t BH = B * H;
  std::vector<double> L(BH * N), Delta(BH * N);
#pragma omp parallel
  {
    std::vector<double> p(static_cast<size_t>(N)), oi(static_cast<size_t>(D));
#pragma omp for schedule(dynamic, 16)
    for (int64_t r = 0; r < BH * N; ++r) {
      const int64_t bh = r / N, i = r % N;
      const int64_t base = bh * N * D;
      const int64_t nk = keys_allowed(i, N, causal);
      const double* doi = dO + base + i * D;
      row_forward(Q + base + i * D, K + base, V + base, nk, D, scale, p.data(),
                  oi.data(), &L[bh * N + i]);
      const double delta = dot(doi, oi.data(), D);
      Delta[bh * N + i] = delta;
      double* oa = Oabs + base + i * D;
      double* qa = dQabs + base + i * D;
      for (int64_t d = 0; d < D; ++d) { oa[d] = 0.0; qa[d] = 0.0; }
      for (int64_t j = 0; j < nk; ++j) {
        const double* vj = V + base + j * D;
        const double* kj = K + base + j * D;
        const double ads = std::fabs(p[j] * (dot(doi, vj, D) - delta));
        for (int64_t d = 0; d < D; ++d) {
          oa[d] += p[j] * std::fabs(vj[d]);
          qa[d] += ads * std::fabs(kj[d]);
        }
      }
      for (int64_t d = 0; d < D; ++d) qa[d] *= scale;
    }
#pragma omp for schedule(dynamic, 16)
    for (int64_t r = 0; r < BH * N; ++r) {
      const int64_t bh = r / N, j = r % N;
      const int64_t base = bh * N * D;
      const double* kj = K + base + j * D;
      const double* vj = V + base + j * D;
      double* ka = dKabs + base + j * D;
      double* va = dVabs + base + j * D;
      for (int64_t d = 0; d < D; ++d) { ka[d] = 0.0; va[d] = 0.0; }
      for (int64_t i = causal ? j : 0; i < N; ++i) {
        const double* qi = Q + base + i * D;
        const double* doi = dO + base + i * D;
        const double pij = std::exp(scale * dot(qi, kj, D) - L[bh * N + i]);
        const double ads = std::fabs(pij * (dot(doi, vj, D) - Delta[bh * N + i]));
        for (int64_t d = 0; d < D; ++d) {
          va[d] += pij * std::fabs(doi[d]);
          ka[d] += ads * std::fabs(qi[d]);
        }
      }
      for (int64_t d = 0; d < D; ++d) ka[d] *= scale;
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
