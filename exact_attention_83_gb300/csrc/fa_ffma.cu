// FFMA (IEEE fp32) kernels: forward, dK/dV and dQ.
//
// These serve fp32 inputs, whose products must not drop to TF32 ("Triton
// FlashAttention", lessons: IEEE-precision dot products for fp32 inputs;
// "FlashAttention-2 from PyTorch to Triton", the harness note on tl.dot and
// TF32), and any (D, dtype) without a tensor-core kernel.  Every product and
// sum is an fp32 FMA; exponentials and logarithms are the full-precision
// exp2f/log2f.
//
// Tiling: 64 query rows x 64 keys per step, 256 threads as a 16 x 16 grid.
// Thread (ty, tx) owns rows 4*ty .. 4*ty+3 and the strided columns
// tx + 16*b (b < 4) of each 64 x 64 score tile, and columns tx + 16*e of each
// 64 x D accumulator.  Tiles are staged in shared memory as fp32 with one
// column of padding (conflict-free strided reads).  Global offsets are int64.
//
// Online softmax in the forward follows "FlashAttention-2 from PyTorch to
// Triton" (running max and sum in fp32, exp2 on scores pre-scaled by
// scale*log2(e), the accumulator rescaled when the max moves, one division at
// the end) and "Triton FlashAttention" (causal key tiles above the diagonal
// are never visited).  The backward follows the FlashAttention-2 split of
// "Triton FlashAttention": one kernel per key tile for dK/dV looping over query
// tiles, one kernel per query tile for dQ, both rebuilding P = exp(S - L).
//
// The kernels take the general geometry of fa_internal.h: each CTA resolves
// its sequence view (packed offsets, lengths Nq != Nk), query head h reads
// key/value head h / (Hq / Hkv), the dK/dV kernel of a key/value head loops
// over every query head of its group, and sequences without keys give dQ = 0
// (and keys nobody attends dK = dV = 0).  With dropout each weight's keep
// decision comes from the shared Philox mask (keep8), scaled by 1 / (1 - p).

#include "fa_internal.h"

#include <cmath>

namespace fa {
namespace {

constexpr int BT = 64;        // rows per tile (queries and keys)
constexpr int NT = 256;       // threads per CTA
constexpr int PLD = BT + 1;   // leading dimension of 64 x 64 smem tiles

// Stage rows [row0, row0 + 64) of a strided N x D matrix as fp32 [64][D + 1];
// rows at or past N are zero.
template <typename T, int D>
__device__ __forceinline__ void stage_tile(float* dst, const T* base, int64_t sn,
                                           int64_t row0, int64_t N) {
  constexpr int LD = D + 1;
  for (int idx = threadIdx.x; idx < BT * D; idx += NT) {
    const int r = idx / D, d = idx % D;
    const int64_t row = row0 + r;
    dst[r * LD + d] = row < N ? Elem<T>::load(base + row * sn + d) : 0.f;
  }
}

struct FfmaArgs {
  const void* q; const void* k; const void* v; const void* dout;
  void* o; float* lse; const float* lse_in; const float* delta;
  void* dq; void* dk; void* dv;
  Geo g;
  int64_t BH, ntiles;    // flat heads of the grid (B*Hq, or B*Hkv for dK/dV) and tiles
  int64_t sq[4], sk[4], sv[4], so[4], sdo[4], sdq[4], sdk[4], sdv[4];
  int causal;
  float scale;
  Dropout drop;
  unsigned int* status;
  const BwdParams* bp;   // host-side only: the call's parameters (profiling events)
};

// Linear block id -> (bh, tile).  With heavy_last_tile, the block order runs
// from the last tile to the first so that, under a causal mask, the longest
// rows start first.
__device__ __forceinline__ void block_coords(const FfmaArgs& a, bool heavy_last_tile,
                                             int64_t& bh, int64_t& tile) {
  const int64_t id = blockIdx.x;
  bh = id % a.BH;
  const int64_t t = id / a.BH;
  tile = heavy_last_tile ? (a.ntiles - 1 - t) : t;
}

// Dropout factor Z_ij of query i, key j (positions in the sequence) of flat
// query head bhq: 1 / (1 - p) if kept, else 0.
__device__ __forceinline__ float drop_factor(const Dropout& d, int64_t i, int64_t j, int64_t bhq) {
  const uint32_t bits = keep8(d, static_cast<uint32_t>(j >> 3), static_cast<uint32_t>(i),
                              static_cast<uint32_t>(bhq));
  return ((bits >> (j & 7)) & 1u) ? d.rscale : 0.f;
}

template <typename T, int D>
__global__ void __launch_bounds__(NT) fwd_ffma_kernel(FfmaArgs a) {
  extern __shared__ float sm[];
  constexpr int LD = D + 1, E = D / 16;
  float* Qs = sm;
  float* Ks = Qs + BT * LD;
  float* Vs = Ks + BT * LD;
  float* Ps = Vs + BT * LD;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  int64_t bh, qt;
  block_coords(a, a.causal != 0, bh, qt);
  const int64_t h = bh % a.g.Hq, hk = h / a.g.G;
  const SeqView sv = seq_view(a.g, bh / a.g.Hq);
  if (!sv.ok) {
    if (threadIdx.x == 0) record_status(a.status, FA_ERR_SEQLENS);
    return;
  }
  const int64_t Nq = sv.nq, Nk = sv.nk;
  const int64_t q0 = qt * BT;
  if (q0 >= Nq) return;
  const T* q = static_cast<const T*>(a.q) + sv.b * a.sq[0] + h * a.sq[1] + sv.q0 * a.sq[2];
  const T* k = static_cast<const T*>(a.k) + sv.b * a.sk[0] + hk * a.sk[1] + sv.k0 * a.sk[2];
  const T* v = static_cast<const T*>(a.v) + sv.b * a.sv[0] + hk * a.sv[1] + sv.k0 * a.sv[2];
  T* o = static_cast<T*>(a.o) + sv.b * a.so[0] + h * a.so[1] + sv.q0 * a.so[2];
  stage_tile<T, D>(Qs, q, a.sq[2], q0, Nq);

  const float c = a.scale * kLog2e;   // scores are kept in the log2 domain
  float m[4], l[4], acc[4][E];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m[i] = -INFINITY; l[i] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[i][e] = 0.f;
  }
  const int64_t kend = a.causal ? min(Nk, q0 + BT) : Nk;
  for (int64_t k0 = 0; k0 < kend; k0 += BT) {
    __syncthreads();
    stage_tile<T, D>(Ks, k, a.sk[2], k0, Nk);
    stage_tile<T, D>(Vs, v, a.sv[2], k0, Nk);
    __syncthreads();
    float s[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) s[i][j] = 0.f;
#pragma unroll 4
    for (int d = 0; d < D; ++d) {
      float qv[4], kv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) qv[i] = Qs[(ty * 4 + i) * LD + d];
#pragma unroll
      for (int j = 0; j < 4; ++j) kv[j] = Ks[(tx + 16 * j) * LD + d];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) s[i][j] = fmaf(qv[i], kv[j], s[i][j]);
    }
    // Ragged keys past N and (on the diagonal tile) keys after the query are
    // excluded.  Interior tiles skip the test.
    const bool edge = (k0 + BT > Nk) || (a.causal && k0 + BT - 1 > q0);
    if (edge) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int64_t kp = k0 + tx + 16 * j, qp = q0 + ty * 4 + i;
          if (kp >= Nk || (a.causal && kp > qp)) s[i][j] = -INFINITY;
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float mx = fmaxf(fmaxf(s[i][0], s[i][1]), fmaxf(s[i][2], s[i][3]));
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float m_new = fmaxf(m[i], mx * c);
      const float alpha = (m[i] == -INFINITY) ? 0.f : exp2f(m[i] - m_new);
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float p = exp2f(fmaf(s[i][j], c, -m_new));
        // l sums the undropped weights; P V takes the dropped, rescaled ones
        const float z = a.drop.on ? drop_factor(a.drop, q0 + ty * 4 + i, k0 + tx + 16 * j, bh) : 1.f;
        Ps[(ty * 4 + i) * PLD + tx + 16 * j] = p * z;
        sum += p;
      }
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      l[i] = fmaf(l[i], alpha, sum);
      m[i] = m_new;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[i][e] *= alpha;
    }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < BT; ++kk) {
      float p[4], vv[E];
#pragma unroll
      for (int i = 0; i < 4; ++i) p[i] = Ps[(ty * 4 + i) * PLD + kk];
#pragma unroll
      for (int e = 0; e < E; ++e) vv[e] = Vs[kk * LD + tx + 16 * e];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int e = 0; e < E; ++e) acc[i][e] = fmaf(p[i], vv[e], acc[i][e]);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t row = q0 + ty * 4 + i;
    if (row >= Nq) continue;
    // a row with no key at all (empty key sequence): O = 0, L = -inf
    const bool any = l[i] > 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e)
      o[row * a.so[2] + tx + 16 * e] = Elem<T>::from_f32(any ? acc[i][e] / l[i] : 0.f);
    if (tx == 0)
      a.lse[lse_index(a.g, sv, h, row)] = l[i] > 0.f ? (m[i] + log2f(l[i])) * kLn2 : -INFINITY;
  }
}

// dK/dV: one CTA per (head, key tile); loops over the query tiles that may
// attend to it (from the diagonal tile when causal).
template <typename T, int D>
__global__ void __launch_bounds__(NT) bwd_dkdv_ffma_kernel(FfmaArgs a) {
  extern __shared__ float sm[];
  constexpr int LD = D + 1, E = D / 16;
  float* Ks = sm;
  float* Vs = Ks + BT * LD;
  float* Qs = Vs + BT * LD;
  float* dOs = Qs + BT * LD;
  float* Ps = dOs + BT * LD;
  float* dSs = Ps + BT * PLD;
  float* L2s = dSs + BT * PLD;   // L * log2(e) of the staged query rows
  float* Dls = L2s + BT;         // Delta of the staged query rows
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  int64_t bhk, kt;
  block_coords(a, false, bhk, kt);
  const int64_t bseq = bhk / a.g.Hkv, hk = bhk % a.g.Hkv;
  const SeqView sv = seq_view(a.g, bseq);
  if (!sv.ok) {
    if (threadIdx.x == 0) record_status(a.status, FA_ERR_SEQLENS);
    return;
  }
  const int64_t Nq = sv.nq, Nk = sv.nk;
  const int64_t k0 = kt * BT;
  if (k0 >= Nk) return;
  const T* k = static_cast<const T*>(a.k) + sv.b * a.sk[0] + hk * a.sk[1] + sv.k0 * a.sk[2];
  const T* v = static_cast<const T*>(a.v) + sv.b * a.sv[0] + hk * a.sv[1] + sv.k0 * a.sv[2];
  stage_tile<T, D>(Ks, k, a.sk[2], k0, Nk);
  stage_tile<T, D>(Vs, v, a.sv[2], k0, Nk);
  const float c = a.scale * kLog2e;
  float dk[4][E], dv[4][E];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int e = 0; e < E; ++e) { dk[i][e] = 0.f; dv[i][e] = 0.f; }

  // every query head that reads this key/value head, then its query tiles
  for (int64_t hg = 0; hg < a.g.G; ++hg)
  for (int64_t q0 = a.causal ? k0 : 0; q0 < Nq; q0 += BT) {
    const int64_t h = hk * a.g.G + hg, bhq = bseq * a.g.Hq + h;
    const T* q = static_cast<const T*>(a.q) + sv.b * a.sq[0] + h * a.sq[1] + sv.q0 * a.sq[2];
    const T* g = static_cast<const T*>(a.dout) + sv.b * a.sdo[0] + h * a.sdo[1] + sv.q0 * a.sdo[2];
    __syncthreads();
    stage_tile<T, D>(Qs, q, a.sq[2], q0, Nq);
    stage_tile<T, D>(dOs, g, a.sdo[2], q0, Nq);
    if (threadIdx.x < BT) {
      const int64_t row = q0 + threadIdx.x;
      const int64_t li = lse_index(a.g, sv, h, row);
      L2s[threadIdx.x] = row < Nq ? a.lse_in[li] * kLog2e : 0.f;
      Dls[threadIdx.x] = row < Nq ? a.delta[li] : 0.f;
    }
    __syncthreads();
    // Transposed score and dP tiles: element (key 4*ty+i, query tx+16*j).
    float s[4][4], dp[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) { s[i][j] = 0.f; dp[i][j] = 0.f; }
#pragma unroll 2
    for (int d = 0; d < D; ++d) {
      float kv[4], vv[4], qv[4], gv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) { kv[i] = Ks[(ty * 4 + i) * LD + d]; vv[i] = Vs[(ty * 4 + i) * LD + d]; }
#pragma unroll
      for (int j = 0; j < 4; ++j) { qv[j] = Qs[(tx + 16 * j) * LD + d]; gv[j] = dOs[(tx + 16 * j) * LD + d]; }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          s[i][j] = fmaf(kv[i], qv[j], s[i][j]);
          dp[i][j] = fmaf(vv[i], gv[j], dp[i][j]);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int ql = tx + 16 * j;
        const int64_t qp = q0 + ql, kp = k0 + ty * 4 + i;
        const bool keep = qp < Nq && (!a.causal || kp <= qp);
        const float p = keep ? exp2f(fmaf(s[i][j], c, -L2s[ql])) : 0.f;
        // dropout: dV takes P o Z, dS = P o (Z o dP - Delta)
        const float z = a.drop.on ? drop_factor(a.drop, qp, kp, bhq) : 1.f;
        Ps[(ty * 4 + i) * PLD + ql] = p * z;
        dSs[(ty * 4 + i) * PLD + ql] = p * fmaf(z, dp[i][j], -Dls[ql]);
      }
    __syncthreads();
#pragma unroll 2
    for (int qq = 0; qq < BT; ++qq) {
      float p[4], ds[4], gv[E], qv[E];
#pragma unroll
      for (int i = 0; i < 4; ++i) { p[i] = Ps[(ty * 4 + i) * PLD + qq]; ds[i] = dSs[(ty * 4 + i) * PLD + qq]; }
#pragma unroll
      for (int e = 0; e < E; ++e) { gv[e] = dOs[qq * LD + tx + 16 * e]; qv[e] = Qs[qq * LD + tx + 16 * e]; }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int e = 0; e < E; ++e) {
          dv[i][e] = fmaf(p[i], gv[e], dv[i][e]);
          dk[i][e] = fmaf(ds[i], qv[e], dk[i][e]);
        }
    }
  }
  T* dkp = static_cast<T*>(a.dk) + sv.b * a.sdk[0] + hk * a.sdk[1] + sv.k0 * a.sdk[2];
  T* dvp = static_cast<T*>(a.dv) + sv.b * a.sdv[0] + hk * a.sdv[1] + sv.k0 * a.sdv[2];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t row = k0 + ty * 4 + i;
    if (row >= Nk) continue;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      dkp[row * a.sdk[2] + tx + 16 * e] = Elem<T>::from_f32(dk[i][e] * a.scale);
      dvp[row * a.sdv[2] + tx + 16 * e] = Elem<T>::from_f32(dv[i][e]);
    }
  }
}

// dQ: one CTA per (head, query tile); loops over the key tiles it attends to.
template <typename T, int D>
__global__ void __launch_bounds__(NT) bwd_dq_ffma_kernel(FfmaArgs a) {
  extern __shared__ float sm[];
  constexpr int LD = D + 1, E = D / 16;
  float* Qs = sm;
  float* dOs = Qs + BT * LD;
  float* Ks = dOs + BT * LD;
  float* Vs = Ks + BT * LD;
  float* dSs = Vs + BT * LD;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  int64_t bh, qt;
  block_coords(a, a.causal != 0, bh, qt);
  const int64_t h = bh % a.g.Hq, hk = h / a.g.G;
  const SeqView sv = seq_view(a.g, bh / a.g.Hq);
  if (!sv.ok) {
    if (threadIdx.x == 0) record_status(a.status, FA_ERR_SEQLENS);
    return;
  }
  const int64_t Nq = sv.nq, Nk = sv.nk;
  const int64_t q0 = qt * BT;
  if (q0 >= Nq) return;
  const T* q = static_cast<const T*>(a.q) + sv.b * a.sq[0] + h * a.sq[1] + sv.q0 * a.sq[2];
  const T* k = static_cast<const T*>(a.k) + sv.b * a.sk[0] + hk * a.sk[1] + sv.k0 * a.sk[2];
  const T* v = static_cast<const T*>(a.v) + sv.b * a.sv[0] + hk * a.sv[1] + sv.k0 * a.sv[2];
  const T* g = static_cast<const T*>(a.dout) + sv.b * a.sdo[0] + h * a.sdo[1] + sv.q0 * a.sdo[2];
  stage_tile<T, D>(Qs, q, a.sq[2], q0, Nq);
  stage_tile<T, D>(dOs, g, a.sdo[2], q0, Nq);
  const float c = a.scale * kLog2e;
  float L2[4], Dl[4], dq[4][E];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t row = q0 + ty * 4 + i;
    const int64_t li = lse_index(a.g, sv, h, row);
    L2[i] = row < Nq ? a.lse_in[li] * kLog2e : 0.f;
    Dl[i] = row < Nq ? a.delta[li] : 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) dq[i][e] = 0.f;
  }
  const int64_t kend = a.causal ? min(Nk, q0 + BT) : Nk;
  for (int64_t k0 = 0; k0 < kend; k0 += BT) {
    __syncthreads();
    stage_tile<T, D>(Ks, k, a.sk[2], k0, Nk);
    stage_tile<T, D>(Vs, v, a.sv[2], k0, Nk);
    __syncthreads();
    float s[4][4], dp[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) { s[i][j] = 0.f; dp[i][j] = 0.f; }
#pragma unroll 2
    for (int d = 0; d < D; ++d) {
      float qv[4], gv[4], kv[4], vv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) { qv[i] = Qs[(ty * 4 + i) * LD + d]; gv[i] = dOs[(ty * 4 + i) * LD + d]; }
#pragma unroll
      for (int j = 0; j < 4; ++j) { kv[j] = Ks[(tx + 16 * j) * LD + d]; vv[j] = Vs[(tx + 16 * j) * LD + d]; }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          s[i][j] = fmaf(qv[i], kv[j], s[i][j]);
          dp[i][j] = fmaf(gv[i], vv[j], dp[i][j]);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t kp = k0 + tx + 16 * j, qp = q0 + ty * 4 + i;
        const bool keep = kp < Nk && (!a.causal || kp <= qp);
        const float p = keep ? exp2f(fmaf(s[i][j], c, -L2[i])) : 0.f;
        const float z = a.drop.on ? drop_factor(a.drop, qp, kp, bh) : 1.f;
        dSs[(ty * 4 + i) * PLD + tx + 16 * j] = p * fmaf(z, dp[i][j], -Dl[i]);
      }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < BT; ++kk) {
      float ds[4], kv[E];
#pragma unroll
      for (int i = 0; i < 4; ++i) ds[i] = dSs[(ty * 4 + i) * PLD + kk];
#pragma unroll
      for (int e = 0; e < E; ++e) kv[e] = Ks[kk * LD + tx + 16 * e];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int e = 0; e < E; ++e) dq[i][e] = fmaf(ds[i], kv[e], dq[i][e]);
    }
  }
  T* dqp = static_cast<T*>(a.dq) + sv.b * a.sdq[0] + h * a.sdq[1] + sv.q0 * a.sdq[2];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t row = q0 + ty * 4 + i;
    if (row >= Nq) continue;
#pragma unroll
    for (int e = 0; e < E; ++e)
      dqp[row * a.sdq[2] + tx + 16 * e] = Elem<T>::from_f32(dq[i][e] * a.scale);
  }
}

constexpr size_t fwd_smem(int D) { return sizeof(float) * (3 * BT * (D + 1) + BT * PLD); }
constexpr size_t dkdv_smem(int D) { return sizeof(float) * (4 * BT * (D + 1) + 2 * BT * PLD + 2 * BT); }
constexpr size_t dq_smem(int D) { return sizeof(float) * (4 * BT * (D + 1) + BT * PLD); }

template <typename Kern>
fa_status launch(Kern kern, size_t smem, int64_t blocks, const FfmaArgs& a, cudaStream_t s) {
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return FA_ERR_LAUNCH;
  if (blocks > 0x7fffffffLL) return FA_ERR_SHAPE;
  kern<<<dim3((unsigned)blocks), dim3(NT), smem, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

template <typename T, int D>
fa_status run_fwd(const FfmaArgs& a, cudaStream_t s) {
  return launch(fwd_ffma_kernel<T, D>, fwd_smem(D), a.BH * a.ntiles, a, s);
}
template <typename T, int D>
fa_status run_bwd(const FfmaArgs& a0, cudaStream_t s) {
  FfmaArgs a = a0;
  prof_record(*a.bp, 0, s);
  a.BH = a.g.B * a.g.Hkv; a.ntiles = (a.g.Nk + BT - 1) / BT;
  fa_status st = launch(bwd_dkdv_ffma_kernel<T, D>, dkdv_smem(D), a.BH * a.ntiles, a, s);
  if (st != FA_OK) return st;
  prof_record(*a.bp, 1, s);
  a.BH = a.g.B * a.g.Hq; a.ntiles = (a.g.Nq + BT - 1) / BT;
  st = launch(bwd_dq_ffma_kernel<T, D>, dq_smem(D), a.BH * a.ntiles, a, s);
  prof_record(*a.bp, 2, s);
  return st;
}

#define FA_DISPATCH(FN, dtype, D, a, s)                                    \
  do {                                                                     \
    switch (dtype) {                                                       \
      case FA_F32:                                                         \
        switch (D) { case 16: return FN<float, 16>(a, s); case 32: return FN<float, 32>(a, s); \
                     case 64: return FN<float, 64>(a, s); case 128: return FN<float, 128>(a, s); } \
        break;                                                             \
      case FA_F16:                                                         \
        switch (D) { case 16: return FN<__half, 16>(a, s); case 32: return FN<__half, 32>(a, s); \
                     case 64: return FN<__half, 64>(a, s); case 128: return FN<__half, 128>(a, s); } \
        break;                                                             \
      case FA_BF16:                                                        \
        switch (D) { case 16: return FN<__nv_bfloat16, 16>(a, s); case 32: return FN<__nv_bfloat16, 32>(a, s); \
                     case 64: return FN<__nv_bfloat16, 64>(a, s); case 128: return FN<__nv_bfloat16, 128>(a, s); } \
        break;                                                             \
    }                                                                      \
    return FA_ERR_ARG;                                                     \
  } while (0)

void copy4(int64_t* dst, const int64_t* src) { for (int i = 0; i < 4; ++i) dst[i] = src[i]; }

}  // namespace

fa_status launch_fwd_ffma(const FwdParams& p, cudaStream_t s) {
  FfmaArgs a{};
  a.q = p.q; a.k = p.k; a.v = p.v; a.o = p.o; a.lse = p.lse;
  a.g = p.g; a.BH = p.g.B * p.g.Hq; a.ntiles = (p.g.Nq + BT - 1) / BT;
  copy4(a.sq, p.sq); copy4(a.sk, p.sk); copy4(a.sv, p.sv); copy4(a.so, p.so);
  a.causal = p.causal; a.scale = p.scale; a.drop = p.drop; a.status = p.status;
  FA_DISPATCH(run_fwd, p.dtype, p.D, a, s);
}

fa_status launch_bwd_ffma(const BwdParams& p, cudaStream_t s) {
  FfmaArgs a{};
  a.q = p.q; a.k = p.k; a.v = p.v; a.dout = p.dout; a.lse_in = p.lse; a.delta = p.delta;
  a.dq = p.dq; a.dk = p.dk; a.dv = p.dv;
  a.g = p.g;
  copy4(a.sq, p.sq); copy4(a.sk, p.sk); copy4(a.sv, p.sv); copy4(a.sdo, p.sdo);
  copy4(a.sdq, p.sdq); copy4(a.sdk, p.sdk); copy4(a.sdv, p.sdv);
  a.causal = p.causal; a.scale = p.scale; a.drop = p.drop; a.status = p.status;
  a.bp = &p;
  FA_DISPATCH(run_bwd, p.dtype, p.D, a, s);
}

}  // namespace fa
