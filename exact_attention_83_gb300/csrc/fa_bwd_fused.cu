// Single-pass tensor-core backward: dK, dV and dQ from one kernel per key
// tile, with dQ accumulated by fp32 reduce-add into a caller workspace, then
// scaled and rounded by a small convert kernel.
//
// "FlashAttention-2 from PyTorch to Triton" (defect 5) names the two ways to
// obtain dQ when the backward iterates over query tiles for each key tile:
// atomics, or a second pass.  The split backward (fa_bwd_tc.cu) is the second
// pass: a dQ kernel that rebuilds S and dP.  This file is the other one: the
// dK/dV kernel's dS tile also yields the partial dQ_i = dS_i K_j of its key
// tile, so S and dP are built once (five products per tile pair instead of
// seven).  The partial sums reach the workspace through TMA bulk tensor
// reductions (cp.reduce.async.bulk.tensor ... .add, f32), whose order between
// key tiles is not fixed: dQ is not bitwise reproducible from run to run, dK
// and dV are.
//
// Per (key tile j, query tile i), 320 threads as in the split dK/dV kernel
// (two elementwise warpgroups, a TMA producer warp, an MMA warp):
//   S^T = K_j Q_i^T,  dP^T = V_j dO_i^T      (SS products into TMEM)
//   P^T, dS^T = P^T o (dP^T - Delta)          (elementwise warps, from L, Delta)
//   dV_j += P^T dO_i,  dK_j += dS^T Q_i       (A = P^T, dS^T from TMEM)
//   dQ_i  = dS_i K_j                          (A = dS from shared memory, MN-major)
// The elementwise warps write each rounded dS^T row twice: into TMEM (the A
// operand of dK) and into a 128 x 128 shared-memory tile (key rows, query
// columns, 128-byte swizzle), which the dQ product reads as an MN-major A
// operand with the key tile K_j as an MN-major B operand.  At D = 128 that
// tile is the dO_i slot, whose last reader, dV_i, has completed by then: the
// Q ring keeps three slots.  dQ_i lands in TMEM (at D = 128 in the dP^T
// columns, free once dK_i has read dS^T); each warpgroup copies its half of
// the columns, 32 at a time, into free shared memory (fp32 rows of 128 bytes,
// swizzled; at D = 128 the dO_i and Q_i slots, whose last readers dQ_i and
// dK_i have completed) and one thread issues the TMA reduction of that
// 128 x 32 box.  That thread releases the slots to the producer once the
// reductions have read them.
//
// Schedule per step i (MMA issue order and elementwise order):
//   MMA:          dK_i, dQ_i, dV_{i+1}, dP^T_{i+1}, S^T_{i+2}
//   elementwise:  dS_i, P_{i+1}, dQ_i out of TMEM and into the workspace
// so P_{i+1} is formed while dK_i and dQ_i run, dV_{i+1} follows dQ_i without
// waiting for the dQ read-out, and at D = 128 only dP^T_{i+1} (which reuses
// the dQ columns) waits for it.
//
// The workspace is fp32 [B, Hq, Nq, Dw] (packed: [Hq, total_q, Dw]), Dw = 64
// for head dimensions up to 64 and 128 otherwise; the caller's buffer is
// zeroed on the stream first.  Query rows past a sequence's end receive exact
// zeros (their probabilities are 0) and keys past its end are masked.
//
// Every mbarrier wait is bounded (tc_common.cuh); the elementwise warpgroups
// hand their staging boxes to the TMA thread through mbarriers as well, so a
// timeout anywhere ends every role.  Before exit the issuing threads wait for
// their reductions to complete.

#include "bwd_common.cuh"

namespace fa {
namespace {

using namespace tc;

template <int D>
struct FusedCfg {
  static constexpr int BT = 128;                 // rows per tile (keys and queries)
  static constexpr int DC = D / 64;              // 128-byte column chunks per row
  static constexpr int CHUNK = BT * 128;         // bytes of one 128-row chunk
  static constexpr int TILE = DC * CHUNK;        // bytes of one 128 x D tile
  static constexpr int THREADS = 320;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr int NQ = 3;                   // Q ring slots
  static constexpr int ND = 2;                   // dO (+ L, Delta) ring slots
  static constexpr int DSLOT = TILE + 1024;      // dO | L*log2e | Delta
  static constexpr int OFF_V = TILE;
  static constexpr int OFF_Q = 2 * TILE;
  static constexpr int OFF_DO = OFF_Q + NQ * TILE;
  // D = 128: dS lives in the dO slot and dQ is staged in the dO and Q slots.
  // D = 64: a dS tile and a staging area of their own (two chunks each).
  static constexpr bool IN_SLOTS = D == 128;
  static constexpr int OFF_DS = OFF_DO + ND * DSLOT;
  static constexpr int OFF_ST = OFF_DS + (IN_SLOTS ? 0 : 2 * CHUNK);
  static constexpr int OFF_BAR = OFF_ST + (IN_SLOTS ? 0 : 2 * CHUNK);
  static constexpr int BAR_BYTES = 256;
  static constexpr int MAX_PAD = D == 128 ? 768 : 1024;
  static constexpr int SMEM = OFF_BAR + BAR_BYTES + MAX_PAD;
  static constexpr uint32_t COL_ST = 0, COL_DPT = 128, COL_DV = 256, COL_DK = 256 + D;
  static constexpr uint32_t COL_DQ = D == 128 ? COL_DPT : 384;
  static constexpr int DW = D;                   // workspace row width (floats)
  static constexpr int ROUNDS = D / 64;          // 32-column boxes per warpgroup and tile
  // arrivals that release a Q or dO slot: the MMA commit, plus at D = 128 the
  // two threads whose reductions read dQ out of it
  static constexpr uint32_t RELEASE = IN_SLOTS ? 3 : 1;
};

struct FusedArgs {
  const float* lse;
  const float* delta;
  void* dv;
  void* dk;
  Geo g;
  int64_t BH;              // B * Hkv
  int dreal;               // head dimension stored (<= D)
  int64_t sdv[4], sdk[4];
  int causal;
  float c;                 // scale * log2(e)
  float scale;
  Dropout drop;
  int split;               // CTAs (one cluster) sharing a key tile's query heads
  unsigned int* status;
  uint64_t timeout_ns;
  int withhold_arrival;    // test-only: CTA 0 withholds one arrival of its first P^T
};

// ---------------------------------------------------------------- local PTX
// 3-D tiled bulk reduction (add) of a shared-memory box into global memory.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, uint32_t src, int32_t c0,
                                                  int32_t c1, int32_t c2) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
      " [%0, {%1, %2, %3}], [%4];" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(c0), "r"(c1), "r"(c2), "r"(src)
      : "memory");
}

// Writes one 128-byte row (8 16-byte units) of a 128-byte-swizzled tile:
// unit u of row r goes to unit u ^ (r mod 8).
__device__ __forceinline__ void st_row_sw128(uint32_t tile, int row, const uint32_t* w) {
  const uint32_t base = tile + static_cast<uint32_t>(row) * 128u;
#pragma unroll
  for (int u = 0; u < 8; ++u)
    st_shared_v4(base + ((static_cast<uint32_t>(u ^ (row & 7))) << 4), w[4 * u], w[4 * u + 1],
                 w[4 * u + 2], w[4 * u + 3]);
}

// What the elementwise threads need to form P for one step.
struct ProbStep {
  const float* L2s;       // L * log2(e) of this half's 64 queries
  bool diag;              // causal diagonal tile
  uint32_t bhq;           // flat query head (dropout numbering)
  int64_t qbase;          // first query (within the sequence) of this half
};

// P^T for this thread's key and its half's 64 queries: exp2(c*S - L*log2 e),
// masked (keys past the sequence, causal diagonal), dropout keep bits into
// `keep` (query qbase + q is bit kbit(q)), and the rounded (dropped)
// P^T stored back over the scores for dV.
template <typename T, bool DROP>
__device__ __forceinline__ void form_probs(float (&p)[64], uint64_t& keep, uint32_t taddr,
                                           const ProbStep& s, float c, bool key_in, int hf, int row,
                                           int lane, int64_t key, const Dropout& drop) {
  tmem_ld64(taddr, p);
#pragma unroll
  for (int q = 0; q < 64; q += 4) {
    const float4 l4 = *reinterpret_cast<const float4*>(s.L2s + q);
    p[q] = ex2(fmaf(p[q], c, -l4.x));
    p[q + 1] = ex2(fmaf(p[q + 1], c, -l4.y));
    p[q + 2] = ex2(fmaf(p[q + 2], c, -l4.z));
    p[q + 3] = ex2(fmaf(p[q + 3], c, -l4.w));
  }
  if (!key_in) {
    // a key past the sequence (packed rows of the next one): no weight
#pragma unroll
    for (int q = 0; q < 64; ++q) p[q] = 0.f;
  }
  if (s.diag) {
    // query (64*hf + q) attends to this key only if it is not earlier
#pragma unroll
    for (int q = 0; q < 64; ++q)
      if (64 * hf + q < row) p[q] = 0.f;
  }
  keep = 0;
  if constexpr (DROP) keep = octet_keep_bits(drop, static_cast<uint32_t>(key >> 3), s.qbase, s.bhq, lane);
  uint32_t w[32];
  const uint32_t kl = static_cast<uint32_t>(keep), kh = static_cast<uint32_t>(keep >> 32);
#pragma unroll
  for (int q = 0; q < 32; ++q) {
    if constexpr (DROP) {
      // P o keep; Z's 1 / (1 - p) scales dV when it is stored
      w[q] = pack2<T>(kept64(kl, kh, kbit(2 * q)) ? p[2 * q] : 0.f,
                      kept64(kl, kh, kbit(2 * q + 1)) ? p[2 * q + 1] : 0.f);
    } else {
      w[q] = pack2<T>(p[2 * q], p[2 * q + 1]);
    }
  }
  tmem_st32(taddr, w);
  tmem_wait_st();
}

template <typename T, int D, bool DROP>
__global__ void __launch_bounds__(320, 1)
    bwd_fused_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo,
                        const __grid_constant__ CUtensorMap tmdq, const FusedArgs a) {
  using C = FusedCfg<D>;
  static_assert(C::SMEM <= 232448, "shared memory per block");
  static_assert(2 * 128 * D * 4 <= C::OFF_DO, "cluster staging fits below the dO slots");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  if (pad > static_cast<uint32_t>(C::MAX_PAD)) {   // never expected: report, do nothing
    if (threadIdx.x == 0) atomicCAS(a.status, 0u, static_cast<unsigned int>(FA_ERR_LAUNCH));
    return;
  }
  uint8_t* smem = smem_raw + pad;
  uint8_t* sK = smem;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sQ = smem + C::OFF_Q;            // slot s: Q tile
  uint8_t* sD = smem + C::OFF_DO;           // slot s: dO tile (then dS at D = 128) | L2 | Delta
  uint8_t* sDS = smem + C::OFF_DS;          // D = 64: dS tile
  uint8_t* sST = smem + C::OFF_ST;          // D = 64: dQ staging boxes
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  Ctl* ctl = reinterpret_cast<Ctl*>(bars + 28);
  const uint32_t b_kv = smem_u32(&bars[0]);
  const uint32_t b_qfull0 = smem_u32(&bars[1]);                  // + 8 * Q slot (3)
  const uint32_t b_qempty0 = smem_u32(&bars[4]);                 // + 8 * Q slot
  const uint32_t b_dfull0 = smem_u32(&bars[7]);                  // + 8 * dO slot (2)
  const uint32_t b_dempty0 = smem_u32(&bars[9]);                 // + 8 * dO slot
  const uint32_t b_sfull = smem_u32(&bars[11]);
  const uint32_t b_dpfull = smem_u32(&bars[12]);
  const uint32_t b_pready0 = smem_u32(&bars[13]);                // + 8 * half
  const uint32_t b_dsready0 = smem_u32(&bars[15]);               // + 8 * half
  const uint32_t b_accdone = smem_u32(&bars[17]);
  const uint32_t b_mmadone = smem_u32(&bars[18]);
  const uint32_t b_dqfull = smem_u32(&bars[19]);                 // dQ_i is in TMEM
  const uint32_t b_dqread = smem_u32(&bars[20]);                 // dQ_i read out (D = 128)
  const uint32_t b_dvdone = smem_u32(&bars[21]);                 // dV_i has completed
  // + 8 * (2 * half + round): box written.  One barrier per round, so a warp
  // that is already writing the next round's box cannot complete this one.
  const uint32_t b_staged0 = smem_u32(&bars[22]);
  const uint32_t b_stfree0 = smem_u32(&bars[26]);                // + 8 * half (D = 64): box read

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = a.split;
  const int rank = static_cast<int>(blockIdx.x % split);
  const int64_t id = blockIdx.x / split;
  const int64_t bhk = id % a.BH;                // b * Hkv + key/value head
  const int64_t kt = id / a.BH;                 // key tile; low tiles (most work) first
  const int64_t bseq = bhk / a.g.Hkv;
  const int32_t hk = static_cast<int32_t>(bhk % a.g.Hkv);
  const SeqView sv = seq_view(a.g, bseq);
  if (!sv.ok) {
    if (threadIdx.x == 0) record_status(a.status, FA_ERR_SEQLENS);
    return;
  }
  const int64_t Nq = sv.nq, Nk = sv.nk;
  if (kt * C::BT >= Nk) return;                 // this key tile lies past the sequence
  const int32_t bb = static_cast<int32_t>(sv.b);
  const int nq = static_cast<int>((Nq + C::BT - 1) / C::BT);
  const int i0 = a.causal ? static_cast<int>(kt) : 0;   // first query tile
  const int per = nq > i0 ? nq - i0 : 0;                 // query tiles per query head
  const int gper = static_cast<int>(a.g.G) / split;      // query heads of this CTA
  const int g0 = rank * gper;                            // its first head within the group
  const int n = per * gper;                              // (query head, query tile) steps
  if (n == 0) {
    // No query attends to these keys: dK = dV = 0 and no dQ contribution.
    if (warp < 8 && rank == 0) {
      const int64_t key = kt * C::BT + (warp & 3) * 32 + lane;
      if (key < Nk) {
        const int64_t* st = (warp >> 2) ? a.sdk : a.sdv;
        T* out = static_cast<T*>((warp >> 2) ? a.dk : a.dv) + bb * st[0] + hk * st[1] +
                 (sv.k0 + key) * st[2];
        for (int d = 0; d < a.dreal; ++d) out[d] = Elem<T>::from_f32(0.f);
      }
    }
    return;
  }

  if (threadIdx.x == 0) {
    mbar_init(b_kv, 1);
    for (int s = 0; s < C::NQ; ++s) {
      mbar_init(b_qfull0 + 8 * s, 1);
      mbar_init(b_qempty0 + 8 * s, C::RELEASE);
    }
    for (int s = 0; s < C::ND; ++s) {
      mbar_init(b_dfull0 + 8 * s, 32);
      mbar_init(b_dempty0 + 8 * s, C::RELEASE);
    }
    mbar_init(b_sfull, 1);
    mbar_init(b_dpfull, 1);
    for (int h = 0; h < 2; ++h) {
      mbar_init(b_pready0 + 8 * h, 128);
      mbar_init(b_dsready0 + 8 * h, 128);
      mbar_init(b_staged0 + 8 * (2 * h), 128);
      mbar_init(b_staged0 + 8 * (2 * h + 1), 128);
      mbar_init(b_stfree0 + 8 * h, 1);
    }
    mbar_init(b_accdone, 1);
    mbar_init(b_mmadone, 1);
    mbar_init(b_dqfull, 1);
    mbar_init(b_dqread, 256);
    mbar_init(b_dvdone, 1);
    ctl->abort = 0;
    mbar_fence_init();
  }
  if (warp == 8) {
    tmem_alloc(smem_u32(&ctl->tmem_base), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  bool ew_ok = false;   // elementwise warps: main loop completed

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    // Lane 0 issues the TMA copies: K and V once, then per step Q into its Q
    // slot and dO into its dO slot, where all 32 lanes also stage L * log2(e)
    // and Delta (4 rows per lane, read from global memory before the slot is
    // free; rows past the sequence get L = +inf, so their probabilities are
    // exactly 0, and Delta = 0).
    if (lane == 0) {
      tma_prefetch_desc(&tmq); tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv); tma_prefetch_desc(&tmdo);
      mbar_arrive_expect_tx(b_kv, 2 * C::TILE);
      for (int c = 0; c < C::DC; ++c) {
        tma_load_4d(smem_u32(sK + c * C::CHUNK), &tmk, b_kv, c * 64,
                    static_cast<int32_t>(sv.k0 + kt * C::BT), hk, bb);
        tma_load_4d(smem_u32(sV + c * C::CHUNK), &tmv, b_kv, c * 64,
                    static_cast<int32_t>(sv.k0 + kt * C::BT), hk, bb);
      }
    }
    uint32_t q_round[C::NQ], d_round[C::ND];
#pragma unroll
    for (int s = 0; s < C::NQ; ++s) q_round[s] = 0;
#pragma unroll
    for (int s = 0; s < C::ND; ++s) d_round[s] = 0;
    bool ok = true;
    for (int it = 0; it < n; ++it) {
      const int64_t q0 = static_cast<int64_t>(i0 + it % per) * C::BT;     // within the sequence
      const int32_t hq = static_cast<int32_t>(hk * a.g.G + g0 + it / per);
      const int qs = it % C::NQ;
      const uint32_t qr = static_cast<uint32_t>(it / C::NQ);
      if (lane == 0) {
        if (qr > 0 && !wait_bounded(b_qempty0 + 8 * qs, (qr - 1) & 1, ctl, a.status, a.timeout_ns))
          ok = false;
        if (ok) {
          mbar_arrive_expect_tx(b_qfull0 + 8 * qs, C::TILE);
          for (int c = 0; c < C::DC; ++c)
            tma_load_4d(smem_u32(sQ + qs * C::TILE + c * C::CHUNK), &tmq, b_qfull0 + 8 * qs, c * 64,
                        static_cast<int32_t>(sv.q0 + q0), hq, bb);
          q_round[qs] = qr + 1;
        }
      }
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      float lv[4], dv[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int64_t q = q0 + lane * 4 + t;
        const int64_t li = lse_index(a.g, sv, hq, q);
        lv[t] = q < Nq ? a.lse[li] * kLog2e : INFINITY;
        dv[t] = q < Nq ? a.delta[li] : 0.f;
      }
      const int ds = it % C::ND;
      const uint32_t dr = static_cast<uint32_t>(it / C::ND);
      if (dr > 0 && !(ok = wait_warp(b_dempty0 + 8 * ds, (dr - 1) & 1, ctl, a.status, a.timeout_ns)))
        break;
      uint8_t* slot = sD + ds * C::DSLOT;
      float* L2s = reinterpret_cast<float*>(slot + C::TILE);
      float* Ds = L2s + 128;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        L2s[lane * 4 + t] = lv[t];
        Ds[lane * 4 + t] = dv[t];
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(b_dfull0 + 8 * ds, C::TILE);
        for (int c = 0; c < C::DC; ++c)
          tma_load_4d(smem_u32(slot + c * C::CHUNK), &tmdo, b_dfull0 + 8 * ds, c * 64,
                      static_cast<int32_t>(sv.q0 + q0), hq, bb);
      } else {
        mbar_arrive(b_dfull0 + 8 * ds);
      }
      d_round[ds] = dr + 1;
    }
    // Drain: every copy issued has landed.
    if (lane == 0) {
      wait_bounded(b_kv, 0, ctl, a.status, a.timeout_ns, false);
      for (int s = 0; s < C::NQ; ++s)
        if (q_round[s]) wait_bounded(b_qfull0 + 8 * s, (q_round[s] - 1) & 1, ctl, a.status,
                                     a.timeout_ns, false);
      for (int s = 0; s < C::ND; ++s)
        if (d_round[s]) wait_bounded(b_dfull0 + 8 * s, (d_round[s] - 1) & 1, ctl, a.status,
                                     a.timeout_ns, false);
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idS = idesc_f16<T>(128, C::BT, false, false);
      const uint32_t idG = idesc_f16<T>(128, D, false, true);
      const uint32_t idQ = idesc_f16<T>(128, D, true, true);
      const uint64_t dK0 = sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dV0 = sdesc_sw128(smem_u32(sV), 16, 1024);
      const uint64_t dQk = sdesc_sw128(smem_u32(sQ), 16, 1024);          // K-major views
      const uint64_t dDk = sdesc_sw128(smem_u32(sD), 16, 1024);
      const uint64_t dQm = sdesc_sw128(smem_u32(sQ), C::CHUNK, 1024);    // MN-major views
      const uint64_t dDm = sdesc_sw128(smem_u32(sD), C::CHUNK, 1024);
      const uint64_t dKm = sdesc_sw128(smem_u32(sK), C::CHUNK, 1024);
      const uint64_t dSm = sdesc_sw128(smem_u32(C::IN_SLOTS ? sD : sDS), C::CHUNK, 1024);
      auto issue_ST = [&](int qs) {   // S^T = K Q^T
        const uint64_t q = dQk + static_cast<uint64_t>((qs * C::TILE) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::CHUNK + (kk & 3) * 32) >> 4;
          mma_ss(tmem + C::COL_ST, dK0 + off, q + off, idS, kk > 0 ? 1u : 0u);
        }
        mma_commit(b_sfull);
      };
      auto issue_DPT = [&](int ds) {  // dP^T = V dO^T
        const uint64_t g = dDk + static_cast<uint64_t>((ds * C::DSLOT) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::CHUNK + (kk & 3) * 32) >> 4;
          mma_ss(tmem + C::COL_DPT, dV0 + off, g + off, idS, kk > 0 ? 1u : 0u);
        }
        mma_commit(b_dpfull);
      };
      // dV += P^T_j dO_j (per half as P^T is ready; B: dO read MN-major, N = d)
      auto issue_DV = [&](int j) -> bool {
        const uint64_t mdo = dDm + static_cast<uint64_t>(((j % C::ND) * C::DSLOT) >> 4);
        for (int h = 0; h < 2; ++h) {
          if (!wait_bounded(b_pready0 + 8 * h, j & 1, ctl, a.status, a.timeout_ns)) return false;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts(tmem + C::COL_DV, tmem + C::COL_ST + 64 * h + 8 * kk,
                   mdo + static_cast<uint64_t>(((64 * h + 16 * kk) * 128) >> 4), idG,
                   (j > 0 || h > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(b_dvdone);
        return true;
      };
      bool ok = wait_bounded(b_kv, 0, ctl, a.status, a.timeout_ns) &&
                wait_bounded(b_qfull0, 0, ctl, a.status, a.timeout_ns) &&
                wait_bounded(b_dfull0, 0, ctl, a.status, a.timeout_ns);
      if (ok) {
        tc_fence_after();
        issue_ST(0);
        issue_DPT(0);
        ok = issue_DV(0);
      }
      if (ok && n > 1) {
        if ((ok = wait_bounded(b_qfull0 + 8, 0, ctl, a.status, a.timeout_ns))) {
          tc_fence_after();
          issue_ST(1);
        }
      }
      for (int it = 0; ok && it < n; ++it) {
        const int qs = it % C::NQ, ds = it % C::ND;
        // dK += dS^T Q (B: this tile's Q read MN-major)
        const uint64_t mq = dQm + static_cast<uint64_t>((qs * C::TILE) >> 4);
        for (int h = 0; ok && h < 2; ++h) {
          if (!(ok = wait_bounded(b_dsready0 + 8 * h, it & 1, ctl, a.status, a.timeout_ns))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts(tmem + C::COL_DK, tmem + C::COL_DPT + 64 * h + 8 * kk,
                   mq + static_cast<uint64_t>(((64 * h + 16 * kk) * 128) >> 4), idG,
                   (it > 0 || h > 0 || kk > 0) ? 1u : 0u);
        }
        if (!ok) break;
        mma_commit(b_qempty0 + 8 * qs);   // Q_i has no reader after dK_i
        // dQ_i = dS_i K: A = dS from shared memory (M = query, MN-major),
        // B = K (N = d, MN-major); 16 keys per product.
        const uint64_t dsm =
            dSm + (C::IN_SLOTS ? static_cast<uint64_t>((ds * C::DSLOT) >> 4) : 0ull);
#pragma unroll
        for (int kk = 0; kk < C::BT / 16; ++kk) {
          const uint64_t off = static_cast<uint64_t>((kk * 16 * 128) >> 4);
          mma_ss(tmem + C::COL_DQ, dsm + off, dKm + off, idQ, kk > 0 ? 1u : 0u);
        }
        mma_commit(b_dqfull);
        mma_commit(b_dempty0 + 8 * ds);   // dO_i / dS_i have no reader after dQ_i
        if (it + 1 < n) {
          const int ds1 = (it + 1) % C::ND;
          if (!(ok = wait_bounded(b_dfull0 + 8 * ds1, ((it + 1) / C::ND) & 1, ctl, a.status,
                                  a.timeout_ns)))
            break;
          tc_fence_after();
          if (!(ok = issue_DV(it + 1))) break;
          if constexpr (C::COL_DQ == C::COL_DPT) {
            // dQ_i occupies the dP^T columns until the elementwise warps read it
            if (!(ok = wait_bounded(b_dqread, it & 1, ctl, a.status, a.timeout_ns))) break;
            tc_fence_after();
          }
          issue_DPT(ds1);
          if (it + 2 < n) {
            const int qs2 = (it + 2) % C::NQ;
            if (!(ok = wait_bounded(b_qfull0 + 8 * qs2, ((it + 2) / C::NQ) & 1, ctl, a.status,
                                    a.timeout_ns)))
              break;
            tc_fence_after();
            issue_ST(qs2);                // P^T_{i+1} was read by dV_{i+1}, issued before
          }
        }
      }
      if (ok) mma_commit(b_accdone);
      mma_commit(b_mmadone);
      wait_bounded(b_mmadone, 0, ctl, a.status, a.timeout_ns, false);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ elementwise + epilogue
    const int hf = warp >> 2, quarter = warp & 3;
    const int row = quarter * 32 + lane;        // TMEM lane: key of S^T/dP^T, query of dQ
    const int64_t key = kt * C::BT + row;
    const bool key_in = key < Nk;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const bool elected = quarter == 0 && lane == 0;   // issues this warpgroup's reductions
    const uint32_t b_staged = b_staged0 + 16 * hf, b_stfree = b_stfree0 + 8 * hf;
    const float c = a.c;
    auto prob_step = [&](int it) {
      ProbStep s;
      const int ds = it % C::ND;
      s.L2s = reinterpret_cast<const float*>(sD + ds * C::DSLOT + C::TILE) + 64 * hf;
      const int i = i0 + it % per;
      s.diag = a.causal && i == kt;
      s.bhq = static_cast<uint32_t>(bseq * a.g.Hq + hk * a.g.G + g0 + it / per);
      s.qbase = static_cast<int64_t>(i) * C::BT + 64 * hf;
      return s;
    };
    float p[64];
    uint64_t keep = 0;
    bool ok = wait_warp(b_sfull, 0, ctl, a.status, a.timeout_ns) &&
              wait_warp(b_dfull0, 0, ctl, a.status, a.timeout_ns);
    if (ok) {
      // the dO slot's arrival also publishes the staged L and Delta
      tc_fence_after();
      form_probs<T, DROP>(p, keep, lane_base + C::COL_ST + 64 * hf, prob_step(0), c, key_in, hf,
                          row, lane, key, a.drop);
      tc_fence_before();
      // A test can withhold this arrival in CTA 0 to make the MMA warp's
      // bounded wait run out (the timeout path, without a fault).
      if (!(a.withhold_arrival && blockIdx.x == 0 && threadIdx.x == 0))
        mbar_arrive(b_pready0 + 8 * hf);
    }
    for (int it = 0; ok && it < n; ++it) {
      const int i = i0 + it % per, ds = it % C::ND, qs = it % C::NQ;
      const int32_t hq = static_cast<int32_t>(hk * a.g.G + g0 + it / per);
      // ---- dS_i (at D = 128 written over dO_i below, so dV_i must be done)
      if (!(ok = wait_warp(b_dpfull, it & 1, ctl, a.status, a.timeout_ns))) break;
      if constexpr (C::IN_SLOTS) {
        if (!(ok = wait_warp(b_dvdone, it & 1, ctl, a.status, a.timeout_ns))) break;
      }
      tc_fence_after();
      {
        const float* Ds = reinterpret_cast<const float*>(sD + ds * C::DSLOT + C::TILE) + 128 +
                          64 * hf;
        float dp[64];
        tmem_ld64(lane_base + C::COL_DPT + 64 * hf, dp);
        if constexpr (DROP) {
          // dS = P o (Z o dP - Delta), Z = keep / (1 - p)
#pragma unroll
          for (int q = 0; q < 64; ++q) {
            const float z = kept64(static_cast<uint32_t>(keep), static_cast<uint32_t>(keep >> 32),
                                   kbit(q)) ? a.drop.rscale : 0.f;
            dp[q] = p[q] * fmaf(z, dp[q], -Ds[q]);
          }
        } else {
#pragma unroll
          for (int q = 0; q < 64; q += 4) {
            const float4 d4 = *reinterpret_cast<const float4*>(Ds + q);
            dp[q] = p[q] * (dp[q] - d4.x);
            dp[q + 1] = p[q + 1] * (dp[q + 1] - d4.y);
            dp[q + 2] = p[q + 2] * (dp[q + 2] - d4.z);
            dp[q + 3] = p[q + 3] * (dp[q + 3] - d4.w);
          }
        }
        uint32_t w[32];
#pragma unroll
        for (int q = 0; q < 32; ++q) w[q] = pack2<T>(dp[2 * q], dp[2 * q + 1]);
        tmem_st32(lane_base + C::COL_DPT + 64 * hf, w);   // dS^T, A operand of dK
        // the same row into shared memory, A operand of dQ (key row `row`,
        // this warpgroup's 64 queries)
        st_row_sw128(smem_u32((C::IN_SLOTS ? sD + ds * C::DSLOT : sDS) + hf * C::CHUNK), row, w);
        fence_async_smem();
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(b_dsready0 + 8 * hf);
      }
      // ---- P_{i+1}, while the tensor cores run dK_i and dQ_i
      if (it + 1 < n) {
        if (!(ok = wait_warp(b_sfull, (it + 1) & 1, ctl, a.status, a.timeout_ns))) break;
        if (!(ok = wait_warp(b_dfull0 + 8 * ((it + 1) % C::ND), ((it + 1) / C::ND) & 1, ctl,
                             a.status, a.timeout_ns)))
          break;
        tc_fence_after();
        form_probs<T, DROP>(p, keep, lane_base + C::COL_ST + 64 * hf, prob_step(it + 1), c, key_in,
                            hf, row, lane, key, a.drop);
        tc_fence_before();
        mbar_arrive(b_pready0 + 8 * hf);
      }
      // ---- dQ_i: this thread holds query row `row` of the tile; warpgroup
      // hf reduces columns (D/2)*hf .. (D/2)*hf + D/2 - 1, 32 per box
      if (!(ok = wait_warp(b_dqfull, it & 1, ctl, a.status, a.timeout_ns))) break;
      tc_fence_after();
      uint32_t x[C::ROUNDS][32];
#pragma unroll
      for (int r = 0; r < C::ROUNDS; ++r)
        tmem_ld32(lane_base + C::COL_DQ + (D / 2) * hf + 32 * r, x[r]);
      tmem_wait_ld();
#pragma unroll
      for (int r = 0; r < C::ROUNDS; ++r) reg_fence32(x[r]);
      if constexpr (C::COL_DQ == C::COL_DPT) {
        tc_fence_before();
        mbar_arrive(b_dqread);            // the dP^T columns may be overwritten
      }
      if constexpr (!C::IN_SLOTS) {
        // the staging box of the previous step has been read
        if (it > 0 && !(ok = wait_warp(b_stfree, (it - 1) & 1, ctl, a.status, a.timeout_ns))) break;
      }
      const int32_t qrow0 = static_cast<int32_t>(sv.q0 + static_cast<int64_t>(i) * C::BT);
      const int32_t plane = static_cast<int32_t>(sv.b * a.g.Hq + hq);
#pragma unroll
      for (int r = 0; r < C::ROUNDS; ++r) {
        // box r: D = 128: the dO_i / dS_i slot (r = 0) and the Q_i slot
        // (r = 1), whose readers dQ_i and dK_i have completed; D = 64: the
        // warpgroup's own staging box
        uint8_t* box = C::IN_SLOTS ? (r == 0 ? sD + ds * C::DSLOT : sQ + qs * C::TILE) : sST;
        const uint32_t bx = smem_u32(box + hf * C::CHUNK);
        st_row_sw128(bx, row, x[r]);
        fence_async_smem();
        mbar_arrive(b_staged + 8 * r);
        if (elected) {
          if (wait_bounded(b_staged + 8 * r, it & 1, ctl, a.status, a.timeout_ns)) {
            const int col = (D / 2) * hf + 32 * r;
            if (col < a.dreal) tma_reduce_add_3d(&tmdq, bx, col, qrow0, plane);
            bulk_commit();
          }
        }
        __syncwarp();
      }
      if (elected) {
        // release what the reductions read (the other warps of this
        // warpgroup go on to the next step meanwhile)
        bulk_wait_read_all();
        if constexpr (C::IN_SLOTS) {
          mbar_arrive(b_dempty0 + 8 * ds);
          mbar_arrive(b_qempty0 + 8 * qs);
        } else {
          mbar_arrive(b_stfree);
        }
      }
      __syncwarp();
    }
    // Every reduction of both warpgroups has completed before any thread
    // goes on: the cluster epilogue below stages partial sums over the Q
    // slots, which the last reductions read.  All 256 elementwise threads
    // reach this barrier (nothing above returns early or waits unbounded).
    if (elected) bulk_wait_all();
    asm volatile("bar.sync 1, 256;" ::: "memory");
    if (ok) ok = wait_warp(b_accdone, 0, ctl, a.status, a.timeout_ns);
    ew_ok = ok;
    if (ok) {
      tc_fence_after();
      const bool store = key_in;
      const uint32_t acc = lane_base + (hf == 0 ? C::COL_DV : C::COL_DK);
      if (split == 1) {
        if (hf == 0) {
          T* out = static_cast<T*>(a.dv) + bb * a.sdv[0] + hk * a.sdv[1] + (sv.k0 + key) * a.sdv[2];
          store_row_cols<T>(acc, DROP ? a.drop.rscale : 1.f, out, store, a.dreal);
        } else {
          T* out = static_cast<T*>(a.dk) + bb * a.sdk[0] + hk * a.sdk[1] + (sv.k0 + key) * a.sdk[2];
          store_row_cols<T>(acc, a.scale, out, store, a.dreal);
        }
      } else if (rank != 0) {
        // partial sums into this CTA's shared memory for rank 0 to read
        stage_partial<D>(smem, hf, row, acc);
      }
    }
  }

  if (split > 1) {
    // Every thread of every CTA of the cluster passes both barriers, also
    // after a timeout (outputs are then undefined but nothing waits forever).
    cluster_sync_all();
    if (warp < 8 && rank == 0 && ew_ok) {
      const int hf = warp >> 2, quarter = warp & 3, row = quarter * 32 + lane;
      const int64_t key = kt * C::BT + row;
      const uint32_t acc = tmem + (static_cast<uint32_t>(quarter * 32) << 16) +
                           (hf == 0 ? C::COL_DV : C::COL_DK);
      T* out = hf == 0
                   ? static_cast<T*>(a.dv) + bb * a.sdv[0] + hk * a.sdv[1] + (sv.k0 + key) * a.sdv[2]
                   : static_cast<T*>(a.dk) + bb * a.sdk[0] + hk * a.sdk[1] + (sv.k0 + key) * a.sdk[2];
      cluster_reduce_store<T, D>(smem, hf, row, acc, split, hf == 0 ? (DROP ? a.drop.rscale : 1.f) : a.scale, out,
                                 key < Nk, a.dreal);
    }
    cluster_sync_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// dQ = scale * workspace, rounded to T, for every query row a sequence owns
// (packed: rows cu_q[0] .. cu_q[B] - 1).  HBM-bound: 8 elements per thread
// (two 16-byte reads, one 16-byte write), grid-stride over the rows.
template <typename T>
__global__ void __launch_bounds__(256)
    dq_convert_kernel(const float* __restrict__ ws, T* dq, Geo g, int dw, int dreal, int64_t s0,
                      int64_t s1, int64_t s2, float scale) {
  const int nv = dreal / 8;
  const int64_t total = g.Bt * g.Hq * g.rows_q * nv;
  int64_t rlo = 0, rhi = g.rows_q;
  if (g.cu_q != nullptr) {
    rlo = max(static_cast<int64_t>(0), static_cast<int64_t>(__ldg(g.cu_q)));
    rhi = min(g.rows_q, static_cast<int64_t>(__ldg(g.cu_q + g.B)));
  }
  for (int64_t v = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; v < total;
       v += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t d8 = v % nv;
    const int64_t rowg = v / nv;                 // (b * Hq + h) * rows_q + row
    const int64_t r = rowg % g.rows_q;
    if (r < rlo || r >= rhi) continue;
    const int64_t bh = rowg / g.rows_q;
    const float* src = ws + rowg * dw + d8 * 8;
    const float4 x = __ldg(reinterpret_cast<const float4*>(src));
    const float4 y = __ldg(reinterpret_cast<const float4*>(src + 4));
    uint4 w;
    w.x = pack2<T>(x.x * scale, x.y * scale);
    w.y = pack2<T>(x.z * scale, x.w * scale);
    w.z = pack2<T>(y.x * scale, y.y * scale);
    w.w = pack2<T>(y.z * scale, y.w * scale);
    *reinterpret_cast<uint4*>(dq + (bh / g.Hq) * s0 + (bh % g.Hq) * s1 + r * s2 + d8 * 8) = w;
  }
}

template <typename T, int D, bool DROP>
fa_status run_bwd_fused(const BwdParams& p, float* ws, cudaStream_t stream) {
  using C = FusedCfg<D>;
  const Geo& g = p.g;
  CUtensorMap mq, mk, mv, mdo, mdq;
  if (!encode_tile_map(&mq, p.q, p.dtype, g.Bt, g.Hq, g.rows_q, p.D, p.sq, 128, 64) ||
      !encode_tile_map(&mk, p.k, p.dtype, g.Bt, g.Hkv, g.rows_k, p.D, p.sk, 128, 64) ||
      !encode_tile_map(&mv, p.v, p.dtype, g.Bt, g.Hkv, g.rows_k, p.D, p.sv, 128, 64) ||
      !encode_tile_map(&mdo, p.dout, p.dtype, g.Bt, g.Hq, g.rows_q, p.D, p.sdo, 128, 64) ||
      !encode_f32_rows_map(&mdq, ws, C::DW, g.rows_q, g.Bt * g.Hq, 32, 128))
    return FA_ERR_LAUNCH;
  const size_t ws_bytes = static_cast<size_t>(g.Bt * g.Hq * g.rows_q) * C::DW * sizeof(float);
  if (cudaMemsetAsync(ws, 0, ws_bytes, stream) != cudaSuccess) return FA_ERR_LAUNCH;

  FusedArgs a{};
  a.lse = p.lse; a.delta = p.delta;
  a.dv = p.dv; a.dk = p.dk;
  a.g = g;
  a.BH = g.B * g.Hkv;
  a.dreal = static_cast<int>(p.D);
  for (int i = 0; i < 4; ++i) { a.sdv[i] = p.sdv[i]; a.sdk[i] = p.sdk[i]; }
  a.causal = p.causal;
  a.c = p.scale * kLog2e;
  a.scale = p.scale;
  a.drop = p.drop;
  a.status = p.status;
  a.timeout_ns = p.timeout_ns;
  a.withhold_arrival = p.withhold_arrival;
  // one CTA per (b, key/value head, key tile); a cluster of `split` CTAs
  // shares a key tile's query heads while the grid is short of two waves
  const int64_t base = a.BH * ((g.Nk + 127) / 128);
  int split = 1;
  while (split < 8 && g.G % (2 * split) == 0 && base * split < 2 * device_sm_count()) split *= 2;
  a.split = split;
  const int64_t blocks = base * split;
  if (blocks > 0x7fffffffLL) return FA_ERR_SHAPE;
  auto k1 = bwd_fused_tc_kernel<T, D, DROP>;
  if (cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
    return FA_ERR_LAUNCH;
  prof_record(p, 0, stream);
  if (split == 1) {
    k1<<<dim3(static_cast<unsigned>(blocks)), dim3(C::THREADS), C::SMEM, stream>>>(mq, mk, mv, mdo,
                                                                                  mdq, a);
  } else {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(split);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, k1, mq, mk, mv, mdo, mdq, a) != cudaSuccess) return FA_ERR_LAUNCH;
  }
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_LAUNCH;
  prof_record(p, 1, stream);

  const int64_t vecs = g.Bt * g.Hq * g.rows_q * (p.D / 8);
  const int64_t want = (vecs + 255) / 256;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
  const unsigned blocks2 = static_cast<unsigned>(want < cap ? (want > 0 ? want : 1) : cap);
  dq_convert_kernel<T><<<blocks2, 256, 0, stream>>>(ws, static_cast<T*>(p.dq), g, C::DW,
                                                    static_cast<int>(p.D), p.sdq[0], p.sdq[1],
                                                    p.sdq[2], p.scale);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_LAUNCH;
  prof_record(p, 2, stream);
  return FA_OK;
}

template <typename T, int D>
fa_status run_bwd_fused_any(const BwdParams& p, float* ws, cudaStream_t s) {
  return p.drop.on ? run_bwd_fused<T, D, true>(p, ws, s) : run_bwd_fused<T, D, false>(p, ws, s);
}

}  // namespace

size_t bwd_fused_workspace_floats(const Geo& g, int64_t D) {
  return static_cast<size_t>(g.Bt * g.Hq * g.rows_q) * (D == 128 ? 128 : 64);
}

fa_status launch_bwd_fused(const BwdParams& p, float* ws, cudaStream_t s) {
  if (p.dtype == FA_BF16) {
    if (p.D == 128) return run_bwd_fused_any<__nv_bfloat16, 128>(p, ws, s);
    if (p.D <= 64) return run_bwd_fused_any<__nv_bfloat16, 64>(p, ws, s);
  } else if (p.dtype == FA_F16) {
    if (p.D == 128) return run_bwd_fused_any<__half, 128>(p, ws, s);
    if (p.D <= 64) return run_bwd_fused_any<__half, 64>(p, ws, s);
  }
  return FA_ERR_DTYPE;
}

}  // namespace fa
