// Tensor-core backward: TMA + tcgen05 + TMEM, warp-specialised, for fp16/bf16
// with D in {64, 128} (16 and 32 run through D = 64 with the head dimension
// zero-filled by the TMA loads), over the general geometry of fa_internal.h
// (sequence views, grouped key/value heads) and, as a template flag, dropout.
//
// The FlashAttention-2 split of "Triton FlashAttention" (project summary): a
// dK/dV kernel that, for each 128-key tile, loops over the query tiles that
// attend to it, and a dQ kernel that, for each 128-query tile, loops over the
// key tiles it attends to.  Neither uses atomics.  Both rebuild the
// probabilities from the saved log-sum-exp, P = exp(S - L)
// ("FlashAttention-2 from PyTorch to Triton", section on the running
// quantities), evaluated as exp2(c * S - L * log2(e)) with c = scale * log2(e),
// and use Delta = rowsum(dO o O) from the preprocess kernel (same page,
// defect 5).  With dS = P o (dP - Delta):
//   dK/dV kernel (key tile j):  S^T = K_j Q_i^T,  dP^T = V_j dO_i^T,
//                               dV_j += P^T dO_i,  dK_j += dS^T Q_i,
//                               dK_j *= scale at the end;
//   dQ kernel (query tile i):   S = Q_i K_j^T,  dP = dO_i V_j^T,
//                               dQ_i += dS K_j,  dQ_i *= scale at the end.
// P^T and dS are rounded to the input type before they enter a product.
//
// Warp roles (320 threads): warps 0-3 and 4-7 are two elementwise warpgroups
// that split the 128 columns of each score tile (64 each; one TMEM lane = one
// row per thread); warp 8 is the TMA producer and owns the TMEM allocation;
// warp 9 issues the MMAs (the whole warp runs the issue loop, one elected
// lane issues).  Each elementwise warpgroup writes
// its rounded P^T / dS into the TMEM columns it alone reads, so the two never
// race.  Both warpgroups release a product's operand on one barrier (256
// arrivals), so the MMA thread waits once per product: the two halves are
// computed side by side, and a wait per half cost the one-lane issuer more
// than the earlier start of the first half saved (dK/dV 2.61 -> 2.45 ms on the
// long causal shape).  The second barrier of each pair is unused.
//
// With grouped heads the dK/dV kernel of a key/value head loops over every
// query head that reads it; when that leaves too few CTAs for the GPU, a
// cluster of CTAs splits the query heads of one key tile and sums its partial
// dK, dV through distributed shared memory (see the kernel).
//
// Every mbarrier wait is bounded (tc_common.cuh); on a timeout the CTA drains
// its copies and MMAs in flight, frees its tensor memory and exits.

#include "bwd_common.cuh"

namespace fa {
namespace {

using namespace tc;

template <int D>
struct BwdShape {
  static constexpr int BT = 128;                 // rows per tile (keys and queries)
  static constexpr int DC = D / 64;              // 128-byte column chunks per row
  static constexpr int CHUNK = BT * 128;         // bytes of one 128-row chunk
  static constexpr int TILE = DC * CHUNK;        // bytes of one 128 x D tile
  static constexpr int THREADS = 320;
  static constexpr uint32_t TMEM_COLS = 512;
};

struct BwdTcArgs {
  const float* lse;
  const float* delta;
  void* out0;              // dK/dV kernel: dV;  dQ kernel: dQ
  void* out1;              // dK/dV kernel: dK
  Geo g;
  int64_t BH;              // dK/dV kernel: B * Hkv;  dQ kernel: B * Hq
  int64_t ntiles;          // dK/dV kernel: key tiles;  dQ kernel: query tiles (longest sequence)
  int64_t hgroup;          // heads per group of the block order (grouped_tile)
  int dreal;               // head dimension stored (<= D; narrower ones run zero-padded)
  int64_t s0[4], s1[4];    // strides of out0, out1
  int causal;
  float c;                 // scale * log2(e)
  float scale;
  Dropout drop;
  int split;               // dK/dV kernel: CTAs (one cluster) sharing a key tile's query heads
  unsigned int* status;
  uint64_t timeout_ns;
};

// ============================================================================
// dK / dV
// ============================================================================
// Shared memory: K_j and V_j (loaded once), a ring of NQ query tiles Q_i and a
// ring of ND slots holding dO_i with its L * log2(e) and Delta.  Q_i is read by
// S^T_i and dK_i, dO_i by dP^T_i and dV_i, so the MMA issue order per query
// tile i,
//     dV_i (once P^T_i is ready),  S^T_{i+1},
//     dK_i (once dS^T_i is ready), dP^T_{i+1},
// needs Q_{i+1} loaded while tile i is still in use (three Q slots) but dO_{i+1}
// only after dK_i (two dO slots).  S^T_{i+1} overwrites P^T_i and dP^T_{i+1}
// overwrites dS^T_i; each is read only by products issued before it.  The next
// tile's scores are therefore ready while the elementwise warps finish dS_i.
// The cluster reduction stages partial sums with stage_row / stage_chunk
// (bwd_common.cuh).

template <int D>
struct DkdvCfg : BwdShape<D> {
  using S = BwdShape<D>;
  static constexpr int NQ = 3;                               // Q ring slots
  static constexpr int ND = 2;                               // dO (+ L, Delta) ring slots
  static constexpr int DSLOT = S::TILE + 1024;               // dO | L*log2e | Delta
  static constexpr int OFF_V = S::TILE;
  static constexpr int OFF_Q = 2 * S::TILE;
  static constexpr int OFF_DO = OFF_Q + NQ * S::TILE;
  static constexpr int OFF_BAR = OFF_DO + ND * DSLOT;
  static constexpr int BAR_BYTES = 256;
  // Up to MAX_PAD bytes to bring the dynamic shared memory base to a 1024-byte
  // boundary (the kernel checks this at entry).
  static constexpr int MAX_PAD = D == 128 ? 768 : 1024;
  static constexpr int SMEM = OFF_BAR + BAR_BYTES + MAX_PAD;
  static constexpr uint32_t COL_ST = 0, COL_DPT = 128, COL_DV = 256, COL_DK = 256 + D;
};

template <typename T, int D, int DROP>
__global__ void __launch_bounds__(320, 1)
    bwd_dkdv_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo,
                       const BwdTcArgs a) {
  using C = DkdvCfg<D>;
  static_assert(C::SMEM <= 232448, "shared memory per block");
  static_assert(2 * 128 * D * 4 <= C::OFF_BAR, "cluster staging fits below the barriers");
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
  uint8_t* sD = smem + C::OFF_DO;           // slot s: dO tile | L2 (128 f32) | Delta (128 f32)
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  Ctl* ctl = reinterpret_cast<Ctl*>(bars + 28);
  const uint32_t b_kv = smem_u32(&bars[0]);
  const uint32_t b_qfull0 = smem_u32(&bars[1]);                  // + 8 * Q slot (3)
  const uint32_t b_qempty0 = smem_u32(&bars[4]);                 // + 8 * Q slot (3)
  const uint32_t b_dfull0 = smem_u32(&bars[7]);                  // + 8 * dO slot (2)
  const uint32_t b_dempty0 = smem_u32(&bars[9]);                 // + 8 * dO slot (2)
  const uint32_t b_sfull = smem_u32(&bars[11]);
  const uint32_t b_dpfull = smem_u32(&bars[12]);
  const uint32_t b_pready0 = smem_u32(&bars[13]);                // + 8 * half
  const uint32_t b_dsready0 = smem_u32(&bars[15]);               // + 8 * half
  const uint32_t b_accdone = smem_u32(&bars[17]);
  const uint32_t b_mmadone = smem_u32(&bars[18]);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // With split S > 1, the S CTAs of a cluster share one key tile: CTA `rank`
  // takes query heads rank*G/S .. (rank+1)*G/S - 1 of the group, and rank 0
  // sums the partial dK, dV through distributed shared memory at the end.
  const int split = a.split;
  const int rank = static_cast<int>(blockIdx.x % split);
  const int64_t id = blockIdx.x / split;
  // Grouped order (grouped_tile): the key-tile CTAs in flight belong to a few
  // heads, whose Q and dO tiles stay in L2; low key tiles (most work) first.
  int64_t bhk, kt;                              // b * Hkv + key/value head, key tile
  grouped_tile(id, a.BH, a.ntiles, a.hgroup, bhk, kt);
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
    // No query attends to these keys: dK = dV = 0 (every CTA of a cluster
    // takes this branch together).
    if (warp < 8 && rank == 0) {
      const int64_t key = kt * C::BT + (warp & 3) * 32 + lane;
      if (key < Nk) {
        const int64_t* st = (warp >> 2) ? a.s1 : a.s0;
        T* out = static_cast<T*>((warp >> 2) ? a.out1 : a.out0) + bb * st[0] + hk * st[1] +
                 (sv.k0 + key) * st[2];
        for (int d = 0; d < a.dreal; ++d) out[d] = Elem<T>::from_f32(0.f);
      }
    }
    return;
  }

  // The producer's lane 0 sets up the barriers and sends the first copies
  // (K, V, Q and dO of the first step) before the block-wide sync, so their
  // latency overlaps the set-up; the first step's L, Delta and the dO
  // barrier's arrivals follow in the producer loop.
  const int64_t q_first = static_cast<int64_t>(i0) * C::BT;
  const int32_t hq_first = static_cast<int32_t>(hk * a.g.G + g0);
  if (warp == 8) {
    if (lane == 0) {
      mbar_init(b_kv, 1);
      for (int s = 0; s < C::NQ; ++s) {
        mbar_init(b_qfull0 + 8 * s, 1);
        mbar_init(b_qempty0 + 8 * s, 1);
      }
      for (int s = 0; s < C::ND; ++s) {
        mbar_init(b_dfull0 + 8 * s, 32);
        mbar_init(b_dempty0 + 8 * s, 1);
      }
      mbar_init(b_sfull, 1);
      mbar_init(b_dpfull, 1);
      for (int h = 0; h < 2; ++h) {
        mbar_init(b_pready0 + 8 * h, 256);
        mbar_init(b_dsready0 + 8 * h, 256);
      }
      mbar_init(b_accdone, 1);
      mbar_init(b_mmadone, 1);
      ctl->abort = 0;
      mbar_fence_init();
      tma_prefetch_desc(&tmq); tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv); tma_prefetch_desc(&tmdo);
      mbar_arrive_expect_tx(b_kv, 2 * C::TILE);
      for (int c = 0; c < C::DC; ++c) {
        tma_load_4d(smem_u32(sK + c * C::CHUNK), &tmk, b_kv, c * 64,
                    static_cast<int32_t>(sv.k0 + kt * C::BT), hk, bb);
        tma_load_4d(smem_u32(sV + c * C::CHUNK), &tmv, b_kv, c * 64,
                    static_cast<int32_t>(sv.k0 + kt * C::BT), hk, bb);
      }
      mbar_arrive_expect_tx(b_qfull0, C::TILE);
      for (int c = 0; c < C::DC; ++c)
        tma_load_4d(smem_u32(sQ + c * C::CHUNK), &tmq, b_qfull0, c * 64,
                    static_cast<int32_t>(sv.q0 + q_first), hq_first, bb);
      mbar_expect_tx(b_dfull0, C::TILE);
      for (int c = 0; c < C::DC; ++c)
        tma_load_4d(smem_u32(sD + c * C::CHUNK), &tmdo, b_dfull0, c * 64,
                    static_cast<int32_t>(sv.q0 + q_first), hq_first, bb);
    }
    __syncwarp();
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
    // Lane 0 issues the TMA copies.  For each query tile: Q into its Q slot,
    // then dO into its dO slot, where all 32 lanes also stage L * log2(e) and
    // Delta (4 rows per lane, read from global memory before the slot is
    // free, so their latency overlaps the wait), both negated so that the
    // elementwise warps add them directly.  Rows past N get L = +inf, so
    // their probabilities are exactly 0, and Delta = 0.
    // (K, V and the first step's Q and dO tiles were sent before the sync)
    uint32_t q_round[C::NQ], d_round[C::ND];
#pragma unroll
    for (int s = 0; s < C::NQ; ++s) q_round[s] = 0;
#pragma unroll
    for (int s = 0; s < C::ND; ++s) d_round[s] = 0;
    bool ok = true;
    for (int it = 0; it < n; ++it) {
      const int64_t q0 = static_cast<int64_t>(i0 + it % per) * C::BT;     // within the sequence
      const int32_t hq = static_cast<int32_t>(hk * a.g.G + g0 + it / per);
      // Q_i
      const int qs = it % C::NQ;
      const uint32_t qr = static_cast<uint32_t>(it / C::NQ);
      if (lane == 0 && it == 0) {
        q_round[0] = 1;                      // sent before the sync
      } else if (lane == 0) {
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
      // dO_i, L, Delta
      float lv[4], dv[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int64_t q = q0 + lane * 4 + t;
        const int64_t li = lse_index(a.g, sv, hq, q);
        lv[t] = q < Nq ? -a.lse[li] * kLog2e : -INFINITY;   // staged negated
        dv[t] = q < Nq ? -a.delta[li] : 0.f;
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
      if (lane == 0 && it > 0) {
        mbar_arrive_expect_tx(b_dfull0 + 8 * ds, C::TILE);
        for (int c = 0; c < C::DC; ++c)
          tma_load_4d(smem_u32(slot + c * C::CHUNK), &tmdo, b_dfull0 + 8 * ds, c * 64,
                      static_cast<int32_t>(sv.q0 + q0), hq, bb);
      } else {
        mbar_arrive(b_dfull0 + 8 * ds);     // step 0: dO sent (expect_tx) before the sync
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
    // The whole warp runs the issue loop and its waits (warp-uniform loop
    // control and descriptor arithmetic); one elected lane issues the
    // products and commits.
    {
      const bool leader = elect_one();
      const uint32_t idS = idesc_f16<T>(128, C::BT, false, false);
      const uint32_t idG = idesc_f16<T>(128, D, false, true);
      const uint64_t dK0 = sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dV0 = sdesc_sw128(smem_u32(sV), 16, 1024);
      const uint64_t dQk = sdesc_sw128(smem_u32(sQ), 16, 1024);          // K-major views
      const uint64_t dDk = sdesc_sw128(smem_u32(sD), 16, 1024);
      const uint64_t dQm = sdesc_sw128(smem_u32(sQ), C::CHUNK, 1024);    // MN-major views
      const uint64_t dDm = sdesc_sw128(smem_u32(sD), C::CHUNK, 1024);
      auto issue_ST = [&](int qs) {   // S^T = K Q^T
        const uint64_t q = dQk + static_cast<uint64_t>((qs * C::TILE) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::CHUNK + (kk & 3) * 32) >> 4;
          if (leader) mma_ss(tmem + C::COL_ST, dK0 + off, q + off, idS, kk > 0 ? 1u : 0u);
        }
        if (leader) mma_commit(b_sfull);
      };
      auto issue_DPT = [&](int ds) {  // dP^T = V dO^T
        const uint64_t g = dDk + static_cast<uint64_t>((ds * C::DSLOT) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::CHUNK + (kk & 3) * 32) >> 4;
          if (leader) mma_ss(tmem + C::COL_DPT, dV0 + off, g + off, idS, kk > 0 ? 1u : 0u);
        }
        if (leader) mma_commit(b_dpfull);
      };
      bool ok = wait_warp(b_kv, 0, ctl, a.status, a.timeout_ns) &&
                wait_warp(b_qfull0, 0, ctl, a.status, a.timeout_ns) &&
                wait_warp(b_dfull0, 0, ctl, a.status, a.timeout_ns);
      if (ok) {
        tc_fence_after();
        issue_ST(0);
        issue_DPT(0);
      }
      for (int it = 0; ok && it < n; ++it) {
        const int qs = it % C::NQ, ds = it % C::ND;
        const bool next = it + 1 < n;
        const int qs1 = (it + 1) % C::NQ, ds1 = (it + 1) % C::ND;
        // dV += P^T dO (B: this tile's dO read MN-major, N = d)
        const uint64_t mdo = dDm + static_cast<uint64_t>((ds * C::DSLOT) >> 4);
        for (int h = 0; ok && h < 2; ++h) {
          if (!(ok = h > 0 || wait_warp(b_pready0, it & 1, ctl, a.status, a.timeout_ns))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            if (leader) mma_ts(tmem + C::COL_DV, tmem + C::COL_ST + 64 * h + 8 * kk,
                   mdo + static_cast<uint64_t>(((64 * h + 16 * kk) * 128) >> 4), idG,
                   (it > 0 || h > 0 || kk > 0) ? 1u : 0u);
        }
        if (!ok) break;
        if (next) {
          if (!(ok = wait_warp(b_qfull0 + 8 * qs1, ((it + 1) / C::NQ) & 1, ctl, a.status,
                                  a.timeout_ns)))
            break;
          tc_fence_after();
          issue_ST(qs1);
        }
        // dK += dS^T Q (B: this tile's Q read MN-major)
        const uint64_t mq = dQm + static_cast<uint64_t>((qs * C::TILE) >> 4);
        for (int h = 0; ok && h < 2; ++h) {
          if (!(ok = h > 0 || wait_warp(b_dsready0, it & 1, ctl, a.status, a.timeout_ns))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            if (leader) mma_ts(tmem + C::COL_DK, tmem + C::COL_DPT + 64 * h + 8 * kk,
                   mq + static_cast<uint64_t>(((64 * h + 16 * kk) * 128) >> 4), idG,
                   (it > 0 || h > 0 || kk > 0) ? 1u : 0u);
        }
        if (!ok) break;
        if (leader) mma_commit(b_qempty0 + 8 * qs);
        if (leader) mma_commit(b_dempty0 + 8 * ds);
        if (next) {
          if (!(ok = wait_warp(b_dfull0 + 8 * ds1, ((it + 1) / C::ND) & 1, ctl, a.status,
                                  a.timeout_ns)))
            break;
          tc_fence_after();
          issue_DPT(ds1);
        }
      }
      if (ok && leader) mma_commit(b_accdone);
      if (leader) mma_commit(b_mmadone);
      wait_bounded(b_mmadone, 0, ctl, a.status, a.timeout_ns, false);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ elementwise + epilogue
    const int hf = warp >> 2, quarter = warp & 3;
    const int row = quarter * 32 + lane;                 // key within the tile
    const int64_t key = kt * C::BT + row;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float c = a.c;
    bool ok = true;
    // Dropout keep bits: bit q set iff weight (query 64*hf + q of the step's
    // query tile, this key) is kept.  The eight lanes of an octet hold eight
    // consecutive keys, whose decisions for one query are one byte of the
    // keep mask or one generator call.  Mask bytes are loaded a step ahead
    // (mb), so their latency overlaps a whole step.
    uint32_t mb[8];
    if constexpr (DROP) {
      static_assert(C::BT == 128, "keep-mask entries cover 128-key tiles");
      if constexpr (DROP == kDropRead)
        octet_mask_load(a.drop, a.g, sv, hk * a.g.G + g0, kt, static_cast<int64_t>(i0) * C::BT + 64 * hf,
                        row >> 3, lane, mb);
    }
    for (int it = 0; it < n; ++it) {
      const int i = i0 + it % per, ds = it % C::ND;
      // keep bits drawn before the scores arrive (positions only), or the
      // prefetched mask bytes exchanged and the next step's loads issued
      uint64_t keep = 0;
      if constexpr (DROP) {
        if constexpr (DROP == kDropRead) {
          keep = octet_mask_bits(mb, lane);
          if (it + 1 < n)
            octet_mask_load(a.drop, a.g, sv, hk * a.g.G + g0 + (it + 1) / per, kt,
                            static_cast<int64_t>(i0 + (it + 1) % per) * C::BT + 64 * hf, row >> 3,
                            lane, mb);
        } else {
          keep = octet_keep_bits(a.drop, static_cast<uint32_t>(key >> 3),
                                 static_cast<int64_t>(i) * C::BT + 64 * hf,
                                 static_cast<uint32_t>(bseq * a.g.Hq + hk * a.g.G + g0 + it / per),
                                 lane);
        }
      }
      if (!(ok = wait_warp(b_sfull, it & 1, ctl, a.status, a.timeout_ns))) break;
      // the dO slot's arrival also publishes the staged L and Delta
      if (!(ok = wait_warp(b_dfull0 + 8 * ds, (it / C::ND) & 1, ctl, a.status, a.timeout_ns))) break;
      tc_fence_after();
      // -L * log2(e) and -Delta of this half's 64 queries
      const float* nL2s = reinterpret_cast<const float*>(sD + ds * C::DSLOT + C::TILE) + 64 * hf;
      const float* nDs = nL2s + 128;
      float p[64];
      tmem_ld64(lane_base + C::COL_ST + 64 * hf, p);
      {
        // P = exp2(c * S - L * log2(e)), two queries per paired instruction
        const uint64_t cc = f32x2(c, c);
#pragma unroll
        for (int q = 0; q < 64; q += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(nL2s + q);
          float x0, x1, x2, x3;
          f32x2_split(fma_f32x2(f32x2(p[q], p[q + 1]), cc, f32x2(l4.x, l4.y)), x0, x1);
          f32x2_split(fma_f32x2(f32x2(p[q + 2], p[q + 3]), cc, f32x2(l4.z, l4.w)), x2, x3);
          p[q] = ex2(x0);
          p[q + 1] = ex2(x1);
          p[q + 2] = ex2(x2);
          p[q + 3] = ex2(x3);
        }
      }
      if (a.causal && i == kt) {
        // diagonal tile: query (64*hf + q) attends to this key only if it is not earlier
#pragma unroll
        for (int q = 0; q < 64; ++q)
          if (64 * hf + q < row) p[q] = 0.f;
      }
      if constexpr (DROP) {
        // P o keep, rounded pairs formed straight from p (no fp32 copy
        // kept); Z's 1 / (1 - p) scales dV when it is stored
        // Queries 8t + e and 8t + e + 1 (e even) are bits t of bytes e and
        // e + 1 of keep: shifted by 7 - t, the pair's flags are those bytes'
        // sign bits, which one prmt spreads over the pair's two halves.
        const uint32_t kl = static_cast<uint32_t>(keep), kh = static_cast<uint32_t>(keep >> 32);
        uint32_t w[32];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const uint32_t xl = kl << (7 - t), xh = kh << (7 - t);
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const int q = 8 * t + e;
            w[q / 2] = pack2<T>(p[q], p[q + 1]) &
                       prmt(e < 4 ? xl : xh, 0u, half_sign_sel(e & 3, (e & 3) + 1));
          }
        }
        tmem_st32(lane_base + C::COL_ST + 64 * hf, w);
      } else {
        tmem_st_packed64<T>(lane_base + C::COL_ST + 64 * hf, p);
      }
      (void)keep;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(b_pready0);

      if (!(ok = wait_warp(b_dpfull, it & 1, ctl, a.status, a.timeout_ns))) break;
      tc_fence_after();
      if constexpr (DROP) {
        // dS = P o (Z o dP - Delta), Z = keep / (1 - p): dP / (1 - p) - Delta
        // for kept weights, -Delta for dropped ones, two queries per paired
        // instruction.  In two halves of 32 queries, so that only 32 of dP
        // are held next to P: half 0's rounded dS lands on columns whose dP
        // was read first, half 1's on half 0's.
        const uint64_t rs2 = f32x2(a.drop.rscale, a.drop.rscale);
        const uint32_t kl = static_cast<uint32_t>(keep), kh = static_cast<uint32_t>(keep >> 32);
        const uint32_t tdp = lane_base + C::COL_DPT + 64 * hf;
#pragma unroll
        for (int hq = 0; hq < 2; ++hq) {
          uint32_t r[32];
          tmem_ld32(tdp + 32 * hq, r);
          tmem_wait_ld();
          reg_fence32(r);
          uint32_t w[16];
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const int q = 32 * hq + j;
            const float2 d2 = *reinterpret_cast<const float2*>(nDs + q);
            float x0, x1;
            f32x2_split(fma_f32x2(f32x2(__uint_as_float(r[j]), __uint_as_float(r[j + 1])), rs2,
                                  f32x2(d2.x, d2.y)),
                        x0, x1);
            x0 = kept64(kl, kh, kbit(q)) ? x0 : d2.x;
            x1 = kept64(kl, kh, kbit(q + 1)) ? x1 : d2.y;
            f32x2_split(mul_f32x2(f32x2(x0, x1), f32x2(p[q], p[q + 1])), x0, x1);
            w[j / 2] = pack2<T>(x0, x1);
          }
          tmem_st16(tdp + 16 * hq, w);
        }
      } else {
        float dp[64];
        tmem_ld64(lane_base + C::COL_DPT + 64 * hf, dp);
#pragma unroll
        for (int q = 0; q < 64; q += 4) {
          // dS = P o (dP - Delta), two queries per paired instruction
          const float4 d4 = *reinterpret_cast<const float4*>(nDs + q);
          uint64_t a01 = add_f32x2(f32x2(dp[q], dp[q + 1]), f32x2(d4.x, d4.y));
          uint64_t a23 = add_f32x2(f32x2(dp[q + 2], dp[q + 3]), f32x2(d4.z, d4.w));
          a01 = mul_f32x2(a01, f32x2(p[q], p[q + 1]));
          a23 = mul_f32x2(a23, f32x2(p[q + 2], p[q + 3]));
          f32x2_split(a01, dp[q], dp[q + 1]);
          f32x2_split(a23, dp[q + 2], dp[q + 3]);
        }
        tmem_st_packed64<T>(lane_base + C::COL_DPT + 64 * hf, dp);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(b_dsready0);
    }
    if (ok) ok = wait_warp(b_accdone, 0, ctl, a.status, a.timeout_ns);
    ew_ok = ok;
    const uint32_t acc = lane_base + (hf == 0 ? C::COL_DV : C::COL_DK);
    const float mul = hf == 0 ? (DROP ? a.drop.rscale : 1.f) : a.scale;
    if (split == 1) {
      // Rows staged in shared memory (the Q ring is idle once every product
      // has completed) as the loads lay them out, then stored by the
      // warpgroup with consecutive threads on consecutive 16 bytes of a row:
      // whole lines per warp store instead of each thread's scattered row.
      // Rows past the sequence (the next packed sequence's) are not written.
      // Every thread of the warpgroup passes the barrier, also after a
      // timeout; the stores go out only if all of them got this far.
      const uint32_t stg = smem_u32(sQ) + static_cast<uint32_t>(hf * C::TILE);
      if (ok) {
        tc_fence_after();
        stage_row_sw128<T>(acc, mul, stg, row, 0, D);
      }
      if (bar_red_and(1 + hf, 128, ok)) {
        const int64_t* st = hf == 0 ? a.s0 : a.s1;
        T* row0 = static_cast<T*>(hf == 0 ? a.out0 : a.out1) + bb * st[0] + hk * st[1] +
                  (sv.k0 + kt * C::BT) * st[2];
        store_staged_tile<T>(stg, D, threadIdx.x & 127, 128, row0, st[2],
                             static_cast<int>(Nk - kt * C::BT < C::BT ? Nk - kt * C::BT : C::BT), a.dreal);
      }
    } else if (ok) {
      tc_fence_after();
      if (rank != 0) {
        // partial sums into this CTA's shared memory for rank 0 to read
        float* st = stage_row<D>(smem, hf, row);
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t t[32];
          tmem_ld32(acc + 32 * cc, t);
          tmem_wait_ld();
          reg_fence32(t);
#pragma unroll
          for (int u = 0; u < 8; ++u)
            *reinterpret_cast<uint4*>(st + 4 * stage_chunk(cc * 8 + u, row)) =
                make_uint4(t[4 * u], t[4 * u + 1], t[4 * u + 2], t[4 * u + 3]);
        }
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
      const uint32_t st = smem_u32(stage_row<D>(smem, hf, row));
      const float mul = hf == 0 ? (DROP ? a.drop.rscale : 1.f) : a.scale;
      T* out = hf == 0
                   ? static_cast<T*>(a.out0) + bb * a.s0[0] + hk * a.s0[1] + (sv.k0 + key) * a.s0[2]
                   : static_cast<T*>(a.out1) + bb * a.s1[0] + hk * a.s1[1] + (sv.k0 + key) * a.s1[2];
#pragma unroll 1
      for (int cc = 0; cc < a.dreal / 32 + (a.dreal % 32 ? 1 : 0); ++cc) {
        uint32_t t[32];
        tmem_ld32(acc + 32 * cc, t);
        tmem_wait_ld();
        reg_fence32(t);
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(t[i]);
        for (int r = 1; r < split; ++r) {
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const float4 x = ld_cluster_f4(cluster_map(st + 16 * stage_chunk(cc * 8 + u, row),
                                                       static_cast<uint32_t>(r)));
            v[4 * u] += x.x; v[4 * u + 1] += x.y; v[4 * u + 2] += x.z; v[4 * u + 3] += x.w;
          }
        }
        if (key < Nk) {
          const int ncol = min(32, a.dreal - 32 * cc);   // 16 or 32
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (8 * u >= ncol) break;
            uint4 w;
            w.x = pack2<T>(v[8 * u] * mul, v[8 * u + 1] * mul);
            w.y = pack2<T>(v[8 * u + 2] * mul, v[8 * u + 3] * mul);
            w.z = pack2<T>(v[8 * u + 4] * mul, v[8 * u + 5] * mul);
            w.w = pack2<T>(v[8 * u + 6] * mul, v[8 * u + 7] * mul);
            *reinterpret_cast<uint4*>(out + 32 * cc + 8 * u) = w;
          }
        }
      }
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

// ============================================================================
// dK / dV, persistent (D <= 64, no dropout, no cluster split): short sequences
// ============================================================================
// At short lengths a dK/dV CTA does 1-8 steps, and a clock64 trace put most
// of its time in set-up, the first loads, the epilogue and the launch of the
// next CTA.  This variant keeps one CTA per SM for the whole launch and walks
// the same (key tile, key/value head) items, most work first, round-robin
// over the CTAs.  Barriers and tensor memory are set up once; K | V are
// double-buffered in shared memory and dV | dK in tensor memory (all 512
// columns: S^T, dP^T, two accumulator pairs), so the producer loads item
// i+1's tiles while item i computes, and item i's epilogue (staged in its own
// shared memory) overlaps item i+1's products.  Every ring phase runs on a
// global step count; per-item barriers on the item count.  The per-step work
// is the non-persistent kernel's (no dropout).
struct DkdvPCfg : BwdShape<64> {
  using S = BwdShape<64>;
  static constexpr int NQ = 3, ND = 2;
  static constexpr int DSLOT = S::TILE + 1024;
  static constexpr int OFF_KV = 0;                           // 2 x (K | V)
  static constexpr int OFF_Q = 4 * S::TILE;
  static constexpr int OFF_DO = OFF_Q + NQ * S::TILE;
  static constexpr int OFF_STG = OFF_DO + ND * DSLOT;        // epilogue staging: dV | dK
  static constexpr int OFF_BAR = OFF_STG + 2 * S::TILE;
  static constexpr int SMEM = OFF_BAR + 512 + 1024;
  static constexpr uint32_t COL_ST = 0, COL_DPT = 128, COL_ACC = 256;   // acc pair b: 256 + 128 b
};

template <typename T>
__global__ void __launch_bounds__(320, 1)
    bwd_dkdv_persist_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                            const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo,
                            const BwdTcArgs a) {
  using C = DkdvPCfg;
  constexpr int D = 64;
  static_assert(C::SMEM <= 232448, "shared memory per block");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sD = smem + C::OFF_DO;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  Ctl* ctl = reinterpret_cast<Ctl*>(bars + 56);
  const uint32_t b_kvfull0 = smem_u32(&bars[0]);       // + 8 * buffer (2)
  const uint32_t b_kvempty0 = smem_u32(&bars[2]);      // + 8 * buffer (2)
  const uint32_t b_qfull0 = smem_u32(&bars[4]);        // + 8 * Q slot (3)
  const uint32_t b_qempty0 = smem_u32(&bars[7]);       // + 8 * Q slot (3)
  const uint32_t b_dfull0 = smem_u32(&bars[10]);       // + 8 * dO slot (2)
  const uint32_t b_dempty0 = smem_u32(&bars[12]);      // + 8 * dO slot (2)
  const uint32_t b_sfull = smem_u32(&bars[14]);
  const uint32_t b_dpfull = smem_u32(&bars[15]);
  const uint32_t b_pready0 = smem_u32(&bars[16]);      // + 8 * half
  const uint32_t b_dsready0 = smem_u32(&bars[18]);     // + 8 * half
  const uint32_t b_accdone0 = smem_u32(&bars[20]);     // + 8 * accumulator pair (2)
  const uint32_t b_accfree0 = smem_u32(&bars[22]);     // + 8 * accumulator pair (2)
  const uint32_t b_mmadone = smem_u32(&bars[24]);
  static_assert(25 * 8 <= 56 * 8, "barriers below the control block");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nitems = a.BH * a.ntiles;
  // One item: key tile kt of key/value head bhk (b * Hkv + head); low tiles
  // (most work under causal masking) first.
  struct Item {
    int64_t kt, bhk, bseq; int32_t hk, bb; SeqView sv; int64_t Nq, Nk; int i0, per, n;
  };
  // Round r of the walk: items r*P .. r*P + P - 1 (P CTAs), taken in snake
  // order (CTA c takes the c-th in even rounds, the c-th from the end in odd
  // ones), which pairs long and short items under causal masking.
  auto item_id = [&](int64_t r) {
    const int64_t P = gridDim.x;
    return r * P + ((r & 1) ? P - 1 - blockIdx.x : blockIdx.x);
  };
  auto item_at = [&](int64_t id) {   // id < 2^31 (checked at launch): 32-bit divisions
    Item it{};
    const uint32_t u = static_cast<uint32_t>(id), bh = static_cast<uint32_t>(a.BH),
                   hkv = static_cast<uint32_t>(a.g.Hkv);
    const uint32_t kt = u / bh, bhk = u - kt * bh, bseq = bhk / hkv;
    it.bhk = bhk; it.kt = kt; it.bseq = bseq;
    it.hk = static_cast<int32_t>(bhk - bseq * hkv);
    it.sv = seq_view(a.g, it.bseq);
    it.bb = static_cast<int32_t>(it.sv.b);
    it.Nq = it.sv.nq; it.Nk = it.sv.nk;
    const int nq = static_cast<int>((it.Nq + C::BT - 1) / C::BT);
    it.i0 = a.causal ? static_cast<int>(it.kt) : 0;
    it.per = nq > it.i0 ? nq - it.i0 : 0;
    it.n = (it.sv.ok && it.kt * C::BT < it.Nk) ? it.per * static_cast<int>(a.g.G) : 0;
    return it;
  };

  if (warp == 8) {
    if (lane == 0) {
      for (int b = 0; b < 2; ++b) {
        mbar_init(b_kvfull0 + 8 * b, 1);
        mbar_init(b_kvempty0 + 8 * b, 1);
        mbar_init(b_accdone0 + 8 * b, 1);
        mbar_init(b_accfree0 + 8 * b, 256);
      }
      for (int s = 0; s < C::NQ; ++s) {
        mbar_init(b_qfull0 + 8 * s, 1);
        mbar_init(b_qempty0 + 8 * s, 1);
      }
      for (int s = 0; s < C::ND; ++s) {
        mbar_init(b_dfull0 + 8 * s, 32);
        mbar_init(b_dempty0 + 8 * s, 1);
      }
      mbar_init(b_sfull, 1);
      mbar_init(b_dpfull, 1);
      for (int h = 0; h < 2; ++h) {
        mbar_init(b_pready0 + 8 * h, 256);
        mbar_init(b_dsready0 + 8 * h, 256);
      }
      mbar_init(b_mmadone, 1);
      ctl->abort = 0;
      mbar_fence_init();
      tma_prefetch_desc(&tmq); tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv); tma_prefetch_desc(&tmdo);
    }
    __syncwarp();
    tmem_alloc(smem_u32(&ctl->tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    // Per item: K, V into buffer (item count) & 1 once the item two back has
    // released it; then per step Q and dO (+ negated L * log2(e) and Delta,
    // staged by all 32 lanes) into their rings, slots and rounds counted
    // over every step this CTA has run.
    uint32_t kv_round[2] = {0u, 0u}, q_round[C::NQ], d_round[C::ND];
#pragma unroll
    for (int s = 0; s < C::NQ; ++s) q_round[s] = 0;
#pragma unroll
    for (int s = 0; s < C::ND; ++s) d_round[s] = 0;
    uint32_t gstep = 0;   // steps of this CTA so far (< 2^31)
    int li = 0;
    bool ok = true;
    for (int64_t r = 0; ok && r * gridDim.x < nitems; ++r) {
      const int64_t id = item_id(r);
      if (id >= nitems) continue;
      const Item itm = item_at(id);
      if (itm.n == 0) continue;
      const int buf = li & 1;
      if (lane == 0) {
        if (li >= 2 && !wait_bounded(b_kvempty0 + 8 * buf, ((li >> 1) - 1) & 1, ctl, a.status,
                                     a.timeout_ns))
          ok = false;
        if (ok) {
          uint8_t* kv = smem + C::OFF_KV + buf * 2 * C::TILE;
          mbar_arrive_expect_tx(b_kvfull0 + 8 * buf, 2 * C::TILE);
          tma_load_4d(smem_u32(kv), &tmk, b_kvfull0 + 8 * buf, 0,
                      static_cast<int32_t>(itm.sv.k0 + itm.kt * C::BT), itm.hk, itm.bb);
          tma_load_4d(smem_u32(kv + C::TILE), &tmv, b_kvfull0 + 8 * buf, 0,
                      static_cast<int32_t>(itm.sv.k0 + itm.kt * C::BT), itm.hk, itm.bb);
          kv_round[buf] = static_cast<uint32_t>(li >> 1) + 1;
        }
      }
      ok = __all_sync(0xffffffffu, ok);
      for (int it = 0; ok && it < itm.n; ++it) {
        const uint32_t g = gstep + static_cast<uint32_t>(it);
        const int64_t q0 = static_cast<int64_t>(itm.i0 + it % itm.per) * C::BT;
        const int32_t hq = static_cast<int32_t>(itm.hk * a.g.G + it / itm.per);
        const int qs = static_cast<int>(g % C::NQ);
        const uint32_t qr = static_cast<uint32_t>(g / C::NQ);
        if (lane == 0) {
          if (qr > 0 && !wait_bounded(b_qempty0 + 8 * qs, (qr - 1) & 1, ctl, a.status, a.timeout_ns))
            ok = false;
          if (ok) {
            mbar_arrive_expect_tx(b_qfull0 + 8 * qs, C::TILE);
            tma_load_4d(smem_u32(sQ + qs * C::TILE), &tmq, b_qfull0 + 8 * qs, 0,
                        static_cast<int32_t>(itm.sv.q0 + q0), hq, itm.bb);
            q_round[qs] = qr + 1;
          }
        }
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        float lv[4], dv[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int64_t q = q0 + lane * 4 + t;
          const int64_t li2 = lse_index(a.g, itm.sv, hq, q);
          lv[t] = q < itm.Nq ? -a.lse[li2] * kLog2e : -INFINITY;   // staged negated
          dv[t] = q < itm.Nq ? -a.delta[li2] : 0.f;
        }
        const int ds = static_cast<int>(g % C::ND);
        const uint32_t dr = static_cast<uint32_t>(g / C::ND);
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
          tma_load_4d(smem_u32(slot), &tmdo, b_dfull0 + 8 * ds, 0,
                      static_cast<int32_t>(itm.sv.q0 + q0), hq, itm.bb);
        } else {
          mbar_arrive(b_dfull0 + 8 * ds);
        }
        d_round[ds] = dr + 1;
      }
      gstep += static_cast<uint32_t>(itm.n);
      ++li;
    }
    // Drain: every copy issued has landed.
    if (lane == 0) {
      for (int b = 0; b < 2; ++b)
        if (kv_round[b]) wait_bounded(b_kvfull0 + 8 * b, (kv_round[b] - 1) & 1, ctl, a.status,
                                      a.timeout_ns, false);
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
    // The non-persistent kernel's order per step; per item K | V from buffer
    // (item count) & 1 and dV | dK into accumulator pair (item count) & 1,
    // whose first product waits until the epilogue of the item two back has
    // read that pair.
    // The whole warp runs the issue loop and its waits (warp-uniform loop
    // control and descriptor arithmetic); one elected lane issues the
    // products and commits.
    {
      const bool leader = elect_one();
      const uint32_t idS = idesc_f16<T>(128, C::BT, false, false);
      const uint32_t idG = idesc_f16<T>(128, D, false, true);
      const uint64_t dKV0 = sdesc_sw128(smem_u32(smem + C::OFF_KV), 16, 1024);
      const uint64_t dQk = sdesc_sw128(smem_u32(sQ), 16, 1024);          // K-major views
      const uint64_t dDk = sdesc_sw128(smem_u32(sD), 16, 1024);
      const uint64_t dQm = sdesc_sw128(smem_u32(sQ), C::CHUNK, 1024);    // MN-major views
      const uint64_t dDm = sdesc_sw128(smem_u32(sD), C::CHUNK, 1024);
      auto issue_ST = [&](int qs, int buf) {   // S^T = K Q^T
        const uint64_t q = dQk + static_cast<uint64_t>((qs * C::TILE) >> 4);
        const uint64_t kd = dKV0 + static_cast<uint64_t>((buf * 2 * C::TILE) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk & 3) * 32) >> 4;
          if (leader) mma_ss(tmem + C::COL_ST, kd + off, q + off, idS, kk > 0 ? 1u : 0u);
        }
        if (leader) mma_commit(b_sfull);
      };
      auto issue_DPT = [&](int ds, int buf) {  // dP^T = V dO^T
        const uint64_t gd = dDk + static_cast<uint64_t>((ds * C::DSLOT) >> 4);
        const uint64_t vd = dKV0 + static_cast<uint64_t>((buf * 2 * C::TILE + C::TILE) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk & 3) * 32) >> 4;
          if (leader) mma_ss(tmem + C::COL_DPT, vd + off, gd + off, idS, kk > 0 ? 1u : 0u);
        }
        if (leader) mma_commit(b_dpfull);
      };
      uint32_t gstep = 0;   // steps of this CTA so far (< 2^31)
      int li = 0;
      bool ok = true;
      for (int64_t r = 0; ok && r * gridDim.x < nitems; ++r) {
        const int64_t id = item_id(r);
        if (id >= nitems) continue;
        const Item itm = item_at(id);
        if (itm.n == 0) continue;
        const int buf = li & 1;
        const uint32_t accv = tmem + C::COL_ACC + 128 * buf, acck = accv + 64;
        ok = wait_warp(b_kvfull0 + 8 * buf, (li >> 1) & 1, ctl, a.status, a.timeout_ns) &&
             wait_warp(b_qfull0 + 8 * static_cast<int>(gstep % C::NQ),
                          static_cast<uint32_t>(gstep / C::NQ) & 1, ctl, a.status, a.timeout_ns) &&
             wait_warp(b_dfull0 + 8 * static_cast<int>(gstep % C::ND),
                          static_cast<uint32_t>(gstep / C::ND) & 1, ctl, a.status, a.timeout_ns);
        if (!ok) break;
        tc_fence_after();
        issue_ST(static_cast<int>(gstep % C::NQ), buf);
        issue_DPT(static_cast<int>(gstep % C::ND), buf);
        if (li >= 2 && !(ok = wait_warp(b_accfree0 + 8 * buf, ((li >> 1) - 1) & 1, ctl, a.status,
                                           a.timeout_ns)))
          break;
        for (int it = 0; ok && it < itm.n; ++it) {
          const uint32_t g = gstep + static_cast<uint32_t>(it);
          const int qs = static_cast<int>(g % C::NQ), ds = static_cast<int>(g % C::ND);
          const bool next = it + 1 < itm.n;
          const int qs1 = static_cast<int>((g + 1) % C::NQ), ds1 = static_cast<int>((g + 1) % C::ND);
          const uint32_t par = g & 1u;
          // dV += P^T dO (B: this step's dO read MN-major, N = d)
          const uint64_t mdo = dDm + static_cast<uint64_t>((ds * C::DSLOT) >> 4);
          for (int h = 0; ok && h < 2; ++h) {
            if (!(ok = h > 0 || wait_warp(b_pready0, par, ctl, a.status, a.timeout_ns))) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              if (leader) mma_ts(accv, tmem + C::COL_ST + 64 * h + 8 * kk,
                     mdo + static_cast<uint64_t>(((64 * h + 16 * kk) * 128) >> 4), idG,
                     (it > 0 || h > 0 || kk > 0) ? 1u : 0u);
          }
          if (!ok) break;
          if (next) {
            if (!(ok = wait_warp(b_qfull0 + 8 * qs1, static_cast<uint32_t>((g + 1) / C::NQ) & 1,
                                    ctl, a.status, a.timeout_ns)))
              break;
            tc_fence_after();
            issue_ST(qs1, buf);
          }
          // dK += dS^T Q (B: this step's Q read MN-major)
          const uint64_t mq = dQm + static_cast<uint64_t>((qs * C::TILE) >> 4);
          for (int h = 0; ok && h < 2; ++h) {
            if (!(ok = h > 0 || wait_warp(b_dsready0, par, ctl, a.status, a.timeout_ns))) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              if (leader) mma_ts(acck, tmem + C::COL_DPT + 64 * h + 8 * kk,
                     mq + static_cast<uint64_t>(((64 * h + 16 * kk) * 128) >> 4), idG,
                     (it > 0 || h > 0 || kk > 0) ? 1u : 0u);
          }
          if (!ok) break;
          if (leader) mma_commit(b_qempty0 + 8 * qs);
          if (leader) mma_commit(b_dempty0 + 8 * ds);
          if (next) {
            if (!(ok = wait_warp(b_dfull0 + 8 * ds1, static_cast<uint32_t>((g + 1) / C::ND) & 1,
                                    ctl, a.status, a.timeout_ns)))
              break;
            tc_fence_after();
            issue_DPT(ds1, buf);
          }
        }
        if (!ok) break;
        if (leader) mma_commit(b_kvempty0 + 8 * buf);
        if (leader) mma_commit(b_accdone0 + 8 * buf);
        gstep += static_cast<uint32_t>(itm.n);
        ++li;
      }
      if (leader) mma_commit(b_mmadone);
      wait_bounded(b_mmadone, 0, ctl, a.status, a.timeout_ns, false);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ elementwise + epilogue
    const int hf = warp >> 2, quarter = warp & 3;
    const int row = quarter * 32 + lane;                 // key within the tile
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float c = a.c;
    const uint32_t stg = smem_u32(smem + C::OFF_STG) + static_cast<uint32_t>(hf * C::TILE);
    uint32_t gstep = 0;   // steps of this CTA so far (< 2^31)
    int li = 0;
    bool ok = true;
    // Epilogue of item `e` (item count `eli`): its accumulator pair, staged in
    // the CTA's own staging tiles (dV | dK) and stored with consecutive
    // threads on consecutive 16 bytes of a row; the pair is released to the
    // MMA thread once read.  Every thread of the warpgroup passes the
    // barrier, also after a timeout.
    T* pend_row0 = nullptr;   // the pending item's first output row (dV or dK of this warpgroup)
    int pend_rows = 0, pend_li = -1;
    auto epilogue = [&](T* row0, int nrows, int eli) {
      const int buf = eli & 1;
      if (ok)
        ok = wait_warp(b_accdone0 + 8 * buf, static_cast<uint32_t>(eli >> 1) & 1, ctl, a.status,
                       a.timeout_ns);
      if (ok) {
        tc_fence_after();
        stage_row_sw128<T>(lane_base + C::COL_ACC + 128 * buf + 64 * hf, hf == 0 ? 1.f : a.scale,
                           stg, row, 0, D);
      }
      tc_fence_before();
      mbar_arrive(b_accfree0 + 8 * buf);
      if (bar_red_and(1 + hf, 128, ok))
        store_staged_tile<T>(stg, D, threadIdx.x & 127, 128, row0, (hf == 0 ? a.s0 : a.s1)[2], nrows,
                             a.dreal);
    };
    // After a wait ran out (ok false) the warp still walks every item and
    // passes each epilogue barrier, doing nothing else, so that the other
    // warps of its warpgroup never wait on it at a barrier.
    for (int64_t r = 0; r * gridDim.x < nitems; ++r) {
      const int64_t id = item_id(r);
      if (id >= nitems) continue;
      const Item itm = item_at(id);
      if (!itm.sv.ok) {
        if (threadIdx.x == 0 && itm.kt == 0) record_status(a.status, FA_ERR_SEQLENS);
        continue;
      }
      if (itm.kt * C::BT >= itm.Nk) continue;           // this key tile lies past the sequence
      if (itm.n == 0) {
        // no query attends to these keys: dK = dV = 0
        const int64_t* st = hf == 0 ? a.s0 : a.s1;
        T* row0 = static_cast<T*>(hf == 0 ? a.out0 : a.out1) + itm.bb * st[0] + itm.hk * st[1] +
                  (itm.sv.k0 + itm.kt * C::BT) * st[2];
        if (row < itm.Nk - itm.kt * C::BT)
          for (int d = 0; d < a.dreal; ++d) row0[row * st[2] + d] = Elem<T>::from_f32(0.f);
        continue;
      }
      for (int it = 0; ok && it < itm.n; ++it) {
        const uint32_t g = gstep + static_cast<uint32_t>(it);
        const int i = itm.i0 + it % itm.per, ds = static_cast<int>(g % C::ND);
        const uint32_t par = g & 1u;
        if (!(ok = wait_warp(b_sfull, par, ctl, a.status, a.timeout_ns))) break;
        // the dO slot's arrival also publishes the staged L and Delta
        if (!(ok = wait_warp(b_dfull0 + 8 * ds, static_cast<uint32_t>(g / C::ND) & 1, ctl, a.status,
                             a.timeout_ns)))
          break;
        tc_fence_after();
        // -L * log2(e) and -Delta of this half's 64 queries
        const float* nL2s = reinterpret_cast<const float*>(sD + ds * C::DSLOT + C::TILE) + 64 * hf;
        const float* nDs = nL2s + 128;
        float p[64];
        tmem_ld64(lane_base + C::COL_ST + 64 * hf, p);
        {
          // P = exp2(c * S - L * log2(e)), two queries per paired instruction
          const uint64_t cc = f32x2(c, c);
#pragma unroll
          for (int q = 0; q < 64; q += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(nL2s + q);
            float x0, x1, x2, x3;
            f32x2_split(fma_f32x2(f32x2(p[q], p[q + 1]), cc, f32x2(l4.x, l4.y)), x0, x1);
            f32x2_split(fma_f32x2(f32x2(p[q + 2], p[q + 3]), cc, f32x2(l4.z, l4.w)), x2, x3);
            p[q] = ex2(x0);
            p[q + 1] = ex2(x1);
            p[q + 2] = ex2(x2);
            p[q + 3] = ex2(x3);
          }
        }
        if (a.causal && i == itm.kt) {
          // diagonal tile: query (64*hf + q) attends to this key only if it is not earlier
#pragma unroll
          for (int q = 0; q < 64; ++q)
            if (64 * hf + q < row) p[q] = 0.f;
        }
        tmem_st_packed64<T>(lane_base + C::COL_ST + 64 * hf, p);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(b_pready0);

        if (!(ok = wait_warp(b_dpfull, par, ctl, a.status, a.timeout_ns))) break;
        tc_fence_after();
        // dS = P o (dP - Delta), two queries per paired instruction, in two
        // halves of 32 columns (only 32 of dP held next to P): half 0's
        // rounded dS lands on columns whose dP was read first, half 1's on
        // half 0's
        const uint32_t tdp = lane_base + C::COL_DPT + 64 * hf;
#pragma unroll
        for (int hq = 0; hq < 2; ++hq) {
          uint32_t r[32];
          tmem_ld32(tdp + 32 * hq, r);
          tmem_wait_ld();
          reg_fence32(r);
          uint32_t w[16];
#pragma unroll
          for (int j2 = 0; j2 < 32; j2 += 2) {
            const int q = 32 * hq + j2;
            const float2 d2 = *reinterpret_cast<const float2*>(nDs + q);
            float x0, x1;
            f32x2_split(mul_f32x2(add_f32x2(f32x2(__uint_as_float(r[j2]), __uint_as_float(r[j2 + 1])),
                                            f32x2(d2.x, d2.y)),
                                  f32x2(p[q], p[q + 1])),
                        x0, x1);
            w[j2 / 2] = pack2<T>(x0, x1);
          }
          tmem_st16(tdp + 16 * hq, w);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(b_dsready0);
      }
      // The previous item's epilogue, deferred to here so that its products
      // have long completed and this item's steps ran without waiting for it.
      if (pend_li >= 0) epilogue(pend_row0, pend_rows, pend_li);
      {
        const int64_t* st = hf == 0 ? a.s0 : a.s1;
        pend_row0 = static_cast<T*>(hf == 0 ? a.out0 : a.out1) + itm.bb * st[0] + itm.hk * st[1] +
                    (itm.sv.k0 + itm.kt * C::BT) * st[2];
        pend_rows = static_cast<int>(itm.Nk - itm.kt * C::BT < C::BT ? itm.Nk - itm.kt * C::BT : C::BT);
      }
      pend_li = li;
      gstep += static_cast<uint32_t>(itm.n);
      ++li;
    }
    if (pend_li >= 0) epilogue(pend_row0, pend_rows, pend_li);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ============================================================================
// dQ
// ============================================================================
// Q_i and dO_i are only A operands (of S = Q K^T and dP = dO V^T), so they are
// copied once into TMEM and their shared memory then holds key tiles: NST
// stages of K_j | V_j, the last of which first receives Q_i and dO_i.
template <int D>
struct DqCfg : BwdShape<D> {
  using S = BwdShape<D>;
  static constexpr int NST = D == 128 ? 3 : 6;               // key-tile stages (K | V)
  static constexpr int STAGE = 2 * S::TILE;
  static constexpr int QSLOT = NST - 1;                      // stage that first holds Q | dO
  static constexpr int OFF_BAR = NST * STAGE;
  static constexpr int SMEM = OFF_BAR + 1024 + 1024;
  // TMEM: Q and dO (input type, two per column), the dQ accumulator, S and dP
  // (fp32; dS is written over the first 32 columns of each dP half).
  static constexpr uint32_t COL_Q = 0, COL_DO = D / 2, COL_DQ = D, COL_S = 256, COL_DP = 384;
};

// Copies this thread's row of a 128-byte-swizzled 128 x D tile (shared
// memory) into D / 2 TMEM columns of its lane, two elements per column, as an
// A operand.
template <int D>
__device__ __forceinline__ void tile_row_to_tmem(const uint8_t* tile, int row, uint32_t taddr) {
#pragma unroll
  for (int ch = 0; ch < D / 64; ++ch) {
    const uint8_t* base = tile + ch * (128 * 128) + row * 128;
    uint32_t w[32];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint4 x = *reinterpret_cast<const uint4*>(base + ((u ^ (row & 7)) << 4));
      w[4 * u] = x.x; w[4 * u + 1] = x.y; w[4 * u + 2] = x.z; w[4 * u + 3] = x.w;
    }
    tmem_st32(taddr + 32 * ch, w);
  }
}

template <typename T, int D, int DROP>
__global__ void __launch_bounds__(320, 1)
    bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo,
                     const BwdTcArgs a) {
  using C = DqCfg<D>;
  // At D <= 64, Q and dO stay in shared memory (their stage is not reused)
  // and S, dP read them from there: no per-CTA copy into TMEM before the
  // first product, which short sequences cannot hide; NST - 1 stages still
  // hold K | V.  At D = 128 the stage is needed for K | V (three stages).
  constexpr bool QS = D == 64;
  constexpr int NR = QS ? C::NST - 1 : C::NST;   // K | V ring stages
  static_assert(C::SMEM <= 232448, "shared memory per block");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sStage = smem;                   // stage st: K | V
  uint8_t* sQ = smem + C::QSLOT * C::STAGE; // Q | dO before they move to TMEM
  uint8_t* sDO = sQ + C::TILE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  Ctl* ctl = reinterpret_cast<Ctl*>(bars + 48);
  const uint32_t b_q = smem_u32(&bars[0]);
  const uint32_t b_kvfull0 = smem_u32(&bars[1]);                 // + 8 * stage
  const uint32_t b_kvempty0 = smem_u32(&bars[1 + C::NST]);       // + 8 * stage
  const uint32_t b_sfull = smem_u32(&bars[1 + 2 * C::NST]);
  const uint32_t b_sfree = smem_u32(&bars[2 + 2 * C::NST]);
  const uint32_t b_dpfull = smem_u32(&bars[3 + 2 * C::NST]);
  const uint32_t b_dsready0 = smem_u32(&bars[4 + 2 * C::NST]);   // + 8 * half
  const uint32_t b_accdone = smem_u32(&bars[6 + 2 * C::NST]);
  const uint32_t b_mmadone = smem_u32(&bars[7 + 2 * C::NST]);
  const uint32_t b_qt = smem_u32(&bars[8 + 2 * C::NST]);         // Q, dO are in TMEM

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t id = blockIdx.x;
  // Grouped order (grouped_tile): the query-tile CTAs in flight belong to a
  // few heads, whose K and V tiles stay in L2; the longest tiles first.
  int64_t bh, t;                                // b * Hq + h
  grouped_tile(id, a.BH, a.ntiles, a.hgroup, bh, t);
  const int64_t qt = a.causal ? (a.ntiles - 1 - t) : t;
  const int64_t h = bh % a.g.Hq;
  const SeqView sv = seq_view(a.g, bh / a.g.Hq);
  if (!sv.ok) {
    if (threadIdx.x == 0) record_status(a.status, FA_ERR_SEQLENS);
    return;
  }
  const int64_t Nq = sv.nq, Nk = sv.nk;
  if (qt * C::BT >= Nq) return;                 // this query tile lies past the sequence
  const int32_t hq = static_cast<int32_t>(h), hk = static_cast<int32_t>(h / a.g.G);
  const int32_t bb = static_cast<int32_t>(sv.b);
  const int nk = static_cast<int>((Nk + C::BT - 1) / C::BT);
  const int n = a.causal ? min(static_cast<int>(qt) + 1, nk) : nk;   // key tiles to visit
  if (n == 0) {
    // No key at all (an empty key sequence): dQ = 0.
    if (warp < 4) {
      const int64_t qrow = qt * C::BT + warp * 32 + lane;
      if (qrow < Nq) {
        T* out = static_cast<T*>(a.out0) + bb * a.s0[0] + hq * a.s0[1] + (sv.q0 + qrow) * a.s0[2];
        for (int d = 0; d < a.dreal; ++d) out[d] = Elem<T>::from_f32(0.f);
      }
    }
    return;
  }

  // The producer's lane 0 sets up the barriers and sends the first copies
  // (Q, dO and the K | V tiles of the stages that do not hold Q | dO) before
  // the block-wide sync, so their latency overlaps the set-up.
  const int jt_early = n < C::QSLOT ? n : C::QSLOT;   // key tiles sent before the sync
  auto load_kv = [&](int jt, int st) {
    uint8_t* stage = sStage + st * C::STAGE;
    mbar_arrive_expect_tx(b_kvfull0 + 8 * st, 2 * C::TILE);
    for (int c = 0; c < C::DC; ++c) {
      const int32_t krow = static_cast<int32_t>(sv.k0 + static_cast<int64_t>(jt) * C::BT);
      tma_load_4d(smem_u32(stage + c * C::CHUNK), &tmk, b_kvfull0 + 8 * st, c * 64, krow, hk, bb);
      tma_load_4d(smem_u32(stage + C::TILE + c * C::CHUNK), &tmv, b_kvfull0 + 8 * st, c * 64,
                  krow, hk, bb);
    }
  };
  if (warp == 8) {
    if (lane == 0) {
      mbar_init(b_q, 1);
      for (int s = 0; s < C::NST; ++s) {
        mbar_init(b_kvfull0 + 8 * s, 1);
        mbar_init(b_kvempty0 + 8 * s, 1);
      }
      mbar_init(b_sfull, 1);
      mbar_init(b_sfree, 256);
      mbar_init(b_dpfull, 1);
      for (int h = 0; h < 2; ++h) mbar_init(b_dsready0 + 8 * h, 256);
      mbar_init(b_accdone, 1);
      mbar_init(b_mmadone, 1);
      mbar_init(b_qt, 256);
      ctl->abort = 0;
      mbar_fence_init();
      tma_prefetch_desc(&tmq); tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv); tma_prefetch_desc(&tmdo);
      mbar_arrive_expect_tx(b_q, 2 * C::TILE);
      for (int c = 0; c < C::DC; ++c) {
        tma_load_4d(smem_u32(sQ + c * C::CHUNK), &tmq, b_q, c * 64,
                    static_cast<int32_t>(sv.q0 + qt * C::BT), hq, bb);
        tma_load_4d(smem_u32(sDO + c * C::CHUNK), &tmdo, b_q, c * 64,
                    static_cast<int32_t>(sv.q0 + qt * C::BT), hq, bb);
      }
      for (int jt = 0; jt < jt_early; ++jt) load_kv(jt, jt);   // stages 0 .. QSLOT - 1, round 0
    }
    __syncwarp();
    tmem_alloc(smem_u32(&ctl->tmem_base), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // (Q, dO and key tiles 0 .. jt_early - 1 were sent before the sync)
      uint32_t last_round[C::NST];
#pragma unroll
      for (int s = 0; s < C::NST; ++s) last_round[s] = s < jt_early ? 1u : 0u;
      for (int jt = jt_early; jt < n; ++jt) {
        const int st = jt % NR;
        const uint32_t r = static_cast<uint32_t>(jt / NR);
        if (r > 0) {
          if (!wait_bounded(b_kvempty0 + 8 * st, (r - 1) & 1, ctl, a.status, a.timeout_ns)) break;
        } else if (!QS && st == C::QSLOT) {
          // this stage still holds Q | dO until they have been copied into TMEM
          if (!wait_bounded(b_qt, 0, ctl, a.status, a.timeout_ns)) break;
        }
        load_kv(jt, st);
        last_round[st] = r + 1;
      }
      wait_bounded(b_q, 0, ctl, a.status, a.timeout_ns, false);
      for (int s = 0; s < C::NST; ++s)
        if (last_round[s]) wait_bounded(b_kvfull0 + 8 * s, (last_round[s] - 1) & 1, ctl, a.status,
                                        a.timeout_ns, false);
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // Order: S_0, dP_0, then per key tile jt: S_jt+1 (once S_jt has been read
    // out of TMEM), dQ += dS_jt K_jt (once dS_jt is ready), dP_jt+1 (it
    // overwrites dS_jt, read only by the dQ products issued before it).
    // The whole warp runs the issue loop and its waits (warp-uniform loop
    // control and descriptor arithmetic); one elected lane issues the
    // products and commits.
    {
      const bool leader = elect_one();
      const uint32_t idS = idesc_f16<T>(128, C::BT, false, false);
      const uint32_t idG = idesc_f16<T>(128, D, false, true);
      const uint64_t dSt0 = sdesc_sw128(smem_u32(sStage), 16, 1024);
      const uint64_t dSt0mn = sdesc_sw128(smem_u32(sStage), C::CHUNK, 1024);
      const uint64_t dQa = sdesc_sw128(smem_u32(sQ), 16, 1024);     // K-major A views (QS)
      const uint64_t dDa = sdesc_sw128(smem_u32(sDO), 16, 1024);
      auto issue_S = [&](int st) {   // S = Q K^T, Q from TMEM (or shared memory, QS)
        const uint64_t kb = dSt0 + static_cast<uint64_t>((st * C::STAGE) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::CHUNK + (kk & 3) * 32) >> 4;
          if constexpr (QS) {
            if (leader) mma_ss(tmem + C::COL_S, dQa + off, kb + off, idS, kk > 0 ? 1u : 0u);
          } else {
            if (leader) mma_ts(tmem + C::COL_S, tmem + C::COL_Q + 8 * kk, kb + off, idS, kk > 0 ? 1u : 0u);
          }
        }
      };
      auto issue_dP = [&](int st) {  // dP = dO V^T, dO from TMEM (or shared memory, QS)
        const uint64_t vb = dSt0 + static_cast<uint64_t>((st * C::STAGE + C::TILE) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::CHUNK + (kk & 3) * 32) >> 4;
          if constexpr (QS) {
            if (leader) mma_ss(tmem + C::COL_DP, dDa + off, vb + off, idS, kk > 0 ? 1u : 0u);
          } else {
            if (leader) mma_ts(tmem + C::COL_DP, tmem + C::COL_DO + 8 * kk, vb + off, idS, kk > 0 ? 1u : 0u);
          }
        }
      };
      bool ok = wait_warp(QS ? b_q : b_qt, 0, ctl, a.status, a.timeout_ns) &&
                wait_warp(b_kvfull0, 0, ctl, a.status, a.timeout_ns);
      if (ok) {
        tc_fence_after();
        issue_S(0);
        if (leader) mma_commit(b_sfull);
        issue_dP(0);
        if (leader) mma_commit(b_dpfull);
      }
      for (int jt = 0; ok && jt < n; ++jt) {
        const int st = jt % NR;
        const bool next = jt + 1 < n;
        const int stn = (jt + 1) % NR;
        if (next) {
          if (!(ok = wait_warp(b_kvfull0 + 8 * stn, ((jt + 1) / NR) & 1, ctl, a.status,
                                  a.timeout_ns)))
            break;
          if (!(ok = wait_warp(b_sfree, jt & 1, ctl, a.status, a.timeout_ns))) break;
          tc_fence_after();
          issue_S(stn);
          if (leader) mma_commit(b_sfull);
        }
        const uint64_t kmn = dSt0mn + static_cast<uint64_t>((st * C::STAGE) >> 4);
        for (int h = 0; ok && h < 2; ++h) {
          if (!(ok = h > 0 || wait_warp(b_dsready0, jt & 1, ctl, a.status, a.timeout_ns))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            if (leader) mma_ts(tmem + C::COL_DQ, tmem + C::COL_DP + 64 * h + 8 * kk,
                   kmn + static_cast<uint64_t>(((64 * h + 16 * kk) * 128) >> 4), idG,
                   (jt > 0 || h > 0 || kk > 0) ? 1u : 0u);
        }
        if (!ok) break;
        if (leader) mma_commit(b_kvempty0 + 8 * st);
        if (next) {
          issue_dP(stn);
          if (leader) mma_commit(b_dpfull);
        }
      }
      if (ok && leader) mma_commit(b_accdone);
      if (leader) mma_commit(b_mmadone);
      wait_bounded(b_mmadone, 0, ctl, a.status, a.timeout_ns, false);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ elementwise + epilogue
    const int hf = warp >> 2, quarter = warp & 3;
    const int row = quarter * 32 + lane;                  // query within the tile
    const int64_t qrow = qt * C::BT + row;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float c = a.c;
    const int64_t li = lse_index(a.g, sv, h, qrow);
    const float l2 = qrow < Nq ? a.lse[li] * kLog2e : INFINITY;
    const float dl = qrow < Nq ? a.delta[li] : 0.f;
    // Q (warps 0-3) and dO (warps 4-7) into TMEM as A operands (not in QS
    // mode, where the products read them from shared memory).
    bool ok = true;
    if constexpr (!QS) {
      ok = wait_warp(b_q, 0, ctl, a.status, a.timeout_ns);
      if (ok) {
        tile_row_to_tmem<D>(hf == 0 ? sQ : sDO, row, lane_base + (hf == 0 ? C::COL_Q : C::COL_DO));
        tmem_wait_st();
      }
      tc_fence_before();
      mbar_arrive(b_qt);
    }
    // Dropout keep bits of this row's 64 keys of a key tile: bit q set iff
    // key 64*hf + q of the tile is kept.  In the keep mask they are bytes
    // 8*hf .. 8*hf + 7 of the row's entry for the tile, loaded a tile ahead
    // (mnext) so their latency overlaps a whole tile.
    const bool mrow = DROP == kDropRead && qrow < Nq;
    const unsigned long long* mptr =
        mrow ? reinterpret_cast<const unsigned long long*>(
                   a.drop.mask + mask_entry(a.drop, a.g, sv, h, 0, qrow) + 8 * hf)
             : nullptr;
    const int64_t mstep = a.g.rows_q * 2;            // one key tile, in 8-byte words
    unsigned long long mnext = (mrow && n > 0) ? __ldg(mptr) : 0ull;
    for (int jt = 0; ok && jt < n; ++jt) {
      // keep bits drawn before the scores arrive (positions only), or the
      // prefetched mask word taken and the next tile's issued
      uint64_t keep = 0;
      if constexpr (DROP) {
        static_assert(C::BT == 128, "keep-mask entries cover 128-key tiles");
        if constexpr (DROP == kDropRead) {
          keep = mnext;
          if (mrow && jt + 1 < n) mnext = __ldg(mptr + (jt + 1) * mstep);
        } else {
          const int64_t kbase = static_cast<int64_t>(jt) * C::BT + 64 * hf;
#pragma unroll
          for (int t = 0; t < 8; ++t)
            keep |= static_cast<uint64_t>(keep8(a.drop, static_cast<uint32_t>((kbase >> 3) + t),
                                                static_cast<uint32_t>(qrow),
                                                static_cast<uint32_t>(bh)))
                    << (8 * t);
        }
      }
      if (!(ok = wait_warp(b_sfull, jt & 1, ctl, a.status, a.timeout_ns))) break;
      tc_fence_after();
      float p[64];
      tmem_ld64(lane_base + C::COL_S + 64 * hf, p);
      tc_fence_before();
      mbar_arrive(b_sfree);                  // S may be overwritten by the next tile
      // keys past N (last tile) and keys after the query (diagonal tile)
      int lim = 63;
      if (a.causal && jt == qt) lim = row - 64 * hf;
      if (jt == nk - 1) lim = min(lim, static_cast<int>(Nk - 1 - static_cast<int64_t>(jt) * C::BT) - 64 * hf);
      {
        // P = exp2(c * S - L * log2(e)), two keys per paired instruction
        const uint64_t cc = f32x2(c, c), nl = f32x2(-l2, -l2);
#pragma unroll
        for (int q = 0; q < 64; q += 2) {
          float x0, x1;
          f32x2_split(fma_f32x2(f32x2(p[q], p[q + 1]), cc, nl), x0, x1);
          p[q] = ex2(x0);
          p[q + 1] = ex2(x1);
        }
      }
      if (lim < 63) {
#pragma unroll
        for (int q = 0; q < 64; ++q)
          if (q > lim) p[q] = 0.f;
      }
      if (!(ok = wait_warp(b_dpfull, jt & 1, ctl, a.status, a.timeout_ns))) break;
      tc_fence_after();
      if constexpr (DROP) {
        // dS = P o (Z o dP - Delta), Z = keep / (1 - p): dP / (1 - p) - Delta
        // for kept weights, -Delta for dropped ones, two keys per paired
        // instruction.  In two halves of 32 keys, so that only 32 of dP are
        // held next to P: half 0's rounded dS lands on columns whose dP was
        // read first, half 1's on half 0's.
        const uint64_t rs2 = f32x2(a.drop.rscale, a.drop.rscale), nd = f32x2(-dl, -dl);
        const uint32_t kl = static_cast<uint32_t>(keep), kh = static_cast<uint32_t>(keep >> 32);
        const uint32_t tdp = lane_base + C::COL_DP + 64 * hf;
#pragma unroll
        for (int hq = 0; hq < 2; ++hq) {
          uint32_t r[32];
          tmem_ld32(tdp + 32 * hq, r);
          tmem_wait_ld();
          reg_fence32(r);
          uint32_t w[16];
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const int q = 32 * hq + j;
            float x0, x1;
            f32x2_split(fma_f32x2(f32x2(__uint_as_float(r[j]), __uint_as_float(r[j + 1])), rs2, nd),
                        x0, x1);
            x0 = kept64(kl, kh, q) ? x0 : -dl;
            x1 = kept64(kl, kh, q + 1) ? x1 : -dl;
            f32x2_split(mul_f32x2(f32x2(x0, x1), f32x2(p[q], p[q + 1])), x0, x1);
            w[j / 2] = pack2<T>(x0, x1);
          }
          tmem_st16(tdp + 16 * hq, w);
        }
      } else {
        float dp[64];
        tmem_ld64(lane_base + C::COL_DP + 64 * hf, dp);
        // dS = P o (dP - Delta), two keys per paired instruction
        const uint64_t nd = f32x2(-dl, -dl);
#pragma unroll
        for (int q = 0; q < 64; q += 2) {
          const uint64_t x = mul_f32x2(add_f32x2(f32x2(dp[q], dp[q + 1]), nd), f32x2(p[q], p[q + 1]));
          f32x2_split(x, dp[q], dp[q + 1]);
        }
        tmem_st_packed64<T>(lane_base + C::COL_DP + 64 * hf, dp);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(b_dsready0);
    }
    if (ok) ok = wait_warp(b_accdone, 0, ctl, a.status, a.timeout_ns);
    // Each warpgroup stages half the columns of its rows in shared memory (the
    // K | V stages are idle once every product has completed) as the loads
    // lay them out; then the 256 threads store the tile with consecutive
    // threads on consecutive 16 bytes of a row (whole lines per warp store).
    // Rows past the sequence and columns past a narrow head dimension are not
    // written.  Every elementwise thread passes the barrier, also after a
    // timeout; the stores go out only if all of them got this far.
    const uint32_t stg = smem_u32(sStage);
    if (ok) {
      tc_fence_after();
      stage_row_sw128<T>(lane_base + C::COL_DQ + (D / 2) * hf, a.scale, stg, row, (D / 2) * hf, D / 2);
    }
    if (bar_red_and(1, 256, ok)) {
      T* row0 = static_cast<T*>(a.out0) + bb * a.s0[0] + hq * a.s0[1] + (sv.q0 + qt * C::BT) * a.s0[2];
      store_staged_tile<T>(stg, D, threadIdx.x, 256, row0, a.s0[2],
                           static_cast<int>(Nq - qt * C::BT < C::BT ? Nq - qt * C::BT : C::BT), a.dreal);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// Longest sequence (query and key rows) for which the D <= 64 backward runs
// the persistent dK/dV kernel.
constexpr int64_t kPersistMaxN = 1024;
// Sequences at most this long run the dQ kernel concurrently with the dK/dV
// kernel (see run_bwd_tc).
constexpr int64_t kConcurrentMaxN = 4096;

// Joins the side stream back into the caller's stream on every return path.
struct SideJoin {
  cudaStream_t caller;
  bool on = false;
  ~SideJoin() {
    if (on) side_end(caller);
  }
  fa_status end() {
    on = false;
    return side_end(caller);
  }
};

template <typename T, int D, int DROP>
fa_status run_bwd_tc(const BwdParams& p, cudaStream_t stream) {
  const Geo& g = p.g;
  // Tensor maps carry the true head dimension (zero fill past it).
  CUtensorMap mq, mk, mv, mdo;
  if (!encode_tile_map(&mq, p.q, p.dtype, g.Bt, g.Hq, g.rows_q, p.D, p.sq, 128, 64) ||
      !encode_tile_map(&mk, p.k, p.dtype, g.Bt, g.Hkv, g.rows_k, p.D, p.sk, 128, 64) ||
      !encode_tile_map(&mv, p.v, p.dtype, g.Bt, g.Hkv, g.rows_k, p.D, p.sv, 128, 64) ||
      !encode_tile_map(&mdo, p.dout, p.dtype, g.Bt, g.Hq, g.rows_q, p.D, p.sdo, 128, 64))
    return FA_ERR_LAUNCH;
  BwdTcArgs a{};
  a.dreal = static_cast<int>(p.D);
  a.lse = p.lse; a.delta = p.delta;
  a.g = g;
  a.causal = p.causal;
  a.c = p.scale * kLog2e;
  a.scale = p.scale;
  a.drop = p.drop;
  a.status = p.status;
  a.timeout_ns = p.timeout_ns;

  // dK / dV: one CTA per (b, key/value head, key tile); with few key/value
  // heads (grouped or multi-query attention) a cluster of `split` CTAs
  // shares each key tile's query heads, so the grid fills the SMs and the
  // heaviest key tiles no longer run alone.
  a.BH = g.B * g.Hkv; a.ntiles = (g.Nk + 127) / 128;
  const int64_t esz = p.dtype == FA_F32 ? 4 : 2;
  // Q and dO of a key/value head's G query heads: the operand all its CTAs read
  a.hgroup = head_group(a.BH, 2 * g.Nq * p.D * esz * g.G);
  const int64_t base1 = a.BH * a.ntiles;
  int split = 1;
  while (split < 8 && g.G % (2 * split) == 0 && base1 * split < 2 * device_sm_count()) split *= 2;
  a.split = split;
  const int64_t blocks1 = base1 * split;
  if (blocks1 > 0x7fffffffLL) return FA_ERR_SHAPE;
  a.out0 = p.dv; a.out1 = p.dk;
  for (int i = 0; i < 4; ++i) { a.s0[i] = p.sdv[i]; a.s1[i] = p.sdk[i]; }
  // Short sequences (a few steps per key tile) at D <= 64 without dropout:
  // Short sequences: the dQ kernel, which shares only inputs with the dK/dV
  // kernel, runs on the device's side stream at the same time, so each fills
  // SMs that the other's small grid and tail leave idle (N = 512: backward
  // 169 -> 155 us).  Longer sequences keep them in sequence: their grids fill
  // the GPU, and each kernel's launch duration stays its own.  Never while
  // the caller's stream is being captured into a graph (the shared side
  // stream would join that capture).
  const bool concurrent = p.allow_side && g.Nq <= kConcurrentMaxN && g.Nk <= kConcurrentMaxN &&
                          !stream_capturing(stream);
  SideJoin join{stream};
  cudaStream_t s2 = stream;
  if (concurrent) {
    const fa_status st = side_begin(stream, &s2);
    if (st != FA_OK) return st;
    join.on = true;
  }
  // the persistent kernel, one CTA per SM walking the key tiles, hides each
  // tile's set-up, first loads and epilogue behind its neighbours'.
  bool persist = false;
  if constexpr (D == 64 && DROP == kDropNone)
    persist = split == 1 && g.Nq <= kPersistMaxN && g.Nk <= kPersistMaxN;
  auto k1 = bwd_dkdv_tc_kernel<T, D, DROP>;
  if (persist) {
    auto kp = bwd_dkdv_persist_kernel<T>;
    if (cudaFuncSetAttribute(kp, cudaFuncAttributeMaxDynamicSharedMemorySize, DkdvPCfg::SMEM) !=
        cudaSuccess)
      return FA_ERR_LAUNCH;
    const int64_t sms = device_sm_count();
    const int64_t grid = base1 < sms ? base1 : sms;
    prof_record(p, 0, stream);
    kp<<<dim3(static_cast<unsigned>(grid)), dim3(DkdvCfg<D>::THREADS), DkdvPCfg::SMEM, stream>>>(
        mq, mk, mv, mdo, a);
  } else {
    if (cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, DkdvCfg<D>::SMEM) !=
        cudaSuccess)
      return FA_ERR_LAUNCH;
    prof_record(p, 0, stream);
  }
  if (persist) {
    // launched above
  } else if (split == 1) {
    k1<<<dim3(static_cast<unsigned>(blocks1)), dim3(DkdvCfg<D>::THREADS), DkdvCfg<D>::SMEM,
         stream>>>(mq, mk, mv, mdo, a);
  } else {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks1));
    cfg.blockDim = dim3(DkdvCfg<D>::THREADS);
    cfg.dynamicSmemBytes = DkdvCfg<D>::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(split);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, k1, mq, mk, mv, mdo, a) != cudaSuccess) return FA_ERR_LAUNCH;
  }
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_LAUNCH;
  prof_record(p, 1, stream);

  // dQ: one CTA per (b, query head, query tile)
  a.split = 1;
  a.BH = g.B * g.Hq; a.ntiles = (g.Nq + 127) / 128;
  // K and V of a query head's key/value head: the operand all its CTAs read
  a.hgroup = head_group(a.BH, 2 * g.Nk * p.D * esz);
  const int64_t blocks2 = a.BH * a.ntiles;
  if (blocks2 > 0x7fffffffLL) return FA_ERR_SHAPE;
  a.out0 = p.dq; a.out1 = nullptr;
  for (int i = 0; i < 4; ++i) { a.s0[i] = p.sdq[i]; a.s1[i] = 0; }
  auto k2 = bwd_dq_tc_kernel<T, D, DROP>;
  if (cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, DqCfg<D>::SMEM) != cudaSuccess)
    return FA_ERR_LAUNCH;
  k2<<<dim3(static_cast<unsigned>(blocks2)), dim3(DqCfg<D>::THREADS), DqCfg<D>::SMEM, s2>>>(
      mq, mk, mv, mdo, a);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_LAUNCH;
  if (concurrent) {
    const fa_status st = join.end();
    if (st != FA_OK) return st;
  }
  prof_record(p, 2, stream);
  return FA_OK;
}

template <typename T, int D>
fa_status run_bwd_tc_any(const BwdParams& p, cudaStream_t s) {
  const int dm = bwd_drop_mode(p.drop);
  return dm == kDropRead ? run_bwd_tc<T, D, kDropRead>(p, s)
         : dm == kDropDraw ? run_bwd_tc<T, D, kDropDraw>(p, s) : run_bwd_tc<T, D, kDropNone>(p, s);
}

}  // namespace

// D = 16 and 32 run through the D = 64 kernels, zero-padded by the TMA loads.
bool have_bwd_tc(int64_t D, fa_dtype dt) {
  return (D == 16 || D == 32 || D == 64 || D == 128) && dt != FA_F32;
}

fa_status launch_bwd_tc(const BwdParams& p, cudaStream_t s) {
  if (p.dtype == FA_BF16) {
    if (p.D == 128) return run_bwd_tc_any<__nv_bfloat16, 128>(p, s);
    if (p.D <= 64) return run_bwd_tc_any<__nv_bfloat16, 64>(p, s);
  } else if (p.dtype == FA_F16) {
    if (p.D == 128) return run_bwd_tc_any<__half, 128>(p, s);
    if (p.D <= 64) return run_bwd_tc_any<__half, 64>(p, s);
  }
  return FA_ERR_ARG;
}

}  // namespace fa
