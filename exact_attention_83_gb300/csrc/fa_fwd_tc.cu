// Tensor-core forward: TMA + tcgen05 + TMEM, warp-specialised, for fp16/bf16
// with D in {64, 128} (16 and 32 run through D = 64 with the head dimension
// zero-filled by the TMA loads).  D = 128 uses fwd_tc_kernel below (two query
// tiles per CTA); D <= 64 uses fwd_tc_1t_kernel further down (one query tile
// per CTA, two CTAs per SM).  Both handle the general geometry of fa_internal.h
// (sequence views, grouped key/value heads) and, as a template flag, dropout.
//
// Algorithm ("FlashAttention-2 from PyTorch to Triton", the running quantities
// m, l, O and the store of L = m + log l; "Triton FlashAttention", the online
// softmax in fp32 with exp2 on scores pre-scaled by log2(e), the accumulator
// rescaled when the max moves, and causal key tiles above the diagonal never
// visited): for each 128-row query tile, loop over 128-key tiles,
//   S = Q K_j^T (tensor cores, fp32 in TMEM),
//   mask keys past the sequence (last tile) and keys after the query
//   (diagonal tile only),
//   m_new = max(m, c * rowmax S) with c = scale * log2(e),
//   P = exp2(c * S - m) rounded to the input type (FIX 1 of the Triton page),
//   l += rowsum P,  O += P V_j (tensor cores, fp32 in TMEM),
// then O / l and L = (m + log2 l) * ln 2.
//
// Lazy rescale: the running max used in the exponent is only moved when the
// row max grows by more than 8 (a factor 2^8 in P); then O (in TMEM) and l
// are multiplied by exp2(m_old - m_new).  Otherwise P is computed against the
// stale max and stays <= 2^8.  The result is the same: numerator and
// denominator share the one max used for that row, and the final division
// cancels it.
//
// fwd_tc_kernel: CTA = two query tiles (256 rows) of one head sharing every
// K/V tile load.
// Warps 0-3: softmax + epilogue of query tile 0 (one TMEM lane = one row per
// thread); warps 4-7: the same for query tile 1; warp 8: TMA producer (lane 0)
// and TMEM allocation; warp 9: MMA issuer (the whole warp runs the issue loop,
// one elected lane issues).  TMEM columns: S0 [0,128),
// S1 [128,256), O0 [256,256+D), O1 [256+D,256+2D); P (input type, packed two
// per column) overwrites the first 64 columns of its S after S is read.
// The MMA issue order S0_0, S1_0, {PV0_j, S0_j+1, PV1_j, S1_j+1} lets one
// tile's softmax overlap the other tile's two MMAs.  A tcgen05.commit tracks
// every earlier MMA of the issuing thread, so when the softmax warps see S_j
// complete, PV_{j-1} of the same tile is complete too and O may be rescaled.
//
// Dropout (FlashAttention-2's dropout of P, decisions from Philox positions):
// each softmax thread evaluates the generator for its row of the next key
// tile before the scores arrive and, when the caller gave a keep mask, stores
// the 16 bytes there for the backward.  P V takes P o keep; the 1 / (1 - p)
// of Z is folded into the final 1 / l.
//
// Every mbarrier wait is bounded (see tc_common.cuh); a wait that runs out
// records FA_ERR_TIMEOUT, the CTA drains its copies and MMAs in flight,
// releases its tensor memory and exits.

#include "tc_common.cuh"

namespace fa {
namespace {

using namespace tc;

template <int D>
struct FwdCfg {
  static constexpr int BM = 128;                  // query rows per tile
  static constexpr int BN = 128;                  // keys per tile
  static constexpr int DC = D / 64;               // 128-byte column chunks per row
  static constexpr int CHUNK = BM * 128;          // bytes of one 128-row chunk
  static constexpr int TILE = DC * CHUNK;         // bytes of one 128 x D tile
  static constexpr int NS = D == 128 ? 4 : 8;     // K/V ring tiles
  static constexpr int NP = NS / 2;               // ring slots of a V tile + a K tile
  static constexpr int PAIR = 2 * TILE;
  static constexpr int OFF_RING = 2 * TILE;
  static constexpr int OFF_BAR = OFF_RING + NS * TILE;
  static constexpr int SMEM = OFF_BAR + 1024 + 1024;   // + barriers, + alignment slack
  static constexpr int THREADS = 320;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_S0 = 0, COL_O0 = 256;
};

// Ring position of each K / V tile when tiles are loaded in consumption order
// K_0, K_1, V_0, K_2, V_1, ...: K_j at 2j - 1 (K_0 at 0), V_j at 2j + 2.
__device__ __forceinline__ int unit_k(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int unit_v(int j) { return 2 * j + 2; }

struct FwdTcArgs {
  void* o;
  float* lse;
  Geo g;
  int64_t BH, npairs;      // B * Hq; query-tile pairs of the longest sequence
  int64_t hgroup;          // heads per group of the block order
  int dreal;               // head dimension stored (<= D; narrower ones run zero-padded)
  int64_t so[4];
  int causal;
  float c;                 // scale * log2(e)
  Dropout drop;
  unsigned int* status;
  uint64_t timeout_ns;
  int withhold_arrival;    // test-only: CTA 0 skips the first S-ready arrival of tile 0
};

template <typename T, int D, int DROP>
__global__ void __launch_bounds__(320, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv, const FwdTcArgs a) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sRing = smem + C::OFF_RING;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  Ctl* ctl = reinterpret_cast<Ctl*>(bars + 40);
  // barrier map
  const uint32_t b_q = smem_u32(&bars[0]);
  const uint32_t b_full0 = smem_u32(&bars[1]);            // + 8 * slot
  const uint32_t b_empty0 = smem_u32(&bars[1 + C::NS]);   // + 8 * slot
  const uint32_t b_sfull0 = smem_u32(&bars[1 + 2 * C::NS]);      // + 8 * g
  const uint32_t b_pready0 = smem_u32(&bars[3 + 2 * C::NS]);     // + 8 * (2 * g + half)
  const uint32_t b_ofinal0 = smem_u32(&bars[7 + 2 * C::NS]);     // + 8 * g
  const uint32_t b_mmadone = smem_u32(&bars[9 + 2 * C::NS]);
  static_assert(10 + 2 * C::NS <= 40, "barriers below the control block");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t id = blockIdx.x;
  // Grouped order (grouped_tile): the CTAs in flight belong to a few heads,
  // whose K and V tiles stay in L2; the longest query-tile pairs first.
  int64_t bh, t;                                // b * Hq + h
  grouped_tile(id, a.BH, a.npairs, a.hgroup, bh, t);
  const int64_t pr = a.causal ? (a.npairs - 1 - t) : t;
  const int64_t h = bh % a.g.Hq;
  const SeqView sv = seq_view(a.g, bh / a.g.Hq);
  if (!sv.ok) {
    if (threadIdx.x == 0) record_status(a.status, FA_ERR_SEQLENS);
    return;
  }
  const int64_t Nq = sv.nq, Nk = sv.nk;
  if (2 * pr * C::BM >= Nq) return;             // both query tiles lie past this sequence
  const int32_t hq = static_cast<int32_t>(h), hk = static_cast<int32_t>(h / a.g.G);
  const int32_t bb = static_cast<int32_t>(sv.b);
  const int nk = static_cast<int>((Nk + C::BN - 1) / C::BN);
  int ntile[2];
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    const int64_t qt = 2 * pr + g;
    const int64_t diag = qt + 1;   // key tiles up to and including the diagonal
    ntile[g] = (qt * C::BM >= Nq) ? 0 : (a.causal ? static_cast<int>(diag < nk ? diag : nk) : nk);
  }
  const int nmax = max(ntile[0], ntile[1]);
  if (nmax == 0) {
    // No key at all (an empty key sequence): O = 0 and L = -inf.
    if (warp < 8) {
      const int64_t qrow = (2 * pr + (warp >> 2)) * C::BM + (warp & 3) * 32 + lane;
      if (qrow < Nq) {
        T* orow = static_cast<T*>(a.o) + bb * a.so[0] + hq * a.so[1] + (sv.q0 + qrow) * a.so[2];
        for (int d = 0; d < a.dreal; ++d) orow[d] = Elem<T>::from_f32(0.f);
        a.lse[lse_index(a.g, sv, h, qrow)] = -INFINITY;
      }
    }
    return;
  }

  // K | V ring units in consumption order, one per step: unit 0 = K_0 (the
  // first score products), unit u >= 1 = V_{u-1} and K_u (step u - 1's P V
  // and next score products; no K_u at u = nmax), in slot u % NP with V in
  // the slot's first tile and K in its second.  The MMA thread stays only a
  // product or two ahead of the tensor pipe, so each wait or commit it makes
  // between products can leave the pipe idle: with one unit per step it
  // waits once and commits once per step for the ring.  The
  // producer's lane 0 sets up the barriers and sends Q and the ring's first
  // round of units before the block-wide sync, so their latency overlaps the
  // set-up.
  uint32_t issued[C::NP];   // producer lane 0: rounds issued per ring slot
#pragma unroll
  for (int s = 0; s < C::NP; ++s) issued[s] = 0;
  auto issue_unit = [&](int u) {
    const int s = u % C::NP;
    const bool hasV = u > 0, hasK = u < nmax;
    mbar_arrive_expect_tx(b_full0 + 8 * s, (hasV ? C::TILE : 0) + (hasK ? C::TILE : 0));
    for (int c = 0; c < C::DC; ++c) {
      if (hasV)
        tma_load_4d(smem_u32(sRing + s * C::PAIR + c * C::CHUNK), &tmv, b_full0 + 8 * s, c * 64,
                    static_cast<int32_t>(sv.k0 + (u - 1) * C::BN), hk, bb);
      if (hasK)
        tma_load_4d(smem_u32(sRing + s * C::PAIR + C::TILE + c * C::CHUNK), &tmk, b_full0 + 8 * s,
                    c * 64, static_cast<int32_t>(sv.k0 + u * C::BN), hk, bb);
    }
    issued[s] = static_cast<uint32_t>(u / C::NP) + 1;
  };
  const int nunits = nmax + 1;
  const int u_early = nunits < C::NP ? nunits : C::NP;   // round 0 of the ring
  if (warp == 8) {
    if (lane == 0) {
      mbar_init(b_q, 1);
      for (int s = 0; s < C::NP; ++s) {
        mbar_init(b_full0 + 8 * s, 1);
        mbar_init(b_empty0 + 8 * s, 1);
      }
      for (int g = 0; g < 2; ++g) {
        mbar_init(b_sfull0 + 8 * g, 1);
        mbar_init(b_pready0 + 8 * (2 * g), 128);
        mbar_init(b_pready0 + 8 * (2 * g + 1), 128);
        mbar_init(b_ofinal0 + 8 * g, 1);
      }
      mbar_init(b_mmadone, 1);
      ctl->abort = 0;
      mbar_fence_init();
      tma_prefetch_desc(&tmq);
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
      const uint32_t qbytes = (ntile[0] > 0 ? C::TILE : 0) + (ntile[1] > 0 ? C::TILE : 0);
      mbar_arrive_expect_tx(b_q, qbytes);
      for (int g = 0; g < 2; ++g) {
        if (ntile[g] == 0) continue;
        for (int c = 0; c < C::DC; ++c)
          tma_load_4d(smem_u32(sQ + g * C::TILE + c * C::CHUNK), &tmq, b_q, c * 64,
                      static_cast<int32_t>(sv.q0 + (2 * pr + g) * C::BM), hq, bb);
      }
      for (int u = 0; u < u_early; ++u) issue_unit(u);
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
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      bool ok = true;
      for (int u = u_early; ok && u < nunits; ++u) {
        const int s = u % C::NP;
        const uint32_t r = static_cast<uint32_t>(u / C::NP);
        if (r > 0 && !(ok = wait_bounded(b_empty0 + 8 * s, (r - 1) & 1, ctl, a.status,
                                         a.timeout_ns)))
          break;
        issue_unit(u);
      }
      // Drain: every copy issued has landed before the CTA may exit.
      wait_bounded(b_q, 0, ctl, a.status, a.timeout_ns, false);
      for (int s = 0; s < C::NP; ++s)
        if (issued[s]) wait_bounded(b_full0 + 8 * s, (issued[s] - 1) & 1, ctl, a.status,
                                    a.timeout_ns, false);
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the issue loop and its waits, so the loop control
    // and descriptor arithmetic are warp-uniform; one elected lane issues
    // the products and commits.  (With the loop inside a one-lane branch the
    // same code issued products more slowly than the tensor pipe ran them.)
    {
      const bool leader = elect_one();
      const uint32_t idS = idesc_f16<T>(128, C::BN, false, false);
      const uint32_t idO = idesc_f16<T>(128, D, false, true);
      // Descriptors are built once and advanced by adding (byte offset >> 4)
      // to the start-address field (addresses stay below 256 KiB, so the
      // 14-bit field never carries).
      const uint64_t dQ0 = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dK0 = sdesc_sw128(smem_u32(sRing + C::TILE), 16, 1024);
      const uint64_t dV0 = sdesc_sw128(smem_u32(sRing), C::CHUNK, 1024);
      auto issue_S = [&](int g, int slot) {
        const uint64_t qa = dQ0 + static_cast<uint64_t>((g * C::TILE) >> 4);
        const uint64_t kb = dK0 + static_cast<uint64_t>((slot * C::PAIR) >> 4);
        const uint32_t d = tmem + C::COL_S0 + 128 * g;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::CHUNK + (kk & 3) * 32) >> 4;
          if (leader) mma_ss(d, qa + off, kb + off, idS, kk > 0 ? 1u : 0u);
        }
      };
      // O_g += P V over keys 64h .. 64h+63 (P columns 32h .. 32h+31)
      auto issue_PV_half = [&](int g, int slot, int hh, bool acc) {
        const uint64_t vb = dV0 + static_cast<uint64_t>((slot * C::PAIR) >> 4);
        const uint32_t d = tmem + C::COL_O0 + D * g, p = tmem + C::COL_S0 + 128 * g;
#pragma unroll
        for (int k4 = 0; k4 < C::BN / 32; ++k4) {
          const int kk = 4 * hh + k4;
          if (leader) mma_ts(d, p + kk * 8, vb + static_cast<uint64_t>((kk * 2048) >> 4), idO,
                 (acc || kk > 0) ? 1u : 0u);
        }
      };
      bool ok = wait_warp(b_q, 0, ctl, a.status, a.timeout_ns) &&
                wait_warp(b_full0, 0, ctl, a.status, a.timeout_ns);
      if (ok) {
        tc_fence_after();
        for (int g = 0; g < 2; ++g)
          if (ntile[g] > 0) {
            issue_S(g, 0);
            // A test can withhold this arrival in CTA 0 to make the softmax
            // warps' bounded wait run out (the timeout path, without a fault).
            if (leader && !(a.withhold_arrival && blockIdx.x == 0 && g == 0))
              mma_commit(b_sfull0 + 8 * g);
          }
        if (leader) mma_commit(b_empty0);
      }
      for (int j = 0; ok && j < nmax; ++j) {
        // unit j + 1: V_j for this step's P V, K_{j+1} for its score products
        const int u = j + 1, su = u % C::NP;
        // (the fence after each P-ready wait below orders the products after
        // this wait too)
        ok = wait_warp(b_full0 + 8 * su, (u / C::NP) & 1, ctl, a.status, a.timeout_ns);
        if (!ok) break;
        for (int g = 0; g < 2 && ok; ++g) {
          if (j >= ntile[g]) continue;
          // P V once the softmax warps have written all of P
          if (!(ok = wait_warp(b_pready0 + 8 * (2 * g), j & 1, ctl, a.status, a.timeout_ns)))
            break;
          tc_fence_after();
          issue_PV_half(g, su, 0, j > 0);
          issue_PV_half(g, su, 1, true);
          if (j + 1 < ntile[g]) {
            issue_S(g, su);
            if (leader) mma_commit(b_sfull0 + 8 * g);
          } else {
            if (leader) mma_commit(b_ofinal0 + 8 * g);
          }
        }
        if (!ok) break;
        if (leader) mma_commit(b_empty0 + 8 * su);
      }
      // Drain: every MMA (and every commit arrival) of this thread is complete.
      if (leader) mma_commit(b_mmadone);
      wait_bounded(b_mmadone, 0, ctl, a.status, a.timeout_ns, false);
    }
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax + epilogue
    const int g = warp >> 2, quarter = warp & 3;
    const int r = quarter * 32 + lane;                       // row in the query tile
    const int64_t qt = 2 * pr + g;
    const int64_t qrow = qt * C::BM + r;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t tS = lane_base + C::COL_S0 + 128 * g;
    const uint32_t tO = lane_base + C::COL_O0 + D * g;
    const float c = a.c;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    const int n = ntile[g];
    // last valid key column of the last key tile
    const int lim_last = static_cast<int>(Nk - 1 - static_cast<int64_t>(nk - 1) * C::BN);
    // keep bits of this row, stored into the caller's keep mask (16 bytes
    // per key tile, tiles rows_q entries apart) for the backward
    uint4* mrow = nullptr;
    if (DROP && a.drop.mask != nullptr && qrow < Nq)
      mrow = reinterpret_cast<uint4*>(a.drop.mask + mask_entry(a.drop, a.g, sv, h, 0, qrow));
    for (int j = 0; j < n; ++j) {
      // Dropout keep bits of this row's 128 keys, drawn before the scores
      // arrive (positions only): bit k of kb[k / 32] is key j*128 + k.
      uint32_t kb[4] = {0u, 0u, 0u, 0u};
      if constexpr (DROP) {
        tile_keep_bits(a.drop, bh, j, qrow, kb);
        if (mrow) mrow[j * a.g.rows_q] = make_uint4(kb[0], kb[1], kb[2], kb[3]);
      }
      if (!(ok = wait_warp(b_sfull0 + 8 * g, j & 1, ctl, a.status, a.timeout_ns))) break;
      tc_fence_after();
      float s[128];
      {
        uint32_t r0[32], r1[32], r2[32], r3[32];
        tmem_ld32(tS + 0, r0);
        tmem_ld32(tS + 32, r1);
        tmem_ld32(tS + 64, r2);
        tmem_ld32(tS + 96, r3);
        tmem_wait_ld();
        reg_fence32(r0); reg_fence32(r1); reg_fence32(r2); reg_fence32(r3);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          s[i] = __uint_as_float(r0[i]);
          s[32 + i] = __uint_as_float(r1[i]);
          s[64 + i] = __uint_as_float(r2[i]);
          s[96 + i] = __uint_as_float(r3[i]);
        }
      }
      // Exclude keys past N (last key tile) and keys after the query (the
      // diagonal tile, the only one a causal row can straddle).
      int lim = C::BN - 1;
      if (a.causal && j == qt) lim = r;
      if (j == nk - 1) lim = min(lim, lim_last);
      if (lim < C::BN - 1) {
#pragma unroll
        for (int kk = 0; kk < C::BN; ++kk)
          if (kk > lim) s[kk] = -INFINITY;
      }
      // Running max: four independent three-input max chains over the scores.
      bool rescale = false;
      float alpha = 1.f;
      {
        float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
        for (int kk = 0; kk < C::BN; kk += 8) {
          m0 = max3f(m0, s[kk], s[kk + 1]);
          m1 = max3f(m1, s[kk + 2], s[kk + 3]);
          m2 = max3f(m2, s[kk + 4], s[kk + 5]);
          m3 = max3f(m3, s[kk + 6], s[kk + 7]);
        }
        const float m_new = fmaxf(m, fmaxf(fmaxf(m0, m1), fmaxf(m2, m3)) * c);
        // Lazy rescale decision (warp-uniform for the TMEM access below).
        if (j == 0) {
          m = m_new;
        } else {
          const bool need = m_new > m + 8.f;
          rescale = __any_sync(0xffffffffu, need);
          if (need) {
            alpha = ex2(m - m_new);
            l *= alpha;
            m = m_new;
          }
        }
      }
      const uint64_t cc = f32x2(c, c), nm = f32x2(-m, -m);
      // P in two halves of 64 keys; each half is released to the MMA thread as
      // soon as it is in tensor memory, so P V on the first half overlaps the
      // exponentials of the second.  Paired fp32 instructions form c * s - m
      // and the row sum two keys at a time.
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t pk[32];
        uint64_t acc = f32x2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float x0, x1;
          f32x2_split(fma_f32x2(f32x2(s[64 * hh + 2 * i], s[64 * hh + 2 * i + 1]), cc, nm), x0, x1);
          const float p0 = ex2(x0), p1 = ex2(x1);
          acc = add_f32x2(acc, f32x2(p0, p1));
          if constexpr (DROP) {
            // l sums the undropped weights; P V takes the kept ones (the
            // 1 / (1 - p) of Z is applied with 1 / l at the end)
            // keys kk, kk + 1 are bits b, b + 1 of byte kk / 8 % 4 of their
            // word (b = kk % 8): shifted by 7 - b and 6 - b they are that
            // byte's sign bits, which one prmt spreads over the pair's halves
            const int kk = 64 * hh + 2 * i, byte = (kk >> 3) & 3, b = kk & 7;
            const uint32_t wk = kb[kk >> 5];
            pk[i] = pack2<T>(p0, p1) & prmt(wk << (7 - b), wk << (6 - b), half_sign_sel(byte, 4 + byte));
          } else {
            pk[i] = pack2<T>(p0, p1);
          }
        }
        tmem_st32(tS + 32 * hh, pk);
        if (hh == 0 && rescale) {
          // O *= alpha before any of P_j is released (P_j V is issued only
          // after the arrivals, and P_{j-1} V completed before S_j did); the
          // first half's scores are dead by now, which keeps registers free
#pragma unroll 1
          for (int cc4 = 0; cc4 < D / 16; ++cc4) {
            uint32_t t[16];
            tmem_ld16(tO + 16 * cc4, t);
            tmem_wait_ld();
            reg_fence16(t);
#pragma unroll
            for (int i = 0; i < 16; ++i) t[i] = __float_as_uint(__uint_as_float(t[i]) * alpha);
            tmem_st16(tO + 16 * cc4, t);
          }
        }
        if (hh == 1) {
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(b_pready0 + 8 * (2 * g));
        }
        float lo, hi;
        f32x2_split(acc, lo, hi);
        l += lo + hi;
      }
      if (!ok) break;
    }
    if (ok && n > 0) ok = wait_warp(b_ofinal0 + 8 * g, 0, ctl, a.status, a.timeout_ns);
    // O / l staged in shared memory over this tile's Q (no product reads it
    // once the tile's last P V, committed after its last S, has completed;
    // the other tile's products may still be using the K | V ring) and
    // stored by the tile's four warps with consecutive threads on
    // consecutive 16 bytes of a row (whole lines per warp store); rows past
    // the sequence are not written.  Every thread of the tile's warpgroup
    // passes the barrier, also after a timeout; the stores go out only if
    // all of them got this far.
    if (n > 0) {
      const uint32_t stg = smem_u32(sQ) + static_cast<uint32_t>(g * C::TILE);
      if (ok) {
        tc_fence_after();
        const float inv = (DROP ? a.drop.rscale : 1.f) / l;   // Z's 1 / (1 - p) with dropout
        stage_row_sw128<T>(tO, inv, stg, r, 0, D);
        if (qrow < Nq) a.lse[lse_index(a.g, sv, h, qrow)] = (m + log2f(l)) * kLn2;
      }
      if (bar_red_and(1 + g, 128, ok)) {
        T* row0 = static_cast<T*>(a.o) + bb * a.so[0] + hq * a.so[1] + (sv.q0 + qt * C::BM) * a.so[2];
        store_staged_tile<T>(stg, D, threadIdx.x & 127, 128, row0, a.so[2],
                             static_cast<int>(Nq - qt * C::BM < C::BM ? Nq - qt * C::BM : C::BM),
                             a.dreal);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ============================================================================
// D <= 64: one query tile per CTA, two CTAs per SM
// ============================================================================
// At D = 64 one query tile needs S (128 columns), O (64) and P (64, two
// input-type values per column) of tensor memory: 256 columns, half an SM's,
// and its operands fit in under half the shared memory.  So two CTAs share an
// SM; each one's softmax overlaps the other's products, and a CTA's start-up
// and epilogue overlap the other's main loop.  With P in its own columns the
// softmax warps release S as soon as they have read it: per key tile j the MMA
// issuer runs S_{j+1} (once S_j has been read) and then P_j V_j (once P_j is
// written); the softmax warps write P_{j+1} only after P_j V_j has completed,
// which also makes O stable for a rescale.  K and V tiles share one ring,
// filled in consumption order K_0, K_1, V_0, K_2, V_1, ...
struct Fwd1Cfg {
  static constexpr int D = 64;
  static constexpr int BM = 128, BN = 128;
  static constexpr int TILE = BM * 128;           // one 128 x 64 tile of 16-bit values
  static constexpr int NS = 5;                    // K/V ring slots
  static constexpr int OFF_RING = TILE;
  static constexpr int OFF_BAR = OFF_RING + NS * TILE;
  static constexpr int SMEM = OFF_BAR + 1024 + 1024;
  static constexpr int THREADS = 192;
  static constexpr uint32_t TMEM_COLS = 256;
  static constexpr uint32_t COL_S = 0, COL_O = 128, COL_P = 192;
};

template <typename T, int DROP>
__global__ void __launch_bounds__(192, 2)
    fwd_tc_1t_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv, const FwdTcArgs a) {
  using C = Fwd1Cfg;
  constexpr int D = C::D;
  static_assert(2 * C::SMEM <= 227 * 1024, "two CTAs per SM");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sRing = smem + C::OFF_RING;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  Ctl* ctl = reinterpret_cast<Ctl*>(bars + 40);
  const uint32_t b_q = smem_u32(&bars[0]);
  const uint32_t b_full0 = smem_u32(&bars[1]);                   // + 8 * slot
  const uint32_t b_empty0 = smem_u32(&bars[1 + C::NS]);          // + 8 * slot
  const uint32_t b_sfull = smem_u32(&bars[1 + 2 * C::NS]);       // S ready
  const uint32_t b_sfree = smem_u32(&bars[2 + 2 * C::NS]);       // S read
  const uint32_t b_pready = smem_u32(&bars[3 + 2 * C::NS]);      // P written
  const uint32_t b_pvdone = smem_u32(&bars[4 + 2 * C::NS]);      // P V done
  const uint32_t b_mmadone = smem_u32(&bars[5 + 2 * C::NS]);
  static_assert(6 + 2 * C::NS <= 40, "barriers below the control block");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t id = blockIdx.x;
  int64_t bh, t;                                // b * Hq + h (grouped order, as above)
  grouped_tile(id, a.BH, a.npairs, a.hgroup, bh, t);
  const int64_t qt = a.causal ? (a.npairs - 1 - t) : t;   // query tile
  const int64_t h = bh % a.g.Hq;
  const SeqView sv = seq_view(a.g, bh / a.g.Hq);
  if (!sv.ok) {
    if (threadIdx.x == 0) record_status(a.status, FA_ERR_SEQLENS);
    return;
  }
  const int64_t Nq = sv.nq, Nk = sv.nk;
  if (qt * C::BM >= Nq) return;                 // this query tile lies past the sequence
  const int32_t hq = static_cast<int32_t>(h), hk = static_cast<int32_t>(h / a.g.G);
  const int32_t bb = static_cast<int32_t>(sv.b);
  const int nk = static_cast<int>((Nk + C::BN - 1) / C::BN);
  const int n = a.causal ? min(static_cast<int>(qt) + 1, nk) : nk;   // key tiles to visit
  if (n == 0) {
    // No key at all (an empty key sequence): O = 0 and L = -inf.
    if (warp < 4) {
      const int64_t qrow = qt * C::BM + warp * 32 + lane;
      if (qrow < Nq) {
        T* orow = static_cast<T*>(a.o) + bb * a.so[0] + hq * a.so[1] + (sv.q0 + qrow) * a.so[2];
        for (int d = 0; d < a.dreal; ++d) orow[d] = Elem<T>::from_f32(0.f);
        a.lse[lse_index(a.g, sv, h, qrow)] = -INFINITY;
      }
    }
    return;
  }

  // K | V ring units in consumption order K_0, K_1, V_0, K_2, V_1, ...; unit
  // 2*n - 1 would be K_n (absent).  The producer's lane 0 sets up the
  // barriers and sends Q and the ring's first round of units before the
  // block-wide sync, so their latency overlaps the set-up.
  uint32_t issued[C::NS];   // producer lane 0: rounds issued per ring slot
#pragma unroll
  for (int s = 0; s < C::NS; ++s) issued[s] = 0;
  auto issue_unit = [&](int u) {
    int j, kv;
    if (u == 0) { j = 0; kv = 0; }
    else if (u & 1) { j = (u + 1) / 2; kv = 0; }
    else { j = (u - 2) / 2; kv = 1; }
    if (j >= n) return;
    const int s = u % C::NS;
    mbar_arrive_expect_tx(b_full0 + 8 * s, C::TILE);
    tma_load_4d(smem_u32(sRing + s * C::TILE), kv ? &tmv : &tmk, b_full0 + 8 * s, 0,
                static_cast<int32_t>(sv.k0 + j * C::BN), hk, bb);
    issued[s] = static_cast<uint32_t>(u / C::NS) + 1;
  };
  const int u_early = 2 * n + 1 < C::NS ? 2 * n + 1 : C::NS;   // round 0 of the ring
  if (warp == 4) {
    if (lane == 0) {
      mbar_init(b_q, 1);
      for (int s = 0; s < C::NS; ++s) {
        mbar_init(b_full0 + 8 * s, 1);
        mbar_init(b_empty0 + 8 * s, 1);
      }
      mbar_init(b_sfull, 1);
      mbar_init(b_sfree, 128);
      mbar_init(b_pready, 128);
      mbar_init(b_pvdone, 1);
      mbar_init(b_mmadone, 1);
      ctl->abort = 0;
      mbar_fence_init();
      tma_prefetch_desc(&tmq);
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
      mbar_arrive_expect_tx(b_q, C::TILE);
      tma_load_4d(smem_u32(sQ), &tmq, b_q, 0, static_cast<int32_t>(sv.q0 + qt * C::BM), hq, bb);
      for (int u = 0; u < u_early; ++u) issue_unit(u);
    }
    __syncwarp();
    tmem_alloc(smem_u32(&ctl->tmem_base), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      bool ok = true;
      for (int u = u_early; ok && u <= 2 * n; ++u) {
        const int s = u % C::NS;
        const uint32_t r = static_cast<uint32_t>(u / C::NS);
        if (r > 0 && !(ok = wait_bounded(b_empty0 + 8 * s, (r - 1) & 1, ctl, a.status,
                                         a.timeout_ns)))
          break;
        issue_unit(u);
      }
      // Drain: every copy issued has landed before the CTA may exit.
      wait_bounded(b_q, 0, ctl, a.status, a.timeout_ns, false);
      for (int s = 0; s < C::NS; ++s)
        if (issued[s]) wait_bounded(b_full0 + 8 * s, (issued[s] - 1) & 1, ctl, a.status,
                                    a.timeout_ns, false);
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    {
      const bool leader = elect_one();
      const uint32_t idS = idesc_f16<T>(128, C::BN, false, false);
      const uint32_t idO = idesc_f16<T>(128, D, false, true);
      const uint64_t dQ0 = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dK0 = sdesc_sw128(smem_u32(sRing), 16, 1024);
      const uint64_t dV0 = sdesc_sw128(smem_u32(sRing), C::TILE, 1024);
      auto slot_of = [](int u) { return u % C::NS; };
      auto parity_of = [](int u) { return static_cast<uint32_t>((u / C::NS) & 1); };
      auto issue_S = [&](int slot) {   // S = Q K^T
        const uint64_t kb = dK0 + static_cast<uint64_t>((slot * C::TILE) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          if (leader) mma_ss(tmem + C::COL_S, dQ0 + ((kk * 32) >> 4), kb + ((kk * 32) >> 4), idS,
                 kk > 0 ? 1u : 0u);
      };
      auto issue_PV = [&](int slot, bool acc) {   // O += P V, P from tensor memory
        const uint64_t vb = dV0 + static_cast<uint64_t>((slot * C::TILE) >> 4);
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk)
          if (leader) mma_ts(tmem + C::COL_O, tmem + C::COL_P + 8 * kk,
                 vb + static_cast<uint64_t>((kk * 2048) >> 4), idO, (acc || kk > 0) ? 1u : 0u);
      };
      bool ok = wait_warp(b_q, 0, ctl, a.status, a.timeout_ns) &&
                wait_warp(b_full0 + 8 * slot_of(unit_k(0)), parity_of(unit_k(0)), ctl,
                             a.status, a.timeout_ns);
      if (ok) {
        tc_fence_after();
        issue_S(slot_of(unit_k(0)));
        // A test can withhold this arrival in CTA 0 to make the softmax warps'
        // bounded wait run out (the timeout path, without a fault).
        if (leader && !(a.withhold_arrival && blockIdx.x == 0)) mma_commit(b_sfull);
        if (leader) mma_commit(b_empty0 + 8 * slot_of(unit_k(0)));
      }
      for (int j = 0; ok && j < n; ++j) {
        if (j + 1 < n) {
          // S_{j+1} once S_j has been read out of TMEM
          const int uk = unit_k(j + 1);
          if (!(ok = wait_warp(b_full0 + 8 * slot_of(uk), parity_of(uk), ctl, a.status,
                                  a.timeout_ns)))
            break;
          if (!(ok = wait_warp(b_sfree, j & 1, ctl, a.status, a.timeout_ns))) break;
          tc_fence_after();
          issue_S(slot_of(uk));
          if (leader) mma_commit(b_sfull);
          if (leader) mma_commit(b_empty0 + 8 * slot_of(uk));
        }
        // P_j V_j once P_j is in TMEM
        const int uv = unit_v(j);
        if (!(ok = wait_warp(b_full0 + 8 * slot_of(uv), parity_of(uv), ctl, a.status,
                                a.timeout_ns)))
          break;
        if (!(ok = wait_warp(b_pready, j & 1, ctl, a.status, a.timeout_ns))) break;
        tc_fence_after();
        issue_PV(slot_of(uv), j > 0);
        if (leader) mma_commit(b_pvdone);
        if (leader) mma_commit(b_empty0 + 8 * slot_of(uv));
      }
      // Drain: every MMA (and every commit arrival) of this thread is complete.
      if (leader) mma_commit(b_mmadone);
      wait_bounded(b_mmadone, 0, ctl, a.status, a.timeout_ns, false);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int r = warp * 32 + lane;                          // row in the query tile
    const int64_t qrow = qt * C::BM + r;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const uint32_t tS = lane_base + C::COL_S;
    const uint32_t tO = lane_base + C::COL_O;
    const uint32_t tP = lane_base + C::COL_P;
    const float c = a.c;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    // last valid key column of the last key tile
    const int lim_last = static_cast<int>(Nk - 1 - static_cast<int64_t>(nk - 1) * C::BN);
    // keep bits of this row, stored into the caller's keep mask (16 bytes
    // per key tile, tiles rows_q entries apart) for the backward
    uint4* mrow = nullptr;
    if (DROP && a.drop.mask != nullptr && qrow < Nq)
      mrow = reinterpret_cast<uint4*>(a.drop.mask + mask_entry(a.drop, a.g, sv, h, 0, qrow));
    for (int j = 0; j < n; ++j) {
      // Dropout keep bits of this row's 128 keys, drawn before the scores
      // arrive (positions only): bit k of kb[k / 32] is key j*128 + k.
      uint32_t kb[4] = {0u, 0u, 0u, 0u};
      if constexpr (DROP) {
        tile_keep_bits(a.drop, bh, j, qrow, kb);
        if (mrow) mrow[j * a.g.rows_q] = make_uint4(kb[0], kb[1], kb[2], kb[3]);
      }
      if (!(ok = wait_warp(b_sfull, j & 1, ctl, a.status, a.timeout_ns))) break;
      tc_fence_after();
      float s[128];
      {
        uint32_t r0[32], r1[32], r2[32], r3[32];
        tmem_ld32(tS + 0, r0);
        tmem_ld32(tS + 32, r1);
        tmem_ld32(tS + 64, r2);
        tmem_ld32(tS + 96, r3);
        tmem_wait_ld();
        reg_fence32(r0); reg_fence32(r1); reg_fence32(r2); reg_fence32(r3);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          s[i] = __uint_as_float(r0[i]);
          s[32 + i] = __uint_as_float(r1[i]);
          s[64 + i] = __uint_as_float(r2[i]);
          s[96 + i] = __uint_as_float(r3[i]);
        }
      }
      // S is in registers: the tensor cores may overwrite it with S_{j+1}.
      tc_fence_before();
      mbar_arrive(b_sfree);
      // Exclude keys past the sequence (last key tile) and keys after the
      // query (the diagonal tile, the only one a causal row can straddle).
      int lim = C::BN - 1;
      if (a.causal && j == qt) lim = r;
      if (j == nk - 1) lim = min(lim, lim_last);
      if (lim < C::BN - 1) {
#pragma unroll
        for (int kk = 0; kk < C::BN; ++kk)
          if (kk > lim) s[kk] = -INFINITY;
      }
      float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
      for (int kk = 0; kk < C::BN; kk += 8) {
        mx0 = max3f(mx0, s[kk], s[kk + 1]);
        mx1 = max3f(mx1, s[kk + 2], s[kk + 3]);
        mx2 = max3f(mx2, s[kk + 4], s[kk + 5]);
        mx3 = max3f(mx3, s[kk + 6], s[kk + 7]);
      }
      const float m_new = fmaxf(m, fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * c);
      // Lazy rescale decision (warp-uniform for the TMEM access below).
      bool rescale = false;
      float alpha = 1.f;
      if (j == 0) {
        m = m_new;
      } else {
        const bool need = m_new > m + 8.f;
        rescale = __any_sync(0xffffffffu, need);
        if (need) {
          alpha = ex2(m - m_new);
          l *= alpha;
          m = m_new;
        }
      }
      const float negm = -m;
      // paired fp32: c * s - m and the row sum two keys at a time
      const uint64_t cc = f32x2(c, c), nm = f32x2(negm, negm);
      uint64_t acc = f32x2(0.f, 0.f);
      // P in two halves of 64 keys (32 columns each); the first half waits
      // (in registers) until P_{j-1} V has finished reading the P columns,
      // which also makes O stable for a rescale.
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float x0, x1;
          f32x2_split(fma_f32x2(f32x2(s[64 * half + 2 * i], s[64 * half + 2 * i + 1]), cc, nm),
                      x0, x1);
          const float p0 = ex2(x0), p1 = ex2(x1);
          acc = add_f32x2(acc, f32x2(p0, p1));
          if constexpr (DROP) {
            // l sums the undropped weights; P V takes the kept ones (the
            // 1 / (1 - p) of Z is applied with 1 / l at the end)
            // keys kk, kk + 1 are bits b, b + 1 of byte kk / 8 % 4 of their
            // word (b = kk % 8): shifted by 7 - b and 6 - b they are that
            // byte's sign bits, which one prmt spreads over the pair's halves
            const int kk = 64 * half + 2 * i, byte = (kk >> 3) & 3, b = kk & 7;
            const uint32_t wk = kb[kk >> 5];
            pk[i] = pack2<T>(p0, p1) & prmt(wk << (7 - b), wk << (6 - b), half_sign_sel(byte, 4 + byte));
          } else {
            pk[i] = pack2<T>(p0, p1);
          }
        }
        if (half == 0 && j > 0) {
          if (!(ok = wait_warp(b_pvdone, (j - 1) & 1, ctl, a.status, a.timeout_ns))) break;
          tc_fence_after();
          if (rescale) {
#pragma unroll 1
            for (int c4 = 0; c4 < D / 32; ++c4) {
              uint32_t t[32];
              tmem_ld32(tO + 32 * c4, t);
              tmem_wait_ld();
              reg_fence32(t);
#pragma unroll
              for (int i = 0; i < 32; ++i) t[i] = __float_as_uint(__uint_as_float(t[i]) * alpha);
              tmem_st32(tO + 32 * c4, t);
            }
          }
        }
        tmem_st32(tP + 32 * half, pk);
      }
      if (!ok) break;
      {
        float lo, hi;
        f32x2_split(acc, lo, hi);
        l += lo + hi;
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(b_pready);
    }
    if (ok) ok = wait_warp(b_pvdone, (n - 1) & 1, ctl, a.status, a.timeout_ns);
    // O / l staged in shared memory (the K | V ring is idle once the last
    // P V has completed) as the loads lay it out, then stored by the four
    // warps with consecutive threads on consecutive 16 bytes of a row (whole
    // lines per warp store); rows past the sequence are not written.  Every
    // softmax thread passes the barrier, also after a timeout; the stores go
    // out only if all of them got this far.
    const uint32_t stg = smem_u32(sRing);
    if (ok) {
      tc_fence_after();
      const float inv = (DROP ? a.drop.rscale : 1.f) / l;   // Z's 1 / (1 - p) with dropout
      stage_row_sw128<T>(tO, inv, stg, r, 0, D);
      if (qrow < Nq) a.lse[lse_index(a.g, sv, h, qrow)] = (m + log2f(l)) * kLn2;
    }
    if (bar_red_and(1, 128, ok)) {
      T* row0 = static_cast<T*>(a.o) + bb * a.so[0] + hq * a.so[1] + (sv.q0 + qt * C::BM) * a.so[2];
      store_staged_tile<T>(stg, D, threadIdx.x, 128, row0, a.so[2],
                           static_cast<int>(Nq - qt * C::BM < C::BM ? Nq - qt * C::BM : C::BM), a.dreal);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <typename T, int D>
fa_status run_fwd_tc(const FwdParams& p, cudaStream_t stream) {
  using C = FwdCfg<D>;
  const Geo& g = p.g;
  // Tensor maps carry the true head dimension; a narrower one than D reads
  // as zeros past its end (TMA fill), which leaves every product exact.
  CUtensorMap mq, mk, mv;
  if (!encode_tile_map(&mq, p.q, p.dtype, g.Bt, g.Hq, g.rows_q, p.D, p.sq, 128, 64) ||
      !encode_tile_map(&mk, p.k, p.dtype, g.Bt, g.Hkv, g.rows_k, p.D, p.sk, 128, 64) ||
      !encode_tile_map(&mv, p.v, p.dtype, g.Bt, g.Hkv, g.rows_k, p.D, p.sv, 128, 64))
    return FA_ERR_LAUNCH;
  FwdTcArgs a{};
  a.dreal = static_cast<int>(p.D);
  a.o = p.o; a.lse = p.lse;
  a.g = g;
  a.BH = g.B * g.Hq; a.npairs = (g.Nq + 255) / 256;
  // K and V of a head: the operand all of its CTAs read
  a.hgroup = head_group(a.BH, 2 * g.Nk * p.D * (p.dtype == FA_F32 ? 4 : 2));
  for (int i = 0; i < 4; ++i) a.so[i] = p.so[i];
  a.causal = p.causal;
  a.c = p.scale * kLog2e;
  a.drop = p.drop;
  a.status = p.status;
  a.timeout_ns = p.timeout_ns;
  a.withhold_arrival = p.withhold_arrival;
  const int64_t blocks = a.BH * a.npairs;
  if (blocks > 0x7fffffffLL) return FA_ERR_SHAPE;
  if constexpr (D == 64) {
    // one query tile per CTA (npairs counts query tiles here), two CTAs per SM
    a.npairs = (g.Nq + 127) / 128;
    const int64_t blocks1 = a.BH * a.npairs;
    if (blocks1 > 0x7fffffffLL) return FA_ERR_SHAPE;
    auto kern = p.drop.on ? fwd_tc_1t_kernel<T, kDropDraw> : fwd_tc_1t_kernel<T, kDropNone>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Fwd1Cfg::SMEM) !=
        cudaSuccess)
      return FA_ERR_LAUNCH;
    kern<<<dim3(static_cast<unsigned>(blocks1)), dim3(Fwd1Cfg::THREADS), Fwd1Cfg::SMEM, stream>>>(
        mq, mk, mv, a);
  } else {
    auto kern = p.drop.on ? fwd_tc_kernel<T, D, kDropDraw> : fwd_tc_kernel<T, D, kDropNone>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
        cudaSuccess)
      return FA_ERR_LAUNCH;
    kern<<<dim3(static_cast<unsigned>(blocks)), dim3(C::THREADS), C::SMEM, stream>>>(mq, mk, mv, a);
  }
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

}  // namespace

// D = 16 and 32 run through the D = 64 kernel, zero-padded by the TMA loads.
bool have_fwd_tc(int64_t D, fa_dtype dt) {
  return (D == 16 || D == 32 || D == 64 || D == 128) && dt != FA_F32;
}

fa_status launch_fwd_tc(const FwdParams& p, cudaStream_t s) {
  if (p.dtype == FA_BF16) {
    if (p.D == 128) return run_fwd_tc<__nv_bfloat16, 128>(p, s);
    if (p.D <= 64) return run_fwd_tc<__nv_bfloat16, 64>(p, s);
  } else if (p.dtype == FA_F16) {
    if (p.D == 128) return run_fwd_tc<__half, 128>(p, s);
    if (p.D <= 64) return run_fwd_tc<__half, 64>(p, s);
  }
  return FA_ERR_ARG;
}

}  // namespace fa
