// Device helpers shared by the tensor-core backward kernels (the split dK/dV
// and dQ kernels of fa_bwd_tc.cu and the single-pass kernel of
// fa_bwd_fused.cu): whole-row TMEM transfers of one elementwise thread, the
// dropout keep bits of a key row, and the cluster reduction of partial dK, dV
// when several CTAs share one key tile's query heads.
#pragma once

#include "tc_common.cuh"

namespace fa {
namespace tc {

// Loads 64 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&x)[64]) {
  uint32_t a[32], b[32];
  tmem_ld32(taddr, a);
  tmem_ld32(taddr + 32, b);
  tmem_wait_ld();
  reg_fence32(a);
  reg_fence32(b);
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    x[i] = __uint_as_float(a[i]);
    x[32 + i] = __uint_as_float(b[i]);
  }
}

// Rounds 64 floats to T, packs two per column and stores 32 TMEM columns.
template <typename T>
__device__ __forceinline__ void tmem_st_packed64(uint32_t taddr, const float (&x)[64]) {
  uint32_t w[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) w[i] = pack2<T>(x[2 * i], x[2 * i + 1]);
  tmem_st32(taddr, w);
}

// Keep bits of the key held by a lane for 64 consecutive queries, as the
// octet exchange below leaves them: query qbase + q is bit kbit(q) (a fixed
// permutation; q is a compile-time constant wherever it is used).
__device__ __forceinline__ constexpr int kbit(int q) { return 8 * (q & 7) + (q >> 3); }

// Transposes the 8 x 8 bit matrix held in (lo, hi) as bytes (byte r, bit c
// -> byte c, bit r): three delta swaps of 7, 14 and 28 bit positions.
__device__ __forceinline__ void bit_transpose8(uint32_t& lo, uint32_t& hi) {
  uint32_t t;
  t = (lo ^ (lo >> 7)) & 0x00AA00AAu; lo ^= t ^ (t << 7);
  t = (hi ^ (hi >> 7)) & 0x00AA00AAu; hi ^= t ^ (t << 7);
  t = (lo ^ (lo >> 14)) & 0x0000CCCCu; lo ^= t ^ (t << 14);
  t = (hi ^ (hi >> 14)) & 0x0000CCCCu; hi ^= t ^ (t << 14);
  t = (lo ^ __funnelshift_r(lo, hi, 28)) & 0xF0F0F0F0u;   // the 64-bit x ^ (x >> 28), low word
  lo ^= t;
  hi ^= t >> 4;
}

// The octet's exchange.  Lane e of the octet (lane & 7) holds b[t], the 8-bit
// keep decisions of query qbase + 8t + e for the octet's eight consecutive
// keys (bit k: key k).  Each lane packs its eight bytes, transposes them as
// an 8 x 8 bit matrix (byte k then holds key k's decisions for its eight
// queries), and the octet transposes the 8 x 8 byte matrix across its lanes
// (three butterfly stages, one shuffle each), so that lane k ends with byte e
// = lane e's byte k: bit 8e + t = kbit(8t + e) is query qbase + 8t + e of
// key k.  Every lane of the warp must call it.
__device__ __forceinline__ uint64_t octet_exchange(const uint32_t (&b)[8], int lane) {
  uint32_t lo = __byte_perm(__byte_perm(b[0], b[1], 0x3340), __byte_perm(b[2], b[3], 0x3340), 0x5410);
  uint32_t hi = __byte_perm(__byte_perm(b[4], b[5], 0x3340), __byte_perm(b[6], b[7], 0x3340), 0x5410);
  bit_transpose8(lo, hi);
  const bool x4 = lane & 4, x2 = lane & 2, x1 = lane & 1;
  // stage 4: swap the off-diagonal 4 x 4 blocks (words)
  const uint32_t r4 = __shfl_xor_sync(0xffffffffu, x4 ? lo : hi, 4);
  if (x4) lo = r4; else hi = r4;
  // stage 2: within each word, swap the off-diagonal 2 x 2 blocks (16-bit halves)
  const uint32_t r2 = __shfl_xor_sync(0xffffffffu, __byte_perm(lo, hi, x2 ? 0x5410 : 0x7632), 2);
  lo = __byte_perm(lo, r2, x2 ? 0x3254 : 0x5410);
  hi = __byte_perm(hi, r2, x2 ? 0x3276 : 0x7610);
  // stage 1: swap single bytes
  const uint32_t r1 = __shfl_xor_sync(0xffffffffu, __byte_perm(lo, hi, x1 ? 0x6420 : 0x7531), 1);
  lo = __byte_perm(lo, r1, x1 ? 0x3514 : 0x5240);
  hi = __byte_perm(hi, r1, x1 ? 0x3716 : 0x7260);
  return static_cast<uint64_t>(hi) << 32 | lo;
}

// Dropout keep bits of the key held by this lane for 64 consecutive queries
// qbase .. qbase + 63 of flat head bhq, drawn: query qbase + q is bit
// kbit(q).  The eight lanes of an octet hold eight consecutive keys
// 8*jg .. 8*jg + 7, which one generator call covers for one query: lane e of
// the octet draws for queries qbase + 8t + e and the octet exchanges the
// results (octet_exchange).  Every lane of the warp must call it.
__device__ __forceinline__ uint64_t octet_keep_bits(const Dropout& d, uint32_t jg, int64_t qbase,
                                                    uint32_t bhq, int lane) {
  const int e = lane & 7;
  uint32_t b[8];
#pragma unroll
  for (int t = 0; t < 8; ++t) b[t] = keep8(d, jg, static_cast<uint32_t>(qbase + 8 * t + e), bhq);
  return octet_exchange(b, lane);
}

// The same bits read from the keep mask (Dropout::mask), in two steps so the
// loads can be issued a step ahead: octet_mask_load reads, for query head h
// of sequence v, key tile jt, the octet's byte `gbyte` (key group mod 16) of
// the 16-byte entries of queries qbase .. qbase + 63 (lane e of the octet
// reads queries qbase + 8t + e; queries past the sequence read as dropped),
// and octet_mask_bits exchanges them within the octet as for drawn bits
// (query qbase + q is bit kbit(q)).  Every lane of the warp must call
// octet_mask_bits.
__device__ __forceinline__ void octet_mask_load(const Dropout& d, const Geo& g, const SeqView& v,
                                                int64_t h, int64_t jt, int64_t qbase, int gbyte,
                                                int lane, uint32_t (&b)[8]) {
  const int e = lane & 7;
  const uint8_t* col = d.mask + mask_entry(d, g, v, h, jt, qbase) + gbyte;
#pragma unroll
  for (int t = 0; t < 8; ++t)
    b[t] = qbase + 8 * t + e < v.nq ? static_cast<uint32_t>(__ldg(col + (8 * t + e) * 16)) : 0u;
}

__device__ __forceinline__ uint64_t octet_mask_bits(const uint32_t (&b)[8], int lane) {
  return octet_exchange(b, lane);
}

// Staging of a CTA's partial dV (t = 0) and dK (t = 1) for the cluster
// reduction: [2][128 rows][D] fp32 at the start of shared memory (operand
// buffers that are idle by then), 16-byte chunk c of row r stored at chunk
// c ^ (r mod 8) so a warp's 32 rows spread over the banks.
template <int D>
__device__ __forceinline__ float* stage_row(uint8_t* smem, int t, int row) {
  return reinterpret_cast<float*>(smem) + (t * 128 + row) * D;
}
__device__ __forceinline__ int stage_chunk(int c, int row) { return c ^ (row & 7); }

// A rank other than 0: copies this thread's accumulator row (D fp32 TMEM
// columns at acc) into its staging row t for rank 0 to read.
template <int D>
__device__ __forceinline__ void stage_partial(uint8_t* smem, int t, int row, uint32_t acc) {
  float* st = stage_row<D>(smem, t, row);
#pragma unroll 1
  for (int cc = 0; cc < D / 32; ++cc) {
    uint32_t v[32];
    tmem_ld32(acc + 32 * cc, v);
    tmem_wait_ld();
    reg_fence32(v);
#pragma unroll
    for (int u = 0; u < 8; ++u)
      *reinterpret_cast<uint4*>(st + 4 * stage_chunk(cc * 8 + u, row)) =
          make_uint4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
  }
}

// Rank 0 (between the two cluster barriers): adds the staged rows t of ranks
// 1 .. split-1 (distributed shared memory) to its own accumulator row at acc,
// scales by mul, rounds to T and, when store, writes the first dreal
// columns to out.
template <typename T, int D>
__device__ __forceinline__ void cluster_reduce_store(uint8_t* smem, int t, int row, uint32_t acc,
                                                     int split, float mul, T* out, bool store,
                                                     int dreal) {
  const uint32_t st = smem_u32(stage_row<D>(smem, t, row));
#pragma unroll 1
  for (int cc = 0; cc < dreal / 32 + (dreal % 32 ? 1 : 0); ++cc) {
    uint32_t w32[32];
    tmem_ld32(acc + 32 * cc, w32);
    tmem_wait_ld();
    reg_fence32(w32);
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(w32[i]);
    for (int r = 1; r < split; ++r) {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float4 x = ld_cluster_f4(cluster_map(st + 16 * stage_chunk(cc * 8 + u, row),
                                                   static_cast<uint32_t>(r)));
        v[4 * u] += x.x; v[4 * u + 1] += x.y; v[4 * u + 2] += x.z; v[4 * u + 3] += x.w;
      }
    }
    if (store) {
      const int ncol = min(32, dreal - 32 * cc);   // 16 or 32
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

}  // namespace tc
}  // namespace fa
