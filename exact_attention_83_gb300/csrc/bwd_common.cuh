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

// The octet's exchange: lane e' of the octet (lane & 7) holds `bits`, the
// 8-bit keep decisions of query 8t + e' for the octet's eight consecutive
// keys; returns, for this lane's key (bit e = lane & 7), the decisions of the
// eight queries 8t .. 8t + 7 as bits 0..7.  Three shuffles and a bit gather;
// every lane of the warp must call it.
__device__ __forceinline__ uint64_t octet_gather8(uint32_t bits, int e) {
  uint64_t x = static_cast<uint64_t>(bits) << (8 * e);
  x |= __shfl_xor_sync(0xffffffffu, x, 1);
  x |= __shfl_xor_sync(0xffffffffu, x, 2);
  x |= __shfl_xor_sync(0xffffffffu, x, 4);
  // bit 8 * e' + e of x is (query 8t + e', this key); gather them
  const uint64_t y = (x >> e) & 0x0101010101010101ull;
  return (y * 0x0102040810204080ull) >> 56;
}

// Dropout keep bits of the key held by this lane for 64 consecutive queries
// qbase .. qbase + 63 of flat head bhq: bit q set iff weight (qbase + q, key)
// is kept.  The eight lanes of an octet hold eight consecutive keys
// 8*jg .. 8*jg + 7, which one generator call covers for one query: lane e of
// the octet draws for query qbase + 8t + e and the octet exchanges the
// results (octet_gather8).  Every lane of the warp must call it.
__device__ __forceinline__ uint64_t octet_keep_bits(const Dropout& d, uint32_t jg, int64_t qbase,
                                                    uint32_t bhq, int lane) {
  const int e = lane & 7;
  uint64_t keep = 0;
#pragma unroll
  for (int t = 0; t < 8; ++t)
    keep |= octet_gather8(keep8(d, jg, static_cast<uint32_t>(qbase + 8 * t + e), bhq), e) << (8 * t);
  return keep;
}

// The same bits read from the keep mask (Dropout::mask), in two steps so the
// loads can be issued a step ahead: octet_mask_load reads, for query head h
// of sequence v, key tile jt, the octet's byte `gbyte` (key group mod 16) of
// the 16-byte entries of queries qbase .. qbase + 63 (lane e of the octet
// reads queries qbase + 8t + e; queries past the sequence read as dropped),
// and octet_mask_bits exchanges them within the octet as for drawn bits.
// Every lane of the warp must call octet_mask_bits.
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
  const int e = lane & 7;
  uint64_t keep = 0;
#pragma unroll
  for (int t = 0; t < 8; ++t) keep |= octet_gather8(b[t], e) << (8 * t);
  return keep;
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
