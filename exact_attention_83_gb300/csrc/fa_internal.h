// Internal declarations shared by the translation units of libfa.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "../../include/fa.h"

namespace fa {

// Problem geometry, validated by the ABI layer.
//  Fixed lengths: B sequences of Nq query and Nk key rows; a tensor row is
//  addressed as (b, h, n).  Packed variable lengths: cu_q / cu_k hold B+1
//  offsets into rows_q / rows_k packed rows, the tensors have one batch entry
//  (b-stride unused), and sequence b's row n is packed row cu[b] + n.
//  Query head h reads key/value head h / G.
struct Geo {
  int64_t B, Hq, Hkv, G;     // G = Hq / Hkv
  int64_t Nq, Nk;            // rows per sequence (upper bounds when packed)
  const int32_t* cu_q;       // device, B+1 entries, or null (fixed lengths)
  const int32_t* cu_k;
  int64_t rows_q, rows_k;    // tensor rows per (b, h): Nq, Nk, or the packed totals
  int64_t Bt;                // batch extent of the tensors: B, or 1 when packed
};

// Dropout of the attention weights: weight (i, j) of query head h in sequence
// b is kept iff 16-bit half (j mod 2) of word ((j mod 8) / 2) of Philox4x32-10
// (Salmon, Moraes, Dror and Shaw, "Parallel Random Numbers: As Easy as 1, 2,
// 3", SC 2011) at counter (j / 8, i, b * Hq + h, offset) under key
// (key0, key1) is >= thr = floor(p * 65536); kept weights are multiplied by
// rscale = 1 / (1 - p).  One generator call serves eight consecutive keys.
// The key of round r (key0 and key1 bumped r times by the two Weyl
// constants) is computed on the host: as a kernel parameter it is read from
// the constant bank and takes no register.
struct Dropout {
  int on;
  uint32_t thr;
  float rscale;
  uint32_t key0, key1, offset;
  uint32_t rk0[10], rk1[10];   // round keys
  // Keep mask, or null: 16 bytes per (sequence-level flat head, key tile of
  // 128, query row); byte g of key tile t is keep8 of key group 16t + g.
  // The forward writes it, the backward reads it.  mask_kt = key tiles per
  // head.
  uint8_t* mask;
  int64_t mask_kt;
};

// Parameters of one forward call.
struct FwdParams {
  const void* q; const void* k; const void* v;
  void* o; float* lse;
  Geo g;
  int64_t D;
  int64_t sq[4], sk[4], sv[4], so[4];   // element strides (b, h, n, d), d == 1
  int causal;
  float scale;
  fa_dtype dtype;
  Dropout drop;
  unsigned int* status;   // device status word (first error a kernel records)
  uint64_t timeout_ns;    // bound on any single device-side wait
  int withhold_arrival;   // test-only: CTA 0 skips one mbarrier arrival (see fa.h)
};

struct PreParams {
  const void* o; const void* dout; float* delta;
  int64_t B, H, N, D;
  int64_t so[4], sdo[4];
  fa_dtype dtype;
};

struct BwdParams {
  const void* q; const void* k; const void* v; const void* dout;
  const float* lse; const float* delta;
  void* dq; void* dk; void* dv;
  Geo g;
  int64_t D;
  int64_t sq[4], sk[4], sv[4], sdo[4], sdq[4], sdk[4], sdv[4];
  int causal;
  float scale;
  fa_dtype dtype;
  Dropout drop;
  unsigned int* status;
  uint64_t timeout_ns;
  const cudaEvent_t* prof;   // 3 events to record around the two kernels, or null
  int withhold_arrival;      // test-only (single-pass backward): see fa.h
  bool allow_side;           // the dQ kernel may run on the device's side stream
};

#ifdef __CUDACC__
// One sequence as a kernel sees it: batch coordinate of the tensors, first
// query / key row, lengths.  ok is false when packed offsets are inconsistent
// (decreasing, past the packed rows, or longer than Nq / Nk); the caller then
// records FA_ERR_SEQLENS and touches nothing of that sequence.
struct SeqView {
  int64_t b, q0, k0, nq, nk;
  bool ok;
};

__device__ __forceinline__ SeqView seq_view(const Geo& g, int64_t b) {
  SeqView v;
  if (g.cu_q == nullptr) {
    v.b = b; v.q0 = 0; v.k0 = 0; v.nq = g.Nq; v.nk = g.Nk; v.ok = true;
    return v;
  }
  const int64_t q0 = __ldg(g.cu_q + b), q1 = __ldg(g.cu_q + b + 1);
  const int64_t k0 = __ldg(g.cu_k + b), k1 = __ldg(g.cu_k + b + 1);
  v.b = 0; v.q0 = q0; v.k0 = k0; v.nq = q1 - q0; v.nk = k1 - k0;
  v.ok = q0 >= 0 && q1 >= q0 && q1 <= g.rows_q && v.nq <= g.Nq &&
         k0 >= 0 && k1 >= k0 && k1 <= g.rows_k && v.nk <= g.Nk;
  return v;
}

// Index of (b, h, row) in the fp32 lse / delta arrays: [Bt, Hq, rows_q].
__device__ __forceinline__ int64_t lse_index(const Geo& g, const SeqView& v, int64_t h,
                                             int64_t row) {
  return (v.b * g.Hq + h) * g.rows_q + v.q0 + row;
}

__device__ __forceinline__ void record_status(unsigned int* status, unsigned int code) {
  atomicCAS(status, 0u, code);
}

// Philox4x32-10: ten rounds of the published round function (each multiplies
// counter words 0 and 2 by the round multipliers and mixes the halves of the
// 64-bit products with words 1 and 3 and the round's key); the round keys are
// the key bumped by the two Weyl constants once per round (Dropout::rk0/rk1).
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, const uint32_t (&rk0)[10],
                                               const uint32_t (&rk1)[10]) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    uint64_t p0, p1;
    asm("mul.wide.u32 %0, %1, %2;" : "=l"(p0) : "r"(c.x), "r"(0xD2511F53u));
    asm("mul.wide.u32 %0, %1, %2;" : "=l"(p1) : "r"(c.z), "r"(0xCD9E8D57u));
    c = make_uint4(static_cast<uint32_t>(p1 >> 32) ^ c.y ^ rk0[r], static_cast<uint32_t>(p1),
                   static_cast<uint32_t>(p0 >> 32) ^ c.w ^ rk1[r], static_cast<uint32_t>(p0));
  }
  return c;
}

// Dropout modes of the tensor-core kernels (template parameter DROP): no
// dropout, keep decisions drawn in the kernel, or read from the keep mask
// (the backward, when the forward left one).
enum : int { kDropNone = 0, kDropDraw = 1, kDropRead = 2 };
inline int bwd_drop_mode(const Dropout& d) {
  return !d.on ? kDropNone : (d.mask != nullptr ? kDropRead : kDropDraw);
}

// Keep bit b (a compile-time constant wherever it is used) of 64 bits held
// as two words: one masked test of one word, no 64-bit shift.
__device__ __forceinline__ bool kept64(uint32_t lo, uint32_t hi, int b) {
  return ((b < 32 ? lo : hi) & (1u << (b & 31))) != 0u;
}

// Byte offset in the keep mask of the 16-byte entry of (query head h of
// sequence v, key tile jt, query row `row` of the sequence); entries of
// consecutive rows are 16 bytes apart.
__device__ __forceinline__ int64_t mask_entry(const Dropout& d, const Geo& g, const SeqView& v,
                                              int64_t h, int64_t jt, int64_t row) {
  return (((v.b * g.Hq + h) * d.mask_kt + jt) * g.rows_q + v.q0 + row) * 16;
}

// The eight keep decisions for keys 8*jg .. 8*jg+7 of query row i in flat
// head bh (= b * Hq + h), as bits 0..7.
__device__ __forceinline__ uint32_t keep8(const Dropout& d, uint32_t jg, uint32_t i,
                                          uint32_t bh) {
  const uint4 r = philox4x32_10(make_uint4(jg, i, bh, d.offset), d.rk0, d.rk1);
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
  // half >= thr as whole-word compares against thr * 2^16: the high half
  // compares as w itself, the low half as w << 16 (fewer integer-pipe
  // instructions than extracting each half)
  const uint32_t t16 = d.thr << 16;
  uint32_t bits = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    bits |= (w[e] >= t16 ? 2u : 0u) << (2 * e);
    bits |= ((w[e] << 16) >= t16 ? 1u : 0u) << (2 * e);
  }
  return bits;
}

// Keep bits of query row `row` in flat head bh (= b * Hq + h) for the 128
// keys of key tile jt, drawn: bit k of kb[k / 32] is key 128 jt + k.
__device__ __forceinline__ void tile_keep_bits(const Dropout& d, int64_t bh, int64_t jt,
                                               int64_t row, uint32_t (&kb)[4]) {
  kb[0] = kb[1] = kb[2] = kb[3] = 0u;
#pragma unroll
  for (int g8 = 0; g8 < 16; ++g8)
    kb[g8 >> 2] |= keep8(d, static_cast<uint32_t>(jt * 16 + g8), static_cast<uint32_t>(row),
                         static_cast<uint32_t>(bh))
                   << (8 * (g8 & 3));
}
#endif

// Records prof[i] on s when profiling events are set.
inline void prof_record(const BwdParams& p, int i, cudaStream_t s) {
  if (p.prof) cudaEventRecord(p.prof[i], s);
}

// Kernel families.  Each launcher returns FA_OK, FA_ERR_LAUNCH, or
// FA_ERR_ARG when it has no kernel compiled for the (D, dtype) asked for.
fa_status launch_fwd_ffma(const FwdParams& p, cudaStream_t s);
fa_status launch_bwd_ffma(const BwdParams& p, cudaStream_t s);
fa_status launch_preprocess(const PreParams& p, cudaStream_t s);
fa_status launch_fwd_tc(const FwdParams& p, cudaStream_t s);
fa_status launch_bwd_tc(const BwdParams& p, cudaStream_t s);
bool have_fwd_tc(int64_t D, fa_dtype dt);
bool have_bwd_tc(int64_t D, fa_dtype dt);
// Single-pass backward (fp16/bf16): dK, dV and dQ through the fp32 workspace
// `ws` of bwd_fused_workspace_floats(g, D) floats, 16-byte aligned.
fa_status launch_bwd_fused(const BwdParams& p, float* ws, cudaStream_t s);
size_t bwd_fused_workspace_floats(const Geo& g, int64_t D);
// Keep mask (fa_dropout_mask): its size in bytes, and the kernel that fills
// the entries the attention kernels read (d.on must be set).
size_t dropout_mask_bytes(const Geo& g);
fa_status launch_dropout_mask(const Geo& g, int causal, const Dropout& d, uint8_t* mask,
                              unsigned int* status, cudaStream_t s);

// Encodes a 4-D tiled TMA map (d, n, h, b) over a strided [B,H,N,D] fp16/bf16
// tensor with 128-byte swizzle and a box of box_cols x box_rows elements.
bool encode_tile_map(CUtensorMap* map, const void* base, fa_dtype dt, int64_t B, int64_t H,
                     int64_t N, int64_t D, const int64_t* strides, uint32_t box_rows,
                     uint32_t box_cols);

// Encodes a 3-D tiled TMA map over `planes` contiguous blocks of `rows` fp32
// rows of `cols` elements, 128-byte swizzle, box of box_cols x box_rows.
bool encode_f32_rows_map(CUtensorMap* map, const float* base, int64_t cols, int64_t rows,
                         int64_t planes, uint32_t box_cols, uint32_t box_rows);

// Number of SMs of the current device (cached per device).
int device_sm_count();

// fa_bwd with the choice of letting the tensor-core dQ kernel use the side
// stream (fa_bwd: yes; fa_bwd_noalloc, which creates nothing: no).
fa_status bwd_square(const void* q, const void* k, const void* v, const void* dout,
                     const float* lse, const float* delta, void* dq, void* dk, void* dv,
                     int64_t B, int64_t H, int64_t N, int64_t D, const int64_t* sq,
                     const int64_t* sk, const int64_t* sv, const int64_t* sdo,
                     const int64_t* sdq, const int64_t* sdk, const int64_t* sdv, int causal,
                     float scale, fa_dtype dtype, cudaStream_t stream, bool allow_side);

// The current device's side stream: side_begin makes it wait for the work
// enqueued so far on `caller` and returns it (holding the device's fork/join
// lock); side_end makes `caller` wait for everything enqueued on the side
// stream since and releases the lock.  Every successful side_begin must be
// followed by side_end on the same thread.
fa_status side_begin(cudaStream_t caller, cudaStream_t* side);
fa_status side_end(cudaStream_t caller);
// True while `s` is being captured into a CUDA graph (or its status cannot
// be read).
bool stream_capturing(cudaStream_t s);

// Heads per group of the grouped block order (grouped_tile), from
// `per_head_bytes` (the operand that all CTAs of a head read) and the current
// device's L2: all BH heads when their operands fit in 3/4 of L2 together,
// else as many as fit in 3/8 of it (at least 1).
int64_t head_group(int64_t BH, int64_t per_head_bytes);

// Grouped block order of the tiled kernels.  Blocks run roughly in index
// order; heads are taken in groups of `hg`, and within a group the tile
// index t varies slowest (t = 0 first: callers map it to their longest
// tile) with the group's heads interleaved.  So the CTAs in flight belong to
// a few heads, whose shared operand stays in L2, while each group still runs
// longest first and the grid ends on short tiles.  With hg >= BH this is the
// plain tile-major order over all heads.  Block `id` of BH * nt maps to head
// `bh` and tile `t`.  The grid holds fewer than 2^31 blocks, so every value
// here fits 32-bit unsigned arithmetic (cheaper divisions in the prologue).
__device__ __forceinline__ void grouped_tile(int64_t id, int64_t BH, int64_t nt, int64_t hg,
                                             int64_t& bh, int64_t& t) {
  const uint32_t i = static_cast<uint32_t>(id), nh = static_cast<uint32_t>(BH);
  const uint32_t g = static_cast<uint32_t>(hg), per = g * static_cast<uint32_t>(nt);
  const uint32_t grp = i / per, rem = i - grp * per;
  const uint32_t g0 = grp * g;
  const uint32_t gh = nh - g0 < g ? nh - g0 : g;     // heads in this group
  const uint32_t tt = rem / gh;
  t = tt;
  bh = g0 + (rem - tt * gh);
}

// Every argument check of fa_bwd_preprocess followed by fa_bwd on a square
// problem (shape, dtype, scale, each tensor's pointer, alignment and strides,
// lse), except the delta pointer, which the caller supplies itself.  Touches
// no device: no context is created and nothing is launched.
fa_status validate_square_bwd(const void* q, const void* k, const void* v, const void* o,
                              const void* dout, const float* lse, const void* dq,
                              const void* dk, const void* dv, int64_t B, int64_t H, int64_t N,
                              int64_t D, const int64_t* sq, const int64_t* sk,
                              const int64_t* sv, const int64_t* so, const int64_t* sdo,
                              const int64_t* sdq, const int64_t* sdk, const int64_t* sdv,
                              int causal, float scale, fa_dtype dtype);

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------- element I/O
template <typename T> struct Elem;
template <> struct Elem<float> {
  static __device__ __forceinline__ float load(const float* p) { return __ldg(p); }
  static __device__ __forceinline__ float to_f32(float x) { return x; }
  static __device__ __forceinline__ float from_f32(float x) { return x; }
};
template <> struct Elem<__half> {
  static __device__ __forceinline__ float load(const __half* p) { return __half2float(__ldg(p)); }
  static __device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
  static __device__ __forceinline__ __half from_f32(float x) { return __float2half_rn(x); }
};
template <> struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float load(const __nv_bfloat16* p) { return __bfloat162float(__ldg(p)); }
  static __device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
  static __device__ __forceinline__ __nv_bfloat16 from_f32(float x) { return __float2bfloat16_rn(x); }
};

}  // namespace fa
