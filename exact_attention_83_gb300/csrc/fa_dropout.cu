// Dropout keep mask drawn without a forward (fa_dropout_mask).
//
// The attention weights' keep decisions (Philox4x32-10 at counter
// (key group, query row, flat head, offset), FlashAttention-2's dropout of P
// regenerated from the seed in the backward) depend on positions only.  The
// tensor-core forward stores the decisions it draws in the caller's keep
// mask, so that the dK/dV and dQ kernels read 1 bit per weight instead of
// evaluating the generator again; this kernel writes the same bytes for a
// backward whose forward kept none.
//
// Work items are (flat head, query tile of 128 rows, key tile of 128 keys):
// a CTA of 128 threads takes one item at a time (one thread per query row,
// 16 generator calls, one 16-byte store), over a grid of a few CTAs per SM
// striding through the items.  Under causal masking items with key tile >
// query tile are skipped: no kernel reads them.

#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kRows = 128;   // query rows per item = threads per CTA
constexpr int kKeys = 128;   // keys per key tile

struct MaskArgs {
  Geo g;
  Dropout drop;
  uint8_t* mask;
  int64_t QT, KT, items;     // query tiles, key tiles per head; QT * KT * B * Hq
  int causal;
  unsigned int* status;
};

__global__ void __launch_bounds__(kRows) dropout_mask_kernel(const __grid_constant__ MaskArgs a) {
  const bool narrow = a.items <= 0xFFFFFFFFll;     // 32-bit index arithmetic suffices
  for (int64_t f = blockIdx.x; f < a.items; f += gridDim.x) {
    int64_t jt, qt, bh;                             // bh = b * Hq + h, b the sequence
    if (narrow) {
      const uint32_t u = static_cast<uint32_t>(f), kt = static_cast<uint32_t>(a.KT),
                     nqt = static_cast<uint32_t>(a.QT);
      const uint32_t t = u / kt, hb = t / nqt;
      jt = u - t * kt; qt = t - hb * nqt; bh = hb;
    } else {
      jt = f % a.KT; qt = (f / a.KT) % a.QT; bh = f / (a.KT * a.QT);
    }
    if (a.causal && jt > qt) continue;
    const SeqView sv = seq_view(a.g, bh / a.g.Hq);
    if (!sv.ok) {
      if (threadIdx.x == 0 && qt == 0 && jt == 0) record_status(a.status, FA_ERR_SEQLENS);
      continue;
    }
    const int64_t row = qt * kRows + threadIdx.x;
    if (row >= sv.nq || jt * kKeys >= sv.nk) continue;
    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int g8 = 0; g8 < 16; ++g8)
      w[g8 >> 2] |= keep8(a.drop, static_cast<uint32_t>(jt * 16 + g8), static_cast<uint32_t>(row),
                          static_cast<uint32_t>(bh))
                    << (8 * (g8 & 3));
    const int64_t off = mask_entry(a.drop, a.g, sv, bh % a.g.Hq, jt, row);
    *reinterpret_cast<uint4*>(a.mask + off) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

}  // namespace

size_t dropout_mask_bytes(const Geo& g) {
  const int64_t kt = (g.Nk + kKeys - 1) / kKeys;
  const double approx = static_cast<double>(g.Bt) * g.Hq * kt * g.rows_q * 16.0;
  if (approx > 9.0e18) return 0;
  return static_cast<size_t>(g.Bt * g.Hq * kt * g.rows_q * 16);
}

fa_status launch_dropout_mask(const Geo& g, int causal, const Dropout& d, uint8_t* mask,
                              unsigned int* status, cudaStream_t s) {
  MaskArgs a{};
  a.g = g;
  a.drop = d;
  a.mask = mask;
  a.QT = (g.Nq + kRows - 1) / kRows;
  a.KT = (g.Nk + kKeys - 1) / kKeys;
  a.drop.mask = nullptr;
  a.drop.mask_kt = a.KT;            // the entry layout the readers use
  a.items = a.QT * a.KT * g.B * g.Hq;
  a.causal = causal;
  a.status = status;
  if (static_cast<double>(a.QT) * static_cast<double>(a.KT) * static_cast<double>(g.B) *
          static_cast<double>(g.Hq) > 9.0e18)
    return FA_ERR_SHAPE;
  if (a.items == 0) return FA_OK;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
  const int64_t blocks = a.items < cap ? a.items : cap;
  dropout_mask_kernel<<<dim3(static_cast<unsigned>(blocks)), dim3(kRows), 0, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

}  // namespace fa
