// Host side of the TMA copies: encodes 4-D tiled tensor maps over the caller's
// strided [B, H, N, D] tensors (dimensions innermost first: d, n, h, b), so a
// permuted view needs no copy and the zero fill past N stops at the end of
// each head, and 3-D maps over contiguous fp32 row blocks (the dQ workspace
// of the single-pass backward, target of bulk reductions).
// cuTensorMapEncodeTiled is reached through the runtime's driver entry
// point, so libfa needs no link against libcuda.
#include "fa_internal.h"

#include <cudaTypedefs.h>

#include <mutex>

namespace fa {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

bool encode_tile_map(CUtensorMap* map, const void* base, fa_dtype dt, int64_t B, int64_t H,
                     int64_t N, int64_t D, const int64_t* s, uint32_t box_rows,
                     uint32_t box_cols) {
  auto fn = encode_fn();
  if (!fn || dt == FA_F32) return false;
  const uint64_t es = 2;
  // A dimension of extent 1 has stride 0 after validation; any multiple of 16
  // bytes serves there, since its coordinate is always 0.
  uint64_t sn = s[2] ? s[2] * es : static_cast<uint64_t>(D) * es;
  uint64_t sh = s[1] ? s[1] * es : sn * static_cast<uint64_t>(N);
  uint64_t sb = s[0] ? s[0] * es : sh * static_cast<uint64_t>(H);
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {sn, sh, sb};
  cuuint32_t box[4] = {box_cols, box_rows, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType type =
      dt == FA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUresult r = fn(map, type, 4, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_f32_rows_map(CUtensorMap* map, const float* base, int64_t cols, int64_t rows,
                         int64_t planes, uint32_t box_cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(planes)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 4,
                           static_cast<cuuint64_t>(cols) * 4 * static_cast<cuuint64_t>(rows)};
  cuuint32_t box[3] = {box_cols, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace fa
