// fa_bwd_noalloc: the backward for callers that cannot allocate device memory.
//
// The regular backward asks the caller for a Delta buffer (one float per query
// row) that lives only between fa_bwd_preprocess and fa_bwd.  Some callers
// cannot provide it because they cannot allocate at that point: code running
// during CUDA graph capture, plugins that receive fixed buffers and no
// allocator, or latency-critical paths that must avoid cudaMalloc's implicit
// synchronisation.  This entry point keeps Delta in a fixed device array that
// belongs to the library instead, and otherwise runs the same preprocess,
// dK/dV and dQ kernels through the existing entry points.
#include "fa_internal.h"

#include <mutex>

namespace {

constexpr int64_t kMaxRows = FA_NOALLOC_MAX_ROWS;   // 16 MiB of fp32

// Library-owned Delta rows.  In host code this name is only a stand-in for
// the device array; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) float fa_noalloc_delta[kMaxRows];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float* g_delta[kMaxDevices];   // device address per device, looked up once

// Once per device, with that device current: the device address of the array.
fa_status scratch_delta(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_LAUNCH;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_delta[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, fa_noalloc_delta) != cudaSuccess || !p) return FA_ERR_LAUNCH;
    g_delta[dev] = static_cast<float*>(p);
  }
  *out = g_delta[dev];
  return FA_OK;
}

}  // namespace

extern "C" fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                    const void* dout, const float* lse, void* dq, void* dk,
                                    void* dv, int64_t B, int64_t H, int64_t N, int64_t D,
                                    const int64_t* sq, const int64_t* sk, const int64_t* sv,
                                    const int64_t* so, const int64_t* sdo, const int64_t* sdq,
                                    const int64_t* sdk, const int64_t* sdv, int causal,
                                    float scale, fa_dtype dtype, cudaStream_t stream) {
  // Every check comes before any device work: an invalid call neither creates
  // a context, nor looks up the array, nor launches anything (so it leaves no
  // stray node in a graph being captured and never writes the shared array).
  if (B < 1 || H < 1 || N < 1) return FA_ERR_SHAPE;
  int64_t bh = 0, rows = 0;
  if (__builtin_mul_overflow(B, H, &bh) || __builtin_mul_overflow(bh, N, &rows)) return FA_ERR_SHAPE;
  if (rows > kMaxRows) return FA_ERR_SCRATCH;
  const fa_status valid = fa::validate_square_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, D,
                                                  sq, sk, sv, so, sdo, sdq, sdk, sdv, causal,
                                                  scale, dtype);
  if (valid != FA_OK) return valid;
  float* delta = nullptr;
  const fa_status st = scratch_delta(&delta);
  if (st != FA_OK) return st;
  // The preprocess writes Delta for every one of the B*H*N rows the backward
  // reads, so stale contents of the array are never used.
  const fa_status pre = fa_bwd_preprocess(o, dout, delta, B, H, N, D, so, sdo, dtype, stream);
  if (pre != FA_OK) return pre;
  // In sequence on `stream`: this entry point creates nothing, not even the
  // side stream fa_bwd may use.
  return fa::bwd_square(q, k, v, dout, lse, delta, dq, dk, dv, B, H, N, D, sq, sk, sv, sdo, sdq, sdk,
                    sdv, causal, scale, dtype, stream, false);
}
