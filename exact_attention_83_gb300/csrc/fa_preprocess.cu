// Backward preprocess: Delta_i = sum_d dO_id * O_id for every row.
//
// "Triton FlashAttention" (project summary) computes rowsum(dO.O) in its own
// small kernel; "FlashAttention-2 from PyTorch to Triton" (defect 5) names the
// same precomputed D = rowsum(dO o O).  The products and the sum are fp32; O
// is the stored (rounded) forward output.
//
// The kernel is HBM-bound: it reads 2 * N * D elements per head and writes
// N floats.  Each thread reads one 16-byte vector of O and one of dO (8
// fp16/bf16 or 4 fp32 elements); the D / VEC threads of a row reduce with
// shuffles.  A grid-stride loop over rows keeps the grid at a multiple of the
// SM count.

#include "fa_internal.h"

namespace fa {
namespace {

template <typename T>
__device__ __forceinline__ float dot16B(const uint4& x, const uint4& y);

template <>
__device__ __forceinline__ float dot16B<float>(const uint4& x, const uint4& y) {
  float acc = __uint_as_float(x.x) * __uint_as_float(y.x);
  acc = fmaf(__uint_as_float(x.y), __uint_as_float(y.y), acc);
  acc = fmaf(__uint_as_float(x.z), __uint_as_float(y.z), acc);
  acc = fmaf(__uint_as_float(x.w), __uint_as_float(y.w), acc);
  return acc;
}

template <typename H2>
__device__ __forceinline__ float2 unpack2(uint32_t w);
template <>
__device__ __forceinline__ float2 unpack2<__half2>(uint32_t w) {
  __half2 h = *reinterpret_cast<__half2*>(&w);
  return __half22float2(h);
}
template <>
__device__ __forceinline__ float2 unpack2<__nv_bfloat162>(uint32_t w) {
  __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&w);
  return __bfloat1622float2(h);
}

template <typename H2>
__device__ __forceinline__ float dot16B_h(const uint4& x, const uint4& y) {
  const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 a = unpack2<H2>(xs[i]), b = unpack2<H2>(ys[i]);
    acc = fmaf(a.x, b.x, acc);
    acc = fmaf(a.y, b.y, acc);
  }
  return acc;
}
template <>
__device__ __forceinline__ float dot16B<__half>(const uint4& x, const uint4& y) { return dot16B_h<__half2>(x, y); }
template <>
__device__ __forceinline__ float dot16B<__nv_bfloat16>(const uint4& x, const uint4& y) { return dot16B_h<__nv_bfloat162>(x, y); }

struct PreArgs {
  const void* o; const void* dout; float* delta;
  int64_t H, N, rows;
  int64_t so[4], sdo[4];
};

template <typename T, int D>
__global__ void __launch_bounds__(256) preprocess_kernel(PreArgs a) {
  constexpr int VEC = 16 / sizeof(T);
  constexpr int TPR = D / VEC;                 // threads per row (2 .. 32)
  constexpr int ROWS_PER_BLOCK = 256 / TPR;
  const int sub = threadIdx.x % TPR;
  const int64_t stride = (int64_t)gridDim.x * ROWS_PER_BLOCK;
  // The loop bound is uniform across the block so every lane reaches the
  // shuffles below.
  for (int64_t base = (int64_t)blockIdx.x * ROWS_PER_BLOCK; base < a.rows; base += stride) {
    const int64_t row = base + threadIdx.x / TPR;
    float acc = 0.f;
    const bool valid = row < a.rows;
    if (valid) {
      const int64_t bh = row / a.N, i = row % a.N, b = bh / a.H, h = bh % a.H;
      const T* o = static_cast<const T*>(a.o) + b * a.so[0] + h * a.so[1] + i * a.so[2] + sub * VEC;
      const T* g = static_cast<const T*>(a.dout) + b * a.sdo[0] + h * a.sdo[1] + i * a.sdo[2] + sub * VEC;
      const uint4 x = __ldg(reinterpret_cast<const uint4*>(o));
      const uint4 y = __ldg(reinterpret_cast<const uint4*>(g));
      acc = dot16B<T>(x, y);
    }
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (valid && sub == 0) a.delta[row] = acc;
  }
}

template <typename T, int D>
fa_status run(const PreArgs& a, cudaStream_t s) {
  constexpr int VEC = 16 / sizeof(T);
  constexpr int ROWS_PER_BLOCK = 256 / (D / VEC);
  const int64_t need = (a.rows + ROWS_PER_BLOCK - 1) / ROWS_PER_BLOCK;
  const int64_t cap = (int64_t)device_sm_count() * 8;
  const int64_t blocks = need < cap ? need : cap;
  preprocess_kernel<T, D><<<dim3((unsigned)blocks), dim3(256), 0, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

}  // namespace

fa_status launch_preprocess(const PreParams& p, cudaStream_t s) {
  PreArgs a{};
  a.o = p.o; a.dout = p.dout; a.delta = p.delta;
  a.H = p.H; a.N = p.N; a.rows = p.B * p.H * p.N;
  for (int i = 0; i < 4; ++i) { a.so[i] = p.so[i]; a.sdo[i] = p.sdo[i]; }
  switch (p.dtype) {
    case FA_F32:
      switch (p.D) { case 16: return run<float, 16>(a, s); case 32: return run<float, 32>(a, s);
                     case 64: return run<float, 64>(a, s); case 128: return run<float, 128>(a, s); }
      break;
    case FA_F16:
      switch (p.D) { case 16: return run<__half, 16>(a, s); case 32: return run<__half, 32>(a, s);
                     case 64: return run<__half, 64>(a, s); case 128: return run<__half, 128>(a, s); }
      break;
    case FA_BF16:
      switch (p.D) { case 16: return run<__nv_bfloat16, 16>(a, s); case 32: return run<__nv_bfloat16, 32>(a, s);
                     case 64: return run<__nv_bfloat16, 64>(a, s); case 128: return run<__nv_bfloat16, 128>(a, s); }
      break;
  }
  return FA_ERR_ARG;
}

}  // namespace fa
