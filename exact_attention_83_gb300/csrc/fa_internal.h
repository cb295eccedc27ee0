// Internal declarations shared by the translation units of libfa.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "../../include/fa.h"

namespace fa {

// Parameters of one forward call, validated by the ABI layer.
struct FwdParams {
  const void* q; const void* k; const void* v;
  void* o; float* lse;
  int64_t B, H, N, D;
  int64_t sq[4], sk[4], sv[4], so[4];   // element strides (b, h, n, d), d == 1
  int causal;
  float scale;
  fa_dtype dtype;
  unsigned int* status;   // device status word (FA_ERR_TIMEOUT on a wait that ran out)
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
  int64_t B, H, N, D;
  int64_t sq[4], sk[4], sv[4], sdo[4], sdq[4], sdk[4], sdv[4];
  int causal;
  float scale;
  fa_dtype dtype;
  unsigned int* status;
  uint64_t timeout_ns;
  const cudaEvent_t* prof;   // 3 events to record around the two kernels, or null
};

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

// Encodes a 4-D tiled TMA map (d, n, h, b) over a strided [B,H,N,D] fp16/bf16
// tensor with 128-byte swizzle and a box of box_cols x box_rows elements.
bool encode_tile_map(CUtensorMap* map, const void* base, fa_dtype dt, int64_t B, int64_t H,
                     int64_t N, int64_t D, const int64_t* strides, uint32_t box_rows,
                     uint32_t box_cols);

// Number of SMs of the current device (cached per device).
int device_sm_count();

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
