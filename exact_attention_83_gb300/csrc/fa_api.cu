// The C ABI of libfa: argument validation, per-device set-up and dispatch.
//
// Nothing here computes attention; every step of the path runs in the kernels
// of the other translation units.  Validation happens before any launch, so an
// invalid call returns its fa_status without touching the device.

#include "fa_internal.h"

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

// Device status word of the current context.  A kernel whose bounded wait
// runs out stores FA_ERR_TIMEOUT here (first writer wins);
// fa_get_device_status reads and clears it.  A file-scope device variable, so
// the library allocates no device memory.
__device__ unsigned int fa_device_status_word;

namespace fa {
namespace {

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;

std::atomic<int> g_path{FA_PATH_AUTO};
std::atomic<uint64_t> g_timeout_ns{kDefaultTimeoutNs};
std::mutex g_mu;
cudaEvent_t g_prof_events[3];
std::atomic<bool> g_prof_on{false};
std::atomic<int> g_withhold_next{0};   // one-shot test switch (fa_test_withhold_next_arrival)
std::atomic<int64_t> g_l2_override{0};  // test switch (fa_test_set_l2_bytes)
struct DeviceInfo {
  int state = 0;              // 0: not set up, 1: ready, -1: not sm_103
  int sm_count = 0;
  int64_t l2_bytes = 0;
  unsigned int* status = nullptr;
};
DeviceInfo g_dev[kMaxDevices];

// Once per device, with that device current: check the architecture, cache
// the SM count and the device address of the status word.
fa_status device_setup(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_LAUNCH;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (d.state == 0) {
    int major = 0, minor = 0, sms = 0, l2 = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
      return FA_ERR_LAUNCH;
    if (major != 10 || minor != 3) {
      d.state = -1;
    } else {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, fa_device_status_word) != cudaSuccess) return FA_ERR_LAUNCH;
      d.status = static_cast<unsigned int*>(p);
      d.sm_count = sms;
      d.l2_bytes = l2;
      d.state = 1;
    }
  }
  if (d.state < 0) return FA_ERR_ARCH;
  *out = &d;
  return FA_OK;
}

int64_t elem_size(fa_dtype dt) { return dt == FA_F32 ? 4 : 2; }

bool mul_ok(int64_t a, int64_t b, int64_t* r) { return !__builtin_mul_overflow(a, b, r); }

fa_status check_shape(int64_t B, int64_t H, int64_t N, int64_t D, fa_dtype dt) {
  if (dt != FA_F32 && dt != FA_F16 && dt != FA_BF16) return FA_ERR_DTYPE;
  if (B < 1 || H < 1 || N < 1) return FA_ERR_SHAPE;
  if (D != 16 && D != 32 && D != 64 && D != 128) return FA_ERR_HEADDIM;
  int64_t bh, bhn, bhnd;
  if (!mul_ok(B, H, &bh) || !mul_ok(bh, N, &bhn) || !mul_ok(bhn, D * 8, &bhnd)) return FA_ERR_SHAPE;
  if (bh > (int64_t)INT32_MAX || N > (int64_t)INT32_MAX) return FA_ERR_SHAPE;
  return FA_OK;
}

// Checks one [B,H,N,D] tensor and copies its strides into dst.  The stride of
// a dimension of extent 1 is never used; it is replaced by 0.
fa_status check_tensor(const void* p, const int64_t* s, int64_t B, int64_t H, int64_t N,
                       fa_dtype dt, int64_t* dst) {
  if (!p || !s) return FA_ERR_NULL;
  if (s[3] != 1) return FA_ERR_STRIDE;
  const int64_t ext[3] = {B, H, N};
  const int64_t es = elem_size(dt);
  if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return FA_ERR_ALIGN;
  for (int i = 0; i < 3; ++i) {
    if (ext[i] == 1) { dst[i] = 0; continue; }
    if (s[i] < 0) return FA_ERR_STRIDE;
    int64_t bytes;
    if (!mul_ok(s[i], es, &bytes)) return FA_ERR_SHAPE;
    if (bytes % 16 != 0) return FA_ERR_ALIGN;
    dst[i] = s[i];
  }
  dst[3] = 1;
  return FA_OK;
}

fa_status check_f32_vec(const void* p) {
  if (!p) return FA_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return FA_ERR_ALIGN;
  return FA_OK;
}

fa_status check_scale(float scale) {
  return (std::isfinite(scale) && scale > 0.f) ? FA_OK : FA_ERR_SCALE;
}

#define FA_TRY(expr)                   \
  do {                                 \
    const fa_status st_ = (expr);      \
    if (st_ != FA_OK) return st_;      \
  } while (0)

bool use_tc(fa_dtype dt) { return g_path.load() == FA_PATH_AUTO && dt != FA_F32; }

// A validated fa_problem.
struct Problem {
  Geo g;
  int64_t D;
  int causal;
  float scale;
  fa_dtype dtype;
  Dropout drop;
};

fa_status check_problem(const fa_problem* pr, Problem* out) {
  if (!pr) return FA_ERR_NULL;
  const fa_dtype dt = pr->dtype;
  if (dt != FA_F32 && dt != FA_F16 && dt != FA_BF16) return FA_ERR_DTYPE;
  if (pr->B < 1 || pr->Hq < 1 || pr->Hkv < 1 || pr->Nq < 1 || pr->Nk < 1) return FA_ERR_SHAPE;
  if (pr->Hq % pr->Hkv != 0) return FA_ERR_SHAPE;
  const int64_t D = pr->D;
  if (D != 16 && D != 32 && D != 64 && D != 128) return FA_ERR_HEADDIM;
  const bool packed = pr->cu_seqlens_q != nullptr;
  if (packed != (pr->cu_seqlens_k != nullptr)) return FA_ERR_SHAPE;
  if (packed && (pr->total_q < 1 || pr->total_k < 1)) return FA_ERR_SHAPE;
  if (packed && (reinterpret_cast<uintptr_t>(pr->cu_seqlens_q) % 4 != 0 ||
                 reinterpret_cast<uintptr_t>(pr->cu_seqlens_k) % 4 != 0))
    return FA_ERR_ALIGN;
  Geo g{};
  g.B = pr->B; g.Hq = pr->Hq; g.Hkv = pr->Hkv; g.G = pr->Hq / pr->Hkv;
  g.Nq = pr->Nq; g.Nk = pr->Nk;
  g.cu_q = pr->cu_seqlens_q; g.cu_k = pr->cu_seqlens_k;
  g.rows_q = packed ? pr->total_q : pr->Nq;
  g.rows_k = packed ? pr->total_k : pr->Nk;
  g.Bt = packed ? 1 : pr->B;
  // Every element count, and the int32 quantities the kernels use (flat head
  // index, row positions, grid sizes), must fit.
  int64_t t;
  const int64_t heads[2] = {g.Hq, g.Hkv}, rows[2] = {g.rows_q, g.rows_k};
  for (int i = 0; i < 2; ++i)
    if (!mul_ok(g.Bt, heads[i], &t) || !mul_ok(t, rows[i], &t) || !mul_ok(t, D * 8, &t))
      return FA_ERR_SHAPE;
  if (!mul_ok(g.B, g.Hq, &t) || t > (int64_t)INT32_MAX) return FA_ERR_SHAPE;
  // TMA row coordinates are int32 and run up to one tile past the last row.
  const int64_t row_max = (int64_t)INT32_MAX - 1024;
  if (g.rows_q > row_max || g.rows_k > row_max || g.Nq > row_max || g.Nk > row_max)
    return FA_ERR_SHAPE;
  FA_TRY(check_scale(pr->scale));
  const float p = pr->dropout_p;
  if (!(p >= 0.f && p < 1.f)) return FA_ERR_ARG;
  Dropout d{};
  if (p > 0.f) {
    d.on = 1;
    const double thr = std::floor(static_cast<double>(p) * 65536.0);
    d.thr = static_cast<uint32_t>(thr < 65535.0 ? thr : 65535.0);
    d.rscale = static_cast<float>(1.0 / (1.0 - static_cast<double>(p)));
    d.key0 = static_cast<uint32_t>(pr->seed & 0xffffffffu);
    d.key1 = static_cast<uint32_t>(pr->seed >> 32);
    d.offset = pr->offset;
    for (int r = 0; r < 10; ++r) {   // Philox4x32 key schedule (Weyl increments)
      d.rk0[r] = d.key0 + static_cast<uint32_t>(r) * 0x9E3779B9u;
      d.rk1[r] = d.key1 + static_cast<uint32_t>(r) * 0xBB67AE85u;
    }
    if (pr->dropout_mask) {
      if (reinterpret_cast<uintptr_t>(pr->dropout_mask) % 16 != 0) return FA_ERR_ALIGN;
      if (dropout_mask_bytes(g) == 0) return FA_ERR_SHAPE;
      d.mask = pr->dropout_mask;
      d.mask_kt = (g.Nk + 127) / 128;
    }
  }
  out->g = g; out->D = D; out->causal = pr->causal ? 1 : 0; out->scale = pr->scale;
  out->dtype = dt; out->drop = d;
  return FA_OK;
}

fa_status run_fwd(const Problem& pb, const void* q, const int64_t* sq, const void* k,
                  const int64_t* sk, const void* v, const int64_t* sv, void* o,
                  const int64_t* so, float* lse, cudaStream_t stream) {
  FwdParams p{};
  const Geo& g = pb.g;
  FA_TRY(check_tensor(q, sq, g.Bt, g.Hq, g.rows_q, pb.dtype, p.sq));
  FA_TRY(check_tensor(k, sk, g.Bt, g.Hkv, g.rows_k, pb.dtype, p.sk));
  FA_TRY(check_tensor(v, sv, g.Bt, g.Hkv, g.rows_k, pb.dtype, p.sv));
  FA_TRY(check_tensor(o, so, g.Bt, g.Hq, g.rows_q, pb.dtype, p.so));
  FA_TRY(check_f32_vec(lse));
  DeviceInfo* dev = nullptr;
  FA_TRY(device_setup(&dev));
  p.q = q; p.k = k; p.v = v; p.o = o; p.lse = lse;
  p.g = g; p.D = pb.D;
  p.causal = pb.causal; p.scale = pb.scale; p.dtype = pb.dtype; p.drop = pb.drop;
  p.status = dev->status; p.timeout_ns = g_timeout_ns.load();
  if (use_tc(pb.dtype) && have_fwd_tc(pb.D, pb.dtype)) {
    p.withhold_arrival = g_withhold_next.exchange(0);
    return launch_fwd_tc(p, stream);   // stores the keep mask as it draws it
  }
  FA_TRY(launch_fwd_ffma(p, stream));
  // the FFMA forward draws inline and stores nothing: fill the caller's keep
  // mask for the backward
  if (p.drop.on && p.drop.mask != nullptr)
    return launch_dropout_mask(g, pb.causal, p.drop, p.drop.mask, p.status, stream);
  return FA_OK;
}

// Validates the backward's tensors and fills p (everything but the path).
fa_status prepare_bwd(const Problem& pb, const void* q, const int64_t* sq, const void* k,
                      const int64_t* sk, const void* v, const int64_t* sv, const void* dout,
                      const int64_t* sdo, const float* lse, const float* delta, void* dq,
                      const int64_t* sdq, void* dk, const int64_t* sdk, void* dv,
                      const int64_t* sdv, BwdParams* out) {
  BwdParams& p = *out;
  p = BwdParams{};
  const Geo& g = pb.g;
  FA_TRY(check_tensor(q, sq, g.Bt, g.Hq, g.rows_q, pb.dtype, p.sq));
  FA_TRY(check_tensor(k, sk, g.Bt, g.Hkv, g.rows_k, pb.dtype, p.sk));
  FA_TRY(check_tensor(v, sv, g.Bt, g.Hkv, g.rows_k, pb.dtype, p.sv));
  FA_TRY(check_tensor(dout, sdo, g.Bt, g.Hq, g.rows_q, pb.dtype, p.sdo));
  FA_TRY(check_tensor(dq, sdq, g.Bt, g.Hq, g.rows_q, pb.dtype, p.sdq));
  FA_TRY(check_tensor(dk, sdk, g.Bt, g.Hkv, g.rows_k, pb.dtype, p.sdk));
  FA_TRY(check_tensor(dv, sdv, g.Bt, g.Hkv, g.rows_k, pb.dtype, p.sdv));
  FA_TRY(check_f32_vec(lse));
  FA_TRY(check_f32_vec(delta));
  DeviceInfo* dev = nullptr;
  FA_TRY(device_setup(&dev));
  p.q = q; p.k = k; p.v = v; p.dout = dout; p.lse = lse; p.delta = delta;
  p.dq = dq; p.dk = dk; p.dv = dv;
  p.g = g; p.D = pb.D;
  p.causal = pb.causal; p.scale = pb.scale; p.dtype = pb.dtype; p.drop = pb.drop;
  p.status = dev->status; p.timeout_ns = g_timeout_ns.load();
  p.prof = g_prof_on.load() ? g_prof_events : nullptr;
  return FA_OK;
}

fa_status run_bwd(const Problem& pb, const void* q, const int64_t* sq, const void* k,
                  const int64_t* sk, const void* v, const int64_t* sv, const void* dout,
                  const int64_t* sdo, const float* lse, const float* delta, void* dq,
                  const int64_t* sdq, void* dk, const int64_t* sdk, void* dv,
                  const int64_t* sdv, cudaStream_t stream, bool allow_side = true) {
  BwdParams p{};
  FA_TRY(prepare_bwd(pb, q, sq, k, sk, v, sv, dout, sdo, lse, delta, dq, sdq, dk, sdk, dv, sdv,
                     &p));
  p.allow_side = allow_side;
  if (use_tc(pb.dtype) && have_bwd_tc(pb.D, pb.dtype)) return launch_bwd_tc(p, stream);
  return launch_bwd_ffma(p, stream);
}

// fa_problem of the square, equal-heads, fixed-length, no-dropout entry points.
fa_problem square_problem(int64_t B, int64_t H, int64_t N, int64_t D, int causal, float scale,
                          fa_dtype dtype) {
  fa_problem pr{};
  pr.B = B; pr.Hq = H; pr.Hkv = H; pr.Nq = N; pr.Nk = N; pr.D = D;
  pr.causal = causal; pr.scale = scale; pr.dtype = dtype;
  return pr;
}

}  // namespace

fa_status validate_square_bwd(const void* q, const void* k, const void* v, const void* o,
                              const void* dout, const float* lse, const void* dq,
                              const void* dk, const void* dv, int64_t B, int64_t H, int64_t N,
                              int64_t D, const int64_t* sq, const int64_t* sk,
                              const int64_t* sv, const int64_t* so, const int64_t* sdo,
                              const int64_t* sdq, const int64_t* sdk, const int64_t* sdv,
                              int causal, float scale, fa_dtype dtype) {
  FA_TRY(check_shape(B, H, N, D, dtype));
  const fa_problem pr = square_problem(B, H, N, D, causal, scale, dtype);
  Problem pb{};
  FA_TRY(check_problem(&pr, &pb));
  int64_t st[4];
  const void* tensors[8] = {q, k, v, o, dout, dq, dk, dv};
  const int64_t* strides[8] = {sq, sk, sv, so, sdo, sdq, sdk, sdv};
  for (int i = 0; i < 8; ++i) FA_TRY(check_tensor(tensors[i], strides[i], B, H, N, dtype, st));
  return check_f32_vec(lse);
}

int device_sm_count() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < kMaxDevices && g_dev[dev].state == 1) return g_dev[dev].sm_count;
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms > 0 ? sms : 1;
}

// Side stream of each device, for a kernel that may overlap the caller's
// stream (the backward's dQ kernel beside its dK/dV kernel).  One fork/join
// at a time per device: the lock is held from side_begin to side_end, so two
// host threads never interleave the records of the shared events.
struct SideStream {
  std::mutex mu;
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
SideStream g_side[kMaxDevices];

fa_status side_begin(cudaStream_t caller, cudaStream_t* side) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_LAUNCH;
  SideStream& ss = g_side[dev];
  ss.mu.lock();
  if (ss.s == nullptr) {
    cudaStream_t st = nullptr;
    cudaEvent_t f = nullptr, j = nullptr;
    if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&f, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&j, cudaEventDisableTiming) != cudaSuccess) {
      if (j) cudaEventDestroy(j);
      if (f) cudaEventDestroy(f);
      if (st) cudaStreamDestroy(st);
      ss.mu.unlock();
      return FA_ERR_LAUNCH;
    }
    ss.s = st; ss.fork = f; ss.join = j;
  }
  if (cudaEventRecord(ss.fork, caller) != cudaSuccess ||
      cudaStreamWaitEvent(ss.s, ss.fork, 0) != cudaSuccess) {
    ss.mu.unlock();
    return FA_ERR_LAUNCH;
  }
  *side = ss.s;
  return FA_OK;
}

fa_status side_end(cudaStream_t caller) {
  int dev = 0;
  cudaGetDevice(&dev);
  SideStream& ss = g_side[dev];
  const bool ok = cudaEventRecord(ss.join, ss.s) == cudaSuccess &&
                  cudaStreamWaitEvent(caller, ss.join, 0) == cudaSuccess;
  ss.mu.unlock();
  return ok ? FA_OK : FA_ERR_LAUNCH;
}

bool stream_capturing(cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
    cudaGetLastError();          // clear the error; treat as capturing
    return true;
  }
  return cs != cudaStreamCaptureStatusNone;
}

int64_t head_group(int64_t BH, int64_t per_head_bytes) {
  int dev = 0;
  cudaGetDevice(&dev);
  int64_t l2 = 0;
  if (dev >= 0 && dev < kMaxDevices && g_dev[dev].state == 1) {
    l2 = g_dev[dev].l2_bytes;
  } else {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev);
    l2 = v;
  }
  const int64_t forced = g_l2_override.load();
  if (forced > 0) l2 = forced;
  // All heads at once when their operands fit in L2 together (the order is
  // then the plain longest-first one); otherwise groups of 3/8 of L2.
  if (per_head_bytes <= 0 || BH * per_head_bytes <= l2 * 3 / 4) return BH;
  const int64_t g = l2 * 3 / 8 / per_head_bytes;
  return g < 1 ? 1 : (g > BH ? BH : g);
}

fa_status bwd_square(const void* q, const void* k, const void* v, const void* dout,
                     const float* lse, const float* delta, void* dq, void* dk, void* dv,
                     int64_t B, int64_t H, int64_t N, int64_t D, const int64_t* sq,
                     const int64_t* sk, const int64_t* sv, const int64_t* sdo,
                     const int64_t* sdq, const int64_t* sdk, const int64_t* sdv, int causal,
                     float scale, fa_dtype dtype, cudaStream_t stream, bool allow_side) {
  FA_TRY(check_shape(B, H, N, D, dtype));
  const fa_problem pr = square_problem(B, H, N, D, causal, scale, dtype);
  Problem pb{};
  FA_TRY(check_problem(&pr, &pb));
  return run_bwd(pb, q, sq, k, sk, v, sv, dout, sdo, lse, delta, dq, sdq, dk, sdk, dv, sdv,
                 stream, allow_side);
}

}  // namespace fa

using namespace fa;

extern "C" {

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int64_t B, int64_t H, int64_t N, int64_t D,
                 const int64_t* sq, const int64_t* sk, const int64_t* sv,
                 const int64_t* so, int causal, float scale, fa_dtype dtype,
                 cudaStream_t stream) {
  FA_TRY(check_shape(B, H, N, D, dtype));
  const fa_problem pr = square_problem(B, H, N, D, causal, scale, dtype);
  Problem pb{};
  FA_TRY(check_problem(&pr, &pb));
  return run_fwd(pb, q, sq, k, sk, v, sv, o, so, lse, stream);
}

fa_status fa_fwd_ex(const fa_problem* prob, const void* q, const int64_t* sq, const void* k,
                    const int64_t* sk, const void* v, const int64_t* sv, void* o,
                    const int64_t* so, float* lse, cudaStream_t stream) {
  Problem pb{};
  FA_TRY(check_problem(prob, &pb));
  return run_fwd(pb, q, sq, k, sk, v, sv, o, so, lse, stream);
}

fa_status fa_bwd_preprocess(const void* o, const void* dout, float* delta,
                            int64_t B, int64_t H, int64_t N, int64_t D,
                            const int64_t* so, const int64_t* sdo, fa_dtype dtype,
                            cudaStream_t stream) {
  PreParams p{};
  FA_TRY(check_shape(B, H, N, D, dtype));
  FA_TRY(check_tensor(o, so, B, H, N, dtype, p.so));
  FA_TRY(check_tensor(dout, sdo, B, H, N, dtype, p.sdo));
  FA_TRY(check_f32_vec(delta));
  DeviceInfo* dev = nullptr;
  FA_TRY(device_setup(&dev));
  p.o = o; p.dout = dout; p.delta = delta;
  p.B = B; p.H = H; p.N = N; p.D = D; p.dtype = dtype;
  return launch_preprocess(p, stream);
}


fa_status fa_bwd(const void* q, const void* k, const void* v, const void* dout,
                 const float* lse, const float* delta, void* dq, void* dk, void* dv,
                 int64_t B, int64_t H, int64_t N, int64_t D,
                 const int64_t* sq, const int64_t* sk, const int64_t* sv,
                 const int64_t* sdo, const int64_t* sdq, const int64_t* sdk,
                 const int64_t* sdv, int causal, float scale, fa_dtype dtype,
                 cudaStream_t stream) {
  return bwd_square(q, k, v, dout, lse, delta, dq, dk, dv, B, H, N, D, sq, sk, sv, sdo, sdq,
                    sdk, sdv, causal, scale, dtype, stream, true);
}

fa_status fa_bwd_ex(const fa_problem* prob, const void* q, const int64_t* sq, const void* k,
                    const int64_t* sk, const void* v, const int64_t* sv, const void* dout,
                    const int64_t* sdo, const float* lse, const float* delta, void* dq,
                    const int64_t* sdq, void* dk, const int64_t* sdk, void* dv,
                    const int64_t* sdv, cudaStream_t stream) {
  Problem pb{};
  FA_TRY(check_problem(prob, &pb));
  return run_bwd(pb, q, sq, k, sk, v, sv, dout, sdo, lse, delta, dq, sdq, dk, sdk, dv, sdv,
                 stream);
}

size_t fa_dropout_mask_bytes(const fa_problem* prob) {
  Problem pb{};
  if (check_problem(prob, &pb) != FA_OK || !pb.drop.on) return 0;
  return dropout_mask_bytes(pb.g);
}

fa_status fa_dropout_mask(const fa_problem* prob, uint8_t* mask, size_t bytes,
                          cudaStream_t stream) {
  if (!prob) return FA_ERR_NULL;
  fa_problem pr = *prob;
  pr.dropout_mask = nullptr;           // the buffer being filled is not an input
  Problem pb{};
  FA_TRY(check_problem(&pr, &pb));
  if (!pb.drop.on) return FA_ERR_ARG;
  if (!mask) return FA_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(mask) % 16 != 0) return FA_ERR_ALIGN;
  const size_t need = dropout_mask_bytes(pb.g);
  if (need == 0) return FA_ERR_SHAPE;
  if (bytes < need) return FA_ERR_SCRATCH;
  DeviceInfo* dev = nullptr;
  FA_TRY(device_setup(&dev));
  return launch_dropout_mask(pb.g, pb.causal, pb.drop, mask, dev->status, stream);
}

size_t fa_bwd_fused_workspace_bytes(const fa_problem* prob) {
  Problem pb{};
  if (check_problem(prob, &pb) != FA_OK) return 0;
  return bwd_fused_workspace_floats(pb.g, pb.D) * sizeof(float);
}

fa_status fa_bwd_fused(const fa_problem* prob, const void* q, const int64_t* sq, const void* k,
                       const int64_t* sk, const void* v, const int64_t* sv, const void* dout,
                       const int64_t* sdo, const float* lse, const float* delta, void* dq,
                       const int64_t* sdq, void* dk, const int64_t* sdk, void* dv,
                       const int64_t* sdv, float* dq_accum, size_t workspace_bytes,
                       cudaStream_t stream) {
  Problem pb{};
  FA_TRY(check_problem(prob, &pb));
  if (pb.dtype == FA_F32) return FA_ERR_DTYPE;
  if (!dq_accum) return FA_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(dq_accum) % 16 != 0) return FA_ERR_ALIGN;
  if (workspace_bytes < bwd_fused_workspace_floats(pb.g, pb.D) * sizeof(float))
    return FA_ERR_SCRATCH;
  BwdParams p{};
  FA_TRY(prepare_bwd(pb, q, sq, k, sk, v, sv, dout, sdo, lse, delta, dq, sdq, dk, sdk, dv, sdv,
                     &p));
  p.withhold_arrival = g_withhold_next.exchange(0);
  return launch_bwd_fused(p, dq_accum, stream);
}

fa_status fa_get_device_status(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_LAUNCH;
  DeviceInfo* dev = nullptr;
  FA_TRY(device_setup(&dev));
  unsigned int word = 0;
  if (cudaMemcpyFromSymbol(&word, fa_device_status_word, sizeof(word)) != cudaSuccess)
    return FA_ERR_LAUNCH;
  if (word != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(fa_device_status_word, &zero, sizeof(zero)) != cudaSuccess)
      return FA_ERR_LAUNCH;
  }
  return static_cast<fa_status>(word);
}

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_NULL: return "FA_ERR_NULL: a required pointer is NULL";
    case FA_ERR_SHAPE: return "FA_ERR_SHAPE: B, H or N < 1, or sizes overflow";
    case FA_ERR_HEADDIM: return "FA_ERR_HEADDIM: D must be 16, 32, 64 or 128";
    case FA_ERR_DTYPE: return "FA_ERR_DTYPE: unknown dtype";
    case FA_ERR_STRIDE: return "FA_ERR_STRIDE: d-stride must be 1 and strides non-negative";
    case FA_ERR_ALIGN: return "FA_ERR_ALIGN: bases and strides must be 16-byte multiples";
    case FA_ERR_LAUNCH: return "FA_ERR_LAUNCH: CUDA error configuring or launching a kernel";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a device-side bounded wait ran out";
    case FA_ERR_ARCH: return "FA_ERR_ARCH: the current device is not sm_103";
    case FA_ERR_SCALE: return "FA_ERR_SCALE: scale must be finite and > 0";
    case FA_ERR_ARG: return "FA_ERR_ARG: invalid argument";
    case FA_ERR_SCRATCH:
      return "FA_ERR_SCRATCH: B*H*N exceeds FA_NOALLOC_MAX_ROWS, or the workspace is too small";
    case FA_ERR_SEQLENS: return "FA_ERR_SEQLENS: packed sequence offsets are inconsistent";
  }
  return "unknown fa_status";
}

fa_status fa_set_path(fa_path path) {
  if (path != FA_PATH_AUTO && path != FA_PATH_FFMA) return FA_ERR_ARG;
  g_path.store(path);
  return FA_OK;
}

void fa_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns ? ns : kDefaultTimeoutNs); }

void fa_set_profile_events(const cudaEvent_t* events) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (events) {
    for (int i = 0; i < 3; ++i) g_prof_events[i] = events[i];
    g_prof_on.store(true);
  } else {
    g_prof_on.store(false);
  }
}

void fa_test_withhold_next_arrival(void) { g_withhold_next.store(1); }

void fa_test_set_l2_bytes(int64_t bytes) { g_l2_override.store(bytes > 0 ? bytes : 0); }

int fa_version(void) { return 0x000300; }

}  // extern "C"
