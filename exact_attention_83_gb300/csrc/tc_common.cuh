// Inline-PTX building blocks for the sm_103a tensor-core kernels: mbarriers,
// TMA tile loads, tcgen05 (tensor memory allocation, MMA, commit, loads and
// stores), shared-memory matrix descriptors and bounded waits.
//
// Encodings follow the PTX ISA for tcgen05:
//  * shared-memory matrix descriptor (64 bit): start address >> 4 in bits
//    0-13, leading-dimension byte offset >> 4 in bits 16-29, stride-dimension
//    byte offset >> 4 in bits 32-45, the fixed value 1 in bits 46-48, base
//    offset 0, swizzle mode in bits 61-63 (2 = 128-byte swizzle);
//  * instruction descriptor for kind::f16 (32 bit): D format in bits 4-5
//    (1 = f32), A format in bits 7-9 and B format in bits 10-12 (0 = f16,
//    1 = bf16), A / B major-ness in bits 15 / 16 (0 = K-major, 1 = MN-major),
//    N >> 3 in bits 17-22, M >> 4 in bits 24-28.
// Tiles are stored the way a TMA load with 128-byte swizzle writes them: rows
// of 128 bytes (64 16-bit elements), 8-row groups 1024 bytes apart, the
// 16-byte chunks of row r XOR-permuted by (r mod 8).  A K-major operand is
// read with SBO = 1024; an MN-major operand with SBO = 1024 between 8-row K
// groups and LBO = the distance between 64-element MN chunks.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "fa_internal.h"

namespace fa {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Raises the transaction count of the barrier's current phase without an
// arrival (the arrivals come separately).
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Per-CTA control block in shared memory.
struct Ctl {
  uint32_t tmem_base;
  volatile int abort;       // set when any wait of this CTA ran out
};

// Bounded wait on phase `parity` of an mbarrier.  Returns true when the phase
// completed.  Returns false when the CTA is aborting (some wait ran out) or
// this wait ran past timeout_ns; in the latter case FA_ERR_TIMEOUT is stored
// in the device status word (first writer wins) and the CTA abort flag is set.
// With honor_abort = false the wait ignores the abort flag (used to drain
// copies in flight before exit).
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, Ctl* ctl,
                                             unsigned int* status, uint64_t timeout_ns,
                                             bool honor_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t spin = 1;; ++spin) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((spin & 31u) == 0) {
      if (honor_abort && ctl->abort) return false;
      if (globaltimer() - t0 > timeout_ns) {
        atomicCAS(status, 0u, static_cast<unsigned int>(FA_ERR_TIMEOUT));
        ctl->abort = 1;
        return false;
      }
    }
  }
}

// Warp-collective form: every lane waits, and the result is made uniform
// across the warp (a lane that gave up makes the whole warp give up), so that
// the warp-collective tcgen05 instructions after it never diverge.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, Ctl* ctl,
                                          unsigned int* status, uint64_t timeout_ns) {
  const bool ok = wait_bounded(bar, parity, ctl, status, timeout_ns);
  return __all_sync(0xffffffffu, ok);
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 4-D tiled load (coordinates innermost first) into shared memory; completion
// is signalled on `bar` as transaction bytes.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t c0, int32_t c1, int32_t c2, int32_t c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// The shared-memory sources of every committed bulk group have been read.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Every committed bulk group has completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy reads (tensor-core operands, TMA sources).
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t x, uint32_t y, uint32_t z,
                                             uint32_t w) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(x), "r"(y), "r"(z),
               "r"(w)
               : "memory");
}
// Barrier `id` (1..15) over `count` threads (a multiple of 32) that also
// returns the AND of every participant's `v`.  Every participating thread
// must reach it, including those whose earlier waits ran out.
__device__ __forceinline__ bool bar_red_and(int id, int count, bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.and.pred p, %2, %3, q;\n"
      " selp.u32 %0, 1, 0, p;\n}" : "=r"(r) : "r"(v ? 1u : 0u), "r"(id), "r"(count) : "memory");
  return r != 0u;
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// One lane of the (fully active) warp, chosen by elect.sync: the issuing
// lane for tensor-core products and commits, whose surrounding loop the whole
// warp runs.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 consecutive 32-bit columns of this thread's lane (warp w reads lanes
// 32*(w%4) .. 32*(w%4)+31; `taddr` carries that lane base).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}


__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

// 16 consecutive 32-bit columns of this thread's lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// Register fence: makes the compiler treat the 32 registers as redefined at
// this point, so no use of a tcgen05.ld destination is scheduled before the
// tcgen05.wait::ld that precedes this call (and no tcgen05.st source is reused
// before the tcgen05.wait::st that precedes it).
__device__ __forceinline__ void reg_fence32(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31])::"memory");
}

__device__ __forceinline__ void reg_fence16(uint32_t (&r)[16]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])::"memory");
}

// ---------------------------------------------------------------- descriptors
// 128-byte-swizzled operand tile in shared memory.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                uint32_t sbo_bytes) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// kind::f16 instruction descriptor with an f32 accumulator.
template <typename T>
constexpr uint32_t idesc_f16(int M, int N, bool a_mn_major, bool b_mn_major) {
  constexpr uint32_t ab = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
  return (1u << 4) | (ab << 7) | (ab << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         ((b_mn_major ? 1u : 0u) << 16) | ((static_cast<uint32_t>(N) >> 3) << 17) |
         ((static_cast<uint32_t>(M) >> 4) << 24);
}

// ---------------------------------------------------------------- packing
template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// prmt.b32: byte n of the result is byte (sel >> 4n) & 7 of {b, a} (a bytes
// 0-3, b bytes 4-7), or, when bit 3 of that nibble is set, that byte's sign
// bit replicated over all 8 bits.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// Mask keeping the 16-bit halves of a packed pair whose flag is set: half 0
// follows bit 7 of byte i0 of {b, a}, half 1 bit 7 of byte i1 (0..7).
__device__ __forceinline__ constexpr uint32_t half_sign_sel(int i0, int i1) {
  return static_cast<uint32_t>((8 | i0) | (8 | i0) << 4 | (8 | i1) << 8 | (8 | i1) << 12);
}

// ---------------------------------------------------------------- clusters
// All threads of every CTA of the cluster (release / acquire).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// ---------------------------------------------------------------- CTA pairs
// cta_group::2 forms of the tensor-core instructions: the two CTAs of a
// cluster of 2 share each MMA (M = 256: rows 0-127 from CTA 0's operands and
// tensor memory, rows 128-255 from CTA 1's; the B operand's N rows are split,
// the first half in CTA 0's shared memory, the second in CTA 1's, at the same
// offset).  Allocation and release are performed by one warp in each CTA; MMAs
// and commits are issued by one thread of CTA 0.  A kernel uses one cta_group
// form throughout.
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void mma_ss_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on the mbarrier at offset `bar` in both CTAs of the pair when
// every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void mma_commit_pair_both(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar), "h"(static_cast<uint16_t>(3))
      : "memory");
}
// The same, on this CTA's barrier only.
__device__ __forceinline__ void mma_commit_pair_local(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
// Arrive (release, cluster scope) on the mbarrier at shared::cluster address
// `remote` (from cluster_map).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t remote) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait (as wait_bounded) on a barrier that threads of the other CTA
// of the cluster also arrive on: acquire at cluster scope.
__device__ __forceinline__ bool wait_bounded_cluster(uint32_t bar, uint32_t parity, Ctl* ctl,
                                                     unsigned int* status, uint64_t timeout_ns,
                                                     bool honor_abort = true) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t spin = 1;; ++spin) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((spin & 31u) == 0) {
      if (honor_abort && ctl->abort) return false;
      if (globaltimer() - t0 > timeout_ns) {
        atomicCAS(status, 0u, static_cast<unsigned int>(FA_ERR_TIMEOUT));
        ctl->abort = 1;
        return false;
      }
    }
  }
}

// Paired fp32 arithmetic (two fp32 lanes in one 64-bit register; one
// instruction does both) and the three-input maximum.
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f32x2_split(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace tc
}  // namespace fa

namespace fa {
namespace tc {

// Epilogue staging: `ncols` (a multiple of 32) fp32 columns of this thread's
// TMEM lane starting at taddr, times `mul`, rounded to T, written as columns
// col0 .. col0 + ncols - 1 (col0 a multiple of 32) of row `row` of a
// shared-memory tile laid out as the 128-byte-swizzled loads are (64-column
// chunks of 128 rows x 128 bytes, chunk c at tile + c * 16384, 16-byte unit u
// of a row at unit u ^ (row % 8)); a warp's eight-row groups cover all banks.
template <typename T>
__device__ __forceinline__ void stage_row_sw128(uint32_t taddr, float mul, uint32_t tile, int row,
                                                int col0, int ncols) {
  for (int c = 0; c < ncols; c += 32) {
    uint32_t t[32];
    tmem_ld32(taddr + c, t);
    tmem_wait_ld();
    reg_fence32(t);
    const int col = col0 + c;
    const uint32_t rbase = tile + static_cast<uint32_t>(col / 64) * 16384u + static_cast<uint32_t>(row) * 128u;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int u = ((col % 64) / 8) + v, e = 8 * v;
      st_shared_v4(rbase + static_cast<uint32_t>((u ^ (row & 7)) * 16),
                   pack2<T>(__uint_as_float(t[e]) * mul, __uint_as_float(t[e + 1]) * mul),
                   pack2<T>(__uint_as_float(t[e + 2]) * mul, __uint_as_float(t[e + 3]) * mul),
                   pack2<T>(__uint_as_float(t[e + 4]) * mul, __uint_as_float(t[e + 5]) * mul),
                   pack2<T>(__uint_as_float(t[e + 6]) * mul, __uint_as_float(t[e + 7]) * mul));
    }
  }
}

// Stores a tile staged by stage_row_sw128 (`ncols` columns, 128 rows) from
// shared memory to global memory, thread t of `nthreads` taking every
// nthreads-th 16-byte unit: consecutive threads write consecutive units of a
// row, so a warp's store covers whole lines.  Rows at or past `nrows` and
// columns at or past `dreal` (a multiple of 8) are not written.
template <typename T>
__device__ __forceinline__ void store_staged_tile(uint32_t tile, int ncols, int t, int nthreads,
                                                  T* row0, int64_t row_stride, int nrows,
                                                  int dreal) {
  const int units = ncols / 8;   // 16-byte units per row
  for (int j = t; j < 128 * units; j += nthreads) {
    const int r = j / units, u = j % units;
    if (r < nrows && 8 * u < dreal) {
      uint32_t x, y, z, w;
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(x), "=r"(y), "=r"(z), "=r"(w)
                   : "r"(tile + static_cast<uint32_t>((u >> 3) * 16384 + r * 128 +
                                                      (((u & 7) ^ (r & 7)) * 16))));
      *reinterpret_cast<uint4*>(row0 + r * row_stride + 8 * u) = make_uint4(x, y, z, w);
    }
  }
}

// Epilogue store: `ncols` (a multiple of 16, at most 128, uniform across the
// warp) fp32 columns of this thread's TMEM lane starting at taddr, times
// `mul`, rounded to T and written to `row` (16-byte vector stores) when
// `store`.  Used with ncols < the accumulator width when a narrow head
// dimension runs zero-padded through a wider kernel.
template <typename T>
__device__ __forceinline__ void store_row_cols(uint32_t taddr, float mul, T* row, bool store,
                                               int ncols) {
  int c = 0;
  // 64 columns per wait: two loads in flight, one latency
  for (; c + 64 <= ncols; c += 64) {
    uint32_t t0[32], t1[32];
    tmem_ld32(taddr + c, t0);
    tmem_ld32(taddr + c + 32, t1);
    tmem_wait_ld();
    reg_fence32(t0);
    reg_fence32(t1);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const uint32_t* t = hh ? t1 : t0;
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        w[i] = pack2<T>(__uint_as_float(t[2 * i]) * mul, __uint_as_float(t[2 * i + 1]) * mul);
      if (store) {
        uint4* dst = reinterpret_cast<uint4*>(row + c + 32 * hh);
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4)
          dst[v4] = make_uint4(w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
      }
    }
  }
  for (; c + 32 <= ncols; c += 32) {
    uint32_t t[32];
    tmem_ld32(taddr + c, t);
    tmem_wait_ld();
    reg_fence32(t);
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      w[i] = pack2<T>(__uint_as_float(t[2 * i]) * mul, __uint_as_float(t[2 * i + 1]) * mul);
    if (store) {
      uint4* dst = reinterpret_cast<uint4*>(row + c);
#pragma unroll
      for (int v4 = 0; v4 < 4; ++v4)
        dst[v4] = make_uint4(w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
    }
  }
  if (c < ncols) {   // 16 columns left
    uint32_t t[16];
    tmem_ld16(taddr + c, t);
    tmem_wait_ld();
    reg_fence16(t);
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      w[i] = pack2<T>(__uint_as_float(t[2 * i]) * mul, __uint_as_float(t[2 * i + 1]) * mul);
    if (store) {
      uint4* dst = reinterpret_cast<uint4*>(row + c);
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
  }
}

}  // namespace tc
}  // namespace fa
