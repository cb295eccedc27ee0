/*
 * fa.h -- C ABI of libfa: exact scaled-dot-product attention, forward and
 * backward, in FlashAttention-2 form, for one NVIDIA GB300 (sm_103a).
 *
 * The operation (sources named by page title and section):
 *
 *   S = scale * Q K^T                      per (b, h); Q, K, V are N x D
 *   causal: key j is kept for query i iff j <= i (top-left aligned)
 *       ("FlashAttention-2 from PyTorch to Triton", the kernel's causal
 *        predicate and its test harness)
 *   L_i = log sum_j exp(S_ij)  (natural log)        P = exp(S - L)
 *   O   = P V
 *       ("FlashAttention-2 from PyTorch to Triton", section on the three
 *        running quantities: L_i = m_i + log(l_i), and the backward's
 *        recovery of P as exp(S - L))
 *   Delta_i = sum_d dO_id O_id
 *       ("Triton FlashAttention", project summary: rowsum(dO.O) is computed
 *        by its own small kernel; "FlashAttention-2 from PyTorch to Triton",
 *        defect 5: the precomputed D = rowsum(dO o O))
 *   dV = P^T dO,  dP = dO V^T,  dS = P o (dP - Delta),
 *   dQ = scale dS K,  dK = scale dS^T Q
 *       (the standard softmax-attention gradient; "Triton FlashAttention":
 *        a dK/dV kernel and a dQ kernel, no atomics, P rebuilt from L)
 *
 * Tensors.  Q, K, V, O, dO, dQ, dK, dV are logical [B, H, N, D] arrays of one
 * element type (fa_dtype) addressed through int64 ELEMENT strides given in the
 * order (b, h, n, d).  The d-stride must be 1; the others are free (permuted
 * views such as [B, N, H, D] storage need no copy).  lse and delta are
 * contiguous fp32 [B, H, N] arrays with 16-byte aligned bases.  All pointers
 * are device pointers.
 *
 * Alignment.  Every tensor base must be 16-byte aligned and every b/h/n stride
 * times the element size must be a multiple of 16 bytes (tiles move by TMA).
 *
 * Shapes.  B, H, N >= 1; D in {16, 32, 64, 128}; Q, K and V share N
 * (fa_fwd_ex / fa_bwd_ex below lift this: Nq != Nk, grouped key/value heads,
 * packed variable lengths, dropout).
 * scale must be finite and > 0 (use 1/sqrt(D) for standard attention).
 *
 * Ownership.  The caller allocates every buffer.  The library allocates no
 * device memory per call and keeps no pointer after a call returns.  Inputs are
 * never written.  Outputs are fully overwritten (no accumulate-into
 * semantics; dQ, dK, dV need no zeroing).  Output buffers must not overlap
 * inputs or each other.
 *
 * Ordering.  Calls are asynchronous on `stream`.  fa_fwd -> fa_bwd_preprocess
 * -> fa_bwd must run in that order on one stream (or be ordered by the caller
 * with events).  The return code reports argument and launch errors only;
 * a device-side wait that runs out is reported by fa_get_device_status.
 * The tensor-core backward may run part of its work on a stream of the
 * library's own (one per device, created on first use and kept): that work
 * starts after everything enqueued on `stream` before the call, and `stream`
 * waits for it before anything enqueued after the call, so the call is
 * ordered on `stream` like a single kernel.
 *
 * Precision.  fp16/bf16: products on tensor cores with fp32 accumulation; the
 * probabilities are rounded to the input type before P.V, dS and P^T before
 * the gradient products; O, dQ, dK, dV are rounded to the input type (RNE).
 * fp32: IEEE fp32 FFMA throughout (no TF32).
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { FA_F32 = 0, FA_F16 = 1, FA_BF16 = 2 } fa_dtype;

typedef enum {
  FA_OK = 0,
  FA_ERR_NULL = 1,     /* a required pointer is NULL                          */
  FA_ERR_SHAPE = 2,    /* B, H or N < 1, or the sizes overflow int64          */
  FA_ERR_HEADDIM = 3,  /* D not in {16, 32, 64, 128}                           */
  FA_ERR_DTYPE = 4,    /* unknown fa_dtype                                     */
  FA_ERR_STRIDE = 5,   /* d-stride != 1, or a negative stride                  */
  FA_ERR_ALIGN = 6,    /* base not 16-byte aligned, or stride*size % 16 != 0   */
  FA_ERR_LAUNCH = 7,   /* CUDA reported an error configuring or launching      */
  FA_ERR_TIMEOUT = 8,  /* a device-side bounded wait ran out (see below)       */
  FA_ERR_ARCH = 9,     /* the current device is not sm_103                      */
  FA_ERR_SCALE = 10,   /* scale is not finite and > 0                          */
  FA_ERR_ARG = 11,     /* another invalid argument (e.g. an unknown option)    */
  FA_ERR_SCRATCH = 12, /* B*H*N above FA_NOALLOC_MAX_ROWS (fa_bwd_noalloc) or */
                       /* a workspace or mask buffer too small              */
  FA_ERR_SEQLENS = 13  /* device-reported: packed offsets inconsistent (below) */
} fa_status;

/*
 * Forward.  Writes O (caller strides so) and lse = L [B, H, N] fp32, natural
 * log units: L_i = log sum_j exp(S_ij) over the kept keys.
 * sq, sk, sv, so: 4 int64 element strides each, order (b, h, n, d).
 */
FA_API fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int64_t B, int64_t H, int64_t N, int64_t D,
                 const int64_t* sq, const int64_t* sk, const int64_t* sv,
                 const int64_t* so, int causal, float scale, fa_dtype dtype,
                 cudaStream_t stream);

/*
 * Backward preprocess.  delta[b,h,i] = sum_d dO[b,h,i,d] * O[b,h,i,d], with
 * the products and the sum in fp32, O being the stored forward output.
 */
FA_API fa_status fa_bwd_preprocess(const void* o, const void* dout, float* delta,
                            int64_t B, int64_t H, int64_t N, int64_t D,
                            const int64_t* so, const int64_t* sdo, fa_dtype dtype,
                            cudaStream_t stream);

/*
 * Backward.  From Q, K, V, dO, the forward's lse and the preprocess's delta,
 * writes dQ, dK, dV (strides sdq, sdk, sdv).  P is rebuilt tile by tile as
 * exp(S - L); no N x N matrix is stored.  Runs a dK/dV kernel and a dQ
 * kernel; neither uses atomics.  With both sequence lengths at most 4096 (and
 * `stream` not being captured into a CUDA graph) the tensor-core dQ kernel
 * runs on the library's stream at the same time as the dK/dV kernel (see
 * Ordering above); otherwise the two run one after the other on `stream`.
 */
FA_API fa_status fa_bwd(const void* q, const void* k, const void* v, const void* dout,
                 const float* lse, const float* delta, void* dq, void* dk, void* dv,
                 int64_t B, int64_t H, int64_t N, int64_t D,
                 const int64_t* sq, const int64_t* sk, const int64_t* sv,
                 const int64_t* sdo, const int64_t* sdq, const int64_t* sdk,
                 const int64_t* sdv, int causal, float scale, fa_dtype dtype,
                 cudaStream_t stream);

/*
 * Backward that needs no device buffer beyond inputs and outputs.  The pages
 * that define the method have no counterpart for this entry point; it serves
 * callers that cannot allocate device memory at the point where they run the
 * backward -- for example code executing while a CUDA graph is being
 * captured (cudaMalloc is not allowed then), code inside a framework or
 * plugin that is handed fixed buffers and no allocator, or latency-critical
 * paths that must not take cudaMalloc's implicit synchronisation.
 *
 * Computes exactly what fa_bwd_preprocess followed by fa_bwd computes, with
 * the same argument meanings, layouts and validation, except that the per-row
 * Delta = rowsum(dO o O) is kept in a buffer inside libfa instead of one the
 * caller passes: a fixed device array of FA_NOALLOC_MAX_ROWS floats (16 MiB)
 * that every GPU which loads this part of the library holds until the
 * process exits.  O is the forward output (strides so).  The call allocates
 * nothing (no cudaMalloc, no cudaFree).
 *
 * Limit: B * H * N <= FA_NOALLOC_MAX_ROWS, else FA_ERR_SCRATCH.
 * Errors: the size limit and every argument check of fa_bwd_preprocess and
 * fa_bwd run before any device work, so an invalid call returns its code
 * without creating a context, looking up the buffer or launching anything.
 * Set-up: the first call on a device (with that device current) looks up the
 * buffer's device address once; make that first call before any stream
 * capture begins.
 * Sharing: every call uses the same buffer and leaves its Delta rows in it.
 * Each call writes all the rows it reads before reading them, so nothing
 * needs to start at zero, but calls whose work overlaps on the GPU (for
 * example on two streams at once) race on the buffer: order them.
 */
#define FA_NOALLOC_MAX_ROWS (1 << 22)
FA_API fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                const void* dout, const float* lse, void* dq, void* dk,
                                void* dv, int64_t B, int64_t H, int64_t N, int64_t D,
                                const int64_t* sq, const int64_t* sk, const int64_t* sv,
                                const int64_t* so, const int64_t* sdo, const int64_t* sdq,
                                const int64_t* sdk, const int64_t* sdv, int causal,
                                float scale, fa_dtype dtype, cudaStream_t stream);

/*
 * General problem for fa_fwd_ex / fa_bwd_ex: query and key lengths that
 * differ, fewer key/value heads than query heads, packed variable-length
 * sequences, and dropout of the attention weights.  fa_fwd / fa_bwd are the
 * case Hq = Hkv, Nq = Nk, fixed lengths, no dropout.
 *
 *   B          number of sequences, >= 1
 *   Hq, Hkv    query heads and key/value heads, >= 1, Hq % Hkv == 0.  Query
 *              head h reads key/value head h / (Hq / Hkv): consecutive query
 *              heads share one (grouped-query attention; Hkv = 1 is
 *              multi-query attention).  dK, dV sum over the sharing heads.
 *   Nq, Nk     fixed lengths: the query / key rows of every sequence (>= 1).
 *              Packed: upper bounds on any sequence's rows (>= 1; the grid is
 *              sized by them).
 *   D          head dimension, 16, 32, 64 or 128
 *   cu_seqlens_q, cu_seqlens_k
 *              both NULL: fixed lengths.  Q, O, dO, dQ are [B, Hq, Nq, D];
 *              K, V, dK, dV are [B, Hkv, Nk, D]; lse and delta are fp32
 *              [B, Hq, Nq].
 *              Both set: DEVICE arrays of B+1 int32 offsets into packed rows,
 *              non-decreasing, from >= 0 up to <= total_q / total_k.
 *              Sequence b owns query rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1
 *              of packed tensors [total_q, Hq, D] (pass their strides as a
 *              [1, Hq, total_q, D] view: the b-stride is ignored) and key rows
 *              cu_seqlens_k[b] .. likewise of [total_k, Hkv, D]; lse and delta
 *              are fp32 [Hq, total_q].  A sequence may be empty.  A sequence
 *              whose offsets break these rules (or is longer than Nq / Nk) is
 *              skipped and the kernels record FA_ERR_SEQLENS, which
 *              fa_get_device_status reports; no memory outside the tensors is
 *              touched.
 *   total_q, total_k  packed rows (>= 1); ignored for fixed lengths
 *   causal     key j is kept for query i iff j <= i, both counted from the
 *              sequence's first row (top-left aligned, as for fa_fwd)
 *   scale, dtype  as for fa_fwd
 *   dropout_p  0 <= p < 1.  With p > 0 each attention weight P_ij of query
 *              head h in sequence b is kept iff the 16-bit half (j mod 2;
 *              0 = low) of word ((j mod 8) / 2) of Philox4x32-10 (Salmon,
 *              Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2,
 *              3", SC 2011) with counter (j / 8, i, b*Hq + h, offset) and key
 *              (seed mod 2^32, seed / 2^32) is >= floor(p * 65536); i, j are
 *              positions within the sequence.  Kept weights are scaled by 1 / (1 - p):
 *              O = (P o Z) V with Z_ij = keep_ij / (1 - p).  L stays the
 *              log-sum-exp of the undropped scores.  fa_bwd_ex with the same
 *              seed and offset rebuilds the same mask:
 *              dV = (P o Z)^T dO, dS = P o (Z o (dO V^T) - Delta).
 *   dropout_mask  optional, may be NULL (also for zero-initialised structs
 *              of callers that do not know the field): a DEVICE buffer of at
 *              least fa_dropout_mask_bytes(prob) bytes, 16-byte aligned, that
 *              carries the keep decisions from the forward to the backward.
 *              With dropout_p > 0, fa_fwd_ex stores every decision it draws
 *              there (the bytes fa_dropout_mask would write), and fa_bwd_ex
 *              reads them instead of evaluating the generator again; results
 *              are bitwise identical either way.  So the backward must get a
 *              buffer that a forward (or fa_dropout_mask) of this same problem
 *              (sizes, lengths, causal, dropout_p, seed, offset) filled: it
 *              trusts the contents, and another problem's buffer gives another
 *              mask without an error.  Ignored when dropout_p = 0.
 *              FA_ERR_ALIGN unless 16-byte aligned.
 *
 * Rows with no key at all (an empty key sequence) get O = 0 and L = -inf;
 * keys that no query attends to get dK = dV = 0.
 */
typedef struct fa_problem {
  int64_t B, Hq, Hkv, Nq, Nk, D;
  const int32_t* cu_seqlens_q;
  const int32_t* cu_seqlens_k;
  int64_t total_q, total_k;
  int causal;
  float scale;
  fa_dtype dtype;
  float dropout_p;
  uint64_t seed;
  uint32_t offset;
  uint8_t* dropout_mask;
} fa_problem;

/*
 * Forward for a general problem.  Tensors as described for fa_problem, with
 * 4 element strides each in the order (b, h, n, d) as for fa_fwd.  Validation
 * and error codes as for fa_fwd, plus FA_ERR_SHAPE for Hq % Hkv != 0 or
 * cu_seqlens pointers of which only one is set, and FA_ERR_ARG for dropout_p
 * outside [0, 1).
 */
FA_API fa_status fa_fwd_ex(const fa_problem* prob, const void* q, const int64_t* sq,
                           const void* k, const int64_t* sk, const void* v,
                           const int64_t* sv, void* o, const int64_t* so, float* lse,
                           cudaStream_t stream);

/*
 * Backward for a general problem: dQ, dK, dV from Q, K, V, dO, the forward's
 * lse and delta = rowsum(dO o O) (fa_bwd_preprocess over the Q-shaped rows:
 * B, Hq, Nq for fixed lengths; 1, Hq, total_q for packed ones).  Same problem
 * description (seed and offset included) as the forward call.  Like fa_bwd,
 * runs its dQ kernel on the library's own stream beside the dK/dV kernel when
 * Nq and Nk are at most 4096 and `stream` is not being captured (see
 * Ordering).
 */
FA_API fa_status fa_bwd_ex(const fa_problem* prob, const void* q, const int64_t* sq,
                           const void* k, const int64_t* sk, const void* v,
                           const int64_t* sv, const void* dout, const int64_t* sdo,
                           const float* lse, const float* delta, void* dq,
                           const int64_t* sdq, void* dk, const int64_t* sdk, void* dv,
                           const int64_t* sdv, cudaStream_t stream);

/*
 * Single-pass backward for a general problem (fp16 / bf16 only): the same
 * inputs, outputs and validation as fa_bwd_ex, computed by one kernel per key
 * tile that also produces each tile's share of dQ ("FlashAttention-2 from
 * PyTorch to Triton", defect 5: dQ accumulated by atomics instead of a second
 * pass).  The shares are summed by fp32 bulk reductions into `dq_accum`, a
 * caller-owned DEVICE buffer of at least fa_bwd_fused_workspace_bytes(prob)
 * bytes, 16-byte aligned, which the call zeroes on `stream` and then converts
 * into dq (scaled, rounded to the input type).  The buffer may be reused once
 * the call's work on `stream` has finished; the call allocates nothing.
 *
 * dK and dV are bitwise reproducible; dQ is not, because the order in which
 * key tiles add into a row is not fixed (results differ from run to run by
 * fp32 rounding).  Query rows that belong to no sequence (packed rows past
 * cu_seqlens_q[B] or before cu_seqlens_q[0]) are left untouched, as by
 * fa_bwd_ex.
 *
 * Errors: those of fa_bwd_ex; FA_ERR_DTYPE for FA_F32; FA_ERR_NULL for a NULL
 * dq_accum; FA_ERR_ALIGN for a dq_accum not 16-byte aligned; FA_ERR_SCRATCH
 * when workspace_bytes is below fa_bwd_fused_workspace_bytes(prob).
 */
FA_API size_t fa_bwd_fused_workspace_bytes(const fa_problem* prob);
FA_API fa_status fa_bwd_fused(const fa_problem* prob, const void* q, const int64_t* sq,
                              const void* k, const int64_t* sk, const void* v,
                              const int64_t* sv, const void* dout, const int64_t* sdo,
                              const float* lse, const float* delta, void* dq,
                              const int64_t* sdq, void* dk, const int64_t* sdk, void* dv,
                              const int64_t* sdv, float* dq_accum, size_t workspace_bytes,
                              cudaStream_t stream);

/*
 * Dropout keep mask of a general problem: the decisions stated for dropout_p
 * under fa_problem, 1 bit per (query, key) pair, in the buffer that
 * fa_problem.dropout_mask names.  fa_fwd_ex fills it as it draws the
 * decisions (in warps of its own, beside the softmax); fa_dropout_mask fills
 * it without a forward, e.g. for a backward whose forward ran without one.
 *
 * Layout (callers need not read it): 16 bytes per (flat head, key tile of 128
 * keys, query row), ordered [Bt][Hq][ceil(Nk / 128)][rows][16] with Bt = B,
 * rows = Nq for fixed lengths and Bt = 1, rows = total_q (the packed row) for
 * packed sequences; byte g of key tile t holds the decisions for keys
 * 8(16t + g) .. 8(16t + g) + 7 of the row as bits 0..7 (set: kept).  Written
 * are the entries the kernels read: rows and key tiles inside the row's
 * sequence and, under causal masking, key tiles t <= row / 128.  1/8 byte
 * per (query, key) pair: 1 GiB for 32 heads of 16384 x 16384.
 *
 * fa_dropout_mask_bytes returns the size for `prob`, or 0 when the problem is
 * invalid or has dropout_p = 0.  fa_dropout_mask fills `mask` (a DEVICE
 * buffer of `bytes` bytes) on `stream` and allocates nothing.  Errors: those
 * of fa_fwd_ex's problem checks; FA_ERR_ARG for dropout_p = 0; FA_ERR_NULL
 * for a NULL mask; FA_ERR_ALIGN unless it is 16-byte aligned; FA_ERR_SCRATCH
 * when bytes < fa_dropout_mask_bytes(prob).  prob->dropout_mask is ignored.
 * Packed sequences whose offsets break the rules above are skipped (the
 * forward reports FA_ERR_SEQLENS for them).
 */
FA_API size_t fa_dropout_mask_bytes(const fa_problem* prob);
FA_API fa_status fa_dropout_mask(const fa_problem* prob, uint8_t* mask, size_t bytes,
                                 cudaStream_t stream);

/*
 * Synchronises `stream`, then reads and clears the device status word of the
 * current device.  Returns FA_OK, FA_ERR_TIMEOUT if a kernel's bounded wait on
 * an mbarrier ran out since the last call (that kernel's outputs are then
 * undefined; the CUDA context stays usable), FA_ERR_SEQLENS if a kernel met
 * inconsistent packed offsets, or FA_ERR_LAUNCH if the stream reported a CUDA
 * error.  The first error recorded since the last call wins.
 */
FA_API fa_status fa_get_device_status(cudaStream_t stream);

/* Static, NUL-terminated name of a status code. */
FA_API const char* fa_status_string(fa_status status);

/*
 * Kernel family selection for later calls in this process (for tests and
 * benchmarks; the default is FA_PATH_AUTO).
 *   FA_PATH_AUTO: tensor-core kernels for fp16/bf16 where compiled, FFMA
 *                 kernels otherwise (always for fp32).
 *   FA_PATH_FFMA: the FFMA kernels for every dtype.
 * fa_bwd_fused has tensor-core kernels only and ignores this setting.
 * Returns FA_ERR_ARG for an unknown value.
 */
typedef enum { FA_PATH_AUTO = 0, FA_PATH_FFMA = 1 } fa_path;
FA_API fa_status fa_set_path(fa_path path);

/*
 * Upper bound, in nanoseconds, on any single device-side wait of the
 * tensor-core kernels (default 2e9 = 2 s).  When a wait runs out the kernel
 * records FA_ERR_TIMEOUT, drains its own copies in flight, releases its tensor
 * memory and returns.  0 restores the default.
 */
FA_API void fa_set_wait_timeout_ns(uint64_t ns);

/*
 * Profiling hook for benchmarks.  When `events` is non-NULL its three handles
 * are copied, and every later fa_bwd call records events[0] before its dK/dV
 * kernel, events[1] after the dK/dV kernel, and events[2] after the dQ
 * kernel, on the call's stream.  When the two kernels run at the same time
 * (see fa_bwd), events[1] marks the dK/dV kernel's end and events[2] the end
 * of both, so events[1] -> events[2] is not the dQ kernel's duration.  NULL turns the hook off.  The caller
 * creates and destroys the events and must not destroy them while the hook is
 * on.
 */
FA_API void fa_set_profile_events(const cudaEvent_t* events);

/*
 * Test hook for the device-side failure path.  The next call that runs the
 * tensor-core forward kernel (fa_fwd, fa_fwd_ex) or the single-pass backward
 * (fa_bwd_fused) launches it with one mbarrier arrival withheld in its first
 * CTA, so that CTA's waiting warps wait until the bounded wait
 * (fa_set_wait_timeout_ns) runs out: the kernel then records FA_ERR_TIMEOUT,
 * drains its copies, MMAs and reductions in flight, frees its tensor memory
 * and returns; fa_get_device_status reports FA_ERR_TIMEOUT and the context
 * stays usable.  That call's outputs are undefined.  One-shot: later calls
 * run normally.  Set a short wait bound first (e.g. 50 ms).
 */
FA_API void fa_test_withhold_next_arrival(void);

/*
 * Test hook for the tiled kernels' block order.  The forward, dK/dV and dQ
 * grids take heads in groups whose shared operand (K and V, or Q and dO) fits
 * in part of the L2 cache, so that the CTAs in flight reuse it from L2; a
 * group holds every head when all fit.  With `bytes` > 0 later calls size the
 * groups as if L2 held that many bytes (small values force several groups,
 * and a partial last one, on small problems); 0 restores the device's own
 * size.  The order changes which CTAs run together, never what any CTA
 * computes, so outputs are bitwise the same for every setting.
 */
FA_API void fa_test_set_l2_bytes(int64_t bytes);

/* Library version, e.g. 0x000100 for 0.1.0. */
FA_API int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
