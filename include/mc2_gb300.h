/*
 * mc2_gb300.h -- C ABI of the GB300 (sm_103a) MC2 fused-linear library.
 *
 * The compute hot paths of the communication-compute fused operations:
 * AllGatherMatmul, AlltoAllQuantMatmul, MatmulReduceScatter (with the weight
 * gradient of the fused linear layers) and QuantAllReduce.  The world_size
 * (rankSize) shards that a collective would deliver are separate device
 * buffers on one GPU; the library reads them in place and never runs a
 * collective.
 *
 * Conventions shared by every call
 *   - Every tensor is a DEVICE pointer, row-major and contiguous, owned by the
 *     caller.  Arrays of per-rank pointers (x_chunks, chunks) are HOST arrays
 *     of device pointers.  Every device pointer must address memory of the
 *     CUDA device current on the calling thread, and `stream` must belong to
 *     that device: the library launches there and does not look up where a
 *     pointer lives (that would be a driver query per pointer per call).
 *   - Each buffer must hold at least the elements that the sizes passed with
 *     it imply, in the stated dtype.  The library sees bare pointers and
 *     cannot check this: a smaller buffer is read or written past its end.
 *     (The Python binding checks every tensor's shape and dtype first.)
 *   - Work is enqueued on `stream` (a cudaStream_t passed as void*; NULL is the
 *     legacy default stream) and the call returns without synchronising.  The
 *     library never allocates device memory: scratch space is the caller's
 *     `workspace`.  The one exception is mc2_alltoall_quant_mm_no_alloc, which
 *     uses a fixed scratch array built into the library (see there).
 *   - Arguments are validated before anything is launched.  A violated
 *     constraint returns a negative mc2_status and launches nothing;
 *     mc2_last_error() then describes which argument failed (thread-local).
 *   - Outputs are deterministic: the same inputs give the same bits on every
 *     call.  The float paths compute each output tile whole in one CTA pair.
 *     The integer GEMM of mc2_alltoall_quant_mm splits the tiles of its last
 *     partial wave by K blocks ("stream-K"): the parts that do not end a tile
 *     write exact int32 partial sums to the workspace and publish them on
 *     per-tile flags with atomic compare-and-swap, and the part that ends the
 *     tile adds them.  Integer sums are exact in any order, so the result is
 *     bit-identical to whole tiles.
 *   - Pointers must be 16-byte aligned and row pitches multiples of 16 bytes
 *     (the tensor-memory-accelerator copies need it); otherwise
 *     MC2_ERR_UNSUPPORTED.
 */
#ifndef MC2_GB300_H
#define MC2_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MC2_OK = 0,
    MC2_ERR_NULL = -1,        /* a required pointer is NULL */
    MC2_ERR_SHAPE = -2,       /* a size breaks a constraint of the op */
    MC2_ERR_DTYPE = -3,       /* a dtype or quant-mode combination is not allowed */
    MC2_ERR_UNSUPPORTED = -4, /* allowed by the op but not by this kernel (alignment, box shape) */
    MC2_ERR_WORKSPACE = -5,   /* workspace missing or smaller than the query returned */
    MC2_ERR_CUDA = -6,        /* a CUDA runtime/driver call failed (no device, launch error) */
    MC2_ERR_TIMEOUT = -7      /* a bounded device-side wait gave up (see mc2_device_status) */
} mc2_status;

typedef enum {
    MC2_F16 = 1,
    MC2_BF16 = 2,
    MC2_F32 = 3,
    MC2_I8 = 4,
    MC2_F8E4M3 = 5,   /* fp8 E4M3FN: bias 7, no infinities, S.1111.111 is NaN */
    MC2_F8E5M2 = 6,   /* fp8 E5M2: bias 15, IEEE-style infinities and NaNs */
    MC2_E8M0 = 7      /* mx scale: an unsigned biased exponent, value 2^(code - 127), 0xFF is NaN */
} mc2_dtype;

/* Quant-mode enumeration of "aclnnAlltoAllQuantMatmul" (函数原型, the
 * x1QuantMode / x2QuantMode / commQuantMode values). */
typedef enum {
    MC2_QUANT_NONE = 0,
    MC2_QUANT_PERTENSOR = 1,
    MC2_QUANT_PERCHANNEL = 2,
    MC2_QUANT_PERTOKEN = 3,
    MC2_QUANT_PERGROUP = 4,
    MC2_QUANT_PERBLOCK = 5,
    MC2_QUANT_MX = 6,
    MC2_QUANT_PERTOKEN_DYNAMIC = 7
} mc2_quant_mode;

/*
 * AllGatherMatmul  ("torch_npu.npu_all_gather_base_mm": 功能说明, 接口原型,
 * 输出说明, 约束说明; x2 passed as w^T as in hyper_parallel mc2.py
 * AllGatherMatmulFunction.forward).
 *
 *   gathered = concat_m(x_chunks[0], ..., x_chunks[world_size-1])   (m, k)
 *   out      = gathered @ x2 (+ bias)                                (m, n)
 *   m = world_size * m_local.  Accumulation is fp32; out is rounded once
 *   (nearest-even) to `dtype`.  bias, if given, is added in fp32 before the
 *   rounding.
 *
 *   x_chunks      host array of world_size device pointers, each (m_local, k);
 *                 chunks that lie back to back (x_chunks[r] = x_chunks[0] +
 *                 r * m_local * k elements, the slices of one receive buffer)
 *                 are read faster when m_local < 128: through one tensor map,
 *                 in 128-row boxes, instead of one small box per chunk
 *   world_size    2, 4 or 8
 *   m_local       rows per rank, >= 1 (this kernel: a multiple of 8)
 *   k             contraction size, 256 <= k < 65535 (this kernel: k % 8 == 0)
 *   x2            (k, n) row-major, or with x2_is_nk != 0 the nn.Linear weight
 *                 w (n, k) row-major such that x2 = w^T
 *   n             output columns, >= 1 (this kernel: n % 8 == 0)
 *   bias          NULL or (n) of `dtype`
 *   dtype         MC2_F16 or MC2_BF16, the type of chunks, x2, bias and out
 *   gather_output nonzero: also write `gathered` (m, k); zero: gathered must be NULL
 *   out           (m, n) of `dtype`
 *
 * Returns MC2_OK or a negative mc2_status; nothing is launched on error.
 */
int mc2_all_gather_mm(const void *const *x_chunks, int world_size, int64_t m_local, int64_t k,
                      const void *x2, int64_t n, int x2_is_nk, const void *bias, int dtype,
                      int gather_output, void *out, void *gathered, void *stream);

/*
 * MatmulReduceScatter  (hyper_parallel mc2.py, module docstring:
 * matmul_reduce_scatter forward Y = ReduceScatter_m(X @ W^T), the dual of
 * AllGatherMatmul; MatmulReduceScatterFunction.forward passes w.t()).  Rank r
 * holds its activations X_r (m, k_local) and its weight shard W_r; the ranks'
 * partial products are summed and the sum's row blocks scattered:
 *
 *   Y      = sum_r X_r @ W_r^T                                  (m, n)
 *   out_j  = Y[j*m/R : (j+1)*m/R, :] (+ bias)                   rank j's output
 *
 *   The sum over ranks and k is accumulated in fp32 (blocks of 1024 k summed
 *   in fp32 registers) and rounded once (nearest-even) to `dtype`; bias, if
 *   given, is added in fp32 before the rounding.
 *
 *   x_chunks    host array of world_size device pointers, each (m, k_local)
 *   w_chunks    host array of world_size device pointers: w (n, k_local)
 *               row-major (w_is_nk != 0, the nn.Linear layout) or x2 = w^T
 *               (k_local, n) row-major (w_is_nk == 0)
 *   world_size  2, 4 or 8;  m % world_size == 0
 *   k_local     256 <= k_local < 65535 (this kernel: k_local % 64 == 0)
 *   n           >= 1 (this kernel: n % 8 == 0)
 *   bias        NULL or (n) of `dtype`
 *   dtype       MC2_F16 or MC2_BF16 for every tensor
 *   out_chunks  host array of world_size device pointers, each (m/world_size, n)
 *
 * Returns MC2_OK or a negative mc2_status; nothing is launched on error.
 */
int mc2_matmul_reduce_scatter(const void *const *x_chunks, const void *const *w_chunks, int world_size, int64_t m,
                              int64_t k_local, int64_t n, int w_is_nk, const void *bias, int dtype,
                              void *const *out_chunks, void *stream);

/*
 * Weight and bias gradients of the fused linear layers  (hyper_parallel
 * mc2.py, module docstring: all_gather_matmul backward dW = dY^T @
 * AllGather_m(X), matmul_reduce_scatter backward dW = AllGather_m(dY)^T @ X;
 * AllGatherMatmulFunction.backward: grad_w = grad_out.t().matmul(gathered),
 * grad_bias = grad_out.sum(dim=0)).  The all-gathered operand is the one the
 * forward call returned (the `gathered` output of mc2_all_gather_mm).
 *
 *   dw[i, j] = sum_t dy[t, i] * x[t, j]        (n, k), the nn.Linear weight layout
 *   db[i]    = sum_t dy[t, i]                  (n)
 *
 *   Both sums are accumulated in fp32 (dw in blocks of 1024 rows summed in fp32
 *   registers; db in the same launch, from the dY tiles the GEMM has in shared
 *   memory, as four interleaved row partials added at the end) and rounded once
 *   (nearest-even) to `dtype`.
 *
 *   dy     (m, n) row-major          x    (m, k) row-major
 *   dw     (n, k) row-major          db   NULL or (n)
 *   dtype  MC2_F16 or MC2_BF16 for every tensor
 *   m, n, k >= 1 and <= INT32_MAX  (this kernel: n % 8 == 0, k % 8 == 0)
 *
 * Returns MC2_OK or a negative mc2_status; nothing is launched on error.
 */
int mc2_matmul_weight_grad(const void *dy, int64_t m, int64_t n, const void *x, int64_t k, int dtype, void *dw,
                           void *db, void *stream);

/*
 * QuantAllReduce  ("QuantAllReduce", ops-transformer mc2/quant_all_reduce:
 * 功能说明 formula output = Reduce(AllGather(scales) * AllGather(x)), reduceOp
 * "sum"; 参数说明 and 约束说明 for the types, the scale layouts and H).
 *
 *   out[t, j] = sum over r of dec(x_r[t, j]) * dec(scales_r[t, j / G])
 *
 *   Every rank receives the same sum, so one output is written.  The products
 *   are added in rank order by fp32 fused multiply-adds and rounded once
 *   (nearest-even) to out_dtype.
 *
 *   x_chunks      host array of world_size device pointers, each (bs, h) codes
 *                 of x_dtype (a (b, s, h) tensor is passed with bs = b * s)
 *   scale_chunks  host array of world_size device pointers:
 *                   scale_dtype MC2_F32  -> fp32 (bs, h / 128): pertoken-pergroup,
 *                                           G = 128
 *                   scale_dtype MC2_E8M0 -> e8m0 codes (bs, h / 64, 2), read flat
 *                                           as (bs, h / 32): mx, G = 32
 *   world_size    2, 4 or 8
 *   bs            tokens, >= 1
 *   h             hidden size, a multiple of 128 in [1024, 8192]
 *   x_dtype       MC2_I8, MC2_F8E4M3 or MC2_F8E5M2 (HiFloat8 is not supported);
 *                 MC2_E8M0 scales need an fp8 x_dtype
 *   out_dtype     MC2_F32, MC2_F16 or MC2_BF16;  out (bs, h)
 *
 * Returns MC2_OK or a negative mc2_status; nothing is launched on error.
 */
int mc2_quant_all_reduce(const void *const *x_chunks, const void *const *scale_chunks, int world_size, int64_t bs,
                         int64_t h, int x_dtype, int scale_dtype, int out_dtype, void *out, void *stream);

/*
 * Workspace size (bytes) that mc2_alltoall_quant_mm needs for these sizes.
 * Same argument meanings and validation as mc2_alltoall_quant_mm.
 */
int mc2_alltoall_quant_mm_workspace(int rank_size, int64_t bs_local, int64_t h, int64_t n,
                                    int x1_quant_mode, int x1_dtype, size_t *bytes);

/*
 * AlltoAllQuantMatmul  ("aclnnAlltoAllQuantMatmul": 功能说明 / 计算公式,
 * 函数原型, 约束说明).  The AlltoAll has already delivered the rank's
 * rank_size received blocks, chunks[r] = commOut[r], each (bs_local, h).
 *
 *   permuted[t, r*h + j] = chunks[r][t, j]            (bs_local, rank_size*h)
 *   x1_quant_mode 7 (per-token dynamic):
 *     y = permuted * x1_scale (smooth, per column; absent = 1), in fp32
 *     x1s[t] = max_j |y[t, j]| / 127;  q = clamp(rne(y / x1s[t]), -127, 127)
 *     (an all-zero row gives x1s = 0, q = 0)
 *   x1_quant_mode 3 (per-token, pre-quantised): q = permuted (int8),
 *     x1s = x1_scale (input)
 *   acc = q @ x2, exact int32
 *   out = bf16_rne(((float(acc) * x1s[t]) * x2_scale[j]) + bias[j]), fp32 ops in
 *         that order
 *
 *   chunks          host array of rank_size device pointers, each (bs_local, h):
 *                   dtype x1_dtype (MC2_BF16 / MC2_F16 for mode 7, MC2_I8 for mode 3)
 *   rank_size       2, 4 or 8
 *   bs_local        BS / rank_size, 1 <= BS <= INT32_MAX
 *   h               1 <= rank_size*h <= 35000, rank_size*h % 16 == 0
 *   x1_scale        mode 7: NULL or the smooth scale (rank_size*h) of x1_dtype;
 *                   mode 3: required per-token scale (bs_local) fp32
 *   x2              int8 (rank_size*h, n), contiguous
 *   x2_scale        fp32 (n), per channel (x2_quant_mode must be 2)
 *   bias            (n), required; bias_dtype MC2_F32 or MC2_BF16
 *   n               1 <= n <= INT32_MAX (this kernel: n % 16 == 0)
 *   out             bf16 (bs_local, n)
 *   alltoall_out    NULL or (rank_size, bs_local, h) of x1_dtype: alltoAllOutOptional,
 *                   read as commOut, the AlltoAll's result before the permute
 *                   (chunks[r] stored as block r); same dtype as x1 (约束说明)
 *   q_out           NULL or int8 (bs_local, rank_size*h): the quantised activations (mode 7)
 *   x1_scale_out    NULL or fp32 (bs_local): the per-token scales (mode 7)
 *   acc_out         NULL or int32 (bs_local, n): the exact accumulators (debug)
 *   workspace       device scratch of at least the bytes the query returns, 16-byte
 *                   aligned; it needs no initialisation (the stream-K flags in it
 *                   carry a per-launch epoch) and may be reused by calls ordered
 *                   on one stream; concurrent calls need their own
 *
 * Returns MC2_OK or a negative mc2_status; nothing is launched on error.
 */
int mc2_alltoall_quant_mm(const void *const *chunks, int rank_size, int64_t bs_local, int64_t h,
                          int x1_dtype, const void *x1_scale, const int8_t *x2, const float *x2_scale,
                          const void *bias, int bias_dtype, int x1_quant_mode, int x2_quant_mode,
                          int64_t n, void *out, void *alltoall_out, int8_t *q_out, float *x1_scale_out,
                          int32_t *acc_out, void *workspace, size_t workspace_bytes, void *stream);

/*
 * AlltoAllQuantMatmul for callers that cannot allocate device memory.  The
 * pages have no counterpart of this call: it is this library's own addition.
 *
 * mc2_alltoall_quant_mm needs a caller-provided workspace.  Some callers cannot
 * provide one: a C or Fortran host program that links only this library and
 * owns no device allocator, or a plugin inside a framework that owns all device
 * memory and forbids its plugins to call cudaMalloc (it can synchronise the
 * device and fragments the framework's pool).  This call takes the same
 * arguments minus the workspace and computes the same result, using a scratch
 * array built into the library instead.
 *
 *   - The scratch is MC2_NO_ALLOC_SCRATCH_BYTES (32 MiB).  Every GPU that
 *     loads the library holds it until the process exits.
 *   - Sizes whose workspace (as mc2_alltoall_quant_mm_workspace reports it)
 *     exceeds that are refused with MC2_ERR_WORKSPACE before anything is
 *     launched.
 *   - The call never calls cudaMalloc, cudaFree or any allocating routine.
 *   - Every call looks up the scratch's device address on the current device
 *     (a lookup, no allocation and no synchronisation), so a device reset
 *     between calls is harmless.  With CUDA's lazy module loading (the default)
 *     the library's device code, this array included, is loaded on a device
 *     the first time it is used there: that first call (of this or any other
 *     entry point) maps the 32 MiB.  A caller that must never see device
 *     memory grow mid-run makes one warm-up call at start-up, and makes its
 *     first call before any stream capture.
 *   - All calls share the one scratch array, and it keeps whatever the last
 *     call wrote (nothing in it needs to start at zero).  Calls whose work can
 *     overlap on the GPU (other streams, other host threads) race on it and
 *     must be serialised by the caller.
 *   - Other arguments, outputs and errors are those of mc2_alltoall_quant_mm.
 */
#define MC2_NO_ALLOC_SCRATCH_BYTES ((size_t)32 << 20)

int mc2_alltoall_quant_mm_no_alloc(const void *const *chunks, int rank_size, int64_t bs_local, int64_t h,
                                   int x1_dtype, const void *x1_scale, const int8_t *x2, const float *x2_scale,
                                   const void *bias, int bias_dtype, int x1_quant_mode, int x2_quant_mode, int64_t n,
                                   void *out, void *alltoall_out, int8_t *q_out, float *x1_scale_out,
                                   int32_t *acc_out, void *stream);

/* Name of a status code (static string). */
const char *mc2_status_str(int status);

/* Description of the last failure on this thread (static per-thread buffer). */
const char *mc2_last_error(void);

/*
 * Device-side status of the kernels launched so far on the current device:
 * synchronises the device, returns MC2_OK or MC2_ERR_TIMEOUT if a bounded wait
 * inside a kernel gave up (the kernel then skipped the rest of its tile loop),
 * and clears the flag.
 */
int mc2_device_status(void);

/*
 * Measurement aid (not one of the operations): lets a caller time each kernel
 * of a call on the call's own stream.  `events` is a host array of `count`
 * cudaEvent_t handles (as void*) created by the caller; count 0 turns it off.
 * While set, every call on this host thread records events[0] on its stream
 * just before its first kernel launch and events[i] just after its i-th
 * launch, for i < count (launches beyond count - 1 record nothing).  So
 * cudaEventElapsedTime(events[i], events[i+1]) is the device time of launch i.
 * The calls launch, in order:
 *   mc2_all_gather_mm, mc2_matmul_reduce_scatter   1: the GEMM
 *   mc2_matmul_weight_grad     1: the GEMM (which also forms db)
 *   mc2_quant_all_reduce       1: the reduction
 *   mc2_alltoall_quant_mm      x1_quant_mode 7: 2 (the fused quant and x2
 *                              widening, the GEMM), or 3 when rank_size*h > 32768
 *                              or h % 8 != 0 (the quant, the x2 widening, the
 *                              GEMM); x1_quant_mode 3: 2 when h % 64 == 0 (the
 *                              widening of the chunks and x2, the GEMM), else 3
 *                              (the permuted widening, the x2 widening, the GEMM)
 * An event between two launches also keeps the second from starting early
 * (programmatic dependent launch), which can add a few microseconds to a
 * call.  The setting is per host thread and stays until changed; the caller
 * keeps the events alive while it is set.
 * Returns MC2_OK, MC2_ERR_SHAPE (count outside [0, 8]) or MC2_ERR_NULL.
 */
int mc2_set_launch_events(void *const *events, int count);

/*
 * Test hook for the bounded waits (not one of the operations).  Arms a fault
 * for the next mc2_alltoall_quant_mm (or _no_alloc) call on this host thread
 * only: in that call's GEMM, every stream-K finishing part expects one more
 * partial sum than any part writes, so its wait on the tile's flag cannot
 * succeed and gives up after `wait_limit_ns` (instead of the usual 2 s).  The
 * kernel then skips those tiles' epilogues (their outputs are left as they
 * were) and raises the device status word: mc2_device_status() afterwards
 * returns MC2_ERR_TIMEOUT and clears it, and the device stays usable.  The
 * hook is consumed by that one call even when its GEMM has no stream-K tail
 * (then nothing waits and nothing is raised).
 * Returns MC2_OK, or MC2_ERR_SHAPE if wait_limit_ns is 0 or above 2 s.
 */
int mc2_test_expire_next_flag_waits(uint64_t wait_limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* MC2_GB300_H */
