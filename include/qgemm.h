/*
 * qgemm.h -- C ABI of libqgemm: block-quantised (GGUF Q4_0 / Q8_0) matrix-vector
 * and skinny matrix-matrix products on one NVIDIA GB300 (sm_103a).
 *
 * Formats ("Engine and kernels", pooled.run, section "What it runs"): a block
 * is 32 weights plus one f16 scale d. Q4_0 stores 4-bit quants q, weight
 * (q - 8) * d; byte j of a block holds element j in its low nibble and element
 * j + 16 in its high nibble. Q8_0 stores int8 q, weight q * d.
 *
 * Layout ("Architecture", pooled.run, section "Memory and caching": matrices are
 * repacked at load time into separate nibble and scale arrays so that kernels
 * read contiguous stripes). A matrix W of `rows` x `k` weights (k a multiple of
 * 32) is passed as two row-major device arrays:
 *   quants: Q4_0 uint8 [rows][k/2]  (16 bytes per block)
 *           Q8_0 int8  [rows][k]    (32 bytes per block)
 *   scales: uint16 [rows][k/32]      (f16 bit patterns)
 * In-block byte order: a block's quant bytes are taken in 16-byte groups (one
 * group for Q4_0, two for Q8_0), and in each group the two 8-byte halves are
 * interleaved byte by byte: stored byte 2m + h is GGUF byte m + 8h of the group
 * (m = 0..7, h = 0..1). qrepack produces this order from GGUF blocks. It lets
 * a tensor-core fragment load hand each lane the bytes of elements 2t, 2t+1,
 * 2t+8, 2t+9 together, so the activations need no reordering on that path.
 * Activations X are f16 [ncols][k] (column c is the c-th input vector), outputs
 * Y are f32 [ncols][rows].
 *
 * Conventions for every entry point:
 *  - Pointers are DEVICE pointers unless stated; the caller owns all memory.
 *    No entry point allocates device memory.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default stream)
 *    and the call returns without synchronising.
 *  - Argument errors (NULL, shape, alignment, type, workspace) are detected on
 *    the host before anything is launched and returned synchronously; nothing
 *    is written. A launch failure returns QG_ERR_CUDA, and qg_last_cuda_error
 *    on the same host thread names the CUDA error behind it.
 *  - Host threads: calls may come from several threads at once (each on its
 *    own stream, or ordered by the caller). Per-device kernel set-up happens
 *    once, under a lock. A thread's first call makes the current device's
 *    primary context current on that thread (cudaSetDevice); make that first
 *    call outside any stream capture.
 *  - Alignment: quant and scale arrays and X must be 16-byte aligned; Y, y0
 *    4-byte aligned; H 2-byte aligned.
 *  - Residual: y0 may be NULL (no residual) or point to f32 [ncols][rows];
 *    y0 == y is allowed (in-place y += W x). Any other overlap of y0 and y is
 *    QG_ERR_ALIAS.
 *  - rows == 0 is a valid empty problem: QG_OK, nothing launched.
 *  - Kernels are launched with programmatic dependent launch: a call's kernels
 *    may start while the previous kernel on `stream` is finishing, and until
 *    that kernel has completed they read only the weight arrays (quants and
 *    scales), never X, y0, ids or outputs. So weights must not be written by
 *    a preceding kernel on the stream that itself lets its dependents start
 *    early (one that calls cudaTriggerProgrammaticLaunchCompletion before its
 *    last write). Ordinary kernels, and qrepack, never do.
 *  - Results are deterministic: the reduction order depends only on the
 *    problem shape, never on timing or on the number of SMs.
 *  - Arithmetic: weights are dequantised exactly (every Q4_0/Q8_0 weight is
 *    exact in f32 as an integer times its scale) and accumulated in f32; no
 *    partial sum is ever held in f16.
 */
#ifndef QGEMM_H
#define QGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *cudaStream_t;

typedef enum {
  QG_OK = 0,
  QG_ERR_NULL = 1,      /* a required pointer is NULL */
  QG_ERR_SHAPE = 2,     /* k <= 0 or k % 32, rows < 0, ncols/topk/n_expert out of range */
  QG_ERR_ALIGN = 3,     /* a pointer violates the alignment rule above */
  QG_ERR_TYPE = 4,      /* unknown quant type */
  QG_ERR_WORKSPACE = 5, /* workspace NULL or smaller than qmoe_workspace_bytes() */
  QG_ERR_CUDA = 6,      /* a CUDA runtime error (launch failure, no device, ...) */
  QG_ERR_ALIAS = 7      /* y0 partially overlaps y */
} qg_status;

typedef enum { QG_Q4_0 = 2, QG_Q8_0 = 8 } qg_type; /* GGUF type ids */

/* Static, NUL-terminated description of a status code. */
const char *qg_status_str(qg_status s);

/* ---------------------------------------------------------------------------
 * Decode GEMV and its batched twins: Y[c] = y0[c] + W X[c], c < ncols, 1 <= ncols <= 8.
 * ("Engine and kernels", section "Kernel families": cooperative GEMV for decode,
 * batched GEMV twins for speculative verify; section "Fewer passes": y += W x.)
 *   nib / qs : quants of W (see layout), scl: scales, rows x k
 *   x        : f16 [ncols][k]
 *   y0       : NULL or f32 [ncols][rows] (may equal y)
 *   y        : f32 [ncols][rows], written
 * ------------------------------------------------------------------------- */
qg_status qgemv_q4_0(const uint8_t *nib, const uint16_t *scl, int rows, int k,
                     const uint16_t *x, int ncols, const float *y0, float *y,
                     cudaStream_t stream);
qg_status qgemv_q8_0(const int8_t *qs, const uint16_t *scl, int rows, int k,
                     const uint16_t *x, int ncols, const float *y0, float *y,
                     cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Prefill GEMM: Y[c] = y0[c] + W X[c] for 1 <= ncols <= 16, reading each weight
 * block once for all columns ("Engine and kernels", section "Kernel families",
 * prefill GEMM; section "Batching and prefill", row-stationary GEMM at 16
 * columns with split-K pinned per shape). Arguments as qgemv_*, `t` selects the
 * quant type of `q`.
 * ------------------------------------------------------------------------- */
qg_status qgemm_cols(qg_type t, const void *q, const uint16_t *scl, int rows, int k,
                     const uint16_t *x, int ncols, const float *y0, float *y,
                     cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Fused FFN gate/up: one sweep over both projections, SiLU(gate) * up applied
 * before the write ("Engine and kernels", section "Kernel families", fused
 * gate/up):  H[c][r] = f16( SiLU(g) * u ),  g = (Wg X[c])[r], u = (Wu X[c])[r],
 * SiLU(z) = z / (1 + e^-z), g and u accumulated in f32.
 *   qg/sg, qu/su : gate and up matrices, both rows x k, same type t
 *   x            : f16 [ncols][k], 1 <= ncols <= 16
 *   h            : f16 [ncols][rows], written
 * ------------------------------------------------------------------------- */
qg_status qffn_gate_up_silu(qg_type t, const void *qg, const uint16_t *sg, const void *qu,
                            const uint16_t *su, int rows, int k, const uint16_t *x,
                            int ncols, uint16_t *h, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Stacked-expert MoE layer ("Engine and kernels", sections "What it runs" and
 * "Kernel families": 256 experts, 8 active per token, plus a shared expert;
 * routing needs no readback. "A 235B model in a browser window", section
 * "A mixture of experts is a different animal": gate, up and down matrices of
 * all experts stacked by role; only the routed experts' slices are read).
 *
 *   gate/up stacks : [n_expert][ffn][hidden] (quants qg/qu, scales sg/su)
 *   down stack     : [n_expert][hidden][ffn] (quants qd, scales sd)
 *   ids            : device int32 [ncols][topk] expert ids (1 <= topk <= 16;
 *                    1 <= n_expert <= QG_MOE_MAX_EXPERTS)
 *   rw             : device f32   [ncols][topk] routing weights
 *   shared         : HOST pointer to a qg_expert of device pointers (one more
 *                    expert of the same shape, added with weight 1), or NULL
 *   x              : f16 [ncols][hidden], 1 <= ncols <= 16
 *   y              : f32 [ncols][hidden] =
 *                    y0 + sum_j rw[c][j] * D_e (SiLU(G_e x_c) * (U_e x_c)) + shared,
 *                    e = ids[c][j]; the intermediate h is rounded to f16.
 *   ws, ws_bytes   : device workspace of at least qmoe_workspace_bytes(...) bytes,
 *                    16-byte aligned; its contents on entry are ignored. When the
 *                    call's work has completed, ws starts with the intermediate h
 *                    of every (column, slot): f16 [ncols][topk + 1][ffn], slot
 *                    topk being the shared expert; slots of invalid ids (and the
 *                    shared slot when shared is NULL) hold unspecified values.
 *                    A caller may read it to check the layer stage by stage.
 *   err_flag       : device int32 or NULL. An id outside [0, n_expert) makes that
 *                    slot contribute 0 and ORs QG_MOE_BAD_ID into *err_flag. The
 *                    library never clears the flag: zero it before the call and
 *                    read it after synchronising. No trap, no abort.
 *   uniq_ids_out   : device int32 [ncols*topk] or NULL: the distinct valid ids in
 *                    ascending order (each expert slice is read once for all
 *                    columns that route to it), padded with -1.
 * ------------------------------------------------------------------------- */
typedef struct qg_expert {
  const void *qg;
  const uint16_t *sg;
  const void *qu;
  const uint16_t *su;
  const void *qd;
  const uint16_t *sd;
} qg_expert;

#define QG_MOE_BAD_ID 1
#define QG_MOE_MAX_EXPERTS (1 << 22)

/* Workspace bytes qmoe_experts needs for this shape; 0 for a shape that it
 * rejects with QG_ERR_SHAPE. */
size_t qmoe_workspace_bytes(int n_expert, int ffn, int hidden, int ncols, int topk);

qg_status qmoe_experts(qg_type t, const void *qg, const uint16_t *sg, const void *qu,
                       const uint16_t *su, const void *qd, const uint16_t *sd,
                       int n_expert, int ffn, int hidden, const int32_t *ids,
                       const float *rw, int topk, const qg_expert *shared,
                       const uint16_t *x, int ncols, const float *y0, float *y,
                       void *ws, size_t ws_bytes, int32_t *err_flag,
                       int32_t *uniq_ids_out, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * qmoe_experts without a caller workspace. The pages have no counterpart to
 * this call: it exists for callers that cannot allocate device memory (a
 * plugin inside a framework that owns all device memory, a fixed memory budget
 * with no room left, a latency-critical loop that must not call cudaMalloc).
 * Arguments and results are those of qmoe_experts minus ws / ws_bytes; the
 * workspace is a QG_MOE_NOALLOC_WS_BYTES array inside the library, held on every
 * GPU that loads the library until the process exits.
 *  - The array is as large as the largest workspace any shape qmoe_experts
 *    accepts needs (16 columns x 32768 h values per column, f16), so every
 *    accepted shape fits. Type and shape errors are those of qmoe_experts; a
 *    problem whose qmoe_workspace_bytes(...) exceeded the array would get
 *    QG_ERR_WORKSPACE before anything is launched.
 *  - The first call on each device (with that device current) looks up the
 *    array's device address and keeps it; make that first call before any
 *    stream capture. The kept address dies with the device's primary context:
 *    do not use this call across cudaDeviceReset.
 *  - All calls share the array: calls whose GPU work overlaps (different
 *    streams, several host threads) race on it. Nothing in it needs clearing.
 *  - After a call's work has completed the array holds that call's h, laid out
 *    as qmoe_experts leaves it in its workspace.
 *  - Allocates nothing (no cudaMalloc, no library allocator).
 * ------------------------------------------------------------------------- */
#define QG_MOE_NOALLOC_WS_BYTES ((size_t)1 << 20) /* 1 MiB */

qg_status qmoe_experts_noalloc(qg_type t, const void *qg, const uint16_t *sg, const void *qu,
                               const uint16_t *su, const void *qd, const uint16_t *sd,
                               int n_expert, int ffn, int hidden, const int32_t *ids,
                               const float *rw, int topk, const qg_expert *shared,
                               const uint16_t *x, int ncols, const float *y0, float *y,
                               int32_t *err_flag, int32_t *uniq_ids_out, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Load-time repack ("Architecture", section "Memory and caching"): GGUF
 * interleaved blocks (per block: f16 d, little endian, then 16 (Q4_0) or 32
 * (Q8_0) quant bytes), rows x k/32 blocks, into the quant and scale arrays of
 * the layout above. gguf must be 2-byte aligned; q_out and scl_out follow the
 * layout's alignment rule.
 * ------------------------------------------------------------------------- */
qg_status qrepack(qg_type t, const void *gguf, int rows, int k, void *q_out,
                  uint16_t *scl_out, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * MoE router ("Engine and kernels", section "Kernel families": router and top-k
 * on the GPU, so routing needs no readback; the output feeds qmoe_experts).
 *   w_router   : f32 [n_expert][hidden] (16-byte aligned), 1 <= n_expert <= 1024
 *   x          : f16 [ncols][hidden], 1 <= ncols <= 16 (the MoE input)
 *   topk       : 1..32, <= n_expert
 *   logits_out : NULL or f32 [ncols][n_expert]: logits = W_router x (f32)
 *   ids_out    : int32 [ncols][topk]: the topk largest logits of each column in
 *                the qargmax_f32 order (lowest expert id on ties)
 *   rw_out     : f32 [ncols][topk]: softmax over those topk logits
 * ------------------------------------------------------------------------- */
qg_status qmoe_router(const float *w_router, const uint16_t *x, int n_expert, int hidden,
                      int ncols, int topk, float *logits_out, int32_t *ids_out, float *rw_out,
                      cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Sampling over f32 logits ("Engine and kernels", section "Kernel families":
 * greedy argmax and top-k on the GPU, so a token reads back a few bytes instead
 * of the logits; section "Fewer passes": lowest-index tie-breaking).
 *   x        : f32 [ncols][n], 4-byte aligned (e.g. the LM-head output of
 *              qgemv_q8_0; its first n rows are the draft head's output)
 *   n        : >= 1 values per column;  ncols: 1..64
 *   Order    : a number ranks before NaN; larger values first; +0 equals -0;
 *              equal values, and NaNs, rank by the lower index.
 * qargmax_f32: idx_out int32 [ncols], the first-ranked element of each column;
 *              val_out NULL or f32 [ncols], its value (the bits of x).
 * qtopk_f32  : the k first-ranked elements of each column in rank order,
 *              1 <= k <= 256, k <= n; idx_out int32 [ncols][k], val_out NULL
 *              or f32 [ncols][k].
 * Both are deterministic. QG_ERR_SHAPE for n, ncols or k out of range.
 * ------------------------------------------------------------------------- */
qg_status qargmax_f32(const float *x, int n, int ncols, int32_t *idx_out, float *val_out,
                      cudaStream_t stream);
qg_status qtopk_f32(const float *x, int n, int ncols, int k, int32_t *idx_out,
                    float *val_out, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Diagnostics: number of kernels this library has launched in this process
 * (monotonic, all devices and threads). Lets a caller count the GPU launches of
 * a region of work. Not part of the method.
 * ------------------------------------------------------------------------- */
uint64_t qg_kernel_launches(void);

/* ---------------------------------------------------------------------------
 * Diagnostics: the current device's error word, read and then cleared.
 * Not part of the method. Every wait of the tensor-core kernel (on its TMA
 * data, on a free pipeline stage, or on the partial tiles of its K split) and
 * of the staged MoE down kernel (on its bulk copies) is bounded (~2 s); a wait
 * that gives up sets bit QG_DEV_ERR_WAIT and the kernel returns without its
 * result, so the outputs of that call are wrong while the context stays
 * usable. The word is shared by every call on the device since the last read.
 *  - bits_out: host pointer, receives the word (0: no error).
 *  - Synchronises the current device (a copy from a device symbol).
 *  - QG_ERR_NULL if bits_out is null, QG_ERR_CUDA if the copies fail.
 * ------------------------------------------------------------------------- */
#define QG_DEV_ERR_WAIT 1
qg_status qg_device_error(int32_t *bits_out);

/* ---------------------------------------------------------------------------
 * Diagnostics: a self-test of the bounded waits. Not part of the method. One
 * thread of one CTA waits on a phase of an mbarrier that nothing completes,
 * first with CTA scope (the form of the tensor-core kernel's stage waits), then
 * with cluster-scope acquire (the form of its K-split handoff). Each wait gives
 * up after its bound (~2 s), sets QG_DEV_ERR_WAIT in the device error word and
 * returns, so the call takes about 4 s and leaves the context usable.
 *  - completed_out: host int32[2], receives per wait 1 if it completed, 0 if it
 *    gave up (both 0 when the bounds work).
 *  - Enqueues on `stream` and synchronises it.
 *  - QG_ERR_NULL if completed_out is null; QG_ERR_CUDA if the launch or a copy
 *    fails.
 * ------------------------------------------------------------------------- */
qg_status qg_wait_selftest(int32_t *completed_out, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Diagnostics: the CUDA runtime error behind the latest QG_ERR_CUDA that a
 * call of this library returned on the calling host thread (a cudaError_t
 * value; 0 if there was none), and its name and description. The string
 * belongs to the library and stays valid until the thread's next call of
 * qg_last_cuda_error_string. Not part of the method.
 * ------------------------------------------------------------------------- */
int qg_last_cuda_error(void);
const char *qg_last_cuda_error_string(void);

#ifdef __cplusplus
}
#endif
#endif /* QGEMM_H */
