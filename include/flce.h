/*
 * flce.h - C ABI of libflce.so, a GB300-native (sm_103a) fused linear cross entropy.
 *
 * The operation
 * -------------
 * A language-model head projection followed by softmax cross entropy, forward and
 * backward in one call. For token rows X[BT,H], head weight W[V,H], optional bias b[V] and
 * targets t[BT], every row i whose target is not ignore_index gets
 *
 *     s_v    = X_i . W_v + b_v                          (logits: fp32 on chip; exp(s_v)
 *                                                       of the chunk's rows stored in the
 *                                                       input dtype, in the workspace)
 *     lse_i  = log sum_v exp(s_v)
 *     loss_i = lse_i - s_{t_i} + z lse_i^2              (z = z_loss_scale)
 *     pred_i = argmax_v s_v (lowest index on ties),     acc_i = [pred_i == t_i]
 *     dS_iv  = c_i (softmax(s)_v (1 + 2 z lse_i) - [v == t_i])
 *     dX_i   = sum_v dS_iv W_v,      dW += dS^T X,      dbias += sum_i dS_i
 *
 * with c_i = g / N_labelled (mean), g (sum) or g_i (none), g the upstream gradient.
 * The logits, grad_input and grad_weight products all run inside this one call, as in
 * "Liger-Kernel PR #1554: skip ignore_index rows" (Summary), and dW is accumulated
 * straight into the caller's destination with no [V,H] temporary, as proposed in "Reduce
 * FLCE weight-gradient allocation overhead across FP16, BF16, and FP32" (Proposed
 * direction). Rows whose target is ignore_index never enter a GEMM, so a NaN stored in
 * them cannot reach any output (PR #1554, Tests), and they get 0 loss, 0 z-loss, 0
 * accuracy, -1 as predicted token and a zero dX row (PR #1554, Details item 1). The
 * per-call transient memory is the caller's workspace, whose size the caller picks and
 * which does not grow with BT beyond 16 bytes per row (the memory/latency trade-off of
 * "feat(flce): expose direct chunk-size control via LIGER_FLCE_CHUNK_SIZE", Summary, made
 * an explicit API argument as the maintainers ask there).
 *
 * Memory and ownership
 * --------------------
 * Every pointer in flce_args is a DEVICE pointer on the current CUDA device, allocated
 * and owned by the caller. The library allocates no device memory, keeps no per-call
 * state between calls and never synchronises the stream. Layouts are dense row-major:
 * X and dX [BT,H], W and dW [V,H], bias and dbias [V], targets/pred/lse [BT].
 * X, W, dX and dW must be 16-byte aligned, the workspace 256-byte aligned.
 *
 * Errors
 * ------
 * flce_fwd_bwd validates its arguments on the host and returns an flce_status at once,
 * launching nothing on error. Errors found on the device (a labelled target outside
 * [0,V), a pipeline wait that ran out) are OR-ed into the device status word and read
 * back with flce_get_status. No kernel traps.
 *
 * Threading: calls on different streams may run concurrently as long as they use
 * different workspaces and status words.
 */
#ifndef FLCE_H_
#define FLCE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FLCE_ABI_VERSION 2

#if defined(__GNUC__)
#define FLCE_API __attribute__((visibility("default")))
#else
#define FLCE_API
#endif

typedef enum flce_status {
  FLCE_OK = 0,
  FLCE_ERR_INVALID_ARG = 1,  /* null pointer, bad shape, bad enum, misaligned pointer   */
  FLCE_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. a dW_dtype)             */
  FLCE_ERR_TARGET_RANGE = 3, /* device: a labelled target outside [0,V); row ignored    */
  FLCE_ERR_WORKSPACE = 4,    /* workspace too small for one 128-row chunk               */
  FLCE_ERR_CUDA = 5,         /* a CUDA runtime call or launch failed                    */
  FLCE_ERR_TIMEOUT = 6,      /* device: a pipeline wait exceeded its limit; outputs are
                                not valid                                               */
  FLCE_ERR_SCRATCH_LIMIT = 7 /* flce_fwd_bwd_noalloc: the problem does not fit the fixed
                                scratch of FLCE_NOALLOC_SCRATCH_BYTES                   */
} flce_status;

typedef enum flce_reduction { FLCE_MEAN = 0, FLCE_SUM = 1, FLCE_NONE = 2 } flce_reduction;

typedef enum flce_dtype { FLCE_F32 = 0, FLCE_BF16 = 1, FLCE_F16 = 2 } flce_dtype;

/* flce_args.flags */
#define FLCE_FLAG_FORCE_SIMT 0x1u /* run the three GEMMs on SIMT fp32-FMA kernels even for
                                     bf16/f16 inputs (fp32 inputs always use them)       */
#define FLCE_FLAG_NO_ROW_REF 0x2u /* always normalise the gradient slab per vocabulary tile
                                     (a full pass over it) instead of the default one-scale-
                                     per-row form of bf16 tensor-core calls without dbias   */
#define FLCE_FLAG_DW_OVERWRITE 0x4u /* dW and dbias receive this call's gradient instead of
                                     accumulating it (no need to zero them first); with no
                                     labelled row they are set to zero                      */
#define FLCE_FLAG_SEPARATE_BWD 0x8u /* run the dX and dW GEMMs as two launches instead of
                                     one launch sharing a work queue (the results are the
                                     same bits either way)                                 */
#define FLCE_FLAG_DEBUG_STALL 0x100u /* testing only: the tensor-core forward GEMM leaves
                                     one pipeline stage unfilled so that its bounded waits
                                     run out; the call must then report FLCE_ERR_TIMEOUT */
#define FLCE_FLAG_DEBUG_STALL_BWD 0x200u /* testing only: the same in the merged dX + dW
                                     launch (its first work item)                          */

/* Stages of one call, in launch order, for the optional profiler (flce_profile_*). */
typedef enum flce_stage {
  FLCE_STAGE_PROLOGUE = 0, /* row compaction + ignored-row outputs (2 kernels)          */
  FLCE_STAGE_GATHER = 1,   /* gather of the chunk's labelled rows of X                  */
  FLCE_STAGE_FWD = 2,      /* logits GEMM with online max / sum-exp / argmax epilogue   */
  FLCE_STAGE_FINALIZE = 3, /* per-row merge: lse, loss, prediction, gradient multipliers */
  FLCE_STAGE_GPASS = 4,    /* gradient of the logits: formed in place (and dbias), or in
                              the row-reference form the Xc row scale plus the per-tile
                              redo launches gated on the chunk's window flag             */
  FLCE_STAGE_DX = 5,       /* dX GEMM                                                   */
  FLCE_STAGE_DW = 6,       /* dW GEMM (accumulating)                                    */
  FLCE_STAGE_REDUCE = 7,   /* mean/sum reductions (and, with FLCE_FLAG_DW_OVERWRITE,
                              the zeroing of dW / dbias when no row is labelled)         */
  FLCE_STAGE_BWD = 8,      /* dX and dW GEMMs in one launch (tensor-core calls with both
                              gradients and 2048-row or larger chunks), with the dX sum  */
  FLCE_STAGE_COUNT = 9
} flce_stage;

/* Opaque profiler: when flce_args.profile is non-NULL, the call records a CUDA event pair
 * on its stream around every launch and tags it with its stage. Host object, owned by the
 * caller; not thread-safe (one profiler per thread/stream). */
typedef struct flce_profile flce_profile;

typedef struct flce_args {
  /* shapes */
  int64_t BT;               /* token rows, >= 1                                          */
  int64_t H;                /* hidden size, >= 1                                         */
  int64_t V;                /* vocabulary size, >= 1                                     */
  int32_t in_dtype;         /* flce_dtype of X, W, bias and dX                           */
  int32_t reduction;        /* flce_reduction                                            */
  /* inputs */
  const void* X;            /* [BT,H]                                                    */
  const void* W;            /* [V,H]                                                     */
  const void* bias;         /* [V] or NULL                                               */
  const int64_t* targets;   /* [BT]; ignore_index marks rows that take no part           */
  int64_t ignore_index;     /* -100 in the usual convention                              */
  float z_loss_scale;       /* z >= 0; 0 disables the z-loss term                        */
  const float* grad_out;    /* NULL means 1.0; [1] for mean/sum, [BT] for none           */
  int32_t want_dX;          /* 1: write dX                                               */
  int32_t want_dW;          /* 1: accumulate dW (and dbias when bias != NULL)            */
  int32_t dW_dtype;         /* flce_dtype of dW/dbias: FLCE_F32, or in_dtype itself
                               (same-dtype accumulation: the call's G^T X is rounded to
                               in_dtype and added in in_dtype); others give
                               FLCE_ERR_UNSUPPORTED                                      */
  uint32_t flags;           /* FLCE_FLAG_*                                               */
  /* outputs (NULL = not wanted, except loss) */
  float* loss;              /* [1] for mean/sum (reduced), [BT] for none (per token)     */
  float* z_loss;            /* same shape and reduction as loss                          */
  float* acc;               /* same shape and reduction as loss (accuracy)               */
  float* lse;               /* [BT] per token; 0 on ignored rows                         */
  int64_t* pred;            /* [BT] per token argmax; -1 on ignored rows                 */
  int32_t* n_labelled;      /* [1] number of rows that entered the loss                  */
  void* dX;                 /* [BT,H] in_dtype, overwritten (zero on ignored rows)       */
  void* dW;                 /* [V,H] dW_dtype, ACCUMULATED (+=); zero it for a fresh grad,
                               or pass FLCE_FLAG_DW_OVERWRITE                            */
  void* dbias;              /* [V] dW_dtype, ACCUMULATED (or overwritten, as dW); used
                               when bias and want_dW; NULL: the bias gradient is not
                               wanted                                                    */
  /* scratch and status */
  void* workspace;          /* device scratch of workspace_bytes, caller-owned           */
  size_t workspace_bytes;   /* >= flce_workspace_size(BT,H,V,in_dtype,0) or any size
                               that fits one 128-row chunk: larger means fewer chunks    */
  int32_t* status;          /* device int; reset to 0 by the call, then OR-ed with
                               (1 << flce_status) per device-side error; may be NULL
                               (a word inside the workspace is used instead)             */
  uint32_t wait_timeout_ms; /* limit of every pipeline wait; 0 means 4000 ms             */
  flce_profile* profile;    /* NULL, or a profiler from flce_profile_create             */
} flce_args;

/* Workspace bytes for a problem, choosing the row-chunk so that the workspace stays
 * within budget_bytes (0 means 3 GiB). The result grows with BT only by 16 bytes per
 * row (the compaction index and per-row loss terms) and is capped by the budget. Returns 0
 * on invalid arguments or when not even one 128-row chunk fits in the budget. */
FLCE_API size_t flce_workspace_size(int64_t BT, int64_t H, int64_t V, int32_t in_dtype,
                           size_t budget_bytes);

/* Rows per chunk that flce_fwd_bwd will use with this workspace size (a multiple of 128),
 * or 0 when the workspace is too small. Host-only; touches no GPU. */
FLCE_API int64_t flce_chunk_rows(int64_t BT, int64_t H, int64_t V, int32_t in_dtype,
                        size_t workspace_bytes);

/* Human-readable plan of a call with this workspace size, for logs and debugging: chunk
 * rows, host chunk launches, vocabulary tiles, the workspace regions with their offsets and
 * sizes, and the GEMM tile shapes and tile counts when every row is labelled (the device
 * balances the rows it actually finds over cdiv(N, R) chunks). Writes at most `out_len`
 * bytes including the terminating NUL into `out` (which may be NULL when out_len is 0) and
 * returns the length of the full text, like snprintf, or -1 for invalid sizes or dtype or
 * a workspace too small for one 128-row chunk. Host-only; touches no GPU. The same text is
 * printed to stderr by every flce_fwd_bwd call, with the path the call takes, when the
 * environment variable FLCE_TRACE is set to a value other than "" or "0" (read once). */
FLCE_API int64_t flce_plan_describe(int64_t BT, int64_t H, int64_t V, int32_t in_dtype,
                                    size_t workspace_bytes, char* out, size_t out_len);

/* Enqueue the fused forward+backward on `stream` (a cudaStream_t; NULL = legacy default
 * stream). Returns FLCE_OK once every kernel is enqueued, or an error code with nothing
 * enqueued (FLCE_ERR_CUDA may follow a partial enqueue if a launch fails). */
FLCE_API int32_t flce_fwd_bwd(const flce_args* args, void* stream);

/* ----------------------------------------------------------------------------------
 * Fused linear JSD / KL distillation (same tile engine).
 *
 * The pages name this sibling op without defining it (a "fused linear KL" loss with its
 * own chunk policy on the Liger-Kernel v0.8.3 commit page; test_fused_linear_jsd.py in
 * "Liger-Kernel PR #1554: skip ignore_index rows", Results). The definition used: teacher
 * P = softmax(X_t W_t^T / T), student Q = softmax(X_s W_s^T / T) per row over V, and
 *     0 < beta < 1: loss_i = beta KL(P||M) + (1-beta) KL(Q||M),  M = beta P + (1-beta) Q
 *     beta = 0:     loss_i = KL(P||Q)        beta = 1:  loss_i = KL(Q||P)
 * reduced over the rows whose label is not ignore_index (all rows when labels is NULL;
 * a label's value is otherwise unused) by mean (over those rows), sum or none. Only the
 * student gets gradients: dX_s = dS W_s, dW_s += dS^T X_s with
 * dS = c_i / T * dloss_i/dz_s. Neither [BT,V] logits nor probabilities reach HBM; the
 * workspace holds two [R, V] slabs (student, teacher) per chunk of R rows.
 * Memory, ownership, errors and threading as for flce_fwd_bwd.
 * ---------------------------------------------------------------------------------- */
typedef struct flce_jsd_args {
  int64_t BT;               /* rows                                                      */
  int64_t Hs;               /* student hidden size                                       */
  int64_t Ht;               /* teacher hidden size                                       */
  int64_t V;                /* vocabulary size (shared)                                  */
  int32_t in_dtype;         /* flce_dtype of Xs, Ws, Xt, Wt and dX                        */
  int32_t reduction;        /* flce_reduction                                            */
  const void* Xs;           /* [BT,Hs] student rows                                      */
  const void* Ws;           /* [V,Hs]  student head                                      */
  const void* Xt;           /* [BT,Ht] teacher rows                                      */
  const void* Wt;           /* [V,Ht]  teacher head                                      */
  const int64_t* labels;    /* [BT] or NULL; rows equal to ignore_index take no part     */
  int64_t ignore_index;
  float beta;               /* in [0, 1]                                                 */
  float temperature;        /* > 0                                                       */
  const float* grad_out;    /* NULL means 1.0; [1] for mean/sum, [BT] for none           */
  int32_t want_dX;          /* 1: write dX_s                                             */
  int32_t want_dW;          /* 1: accumulate dW_s                                        */
  int32_t dW_dtype;         /* FLCE_F32 or in_dtype                                      */
  uint32_t flags;           /* FLCE_FLAG_FORCE_SIMT, FLCE_FLAG_DW_OVERWRITE              */
  float* loss;              /* [1] for mean/sum, [BT] for none                           */
  int32_t* n_labelled;      /* [1] or NULL                                               */
  void* dX;                 /* [BT,Hs] in_dtype, overwritten (zero on ignored rows)      */
  void* dW;                 /* [V,Hs] dW_dtype, ACCUMULATED (or overwritten, as above)   */
  void* workspace;          /* device scratch, 256-byte aligned                          */
  size_t workspace_bytes;   /* >= flce_jsd_workspace_size(...) for a chosen budget       */
  int32_t* status;          /* device int or NULL, as in flce_args                       */
  uint32_t wait_timeout_ms; /* 0 means 4000 ms                                           */
  flce_profile* profile;    /* NULL, or a profiler (stages as for flce_fwd_bwd; the
                               divergence and gradient passes count as FLCE_STAGE_GPASS) */
} flce_jsd_args;

/* x[i] *= *g for 0 <= i < n, unless *g == 1 exactly: g is read on the device, so scaling
 * by an upstream gradient that lives on the GPU needs no host synchronisation and costs
 * nothing in the common case g == 1 (the torch autograd op scales the gradients it
 * computed in the forward this way). x: device array of n elements of `dtype`
 * (FLCE_F32, FLCE_BF16 or FLCE_F16), scaled in place; g: device pointer to one float.
 * Enqueued on `stream`; returns FLCE_ERR_INVALID_ARG for null pointers, n < 0 or an
 * unknown dtype, FLCE_ERR_CUDA if the launch fails. No counterpart on the pages: it is
 * plumbing for the autograd binding. */
FLCE_API int32_t flce_scale_by(void* x, int64_t n, int32_t dtype, const float* g, void* stream);

/* Workspace bytes for the distillation op within budget_bytes (0 means 6 GiB: its workspace
 * holds two logit-sized slabs, one per head); 0 when
 * not even one 128-row chunk fits or on invalid arguments. */
FLCE_API size_t flce_jsd_workspace_size(int64_t BT, int64_t Hs, int64_t Ht, int64_t V,
                                        int32_t in_dtype, size_t budget_bytes);

/* Enqueue the fused linear JSD forward+backward on `stream`; host-side errors return at
 * once with nothing enqueued, device-side ones go to the status word. */
FLCE_API int32_t flce_fused_linear_jsd(const flce_jsd_args* args, void* stream);

/* Size of the fixed device scratch used by flce_fwd_bwd_noalloc (128 MiB). */
#define FLCE_NOALLOC_SCRATCH_BYTES ((size_t)128 << 20)

/* Same operation and arguments as flce_fwd_bwd, for callers that cannot allocate device
 * memory (a framework that owns all device memory through its own pool, code that must
 * not allocate after start-up, a foreign-function layer that forwards only the op's
 * inputs and outputs). The pages have no counterpart of this entry point.
 *
 * Instead of a caller workspace it uses a scratch array of FLCE_NOALLOC_SCRATCH_BYTES
 * compiled into the library: every GPU that loads the library holds that memory until the
 * process exits. args->workspace must be NULL, args->workspace_bytes 0 and args->profile
 * NULL (FLCE_ERR_INVALID_ARG otherwise). Problems whose 128-row chunk does not fit the
 * scratch (roughly 2 * V * 128 + 16 * BT bytes and more) are rejected with
 * FLCE_ERR_SCRATCH_LIMIT before anything is enqueued; fitting problems run in chunks of
 * as many rows as the scratch holds. The call allocates nothing: no cudaMalloc, no
 * cudaFree, no allocating library routine.
 *
 * The first call on each device, with that device current, looks up the scratch's device
 * address (cudaGetSymbolAddress) and caches it; make that first call before any stream
 * capture. All calls share the one scratch array and it keeps the last call's contents:
 * calls that overlap on the GPU (on streams with no ordering between them) race on it. */
FLCE_API int32_t flce_fwd_bwd_noalloc(const flce_args* args, void* stream);

/* Synchronise `stream`, read the device status word and return the most severe code it
 * holds (FLCE_ERR_TIMEOUT, then FLCE_ERR_TARGET_RANGE, else FLCE_OK); FLCE_ERR_CUDA if the
 * stream reports an error. `status` is the pointer given in flce_args.status, or NULL
 * together with the workspace pointer when flce_args.status was NULL. */
FLCE_API int32_t flce_get_status(const int32_t* status, const void* workspace, void* stream);

/* Profiler: create, forget recorded launches (events are kept for reuse), destroy. */
FLCE_API flce_profile* flce_profile_create(void);
FLCE_API void flce_profile_reset(flce_profile* prof);
FLCE_API void flce_profile_destroy(flce_profile* prof);

/* Synchronise on the last recorded event, then write per stage the summed device time
 * (ms) and the number of kernel launches recorded since the last reset. `n` entries of
 * each array are written (up to FLCE_STAGE_COUNT). Returns FLCE_OK or FLCE_ERR_CUDA. */
FLCE_API int32_t flce_profile_read(flce_profile* prof, float* ms, int32_t* launches, int32_t n);

/* Name of the CUDA runtime error behind the last FLCE_ERR_CUDA returned on this host
 * thread ("cudaSuccess" if none). The string is static; do not free it. */
FLCE_API const char* flce_last_cuda_error(void);

/* Human-readable name of an flce_status value. */
FLCE_API const char* flce_status_string(int32_t code);

/* FLCE_ABI_VERSION of the loaded library. */
FLCE_API int32_t flce_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FLCE_H_ */
