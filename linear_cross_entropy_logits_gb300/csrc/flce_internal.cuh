// Internal declarations shared by the translation units of libflce.so.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>
#include <stddef.h>

#include "../../include/flce.h"

#include <vector>

namespace flce {

// Vocabulary tile of the forward statistics: every forward GEMM (tensor-core or SIMT)
// produces one (max, sum-exp, argmax) triple per row and per VT columns.
constexpr int VT = 256;
constexpr int CHUNK_ALIGN = 128;   // row-chunk granularity (one tensor-core M tile)
constexpr int RED_BLOCKS = 128;   // blocks of the final mean / sum reduction (a fixed split: deterministic)
// Tile-shape thresholds of the tensor-core GEMMs (the reasons are at their use in
// flce_tc.cu): the dW GEMM takes 256 x 512 pair tiles (and, with dX, the merged launch)
// from chunks of this many rows on, the forward from this hidden size on.
#ifndef FLCE_DW_WIDE_MIN_ROWS
#define FLCE_DW_WIDE_MIN_ROWS 2048
#endif
#ifndef FLCE_FWD_WIDE_MIN_H
#define FLCE_FWD_WIDE_MIN_H 4096
#endif
constexpr int DW_WIDE_MIN_ROWS = FLCE_DW_WIDE_MIN_ROWS;
constexpr int FWD_WIDE_MIN_H = FLCE_FWD_WIDE_MIN_H;
constexpr uint32_t DEFAULT_TIMEOUT_MS = 4000;
// Default workspace budget: 3 GiB, about 1% of a GB300's 288 GB of HBM. It holds the
// whole 8192-row chunk of a Llama-3.1-8B head (one pass of W per GEMM, one dW
// read-modify-write per call); callers that need less transient memory pass a budget.
constexpr size_t DEFAULT_BUDGET = (size_t)3 << 30;

// Device status bits (1 << flce_status).
constexpr int ST_TARGET_RANGE = 1 << FLCE_ERR_TARGET_RANGE;
constexpr int ST_TIMEOUT = 1 << FLCE_ERR_TIMEOUT;

// Per-call values produced on the device by the compaction kernel and read by every
// later kernel of the call (no host synchronisation anywhere).
struct Ctrl {
  int n_lab;      // rows that enter the loss
  int n_chunks;   // cdiv(n_lab, R)
  int r_eff;      // rows per chunk, a multiple of 128, <= R, balanced over the chunks
  int status;     // status word used when the caller passes none
  float cbar;     // uniform gradient factor: g/n_lab (mean), g (sum), 1 (none)
  float inv_n;    // 1/n_lab for mean (0 when n_lab == 0), 1 for sum
  int fb;         // row-reference mode: 1 when a row of the current chunk left the window
  int queue;      // work-item counter of the merged dX + dW launch (zeroed before it)
  int red_done;   // blocks of the final reduction that wrote their partial sums (zeroed by compaction)
  double red[RED_BLOCKS][3];  // per-block partial sums of loss, z-loss and accuracy
};

// Workspace layout for one call; every region is 256-byte aligned.
struct Plan {
  int64_t BT, H, V;
  int esz;       // bytes per input element
  int64_t Hp;    // X-chunk row pitch (elements), multiple of 64
  int64_t nvt;   // vocabulary tiles of VT columns
  int64_t Vp;    // slab row pitch (elements) = nvt * VT
  int64_t R;     // max rows per chunk (multiple of 128)
  int64_t kmax;  // chunks the host enqueues = cdiv(BT, R)
  size_t off_ctrl, off_idx, off_rloss, off_rz, off_racc;
  size_t off_xc, off_stm, off_sts, off_sti, off_tgt, off_lse, off_arow, off_rsc, off_rmax, off_slab,
      off_dxacc;
  size_t total;
};

inline int dtype_size(int dt) { return dt == FLCE_F32 ? 4 : 2; }
bool plan_layout(int64_t BT, int64_t H, int64_t V, int dt, int64_t R, Plan* p);
int64_t plan_rows_for_bytes(int64_t BT, int64_t H, int64_t V, int dt, size_t bytes);

// Views of the workspace regions handed to kernels.
struct Work {
  Ctrl* ctrl;
  int* idx;        // [BT] labelled rows, ascending
  float* rloss;    // [BT] per labelled row (compacted order) loss
  float* rz;       // [BT] z-loss
  float* racc;     // [BT] accuracy
  void* xc;        // [R, Hp] gathered rows of the current chunk (zero past its end)
  float* stm;      // [R, nvt] tile max; rewritten by finalize as the G multiplier
  float* sts;      // [R, nvt] tile sum of exp(s - tile max)
  int* sti;        // [R, nvt] tile argmax (lowest index)
  float* tgt;      // [R] target logit
  float* lse;      // [R] row logsumexp
  float* arow;     // [R] per-row factor a_i (g_i for none, 1 otherwise)
  float* rsc;      // [R] row-reference mode: G row scale a_i (1 + 2 z lse_i) exp(-lse_i)
  int* rmax;       // [R] largest tile maximum of the row written so far by the forward
                   // (order-preserving integer key, max_key), reset by the gather; lets a
                   // tile skip its argmax search where it cannot hold the row's maximum
  void* slab;      // [R, Vp] exp(s - tile max) (row-reference mode: exp(s)), then G, in the
                   // input dtype
  float* dxacc;    // [2, R, H] fp32 dX accumulator buffers of the tensor-core path (K
                   // splits 0-1 add into the first, 2-3 into the second)
  int* status;     // device status word
};
Work make_work(const Plan& p, void* ws, int32_t* user_status);

// Everything a kernel of one call needs (passed by value).
struct CallArgs {
  int64_t BT, H, V, Hp, Vp, nvt, R;
  int dt;
  int reduction;
  float z;
  int64_t ignore_index;
  const void* X;
  const void* W;
  const void* bias;
  const int64_t* targets;
  const float* grad_out;
  float* loss;
  float* z_loss;
  float* acc;
  float* lse_out;
  int64_t* pred;
  int32_t* n_labelled;
  void* dX;
  void* dW;        // [V, H] in dW_dt (fp32, or the input dtype for same-dtype accumulation)
  void* dbias;     // [V] in dW_dt
  int dW_dt;
  int want_dX, want_dW;
  Work w;
  uint64_t timeout_ns;
  uint32_t flags;
  float logit_scale;     // logits = (X W^T) * logit_scale + bias (1/T for distillation)
  int labels_are_masks;  // 1: any target != ignore_index marks a row (no range check)
  // Row-reference mode (bf16 tensor-core path): the forward stores exp(s) instead of
  // exp(s - tile max), so that G = rsc_i * slab' with one scale per row (slab' = the slab
  // with the target element patched by finalize); dX applies rsc in its epilogue and dW
  // reads Xc pre-scaled by rsc. No gradient pass over the slab.
  int ref_mode;
  const int* run_if;     // when set, the kernel does nothing unless *run_if != 0
};

// Row-reference window: the row max m must satisfy |m| <= REF_WINDOW so that exp(s) and
// its sums stay in the normal fp32/bf16 range, and the row scale must lie in
// [exp(-REF_SCALE_LOG), exp(REF_SCALE_LOG)] (or be 0) so that the pre-scaled Xc rows stay
// normal. A row outside sets Ctrl::fb and the chunk is redone with per-tile maxima.
constexpr float REF_WINDOW = 60.0f;
constexpr float REF_SCALE_LOG = 70.0f;

// ---- launchers (flce_kernels.cu) ----
cudaError_t launch_prologue(const CallArgs& a, cudaStream_t s);          // compact + ignored rows
cudaError_t launch_gather(const CallArgs& a, int chunk, cudaStream_t s);
cudaError_t launch_fwd_simt(const CallArgs& a, int chunk, cudaStream_t s);
cudaError_t launch_finalize(const CallArgs& a, int chunk, cudaStream_t s);
cudaError_t launch_gpass(const CallArgs& a, int chunk, cudaStream_t s);
cudaError_t launch_scale_x(const CallArgs& a, int chunk, cudaStream_t s);  // Xc rows *= rsc
cudaError_t launch_zero_if_empty(const CallArgs& a, cudaStream_t s);     // dW overwrite, N = 0
cudaError_t launch_scale_by(void* x, int64_t n, int dtype, const float* g, cudaStream_t s);
cudaError_t launch_dx_simt(const CallArgs& a, int chunk, cudaStream_t s);
cudaError_t launch_dw_simt(const CallArgs& a, int chunk, cudaStream_t s);
cudaError_t launch_epilogue(const CallArgs& a, cudaStream_t s);          // reductions

// ---- launchers (flce_tc.cu): tcgen05 tensor-core GEMMs, bf16/f16 only ----
bool tc_supported(const CallArgs& a);
cudaError_t launch_fwd_tc(const CallArgs& a, int chunk, cudaStream_t s);
cudaError_t launch_dx_tc(const CallArgs& a, int chunk, cudaStream_t s);
cudaError_t launch_dw_tc(const CallArgs& a, int chunk, cudaStream_t s);
// dX and dW in one persistent launch with a device-wide work queue; for chunks whose dW
// takes the 256 x 512 tile (bwd_merged_supported)
bool bwd_merged_supported(const CallArgs& a);
cudaError_t launch_bwd_tc(const CallArgs& a, int chunk, cudaStream_t s);
cudaError_t launch_dx_store(const CallArgs& a, int chunk, cudaStream_t s);  // dxacc -> dX rows

int num_sms();

// ---- device helpers ----
template <typename T> __device__ __forceinline__ float to_f(T v);
template <> __device__ __forceinline__ float to_f<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }
template <> __device__ __forceinline__ float to_f<__half>(__half v) { return __half2float(v); }

template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }
template <> __device__ __forceinline__ __half from_f<__half>(float v) { return __float2half_rn(v); }

// Chunk k covers compacted rows [row0, row0 + rows); false when chunk k is empty.
__device__ __forceinline__ bool chunk_bounds(const Ctrl* c, int k, int& row0, int& rows) {
  const int n = c->n_lab;
  if (k >= c->n_chunks) return false;
  row0 = k * c->r_eff;
  rows = n - row0 < c->r_eff ? n - row0 : c->r_eff;
  return rows > 0;
}

constexpr float LOG2E = 1.4426950408889634f;

// Order-preserving integer key of a float (a > b  <=>  key(a) > key(b) for non-NaN a, b),
// so that a row's running maximum can be kept with integer atomicMax.
__device__ __forceinline__ int max_key(float f) {
  const int i = __float_as_int(f);
  return i >= 0 ? i : (i ^ 0x7fffffff);
}
__device__ __forceinline__ float max_key_value(int k) {
  return __int_as_float(k >= 0 ? k : (k ^ 0x7fffffff));
}
constexpr int MAX_KEY_NEG_INF = (int)(0xff800000u ^ 0x7fffffffu);  // max_key(-inf)

}  // namespace flce

// Optional per-launch CUDA-event timing (flce_profile_*).
struct flce_profile {
  std::vector<cudaEvent_t> ev;  // pairs: ev[2i] before, ev[2i+1] after launch i
  std::vector<int> stage;       // stage of pair i
  std::vector<int> nkern;       // kernels launched by pair i
  size_t used = 0;              // pairs recorded since the last reset
};

namespace flce {
// Record `launch` on `s`, bracketed by an event pair when profiling.
template <typename F>
inline cudaError_t staged(flce_profile* prof, int stage, int nkern, cudaStream_t s, F&& launch) {
  if (!prof) return launch();
  if (prof->used * 2 + 2 > prof->ev.size()) {
    for (int i = 0; i < 2; ++i) {
      cudaEvent_t e;
      cudaError_t r = cudaEventCreate(&e);
      if (r != cudaSuccess) return r;
      prof->ev.push_back(e);
    }
    prof->stage.push_back(0);
    prof->nkern.push_back(0);
  }
  const size_t i = prof->used++;
  prof->stage[i] = stage;
  prof->nkern[i] = nkern;
  cudaError_t r = cudaEventRecord(prof->ev[2 * i], s);
  if (r != cudaSuccess) return r;
  r = launch();
  if (r != cudaSuccess) return r;
  return cudaEventRecord(prof->ev[2 * i + 1], s);
}
}  // namespace flce

