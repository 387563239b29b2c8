// C ABI of libflce.so: argument validation, workspace planning and the per-call launch
// sequence. Declarations and their contracts are in include/flce.h.
//
// Launch sequence of one call (all on the caller's stream, no host synchronisation):
//   compact + ignored rows  ->  for each row chunk: gather, forward GEMM (statistics and
//   exp slab), finalize (lse, loss, prediction), gradient formation, dX GEMM, dW GEMM
//   ->  reductions.
// The number of chunks the host enqueues is cdiv(BT, R); chunks past the labelled count
// (known only on the device) exit at once, so the transient memory is the workspace the
// caller sized, whatever the labelled share.
#include <atomic>
#include <mutex>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <string>
#include <vector>

#include "flce_internal.cuh"

namespace flce {

namespace {
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t rup(int64_t a, int64_t b) { return cdiv(a, b) * b; }
inline size_t rup_sz(size_t a, size_t b) { return (a + b - 1) / b * b; }
inline bool aligned(const void* p, size_t n) { return ((uintptr_t)p % n) == 0; }
}  // namespace

bool plan_layout(int64_t BT, int64_t H, int64_t V, int dt, int64_t R, Plan* p) {
  if (BT <= 0 || H <= 0 || V <= 0 || R <= 0) return false;
  Plan q;
  q.BT = BT;
  q.H = H;
  q.V = V;
  q.esz = dtype_size(dt);
  q.Hp = rup(H, 64);
  q.nvt = cdiv(V, VT);
  q.Vp = q.nvt * VT;
  q.R = R;
  q.kmax = cdiv(BT, R);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = rup_sz(off + bytes, 256);
    return o;
  };
  q.off_ctrl = take(sizeof(Ctrl));
  q.off_idx = take(4 * (size_t)BT);
  q.off_rloss = take(4 * (size_t)BT);
  q.off_rz = take(4 * (size_t)BT);
  q.off_racc = take(4 * (size_t)BT);
  q.off_xc = take((size_t)R * q.Hp * q.esz);
  q.off_stm = take(4 * (size_t)q.nvt * R);
  q.off_sts = take(4 * (size_t)q.nvt * R);
  q.off_sti = take(4 * (size_t)q.nvt * R);
  q.off_tgt = take(4 * (size_t)R);
  q.off_lse = take(4 * (size_t)R);
  q.off_arow = take(4 * (size_t)R);
  q.off_rsc = take(4 * (size_t)R);
  q.off_rmax = take(4 * (size_t)R);
  q.off_slab = take((size_t)R * q.Vp * q.esz);
  // two fp32 dX accumulator buffers of the tensor-core path (16-bit inputs only)
  q.off_dxacc = take(q.esz == 2 ? 2 * (size_t)R * H * 4 : 0);
  q.total = off;
  *p = q;
  return true;
}

int64_t plan_rows_for_bytes(int64_t BT, int64_t H, int64_t V, int dt, size_t bytes) {
  Plan p;
  const int64_t cap = rup(BT, CHUNK_ALIGN);
  if (!plan_layout(BT, H, V, dt, CHUNK_ALIGN, &p) || p.total > bytes) return 0;
  // per-row cost from two layouts, then step down until it fits
  Plan p2;
  plan_layout(BT, H, V, dt, 2 * CHUNK_ALIGN, &p2);
  const size_t per128 = p2.total - p.total;
  int64_t R = CHUNK_ALIGN + (int64_t)((bytes - p.total) / (per128 ? per128 : 1)) * CHUNK_ALIGN;
  if (R > cap) R = cap;
  while (R > CHUNK_ALIGN) {
    if (plan_layout(BT, H, V, dt, R, &p) && p.total <= bytes) break;
    R -= CHUNK_ALIGN;
  }
  return R;
}

Work make_work(const Plan& p, void* ws, int32_t* user_status) {
  char* b = (char*)ws;
  Work w;
  w.ctrl = (Ctrl*)(b + p.off_ctrl);
  w.idx = (int*)(b + p.off_idx);
  w.rloss = (float*)(b + p.off_rloss);
  w.rz = (float*)(b + p.off_rz);
  w.racc = (float*)(b + p.off_racc);
  w.xc = b + p.off_xc;
  w.stm = (float*)(b + p.off_stm);
  w.sts = (float*)(b + p.off_sts);
  w.sti = (int*)(b + p.off_sti);
  w.tgt = (float*)(b + p.off_tgt);
  w.lse = (float*)(b + p.off_lse);
  w.arow = (float*)(b + p.off_arow);
  w.rsc = (float*)(b + p.off_rsc);
  w.rmax = (int*)(b + p.off_rmax);
  w.slab = b + p.off_slab;
  w.dxacc = (float*)(b + p.off_dxacc);
  w.status = user_status ? (int*)user_status : &w.ctrl->status;
  return w;
}

int num_sms() {
  // per-device cache; concurrent first calls may both query and store the same value
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 132;
  if (dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 132;
  if (dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

static int32_t validate(const flce_args* x) {
  if (!x) return FLCE_ERR_INVALID_ARG;
  if (x->BT <= 0 || x->H <= 0 || x->V <= 0) return FLCE_ERR_INVALID_ARG;
  if (x->BT > 0x7fffffffLL || x->H > 0x7fffffffLL || x->V > 0x7fffffffLL) return FLCE_ERR_INVALID_ARG;
  if (x->in_dtype != FLCE_F32 && x->in_dtype != FLCE_BF16 && x->in_dtype != FLCE_F16)
    return FLCE_ERR_INVALID_ARG;
  if (x->reduction != FLCE_MEAN && x->reduction != FLCE_SUM && x->reduction != FLCE_NONE)
    return FLCE_ERR_INVALID_ARG;
  if (!x->X || !x->W || !x->targets || !x->loss || !x->workspace) return FLCE_ERR_INVALID_ARG;
  if (!(x->z_loss_scale >= 0.0f) || x->z_loss_scale > 1e30f) return FLCE_ERR_INVALID_ARG;
  if (x->want_dX && !x->dX) return FLCE_ERR_INVALID_ARG;
  if (x->want_dW && !x->dW) return FLCE_ERR_INVALID_ARG;
  // dW / dbias accumulate in fp32, or in the input dtype itself (same-dtype accumulation)
  if (x->want_dW && x->dW_dtype != FLCE_F32 && x->dW_dtype != x->in_dtype) return FLCE_ERR_UNSUPPORTED;
  const int esz = dtype_size(x->in_dtype);
  if (!aligned(x->X, 16) || !aligned(x->W, 16) || !aligned(x->workspace, 256)) return FLCE_ERR_INVALID_ARG;
  if (x->want_dX && !aligned(x->dX, 16)) return FLCE_ERR_INVALID_ARG;
  if (x->want_dW && !aligned(x->dW, 16)) return FLCE_ERR_INVALID_ARG;
  if (x->bias && !aligned(x->bias, esz)) return FLCE_ERR_INVALID_ARG;
  if (x->dbias && !aligned(x->dbias, dtype_size(x->dW_dtype == FLCE_F32 ? FLCE_F32 : x->in_dtype)))
    return FLCE_ERR_INVALID_ARG;
  if (!aligned(x->targets, 8) || (x->pred && !aligned(x->pred, 8))) return FLCE_ERR_INVALID_ARG;
  if (!aligned(x->loss, 4) || (x->status && !aligned(x->status, 4))) return FLCE_ERR_INVALID_ARG;
  return FLCE_OK;
}

}  // namespace flce

using namespace flce;

static thread_local cudaError_t g_last_cuda_error = cudaSuccess;

extern "C" const char* flce_last_cuda_error(void) { return cudaGetErrorName(g_last_cuda_error); }

extern "C" flce_profile* flce_profile_create(void) { return new (std::nothrow) flce_profile(); }

extern "C" void flce_profile_reset(flce_profile* prof) {
  if (prof) prof->used = 0;
}

extern "C" void flce_profile_destroy(flce_profile* prof) {
  if (!prof) return;
  for (cudaEvent_t e : prof->ev) cudaEventDestroy(e);
  delete prof;
}

extern "C" int32_t flce_profile_read(flce_profile* prof, float* ms, int32_t* launches, int32_t n) {
  if (!prof || n < 0) return FLCE_ERR_INVALID_ARG;
  const int m = n < FLCE_STAGE_COUNT ? n : FLCE_STAGE_COUNT;
  for (int k = 0; k < m; ++k) {
    if (ms) ms[k] = 0.0f;
    if (launches) launches[k] = 0;
  }
  if (prof->used == 0) return FLCE_OK;
  if (cudaEventSynchronize(prof->ev[2 * prof->used - 1]) != cudaSuccess) return FLCE_ERR_CUDA;
  for (size_t i = 0; i < prof->used; ++i) {
    float t = 0.0f;
    if (cudaEventElapsedTime(&t, prof->ev[2 * i], prof->ev[2 * i + 1]) != cudaSuccess) return FLCE_ERR_CUDA;
    const int k = prof->stage[i];
    if (k < m) {
      if (ms) ms[k] += t;
      if (launches) launches[k] += prof->nkern[i];
    }
  }
  return FLCE_OK;
}

extern "C" size_t flce_workspace_size(int64_t BT, int64_t H, int64_t V, int32_t in_dtype,
                                      size_t budget_bytes) {
  if (BT <= 0 || H <= 0 || V <= 0) return 0;
  if (in_dtype != FLCE_F32 && in_dtype != FLCE_BF16 && in_dtype != FLCE_F16) return 0;
  const size_t budget = budget_bytes ? budget_bytes : DEFAULT_BUDGET;
  const int64_t R = plan_rows_for_bytes(BT, H, V, in_dtype, budget);
  if (R <= 0) return 0;
  Plan p;
  if (!plan_layout(BT, H, V, in_dtype, R, &p)) return 0;
  return p.total;
}

extern "C" int64_t flce_chunk_rows(int64_t BT, int64_t H, int64_t V, int32_t in_dtype,
                                   size_t workspace_bytes) {
  if (BT <= 0 || H <= 0 || V <= 0) return 0;
  if (in_dtype != FLCE_F32 && in_dtype != FLCE_BF16 && in_dtype != FLCE_F16) return 0;
  return plan_rows_for_bytes(BT, H, V, in_dtype, workspace_bytes);
}

extern "C" int64_t flce_plan_describe(int64_t BT, int64_t H, int64_t V, int32_t in_dtype,
                                      size_t workspace_bytes, char* out, size_t out_len) {
  if (BT <= 0 || H <= 0 || V <= 0) return -1;
  if (in_dtype != FLCE_F32 && in_dtype != FLCE_BF16 && in_dtype != FLCE_F16) return -1;
  if (out == nullptr && out_len != 0) return -1;
  const int64_t R = plan_rows_for_bytes(BT, H, V, in_dtype, workspace_bytes);
  Plan p;
  if (R <= 0 || !plan_layout(BT, H, V, in_dtype, R, &p)) return -1;
  static const char* const names[3] = {"f32", "bf16", "f16"};
  std::string t;
  char line[256];
  auto add = [&](const char* fmt, auto... v) {
    snprintf(line, sizeof(line), fmt, v...);
    t += line;
  };
  add("flce plan: BT=%lld H=%lld V=%lld dtype=%s workspace=%zu B (%zu B used)\n", (long long)BT,
      (long long)H, (long long)V, names[in_dtype], workspace_bytes, p.total);
  add("  chunk rows R=%lld, host chunk launches cdiv(BT,R)=%lld (the device runs cdiv(N,R) of them "
      "for N labelled rows)\n", (long long)R, (long long)p.kmax);
  add("  vocabulary tiles: %lld x %d columns (slab pitch %lld), H padded to %lld\n", (long long)p.nvt,
      VT, (long long)p.Vp, (long long)p.Hp);
  const struct {
    const char* name;
    size_t off, next;
  } reg[] = {{"ctrl", p.off_ctrl, p.off_idx},        {"idx", p.off_idx, p.off_rloss},
             {"rloss", p.off_rloss, p.off_rz},       {"rz", p.off_rz, p.off_racc},
             {"racc", p.off_racc, p.off_xc},         {"xc", p.off_xc, p.off_stm},
             {"stm", p.off_stm, p.off_sts},          {"sts", p.off_sts, p.off_sti},
             {"sti", p.off_sti, p.off_tgt},          {"tgt", p.off_tgt, p.off_lse},
             {"lse", p.off_lse, p.off_arow},         {"arow", p.off_arow, p.off_rsc},
             {"rsc", p.off_rsc, p.off_rmax},         {"rmax", p.off_rmax, p.off_slab},
             {"slab", p.off_slab, p.off_dxacc},
             {"dxacc", p.off_dxacc, p.total}};
  for (const auto& r : reg)
    if (r.next > r.off) add("  workspace %-6s at %12zu, %12zu B\n", r.name, r.off, r.next - r.off);
  if (in_dtype == FLCE_F32 || H % 8 != 0) {
    add("  GEMMs: SIMT fp32-FMA kernels (%s)\n", in_dtype == FLCE_F32 ? "fp32 inputs" : "H not a multiple of 8");
  } else {
    const int64_t mt = (R + 255) / 256, ht = (H + 255) / 256, vt = (V + 255) / 256;
    const bool wide_dw = R >= DW_WIDE_MIN_ROWS;
    const bool wide_fwd = H >= FWD_WIDE_MIN_H;
    add("  GEMMs (tcgen05, CTA pairs) per full chunk: forward %lld tiles of %s; dX %lld tiles of "
        "256x512 (K = V, up to 4 K splits); dW %lld tiles of %s; %s\n",
        (long long)(wide_fwd ? mt * ((p.nvt + 1) / 2) : mt * p.nvt), wide_fwd ? "256x512" : "256x256",
        (long long)(mt * ((ht + 1) / 2)), (long long)(wide_dw ? vt * ((ht + 1) / 2) : vt * ht),
        wide_dw ? "256x512" : "256x256",
        wide_dw ? "dX and dW in one launch over a work queue (calls with both gradients)"
                : "dX and dW in two launches");
  }
  const int64_t n = (int64_t)t.size();
  if (out_len > 0) {
    const size_t c = (size_t)n < out_len - 1 ? (size_t)n : out_len - 1;
    memcpy(out, t.data(), c);
    out[c] = '\0';
  }
  return n;
}

// FLCE_TRACE (environment, read once; any value but empty or "0"): every call prints its
// plan (flce_plan_describe) and the path it takes to stderr, before it enqueues any work.
static bool trace_enabled() {
  static const bool on = [] {
    const char* e = getenv("FLCE_TRACE");
    return e != nullptr && e[0] != '\0' && strcmp(e, "0") != 0;
  }();
  return on;
}

static void trace_call(const flce_args* x, bool tc, bool ref, const char* bwd) {
  const int64_t n = flce_plan_describe(x->BT, x->H, x->V, x->in_dtype, x->workspace_bytes, nullptr, 0);
  if (n > 0) {
    std::string t((size_t)n + 1, '\0');
    flce_plan_describe(x->BT, x->H, x->V, x->in_dtype, x->workspace_bytes, &t[0], t.size());
    fputs(t.c_str(), stderr);
  }
  static const char* const red[3] = {"mean", "sum", "none"};
  fprintf(stderr,
          "  call: reduction=%s z=%g dX=%d dW=%d bias=%d flags=0x%x; GEMMs on %s; gradient form %s; %s\n",
          red[x->reduction], (double)x->z_loss_scale, x->want_dX ? 1 : 0, x->want_dW ? 1 : 0,
          x->bias != nullptr ? 1 : 0, (unsigned)x->flags, tc ? "tcgen05" : "SIMT fp32 FMA",
          ref ? "row-reference (exp(s) slab)" : "per-tile (exp(s - tile max) slab)",
          bwd);
}

extern "C" int32_t flce_fwd_bwd(const flce_args* x, void* stream) {
  const int32_t v = validate(x);
  if (v != FLCE_OK) return v;
  const int64_t R = plan_rows_for_bytes(x->BT, x->H, x->V, x->in_dtype, x->workspace_bytes);
  if (R <= 0) return FLCE_ERR_WORKSPACE;
  Plan p;
  if (!plan_layout(x->BT, x->H, x->V, x->in_dtype, R, &p)) return FLCE_ERR_INVALID_ARG;

  CallArgs a;
  memset(&a, 0, sizeof(a));
  a.BT = x->BT;
  a.H = x->H;
  a.V = x->V;
  a.Hp = p.Hp;
  a.Vp = p.Vp;
  a.nvt = p.nvt;
  a.R = p.R;
  a.dt = x->in_dtype;
  a.reduction = x->reduction;
  a.z = x->z_loss_scale;
  a.ignore_index = x->ignore_index;
  a.X = x->X;
  a.W = x->W;
  a.bias = x->bias;
  a.targets = x->targets;
  a.grad_out = x->grad_out;
  a.loss = x->loss;
  a.z_loss = x->z_loss;
  a.acc = x->acc;
  a.lse_out = x->lse;
  a.pred = x->pred;
  a.n_labelled = x->n_labelled;
  a.want_dX = x->want_dX ? 1 : 0;
  a.want_dW = x->want_dW ? 1 : 0;
  a.dX = a.want_dX ? x->dX : nullptr;
  a.dW = a.want_dW ? x->dW : nullptr;
  a.dbias = (a.want_dW && x->bias) ? x->dbias : nullptr;
  a.dW_dt = x->dW_dtype;
  a.w = make_work(p, x->workspace, x->status);
  const uint32_t tmo_ms = x->wait_timeout_ms ? x->wait_timeout_ms : DEFAULT_TIMEOUT_MS;
  a.timeout_ns = (uint64_t)tmo_ms * 1000000ull;
  a.flags = x->flags;
  a.logit_scale = 1.0f;
  a.labels_are_masks = 0;

  cudaStream_t s = (cudaStream_t)stream;
  const bool tc = !(x->flags & FLCE_FLAG_FORCE_SIMT) && tc_supported(a);
  const bool grads = a.want_dX || a.want_dW;

#define FLCE_TRY(expr)                    \
  do {                                    \
    const cudaError_t e_ = (expr);        \
    if (e_ != cudaSuccess) {              \
      g_last_cuda_error = e_;             \
      return FLCE_ERR_CUDA;               \
    }                                     \
  } while (0)

  // Row-reference mode (bf16 tensor-core calls with gradients and no dbias): the forward
  // stores exp(s), finalize turns it into G up to one scale per row, and the gradient pass
  // over the slab is skipped. A chunk with a row outside the window is redone per tile by
  // three launches that do nothing otherwise (run_if = the chunk's flag).
  const bool ref = tc && grads && a.dt == FLCE_BF16 && a.dbias == nullptr &&
                   !(x->flags & FLCE_FLAG_NO_ROW_REF);
  if (trace_enabled())
    trace_call(x, tc, ref,
               !grads ? "no backward"
               : (tc && bwd_merged_supported(a)) ? "dX and dW in one launch"
                                                 : "backward GEMMs in separate launches");
  flce_profile* prof = x->profile;
  FLCE_TRY(cudaMemsetAsync(a.w.status, 0, sizeof(int), s));
  FLCE_TRY(staged(prof, FLCE_STAGE_PROLOGUE, 2, s, [&] { return launch_prologue(a, s); }));
  CallArgs ar = a;
  ar.ref_mode = ref ? 1 : 0;
  CallArgs afb = a;
  afb.run_if = &a.w.ctrl->fb;
  for (int k = 0; k < (int)p.kmax; ++k) {
    FLCE_TRY(staged(prof, FLCE_STAGE_GATHER, 1, s, [&] { return launch_gather(a, k, s); }));
    FLCE_TRY(staged(prof, FLCE_STAGE_FWD, 1, s,
                    [&] { return tc ? launch_fwd_tc(ar, k, s) : launch_fwd_simt(a, k, s); }));
    FLCE_TRY(staged(prof, FLCE_STAGE_FINALIZE, 1, s, [&] { return launch_finalize(ar, k, s); }));
    if (ref) {
      FLCE_TRY(staged(prof, FLCE_STAGE_GPASS, a.want_dW ? 4 : 3, s, [&] {
        cudaError_t e = a.want_dW ? launch_scale_x(ar, k, s) : cudaSuccess;
        if (e == cudaSuccess) e = launch_fwd_tc(afb, k, s);
        if (e == cudaSuccess) e = launch_finalize(afb, k, s);
        if (e == cudaSuccess) e = launch_gpass(afb, k, s);
        return e;
      }));
    } else if (grads) {
      FLCE_TRY(staged(prof, FLCE_STAGE_GPASS, 1, s, [&] { return launch_gpass(a, k, s); }));
    }
    if (tc && bwd_merged_supported(a)) {
      // dX and dW in one launch (shared work queue), then the dX sum and scatter
      FLCE_TRY(staged(prof, FLCE_STAGE_BWD, 2, s, [&] {
        cudaError_t e = cudaMemsetAsync(a.w.dxacc, 0, 2 * (size_t)a.R * a.H * 4, s);
        if (e != cudaSuccess) return e;
        e = launch_bwd_tc(ar, k, s);
        if (e != cudaSuccess) return e;
        return launch_dx_store(a, k, s);
      }));
      continue;
    }
    if (a.want_dX) {
      if (tc) {
        FLCE_TRY(staged(prof, FLCE_STAGE_DX, 2, s, [&] {
          cudaError_t e = cudaMemsetAsync(a.w.dxacc, 0, 2 * (size_t)a.R * a.H * 4, s);
          if (e != cudaSuccess) return e;
          e = launch_dx_tc(ar, k, s);
          if (e != cudaSuccess) return e;
          return launch_dx_store(a, k, s);
        }));
      } else {
        FLCE_TRY(staged(prof, FLCE_STAGE_DX, 1, s, [&] { return launch_dx_simt(a, k, s); }));
      }
    }
    if (a.want_dW)
      FLCE_TRY(staged(prof, FLCE_STAGE_DW, 1, s,
                      [&] { return tc ? launch_dw_tc(a, k, s) : launch_dw_simt(a, k, s); }));
  }
  if (a.reduction != FLCE_NONE)
    FLCE_TRY(staged(prof, FLCE_STAGE_REDUCE, 1, s, [&] { return launch_epilogue(a, s); }));
  if (a.want_dW && (x->flags & FLCE_FLAG_DW_OVERWRITE))
    FLCE_TRY(staged(prof, FLCE_STAGE_REDUCE, 1, s, [&] { return launch_zero_if_empty(a, s); }));
#undef FLCE_TRY
  return FLCE_OK;
}

extern "C" int32_t flce_scale_by(void* x, int64_t n, int32_t dtype, const float* g, void* stream) {
  if (x == nullptr || g == nullptr || n < 0) return FLCE_ERR_INVALID_ARG;
  if (dtype != FLCE_F32 && dtype != FLCE_BF16 && dtype != FLCE_F16) return FLCE_ERR_INVALID_ARG;
  if (n == 0) return FLCE_OK;
  const cudaError_t e = launch_scale_by(x, n, dtype, g, (cudaStream_t)stream);
  if (e != cudaSuccess) {
    g_last_cuda_error = e;
    return FLCE_ERR_CUDA;
  }
  return FLCE_OK;
}

extern "C" int32_t flce_get_status(const int32_t* status, const void* workspace, void* stream) {
  const int32_t* word = status;
  if (!word) {
    if (!workspace) return FLCE_ERR_INVALID_ARG;
    word = (const int32_t*)&((const Ctrl*)workspace)->status;  // Ctrl sits at offset 0
  }
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return FLCE_ERR_CUDA;
  int32_t h = 0;
  if (cudaMemcpy(&h, word, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return FLCE_ERR_CUDA;
  if (h & ST_TIMEOUT) return FLCE_ERR_TIMEOUT;
  if (h & ST_TARGET_RANGE) return FLCE_ERR_TARGET_RANGE;
  return FLCE_OK;
}

extern "C" const char* flce_status_string(int32_t code) {
  switch (code) {
    case FLCE_OK: return "FLCE_OK";
    case FLCE_ERR_INVALID_ARG: return "FLCE_ERR_INVALID_ARG";
    case FLCE_ERR_UNSUPPORTED: return "FLCE_ERR_UNSUPPORTED";
    case FLCE_ERR_TARGET_RANGE: return "FLCE_ERR_TARGET_RANGE";
    case FLCE_ERR_WORKSPACE: return "FLCE_ERR_WORKSPACE";
    case FLCE_ERR_CUDA: return "FLCE_ERR_CUDA";
    case FLCE_ERR_TIMEOUT: return "FLCE_ERR_TIMEOUT";
    case FLCE_ERR_SCRATCH_LIMIT: return "FLCE_ERR_SCRATCH_LIMIT";
    default: return "FLCE_ERR_UNKNOWN";
  }
}

extern "C" int32_t flce_abi_version(void) { return FLCE_ABI_VERSION; }
