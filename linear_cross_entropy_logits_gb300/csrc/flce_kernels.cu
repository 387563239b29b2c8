// Row compaction, per-chunk gather, forward-statistics merge, gradient formation,
// reductions, and the SIMT (fp32 FMA) GEMMs used for fp32 inputs.
//
// The row-skipping idea follows "Liger-Kernel PR #1554: skip ignore_index rows"
// (Summary): rows whose target is ignore_index take no part in any product. Here the
// compaction is exact (every ignored row is removed, not only whole chunks) and happens
// on the device, so no host synchronisation is needed.
#include "flce_internal.cuh"

#include <math.h>

namespace flce {

namespace {

__host__ __device__ inline int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }
__host__ __device__ inline int64_t rup64(int64_t a, int64_t b) { return cdiv64(a, b) * b; }

__device__ __forceinline__ bool is_labelled(int64_t t, int64_t ignore_index, int64_t V) {
  return t != ignore_index && t >= 0 && t < V;
}

// ---------------------------------------------------------------------------------------
// Compaction: a stable list of labelled rows (ascending), the labelled count, the chunk
// geometry and the uniform gradient factor. One block; BT is scanned 1024 rows at a time.
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) k_compact(const __grid_constant__ CallArgs a) {
  __shared__ int warp_incl[32];
  __shared__ int s_base;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  if (tid == 0) s_base = 0;
  int bad = 0;
  __syncthreads();
  for (int64_t b0 = 0; b0 < a.BT; b0 += 1024) {
    const int64_t i = b0 + tid;
    int lab = 0;
    if (i < a.BT) {
      if (a.targets == nullptr) {
        lab = 1;  // no labels: every row takes part
      } else {
        const int64_t t = a.targets[i];
        if (t != a.ignore_index) {
          if (a.labels_are_masks || (t >= 0 && t < a.V)) lab = 1;
          else bad = 1;
        }
      }
    }
    const unsigned m = __ballot_sync(0xffffffffu, lab);
    const int wpre = __popc(m & ((1u << lane) - 1u));
    if (lane == 0) warp_incl[wid] = __popc(m);
    __syncthreads();
    if (wid == 0) {
      int v = warp_incl[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
      }
      warp_incl[lane] = v;
    }
    __syncthreads();
    const int base = s_base;
    const int wbase = wid ? warp_incl[wid - 1] : 0;
    if (lab) a.w.idx[base + wbase + wpre] = (int)i;
    __syncthreads();
    if (tid == 0) s_base = base + warp_incl[31];
    __syncthreads();
  }
  if (bad) atomicOr(a.w.status, ST_TARGET_RANGE);
  if (tid == 0) {
    // Fields are written one by one: the status word may live inside Ctrl and other
    // threads may be OR-ing into it.
    const int n = s_base;
    Ctrl* c = a.w.ctrl;
    const int nch = n > 0 ? (int)cdiv64(n, a.R) : 0;
    c->n_lab = n;
    c->n_chunks = nch;
    c->red_done = 0;
    c->r_eff = n > 0 ? (int)rup64(cdiv64(n, nch), CHUNK_ALIGN) : 0;
    float g = 1.0f;
    if (a.reduction != FLCE_NONE && a.grad_out != nullptr) g = a.grad_out[0];
    if (a.reduction == FLCE_MEAN) {
      c->cbar = n > 0 ? g / (float)n : 0.0f;
      c->inv_n = n > 0 ? 1.0f / (float)n : 0.0f;
    } else if (a.reduction == FLCE_SUM) {
      c->cbar = g;
      c->inv_n = 1.0f;
    } else {
      c->cbar = 1.0f;
      c->inv_n = 1.0f;
    }
    if (a.n_labelled) *a.n_labelled = n;
  }
}

// Ignored rows: per-token outputs (PR #1554, Details item 1) and a zero dX row.
__global__ void __launch_bounds__(256) k_ignored(const __grid_constant__ CallArgs a) {
  if (a.targets == nullptr) return;  // no labels: no ignored rows
  for (int64_t i = blockIdx.x; i < a.BT; i += gridDim.x) {
    const int64_t t = a.targets[i];
    if (a.labels_are_masks ? t != a.ignore_index : is_labelled(t, a.ignore_index, a.V)) continue;
    if (threadIdx.x == 0) {
      if (a.reduction == FLCE_NONE) {
        if (a.loss) a.loss[i] = 0.0f;
        if (a.z_loss) a.z_loss[i] = 0.0f;
        if (a.acc) a.acc[i] = 0.0f;
      }
      if (a.lse_out) a.lse_out[i] = 0.0f;
      if (a.pred) a.pred[i] = -1;
    }
    if (a.want_dX) {
      const int esz = a.dt == FLCE_F32 ? 4 : 2;
      const int64_t bytes = a.H * esz;
      char* row = (char*)a.dX + i * bytes;
      if ((bytes & 15) == 0) {
        uint4* r4 = (uint4*)row;
        for (int64_t j = threadIdx.x; j < bytes / 16; j += blockDim.x) r4[j] = make_uint4(0, 0, 0, 0);
      } else {
        for (int64_t j = threadIdx.x; j < bytes; j += blockDim.x) row[j] = 0;
      }
    }
  }
}

// ---------------------------------------------------------------------------------------
// Gather the chunk's labelled rows of X into the dense chunk buffer; rows past the chunk
// end (up to the next multiple of 128) and columns past H are zero, so that no stale or
// uninitialised value ever enters a GEMM.
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_gather(const __grid_constant__ CallArgs a, int chunk) {
  int row0, rows;
  if (!chunk_bounds(a.w.ctrl, chunk, row0, rows)) return;
  if (blockIdx.x == 0 && threadIdx.x == 0) a.w.ctrl->fb = 0;  // row-reference window flag
  const int lim = (int)rup64(rows, CHUNK_ALIGN);
  const int esz = a.dt == FLCE_F32 ? 4 : 2;
  const int64_t src_bytes = a.H * esz, dst_bytes = a.Hp * esz;
  // 64 threads per row, four rows per block at a time; each thread keeps up to eight 16-byte
  // loads in flight before it stores them
  const int grp = threadIdx.x >> 6, lt = threadIdx.x & 63;
  for (int r = blockIdx.x * 4 + grp; r < lim; r += gridDim.x * 4) {
    if (lt == 0 && a.w.rmax != nullptr) a.w.rmax[r] = MAX_KEY_NEG_INF;
    char* dst = (char*)a.w.xc + (int64_t)r * dst_bytes;
    if (r < rows) {
      const char* src = (const char*)a.X + (int64_t)a.w.idx[row0 + r] * src_bytes;
      if ((src_bytes & 15) == 0) {
        const uint4* s4 = (const uint4*)src;
        uint4* d4 = (uint4*)dst;
        const int64_t n16 = src_bytes / 16;
        for (int64_t j0 = lt; j0 < n16; j0 += 64 * 8) {
          uint4 v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u)
            if (j0 + 64 * u < n16) v[u] = s4[j0 + 64 * u];
#pragma unroll
          for (int u = 0; u < 8; ++u)
            if (j0 + 64 * u < n16) d4[j0 + 64 * u] = v[u];
        }
      } else {
        for (int64_t j = lt; j < src_bytes; j += 64) dst[j] = src[j];
      }
      for (int64_t j = src_bytes + lt; j < dst_bytes; j += 64) dst[j] = 0;
    } else {
      uint4* d4 = (uint4*)dst;
      for (int64_t j = lt; j < dst_bytes / 16; j += 64) d4[j] = make_uint4(0, 0, 0, 0);
    }
  }
}

// ---------------------------------------------------------------------------------------
// Finalize: one warp per row merges the row's per-tile (max, sum-exp, argmax) triples,
// giving lse, loss, z-loss, prediction and accuracy; then turns each tile max into the
// multiplier that maps the stored exp(s - tile max) to the row's gradient
// a_i (1 + 2 z lse) exp(s - lse). The merge order is fixed (lane-strided tiles, then an
// xor butterfly whose combine is commutative), so every lane and every run agree bitwise.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void lse_combine(float& M, float& S, int& am, float M2, float S2, int a2) {
  const float Mn = fmaxf(M, M2);
  const float Sn = Mn == -INFINITY ? 0.0f : S * expf(M - Mn) + S2 * expf(M2 - Mn);
  am = M > M2 ? am : (M2 > M ? a2 : min(am, a2));
  M = Mn;
  S = Sn;
}

// Row-reference mode: the tile sums are all relative to the same reference (0), so they
// add; the maxima only decide the argmax and the window.
__device__ __forceinline__ void ref_combine(float& M, float& S, int& am, float M2, float S2, int a2) {
  am = M > M2 ? am : (M2 > M ? a2 : min(am, a2));
  M = fmaxf(M, M2);
  S += S2;
}

__global__ void __launch_bounds__(256) k_finalize(const __grid_constant__ CallArgs a, int chunk) {
  if (a.run_if != nullptr && *a.run_if == 0) return;
  int row0, rows;
  if (!chunk_bounds(a.w.ctrl, chunk, row0, rows)) return;
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (r >= rows) return;  // warp-uniform
  const int nvt = (int)a.nvt;
  float* stm = a.w.stm + (int64_t)r * nvt;
  const float* sts = a.w.sts + (int64_t)r * nvt;
  const int* sti = a.w.sti + (int64_t)r * nvt;

  float M = -INFINITY, S = 0.0f;
  int am = 0x7fffffff;
  if (a.ref_mode) {
    // eight tiles' loads per lane in flight, merged in the same order as one at a time
    int t = lane;
    for (; t + 32 * 7 < nvt; t += 32 * 8) {
      float m8[8], s8[8];
      int i8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        m8[u] = stm[t + 32 * u];
        s8[u] = sts[t + 32 * u];
        i8[u] = sti[t + 32 * u];
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) ref_combine(M, S, am, m8[u], s8[u], i8[u]);
    }
    for (; t < nvt; t += 32) ref_combine(M, S, am, stm[t], sts[t], sti[t]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float M2 = __shfl_xor_sync(0xffffffffu, M, o);
      const float S2 = __shfl_xor_sync(0xffffffffu, S, o);
      const int a2 = __shfl_xor_sync(0xffffffffu, am, o);
      ref_combine(M, S, am, M2, S2, a2);
    }
  } else {
    for (int t = lane; t < nvt; t += 32) lse_combine(M, S, am, stm[t], sts[t], sti[t]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float M2 = __shfl_xor_sync(0xffffffffu, M, o);
      const float S2 = __shfl_xor_sync(0xffffffffu, S, o);
      const int a2 = __shfl_xor_sync(0xffffffffu, am, o);
      lse_combine(M, S, am, M2, S2, a2);
    }
  }
  const float lse = a.ref_mode ? logf(S) : M + logf(S);

  const int row = a.w.idx[row0 + r];
  const int64_t tg = a.targets[row];
  float ar = 1.0f;
  if (a.reduction == FLCE_NONE && a.grad_out != nullptr) ar = a.grad_out[row];
  const float zf = 1.0f + 2.0f * a.z * lse;
  if (a.ref_mode) {
    // G_iv = rsc_i * slab'_iv with rsc_i = a_i (1 + 2 z lse_i) exp(-lse_i); the target
    // element becomes exp(s_t) - exp(lse_i) / (1 + 2 z lse_i), so that rsc_i times it is
    // a_i ((1 + 2 z lse_i) p_t - 1). Rows outside the window flag the chunk.
    const float sc = ar * zf * expf(-lse);
    const bool ok = fabsf(M) <= REF_WINDOW && S > 0.0f && isfinite(S) && fabsf(zf) >= 1e-3f &&
                    (sc == 0.0f || fabsf(logf(fabsf(sc))) <= REF_SCALE_LOG);
    if (lane != 0) return;
    if (!ok) {
      a.w.ctrl->fb = 1;
    } else {
      a.w.rsc[r] = sc;
      ((__nv_bfloat16*)a.w.slab)[(int64_t)r * a.Vp + tg] =
          __float2bfloat16_rn(expf(a.w.tgt[r]) - expf(lse) / zf);
    }
  } else {
    const float f = ar * zf;
    for (int t = lane; t < nvt; t += 32) stm[t] = f * expf(stm[t] - lse);
    if (lane != 0) return;
  }
  const float zl = a.z * lse * lse;
  const float loss = (lse - a.w.tgt[r]) + zl;
  const float accv = ((int64_t)am == tg) ? 1.0f : 0.0f;
  a.w.lse[r] = lse;
  a.w.arow[r] = ar;
  if (a.lse_out) a.lse_out[row] = lse;
  if (a.pred) a.pred[row] = am;
  if (a.reduction == FLCE_NONE) {
    a.loss[row] = loss;
    if (a.z_loss) a.z_loss[row] = zl;
    if (a.acc) a.acc[row] = accv;
  }
  a.w.rloss[row0 + r] = loss;
  a.w.rz[row0 + r] = zl;
  a.w.racc[row0 + r] = accv;
}

// ---------------------------------------------------------------------------------------
// Gradient formation: G[r, v] = mult[r, tile(v)] * e[r, v] - a_r [v == t_r], in place in
// the slab; rows past the chunk end up to the next multiple of 64 are zeroed (the dW GEMM
// reduces over them). With dbias wanted, one block owns a whole column strip and adds its
// column sums to dbias in a fixed order.
// ---------------------------------------------------------------------------------------
template <typename T> struct Vec8;
template <> struct Vec8<__nv_bfloat16> {
  __device__ static void load(const __nv_bfloat16* p, float (&f)[8]) {
    const uint4 u = *(const uint4*)p;
    const __nv_bfloat162* h = (const __nv_bfloat162*)&u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 x = __bfloat1622float2(h[j]);
      f[2 * j] = x.x;
      f[2 * j + 1] = x.y;
    }
  }
  __device__ static void store(__nv_bfloat16* p, const float (&f)[8]) {
    uint4 u;
    __nv_bfloat162* h = (__nv_bfloat162*)&u;
#pragma unroll
    for (int j = 0; j < 4; ++j) h[j] = __floats2bfloat162_rn(f[2 * j], f[2 * j + 1]);
    *(uint4*)p = u;
  }
};
template <> struct Vec8<__half> {
  __device__ static void load(const __half* p, float (&f)[8]) {
    const uint4 u = *(const uint4*)p;
    const __half2* h = (const __half2*)&u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 x = __half22float2(h[j]);
      f[2 * j] = x.x;
      f[2 * j + 1] = x.y;
    }
  }
  __device__ static void store(__half* p, const float (&f)[8]) {
    uint4 u;
    __half2* h = (__half2*)&u;
#pragma unroll
    for (int j = 0; j < 4; ++j) h[j] = __floats2half2_rn(f[2 * j], f[2 * j + 1]);
    *(uint4*)p = u;
  }
};
template <> struct Vec8<float> {
  __device__ static void load(const float* p, float (&f)[8]) {
    const float4 x = *(const float4*)p, y = *(const float4*)(p + 4);
    f[0] = x.x; f[1] = x.y; f[2] = x.z; f[3] = x.w;
    f[4] = y.x; f[5] = y.y; f[6] = y.z; f[7] = y.w;
  }
  __device__ static void store(float* p, const float (&f)[8]) {
    *(float4*)p = make_float4(f[0], f[1], f[2], f[3]);
    *(float4*)(p + 4) = make_float4(f[4], f[5], f[6], f[7]);
  }
};

template <typename T>
__global__ void __launch_bounds__(256) k_gpass(const __grid_constant__ CallArgs a, int chunk,
                                               int rows_per_block, int do_dbias) {
  if (a.run_if != nullptr && *a.run_if == 0) return;
  int row0, rows;
  if (!chunk_bounds(a.w.ctrl, chunk, row0, rows)) return;
  const int t = blockIdx.x;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int rlim = (int)rup64(rows, 64);
  const int rb0 = blockIdx.y * rows_per_block;
  const int rb1 = min(rb0 + rows_per_block, rlim);
  const int64_t c0 = (int64_t)t * VT + tx * 8;
  T* slab = (T*)a.w.slab;
  float cs[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int r = rb0 + ty; r < rb1; r += 8) {
    T* p = slab + (int64_t)r * a.Vp + c0;
    float f[8];
    if (r < rows) {
      const float m = a.w.stm[(int64_t)r * a.nvt + t];
      const float ar = a.w.arow[r];
      const int64_t tg = a.targets[a.w.idx[row0 + r]];
      Vec8<T>::load(p, f);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float g = m * f[j];
        if (c0 + j == tg) g -= ar;
        f[j] = g;
        cs[j] += g;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) f[j] = 0.0f;
    }
    Vec8<T>::store(p, f);
  }
  if (do_dbias) {
    __shared__ float red[8][VT];
#pragma unroll
    for (int j = 0; j < 8; ++j) red[ty][tx * 8 + j] = cs[j];
    __syncthreads();
    const float cb = a.w.ctrl->cbar;
    for (int c = threadIdx.x; c < VT; c += blockDim.x) {
      float s = 0.0f;
#pragma unroll
      for (int y = 0; y < 8; ++y) s += red[y][c];
      const int64_t v = (int64_t)t * VT + c;
      if (v < a.V) {
        const bool ovw = (a.flags & FLCE_FLAG_DW_OVERWRITE) && chunk == 0;
        if (a.dW_dt == FLCE_F32) {
          float* db = (float*)a.dbias;
          db[v] = ovw ? cb * s : db[v] + cb * s;
        } else {
          T* db = (T*)a.dbias;  // same-dtype accumulation
          db[v] = from_f<T>(ovw ? cb * s : to_f<T>(db[v]) + cb * s);
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------------------
// Row-reference mode: Xc rows *= rsc (bf16, in place) for the dW GEMM, unless the chunk
// left the window (then Xc stays as gathered for the per-tile redo).
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_scale_x(const __grid_constant__ CallArgs a, int chunk) {
  int row0, rows;
  if (!chunk_bounds(a.w.ctrl, chunk, row0, rows)) return;
  if (a.w.ctrl->fb) return;
  // 64 threads per row (a row is Hp / 8 16-byte units; the pad columns hold zeros, which
  // stay zero), up to eight units in flight per thread
  const int grp = threadIdx.x >> 6, lt = threadIdx.x & 63;
  const int64_t n16 = a.Hp / 8;
  for (int r = blockIdx.x * 4 + grp; r < rows; r += gridDim.x * 4) {
    const float sc = a.w.rsc[r];
    uint4* xr = (uint4*)((__nv_bfloat16*)a.w.xc + (int64_t)r * a.Hp);
    for (int64_t j0 = lt; j0 < n16; j0 += 64 * 8) {
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (j0 + 64 * u < n16) v[u] = xr[j0 + 64 * u];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (j0 + 64 * u >= n16) continue;
        __nv_bfloat162* h = (__nv_bfloat162*)&v[u];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 f = __bfloat1622float2(h[k]);
          h[k] = __floats2bfloat162_rn(f.x * sc, f.y * sc);
        }
        xr[j0 + 64 * u] = v[u];
      }
    }
  }
}

// ---------------------------------------------------------------------------------------
// dW / dbias overwrite with no labelled row: no chunk ran, so the destinations are zeroed
// here (every block returns at once when n_lab > 0).
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_zero_if_empty(const __grid_constant__ CallArgs a) {
  if (a.w.ctrl->n_lab > 0) return;
  const int esz = a.dW_dt == FLCE_F32 ? 4 : 2;
  const int64_t nw = a.V * a.H * esz, nb = a.dbias ? a.V * esz : 0;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nw; i += stride)
    ((char*)a.dW)[i] = 0;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nb; i += stride)
    ((char*)a.dbias)[i] = 0;
}

// x[i] *= *g unless *g == 1 (device-side test; see flce_scale_by).
template <typename T>
__global__ void __launch_bounds__(256) k_scale_by(T* x, int64_t n, const float* g) {
  const float f = *g;
  if (f == 1.0f) return;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    x[i] = from_f<T>(to_f<T>(x[i]) * f);
}

// ---------------------------------------------------------------------------------------
// Final reductions (mean/sum) of loss, z-loss and accuracy over the labelled rows, in a
// fixed order (deterministic): block b adds rows [b*per, (b+1)*per) in float64, and the
// last block to finish adds the RED_BLOCKS partial sums in block order. GB300 runs float64
// at a small fraction of its fp32 rate, so one block alone would take tens of microseconds.
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_reduce(const __grid_constant__ CallArgs a) {
  __shared__ double red[3][8];
  __shared__ bool last;
  Ctrl* c = a.w.ctrl;
  const int n = c->n_lab;
  const int per = (n + RED_BLOCKS - 1) / RED_BLOCKS;
  const int i0 = blockIdx.x * per, i1 = min(n, i0 + per);
  double s0 = 0.0, s1 = 0.0, s2 = 0.0;
  for (int i = i0 + threadIdx.x; i < i1; i += blockDim.x) {
    s0 += a.w.rloss[i];
    s1 += a.w.rz[i];
    s2 += a.w.racc[i];
  }
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s0 += __shfl_down_sync(0xffffffffu, s0, o);
    s1 += __shfl_down_sync(0xffffffffu, s1, o);
    s2 += __shfl_down_sync(0xffffffffu, s2, o);
  }
  if (lane == 0) {
    red[0][wid] = s0;
    red[1][wid] = s1;
    red[2][wid] = s2;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double q[3] = {0.0, 0.0, 0.0};
    for (int w = 0; w < 8; ++w)
      for (int k = 0; k < 3; ++k) q[k] += red[k][w];
    for (int k = 0; k < 3; ++k) c->red[blockIdx.x][k] = q[k];
    __threadfence();
    last = atomicAdd(&c->red_done, 1) == RED_BLOCKS - 1;
  }
  __syncthreads();
  if (!last || wid != 0) return;
  // the last block to finish adds the partial sums in block order
  __threadfence();
  s0 = s1 = s2 = 0.0;
  for (int b = lane; b < RED_BLOCKS; b += 32) {
    s0 += __ldcg(&c->red[b][0]);
    s1 += __ldcg(&c->red[b][1]);
    s2 += __ldcg(&c->red[b][2]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s0 += __shfl_down_sync(0xffffffffu, s0, o);
    s1 += __shfl_down_sync(0xffffffffu, s1, o);
    s2 += __shfl_down_sync(0xffffffffu, s2, o);
  }
  if (lane == 0) {
    double d = 1.0;
    if (a.reduction == FLCE_MEAN) d = n > 0 ? (double)n : 0.0;
    const double q0 = d > 0.0 ? s0 / d : 0.0, q1 = d > 0.0 ? s1 / d : 0.0, q2 = d > 0.0 ? s2 / d : 0.0;
    a.loss[0] = (float)q0;
    if (a.z_loss) a.z_loss[0] = (float)q1;
    if (a.acc) a.acc[0] = (float)q2;
    c->red_done = 0;
  }
}

// ---------------------------------------------------------------------------------------
// SIMT GEMM core (fp32 FMA; the fp32-input path, and 16-bit inputs whose H is not a
// multiple of 8 or that force it): one block computes a (16 TM) x (16 TN) tile of
// C = A B over K. 256 threads as 16 x 16; thread (ty, tx) keeps TM x TN accumulators for
// rows ty*4 + 64*(i/4) + i%4 and columns tx*4 + 64*(j/4) + j%4, so that its shared-memory
// reads are float4 and a warp's reads hit distinct banks (or broadcast). The operands
// pass through shared memory SK = 16 k at a time, in two buffers: the next step's elements
// are loaded into registers while the current step is multiplied.
// KC: the operand's K index is the contiguous one (element (e, k) at p[e * ld + k]);
// otherwise its row index e is (p[k * ld + e]). Elements outside the extents read as 0.
// ---------------------------------------------------------------------------------------
// Row / column of accumulator (i, j) of thread (ty, tx) within the block tile.
__device__ __forceinline__ int simt_row(int i, int ty) { return (i >> 2) * 64 + ty * 4 + (i & 3); }
__device__ __forceinline__ int simt_col(int j, int tx) { return (j >> 2) * 64 + tx * 4 + (j & 3); }
// Thread coordinates in the 16 x 16 grid. The index that keeps more accumulators per thread
// runs slower across a warp, so a warp's reads of that operand are two float4 broadcasts
// (the forward's 4 x 16 accumulators per thread: 6 shared-memory wavefronts per k, not 9).
template <int TM, int TN>
__device__ __forceinline__ void simt_txy(int tid, int& tx, int& ty) {
  if (TN > TM) {
    ty = tid & 15;
    tx = tid >> 4;
  } else {
    tx = tid & 15;
    ty = tid >> 4;
  }
}

constexpr int SK = 16;

template <typename T, int E, bool KC>
struct SimtOperand {
  static constexpr int PER = E * SK / 256;  // elements per thread per step
  static constexpr int PITCH = E + 4;       // shared-memory row pitch (floats, 16-byte rows)
  float r[PER];
  __device__ __forceinline__ void load(const T* p, int64_t ld, int64_t e0, int64_t ext, int64_t k0, int64_t K,
                                       int tid) {
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      int e, k;
      if (KC) {
        k = tid % SK;
        e = tid / SK + (256 / SK) * i;
      } else {
        e = tid % E;
        k = tid / E + (256 / E) * i;
      }
      const int64_t ge = e0 + e, gk = k0 + k;
      r[i] = (ge < ext && gk < K) ? to_f<T>(KC ? p[ge * ld + gk] : p[gk * ld + ge]) : 0.0f;
    }
  }
  __device__ __forceinline__ void store(float* s, int tid) const {
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      int e, k;
      if (KC) {
        k = tid % SK;
        e = tid / SK + (256 / SK) * i;
      } else {
        e = tid % E;
        k = tid / E + (256 / E) * i;
      }
      s[k * PITCH + e] = r[i];
    }
  }
};

template <int TM, int TN>
__device__ __forceinline__ void simt_step(const float* as, const float* bs, float (&acc)[TM][TN], int ty, int tx) {
  constexpr int PA = 16 * TM + 4, PB = 16 * TN + 4;
#pragma unroll
  for (int k = 0; k < SK; ++k) {
    float av[TM], bv[TN];
#pragma unroll
    for (int g = 0; g < TM / 4; ++g) {
      const float4 v = *(const float4*)&as[k * PA + g * 64 + ty * 4];
      av[4 * g] = v.x;
      av[4 * g + 1] = v.y;
      av[4 * g + 2] = v.z;
      av[4 * g + 3] = v.w;
    }
#pragma unroll
    for (int g = 0; g < TN / 4; ++g) {
      const float4 v = *(const float4*)&bs[k * PB + g * 64 + tx * 4];
      bv[4 * g] = v.x;
      bv[4 * g + 1] = v.y;
      bv[4 * g + 2] = v.z;
      bv[4 * g + 3] = v.w;
    }
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
  }
}

// Shared memory of one block tile: two buffers of each operand's 16-k slice.
template <int TM, int TN>
__host__ __device__ constexpr int simt_smem_floats() {
  return 2 * SK * ((16 * TM + 4) + (16 * TN + 4));
}

// acc = A[m0 : m0 + 16 TM, 0 : K] B[0 : K, n0 : n0 + 16 TN] (rows past M / columns past N
// and k past K count as zero). Every thread of the block calls it.
template <typename T, int TM, int TN, bool AKC, bool BKC>
__device__ __forceinline__ void simt_gemm_tile(const T* A, int64_t lda, int64_t m0, int64_t M, const T* B,
                                               int64_t ldb, int64_t n0, int64_t N, int64_t K, float* smem,
                                               float (&acc)[TM][TN]) {
  constexpr int BM = 16 * TM, BN = 16 * TN;
  constexpr int SA = SK * (BM + 4), SB = SK * (BN + 4);
  const int tid = threadIdx.x;
  int tx, ty;
  simt_txy<TM, TN>(tid, tx, ty);
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) acc[i][j] = 0.0f;
  const int64_t nk = (K + SK - 1) / SK;
  if (nk == 0) return;
  SimtOperand<T, BM, AKC> oa;
  SimtOperand<T, BN, BKC> ob;
  oa.load(A, lda, m0, M, 0, K, tid);
  ob.load(B, ldb, n0, N, 0, K, tid);
  oa.store(smem, tid);
  ob.store(smem + 2 * SA, tid);
  __syncthreads();
  for (int64_t kt = 0; kt < nk; ++kt) {
    const int cur = (int)(kt & 1), nxt = cur ^ 1;
    const bool more = kt + 1 < nk;
    if (more) {
      oa.load(A, lda, m0, M, (kt + 1) * SK, K, tid);
      ob.load(B, ldb, n0, N, (kt + 1) * SK, K, tid);
    }
    simt_step<TM, TN>(smem + cur * SA, smem + 2 * SA + cur * SB, acc, ty, tx);
    if (more) {
      oa.store(smem + nxt * SA, tid);
      ob.store(smem + 2 * SA + nxt * SB, tid);
    }
    __syncthreads();
  }
}


// ---------------------------------------------------------------------------------------
// SIMT forward: a 64-row x 256-column logit tile per block (one vocabulary tile), then the
// same per-tile statistics and stored exp(s - tile max) as the tensor-core forward. The
// tile is staged in shared memory 32 rows at a time for the row statistics.
// ---------------------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256, 2) k_fwd_simt(const __grid_constant__ CallArgs a, int chunk) {
  int row0, rows;
  if (!chunk_bounds(a.w.ctrl, chunk, row0, rows)) return;
  const int mb = blockIdx.x;
  if (mb * 64 >= rows) return;
  const int t = blockIdx.y;
  __shared__ __align__(16) float smem[simt_smem_floats<4, 16>()];
  static_assert(simt_smem_floats<4, 16>() >= 32 * 257, "row staging");
  float acc[4][16];
  simt_gemm_tile<T, 4, 16, true, true>((const T*)a.w.xc, a.Hp, (int64_t)mb * 64, rows, (const T*)a.W, a.H,
                                       (int64_t)t * VT, a.V, a.H, smem, acc);
  const int tid = threadIdx.x;
  int tx, ty;
  simt_txy<4, 16>(tid, tx, ty);
  const int64_t V = a.V;
  float bj[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int64_t v = (int64_t)t * VT + simt_col(j, tx);
    bj[j] = (a.bias != nullptr && v < V) ? to_f<T>(((const T*)a.bias)[v]) : 0.0f;
  }
  float* Ss = smem;  // Ss[r * 257 + c], 32 rows
  const int lane = tid & 31, warp = tid >> 5;
  T* slab = (T*)a.w.slab;
  for (int h = 0; h < 2; ++h) {
    if ((ty >> 3) == h) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 16; ++j)
          Ss[(ty * 4 + i - 32 * h) * 257 + simt_col(j, tx)] = fmaf(acc[i][j], a.logit_scale, bj[j]);
    }
    __syncthreads();
    for (int il = warp; il < 32; il += 8) {
      const int rr = mb * 64 + 32 * h + il;
      if (rr >= rows) continue;
      const int64_t tg = a.targets ? a.targets[a.w.idx[row0 + rr]] : -1;
      float mx = -INFINITY;
      int ai = t * VT;
      float tl = 0.0f;
      bool ht = false;
      for (int j = lane; j < VT; j += 32) {
        const int64_t v = (int64_t)t * VT + j;
        if (v < V) {
          const float s = Ss[il * 257 + j];
          if (s > mx) {
            mx = s;
            ai = (int)v;
          }
          if (v == tg) {
            tl = s;
            ht = true;
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, mx, o);
        const int oi = __shfl_xor_sync(0xffffffffu, ai, o);
        if (om > mx || (om == mx && oi < ai)) {
          mx = om;
          ai = oi;
        }
      }
      float sum = 0.0f;
      for (int j = lane; j < VT; j += 32) {
        const int64_t v = (int64_t)t * VT + j;
        const float e = v < V ? expf(Ss[il * 257 + j] - mx) : 0.0f;
        sum += e;
        slab[(int64_t)rr * a.Vp + v] = from_f<T>(e);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      const unsigned hb = __ballot_sync(0xffffffffu, ht);
      if (hb) tl = __shfl_sync(0xffffffffu, tl, __ffs(hb) - 1);
      if (lane == 0) {
        const int64_t o = (int64_t)rr * a.nvt + t;
        a.w.stm[o] = mx;
        a.w.sts[o] = sum;
        a.w.sti[o] = ai;
        if (hb) a.w.tgt[rr] = tl;
      }
    }
    __syncthreads();  // the staging rows are rewritten by the next half
  }
}

// ---------------------------------------------------------------------------------------
// SIMT GEMMs of the backward, (16 TL) x (16 TL) output tiles on the core above (TL = 8;
// 4 when the 128 x 128 grid would leave most SMs idle: every output still sums its k in
// the same order, so the two tile sizes give the same bits).
//   MODE 0 (dX): dX[idx[r]] = cbar * sum_v G[r, v] W[v, :]        (M = rows, K = V)
//   MODE 1 (dW): dW[v]     += cbar * sum_r G[r, v] Xc[r, :]       (M = V, K = rows)
// ---------------------------------------------------------------------------------------
template <typename T, int MODE, int TL>
__global__ void __launch_bounds__(256, 2) k_gemm_simt(const __grid_constant__ CallArgs a, int chunk) {
  int row0, rows;
  if (!chunk_bounds(a.w.ctrl, chunk, row0, rows)) return;
  // dW overwrite: the first chunk stores, later chunks accumulate
  const bool ovw = (a.flags & FLCE_FLAG_DW_OVERWRITE) && chunk == 0;
  const int64_t M = MODE == 0 ? rows : a.V;
  const int64_t N = a.H;
  const int64_t K = MODE == 0 ? a.V : rows;
  const int64_t m0 = (int64_t)blockIdx.y * (16 * TL), n0 = (int64_t)blockIdx.x * (16 * TL);
  if (m0 >= M) return;
  __shared__ __align__(16) float smem[simt_smem_floats<TL, TL>()];
  float acc[TL][TL];
  const T* G = (const T*)a.w.slab;
  if constexpr (MODE == 0)
    simt_gemm_tile<T, TL, TL, true, false>(G, a.Vp, m0, M, (const T*)a.W, a.H, n0, N, K, smem, acc);
  else
    simt_gemm_tile<T, TL, TL, false, false>(G, a.Vp, m0, M, (const T*)a.w.xc, a.Hp, n0, N, K, smem, acc);
  const int tid = threadIdx.x;
  int tx, ty;
  simt_txy<TL, TL>(tid, tx, ty);
  const float cb = a.w.ctrl->cbar;
#pragma unroll
  for (int i = 0; i < TL; ++i) {
    const int64_t m = m0 + simt_row(i, ty);
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < TL; ++j) {
      const int64_t n = n0 + simt_col(j, tx);
      if (n >= N) continue;
      if (MODE == 0) {
        const int64_t orow = a.w.idx[row0 + m];
        ((T*)a.dX)[orow * a.H + n] = from_f<T>(cb * acc[i][j]);
      } else if (a.dW_dt == FLCE_F32) {
        float* w = (float*)a.dW + m * a.H + n;
        *w = ovw ? cb * acc[i][j] : *w + cb * acc[i][j];
      } else {
        T* w = (T*)a.dW + m * a.H + n;  // same-dtype accumulation
        *w = from_f<T>(ovw ? cb * acc[i][j] : to_f<T>(*w) + cb * acc[i][j]);
      }
    }
  }
}

// dX rows of the chunk: dX[idx[row0 + r]] = dxacc[r] in the input dtype (the tensor-core
// dX GEMM accumulates cbar * G W into the fp32 buffer dxacc).
template <typename T>
__global__ void __launch_bounds__(256) k_dx_store(const __grid_constant__ CallArgs a, int chunk) {
  int row0, rows;
  if (!chunk_bounds(a.w.ctrl, chunk, row0, rows)) return;
  const int64_t H = a.H;
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    const float* src = a.w.dxacc + (int64_t)r * H;
    const float* src2 = src + a.R * H;  // second accumulator buffer (K splits 2-3)
    T* dst = (T*)a.dX + (int64_t)a.w.idx[row0 + r] * H;
    for (int64_t j = (int64_t)threadIdx.x * 8; j < H; j += (int64_t)blockDim.x * 8) {
      float f[8], g[8];
      Vec8<float>::load(src + j, f);
      Vec8<float>::load(src2 + j, g);
#pragma unroll
      for (int k = 0; k < 8; ++k) f[k] += g[k];
      Vec8<T>::store(dst + j, f);
    }
  }
}

template <typename T>
cudaError_t gpass_t(const CallArgs& a, int chunk, cudaStream_t s) {
  const bool dbias = a.want_dW && a.bias != nullptr && a.dbias != nullptr;
  const int rlim = (int)rup64(a.R, 64);
  int rpb = dbias ? rlim : 256;
  const int ry = (int)cdiv64(rlim, rpb);
  dim3 grid((unsigned)a.nvt, (unsigned)ry);
  k_gpass<T><<<grid, 256, 0, s>>>(a, chunk, rpb, dbias ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prologue(const CallArgs& a, cudaStream_t s) {
  k_compact<<<1, 1024, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t blocks = a.BT < 8LL * num_sms() ? a.BT : 8LL * num_sms();
  k_ignored<<<(unsigned)blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_gather(const CallArgs& a, int chunk, cudaStream_t s) {
  const int64_t blocks = cdiv64(a.R, 4) < 4LL * num_sms() ? cdiv64(a.R, 4) : 4LL * num_sms();
  k_gather<<<(unsigned)blocks, 256, 0, s>>>(a, chunk);
  return cudaGetLastError();
}

cudaError_t launch_zero_if_empty(const CallArgs& a, cudaStream_t s) {
  k_zero_if_empty<<<(unsigned)(2 * num_sms()), 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_scale_by(void* x, int64_t n, int dtype, const float* g, cudaStream_t s) {
  const unsigned blocks = (unsigned)(4 * num_sms());
  switch (dtype) {
    case FLCE_F32: k_scale_by<float><<<blocks, 256, 0, s>>>((float*)x, n, g); break;
    case FLCE_BF16: k_scale_by<__nv_bfloat16><<<blocks, 256, 0, s>>>((__nv_bfloat16*)x, n, g); break;
    default: k_scale_by<__half><<<blocks, 256, 0, s>>>((__half*)x, n, g); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_scale_x(const CallArgs& a, int chunk, cudaStream_t s) {
  const int64_t blocks = cdiv64(a.R, 4) < 4LL * num_sms() ? cdiv64(a.R, 4) : 4LL * num_sms();
  k_scale_x<<<(unsigned)blocks, 256, 0, s>>>(a, chunk);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const CallArgs& a, int chunk, cudaStream_t s) {
  k_finalize<<<(unsigned)cdiv64(a.R, 8), 256, 0, s>>>(a, chunk);
  return cudaGetLastError();
}

cudaError_t launch_gpass(const CallArgs& a, int chunk, cudaStream_t s) {
  switch (a.dt) {
    case FLCE_BF16: return gpass_t<__nv_bfloat16>(a, chunk, s);
    case FLCE_F16: return gpass_t<__half>(a, chunk, s);
    default: return gpass_t<float>(a, chunk, s);
  }
}

cudaError_t launch_fwd_simt(const CallArgs& a, int chunk, cudaStream_t s) {
  dim3 grid((unsigned)cdiv64(a.R, 64), (unsigned)a.nvt);
  switch (a.dt) {
    case FLCE_BF16: k_fwd_simt<__nv_bfloat16><<<grid, 256, 0, s>>>(a, chunk); break;
    case FLCE_F16: k_fwd_simt<__half><<<grid, 256, 0, s>>>(a, chunk); break;
    default: k_fwd_simt<float><<<grid, 256, 0, s>>>(a, chunk); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_dx_simt(const CallArgs& a, int chunk, cudaStream_t s) {
  if (cdiv64(a.H, 128) * cdiv64(a.R, 128) < num_sms()) {  // few output tiles: 64 x 64
    dim3 grid((unsigned)cdiv64(a.H, 64), (unsigned)cdiv64(a.R, 64));
    switch (a.dt) {
      case FLCE_BF16: k_gemm_simt<__nv_bfloat16, 0, 4><<<grid, 256, 0, s>>>(a, chunk); break;
      case FLCE_F16: k_gemm_simt<__half, 0, 4><<<grid, 256, 0, s>>>(a, chunk); break;
      default: k_gemm_simt<float, 0, 4><<<grid, 256, 0, s>>>(a, chunk); break;
    }
    return cudaGetLastError();
  }
  dim3 grid((unsigned)cdiv64(a.H, 128), (unsigned)cdiv64(a.R, 128));
  switch (a.dt) {
    case FLCE_BF16: k_gemm_simt<__nv_bfloat16, 0, 8><<<grid, 256, 0, s>>>(a, chunk); break;
    case FLCE_F16: k_gemm_simt<__half, 0, 8><<<grid, 256, 0, s>>>(a, chunk); break;
    default: k_gemm_simt<float, 0, 8><<<grid, 256, 0, s>>>(a, chunk); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_dw_simt(const CallArgs& a, int chunk, cudaStream_t s) {
  dim3 grid((unsigned)cdiv64(a.H, 128), (unsigned)cdiv64(a.V, 128));
  switch (a.dt) {
    case FLCE_BF16: k_gemm_simt<__nv_bfloat16, 1, 8><<<grid, 256, 0, s>>>(a, chunk); break;
    case FLCE_F16: k_gemm_simt<__half, 1, 8><<<grid, 256, 0, s>>>(a, chunk); break;
    default: k_gemm_simt<float, 1, 8><<<grid, 256, 0, s>>>(a, chunk); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_dx_store(const CallArgs& a, int chunk, cudaStream_t s) {
  const int64_t blocks = a.R < 8LL * num_sms() ? a.R : 8LL * num_sms();
  if (a.dt == FLCE_BF16) k_dx_store<__nv_bfloat16><<<(unsigned)blocks, 256, 0, s>>>(a, chunk);
  else k_dx_store<__half><<<(unsigned)blocks, 256, 0, s>>>(a, chunk);
  return cudaGetLastError();
}

cudaError_t launch_epilogue(const CallArgs& a, cudaStream_t s) {
  if (a.reduction == FLCE_NONE) return cudaSuccess;
  k_reduce<<<RED_BLOCKS, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace flce
