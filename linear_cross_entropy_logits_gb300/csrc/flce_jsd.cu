// Fused linear JSD / KL distillation on the FLCE tile engine.
//
// The pages name this sibling op ("fused linear KL" on the Liger-Kernel v0.8.3 commit
// page; test_fused_linear_jsd.py in "Liger-Kernel PR #1554: skip ignore_index rows",
// Results) without defining it; the reading used (see include/flce.h) is the generalised
// Jensen-Shannon divergence between the teacher P = softmax(X_t W_t^T / T) and the student
// Q = softmax(X_s W_s^T / T), with beta = 0 giving KL(P||Q) and beta = 1 KL(Q||P).
//
// Per row chunk: gather student and teacher rows; the forward GEMM twice (student and
// teacher, logits scaled by 1/T in the epilogue, each writing per-tile statistics and its
// exp slab); k_jsd_finalize (both lse, per-tile log offsets); k_jsd_rows (per row: the
// divergence terms and sum_v Q g in a fixed order, then dloss/dz into the student slab in
// place, both passes over a row while it is still in L2); then the same dX / dW GEMMs as
// the cross-entropy op. The only [R, V] data in HBM are the two per-chunk exp slabs.
#include <math.h>
#include <string.h>

#include <atomic>

#include "flce_internal.cuh"

namespace flce {
namespace {

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t rup(int64_t a, int64_t b) { return cdiv(a, b) * b; }
inline size_t rup_sz(size_t a, size_t b) { return (a + b - 1) / b * b; }
__host__ __device__ inline int64_t rup64(int64_t a, int64_t b) { return (a + b - 1) / b * b; }

struct JsdPlan {
  int64_t BT, Hs, Ht, V, Hsp, Htp, nvt, Vp, R, kmax;
  int esz;
  size_t off_ctrl, off_idx, off_rloss, off_rz, off_racc;
  size_t off_xcs, off_xct, off_stm_s, off_sts_s, off_sti_s, off_stm_t, off_sts_t, off_sti_t;
  size_t off_tgt_s, off_tgt_t, off_lse_s, off_lse_t, off_arow;
  size_t off_slab_s, off_slab_t, off_dxacc;
  size_t total;
};

bool jsd_layout(int64_t BT, int64_t Hs, int64_t Ht, int64_t V, int dt, int64_t R, JsdPlan* p) {
  if (BT <= 0 || Hs <= 0 || Ht <= 0 || V <= 0 || R <= 0) return false;
  JsdPlan q;
  q.BT = BT;
  q.Hs = Hs;
  q.Ht = Ht;
  q.V = V;
  q.esz = dtype_size(dt);
  q.Hsp = rup(Hs, 64);
  q.Htp = rup(Ht, 64);
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
  const size_t st = 4 * (size_t)q.nvt * R;
  q.off_ctrl = take(sizeof(Ctrl));
  q.off_idx = take(4 * (size_t)BT);
  q.off_rloss = take(4 * (size_t)BT);
  q.off_rz = take(4 * (size_t)BT);
  q.off_racc = take(4 * (size_t)BT);
  q.off_xcs = take((size_t)R * q.Hsp * q.esz);
  q.off_xct = take((size_t)R * q.Htp * q.esz);
  q.off_stm_s = take(st);
  q.off_sts_s = take(st);
  q.off_sti_s = take(st);
  q.off_stm_t = take(st);
  q.off_sts_t = take(st);
  q.off_sti_t = take(st);
  q.off_tgt_s = take(4 * (size_t)R);
  q.off_tgt_t = take(4 * (size_t)R);
  q.off_lse_s = take(4 * (size_t)R);
  q.off_lse_t = take(4 * (size_t)R);
  q.off_arow = take(4 * (size_t)R);
  q.off_slab_s = take((size_t)R * q.Vp * q.esz);
  q.off_slab_t = take((size_t)R * q.Vp * q.esz);
  q.off_dxacc = take(q.esz == 2 ? 2 * (size_t)R * Hs * 4 : 0);  // two fp32 buffers
  q.total = off;
  *p = q;
  return true;
}

int64_t jsd_rows_for_bytes(int64_t BT, int64_t Hs, int64_t Ht, int64_t V, int dt, size_t bytes) {
  JsdPlan p, p2;
  if (!jsd_layout(BT, Hs, Ht, V, dt, CHUNK_ALIGN, &p) || p.total > bytes) return 0;
  jsd_layout(BT, Hs, Ht, V, dt, 2 * CHUNK_ALIGN, &p2);
  const size_t per128 = p2.total - p.total;
  int64_t R = CHUNK_ALIGN + (int64_t)((bytes - p.total) / (per128 ? per128 : 1)) * CHUNK_ALIGN;
  const int64_t cap = rup(BT, CHUNK_ALIGN);
  if (R > cap) R = cap;
  while (R > CHUNK_ALIGN) {
    if (jsd_layout(BT, Hs, Ht, V, dt, R, &p) && p.total <= bytes) break;
    R -= CHUNK_ALIGN;
  }
  return R;
}

// Everything the JSD kernels need: the student and teacher views of the engine, and the
// distillation parameters.
struct JsdArgs {
  CallArgs s, t;
  float beta, inv_T;
};

__device__ __forceinline__ void lse_merge(float& M, float& S, float M2, float S2) {
  const float Mn = fmaxf(M, M2);
  S = Mn == -INFINITY ? 0.0f : S * expf(M - Mn) + S2 * expf(M2 - Mn);
  M = Mn;
}

// Row lse of the student and the teacher from their per-tile (max, sum-exp) statistics, in
// a fixed order; each tile max is then rewritten as the tile's log offset m - lse, so that
// log Q = log e + offset and Q = e * exp(offset) for the stored e = exp(z - m).
__global__ void __launch_bounds__(256) k_jsd_finalize(const __grid_constant__ JsdArgs j, int chunk) {
  int row0, rows;
  if (!chunk_bounds(j.s.w.ctrl, chunk, row0, rows)) return;
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (r >= rows) return;  // warp-uniform
  const int nvt = (int)j.s.nvt;
  float lse2[2];
#pragma unroll
  for (int side = 0; side < 2; ++side) {
    const Work& w = side == 0 ? j.s.w : j.t.w;
    float* stm = w.stm + (int64_t)r * nvt;
    const float* sts = w.sts + (int64_t)r * nvt;
    float M = -INFINITY, S = 0.0f;
    for (int t = lane; t < nvt; t += 32) lse_merge(M, S, stm[t], sts[t]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float M2 = __shfl_xor_sync(0xffffffffu, M, o);
      const float S2 = __shfl_xor_sync(0xffffffffu, S, o);
      lse_merge(M, S, M2, S2);
    }
    const float lse = M + logf(S);
    for (int t = lane; t < nvt; t += 32) stm[t] -= lse;
    lse2[side] = lse;
  }
  if (lane == 0) {
    const int row = j.s.w.idx[row0 + r];
    j.s.w.lse[r] = lse2[0];
    j.t.w.lse[r] = lse2[1];
    float ar = 1.0f;
    if (j.s.reduction == FLCE_NONE && j.s.grad_out != nullptr) ar = j.s.grad_out[row];
    j.s.w.arow[r] = ar;
  }
}

// Logs in base 2, from the hardware approximation (lg2.approx.ftz: absolute error about
// 2^-22 near 1, relative error a few ulp elsewhere), far below the 2^-9 relative rounding
// of the stored e. Arguments are clamped to a normal float so that 0 * log(0) terms vanish
// (e underflows to 0 in the 16-bit slab for very unlikely tokens). Working in base 2 and
// scaling the per-tile sums by ln 2 once keeps these passes to three special-function
// operations per element.
__device__ __forceinline__ float lg2_clamped(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(fmaxf(x, 1e-37f)));
  return y;
}
constexpr float LN2 = 0.6931471805599453f;

// Eight consecutive slab elements: a raw 16-byte (32-byte for fp32) vector load, kept packed
// in registers until it is converted, and the matching converting store.
template <typename T> struct Load8;
template <> struct Load8<__nv_bfloat16> {
  struct Raw { uint4 u; };
  __device__ static Raw load(const __nv_bfloat16* p) { return Raw{*(const uint4*)p}; }
  __device__ static void cvt(const Raw& r, float (&f)[8]) {
    const __nv_bfloat162* h = (const __nv_bfloat162*)&r.u;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 x = __bfloat1622float2(h[k]);
      f[2 * k] = x.x;
      f[2 * k + 1] = x.y;
    }
  }
  __device__ static void store(__nv_bfloat16* p, const float (&f)[8]) {
    uint4 u;
    __nv_bfloat162* h = (__nv_bfloat162*)&u;
#pragma unroll
    for (int k = 0; k < 4; ++k) h[k] = __floats2bfloat162_rn(f[2 * k], f[2 * k + 1]);
    *(uint4*)p = u;
  }
};
template <> struct Load8<__half> {
  struct Raw { uint4 u; };
  __device__ static Raw load(const __half* p) { return Raw{*(const uint4*)p}; }
  __device__ static void cvt(const Raw& r, float (&f)[8]) {
    const __half2* h = (const __half2*)&r.u;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 x = __half22float2(h[k]);
      f[2 * k] = x.x;
      f[2 * k + 1] = x.y;
    }
  }
  __device__ static void store(__half* p, const float (&f)[8]) {
    uint4 u;
    __half2* h = (__half2*)&u;
#pragma unroll
    for (int k = 0; k < 4; ++k) h[k] = __floats2half2_rn(f[2 * k], f[2 * k + 1]);
    *(uint4*)p = u;
  }
};
template <> struct Load8<float> {
  struct Raw { float4 a, b; };
  __device__ static Raw load(const float* p) { return Raw{*(const float4*)p, *(const float4*)(p + 4)}; }
  __device__ static void cvt(const Raw& r, float (&f)[8]) {
    f[0] = r.a.x; f[1] = r.a.y; f[2] = r.a.z; f[3] = r.a.w;
    f[4] = r.b.x; f[5] = r.b.y; f[6] = r.b.z; f[7] = r.b.w;
  }
  __device__ static void store(float* p, const float (&f)[8]) {
    *(float4*)p = make_float4(f[0], f[1], f[2], f[3]);
    *(float4*)(p + 4) = make_float4(f[4], f[5], f[6], f[7]);
  }
};

// Eight slab columns per lane; a warp covers one 256-column tile, and each warp keeps
// RU tiles' loads in flight so that enough bytes are outstanding to cover DRAM latency.
// 24 warps x 2 tiles (768 threads, 80 registers) ran faster than 16 x 4, 32 x 1 or 8 x 8:
// the kernel needs both the bytes in flight and the warps to hide its arithmetic.
#ifndef FLCE_JR_RU
#define FLCE_JR_RU 2
#endif
constexpr int RU = FLCE_JR_RU;

// Both elementwise passes in one kernel, one row at a time per CTA (persistent, one CTA
// per SM): pass 1 reads the row of both slabs and sums the divergence terms and Q g (g =
// dloss/dQ up to a constant) with a fixed-order block reduction, giving loss_i and
// S_i = sum_v Q_v g_v; pass 2 reads the row again, while it is still in L2 (one row per SM
// in flight, about 0.5 MB each at V = 128256), and writes dS over the student slab; over
// the first JR_XTILES tiles it reads only the student row and the log ratio pass 1 kept in
// shared memory (no log in pass 2 there). DRAM moves each slab row once plus the dS write. The slab's pad columns (v >= V) hold exact
// zeros, whose terms vanish and whose dS is zero, so no column test is needed.
#ifndef FLCE_JR_THREADS
#define FLCE_JR_THREADS 768
#endif
constexpr int JR_THREADS = FLCE_JR_THREADS;
static_assert(JR_THREADS % 32 == 0 && JR_THREADS >= 64 && JR_THREADS <= 1024, "whole warps, one CTA");
static_assert(RU >= 1, "at least one tile in flight per warp");
constexpr int JR_WARPS = JR_THREADS / 32;
// Pass 1 also keeps the log ratio x = log2(Q / R) of the row's first JR_XTILES tiles in
// shared memory (fp16, 200 KB), R = M (0 < beta < 1) or P (beta = 1); pass 2 then forms
// dS there from Q and x alone, without the teacher row and without a log. x <= log2(1 /
// (1 - beta)) for 0 < beta < 1, and |x| < 256 for beta = 1 (both logs are clamped), so
// fp16 keeps it to 2^-11 relative, below the 2^-9 rounding of the stored e.
constexpr int JR_XTILES = 400;

// 8 values <-> one 16-byte shared-memory word of fp16. The conversion saturates at the
// largest finite fp16 (|x| past 65504 needs logit gaps beyond ~45000 after the temperature;
// there Q underflows to 0, and a finite x keeps Q * x at 0 instead of NaN).
__device__ __forceinline__ void xs_store(uint32_t addr, const float (&x)[8]) {
  uint32_t h[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)  // upper half <- the odd column, lower half <- the even one
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(h[k]) : "f"(x[2 * k + 1]), "f"(x[2 * k]));
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(h[0]), "r"(h[1]), "r"(h[2]), "r"(h[3])
               : "memory");
}
__device__ __forceinline__ void xs_load(uint32_t addr, float (&x)[8]) {
  uint32_t h[4];
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3]) : "r"(addr)
               : "memory");
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 v = __half22float2(*(__half2*)&h[k]);
    x[2 * k] = v.x;
    x[2 * k + 1] = v.y;
  }
}

template <typename T>
__global__ void __launch_bounds__(JR_THREADS, 1) k_jsd_rows(const __grid_constant__ JsdArgs j, int chunk,
                                                           int grads, int xt) {
  int row0, rows;
  if (!chunk_bounds(j.s.w.ctrl, chunk, row0, rows)) return;
  __shared__ float red_t[JR_WARPS], red_g[JR_WARPS];
  __shared__ float row_S;
  extern __shared__ __align__(16) uint8_t xs_raw[];  // xt tiles x 256 fp16 values
  const uint32_t xs0 = (uint32_t)__cvta_generic_to_shared(xs_raw);
  const int lane = threadIdx.x & 31, wp = threadIdx.x >> 5;
  const int rlim = grads ? (int)rup64(rows, 64) : rows;
  const int nvt = (int)j.s.nvt;
  const float beta = j.beta, omb = 1.0f - beta;
  const float cg = (beta == 1.0f ? 1.0f : omb) * LN2;
  constexpr int RUJ = sizeof(T) == 4 ? (RU > 1 ? RU / 2 : 1) : RU;  // tiles in flight per warp (fp32 rows are twice the bytes)
  for (int r = blockIdx.x; r < rlim; r += gridDim.x) {
    const bool live = r < rows;
    const T* s_row = (const T*)j.s.w.slab + (int64_t)r * j.s.Vp;
    const T* t_row = (const T*)j.t.w.slab + (int64_t)r * j.t.Vp;
    const float* soff = j.s.w.stm + (int64_t)r * nvt;
    const float* toff = j.t.w.stm + (int64_t)r * nvt;
    float S = 0.0f;
    if (live) {
      // ---- pass 1: warp wp takes tiles wp, wp + JR_WARPS, ... RUJ at a time
      float tm = 0.0f, g = 0.0f;
      for (int t0 = wp; t0 < nvt; t0 += JR_WARPS * RUJ) {
        typename Load8<T>::Raw rs[RUJ], rt[RUJ];
        float lqo[RUJ], lpo[RUJ];
#pragma unroll
        for (int u = 0; u < RUJ; ++u) {
          const int t = t0 + u * JR_WARPS < nvt ? t0 + u * JR_WARPS : t0;  // re-read t0 past the end
          lqo[u] = soff[t];
          lpo[u] = toff[t];
          rs[u] = Load8<T>::load(s_row + (int64_t)t * VT + lane * 8);
          rt[u] = Load8<T>::load(t_row + (int64_t)t * VT + lane * 8);
        }
#pragma unroll
        for (int u = 0; u < RUJ; ++u) {
          if (t0 + u * JR_WARPS >= nvt) continue;
          float es[8], et[8];
          Load8<T>::cvt(rs[u], es);
          Load8<T>::cvt(rt[u], et);
          const float qm = expf(lqo[u]), pm = expf(lpo[u]);
          const float lq2 = lqo[u] * LOG2E, lp2 = lpo[u] * LOG2E;
          // 0 < beta < 1: (1 - beta) Q and beta P straight from the stored e
          const float qmo = omb * qm, pmb = beta * pm;
          float xr[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float lQ = lg2_clamped(es[k]) + lq2, lP = lg2_clamped(et[k]) + lp2;
            if (beta == 0.0f) {
              tm = fmaf(et[k] * pm, lP - lQ, tm);
            } else if (beta == 1.0f) {
              xr[k] = lQ - lP;
              const float x = (es[k] * qm) * xr[k];
              tm += x;
              g += x;
            } else {
              const float Qo = es[k] * qmo, Pb = et[k] * pmb;
              const float lM = lg2_clamped(Qo + Pb);
              xr[k] = lQ - lM;
              g = fmaf(Qo, xr[k], g);       // (1 - beta) Q log(Q / M)
              tm = fmaf(Pb, lP - lM, tm);   // beta P log(P / M); the Q part is added below
            }
          }
          const int t = t0 + u * JR_WARPS;
          if (t < xt) xs_store(xs0 + (uint32_t)(t * VT + lane * 8) * 2u, xr);
        }
      }
      if (beta != 0.0f && beta != 1.0f) tm += g;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        tm += __shfl_xor_sync(0xffffffffu, tm, o);
        g += __shfl_xor_sync(0xffffffffu, g, o);
      }
      if (lane == 0) {
        red_t[wp] = tm;
        red_g[wp] = g;
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        float L = 0.0f, G = 0.0f;
        for (int w = 0; w < JR_WARPS; ++w) {  // fixed order
          L += red_t[w];
          G += red_g[w];
        }
        L *= LN2;
        G *= LN2;
        row_S = G;
        const int row = j.s.w.idx[row0 + r];
        j.s.w.rloss[row0 + r] = L;
        j.s.w.rz[row0 + r] = 0.0f;
        j.s.w.racc[row0 + r] = 0.0f;
        if (j.s.reduction == FLCE_NONE) j.s.loss[row] = L;
      }
      __syncthreads();
      S = row_S;
    }
    if (grads) {
      // ---- pass 2: dS = a_i / T * dloss_i/dz_s over the student row, with dloss/dz_s =
      // Q ((1 - beta) ln2 (lQ2 - lM2) - S) in base-2 logs (M = P when beta = 1, and Q - P when
      // beta = 0); rows past the chunk up to the next multiple of 64 are written as zeros
      // (the dW GEMM reduces over them)
      T* d_row = (T*)j.s.w.slab + (int64_t)r * j.s.Vp;
      const float f = live ? j.s.w.arow[r] * j.inv_T : 0.0f;
      for (int t0 = wp; t0 < nvt; t0 += JR_WARPS * RUJ) {
        typename Load8<T>::Raw rs[RUJ], rt[RUJ];
        float lqo[RUJ], lpo[RUJ];
        if (live) {
#pragma unroll
          for (int u = 0; u < RUJ; ++u) {
            const int t = t0 + u * JR_WARPS < nvt ? t0 + u * JR_WARPS : t0;
            lqo[u] = soff[t];
            rs[u] = Load8<T>::load(s_row + (int64_t)t * VT + lane * 8);
            if (t >= xt) {
              lpo[u] = toff[t];
              rt[u] = Load8<T>::load(t_row + (int64_t)t * VT + lane * 8);
            }
          }
        }
#pragma unroll
        for (int u = 0; u < RUJ; ++u) {
          const int t = t0 + u * JR_WARPS;
          if (t >= nvt) continue;
          float out[8];
          if (live && t < xt) {
            float es[8], xr[8];
            Load8<T>::cvt(rs[u], es);
            xs_load(xs0 + (uint32_t)(t * VT + lane * 8) * 2u, xr);
            const float qm = expf(lqo[u]);
#pragma unroll
            for (int k = 0; k < 8; ++k) out[k] = f * ((es[k] * qm) * fmaf(cg, xr[k], -S));
          } else if (live) {
            float es[8], et[8];
            Load8<T>::cvt(rs[u], es);
            Load8<T>::cvt(rt[u], et);
            const float qm = expf(lqo[u]), pm = expf(lpo[u]);
            const float lq2 = lqo[u] * LOG2E, lp2 = lpo[u] * LOG2E;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const float Q = es[k] * qm, P = et[k] * pm;
              float dz;
              if (beta == 0.0f) {
                dz = Q - P;
              } else {
                const float lQ = lg2_clamped(es[k]) + lq2;
                const float lR = beta == 1.0f ? lg2_clamped(et[k]) + lp2
                                              : lg2_clamped(es[k] * (omb * qm) + et[k] * (beta * pm));
                dz = Q * fmaf(cg, lQ - lR, -S);
              }
              out[k] = f * dz;
            }
          } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) out[k] = 0.0f;
          }
          Load8<T>::store(d_row + (int64_t)t * VT + lane * 8, out);
        }
      }
    }
    __syncthreads();  // red_t / red_g / row_S are reused by the next row
  }
}

template <typename T>
cudaError_t launch_jsd_rows(const JsdArgs& j, int chunk, cudaStream_t s, bool grads) {
  int g = num_sms();
  if (g > j.s.R) g = (int)j.s.R;
  // x is kept for 16-bit slabs with gradients and beta > 0 (beta = 0 needs P, not a log)
  int xt = 0;
  if (grads && sizeof(T) == 2 && j.beta > 0.0f) xt = j.s.nvt < JR_XTILES ? (int)j.s.nvt : JR_XTILES;
  const size_t smem = (size_t)xt * VT * 2;
  // the shared-memory limit (the largest any launch asks for) is set on a device's first
  // launch and persists, so later launches, including ones captured into a CUDA graph,
  // enqueue the kernel only; concurrent first launches may both set it
  static std::atomic<int> attr_set[64];
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (smem > 0 && (dev < 0 || dev >= 64 || attr_set[dev].load(std::memory_order_relaxed) == 0)) {
    e = cudaFuncSetAttribute(k_jsd_rows<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)((size_t)JR_XTILES * VT * 2));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev].store(1, std::memory_order_relaxed);
  }
  k_jsd_rows<T><<<(unsigned)g, JR_THREADS, smem, s>>>(j, chunk, grads ? 1 : 0, xt);
  return cudaGetLastError();
}

cudaError_t jsd_rows(const JsdArgs& j, int chunk, cudaStream_t s, bool grads) {
  switch (j.s.dt) {
    case FLCE_BF16: return launch_jsd_rows<__nv_bfloat16>(j, chunk, s, grads);
    case FLCE_F16: return launch_jsd_rows<__half>(j, chunk, s, grads);
    default: return launch_jsd_rows<float>(j, chunk, s, grads);
  }
}


inline bool aligned(const void* p, size_t n) { return ((uintptr_t)p % n) == 0; }

int32_t jsd_validate(const flce_jsd_args* x) {
  if (!x) return FLCE_ERR_INVALID_ARG;
  if (x->BT <= 0 || x->Hs <= 0 || x->Ht <= 0 || x->V <= 0) return FLCE_ERR_INVALID_ARG;
  if (x->BT > 0x7fffffffLL || x->Hs > 0x7fffffffLL || x->Ht > 0x7fffffffLL || x->V > 0x7fffffffLL)
    return FLCE_ERR_INVALID_ARG;
  if (x->in_dtype != FLCE_F32 && x->in_dtype != FLCE_BF16 && x->in_dtype != FLCE_F16)
    return FLCE_ERR_INVALID_ARG;
  if (x->reduction != FLCE_MEAN && x->reduction != FLCE_SUM && x->reduction != FLCE_NONE)
    return FLCE_ERR_INVALID_ARG;
  if (!x->Xs || !x->Ws || !x->Xt || !x->Wt || !x->loss || !x->workspace) return FLCE_ERR_INVALID_ARG;
  if (!(x->beta >= 0.0f && x->beta <= 1.0f)) return FLCE_ERR_INVALID_ARG;
  if (!(x->temperature > 0.0f) || x->temperature > 1e30f) return FLCE_ERR_INVALID_ARG;
  if (x->want_dX && !x->dX) return FLCE_ERR_INVALID_ARG;
  if (x->want_dW && !x->dW) return FLCE_ERR_INVALID_ARG;
  if (x->want_dW && x->dW_dtype != FLCE_F32 && x->dW_dtype != x->in_dtype) return FLCE_ERR_UNSUPPORTED;
  if (!aligned(x->Xs, 16) || !aligned(x->Ws, 16) || !aligned(x->Xt, 16) || !aligned(x->Wt, 16) ||
      !aligned(x->workspace, 256))
    return FLCE_ERR_INVALID_ARG;
  if (x->want_dX && !aligned(x->dX, 16)) return FLCE_ERR_INVALID_ARG;
  if (x->want_dW && !aligned(x->dW, 16)) return FLCE_ERR_INVALID_ARG;
  if (x->labels && !aligned(x->labels, 8)) return FLCE_ERR_INVALID_ARG;
  if (!aligned(x->loss, 4) || (x->status && !aligned(x->status, 4))) return FLCE_ERR_INVALID_ARG;
  return FLCE_OK;
}

}  // namespace
}  // namespace flce

using namespace flce;

extern "C" size_t flce_jsd_workspace_size(int64_t BT, int64_t Hs, int64_t Ht, int64_t V, int32_t in_dtype,
                                          size_t budget_bytes) {
  if (BT <= 0 || Hs <= 0 || Ht <= 0 || V <= 0) return 0;
  if (in_dtype != FLCE_F32 && in_dtype != FLCE_BF16 && in_dtype != FLCE_F16) return 0;
  const int64_t R = jsd_rows_for_bytes(BT, Hs, Ht, V, in_dtype, budget_bytes ? budget_bytes : 2 * DEFAULT_BUDGET);
  if (R <= 0) return 0;
  JsdPlan p;
  if (!jsd_layout(BT, Hs, Ht, V, in_dtype, R, &p)) return 0;
  return p.total;
}

extern "C" int32_t flce_fused_linear_jsd(const flce_jsd_args* x, void* stream) {
  const int32_t v = jsd_validate(x);
  if (v != FLCE_OK) return v;
  const int64_t R = jsd_rows_for_bytes(x->BT, x->Hs, x->Ht, x->V, x->in_dtype, x->workspace_bytes);
  if (R <= 0) return FLCE_ERR_WORKSPACE;
  JsdPlan p;
  if (!jsd_layout(x->BT, x->Hs, x->Ht, x->V, x->in_dtype, R, &p)) return FLCE_ERR_INVALID_ARG;
  char* b = (char*)x->workspace;

  CallArgs s;
  memset(&s, 0, sizeof(s));
  s.BT = x->BT;
  s.V = x->V;
  s.Vp = p.Vp;
  s.nvt = p.nvt;
  s.R = p.R;
  s.dt = x->in_dtype;
  s.reduction = x->reduction;
  s.ignore_index = x->ignore_index;
  s.grad_out = x->grad_out;
  s.loss = x->loss;
  s.n_labelled = x->n_labelled;
  s.want_dX = x->want_dX ? 1 : 0;
  s.want_dW = x->want_dW ? 1 : 0;
  s.dW_dt = x->dW_dtype;
  s.timeout_ns = (uint64_t)(x->wait_timeout_ms ? x->wait_timeout_ms : DEFAULT_TIMEOUT_MS) * 1000000ull;
  s.flags = x->flags;
  s.logit_scale = 1.0f / x->temperature;
  s.labels_are_masks = 1;
  // shared workspace regions
  s.w.ctrl = (Ctrl*)(b + p.off_ctrl);
  s.w.idx = (int*)(b + p.off_idx);
  s.w.rloss = (float*)(b + p.off_rloss);
  s.w.rz = (float*)(b + p.off_rz);
  s.w.racc = (float*)(b + p.off_racc);
  s.w.arow = (float*)(b + p.off_arow);
  s.w.status = x->status ? (int*)x->status : &s.w.ctrl->status;
  CallArgs t = s;
  // student view
  s.H = x->Hs;
  s.Hp = p.Hsp;
  s.X = x->Xs;
  s.W = x->Ws;
  s.dX = s.want_dX ? x->dX : nullptr;
  s.dW = s.want_dW ? x->dW : nullptr;
  s.w.xc = b + p.off_xcs;
  s.w.stm = (float*)(b + p.off_stm_s);
  s.w.sts = (float*)(b + p.off_sts_s);
  s.w.sti = (int*)(b + p.off_sti_s);
  s.w.tgt = (float*)(b + p.off_tgt_s);
  s.w.lse = (float*)(b + p.off_lse_s);
  s.w.slab = b + p.off_slab_s;
  s.w.dxacc = (float*)(b + p.off_dxacc);
  // teacher view (forward only)
  t.H = x->Ht;
  t.Hp = p.Htp;
  t.X = x->Xt;
  t.W = x->Wt;
  t.want_dX = t.want_dW = 0;
  t.w.xc = b + p.off_xct;
  t.w.stm = (float*)(b + p.off_stm_t);
  t.w.sts = (float*)(b + p.off_sts_t);
  t.w.sti = (int*)(b + p.off_sti_t);
  t.w.tgt = (float*)(b + p.off_tgt_t);
  t.w.lse = (float*)(b + p.off_lse_t);
  t.w.slab = b + p.off_slab_t;
  t.w.dxacc = nullptr;
  // compaction reads the labels; the forward GEMMs gather no target logit
  CallArgs comp = s;
  comp.targets = x->labels;
  s.targets = nullptr;
  t.targets = nullptr;

  JsdArgs j;
  j.s = s;
  j.t = t;
  j.beta = x->beta;
  j.inv_T = 1.0f / x->temperature;

  cudaStream_t st = (cudaStream_t)stream;
  const bool tc = !(x->flags & FLCE_FLAG_FORCE_SIMT) && tc_supported(s) && tc_supported(t);
  const bool grads = s.want_dX || s.want_dW;
#define JSD_TRY(expr)                     \
  do {                                    \
    if ((expr) != cudaSuccess) return FLCE_ERR_CUDA; \
  } while (0)
  flce_profile* prof = x->profile;
  JSD_TRY(cudaMemsetAsync(s.w.status, 0, sizeof(int), st));
  JSD_TRY(staged(prof, FLCE_STAGE_PROLOGUE, 2, st, [&] { return launch_prologue(comp, st); }));
  for (int k = 0; k < (int)p.kmax; ++k) {
    JSD_TRY(staged(prof, FLCE_STAGE_GATHER, 2, st, [&] {
      cudaError_t e = launch_gather(s, k, st);
      return e != cudaSuccess ? e : launch_gather(t, k, st);
    }));
    JSD_TRY(staged(prof, FLCE_STAGE_FWD, 2, st, [&] {
      cudaError_t e = tc ? launch_fwd_tc(s, k, st) : launch_fwd_simt(s, k, st);
      return e != cudaSuccess ? e : (tc ? launch_fwd_tc(t, k, st) : launch_fwd_simt(t, k, st));
    }));
    JSD_TRY(staged(prof, FLCE_STAGE_FINALIZE, 1, st, [&] {
      k_jsd_finalize<<<(unsigned)cdiv(p.R, 8), 256, 0, st>>>(j, k);
      return cudaGetLastError();
    }));
    JSD_TRY(staged(prof, FLCE_STAGE_GPASS, 1, st, [&] { return jsd_rows(j, k, st, grads); }));
    if (tc && bwd_merged_supported(s)) {
      // the student's dX and dW in one launch (shared work queue), then the dX sum
      JSD_TRY(staged(prof, FLCE_STAGE_BWD, 2, st, [&] {
        cudaError_t e = cudaMemsetAsync(s.w.dxacc, 0, 2 * (size_t)p.R * s.H * 4, st);
        if (e == cudaSuccess) e = launch_bwd_tc(s, k, st);
        return e != cudaSuccess ? e : launch_dx_store(s, k, st);
      }));
      continue;
    }
    if (s.want_dX) {
      if (tc) {
        JSD_TRY(staged(prof, FLCE_STAGE_DX, 2, st, [&] {
          cudaError_t e = cudaMemsetAsync(s.w.dxacc, 0, 2 * (size_t)p.R * s.H * 4, st);
          if (e == cudaSuccess) e = launch_dx_tc(s, k, st);
          return e != cudaSuccess ? e : launch_dx_store(s, k, st);
        }));
      } else {
        JSD_TRY(staged(prof, FLCE_STAGE_DX, 1, st, [&] { return launch_dx_simt(s, k, st); }));
      }
    }
    if (s.want_dW)
      JSD_TRY(staged(prof, FLCE_STAGE_DW, 1, st,
                     [&] { return tc ? launch_dw_tc(s, k, st) : launch_dw_simt(s, k, st); }));
  }
  if (s.reduction != FLCE_NONE)
    JSD_TRY(staged(prof, FLCE_STAGE_REDUCE, 1, st, [&] { return launch_epilogue(s, st); }));
  if (s.want_dW && (x->flags & FLCE_FLAG_DW_OVERWRITE))
    JSD_TRY(staged(prof, FLCE_STAGE_REDUCE, 1, st, [&] { return launch_zero_if_empty(s, st); }));
#undef JSD_TRY
  return FLCE_OK;
}
