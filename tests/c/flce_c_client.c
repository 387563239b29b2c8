/*
 * A plain C client of libflce.so: no PyTorch, no C++. It reads a problem from a binary
 * file (written by the test that builds and runs it), copies it to the GPU with the CUDA
 * runtime, calls flce_workspace_size / flce_fwd_bwd / flce_get_status through the C ABI,
 * and writes loss, lse, pred, dX and dW back to a binary file.
 *
 * Input file layout (little-endian): int64 BT, H, V; float z; int64 reduction; then
 * X [BT*H] and W [V*H] as raw bf16 (uint16), targets [BT] int64.
 * Output file: int32 status, float loss, float lse[BT], int64 pred[BT], uint16 dX[BT*H]
 * (bf16), float dW[V*H].
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "flce.h"

#define CHECK(x)                                                      \
  do {                                                                \
    cudaError_t e_ = (x);                                             \
    if (e_ != cudaSuccess) {                                          \
      fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));        \
      return 2;                                                       \
    }                                                                 \
  } while (0)

static int read_all(FILE* f, void* p, size_t n) { return fread(p, 1, n, f) == n ? 0 : 1; }

int main(int argc, char** argv) {
  if (argc != 3) {
    fprintf(stderr, "usage: %s in.bin out.bin\n", argv[0]);
    return 1;
  }
  FILE* f = fopen(argv[1], "rb");
  if (!f) return 1;
  int64_t BT, H, V, red;
  float z;
  if (read_all(f, &BT, 8) || read_all(f, &H, 8) || read_all(f, &V, 8) || read_all(f, &z, 4) ||
      read_all(f, &red, 8))
    return 1;
  const size_t nx = (size_t)(BT * H), nw = (size_t)(V * H);
  uint16_t* hX = malloc(nx * 2);
  uint16_t* hW = malloc(nw * 2);
  int64_t* ht = malloc((size_t)BT * 8);
  if (read_all(f, hX, nx * 2) || read_all(f, hW, nw * 2) || read_all(f, ht, (size_t)BT * 8)) return 1;
  fclose(f);

  void *dXin, *dWin, *dT, *dWs, *ddX, *dWgrad;
  float *dloss, *dlse;
  int64_t* dpred;
  int32_t *dstat, *dnl;
  CHECK(cudaMalloc(&dXin, nx * 2));
  CHECK(cudaMalloc(&dWin, nw * 2));
  CHECK(cudaMalloc(&dT, (size_t)BT * 8));
  CHECK(cudaMalloc(&ddX, nx * 2));
  CHECK(cudaMalloc(&dWgrad, nw * 4));
  CHECK(cudaMalloc((void**)&dloss, (red == FLCE_NONE ? (size_t)BT : 1) * 4));
  CHECK(cudaMalloc((void**)&dlse, (size_t)BT * 4));
  CHECK(cudaMalloc((void**)&dpred, (size_t)BT * 8));
  CHECK(cudaMalloc((void**)&dstat, 4));
  CHECK(cudaMalloc((void**)&dnl, 4));
  CHECK(cudaMemcpy(dXin, hX, nx * 2, cudaMemcpyHostToDevice));
  CHECK(cudaMemcpy(dWin, hW, nw * 2, cudaMemcpyHostToDevice));
  CHECK(cudaMemcpy(dT, ht, (size_t)BT * 8, cudaMemcpyHostToDevice));
  CHECK(cudaMemset(dWgrad, 0, nw * 4));

  const size_t wsb = flce_workspace_size(BT, H, V, FLCE_BF16, 0);
  if (wsb == 0) return 3;
  CHECK(cudaMalloc(&dWs, wsb));
  cudaStream_t s;
  CHECK(cudaStreamCreate(&s));

  flce_args a;
  memset(&a, 0, sizeof(a));
  a.BT = BT;
  a.H = H;
  a.V = V;
  a.in_dtype = FLCE_BF16;
  a.reduction = (int32_t)red;
  a.X = dXin;
  a.W = dWin;
  a.targets = (const int64_t*)dT;
  a.ignore_index = -100;
  a.z_loss_scale = z;
  a.want_dX = 1;
  a.want_dW = 1;
  a.dW_dtype = FLCE_F32;
  a.loss = dloss;
  a.lse = dlse;
  a.pred = dpred;
  a.n_labelled = dnl;
  a.dX = ddX;
  a.dW = dWgrad;
  a.workspace = dWs;
  a.workspace_bytes = wsb;
  a.status = dstat;
  int32_t rc = flce_fwd_bwd(&a, s);
  if (rc != FLCE_OK) {
    fprintf(stderr, "flce_fwd_bwd: %s (%s)\n", flce_status_string(rc), flce_last_cuda_error());
    return 4;
  }
  const int32_t st = flce_get_status(dstat, NULL, s);

  float loss0;
  float* hlse = malloc((size_t)BT * 4);
  int64_t* hpred = malloc((size_t)BT * 8);
  uint16_t* hdX = malloc(nx * 2);
  float* hdW = malloc(nw * 4);
  CHECK(cudaMemcpy(&loss0, dloss, 4, cudaMemcpyDeviceToHost));
  CHECK(cudaMemcpy(hlse, dlse, (size_t)BT * 4, cudaMemcpyDeviceToHost));
  CHECK(cudaMemcpy(hpred, dpred, (size_t)BT * 8, cudaMemcpyDeviceToHost));
  CHECK(cudaMemcpy(hdX, ddX, nx * 2, cudaMemcpyDeviceToHost));
  CHECK(cudaMemcpy(hdW, dWgrad, nw * 4, cudaMemcpyDeviceToHost));

  FILE* o = fopen(argv[2], "wb");
  if (!o) return 1;
  fwrite(&st, 4, 1, o);
  fwrite(&loss0, 4, 1, o);
  fwrite(hlse, 4, (size_t)BT, o);
  fwrite(hpred, 8, (size_t)BT, o);
  fwrite(hdX, 2, nx, o);
  fwrite(hdW, 4, nw, o);
  fclose(o);
  cudaStreamDestroy(s);
  printf("ok status=%d loss=%.6f ws=%zu\n", st, loss0, wsb);
  return 0;
}
