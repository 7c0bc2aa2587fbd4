/*
 * A plain C caller of the library (no Python, no torch): reads a problem from
 * a binary file, runs kd_topk_kl_fused_step on device buffers it allocates
 * itself, and writes the results to another binary file.
 *
 *   c_abi_client in.bin out.bin
 *
 * in.bin : int64 T; int32 d, V, K, chunk; then H [T,d] and W [V,d] as bf16
 *          bits (uint16), idx [T,K] int32, p [T,K] float32.
 * out.bin: float32 loss; lse [T]; dH [T,d]; dW [V,d].
 * Exit status 0 on success; any failing call is reported on stderr.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime.h>

#include "kdtopk.h"

#define CUDA_OK(call)                                                             \
  do {                                                                            \
    cudaError_t e_ = (call);                                                      \
    if (e_ != cudaSuccess) {                                                      \
      fprintf(stderr, "%s failed: %s\n", #call, cudaGetErrorString(e_));          \
      return 2;                                                                   \
    }                                                                             \
  } while (0)

static int read_all(FILE* f, void* dst, size_t bytes) { return fread(dst, 1, bytes, f) == bytes ? 0 : 1; }
static int write_all(FILE* f, const void* src, size_t bytes) { return fwrite(src, 1, bytes, f) == bytes ? 0 : 1; }

int main(int argc, char** argv) {
  if (argc != 3) {
    fprintf(stderr, "usage: %s in.bin out.bin\n", argv[0]);
    return 1;
  }
  FILE* in = fopen(argv[1], "rb");
  if (!in) {
    perror("open input");
    return 1;
  }
  int64_t T = 0;
  int32_t dims[4];
  if (read_all(in, &T, sizeof T) || read_all(in, dims, sizeof dims)) return 1;
  const int d = dims[0], V = dims[1], K = dims[2], chunk = dims[3];
  const size_t nH = (size_t)T * d, nW = (size_t)V * d, nC = (size_t)T * K;
  uint16_t* H = malloc(nH * 2);
  uint16_t* W = malloc(nW * 2);
  int32_t* idx = malloc(nC * 4);
  float* p = malloc(nC * 4);
  float* lse = malloc((size_t)T * 4);
  float* dH = malloc(nH * 4);
  float* dW = malloc(nW * 4);
  if (!H || !W || !idx || !p || !lse || !dH || !dW) return 1;
  if (read_all(in, H, nH * 2) || read_all(in, W, nW * 2) || read_all(in, idx, nC * 4) || read_all(in, p, nC * 4))
    return 1;
  fclose(in);

  void *dH_in, *dW_in, *dIdx, *dP, *dLoss, *dLse, *ddH, *ddW, *ws;
  CUDA_OK(cudaMalloc(&dH_in, nH * 2));
  CUDA_OK(cudaMalloc(&dW_in, nW * 2));
  CUDA_OK(cudaMalloc(&dIdx, nC * 4));
  CUDA_OK(cudaMalloc(&dP, nC * 4));
  CUDA_OK(cudaMalloc(&dLoss, 4));
  CUDA_OK(cudaMalloc(&dLse, (size_t)T * 4));
  CUDA_OK(cudaMalloc(&ddH, nH * 4));
  CUDA_OK(cudaMalloc(&ddW, nW * 4));
  CUDA_OK(cudaMemcpy(dH_in, H, nH * 2, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(dW_in, W, nW * 2, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(dIdx, idx, nC * 4, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(dP, p, nC * 4, cudaMemcpyHostToDevice));

  const size_t ws_bytes = kd_topk_kl_workspace_size(T, d, V, K, chunk, KD_WS_FUSED);
  if (ws_bytes == 0) {
    fprintf(stderr, "kd_topk_kl_workspace_size rejected the sizes\n");
    return 3;
  }
  CUDA_OK(cudaMalloc(&ws, ws_bytes));

  kd_status st = kd_topk_kl_fused_step(dH_in, dW_in, (const int32_t*)dIdx, (const float*)dP, T, d, V, K, chunk,
                                       1.0f, (float*)dLoss, (float*)dLse, NULL, (float*)ddH, (float*)ddW, 0, ws,
                                       ws_bytes, NULL);
  if (st != KD_OK) {
    fprintf(stderr, "kd_topk_kl_fused_step: %s\n", kd_status_string(st));
    return 4;
  }
  st = kd_topk_kl_device_status(ws, NULL);
  if (st != KD_OK) {
    fprintf(stderr, "device status: %s\n", kd_status_string(st));
    return 5;
  }
  float loss = 0.f;
  CUDA_OK(cudaMemcpy(&loss, dLoss, 4, cudaMemcpyDeviceToHost));
  CUDA_OK(cudaMemcpy(lse, dLse, (size_t)T * 4, cudaMemcpyDeviceToHost));
  CUDA_OK(cudaMemcpy(dH, ddH, nH * 4, cudaMemcpyDeviceToHost));
  CUDA_OK(cudaMemcpy(dW, ddW, nW * 4, cudaMemcpyDeviceToHost));

  FILE* out = fopen(argv[2], "wb");
  if (!out) {
    perror("open output");
    return 1;
  }
  if (write_all(out, &loss, 4) || write_all(out, lse, (size_t)T * 4) || write_all(out, dH, nH * 4) ||
      write_all(out, dW, nW * 4))
    return 1;
  fclose(out);
  cudaFree(dH_in);
  cudaFree(dW_in);
  cudaFree(dIdx);
  cudaFree(dP);
  cudaFree(dLoss);
  cudaFree(dLse);
  cudaFree(ddH);
  cudaFree(ddW);
  cudaFree(ws);
  free(H);
  free(W);
  free(idx);
  free(p);
  free(lse);
  free(dH);
  free(dW);
  return 0;
}
