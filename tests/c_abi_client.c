/*
 * A plain C client of libattn.so (no PyTorch): reads B, H, S, causal and BF16 Q, K, V from a
 * binary file, runs attn_fwd or attn_fwd_causal through the C ABI on device buffers it
 * allocates with the CUDA runtime, and writes BF16 O and fp32 lse to another file.
 *
 *   input  file: int32 B, H, S, causal; then Q, K, V as uint16 BF16 [B, H, S, 128] each
 *   output file: O as uint16 BF16 [B, H, S, 128], then lse as float32 [B, H, S]
 *
 * Exit status: 0 on success; 2 bad usage or I/O; 3 a CUDA runtime call failed; 10 + the
 * attn_status code if the library call failed; 20 if a bounded wait gave up.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime.h>

#include "attn.h"

static int check(cudaError_t e, const char* what) {
  if (e != cudaSuccess) {
    fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
    return 1;
  }
  return 0;
}

int main(int argc, char** argv) {
  if (argc != 3) {
    fprintf(stderr, "usage: %s input.bin output.bin\n", argv[0]);
    return 2;
  }
  FILE* f = fopen(argv[1], "rb");
  if (!f) return 2;
  int32_t hdr[4];
  if (fread(hdr, sizeof(int32_t), 4, f) != 4) return 2;
  const int B = hdr[0], H = hdr[1], S = hdr[2], causal = hdr[3];
  const size_t n = (size_t)B * H * S * 128, rows = (size_t)B * H * S;
  uint16_t* host = (uint16_t*)malloc(3 * n * sizeof(uint16_t));
  float* lse_h = (float*)malloc(rows * sizeof(float));
  if (!host || !lse_h) return 2;
  if (fread(host, sizeof(uint16_t), 3 * n, f) != 3 * n) return 2;
  fclose(f);

  void *q, *k, *v, *o;
  float* lse;
  if (check(cudaMalloc(&q, n * 2), "cudaMalloc") || check(cudaMalloc(&k, n * 2), "cudaMalloc") ||
      check(cudaMalloc(&v, n * 2), "cudaMalloc") || check(cudaMalloc(&o, n * 2), "cudaMalloc") ||
      check(cudaMalloc((void**)&lse, rows * sizeof(float)), "cudaMalloc"))
    return 3;
  cudaStream_t stream;
  if (check(cudaStreamCreate(&stream), "cudaStreamCreate")) return 3;
  if (check(cudaMemcpy(q, host, n * 2, cudaMemcpyHostToDevice), "copy q") ||
      check(cudaMemcpy(k, host + n, n * 2, cudaMemcpyHostToDevice), "copy k") ||
      check(cudaMemcpy(v, host + 2 * n, n * 2, cudaMemcpyHostToDevice), "copy v"))
    return 3;

  const float scale = 0.08838834764831845f; /* 1/sqrt(128) */
  const int st = causal ? attn_fwd_causal(q, k, v, o, lse, B, H, S, 128, scale, stream)
                        : attn_fwd(q, k, v, o, lse, B, H, S, 128, scale, stream);
  if (st != ATTN_OK) {
    fprintf(stderr, "attn: %s\n", attn_status_string(st));
    return 10 + st;
  }
  if (check(cudaStreamSynchronize(stream), "synchronize")) return 3;
  unsigned int word = 0;
  if (attn_device_status(&word, 1) != ATTN_OK || word != 0) {
    fprintf(stderr, "status word %#x\n", word);
    return 20;
  }
  if (check(cudaMemcpy(host, o, n * 2, cudaMemcpyDeviceToHost), "copy o") ||
      check(cudaMemcpy(lse_h, lse, rows * sizeof(float), cudaMemcpyDeviceToHost), "copy lse"))
    return 3;

  FILE* g = fopen(argv[2], "wb");
  if (!g) return 2;
  if (fwrite(host, sizeof(uint16_t), n, g) != n || fwrite(lse_h, sizeof(float), rows, g) != rows) return 2;
  fclose(g);
  printf("attn version %d.%d: B=%d H=%d S=%d causal=%d ok\n", attn_version() >> 16, attn_version() & 0xFFFF, B,
         H, S, causal);
  cudaFree(q);
  cudaFree(k);
  cudaFree(v);
  cudaFree(o);
  cudaFree(lse);
  cudaStreamDestroy(stream);
  free(host);
  free(lse_h);
  return 0;
}
