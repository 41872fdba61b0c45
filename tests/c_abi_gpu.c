/* A decode driven from C alone: device buffers through the CUDA runtime, the
 * call through include/vt_paged_attn.h, and the result compared with the C
 * oracle (oracle_decode, fp64) on the same host data.  A small batch of bf16
 * pages (contexts 1, 33 and 100 tokens, GQA 4, head_dim 128, a permuted page
 * pool whose unused slots hold NaN), with and without a window.  Exit status
 * 0 and "c abi gpu: ok" when every output is within the bf16 tolerances. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "vt_paged_attn.h"

/* the oracle's entry point (oracle/paged_attn_oracle.c) */
int oracle_decode(double* out, const void* q, const void* k_cache, const void* v_cache, int elem,
                  const int32_t* block_tables, const int32_t* context_lens, int num_seqs, int num_q_heads,
                  int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq, int num_blocks,
                  double scale, int window);

enum { B = 3, HQ = 8, HKV = 2, D = 128, P = 32, MAXB = 4, NB = 9 };

static uint32_t lcg_state = 12345u;
static float uniform(void) { /* [-1, 1) */
  lcg_state = lcg_state * 1664525u + 1013904223u;
  return (float)((lcg_state >> 8) & 0xffffffu) / 8388608.0f - 1.0f;
}
static uint16_t to_bf16(float x) { /* round to nearest even */
  uint32_t u;
  memcpy(&u, &x, 4);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}
static float from_bf16(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float x;
  memcpy(&x, &u, 4);
  return x;
}

#define CUDA(call)                                                          \
  do {                                                                      \
    cudaError_t e_ = (call);                                                \
    if (e_ != cudaSuccess) {                                                \
      printf("CUDA error %s at %s:%d\n", cudaGetErrorString(e_), __FILE__, __LINE__); \
      return 1;                                                             \
    }                                                                       \
  } while (0)

int main(void) {
  static uint16_t q[B * HQ * D], kc[NB * P * HKV * D], vc[NB * P * HKV * D], out[B * HQ * D];
  static double ref[B * HQ * D];
  const int32_t lens[B] = {1, 33, 100};
  const int32_t perm[NB] = {5, 2, 7, 0, 8, 3, 1, 6, 4};
  int32_t bt[B * MAXB];
  size_t i;
  int b, j, w, used = 0;
  const float scale = 0.0883883476f; /* 1 / sqrt(128) */
  void *dq, *dk, *dv, *dout, *dbt, *dcl;

  for (i = 0; i < B * HQ * D; ++i) q[i] = to_bf16(uniform());
  for (i = 0; i < (size_t)NB * P * HKV * D; ++i) {
    kc[i] = 0x7fc0u; /* NaN: slots no context reaches */
    vc[i] = 0x7fc0u;
  }
  for (b = 0; b < B; ++b) {
    const int pages = (lens[b] + P - 1) / P;
    for (j = 0; j < MAXB; ++j) bt[b * MAXB + j] = perm[(used + j) % NB];
    for (j = 0; j < pages; ++j) {
      const int page = bt[b * MAXB + j];
      int slot;
      for (slot = 0; slot < P && j * P + slot < lens[b]; ++slot)
        for (i = 0; i < (size_t)HKV * D; ++i) {
          kc[((size_t)page * P + slot) * HKV * D + i] = to_bf16(uniform());
          vc[((size_t)page * P + slot) * HKV * D + i] = to_bf16(uniform());
        }
    }
    used += pages;
  }

  CUDA(cudaMalloc(&dq, sizeof q));
  CUDA(cudaMalloc(&dk, sizeof kc));
  CUDA(cudaMalloc(&dv, sizeof vc));
  CUDA(cudaMalloc(&dout, sizeof out));
  CUDA(cudaMalloc(&dbt, sizeof bt));
  CUDA(cudaMalloc(&dcl, sizeof lens));
  CUDA(cudaMemcpy(dq, q, sizeof q, cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(dk, kc, sizeof kc, cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(dv, vc, sizeof vc, cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(dbt, bt, sizeof bt, cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(dcl, lens, sizeof lens, cudaMemcpyHostToDevice));

  for (w = 0; w < 2; ++w) {
    const int window = w ? 40 : 0;
    unsigned status = 1u;
    double err2 = 0.0, ref2 = 0.0, maxabs = 0.0;
    vt_status st = vt_paged_attn_decode(dout, dq, dk, dv, (const int32_t*)dbt, (const int32_t*)dcl, B, HQ, HKV, D,
                                        P, scale, window, NULL, MAXB, NB, VT_BF16);
    if (st != VT_OK) {
      printf("decode: %s (%s)\n", vt_status_string(st), vt_last_cuda_error());
      return 1;
    }
    CUDA(cudaDeviceSynchronize());
    if (vt_paged_attn_device_status(NULL, &status) != VT_OK || status != 0u) {
      printf("device status %u\n", status);
      return 1;
    }
    CUDA(cudaMemcpy(out, dout, sizeof out, cudaMemcpyDeviceToHost));
    if (oracle_decode(ref, q, kc, vc, 0, bt, lens, B, HQ, HKV, D, P, MAXB, NB, scale, window) != 0) {
      printf("oracle failed\n");
      return 1;
    }
    for (i = 0; i < B * HQ * D; ++i) {
      const double e = (double)from_bf16(out[i]) - ref[i];
      if (!(fabs(e) <= maxabs)) maxabs = fabs(e); /* also catches NaN */
      err2 += e * e;
      ref2 += ref[i] * ref[i];
    }
    printf("window %d: nmse %.3e max|err| %.3e\n", window, err2 / ref2, maxabs);
    if (!(err2 / ref2 <= 5e-4) || !(maxabs <= 2e-2)) {
      printf("c abi gpu: FAIL\n");
      return 1;
    }
  }
  cudaFree(dq);
  cudaFree(dk);
  cudaFree(dv);
  cudaFree(dout);
  cudaFree(dbt);
  cudaFree(dcl);
  printf("c abi gpu: ok\n");
  return 0;
}
