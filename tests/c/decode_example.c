/* A plain C caller of the library: no PyTorch, only the CUDA runtime for
 * device memory.  One sequence, one KV group of four query heads, 4096
 * tokens of random bf16 keys and values: quantise, run one certified
 * decode step, read o, beta and the stop level back, check the device
 * status word.  Exit status 0 on success.
 *
 * Build (from the repository root):
 *   cc -std=c11 -I include -I /usr/local/cuda/include tests/c/decode_example.c \
 *      -L certified_sparse_attention_gb300/_lib -lcsa \
 *      -L /usr/local/cuda/lib64 -lcudart -lm -o decode_example
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "csa.h"

static uint16_t to_bf16(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);          /* round to nearest even */
  return (uint16_t)(u >> 16);
}

/* xorshift64* stream, Box-Muller normals */
static uint64_t rng_state = 0x9E3779B97F4A7C15ull;
static double uniform01(void) {
  rng_state ^= rng_state >> 12;
  rng_state ^= rng_state << 25;
  rng_state ^= rng_state >> 27;
  return ((rng_state * 0x2545F4914F6CDD1Dull) >> 11) * (1.0 / 9007199254740992.0) + 1e-300;
}
static float normal(void) {
  return (float)(sqrt(-2.0 * log(uniform01())) * cos(6.283185307179586 * uniform01()));
}

#define CHECK_CUDA(x) do { if ((x) != cudaSuccess) { fprintf(stderr, "cuda: %s\n", #x); return 1; } } while (0)
#define CHECK_CSA(x) do { csa_status s_ = (x); if (s_ != CSA_OK) { \
    fprintf(stderr, "%s: %s\n", #x, csa_status_string(s_)); return 1; } } while (0)

int main(void) {
  const int B = 1, Hq = 4, Hkv = 1, d = 128;
  const int64_t n = 4096;
  csa_shape shape = {B, Hq, Hkv, d, n, CSA_BF16};
  csa_params params = {0.05f, 0.05f, 2, CSA_MEASURE_VALUE, -1, 0, 0};
  const int64_t nblk = (n + 63) / 64;
  const size_t kv_elems = (size_t)B * Hkv * n * d;

  uint16_t* hq = malloc((size_t)B * Hq * d * 2);
  uint16_t* hk = malloc(kv_elems * 2);
  uint16_t* hv = malloc(kv_elems * 2);
  if (!hq || !hk || !hv) return 1;
  for (size_t i = 0; i < kv_elems; ++i) { hk[i] = to_bf16(normal()); hv[i] = to_bf16(normal()); }
  for (int i = 0; i < B * Hq * d; ++i) hq[i] = to_bf16(3.0f * normal());

  void *q, *K, *V, *K4, *bounds, *vmax, *vnorm2, *o, *beta, *level, *kread, *ws;
  size_t ws_bytes = csa_workspace_size(&shape, &params);
  if (ws_bytes == 0) return 1;
  CHECK_CUDA(cudaMalloc(&q, (size_t)B * Hq * d * 2));
  CHECK_CUDA(cudaMalloc(&K, kv_elems * 2));
  CHECK_CUDA(cudaMalloc(&V, kv_elems * 2));
  CHECK_CUDA(cudaMalloc(&K4, (size_t)B * Hkv * nblk * 64 * (d / 2)));
  CHECK_CUDA(cudaMalloc(&bounds, (size_t)B * Hkv * nblk * 2 * d * 4));
  CHECK_CUDA(cudaMalloc(&vmax, (size_t)B * Hkv * nblk * 4));
  CHECK_CUDA(cudaMalloc(&vnorm2, (size_t)B * Hkv * n * 4));
  CHECK_CUDA(cudaMalloc(&o, (size_t)B * Hq * d * 4));
  CHECK_CUDA(cudaMalloc(&beta, (size_t)B * Hq * 4));
  CHECK_CUDA(cudaMalloc(&level, (size_t)B * Hq * 4));
  CHECK_CUDA(cudaMalloc(&kread, (size_t)B * Hq * 4));
  CHECK_CUDA(cudaMalloc(&ws, ws_bytes));
  CHECK_CUDA(cudaMemcpy(q, hq, (size_t)B * Hq * d * 2, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(K, hk, kv_elems * 2, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(V, hv, kv_elems * 2, cudaMemcpyHostToDevice));

  const int64_t len[1] = {n};
  const uint64_t seed[1] = {20261202ull};
  CHECK_CSA(csa_quantize_keys(&shape, K, V, len, 0, K4, bounds, vmax, vnorm2, NULL));
  CHECK_CSA(csa_decode_step(&shape, &params, q, K, V, K4, bounds, vmax, vnorm2, len, seed,
                            o, beta, level, kread, NULL, ws, ws_bytes, NULL));
  CHECK_CSA(csa_check(ws, NULL));

  float ho[4 * 128], hb[4];
  int32_t hl[4], hkr[4];
  CHECK_CUDA(cudaMemcpy(ho, o, sizeof(ho), cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(hb, beta, sizeof(hb), cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(hl, level, sizeof(hl), cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(hkr, kread, sizeof(hkr), cudaMemcpyDeviceToHost));
  for (int h = 0; h < Hq; ++h) {
    if (!isfinite(hb[h]) || hb[h] < 0.f || hkr[h] < 64 || hkr[h] > n) return 2;
    for (int c = 0; c < d; ++c)
      if (!isfinite(ho[h * d + c])) return 2;
    printf("head %d: level %d beta %.4g keys_read %d\n", h, hl[h], hb[h], hkr[h]);
  }
  return 0;
}
