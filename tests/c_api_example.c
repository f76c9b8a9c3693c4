/*
 * A plain-C user of the library: one MoE layer through include/cb_moe.h and
 * the CUDA runtime only (no C++, no PyTorch).  tests/test_c_api_example.py
 * compiles and links it on every machine and runs it where a GB300 is
 * present.
 *
 * Usage: c_api_example   (prints "ok" and exits 0 on success)
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "cb_moe.h"

#define CHECK(call)                                                   \
  do {                                                                \
    cb_status_t st_ = (call);                                         \
    if (st_ != CB_OK) {                                               \
      fprintf(stderr, "%s: %s\n", #call, cb_status_string(st_));      \
      return 1;                                                       \
    }                                                                 \
  } while (0)

/* bf16 bits of a float (round to nearest even) */
static uint16_t to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

/* a device buffer of n bf16 values drawn from [-scale, scale) */
static void *device_bf16(size_t n, float scale, unsigned *seed) {
  uint16_t *h = (uint16_t *)malloc(n * 2);
  void *d = NULL;
  for (size_t i = 0; i < n; ++i) {
    *seed = *seed * 1664525u + 1013904223u;
    h[i] = to_bf16(((float)(*seed >> 8) / 16777216.0f * 2.0f - 1.0f) * scale);
  }
  if (cudaMalloc(&d, n * 2) != cudaSuccess || cudaMemcpy(d, h, n * 2, cudaMemcpyHostToDevice) != cudaSuccess) d = NULL;
  free(h);
  return d;
}

int main(void) {
  const int T = 256, d = 512, f = 1024, E = 8, k = 2;
  unsigned seed = 1;
  cb_moe_config_t cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.n_tokens = T;
  cfg.d_model = d;
  cfg.d_ff = f;
  cfg.n_experts = E;
  cfg.top_k = k;
  cfg.wdtype = CB_W_BF16;
  cfg.router_mode = CB_ROUTER_SOFTMAX_TOPK;

  uint64_t bytes = 0;
  CHECK(cb_moe_device_bytes(&cfg, &bytes));
  int n_dev = 0;
  if (cudaGetDeviceCount(&n_dev) != cudaSuccess || n_dev == 0) {
    printf("workspace %.1f MB; no GPU here, nothing run\n", (double)bytes / 1e6);
    return 0;
  }

  cb_moe_weights_t w;
  memset(&w, 0, sizeof w);
  w.w_router = device_bf16((size_t)E * d, 0.3f, &seed);
  w.w_gate = device_bf16((size_t)E * f * d, 0.02f, &seed);
  w.w_up = device_bf16((size_t)E * f * d, 0.02f, &seed);
  w.w_down = device_bf16((size_t)E * d * f, 0.02f, &seed);
  void *x = device_bf16((size_t)T * d, 1.0f, &seed);
  void *out = NULL;
  if (!w.w_router || !w.w_gate || !w.w_up || !w.w_down || !x || cudaMalloc(&out, (size_t)T * d * 2) != cudaSuccess) {
    fprintf(stderr, "device allocation failed\n");
    return 1;
  }

  cb_moe_t *h = NULL;
  CHECK(cb_moe_init(&cfg, &w, &h));
  /* the handle copied the weights: the caller's copies may go */
  cudaFree((void *)w.w_router);
  cudaFree((void *)w.w_gate);
  cudaFree((void *)w.w_up);
  cudaFree((void *)w.w_down);

  cudaStream_t s;
  if (cudaStreamCreate(&s) != cudaSuccess) return 1;
  for (int i = 0; i < 3; ++i) CHECK(cb_moe_forward(h, x, out, s));
  if (cudaStreamSynchronize(s) != cudaSuccess) return 1;
  CHECK(cb_moe_last_error(h));

  cb_routing_view_t v;
  CHECK(cb_moe_routing(h, &v));
  int32_t counts[8], total = 0;
  if (cudaMemcpy(counts, v.counts, sizeof counts, cudaMemcpyDeviceToHost) != cudaSuccess) return 1;
  for (int e = 0; e < E; ++e) total += counts[e];
  if (total != T * k) {
    fprintf(stderr, "routed rows %d, expected %d\n", total, T * k);
    return 1;
  }
  uint16_t first[4];
  if (cudaMemcpy(first, out, sizeof first, cudaMemcpyDeviceToHost) != cudaSuccess) return 1;

  CHECK(cb_moe_free(h));
  cudaStreamDestroy(s);
  cudaFree(x);
  cudaFree(out);
  printf("out[0][0..3] bf16 bits %04x %04x %04x %04x\nok\n", first[0], first[1], first[2], first[3]);
  return 0;
}
