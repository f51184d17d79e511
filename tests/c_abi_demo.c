/*
 * A plain C caller of the okv C ABI: no Python, no torch, device buffers from cudaMalloc.
 *
 * One small request (fp32, 4 query / 2 KV heads, d 32, 100 tokens = 7 blocks of 16) goes through
 * okv_stage (cap 1.0) and okv_attend. The budget (8 slots) covers the context, so every block is
 * staged and the sparse attention must equal dense softmax attention, which this program
 * computes itself in double precision from the same host KV (OasisKV, "4 System Design":
 * attention over the resident KV; with the whole context resident that is ordinary decode
 * attention). Prints one line and exits 0 when the maximum absolute error is at most 1e-5.
 */
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "okv.h"

enum { L = 1, HQ = 4, HKV = 2, D = 32, BS = 16, NTOK = 100, CAP = 8, G = HQ / HKV };

static okv_ctx* ctx = NULL;

static int check(okv_status s, const char* what) {
  if (s == OKV_OK) return 0;
  fprintf(stderr, "%s: %s (%s)\n", what, okv_status_string(s), ctx ? okv_last_error(ctx) : "");
  return 1;
}

/* deterministic values in [-1, 1) from a small integer hash */
static float value(unsigned kind, unsigned h, unsigned t, unsigned c) {
  unsigned x = kind * 0x9E3779B9u ^ h * 0x85EBCA6Bu ^ t * 0xC2B2AE35u ^ c * 0x27D4EB2Fu;
  x ^= x >> 16;
  x *= 0x7FEB352Du;
  x ^= x >> 15;
  x *= 0x846CA68Bu;
  x ^= x >> 16;
  return (float)((double)(x & 0xFFFFFu) / 524288.0 - 1.0);
}

static size_t kv_index(int h, int t, int which, int c) {
  const int b = t / BS, i = t % BS;
  return ((((size_t)h * CAP + b) * 2 + which) * BS + i) * D + c;
}

int main(void) {
  okv_config cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.layers = L;
  cfg.q_heads = HQ;
  cfg.kv_heads = HKV;
  cfg.head_dim = D;
  cfg.block_size = BS;
  cfg.budget_tokens = CAP * BS;
  cfg.max_requests = 1;
  cfg.max_blocks_per_request = CAP;
  cfg.fetch_cap = 1.0f;
  cfg.dtype = OKV_F32;
  if (check(okv_create(&cfg, &ctx), "okv_create")) return 1;

  const size_t host_bytes = (size_t)L * HKV * CAP * 2 * BS * D * sizeof(float);
  void* host = NULL;
  if (check(okv_host_alloc((int64_t)host_bytes, &host), "okv_host_alloc")) return 1;
  float* kv = (float*)host; /* [L][Hkv][cap][2][bs][d], K then V */
  memset(kv, 0, host_bytes);
  for (int h = 0; h < HKV; ++h)
    for (int t = 0; t < NTOK; ++t)
      for (int c = 0; c < D; ++c) {
        kv[kv_index(h, t, 0, c)] = value(1, h, t, c);
        kv[kv_index(h, t, 1, c)] = value(2, h, t, c);
      }
  if (check(okv_add_request(ctx, 0, host, CAP, NTOK, NULL), "okv_add_request")) return 1;

  float q_host[HQ * D], out_host[HQ * D];
  for (int j = 0; j < HQ; ++j)
    for (int c = 0; c < D; ++c) q_host[j * D + c] = value(3, j, 0, c);
  float *q = NULL, *out = NULL;
  if (cudaMalloc((void**)&q, sizeof q_host) != cudaSuccess || cudaMalloc((void**)&out, sizeof q_host) != cudaSuccess) {
    fprintf(stderr, "cudaMalloc failed\n");
    return 1;
  }
  cudaMemcpy(q, q_host, sizeof q_host, cudaMemcpyHostToDevice);

  /* the query serves as its own draft: stage every block, then attend */
  if (check(okv_stage(ctx, 0, q, 0, 1.0f, NULL), "okv_stage")) return 1;
  if (check(okv_attend(ctx, 0, q, out, NULL), "okv_attend")) return 1;
  if (cudaDeviceSynchronize() != cudaSuccess) {
    fprintf(stderr, "cudaDeviceSynchronize failed\n");
    return 1;
  }
  if (check(okv_sync(ctx, 10000), "okv_sync")) return 1;
  cudaMemcpy(out_host, out, sizeof out_host, cudaMemcpyDeviceToHost);

  int32_t counts[HKV], ids[HKV * CAP];
  if (check(okv_read_selection(ctx, 0, counts, ids, NULL), "okv_read_selection")) return 1;
  const int nb = (NTOK + BS - 1) / BS;
  for (int h = 0; h < HKV; ++h)
    if (counts[h] != nb) {
      fprintf(stderr, "kv head %d selected %d blocks, expected %d\n", h, counts[h], nb);
      return 1;
    }

  /* dense softmax attention in double precision: softmax(q.k / sqrt(d)) v over all tokens */
  double max_err = 0.0;
  for (int j = 0; j < HQ; ++j) {
    const int h = j / G;
    double z[NTOK], zmax = -INFINITY;
    for (int t = 0; t < NTOK; ++t) {
      double dot = 0.0;
      for (int c = 0; c < D; ++c) dot += (double)q_host[j * D + c] * kv[kv_index(h, t, 0, c)];
      z[t] = dot / sqrt((double)D);
      if (z[t] > zmax) zmax = z[t];
    }
    double den = 0.0;
    for (int t = 0; t < NTOK; ++t) {
      z[t] = exp(z[t] - zmax);
      den += z[t];
    }
    for (int c = 0; c < D; ++c) {
      double o = 0.0;
      for (int t = 0; t < NTOK; ++t) o += z[t] * kv[kv_index(h, t, 1, c)];
      const double err = fabs(o / den - out_host[j * D + c]);
      if (err > max_err) max_err = err;
    }
  }

  cudaFree(q);
  cudaFree(out);
  okv_destroy(ctx);
  okv_host_free(host);
  printf("c abi demo: %d blocks staged per kv head, attention max abs error %.3g\n", nb, max_err);
  return max_err <= 1e-5 ? 0 : 1;
}
