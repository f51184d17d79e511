// Block key summaries: build from host KV, and the append path that keeps them current.
//
// OasisKV (paperlayer.ai/abs/2608.08097v1, "4 System Design"): the prototype keeps a
// coordinate-wise minimum and maximum key per block, two vectors per block, in HBM. Min and
// max are exact in any evaluation order; ties keep the earlier token (strict comparison),
// so the stored bit patterns are fixed by the data alone.
#include <cuda_bf16.h>

#include "okv_internal.h"

namespace okv {
namespace {

template <typename T>
struct Vec;  // 16-byte vector of storage elements
template <>
struct Vec<float> {
  static constexpr int N = 4;
};
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
};

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

__device__ __forceinline__ void record_error(int32_t* err, int32_t code, int32_t a, int32_t b,
                                             int32_t c) {
  if (atomicCAS(err, 0, code) == 0) {
    err[1] = a;
    err[2] = b;
    err[3] = c;
  }
}

// One thread per (layer, head, block, 16-byte vector of dims).
template <typename T>
__global__ void summary_build_kernel(Geom G, int32_t layer_begin, int32_t n_layers, int32_t req,
                                     const uint8_t* __restrict__ host_kv, int32_t cap_blocks,
                                     int32_t n_tok, uint8_t* __restrict__ summ_base) {
  constexpr int V = Vec<T>::N;
  const int32_t nvec = G.d / V;
  const int32_t nb = (n_tok + G.bs - 1) / G.bs;
  const int64_t total = (int64_t)n_layers * G.Hkv * nb * nvec;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t v = (int32_t)(i % nvec);
    int64_t rest = i / nvec;
    const int32_t b = (int32_t)(rest % nb);
    rest /= nb;
    const int32_t h = (int32_t)(rest % G.Hkv);
    const int32_t layer = layer_begin + (int32_t)(rest / G.Hkv);
    const int32_t nv = min(G.bs, n_tok - b * G.bs);
    const T* kblk = reinterpret_cast<const T*>(
        host_kv + (((int64_t)layer * G.Hkv + h) * cap_blocks + b) * G.block_bytes);
    union U {
      uint4 u;
      T e[V];
    } x, mn, mx;
    mn.u = *reinterpret_cast<const uint4*>(kblk + v * V);
    mx.u = mn.u;
    for (int32_t t = 1; t < nv; ++t) {
      x.u = *reinterpret_cast<const uint4*>(kblk + (int64_t)t * G.d + v * V);
#pragma unroll
      for (int e = 0; e < V; ++e) {
        if (to_f(x.e[e]) < to_f(mn.e[e])) mn.e[e] = x.e[e];
        if (to_f(x.e[e]) > to_f(mx.e[e])) mx.e[e] = x.e[e];
      }
    }
    T* out = reinterpret_cast<T*>(summ_base) +
             ((((int64_t)layer * G.R + req) * G.Hkv + h) * G.nb_max + b) * 2 * G.d;
    *reinterpret_cast<uint4*>(out + v * V) = mn.u;
    *reinterpret_cast<uint4*>(out + G.d + v * V) = mx.u;
  }
}

// grid (n_active, Hkv), one thread per dimension. The last of a request's Hkv CTAs to finish
// (counted in arrivals[r], which starts at zero and is left at zero) advances its length.
template <typename T>
__global__ void append_kernel(Geom G, LayerState S, ReqTables T_, int32_t layer,
                              const T* __restrict__ k_new, const T* __restrict__ v_new,
                              int32_t* __restrict__ arrivals, int32_t* err) {
  const int32_t r = T_.active[blockIdx.x];
  const int32_t h = blockIdx.y;
  const int32_t pos = S.len[r];
  const int32_t cap = T_.cap_blocks[r];
  const int32_t lcap = T_.local_cap[r];
  const int64_t unit = (int64_t)r * G.Hkv + h;
  __shared__ int32_t tail_slot;   // slot holding the tail block, or -1
  __shared__ int32_t kept_entry;  // decode-side entry of the tail block (partial staging), or -1
  __shared__ int32_t skip;        // a check failed: write nothing
  if (threadIdx.x == 0) {
    tail_slot = -1;
    kept_entry = -1;
    skip = 0;
    if (pos < 0 || pos >= cap * G.bs || pos >= G.nb_max * G.bs) {
      record_error(err, kErrCapacity, layer, r, pos);
      skip = 1;
    } else if (lcap > 0) {
      const int32_t e = S.local_of[unit * G.nb_max + pos / G.bs];
      if (e >= lcap) {
        record_error(err, kErrLocalRange, layer, r, e);
        skip = 1;
      } else {
        kept_entry = e;
      }
    }
  }
  __syncthreads();
  if (!skip) {
    const int32_t b = pos / G.bs, t = pos % G.bs;
    const int64_t kofs = (int64_t)t * G.d, vofs = (int64_t)(G.bs + t) * G.d;
    for (int32_t s = threadIdx.x; s < G.kb; s += blockDim.x)
      if (S.slot_block[unit * G.kb + s] == b) tail_slot = s;
    __syncthreads();
    T* host = reinterpret_cast<T*>(T_.host_kv[r] + (((int64_t)layer * G.Hkv + h) * cap + b) * G.block_bytes);
    T* pool = tail_slot >= 0 ? reinterpret_cast<T*>(S.pool + (unit * G.kb + tail_slot) * G.block_bytes) : nullptr;
    // a partially staged request also writes the decode side's kept copy of the block, if any
    T* kept = kept_entry >= 0 ? reinterpret_cast<T*>(T_.local_kv[r] +
                                                     (((int64_t)layer * G.Hkv + h) * lcap + kept_entry) *
                                                         G.block_bytes)
                              : nullptr;
    T* summ = reinterpret_cast<T*>(S.summ) + (unit * G.nb_max + b) * 2 * G.d;
    for (int32_t c = threadIdx.x; c < G.d; c += blockDim.x) {
      const T k = k_new[unit * G.d + c];
      const T v = v_new[unit * G.d + c];
      host[kofs + c] = k;
      host[vofs + c] = v;
      if (pool) {
        pool[kofs + c] = k;
        pool[vofs + c] = v;
      }
      if (kept) {
        kept[kofs + c] = k;
        kept[vofs + c] = v;
      }
      if (t == 0) {
        summ[c] = k;
        summ[G.d + c] = k;
      } else {
        if (to_f(k) < to_f(summ[c])) summ[c] = k;
        if (to_f(k) > to_f(summ[G.d + c])) summ[G.d + c] = k;
      }
    }
  }
  // every CTA of the request has read the length before the last one advances it
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0 && atomicAdd(&arrivals[r], 1) == G.Hkv - 1) {
    arrivals[r] = 0;
    __threadfence();
    S.len[r] = pos + 1;
    S.len_act[blockIdx.x] = pos + 1;
  }
}

// grid (layers, Hkv): empty pool, tables and decode-side tier of one request on every layer.
__global__ void reset_request_kernel(Geom G, StateBase B, RequestInit q) {
  const int32_t layer = blockIdx.x, h = blockIdx.y;
  const int64_t units = (int64_t)G.R * G.Hkv;
  const int64_t u = (int64_t)layer * units + (int64_t)q.req * G.Hkv + h;
  for (int32_t i = threadIdx.x; i < G.kb; i += blockDim.x) {
    B.slot_block[u * G.kb + i] = -1;
    B.stamp[u * G.kb + i] = -1;
  }
  for (int32_t i = threadIdx.x; i < G.nb_max; i += blockDim.x) B.local_of[u * G.nb_max + i] = -1;
  if (threadIdx.x == 0) {
    B.n_sel[u] = 0;
    B.n_fetch[u] = 0;
    B.local_used[u] = 0;
    if (h == 0) B.len[(int64_t)layer * G.R + q.req] = q.n_tok;
    if (h == 0 && layer == 0) {
      B.host_kv_tab[q.req] = q.host_kv;
      B.cap_tab[q.req] = q.cap;
      B.local_kv_tab[q.req] = q.local_kv;
      B.local_cap_tab[q.req] = q.local_cap;
    }
  }
}

}  // namespace

cudaError_t launch_summary_build(const Geom& G, int32_t layer_begin, int32_t layer_end,
                                 int32_t req, uint64_t host_kv, int32_t cap_blocks,
                                 int32_t n_tok, uint8_t* summ_base, int32_t* err,
                                 cudaStream_t s) {
  (void)err;
  if (n_tok <= 0 || layer_end <= layer_begin) return cudaSuccess;
  const int32_t nb = (n_tok + G.bs - 1) / G.bs;
  const int32_t V = G.dtype == OKV_F32 ? 4 : 8;
  const int64_t total = (int64_t)(layer_end - layer_begin) * G.Hkv * nb * (G.d / V);
  const int threads = 256;
  const int64_t want = (total + threads - 1) / threads;
  const int blocks = (int)(want < 152 * 32 ? want : 152 * 32);
  const uint8_t* src = reinterpret_cast<const uint8_t*>(host_kv);
  if (G.dtype == OKV_F32)
    summary_build_kernel<float><<<blocks, threads, 0, s>>>(G, layer_begin, layer_end - layer_begin,
                                                          req, src, cap_blocks, n_tok, summ_base);
  else
    summary_build_kernel<__nv_bfloat16><<<blocks, threads, 0, s>>>(
        G, layer_begin, layer_end - layer_begin, req, src, cap_blocks, n_tok, summ_base);
  return cudaGetLastError();
}

cudaError_t launch_append(const Geom& G, const LayerState& S, const ReqTables& T, int32_t n_active,
                          int32_t layer, const void* k_new, const void* v_new, int32_t* arrivals,
                          int32_t* err, cudaStream_t s) {
  if (n_active <= 0) return cudaSuccess;
  dim3 grid(n_active, G.Hkv);
  const int threads = G.d < 256 ? G.d : 256;
  if (G.dtype == OKV_F32)
    append_kernel<float><<<grid, threads, 0, s>>>(G, S, T, layer, (const float*)k_new,
                                                  (const float*)v_new, arrivals, err);
  else
    append_kernel<__nv_bfloat16><<<grid, threads, 0, s>>>(
        G, S, T, layer, (const __nv_bfloat16*)k_new, (const __nv_bfloat16*)v_new, arrivals, err);
  return cudaGetLastError();
}

cudaError_t launch_reset_request(const Geom& G, const StateBase& B, const RequestInit& q, cudaStream_t s) {
  dim3 grid(G.L, G.Hkv);
  reset_request_kernel<<<grid, 256, 0, s>>>(G, B, q);
  return cudaGetLastError();
}

}  // namespace okv
