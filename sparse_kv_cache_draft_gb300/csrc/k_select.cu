// Lookahead block scoring, per-head top-K and KV selection (diff / admit / evict).
//
// OasisKV (paperlayer.ai/abs/2608.08097v1, "4 System Design"): the draft query scans the
// per-block min/max key summaries to rank blocks; each layer's background chain is top-K
// prediction, then KV selection, which moves at most C blocks per KV head, keeps resident
// predicted blocks and pairs admitted blocks with least-recently-selected eviction targets.
#include <cuda_bf16.h>

#include "okv_internal.h"

namespace okv {
namespace {

constexpr int kScoreThreads = 256;

__device__ __forceinline__ void record_error(int32_t* err, int32_t code, int32_t a, int32_t b,
                                             int32_t c) {
  if (atomicCAS(err, 0, code) == 0) {
    err[1] = a;
    err[2] = b;
    err[3] = c;
  }
}

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

// Order-preserving map of a binary32 score to an unsigned key (larger score, larger key).
__device__ __forceinline__ uint32_t orderable(float s) {
  const uint32_t u = __float_as_uint(s + 0.0f);  // -0 becomes +0: equal scores tie
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float from_orderable(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// ---- score + top-K ------------------------------------------------------------------------
//
// Score of block b for KV head h: sum over the g query heads of the group of
// sum_c max(q_c kmin_c, q_c kmax_c) = sum_c (P_c kmax_c + N_c kmin_c), P_c (N_c) being the sum
// of the group's positive (negative) query coordinates. One CTA per unit; each warp reads one
// 16-byte vector per lane of a block's [kmin | kmax] record (2d elements), multiplies by the
// matching N or P coefficient and reduces across the warp. Keys (orderable score, ~block id)
// then go through a bitonic sort in shared memory, descending: score desc, block id asc.
template <typename T>
__global__ void __launch_bounds__(kScoreThreads)
score_topk_kernel(Geom G, LayerState S, ReqTables RT, int32_t np2, const T* __restrict__ draft,
                  int32_t* err) {
  constexpr int V = 16 / sizeof(T);
  extern __shared__ __align__(16) uint8_t smem[];
  float* coef = reinterpret_cast<float*>(smem);                               // [2d]
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(coef + 2 * G.d);  // [np2]

  const int32_t a = blockIdx.x / G.Hkv, h = blockIdx.x % G.Hkv;
  const int32_t r = RT.active[a];
  const int64_t unit = (int64_t)r * G.Hkv + h;
  const int32_t len = S.len[r];
  const int32_t nb = (len + G.bs - 1) / G.bs;
  if (nb > np2 || nb > G.nb_max) {
    if (threadIdx.x == 0) record_error(err, kErrLength, -1, r, len);
    return;
  }

  // P_c (max part, multiplies kmax) and N_c (min part, multiplies kmin), group heads in order
  for (int32_t c = threadIdx.x; c < G.d; c += blockDim.x) {
    float p = 0.f, n = 0.f;
    for (int32_t j = 0; j < G.g; ++j) {
      const float x = to_f(draft[((int64_t)r * G.Hq + h * G.g + j) * G.d + c]);
      p += x > 0.f ? x : 0.f;
      n += x < 0.f ? x : 0.f;
    }
    coef[c] = n;
    coef[G.d + c] = p;
  }
  __syncthreads();

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int32_t nvec = 2 * G.d / V;  // 16-byte vectors per summary record
  const T* summ = reinterpret_cast<const T*>(S.summ) + unit * G.nb_max * 2 * G.d;
  constexpr int U = 4;  // blocks in flight per warp
  for (int32_t b0 = warp * U; b0 < nb; b0 += nwarps * U) {
    float part[U];
#pragma unroll
    for (int u = 0; u < U; ++u) part[u] = 0.f;
    for (int32_t v = lane; v < nvec; v += 32) {
      union {
        uint4 u4;
        T e[V];
      } x[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int32_t b = b0 + u;
        if (b < nb)
          x[u].u4 = __ldcs(reinterpret_cast<const uint4*>(summ + (int64_t)b * 2 * G.d) + v);
        else
          x[u].u4 = make_uint4(0, 0, 0, 0);
      }
      const float* cf = coef + v * V;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < V; ++e) acc = fmaf(cf[e], to_f(x[u].e[e]), acc);
        part[u] += acc;
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) part[u] += __shfl_xor_sync(0xffffffffu, part[u], o);
    }
    if (lane < U) {
      float s = part[0];
#pragma unroll
      for (int u = 1; u < U; ++u)
        if (lane == u) s = part[u];
      const int32_t b = b0 + lane;
      if (b < nb)
        keys[b] = ((unsigned long long)orderable(s) << 32) | (unsigned long long)(~(uint32_t)b);
    }
  }
  for (int32_t i = nb + threadIdx.x; i < np2; i += blockDim.x) keys[i] = 0ull;  // below any score
  __syncthreads();

  // bitonic sort, descending
  for (int32_t k = 2; k <= np2; k <<= 1) {
    for (int32_t j = k >> 1; j > 0; j >>= 1) {
      for (int32_t i = threadIdx.x; i < np2; i += blockDim.x) {
        const int32_t ixj = i ^ j;
        if (ixj > i) {
          const unsigned long long x = keys[i], y = keys[ixj];
          const bool desc = (i & k) == 0;
          if (desc ? (x < y) : (x > y)) {
            keys[i] = y;
            keys[ixj] = x;
          }
        }
      }
      __syncthreads();
    }
  }

  const int32_t n = nb < G.kb ? nb : G.kb;
  for (int32_t i = threadIdx.x; i < n; i += blockDim.x) {
    const unsigned long long k = keys[i];
    S.sel_ids[unit * G.kb + i] = (int32_t)(~(uint32_t)(k & 0xFFFFFFFFull));
    S.sel_scores[unit * G.kb + i] = from_orderable((uint32_t)(k >> 32));
  }
  if (threadIdx.x == 0) S.n_sel[unit] = n;
}

// ---- diff / admit / evict ----------------------------------------------------------------
//
// One CTA per unit, one thread per slot (and per selection entry):
//  hits (selected and resident) keep their slot and get stamp = step;
//  misses are ranked in selection order and the first min(C, #misses) are admitted;
//  targets are free slots by ascending slot, then unselected resident blocks by
//  (stamp asc, block id asc); each admitted block takes the target of its rank, the evicted
//  block leaves the resident map, and (block, slot) is appended to the fetch list.
__global__ void select_kernel(Geom G, LayerState S, ReqTables RT, int32_t cap_blocks, int32_t step,
                              Counters* ctr, int32_t* err) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int32_t kb = G.kb;
  unsigned long long* tkey = reinterpret_cast<unsigned long long*>(smem);  // [kb]
  int32_t* sb = reinterpret_cast<int32_t*>(tkey + kb);                     // [kb] slot -> block
  int32_t* st = sb + kb;                                                   // [kb] stamps
  int32_t* hit = st + kb;                                                  // [kb]
  int32_t* target = hit + kb;                                              // [kb]
  int32_t* warp_miss = target + kb;                                        // [32]

  const int32_t a = blockIdx.x / G.Hkv, h = blockIdx.x % G.Hkv;
  const int32_t r = RT.active[a];
  const int64_t unit = (int64_t)r * G.Hkv + h;
  const int32_t tid = threadIdx.x;
  const int32_t n_sel = S.n_sel[unit];
  const int32_t nb = (S.len[r] + G.bs - 1) / G.bs;
  int16_t* resident = S.resident + unit * G.nb_max;

  if (tid < kb) {
    sb[tid] = S.slot_block[unit * kb + tid];
    st[tid] = S.stamp[unit * kb + tid];
    hit[tid] = 0;
  }
  __syncthreads();

  int32_t b = -1;
  bool miss = false;
  if (tid < n_sel) {
    b = S.sel_ids[unit * kb + tid];
    if (b < 0 || b >= nb || b >= G.nb_max) {
      record_error(err, kErrBlockRange, -1, r, b);
      b = -1;
    } else {
      const int32_t s = resident[b];
      if (s >= kb) {
        record_error(err, kErrSlotRange, -1, r, s);
      } else if (s >= 0) {
        hit[s] = 1;
        st[s] = step;
      } else {
        miss = true;
      }
    }
  }
  // rank of each miss in selection order
  const unsigned ballot = __ballot_sync(0xffffffffu, miss);
  const int lane = tid & 31, warp = tid >> 5;
  if (lane == 0) warp_miss[warp] = __popc(ballot);
  __syncthreads();
  int32_t before = 0, n_miss = 0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
    if (w < warp) before += warp_miss[w];
    n_miss += warp_miss[w];
  }
  const int32_t rank = before + __popc(ballot & ((1u << lane) - 1u));
  const int32_t n_admit = n_miss < cap_blocks ? n_miss : cap_blocks;

  // eviction-target keys: free slots (class 0, by slot), unselected resident (class 1)
  if (tid < kb) {
    unsigned long long k;
    if (sb[tid] < 0)
      k = (unsigned long long)tid;
    else if (!hit[tid])
      k = (1ull << 63) | ((unsigned long long)((uint32_t)st[tid] ^ 0x80000000u) << 31) |
          (unsigned long long)(uint32_t)sb[tid];
    else
      k = ~0ull;  // protected: never a target
    tkey[tid] = k;
  }
  __syncthreads();
  if (tid < kb && tkey[tid] != ~0ull) {
    const unsigned long long mine = tkey[tid];
    int32_t pos = 0;
    for (int32_t o = 0; o < kb; ++o) pos += tkey[o] < mine;
    if (pos < n_admit) target[pos] = tid;
  }
  __syncthreads();

  if (miss && rank < n_admit) {
    const int32_t s = target[rank];
    const int32_t old = sb[s];
    if (old >= 0) resident[old] = -1;
    resident[b] = (int16_t)s;
    sb[s] = b;
    st[s] = step;
    S.fetch[(unit * kb + rank) * 2 + 0] = b;
    S.fetch[(unit * kb + rank) * 2 + 1] = s;
  }
  __syncthreads();
  if (tid < kb) {
    S.slot_block[unit * kb + tid] = sb[tid];
    S.stamp[unit * kb + tid] = st[tid];
  }
  if (tid == 0) {
    S.n_fetch[unit] = n_admit;
    if (n_admit > 0) atomicAdd(&ctr->fetched_blocks, (unsigned long long)n_admit);
  }
}

}  // namespace

cudaError_t launch_score_topk(const Geom& G, const LayerState& S, const ReqTables& T,
                              int32_t n_active, int32_t max_nb, const void* draft, int32_t* err,
                              cudaStream_t s) {
  if (n_active <= 0) return cudaSuccess;
  int32_t np2 = 32;
  while (np2 < max_nb) np2 <<= 1;
  const size_t smem = (size_t)2 * G.d * sizeof(float) + (size_t)np2 * sizeof(unsigned long long);
  const int grid = n_active * G.Hkv;
  cudaError_t e;
  if (G.dtype == OKV_F32) {
    e = cudaFuncSetAttribute(score_topk_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    score_topk_kernel<float><<<grid, kScoreThreads, smem, s>>>(G, S, T, np2, (const float*)draft, err);
  } else {
    e = cudaFuncSetAttribute(score_topk_kernel<__nv_bfloat16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    score_topk_kernel<__nv_bfloat16><<<grid, kScoreThreads, smem, s>>>(
        G, S, T, np2, (const __nv_bfloat16*)draft, err);
  }
  return cudaGetLastError();
}

cudaError_t launch_select(const Geom& G, const LayerState& S, const ReqTables& T, int32_t n_active,
                          int32_t cap_blocks, int32_t step, Counters* ctr, int32_t* err,
                          cudaStream_t s) {
  if (n_active <= 0) return cudaSuccess;
  const int threads = ((G.kb + 31) / 32) * 32;
  const size_t smem = (size_t)G.kb * (sizeof(unsigned long long) + 4 * sizeof(int32_t)) + 32 * sizeof(int32_t);
  select_kernel<<<n_active * G.Hkv, threads, smem, s>>>(G, S, T, cap_blocks, step, ctr, err);
  return cudaGetLastError();
}

}  // namespace okv
