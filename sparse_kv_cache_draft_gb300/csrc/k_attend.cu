// Sparse GQA decode attention over the resident slot pool.
//
// OasisKV (paperlayer.ai/abs/2608.08097v1, "4 System Design"): attention runs only over the
// KV blocks resident in HBM. For every request and query head h of KV head k:
//   o_h = sum_j softmax_j(q_h . k_j / sqrt(d)) v_j
// over every valid token j of every occupied slot of unit (layer, request, k).
//
// Two paths:
//  * attend_mma_kernel (bf16, head_dim 128, block 16, GQA group <= 8): each warp streams its
//    slots through a ring of shared-memory stages filled by 3-D TMA tensor copies (one 8 KiB
//    copy per slot, 128-byte swizzle, mbarrier completion). QK^T and PV run on the tensor
//    cores as mma.m16n8k16 with the 16 tokens of a block as M and the query heads of the
//    group as N (8 columns; heads past g are zero). The online softmax lives in registers:
//    in this orientation a lane's accumulator columns and softmax statistics belong to the
//    same two heads, so rescaling needs no data exchange.
//  * attend_simt_kernel (binary32 or any other shape): one warp per slot, lanes across head
//    dimensions, binary32 throughout.
// Both split the slots of a unit across `split` CTAs when there are too few units to fill the
// GPU; a combine kernel then merges the partial (max, sum, output) triples.
#include <cuda_bf16.h>
#include <stdio.h>
#include <stdlib.h>

#include <mutex>

#include "okv_internal.h"
#include "ptx.cuh"

namespace okv {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMmaD = 128;
constexpr int kSlotBytes = 8192;  // K and V of 16 tokens x 128 dims, bf16
constexpr int kMaxG = 8;

__device__ __forceinline__ void mma_bf16(float* c, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
      " {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Token held by M-row r (0..15) of the QK^T tile (and by k-slot r of the PV tile). The order is
// chosen so that every 16-byte shared-memory read of the swizzled slot image is conflict-free.
__device__ __forceinline__ int token_of_row(int r) {
  const int lo = r & 7;
  const int t = (lo & 1) ? 4 + (((lo >> 1) + 1) & 3) : (lo >> 1);
  return (r & 8) + t;
}
// Byte offset in the smem slot image of 16-byte chunk `c8` (0..7) of half `hf` of row `row`
// (rows 0..15 = K tokens, 16..31 = V tokens, 256 bytes each), after the 128-byte TMA swizzle
// (16-byte chunk index XOR 128-byte line index mod 8; the stage is 1024-byte aligned).
__device__ __forceinline__ uint32_t swz(int row, int hf, int c8) {
  return (uint32_t)(row * 256 + hf * 128 + ((c8 ^ ((2 * row + hf) & 7)) << 4));
}

// Collect the occupied slots of [s_lo, s_hi) of one unit as (slot << 8 | valid tokens).
__device__ int32_t build_items(const Geom& G, const int32_t* slot_block, int32_t s_lo, int32_t s_hi,
                               int32_t len, int32_t r, int32_t* items, int32_t* scratch,
                               int32_t* err) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  int32_t base = 0;
  for (int32_t s0 = s_lo; s0 < s_hi; s0 += blockDim.x) {
    const int32_t s = s0 + threadIdx.x;
    int32_t item = -1;
    if (s < s_hi) {
      const int32_t b = slot_block[s];
      if (b >= 0) {
        // tokens of block b within the context, in 64 bits: b * bs may pass 2^31 for a block id
        // that fails the check
        const int64_t rem = (int64_t)len - (int64_t)b * G.bs;
        if (rem <= 0 || b >= G.nb_max)
          record_error(err, kErrBlockRange, -2, r, b);
        else
          item = (s << 8) | (int32_t)(rem < G.bs ? rem : G.bs);
      }
    }
    const unsigned ballot = __ballot_sync(0xffffffffu, item >= 0);
    if (lane == 0) scratch[warp] = __popc(ballot);
    __syncthreads();
    int32_t before = 0, total = 0;
    for (int w = 0; w < nwarps; ++w) {
      if (w < warp) before += scratch[w];
      total += scratch[w];
    }
    if (item >= 0) items[base + before + __popc(ballot & ((1u << lane) - 1u))] = item;
    base += total;
    __syncthreads();
  }
  return base;
}

// The rows one unit's attention computes: rows 0..g-1 are the group's query heads of q; with a
// draft query (look-ahead attention) rows g..2g-1 are the same heads of the draft, attending
// over the same resident K and V.
template <typename T>
struct Rows {
  const T* q;
  const T* dq;  // NULL: no draft rows
  T* out;
  T* dout;
  int32_t n;    // g or 2g
  __device__ __forceinline__ const T* in(const Geom& G, int32_t r, int32_t h, int32_t j) const {
    return (j < G.g ? q : dq) + ((int64_t)r * G.Hq + h * G.g + (j < G.g ? j : j - G.g)) * G.d;
  }
  __device__ __forceinline__ T* dst(const Geom& G, int32_t r, int32_t h, int32_t j) const {
    return (j < G.g ? out : dout) + ((int64_t)r * G.Hq + h * G.g + (j < G.g ? j : j - G.g)) * G.d;
  }
};

__device__ __forceinline__ void store_out(float* p, float x) { *p = x; }
__device__ __forceinline__ void store_out(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// The split partials of unit `ua` are complete when the last of its `split` CTAs arrives; that
// CTA merges the (max, sum, o) triples and writes the output. Returns false in the other CTAs.
template <typename T>
__device__ bool finish_split(const Geom& G, int32_t r, int32_t h, int32_t ua, int32_t split,
                             const float* __restrict__ partials, int32_t* __restrict__ arrivals,
                             const Rows<T>& rows) {
  __shared__ int32_t last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    last = atomicAdd(&arrivals[ua], 1) == split - 1;
    if (last) arrivals[ua] = 0;
  }
  __syncthreads();
  if (!last) return false;
  __threadfence();
  const int32_t nr = rows.n;
  const int64_t stride = (int64_t)nr * (G.d + 2);
  const float* base = partials + (int64_t)ua * split * stride;
  for (int32_t idx = threadIdx.x; idx < nr * G.d; idx += blockDim.x) {
    const int head = idx / G.d, dim = idx % G.d;
    float M = -INFINITY;
    for (int p = 0; p < split; ++p) M = fmaxf(M, __ldcg(base + p * stride + nr * G.d + head));
    float acc = 0.f, l = 0.f;
    if (M != -INFINITY) {
      for (int p = 0; p < split; ++p) {
        const float f = exp2f(__ldcg(base + p * stride + nr * G.d + head) - M);
        acc += f * __ldcg(base + p * stride + head * G.d + dim);
        l += f * __ldcg(base + p * stride + nr * G.d + nr + head);
      }
    }
    store_out(rows.dst(G, r, h, head) + dim, l > 0.f ? acc / l : 0.f);
  }
  return true;
}

// ---- tensor-core path ------------------------------------------------------------------------

template <int NW, int NS>
struct MmaSmem {
  static constexpr int kRing = NW * NS * kSlotBytes;
  static constexpr int kBars = NW * NS * 8;
  static size_t bytes(int kb) { return 1024 + kRing + kBars + (size_t)(kb + 64) * 4; }
};

template <int NW, int NS>
__global__ void __launch_bounds__(NW * 32)
attend_mma_kernel(Geom G, LayerState S, ReqTables RT, const __grid_constant__ CUtensorMap pool_map,
                  int64_t row_base, int32_t split, const Rows<__nv_bfloat16> rows,
                  float* __restrict__ partials, int32_t* __restrict__ arrivals, Counters* ctr,
                  int32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring + MmaSmem<NW, NS>::kRing);
  int32_t* items = reinterpret_cast<int32_t*>(bars + NW * NS);
  int32_t* scratch = items + G.kb;

  const int32_t ua = blockIdx.x / split, part = blockIdx.x % split;
  const int32_t a = ua / G.Hkv, h = ua % G.Hkv;
  const int32_t r = RT.active[a];
  const int64_t unit = (int64_t)r * G.Hkv + h;
  const int32_t len = S.len[r];
  const int32_t chunk = (G.kb + split - 1) / split;
  const int32_t s_lo = part * chunk, s_hi = min(G.kb, s_lo + chunk);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gi = lane >> 2, ti = lane & 3;

  if (threadIdx.x < NW * NS) mbar_init(smem_u32(&bars[threadIdx.x]), 1);
  fence_mbar_init();
  const int32_t n_items = build_items(G, S.slot_block + unit * G.kb, s_lo, s_hi, len, r, items,
                                      scratch, err);
  __syncthreads();  // barriers initialised and the item list complete for every warp
  if (threadIdx.x == 0 && n_items > 0) atomicAdd(&ctr->attended_slots, (unsigned long long)n_items);

  const int32_t my_count = n_items > warp ? (n_items - warp + NW - 1) / NW : 0;
  const uint32_t ring_w = smem_u32(ring + warp * NS * kSlotBytes);
  const uint32_t bar_w = smem_u32(&bars[warp * NS]);
  const int64_t unit_row = row_base + unit * G.kb * 32;

  if (lane == 0) {
    for (int st = 0; st < NS && st < my_count; ++st) {
      const int32_t slot = items[warp + st * NW] >> 8;
      mbar_expect_tx(bar_w + st * 8, kSlotBytes);
      tma_load_3d(ring_w + st * kSlotBytes, &pool_map, bar_w + st * 8, 0, 0,
                  (int32_t)(unit_row + (int64_t)slot * 32));
    }
  }

  // query fragments (B operand of QK^T): head gi of the group, dims in the permuted k order
  uint32_t qb[8][2];
  {
    const bool real = gi < rows.n;
    const __nv_bfloat16* qh = rows.in(G, r, h, real ? gi : 0);
#pragma unroll
    for (int hf = 0; hf < 2; ++hf)
#pragma unroll
      for (int s = 0; s < 2; ++s)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int base = 64 * hf + 8 * ((ti & 1) + 4 * (ti >> 1) + 2 * s) + 4 * e;
          uint2 v = real ? *reinterpret_cast<const uint2*>(qh + base) : make_uint2(0, 0);
          qb[4 * hf + 2 * s + e][0] = v.x;
          qb[4 * hf + 2 * s + e][1] = v.y;
        }
  }

  const float scale = kLog2e * rsqrtf((float)kMmaD);
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float o[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  const int rowA = token_of_row(gi), rowB = 8 + rowA;
  const int tv0 = token_of_row(2 * ti), tv1 = token_of_row(2 * ti + 1);
  bool ok = true;
  int32_t issued = my_count < NS ? my_count : NS;
  int32_t consumed = 0;

  for (int32_t k = 0; k < my_count; ++k) {
    const int st = k % NS;
    const uint32_t bar = bar_w + st * 8;
    if (!mbar_wait_bounded(bar, (uint32_t)((k / NS) & 1))) {
      if (lane == 0) record_error(err, kErrTimeout, -3, r, k);
      ok = false;
      consumed = k;
      break;
    }
    const uint32_t sb = ring_w + st * kSlotBytes;
    const int32_t nv = items[warp + k * NW] & 0xFF;

    // S^T = K Q^T : 16 tokens x 8 heads
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int hf = 0; hf < 2; ++hf)
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        const int c8 = (ti & 1) + 4 * (ti >> 1) + 2 * s;
        const uint4 xa = lds128(sb + swz(rowA, hf, c8));
        const uint4 xb = lds128(sb + swz(rowB, hf, c8));
        mma_bf16(sc, xa.x, xb.x, xa.y, xb.y, qb[4 * hf + 2 * s][0], qb[4 * hf + 2 * s][1]);
        mma_bf16(sc, xa.z, xb.z, xa.w, xb.w, qb[4 * hf + 2 * s + 1][0], qb[4 * hf + 2 * s + 1][1]);
      }
    // scale to log2 units, mask tokens past the block's valid count
    sc[0] = rowA < nv ? sc[0] * scale : -INFINITY;
    sc[1] = rowA < nv ? sc[1] * scale : -INFINITY;
    sc[2] = rowB < nv ? sc[2] * scale : -INFINITY;
    sc[3] = rowB < nv ? sc[3] * scale : -INFINITY;
    float mx0 = fmaxf(sc[0], sc[2]), mx1 = fmaxf(sc[1], sc[3]);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);
    const float al0 = exp2f(m_run[0] - mn0), al1 = exp2f(m_run[1] - mn1);
    m_run[0] = mn0;
    m_run[1] = mn1;
    const float p0 = exp2f(sc[0] - mn0), p1 = exp2f(sc[1] - mn1);
    const float p2 = exp2f(sc[2] - mn0), p3 = exp2f(sc[3] - mn1);
    l_run[0] = l_run[0] * al0 + p0 + p2;
    l_run[1] = l_run[1] * al1 + p1 + p3;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      o[i][0] *= al0;
      o[i][1] *= al1;
      o[i][2] *= al0;
      o[i][3] *= al1;
    }
    // P as the B operand of PV: transpose the (token, head) bf16 pairs
    const uint32_t pb0 = movmatrix_trans(pack_bf16x2(p0, p1));
    const uint32_t pb1 = movmatrix_trans(pack_bf16x2(p2, p3));

    // O^T += V^T P : 128 dims x 8 heads, two rounds of 64 dims
#pragma unroll
    for (int om = 0; om < 2; ++om) {
      const uint4 x0 = lds128(sb + swz(16 + tv0, om, gi));
      const uint4 x1 = lds128(sb + swz(16 + tv1, om, gi));
      const uint4 x2 = lds128(sb + swz(24 + tv0, om, gi));
      const uint4 x3 = lds128(sb + swz(24 + tv1, om, gi));
      const uint32_t w0[4] = {x0.x, x0.y, x0.z, x0.w}, w1[4] = {x1.x, x1.y, x1.z, x1.w};
      const uint32_t w2[4] = {x2.x, x2.y, x2.z, x2.w}, w3[4] = {x3.x, x3.y, x3.z, x3.w};
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        mma_bf16(o[om * 4 + qq], __byte_perm(w0[qq], w1[qq], 0x5410), __byte_perm(w0[qq], w1[qq], 0x7632),
                 __byte_perm(w2[qq], w3[qq], 0x5410), __byte_perm(w2[qq], w3[qq], 0x7632), pb0, pb1);
      }
    }

    __syncwarp();
    if (lane == 0 && k + NS < my_count) {
      const int32_t slot = items[warp + (k + NS) * NW] >> 8;
      fence_proxy_async();
      mbar_expect_tx(bar, kSlotBytes);
      tma_load_3d(sb, &pool_map, bar, 0, 0, (int32_t)(unit_row + (int64_t)slot * 32));
      ++issued;
    }
    issued = __shfl_sync(0xffffffffu, issued, 0);
  }
  if (!ok) {
    // drain this warp's copies still in flight before the ring is reused (bounded)
    for (int32_t k = consumed; k < issued; ++k) mbar_wait_bounded(bar_w + (k % NS) * 8, (uint32_t)((k / NS) & 1));
  }
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], off);
    l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], off);
  }
  __syncthreads();  // every stage consumed: the ring becomes the combine buffer

  float* ow = reinterpret_cast<float*>(ring);   // [NW][8 heads][128]
  float* mw = ow + NW * 8 * kMmaD;              // [NW][8]
  float* lw = mw + NW * 8;                      // [NW][8]
  {
    float* mine = ow + warp * 8 * kMmaD;
#pragma unroll
    for (int om = 0; om < 2; ++om)
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        const int dim = 8 * (gi + 8 * om) + 2 * qq;
        mine[(2 * ti) * kMmaD + dim] = o[om * 4 + qq][0];
        mine[(2 * ti + 1) * kMmaD + dim] = o[om * 4 + qq][1];
        mine[(2 * ti) * kMmaD + dim + 1] = o[om * 4 + qq][2];
        mine[(2 * ti + 1) * kMmaD + dim + 1] = o[om * 4 + qq][3];
      }
    if (gi == 0) {
      mw[warp * 8 + 2 * ti] = m_run[0];
      mw[warp * 8 + 2 * ti + 1] = m_run[1];
      lw[warp * 8 + 2 * ti] = l_run[0];
      lw[warp * 8 + 2 * ti + 1] = l_run[1];
    }
  }
  __syncthreads();
  const int32_t nr = rows.n;
  const int32_t nval = nr * kMmaD;
  for (int32_t idx = threadIdx.x; idx < nval; idx += blockDim.x) {
    const int head = idx / kMmaD, dim = idx % kMmaD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, mw[w * 8 + head]);
    float acc = 0.f, l = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float f = exp2f(mw[w * 8 + head] - M);
        acc += f * ow[(w * 8 + head) * kMmaD + dim];
        l += f * lw[w * 8 + head];
      }
    }
    if (split == 1) {
      rows.dst(G, r, h, head)[dim] = __float2bfloat16_rn(l > 0.f ? acc / l : 0.f);
    } else {
      const int64_t pu = (int64_t)ua * split + part;
      float* po = partials + pu * nr * (kMmaD + 2);
      po[head * kMmaD + dim] = acc;
      if (dim == 0) {
        po[nr * kMmaD + head] = M;
        po[nr * kMmaD + nr + head] = l;
      }
    }
  }
  if (split > 1) finish_split(G, r, h, ua, split, partials, arrivals, rows);
}

// ---- CUDA-core path ---------------------------------------------------------------------------

__device__ __forceinline__ float ld_f(const float* p) { return *p; }
__device__ __forceinline__ float ld_f(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st_f(float* p, float x) { *p = x; }
__device__ __forceinline__ void st_f(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

constexpr int kSimtWarps = 4;
constexpr int kSimtMaxDv = 8;  // head_dim <= 256

template <typename T>
__global__ void __launch_bounds__(kSimtWarps * 32)
attend_simt_kernel(Geom G, LayerState S, ReqTables RT, int32_t split, const Rows<T> rows,
                   float* __restrict__ partials, int32_t* __restrict__ arrivals, Counters* ctr,
                   int32_t* err) {
  extern __shared__ __align__(16) uint8_t smem[];
  int32_t* items = reinterpret_cast<int32_t*>(smem);   // [kb]
  int32_t* scratch = items + G.kb;                     // [32]
  float* ow = reinterpret_cast<float*>(scratch + 32);  // [NW][rows][d]
  const int32_t nr = rows.n;
  float* mw = ow + kSimtWarps * nr * G.d;              // [NW][rows]
  float* lw = mw + kSimtWarps * nr;                    // [NW][rows]

  const int32_t ua = blockIdx.x / split, part = blockIdx.x % split;
  const int32_t a = ua / G.Hkv, h = ua % G.Hkv;
  const int32_t r = RT.active[a];
  const int64_t unit = (int64_t)r * G.Hkv + h;
  const int32_t len = S.len[r];
  const int32_t chunk = (G.kb + split - 1) / split;
  const int32_t s_lo = part * chunk, s_hi = min(G.kb, s_lo + chunk);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int32_t n_items = build_items(G, S.slot_block + unit * G.kb, s_lo, s_hi, len, r, items, scratch, err);
  __syncthreads();
  if (threadIdx.x == 0 && n_items > 0) atomicAdd(&ctr->attended_slots, (unsigned long long)n_items);

  const int dv = G.d / 32;
  const float scale = kLog2e / sqrtf((float)G.d);
  float qv[kMaxG][kSimtMaxDv], ov[kMaxG][kSimtMaxDv], m[kMaxG], l[kMaxG];
#pragma unroll
  for (int j = 0; j < kMaxG; ++j) {
    m[j] = -INFINITY;
    l[j] = 0.f;
#pragma unroll
    for (int i = 0; i < kSimtMaxDv; ++i) {
      ov[j][i] = 0.f;
      qv[j][i] = (j < nr && i < dv) ? ld_f(rows.in(G, r, h, j) + lane + 32 * i) * scale : 0.f;
    }
  }
  for (int32_t it = warp; it < n_items; it += kSimtWarps) {
    const int32_t slot = items[it] >> 8, nv = items[it] & 0xFF;
    const T* kp = reinterpret_cast<const T*>(S.pool + (unit * G.kb + slot) * G.block_bytes);
    const T* vp = kp + (int64_t)G.bs * G.d;
    for (int32_t t = 0; t < nv; ++t) {
      float kx[kSimtMaxDv], vx[kSimtMaxDv];
#pragma unroll
      for (int i = 0; i < kSimtMaxDv; ++i) {
        kx[i] = i < dv ? ld_f(kp + (int64_t)t * G.d + lane + 32 * i) : 0.f;
        vx[i] = i < dv ? ld_f(vp + (int64_t)t * G.d + lane + 32 * i) : 0.f;
      }
#pragma unroll
      for (int j = 0; j < kMaxG; ++j) {
        if (j >= nr) break;
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < kSimtMaxDv; ++i) s = fmaf(qv[j][i], kx[i], s);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        const float mn = fmaxf(m[j], s);
        const float al = exp2f(m[j] - mn), p = exp2f(s - mn);
        m[j] = mn;
        l[j] = l[j] * al + p;
#pragma unroll
        for (int i = 0; i < kSimtMaxDv; ++i) ov[j][i] = ov[j][i] * al + p * vx[i];
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kMaxG; ++j) {
    if (j >= nr) break;
#pragma unroll
    for (int i = 0; i < kSimtMaxDv; ++i)
      if (i < dv) ow[(warp * nr + j) * G.d + lane + 32 * i] = ov[j][i];
    if (lane == 0) {
      mw[warp * nr + j] = m[j];
      lw[warp * nr + j] = l[j];
    }
  }
  __syncthreads();
  for (int32_t idx = threadIdx.x; idx < nr * G.d; idx += blockDim.x) {
    const int head = idx / G.d, dim = idx % G.d;
    float M = -INFINITY;
    for (int w = 0; w < kSimtWarps; ++w) M = fmaxf(M, mw[w * nr + head]);
    float acc = 0.f, ls = 0.f;
    if (M != -INFINITY) {
      for (int w = 0; w < kSimtWarps; ++w) {
        const float f = exp2f(mw[w * nr + head] - M);
        acc += f * ow[(w * nr + head) * G.d + dim];
        ls += f * lw[w * nr + head];
      }
    }
    if (split == 1) {
      st_f(rows.dst(G, r, h, head) + dim, ls > 0.f ? acc / ls : 0.f);
    } else {
      const int64_t pu = (int64_t)ua * split + part;
      float* po = partials + pu * nr * (G.d + 2);
      po[head * G.d + dim] = acc;
      if (dim == 0) {
        po[nr * G.d + head] = M;
        po[nr * G.d + nr + head] = ls;
      }
    }
  }
  if (split > 1) finish_split(G, r, h, ua, split, partials, arrivals, rows);
}

// Tile shape of the tensor-core path, chosen at first use (OKV_ATTEND_TILE=<warps>x<stages>).
struct MmaShape {
  int nw, ns;
};

MmaShape mma_shape() {
  static MmaShape sh = [] {
    MmaShape s{4, 3};
    if (const char* e = getenv("OKV_ATTEND_TILE")) {
      int w = 0, st = 0;
      if (sscanf(e, "%dx%d", &w, &st) == 2) {
        if ((w == 4 && (st == 2 || st == 3 || st == 4)) || (w == 8 && (st == 2 || st == 3))) s = {w, st};
      }
    }
    return s;
  }();
  return sh;
}

bool use_mma(const Geom& G) {
  return G.dtype == OKV_BF16 && G.d == kMmaD && G.bs == 16 && G.g <= kMaxG && G.kb <= 1024;
}

int32_t pick_split(const Geom& G, int32_t n_active, int ctas_per_sm, int warps) {
  const int32_t units = n_active * G.Hkv;
  if (const char* e = getenv("OKV_ATTEND_SPLIT")) {
    const int v = atoi(e);
    if (v >= 1 && v <= G.kb) return v;
  }
  int sms = 152;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // Fewer units than SMs: split until every SM has a CTA. From one to four units per SM: one CTA
  // per unit (a split's partials, merge and shorter CTAs cost more than its waves save: 48.8
  // against 77 us per launch alone at 256 units, and +22% decode tok/s with two staging lanes
  // at the 32B-class shapes). Beyond that, about four waves: at 1024 units (Qwen3-8B shapes,
  // batch 128) a split of 2 measured 5% more tok/s in the step than one CTA per unit, although
  // slower alone, the step there being bound by the host link that a faster attention slows.
  int32_t split;
  if (units < sms)
    split = (sms + units - 1) / units;
  else if (units < 4 * sms)
    split = 1;
  else {
    const int32_t target = sms * ctas_per_sm * 4;  // about four waves
    split = units >= target ? 1 : (target + units - 1) / units;
  }
  const int32_t max_split = G.kb / (2 * warps) > 0 ? G.kb / (2 * warps) : 1;
  return split < max_split ? split : max_split;
}

template <int NW, int NS>
cudaError_t run_mma(const Geom& G, const LayerState& S, const ReqTables& T, int32_t n_active,
                    int32_t layer, const Rows<__nv_bfloat16>& rows, const CUtensorMap* map, void* partials,
                    int32_t* arrivals, Counters* ctr, int32_t* err, cudaStream_t s, int32_t split) {
  const size_t smem = MmaSmem<NW, NS>::bytes(G.kb);
  cudaError_t e = cudaFuncSetAttribute(attend_mma_kernel<NW, NS>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // the pool tensor map spans every layer: rows of 256 bytes, 32 rows (K then V) per slot
  const int64_t row_base = (int64_t)layer * G.R * G.Hkv * G.kb * 32;
  attend_mma_kernel<NW, NS><<<n_active * G.Hkv * split, NW * 32, smem, s>>>(
      G, S, T, *map, row_base, split, rows, (float*)partials, arrivals, ctr, err);
  return cudaGetLastError();
}

// The largest split whose partials ([units x split][rows][d + 2] binary32) fit `ws_bytes`, at
// most `want` (the split is chosen at each launch, e.g. from OKV_ATTEND_SPLIT, while the
// workspace was sized when it was allocated).
int32_t fit_split(const Geom& G, int32_t n_active, int32_t nrows, int32_t want, size_t ws_bytes) {
  const size_t per = (size_t)n_active * G.Hkv * nrows * (G.d + 2) * sizeof(float);
  int32_t split = want;
  while (split > 1 && per * (size_t)split > ws_bytes) --split;
  return split;
}

// One attention launch over `nrows` rows (the group's heads of q, then, if dq is given, of dq).
cudaError_t launch_rows(const Geom& G, const LayerState& S, const ReqTables& T, int32_t n_active,
                        int32_t layer, const void* q, const void* dq, void* out, void* dout, int32_t nrows,
                        const CUtensorMap* pool_map, void* partials, size_t ws_bytes, int32_t* arrivals,
                        Counters* ctr, int32_t* err, cudaStream_t s, int32_t* used_split) {
  cudaError_t e;
  int32_t split;
  if (use_mma(G)) {
    const Rows<__nv_bfloat16> rows{(const __nv_bfloat16*)q, (const __nv_bfloat16*)dq, (__nv_bfloat16*)out,
                                   (__nv_bfloat16*)dout, nrows};
    const MmaShape sh = mma_shape();
    split = fit_split(G, n_active, nrows, pick_split(G, n_active, 2, sh.nw), ws_bytes);
    if (sh.nw == 8 && sh.ns == 2)
      e = run_mma<8, 2>(G, S, T, n_active, layer, rows, pool_map, partials, arrivals, ctr, err, s, split);
    else if (sh.nw == 8 && sh.ns == 3)
      e = run_mma<8, 3>(G, S, T, n_active, layer, rows, pool_map, partials, arrivals, ctr, err, s, split);
    else if (sh.ns == 2)
      e = run_mma<4, 2>(G, S, T, n_active, layer, rows, pool_map, partials, arrivals, ctr, err, s, split);
    else if (sh.ns == 4)
      e = run_mma<4, 4>(G, S, T, n_active, layer, rows, pool_map, partials, arrivals, ctr, err, s, split);
    else
      e = run_mma<4, 3>(G, S, T, n_active, layer, rows, pool_map, partials, arrivals, ctr, err, s, split);
  } else {
    split = fit_split(G, n_active, nrows, pick_split(G, n_active, 4, kSimtWarps), ws_bytes);
    const size_t smem = (size_t)(G.kb + 32) * 4 + (size_t)kSimtWarps * nrows * (G.d + 2) * 4;
    const int grid = n_active * G.Hkv * split;
    if (G.dtype == OKV_F32) {
      const Rows<float> rows{(const float*)q, (const float*)dq, (float*)out, (float*)dout, nrows};
      e = cudaFuncSetAttribute(attend_simt_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess)
        attend_simt_kernel<float><<<grid, kSimtWarps * 32, smem, s>>>(G, S, T, split, rows, (float*)partials,
                                                                      arrivals, ctr, err);
    } else {
      const Rows<__nv_bfloat16> rows{(const __nv_bfloat16*)q, (const __nv_bfloat16*)dq, (__nv_bfloat16*)out,
                                     (__nv_bfloat16*)dout, nrows};
      e = cudaFuncSetAttribute(attend_simt_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess)
        attend_simt_kernel<__nv_bfloat16><<<grid, kSimtWarps * 32, smem, s>>>(G, S, T, split, rows,
                                                                              (float*)partials, arrivals, ctr, err);
    }
    if (e == cudaSuccess) e = cudaGetLastError();
  }
  *used_split = split;
  return e;
}

}  // namespace

bool attend_uses_tensor_cores(const Geom& G) { return use_mma(G); }

size_t attend_workspace_bytes(const Geom& G, int32_t n_active) {
  const int warps = use_mma(G) ? mma_shape().nw : kSimtWarps;
  const int32_t n = n_active > 0 ? n_active : 1;
  const int32_t split = pick_split(G, n, use_mma(G) ? 2 : 4, warps);
  const int32_t rows = 2 * G.g <= kMaxG ? 2 * G.g : G.g;  // room for look-ahead rows
  return (size_t)n * G.Hkv * split * rows * (G.d + 2) * sizeof(float);
}

cudaError_t launch_attend(const Geom& G, const LayerState& S, const ReqTables& T, int32_t n_active,
                          int32_t layer, const void* q, void* out, const void* dq, void* dout,
                          const CUtensorMap* pool_map, void* partials, size_t ws_bytes, int32_t* arrivals,
                          Counters* ctr, int32_t* err, cudaStream_t s, int* n_launches, int* used_split) {
  *n_launches = 0;
  *used_split = 0;
  if (n_active <= 0) return cudaSuccess;
  cudaError_t e;
  if (!dq || 2 * G.g <= kMaxG) {
    // one pass: the draft heads (if any) ride in the MMA's spare columns next to the query heads
    e = launch_rows(G, S, T, n_active, layer, q, dq, out, dout, dq ? 2 * G.g : G.g, pool_map, partials,
                    ws_bytes, arrivals, ctr, err, s, used_split);
    if (e != cudaSuccess) return e;
    *n_launches = 1;
  } else {
    // a group too wide for both: two passes over the resident set
    e = launch_rows(G, S, T, n_active, layer, q, nullptr, out, nullptr, G.g, pool_map, partials, ws_bytes,
                    arrivals, ctr, err, s, used_split);
    if (e != cudaSuccess) return e;
    e = launch_rows(G, S, T, n_active, layer, dq, nullptr, dout, nullptr, G.g, pool_map, partials, ws_bytes,
                    arrivals, ctr, err, s, used_split);
    if (e != cudaSuccess) return e;
    *n_launches = 2;
  }
  return cudaSuccess;
}

}  // namespace okv

// ---- allocation-free variant ------------------------------------------------------------------
//
// For callers that cannot allocate device memory, okv_attend_static runs the same attention
// kernels over caller-provided inputs and outputs. Its only workspace (the split partials,
// the request-id list and the error word / counters the kernels write) lives in one fixed,
// file-scope device array that every GPU loading this library holds until the process exits.

namespace {

constexpr size_t kStaticScratchBytes = (size_t)16 << 20;  // 16 MiB
constexpr int32_t kStaticMaxRequests = 16384;
constexpr size_t kStaticIdsOffset = 256;                  // [0, 256): error word, counters
constexpr int32_t kStaticMaxUnits = kStaticMaxRequests * 8;
constexpr size_t kStaticArrivalsOffset = kStaticIdsOffset + (size_t)kStaticMaxRequests * 4;
constexpr size_t kStaticPartialsOffset = kStaticArrivalsOffset + (size_t)kStaticMaxUnits * 4;

static __device__ __align__(256) unsigned char okv_static_scratch[kStaticScratchBytes];

__global__ void static_init_kernel(int32_t* ids, int32_t n, int32_t* err, okv::Counters* ctr) {
  const int32_t i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) ids[i] = i;
  if (i < 4) err[i] = 0;
  if (i == 0) {
    ctr->fetched_blocks = 0;
    ctr->attended_slots = 0;
  }
}

void* driver_entry(const char* name) {
  void* f = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return f;
}

std::mutex g_static_mu;
struct StaticDevice {
  unsigned long long ctx_id;  // the CUDA context the array was set up in (0: not yet)
  void* base;                 // device address of okv_static_scratch in that context
};
StaticDevice g_static[256] = {};  // per device ordinal

// With the device current: resolve the array's device address (host code cannot use the symbol
// itself) and, the first time in each CUDA context of the device, fill the constant part (the
// request ids 0..max-1). A context that was reset and created again (cudaDeviceReset) gets a new
// context id, so its array is set up again.
cudaError_t static_scratch(void** base) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 256) return cudaErrorInvalidDevice;
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, okv_static_scratch);  // also makes the device's context current
  if (e != cudaSuccess) return e;
  // driver calls through entry points, so the library keeps no link-time dependency on libcuda
  typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
  typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);
  static const CtxGetCurrentFn get_current = reinterpret_cast<CtxGetCurrentFn>(driver_entry("cuCtxGetCurrent"));
  static const CtxGetIdFn get_id = reinterpret_cast<CtxGetIdFn>(driver_entry("cuCtxGetId"));
  CUcontext cu = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&cu) != CUDA_SUCCESS || !cu || get_id(cu, &id) != CUDA_SUCCESS)
    return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (g_static[dev].ctx_id != id || g_static[dev].base != p) {
    unsigned char* b = static_cast<unsigned char*>(p);
    static_init_kernel<<<(kStaticMaxRequests + 255) / 256, 256>>>(
        reinterpret_cast<int32_t*>(b + kStaticIdsOffset), kStaticMaxRequests, reinterpret_cast<int32_t*>(b),
        reinterpret_cast<okv::Counters*>(b + 16));
    e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    g_static[dev].ctx_id = id;
    g_static[dev].base = p;
  }
  *base = p;
  return cudaSuccess;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = reinterpret_cast<EncodeTiledFn>(driver_entry("cuTensorMapEncodeTiled"));
  return fn;
}

}  // namespace

extern "C" okv_status okv_attend_static(int32_t n_requests, int32_t q_heads, int32_t kv_heads,
                                        int32_t head_dim, int32_t block_size, int32_t slots,
                                        int32_t dtype, const void* pool, const int32_t* slot_block,
                                        const int32_t* lengths, const void* q, void* out,
                                        void* stream) {
  using namespace okv;
  if (n_requests <= 0 || n_requests > kStaticMaxRequests) return OKV_EINVAL;
  if ((int64_t)n_requests * kv_heads > kStaticMaxUnits) return OKV_EINVAL;
  if (q_heads <= 0 || kv_heads <= 0 || q_heads % kv_heads || q_heads / kv_heads > kMaxG) return OKV_EINVAL;
  if (head_dim <= 0 || head_dim % 32 || head_dim > 256 || block_size <= 0 || block_size > 64) return OKV_EINVAL;
  if (slots <= 0 || slots > 1024 || (dtype != OKV_F32 && dtype != OKV_BF16)) return OKV_EINVAL;
  if (!pool || !slot_block || !lengths || !q || !out) return OKV_EINVAL;
  Geom G{};
  G.L = 1;
  G.Hq = q_heads;
  G.Hkv = kv_heads;
  G.g = q_heads / kv_heads;
  G.d = head_dim;
  G.bs = block_size;
  G.kb = slots;
  G.R = n_requests;
  G.nb_max = (int32_t)(INT32_MAX / block_size);  // block ids are checked against each request's length
  G.dtype = dtype;
  G.elem = dtype == OKV_F32 ? 4 : 2;
  G.block_bytes = (int64_t)2 * block_size * head_dim * G.elem;
  if ((block_size * head_dim * G.elem) % 16) return OKV_EINVAL;
  // the split partials must fit in the fixed workspace
  if (attend_workspace_bytes(G, n_requests) > kStaticScratchBytes - kStaticPartialsOffset) return OKV_EINVAL;

  // the kernels run on `stream` with the array's address on the current device: both must agree
  if (stream) {
    int dev = 0, sdev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaStreamGetDevice((cudaStream_t)stream, &sdev) != cudaSuccess)
      return OKV_ECUDA;
    if (sdev != dev) return OKV_EINVAL;
  }
  void* base = nullptr;
  if (static_scratch(&base) != cudaSuccess) return OKV_ECUDA;
  unsigned char* b = static_cast<unsigned char*>(base);
  LayerState S{};
  S.pool = static_cast<uint8_t*>(const_cast<void*>(pool));
  S.slot_block = const_cast<int32_t*>(slot_block);
  S.len = const_cast<int32_t*>(lengths);
  ReqTables T{};
  T.active = reinterpret_cast<const int32_t*>(b + kStaticIdsOffset);
  CUtensorMap map;
  const CUtensorMap* pmap = nullptr;
  if (use_mma(G)) {
    const uint64_t rows = (uint64_t)n_requests * kv_heads * slots * 32;
    EncodeTiledFn fn = encode_fn();
    if (!fn || rows >= (1ull << 31) || (reinterpret_cast<uintptr_t>(pool) & 15)) return OKV_EINVAL;
    const cuuint64_t dims[3] = {64, 2, rows};
    const cuuint64_t strides[2] = {128, 256};
    const cuuint32_t box[3] = {64, 2, 32};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (fn(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(pool), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return OKV_EINVAL;
    pmap = &map;
  }
  // the split arrival counters must start at zero (the kernel leaves them at zero, but a call
  // may follow any earlier one), and the error word starts clear for each call: clear both on
  // the stream first
  int32_t* arrivals = reinterpret_cast<int32_t*>(b + kStaticArrivalsOffset);
  if (cudaMemsetAsync(arrivals, 0, (size_t)n_requests * kv_heads * 4, (cudaStream_t)stream) != cudaSuccess ||
      cudaMemsetAsync(b, 0, 16, (cudaStream_t)stream) != cudaSuccess)
    return OKV_ECUDA;
  int n_launch = 0, split = 0;
  cudaError_t e = launch_attend(G, S, T, n_requests, 0, q, out, nullptr, nullptr, pmap, b + kStaticPartialsOffset,
                                kStaticScratchBytes - kStaticPartialsOffset, arrivals,
                                reinterpret_cast<Counters*>(b + 16), reinterpret_cast<int32_t*>(b),
                                (cudaStream_t)stream, &n_launch, &split);
  return e == cudaSuccess ? OKV_OK : OKV_ECUDA;
}
