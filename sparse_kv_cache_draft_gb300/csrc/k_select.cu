// Lookahead block scoring, per-head top-K and KV selection (diff / admit / evict).
//
// OasisKV (paperlayer.ai/abs/2608.08097v1, "4 System Design"): the draft query scans the
// per-block min/max key summaries to rank blocks; each layer's background chain is top-K
// prediction, then KV selection, which moves at most C blocks per KV head, keeps resident
// predicted blocks and pairs admitted blocks with least-recently-selected eviction targets.
#include <cuda_bf16.h>

#include "okv_internal.h"
#include "ptx.cuh"

namespace okv {
namespace {

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

// ---- block-wide helpers -------------------------------------------------------------------

// Exclusive prefix count of `flag` over the thread order of one pass of the block (index
// base + threadIdx.x); returns this thread's rank and sets *total to the pass's count.
__device__ __forceinline__ int32_t block_rank(bool flag, int32_t* scratch, int32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const unsigned ballot = __ballot_sync(0xffffffffu, flag);
  if (lane == 0) scratch[warp] = __popc(ballot);
  __syncthreads();
  int32_t before = 0, all = 0;
  for (int w = 0; w < nwarps; ++w) {
    if (w < warp) before += scratch[w];
    all += scratch[w];
  }
  __syncthreads();
  *total = all;
  return before + __popc(ballot & ((1u << lane) - 1u));
}

// ---- block scores -------------------------------------------------------------------------
//
// Score of block b for KV head h: sum over the g query heads of the group of
// sum_c max(q_c kmin_c, q_c kmax_c) = sum_c (P_c kmax_c + N_c kmin_c), P_c (N_c) being the sum
// of the group's positive (negative) query coordinates, computed once per unit by coef_kernel.
// One CTA scores up to kScoreChunk blocks of one unit: each warp takes 8 blocks at a time, one
// 16-byte load per lane per block of the block's [kmin | kmax] record (2d elements) with the
// lane's coefficients in registers, and reduces the 8 block sums across the warp. The order-preserving 32-bit image of each
// binary32 score goes to `ord_out`. (Staging the chunk through shared memory with one bulk TMA
// copy was measured slower: its 64 KiB buffer leaves 3 scoring CTAs per SM and the selection
// tails hold them.)
constexpr int kScoreChunk = 128;
constexpr int kStageThreads = 256;

// Coefficients of the factorised score, per unit (layer, request, KV head): N_c (sum of the
// group's negative draft coordinates c) then P_c (of its positive ones), [2d] binary32, summed
// over the group's heads in head order. One CTA per (layer, active request), one thread per
// coordinate and KV head.
template <typename T>
__global__ void coef_kernel(Geom G, const int32_t* __restrict__ active, const T* __restrict__ draft,
                            float* __restrict__ coef, int64_t draft_layer_stride, int64_t coef_layer_stride) {
  const int32_t a = blockIdx.x, layer = blockIdx.y;
  const int32_t r = active[a];
  const T* dq = draft + layer * draft_layer_stride + (int64_t)r * G.Hq * G.d;
  float* out = coef + layer * coef_layer_stride + (int64_t)r * G.Hkv * 2 * G.d;
  for (int32_t i = threadIdx.x; i < G.Hkv * G.d; i += blockDim.x) {
    const int32_t h = i / G.d, c = i % G.d;
    float p = 0.f, n = 0.f;
    for (int32_t j = 0; j < G.g; ++j) {
      const float x = to_f(dq[(int64_t)(h * G.g + j) * G.d + c]);
      p += x > 0.f ? x : 0.f;
      n += x < 0.f ? x : 0.f;
    }
    out[(int64_t)h * 2 * G.d + c] = n;
    out[(int64_t)h * 2 * G.d + G.d + c] = p;
  }
}

template <typename T>
__device__ void score_chunk(const Geom& G, const LayerState& S, int32_t r, int32_t h, int32_t b_lo,
                            int32_t b_hi, const float* __restrict__ coef, uint32_t* __restrict__ ord_out) {
  constexpr int V = 16 / sizeof(T);
  const int64_t unit = (int64_t)r * G.Hkv + h;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  coef += unit * 2 * G.d;  // this unit's [N | P]
  const int32_t nvec = 2 * G.d / V;  // 16-byte vectors per summary record
  const T* summ = reinterpret_cast<const T*>(S.summ) + unit * G.nb_max * 2 * G.d;
  uint32_t* ord = ord_out + unit * G.nb_max;
  if (nvec <= 32) {
    // one vector per lane (bf16 up to d = 128, fp32 up to d = 64): coefficients in registers,
    // 8 blocks of loads in flight per warp
    constexpr int U = 8;
    float cf[V];
#pragma unroll
    for (int e = 0; e < V; ++e) cf[e] = lane < nvec ? __ldg(coef + lane * V + e) : 0.f;
    for (int32_t b0 = b_lo + warp * U; b0 < b_hi; b0 += nwarps * U) {
      union {
        uint4 u4;
        T e[V];
      } x[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int32_t b = b0 + u;
        x[u].u4 = (b < b_hi && lane < nvec)
                      ? __ldcs(reinterpret_cast<const uint4*>(summ + (int64_t)b * 2 * G.d) + lane)
                      : make_uint4(0, 0, 0, 0);
      }
      float p8[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < V; ++e) acc = fmaf(cf[e], to_f(x[u].e[e]), acc);
        p8[u] = acc;
      }
      // transposing butterfly: each exchange halves the values a lane carries, so the 8 block
      // sums take 9 shuffles; lane quad q ends with the sum of block (bit4, bit3, bit2 of lane)
      float p4[4], p2[2];
      const bool b16 = lane & 16, b8 = lane & 8, b4 = lane & 4;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        p4[i] = (b16 ? p8[i + 4] : p8[i]) + __shfl_xor_sync(0xffffffffu, b16 ? p8[i] : p8[i + 4], 16);
#pragma unroll
      for (int i = 0; i < 2; ++i)
        p2[i] = (b8 ? p4[i + 2] : p4[i]) + __shfl_xor_sync(0xffffffffu, b8 ? p4[i] : p4[i + 2], 8);
      float sc = (b4 ? p2[1] : p2[0]) + __shfl_xor_sync(0xffffffffu, b4 ? p2[0] : p2[1], 4);
      sc += __shfl_xor_sync(0xffffffffu, sc, 2);
      sc += __shfl_xor_sync(0xffffffffu, sc, 1);
      const int32_t b = b0 + (b16 ? 4 : 0) + (b8 ? 2 : 0) + (b4 ? 1 : 0);
      if ((lane & 3) == 0 && b < b_hi) ord[b] = orderable(sc);
    }
    return;
  }
  for (int32_t b = b_lo + warp; b < b_hi; b += nwarps) {
    float part = 0.f;
    for (int32_t v = lane; v < nvec; v += 32) {
      union {
        uint4 u4;
        T e[V];
      } x;
      x.u4 = __ldcs(reinterpret_cast<const uint4*>(summ + (int64_t)b * 2 * G.d) + v);
      const float* cf = coef + v * V;
#pragma unroll
      for (int e = 0; e < V; ++e) part = fmaf(__ldg(cf + e), to_f(x.e[e]), part);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0) ord[b] = orderable(part);
  }
}

// ---- top-K and diff / admit / evict (one unit) ---------------------------------------------
//
// Top-K: a most-significant-digit radix select over the order-preserving score images (8-bit
// digits, warp-aggregated histogram counts) narrows a prefix until the K-th largest image lies
// in a digit bin that is taken whole, or until the image T itself is known. The selection is
// then every image above the prefix plus, among the images equal to it, the lowest block ids
// needed to make K: an ordered compaction in block-id order (warp-contiguous segments, ballot
// prefix counts) writes them in id order, and each one's place in (score desc, block id asc)
// order is its rank, counted against the K candidates, so equal scores resolve to the lower
// block id.
//
// Diff / admit / evict: a block -> slot map of the unit's slot table is built in shared memory;
// hits (selected and resident) keep their slot and get stamp = step; misses are ranked in
// selection order and the first min(C, #misses) are admitted; targets are free slots by
// ascending slot, then unselected resident blocks by (stamp asc, block id asc); each admitted
// block takes the target of its rank and (block, slot) is appended to the fetch list.
//
// With pred_ids / pred_n set, only the top-K is computed and written there (prediction only:
// the unit's selection, slot table and fetch list are left as they are).
__host__ __device__ inline size_t align16(size_t n) { return (n + 15) & ~size_t(15); }

__host__ __device__ inline size_t select_bytes(const Geom& G, int32_t nb_cap) {
  return (size_t)G.kb * 8 /* tkey */ + (size_t)G.kb * 8 /* candidates */ + (size_t)6 * G.kb * 4 + 48 * 4 +
         256 * 4 /* histogram */ + align16((size_t)nb_cap * 4) + align16((size_t)nb_cap * 2);
}

// lcap >= 0: the request is partially staged with a decode-side tier of lcap entries per unit,
// and its fetch list is routed through that tier (S.route).
__device__ void select_unit(const Geom& G, const LayerState& S, int32_t r, int32_t h, int32_t nb,
                            int32_t nb_cap, const uint32_t* ord_in, int32_t cap_blocks, int32_t step,
                            int32_t lcap, Counters* ctr, int32_t* err, uint8_t* smem, int32_t* pred_ids,
                            int32_t* pred_n) {
  // the Kb-sized arrays first: every address below derives from kernel parameters alone
  unsigned long long* tkey = reinterpret_cast<unsigned long long*>(smem);  // [kb] eviction order
  uint32_t* ckey = reinterpret_cast<uint32_t*>(tkey + G.kb);  // [kb] selected images, in block-id order
  int32_t* cid = reinterpret_cast<int32_t*>(ckey + G.kb);     // [kb] their block ids
  int32_t* sb = cid + G.kb;       // [kb] slot -> block
  int32_t* st = sb + G.kb;        // [kb] stamps
  int32_t* hit = st + G.kb;       // [kb]
  int32_t* target = hit + G.kb;   // [kb]
  int32_t* selid = target + G.kb; // [kb] selection, in order
  int32_t* missrank = selid + G.kb;  // [kb] rank of a miss, or -1
  int32_t* fblk = hit;            // [kb] block of each fetch entry (reuses `hit` once it is read)
  int32_t* scratch = missrank + G.kb;  // [48]
  uint32_t* hist = reinterpret_cast<uint32_t*>(scratch + 48);  // [256]
  uint32_t* ord = hist + 256;                                   // [nb_cap] score images
  int16_t* b2s = reinterpret_cast<int16_t*>(reinterpret_cast<uint8_t*>(ord) + align16((size_t)nb_cap * 4));  // [nb_cap]

  const int64_t unit = (int64_t)r * G.Hkv + h;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const bool predict = pred_ids != nullptr;
  // the scores were written by the other CTAs of this unit: read them past L1
  uint32_t all_or = 0u, all_and = ~0u;  // bits set in some / every image of the unit
  for (int32_t b = tid; b < nb; b += blockDim.x) {
    const uint32_t u = __ldcg(ord_in + unit * G.nb_max + b);
    ord[b] = u;
    b2s[b] = -1;
    all_or |= u;
    all_and &= u;
  }
  all_or = __reduce_or_sync(0xffffffffu, all_or);
  all_and = __reduce_and_sync(0xffffffffu, all_and);
  if (lane == 0) {
    scratch[24 + warp] = (int32_t)all_or;
    scratch[36 + warp] = (int32_t)all_and;
  }
  if (!predict)
    for (int32_t s = tid; s < G.kb; s += blockDim.x) {
      sb[s] = S.slot_block[unit * G.kb + s];
      st[s] = S.stamp[unit * G.kb + s];
      hit[s] = 0;
    }
  __syncthreads();
  if (!predict)
    for (int32_t s = tid; s < G.kb; s += blockDim.x) {
      const int32_t b = sb[s];
      if (b >= nb) record_error(err, kErrBlockRange, -1, r, b);
      else if (b >= 0) b2s[b] = (int16_t)s;
    }

  // ---- top-K: radix select. Invariant: the K largest images are those whose masked image is
  // above `prefix` plus the first `krem` (by block id) of those whose masked image equals it.
  // The bits above the highest bit in which the unit's images differ are common to all of them,
  // so the digits start there (8 bits at a time); when every image is equal no digit is needed ----
  const int32_t K = nb < G.kb ? nb : G.kb;
  uint32_t prefix = 0, mask = 0;
  int32_t krem = K;
  if (K < nb) {
    uint32_t any = 0u, every = ~0u;
    for (int w = 0; w < nwarps; ++w) {
      any |= (uint32_t)scratch[24 + w];
      every &= (uint32_t)scratch[36 + w];
    }
    const uint32_t differ = any ^ every;
    const int top0 = differ ? 31 - __clz(differ) : -1;
    // the bits above top0 (every bit if no two images differ)
    mask = top0 < 0 ? ~0u : (top0 >= 31 ? 0u : ~((2u << top0) - 1u));
    prefix = every & mask;
    for (int top = top0; top >= 0;) {
      const int lo = top >= 7 ? top - 7 : 0;
      const uint32_t dmask = (2u << (top - lo)) - 1u;  // the digit's bits, shifted down to bit 0
      for (int32_t i = tid; i < 256; i += blockDim.x) hist[i] = 0;
      __syncthreads();
#pragma unroll 1
      for (int32_t b0 = 0; b0 < nb; b0 += blockDim.x) {
        const int32_t b = b0 + tid;
        const uint32_t u = b < nb ? ord[b] : 0u;
        const bool in = b < nb && (u & mask) == prefix;
        // lanes with the same digit add once, by their lowest lane (the leading digits of a
        // unit's scores are mostly equal, and one shared atomic per lane would serialise)
        const uint32_t dg = in ? ((u >> lo) & dmask) : (256u + (uint32_t)lane);
        const unsigned grp = __match_any_sync(0xffffffffu, dg);
        if (in && (__ffs(grp) - 1) == lane) atomicAdd(&hist[dg], (uint32_t)__popc(grp));
      }
      __syncthreads();
      if (warp == 0) {
        // lane l owns digits 255 - 8l .. 248 - 8l (high to low); the lane whose digits hold the
        // K-th image walks them again
        uint32_t own = 0;
        for (int i = 0; i < 8; ++i) own += hist[255 - 8 * lane - i];
        uint32_t incl = own;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const uint32_t excl = incl - own;
        if (excl < (uint32_t)krem && (uint32_t)krem <= incl) {
          uint32_t run = excl;
          for (int i = 0; i < 8; ++i) {
            const uint32_t c = hist[255 - 8 * lane - i];
            if (run + c >= (uint32_t)krem) {
              scratch[32] = 255 - 8 * lane - i;
              scratch[33] = krem - (int32_t)run;
              scratch[34] = (int32_t)c;
              break;
            }
            run += c;
          }
        }
      }
      __syncthreads();
      prefix |= (uint32_t)scratch[32] << lo;
      mask |= dmask << lo;
      krem = scratch[33];
      const bool whole = scratch[34] == krem;  // the bin of the K-th image is taken whole
      __syncthreads();
      if (whole) break;
      top = lo - 1;
    }
  }
  // ---- ordered compaction, in block-id order: every image above the prefix, and the first krem
  // equal to it. Warp w walks blocks [w*seg, (w+1)*seg) twice: counts, then places ----
  {
    const int32_t seg = (((nb + nwarps - 1) / nwarps) + 31) & ~31;
    const int32_t lo = warp * seg, hi = min(nb, lo + seg);
    const unsigned below = (1u << lane) - 1u;
    int32_t n_eq = 0, n_gt = 0;
#pragma unroll 1
    for (int32_t b0 = lo; b0 < hi; b0 += 32) {
      const int32_t b = b0 + lane;
      const uint32_t m = b < hi ? (ord[b] & mask) : 0u;
      n_eq += __popc(__ballot_sync(0xffffffffu, b < hi && m == prefix));
      n_gt += __popc(__ballot_sync(0xffffffffu, b < hi && m > prefix));
    }
    if (lane == 0) {
      scratch[warp] = n_eq;
      scratch[16 + warp] = n_gt;
    }
    __syncthreads();
    int32_t eq_base = 0, gt_base = 0;
    for (int w = 0; w < warp; ++w) {
      eq_base += scratch[w];
      gt_base += scratch[16 + w];
    }
#pragma unroll 1
    for (int32_t b0 = lo; b0 < hi; b0 += 32) {
      const int32_t b = b0 + lane;
      const uint32_t u = b < hi ? ord[b] : 0u;
      const uint32_t m = u & mask;
      const bool eq = b < hi && m == prefix, gt = b < hi && m > prefix;
      const unsigned beq = __ballot_sync(0xffffffffu, eq), bgt = __ballot_sync(0xffffffffu, gt);
      const int32_t eb = eq_base + __popc(beq & below), gb = gt_base + __popc(bgt & below);
      if (gt || (eq && eb < krem)) {
        const int32_t pos = gb + min(eb, krem);
        ckey[pos] = u;
        cid[pos] = b;
      }
      eq_base += __popc(beq);
      gt_base += __popc(bgt);
    }
  }
  __syncthreads();
  // ---- order: the rank of candidate i in (image desc, block id asc); candidates are in id order,
  // so an equal image ranks before i exactly when its candidate index is lower ----
  // (with K at most half the CTA, two threads count the ranks of one candidate, half each)
  const bool pairs = 2 * K <= (int32_t)blockDim.x;
  for (int32_t i0 = 0; i0 < K; i0 += pairs ? (int32_t)blockDim.x / 2 : (int32_t)blockDim.x) {
    const int32_t i = i0 + (pairs ? tid >> 1 : tid);
    const int32_t j0 = pairs && (tid & 1) ? K / 2 : 0, j1 = pairs && !(tid & 1) ? K / 2 : K;
    const uint32_t u = i < K ? ckey[i] : 0u;
    int32_t rank = 0;
    if (i < K) {
#pragma unroll 4
      for (int32_t j = j0; j < j1; ++j) {
        const uint32_t x = ckey[j];
        rank += (x > u) | ((x == u) & (j < i));
      }
    }
    if (pairs) rank += __shfl_xor_sync(0xffffffffu, rank, 1);
    if (i >= K || (pairs && (tid & 1))) continue;
    const int32_t b = cid[i];
    if (predict) {
      pred_ids[unit * G.kb + rank] = b;
      continue;
    }
    selid[rank] = b;
    S.sel_ids[unit * G.kb + rank] = b;
    S.sel_scores[unit * G.kb + rank] = from_orderable(u);
    const int32_t s = b2s[b];
    if (s >= 0) {
      hit[s] = 1;
      st[s] = step;
      missrank[rank] = -1;
    } else {
      missrank[rank] = 0;
    }
  }
  if (predict) {
    if (tid == 0) pred_n[unit] = K;
    return;
  }
  if (tid == 0) S.n_sel[unit] = K;
  __syncthreads();

  // ---- diff / admit / evict ----
  int32_t n_miss = 0;
  for (int32_t i0 = 0; i0 < K; i0 += blockDim.x) {
    const int32_t i = i0 + tid;
    const bool miss = i < K && missrank[i] == 0;
    int32_t n;
    const int32_t rk = n_miss + block_rank(miss, scratch, &n);
    if (miss) missrank[i] = rk;
    n_miss += n;
  }
  const int32_t n_admit = n_miss < cap_blocks ? n_miss : cap_blocks;
  for (int32_t s = tid; s < G.kb; s += blockDim.x) {
    unsigned long long k;
    if (sb[s] < 0)
      k = (unsigned long long)s;  // free slots first, by slot
    else if (!hit[s])
      k = (1ull << 63) | ((unsigned long long)((uint32_t)st[s] ^ 0x80000000u) << 31) |
          (unsigned long long)(uint32_t)sb[s];  // then least recently selected, by block id
    else
      k = ~0ull;  // selected and resident: never a target
    tkey[s] = k;
  }
  __syncthreads();
  if (n_admit > 0) {
    // each slot's rank among the targets (two threads per slot when the slots fill half the CTA)
    const bool tpairs = 2 * G.kb <= (int32_t)blockDim.x;
    for (int32_t s0 = 0; s0 < G.kb; s0 += tpairs ? (int32_t)blockDim.x / 2 : (int32_t)blockDim.x) {
      const int32_t s = s0 + (tpairs ? tid >> 1 : tid);
      const int32_t o0 = tpairs && (tid & 1) ? G.kb / 2 : 0, o1 = tpairs && !(tid & 1) ? G.kb / 2 : G.kb;
      const unsigned long long mine = s < G.kb ? tkey[s] : ~0ull;
      int32_t pos = 0;
      if (mine != ~0ull) {
#pragma unroll 4
        for (int32_t o = o0; o < o1; ++o) pos += tkey[o] < mine;
      }
      if (tpairs) pos += __shfl_xor_sync(0xffffffffu, pos, 1);
      if (s < G.kb && mine != ~0ull && !(tpairs && (tid & 1)) && pos < n_admit) target[pos] = s;
    }
  }
  __syncthreads();
  for (int32_t i = tid; i < K; i += blockDim.x) {
    const int32_t rk = missrank[i];
    if (rk < 0 || rk >= n_admit) continue;
    const int32_t b = selid[i];
    const int32_t s = target[rk];
    sb[s] = b;
    st[s] = step;
    fblk[rk] = b;
    S.fetch[(unit * G.kb + rk) * 2 + 0] = b;
    S.fetch[(unit * G.kb + rk) * 2 + 1] = s;
  }
  __syncthreads();

  // ---- decode-side tier (partially staged requests): in fetch order, a block already kept is
  // read from its entry; the k-th block fetched for the first time is read from the full copy
  // and kept in entry used + k while entries remain, else read from the full copy only ----
  int32_t n_fresh = 0;
  const int32_t used0 = lcap >= 0 ? S.local_used[unit] : 0;
  if (lcap < 0) {
    for (int32_t i = tid; i < n_admit; i += blockDim.x) S.route[unit * G.kb + i] = -1;
  } else {
    for (int32_t i0 = 0; i0 < n_admit; i0 += blockDim.x) {
      const int32_t i = i0 + tid;
      const int32_t e = i < n_admit ? S.local_of[unit * G.nb_max + fblk[i]] : 0;
      const bool fresh = i < n_admit && e < 0;
      int32_t n;
      const int32_t k = n_fresh + block_rank(fresh, scratch, &n);
      n_fresh += n;
      if (i >= n_admit) continue;
      int32_t route = 2 * e;
      if (fresh) {
        route = -1;
        if (used0 + k < lcap) {
          route = 2 * (used0 + k) + 1;
          S.local_of[unit * G.nb_max + fblk[i]] = used0 + k;
        }
      }
      S.route[unit * G.kb + i] = route;
    }
  }
  for (int32_t s = tid; s < G.kb; s += blockDim.x) {
    S.slot_block[unit * G.kb + s] = sb[s];
    S.stamp[unit * G.kb + s] = st[s];
  }
  if (tid == 0) {
    S.n_fetch[unit] = n_admit;
    if (n_admit > 0) atomicAdd(&ctr->fetched_blocks, (unsigned long long)n_admit);
    if (lcap >= 0 && n_admit > 0) {
      const int32_t room = lcap - used0 > 0 ? lcap - used0 : 0;
      const int32_t fills = n_fresh < room ? n_fresh : room;
      S.local_used[unit] = used0 + fills;
      atomicAdd(&ctr->local_hits, (unsigned long long)(n_admit - n_fresh));
      atomicAdd(&ctr->local_fills, (unsigned long long)fills);
      atomicAdd(&ctr->full_reads, (unsigned long long)n_fresh);
    }
  }
}

// One CTA scores kScoreChunk blocks of one unit; the last of the unit's `chunks` CTAs to finish
// (counted in `arrivals`, which it resets) then selects for the unit.
template <typename T>
__global__ void __launch_bounds__(kStageThreads)
stage_kernel(Geom G, LayerState S, ReqTables RT, int32_t chunks, int32_t nb_cap,
             const float* __restrict__ coef, uint32_t* __restrict__ ord, int32_t* __restrict__ arrivals,
             int32_t cap_blocks, int32_t step, Counters* ctr, int32_t* err, int32_t* pred_ids,
             int32_t* pred_n) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int32_t last;
  const int32_t ua = blockIdx.x / chunks, chunk = blockIdx.x % chunks;
  const int32_t a = ua / G.Hkv, h = ua % G.Hkv;
  const int32_t r = RT.active[a];
  const int32_t len = S.len_act[a];  // (not S.len[r]: no wait for r first)
  const int32_t nb = (len + G.bs - 1) / G.bs;
  const int32_t b_lo = chunk * kScoreChunk;
  const bool bad = len < 0 || nb > G.nb_max || nb > nb_cap;
  if (bad && threadIdx.x == 0 && chunk == 0) record_error(err, kErrLength, -1, r, len);
  if (!bad && b_lo < nb)
    score_chunk<T>(G, S, r, h, b_lo, min(nb, b_lo + kScoreChunk), coef, ord);
  // the barrier orders every thread's score images before thread 0's device-scope fence, which
  // then releases them all ahead of the arrival (one fence per CTA instead of one per thread)
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    last = atomicAdd(&arrivals[ua], 1) == chunks - 1;
    if (last) arrivals[ua] = 0;
  }
  __syncthreads();
  if (!last || bad) return;
  __threadfence();
  select_unit(G, S, r, h, nb, nb_cap, ord, cap_blocks, step, RT.local_cap[r], ctr, err, smem + 16, pred_ids,
              pred_n);
}

}  // namespace

size_t stage_smem_bytes(const Geom& G, int32_t nb_cap) {
  return 16 + select_bytes(G, nb_cap > 0 ? nb_cap : 1);
}

cudaError_t launch_coef(const Geom& G, const int32_t* active, int32_t n_active, int32_t layers, const void* draft,
                        int64_t draft_layer_stride, float* coef, int64_t coef_layer_stride, cudaStream_t s) {
  if (n_active <= 0 || layers <= 0) return cudaSuccess;
  const dim3 grid((unsigned)n_active, (unsigned)layers);
  const int threads = G.Hkv * G.d < 256 ? ((G.Hkv * G.d + 31) / 32) * 32 : 256;
  if (G.dtype == OKV_F32)
    coef_kernel<float><<<grid, threads, 0, s>>>(G, active, (const float*)draft, coef, draft_layer_stride,
                                                coef_layer_stride);
  else
    coef_kernel<__nv_bfloat16><<<grid, threads, 0, s>>>(G, active, (const __nv_bfloat16*)draft, coef,
                                                        draft_layer_stride, coef_layer_stride);
  return cudaGetLastError();
}

cudaError_t launch_stage(const Geom& G, const LayerState& S, const ReqTables& T, int32_t n_active,
                         int32_t max_nb, const float* coef, uint32_t* scores, int32_t* arrivals,
                         int32_t cap_blocks, int32_t step, Counters* ctr, int32_t* err, cudaStream_t s,
                         int* n_launches, int32_t* pred_ids, int32_t* pred_n) {
  *n_launches = 0;
  if (n_active <= 0) return cudaSuccess;
  const int32_t nb_cap = max_nb > 0 ? max_nb : 1;
  const int32_t chunks = (nb_cap + kScoreChunk - 1) / kScoreChunk;
  const size_t smem = stage_smem_bytes(G, nb_cap);
  const int grid = n_active * G.Hkv * chunks;
  cudaError_t e;
  if (G.dtype == OKV_F32) {
    e = cudaFuncSetAttribute(stage_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    stage_kernel<float><<<grid, kStageThreads, smem, s>>>(G, S, T, chunks, nb_cap, coef, scores, arrivals,
                                                          cap_blocks, step, ctr, err, pred_ids, pred_n);
  } else {
    e = cudaFuncSetAttribute(stage_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    stage_kernel<__nv_bfloat16><<<grid, kStageThreads, smem, s>>>(G, S, T, chunks, nb_cap, coef, scores, arrivals,
                                                                  cap_blocks, step, ctr, err, pred_ids, pred_n);
  }
  e = cudaGetLastError();
  if (e == cudaSuccess) *n_launches = 1;
  return e;
}

}  // namespace okv
