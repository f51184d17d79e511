// KV transfer: copy the admitted blocks from page-locked host memory into their HBM slots.
//
// OasisKV (paperlayer.ai/abs/2608.08097v1, "4 System Design"): the selected non-resident
// blocks are prefetched asynchronously from off-GPU memory into HBM, overlapped with the
// forward pass. Here the SMs read the host buffer directly over the host link (the buffer is
// device-mapped), one warp per block: every lane issues all of its 16-byte loads of the block
// before storing, so a warp keeps a whole block in flight.
//
// Partially staged requests (same section, last bullet: the prefill side keeps the full KV
// cache until the request completes, the decode side a demand-filled subset): a block comes
// from the decode side's kept copy when it has one; a block fetched for the first time comes
// from the full copy and is also written to the decode-side entry the selection assigned.
#include <stdlib.h>
#include <string.h>

#include "okv_internal.h"

namespace okv {
namespace {

constexpr int kGatherWarps = 2;

__device__ __forceinline__ void record_error(int32_t* err, int32_t code, int32_t a, int32_t b,
                                             int32_t c) {
  if (atomicCAS(err, 0, code) == 0) {
    err[1] = a;
    err[2] = b;
    err[3] = c;
  }
}

// One work item resolved to its copy: source (host copy, or the decode side's kept copy),
// destination slot, and the decode-side entry to fill (or null). `ok` is false for an item past
// its unit's fetch count or one that failed a bounds check (recorded in `err`).
struct Copy {
  const uint4* src;
  uint4* dst;
  uint4* keep;
  bool ok;
};

__device__ __forceinline__ Copy resolve(const Geom& G, const LayerState& S, const ReqTables& RT, int32_t layer,
                                        int32_t cmax, int64_t it, int lane, int32_t* err) {
  Copy c{nullptr, nullptr, nullptr, false};
  const int32_t ua = (int32_t)(it / cmax), e = (int32_t)(it % cmax);
  const int32_t a = ua / G.Hkv, h = ua % G.Hkv;
  const int32_t r = RT.active[a];
  const int64_t unit = (int64_t)r * G.Hkv + h;
  if (e >= S.n_fetch[unit]) return c;
  const int32_t b = S.fetch[(unit * G.kb + e) * 2 + 0];
  const int32_t s = S.fetch[(unit * G.kb + e) * 2 + 1];
  const int32_t cap = RT.cap_blocks[r];
  if (b < 0 || b >= cap || s < 0 || s >= G.kb) {
    if (lane == 0) record_error(err, b < 0 || b >= cap ? kErrBlockRange : kErrSlotRange, layer, r, e);
    return c;
  }
  c.src = reinterpret_cast<const uint4*>(RT.host_kv[r] + (((int64_t)layer * G.Hkv + h) * cap + b) * G.block_bytes);
  c.dst = reinterpret_cast<uint4*>(S.pool + (unit * G.kb + s) * G.block_bytes);
  const int32_t lcap = RT.local_cap[r];
  if (lcap >= 0) {
    // partially staged request: read the decode side's kept copy, or read the full copy and
    // keep it in the entry the selection assigned
    const int32_t route = S.route[unit * G.kb + e];
    if (route >= 0) {
      const int32_t ent = route >> 1;
      if (ent >= lcap) {
        if (lane == 0) record_error(err, kErrLocalRange, layer, r, ent);
        return c;
      }
      uint4* kept =
          reinterpret_cast<uint4*>(RT.local_kv[r] + (((int64_t)layer * G.Hkv + h) * lcap + ent) * G.block_bytes);
      if (route & 1)
        c.keep = kept;
      else
        c.src = kept;
    }
  }
  c.ok = true;
  return c;
}

// Persistent grid over work items, item i being entry i % cmax of active unit i / cmax (items
// past the unit's fetch count are skipped). With `work` set, warps claim items one at a time
// from work[0], so they finish together instead of at the end of fixed shares whose host-read
// latencies differ; the last CTA to leave (counted in work[1]) resets both counters. Without
// it, warp w copies items w, w + nwarps, ... A warp claims and resolves its next item while
// the host reads of the current one are in flight, so the chain of bookkeeping loads (claim,
// request, fetch entry, host pointer) overlaps the copy instead of preceding it. Measured on
// GB300 against the same grid without it, in interleaved pairs: the in-step link rate 0.84-0.90
// of the pinned-copy rate against 0.81-0.86 and +0.7% median tok/s (6 of 8 pairs) at Qwen3-8B
// 16K batch 128; +1.5% to +3.5% (5 of 5) at mixed lengths with appends; even at 32K batch 32.
template <int kVecPerLane>
__global__ void __launch_bounds__(kGatherWarps * 32)
gather_kernel(Geom G, LayerState S, ReqTables RT, int32_t layer, int32_t n_units, int32_t cmax,
              int32_t* work, int32_t* err) {
  const int lane = threadIdx.x & 31;
  const int64_t nw = (int64_t)gridDim.x * kGatherWarps;
  const int64_t total = (int64_t)n_units * cmax;
  const int32_t nvec = (int32_t)(G.block_bytes / 16);
  auto next = [&](int64_t prev) -> int64_t {
    if (!work) return prev + nw;
    int32_t claimed = 0;
    if (lane == 0) claimed = atomicAdd(&work[0], 1);
    return __shfl_sync(0xffffffffu, claimed, 0);
  };
  int64_t it = work ? next(0) : (int64_t)blockIdx.x * kGatherWarps + (threadIdx.x >> 5);
  Copy cur{nullptr, nullptr, nullptr, false};
  if (it < total) cur = resolve(G, S, RT, layer, cmax, it, lane, err);
  while (it < total) {
    uint4 x[kVecPerLane];
    if (cur.ok) {
#pragma unroll
      for (int i = 0; i < kVecPerLane; ++i) {
        const int32_t v = i * 32 + lane;
        if (v < nvec) x[i] = __ldcs(cur.src + v);
      }
    }
    // the next item, while this one's first host reads are in flight
    const int64_t nit = next(it);
    Copy nc{nullptr, nullptr, nullptr, false};
    if (nit < total) nc = resolve(G, S, RT, layer, cmax, nit, lane, err);
    if (cur.ok) {
      for (int32_t base = 0;;) {
#pragma unroll
        for (int i = 0; i < kVecPerLane; ++i) {
          const int32_t v = base + i * 32 + lane;
          if (v < nvec) __stcs(cur.dst + v, x[i]);
        }
        if (cur.keep) {
#pragma unroll
          for (int i = 0; i < kVecPerLane; ++i) {
            const int32_t v = base + i * 32 + lane;
            if (v < nvec) __stcs(cur.keep + v, x[i]);
          }
        }
        base += 32 * kVecPerLane;
        if (base >= nvec) break;
#pragma unroll
        for (int i = 0; i < kVecPerLane; ++i) {
          const int32_t v = base + i * 32 + lane;
          if (v < nvec) x[i] = __ldcs(cur.src + v);
        }
      }
    }
    it = nit;
    cur = nc;
  }
  if (work) {
    __syncthreads();
    if (threadIdx.x == 0 && atomicAdd(&work[1], 1) == (int32_t)gridDim.x - 1) {
      work[0] = 0;
      work[1] = 0;
    }
  }
}

}  // namespace

cudaError_t launch_gather(const Geom& G, const LayerState& S, const ReqTables& T, int32_t n_active,
                          int32_t layer, int32_t max_fetch, int32_t* work, int32_t* err, cudaStream_t s) {
  if (n_active <= 0 || max_fetch <= 0) return cudaSuccess;
  // A few warps keep enough host reads in flight to fill the host link; more of them only slow
  // the HBM-bound kernels running beside the gather. 128 warps, spread as 64 CTAs of 2 over as
  // many SMs: measured on GB300 at Qwen3-8B batch 128, 64 CTAs of 2 warps beat 32 of 4 in 5 of 6
  // interleaved pairs (about +3% tok/s, the link at 0.82-0.86 of the pinned-copy rate in the
  // step), 16 of 8 lost 3-8% and 128 of 1 lost e2e rate. OKV_GATHER_CTAS overrides the count.
  static int ctas = [] {
    int n = 0;
    if (const char* e = getenv("OKV_GATHER_CTAS")) n = atoi(e);
    return n > 0 ? n : 64;
  }();
  const int64_t items = (int64_t)n_active * G.Hkv * max_fetch;
  const int64_t want = (items + kGatherWarps - 1) / kGatherWarps;
  const int grid = (int)(want < ctas ? want : ctas);
  static const bool dynamic = [] {
    const char* e = getenv("OKV_GATHER_DYNAMIC");
    return !(e && strcmp(e, "0") == 0);
  }();
  gather_kernel<16><<<grid, kGatherWarps * 32, 0, s>>>(G, S, T, layer, n_active * G.Hkv, max_fetch,
                                                       dynamic ? work : nullptr, err);
  return cudaGetLastError();
}

}  // namespace okv
