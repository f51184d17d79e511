// Internal declarations of the okv CUDA library (sm_103a). Not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "../../include/okv.h"

namespace okv {

// Device error word: [0] = first error code (0 = none), [1..3] = details of that error.
enum DeviceError : int32_t {
  kErrNone = 0,
  kErrBlockRange = 1,   // a block id outside [0, nb) of its unit
  kErrSlotRange = 2,    // a slot outside [0, Kb)
  kErrCapacity = 3,     // an append past the request's host capacity
  kErrLength = 4,       // a context length outside [0, max_blocks * block_size]
  kErrTimeout = 5,      // a bounded wait for an asynchronous copy gave up
  kErrLocalRange = 6,   // a decode-side tier entry outside [0, local_cap)
};

// Geometry shared by host and kernels (passed by value).
struct Geom {
  int32_t L, Hq, Hkv, g, d, bs, kb, R, nb_max;
  int32_t dtype;       // OKV_F32 / OKV_BF16
  int32_t elem;        // bytes per element
  int64_t block_bytes; // 2 * bs * d * elem: K and V of one block of one unit
};

// Per-layer views of the device state, all indexed [R][Hkv]...
struct LayerState {
  uint8_t* summ;        // [R][Hkv][nb_max][2][d] storage
  uint8_t* pool;        // [R][Hkv][kb][2][bs][d] storage
  int32_t* slot_block;  // [R][Hkv][kb] slot -> block or -1
  int32_t* stamp;       // [R][Hkv][kb]
  int32_t* sel_ids;     // [R][Hkv][kb]
  float* sel_scores;    // [R][Hkv][kb]
  int32_t* n_sel;       // [R][Hkv]
  int32_t* fetch;       // [R][Hkv][kb][2] (block, slot)
  int32_t* n_fetch;     // [R][Hkv]
  int32_t* len;         // [R] tokens of each request at this layer
  int32_t* len_act;     // [n_active] the same, indexed by position in the active list
  // decode-side tier of partially staged requests
  int32_t* local_of;    // [R][Hkv][nb_max] block -> kept entry or -1
  int32_t* local_used;  // [R][Hkv] entries in use
  int32_t* route;       // [R][Hkv][kb] per fetch entry: 2e = read kept entry e, 2e+1 = read the
                        // full copy and keep it in entry e, -1 = read the full copy only
};

// Per-request device-side tables (shared by all layers).
struct ReqTables {
  const int32_t* active;    // [n_active] compact list of active request ids
  const uint64_t* host_kv;  // [R] device address of the request's host KV buffer
  const int32_t* cap_blocks;// [R]
  const uint64_t* local_kv; // [R] device address of the decode-side tier, 0 for none
  const int32_t* local_cap; // [R] entries per unit of the decode-side tier; -1: full-KV request
};

struct Counters {
  unsigned long long fetched_blocks;
  unsigned long long attended_slots;
  unsigned long long local_hits;   // fetches of partially staged requests served by a kept copy
  unsigned long long local_fills;  // ... read from the full copy and kept
  unsigned long long full_reads;   // ... read from the full copy (fills included)
};

// ---- kernel launchers (defined in the k_*.cu files) --------------------------------------
// Every launcher enqueues on `s` and returns cudaGetLastError().

cudaError_t launch_summary_build(const Geom& G, int32_t layer_begin, int32_t layer_end,
                                 int32_t req, uint64_t host_kv, int32_t cap_blocks,
                                 int32_t n_tok, uint8_t* summ_base, int32_t* err,
                                 cudaStream_t s);
// Append one token per active request at `layer` and advance the lengths; `arrivals`: [R] int32
// that start at zero and are left at zero.
cudaError_t launch_append(const Geom& G, const LayerState& S, const ReqTables& T, int32_t n_active,
                          int32_t layer, const void* k_new, const void* v_new, int32_t* arrivals,
                          int32_t* err, cudaStream_t s);
// Empties request `req`'s pool, tables and decode-side tier on every layer and records its
// buffers (local_cap -1 and local_kv 0 for a request that holds its full KV).
struct RequestInit {
  int32_t req, n_tok, cap, local_cap;
  uint64_t host_kv, local_kv;
};
struct StateBase {  // whole-context arrays, [layers] x per-layer block
  int32_t *slot_block, *stamp, *n_sel, *n_fetch, *len, *local_of, *local_used;
  uint64_t *host_kv_tab, *local_kv_tab;
  int32_t *cap_tab, *local_cap_tab;
};
cudaError_t launch_reset_request(const Geom& G, const StateBase& B, const RequestInit& q, cudaStream_t s);
// Staging of one layer for every active unit: block scores (into `scores`, a [R][Hkv][nb_max]
// uint32 workspace) by chunks of blocks; the last chunk of each unit to finish (counted in
// `arrivals`, [R * Hkv] int32 that start at zero and are left at zero) runs the unit's top-K and
// diff / admit / evict. One launch. With pred_ids / pred_n ([R][Hkv][Kb], [R][Hkv]) only the top-K
// is computed, into them.
// Dynamic shared memory of one staging CTA for contexts of up to nb_cap blocks: the selection
// keeps per-block arrays of the unit (score images, block -> slot map, candidates) on chip.
size_t stage_smem_bytes(const Geom& G, int32_t nb_cap);
// The scoring's coefficients of `layers` layers of draft queries (layer l at draft +
// l * draft_layer_stride elements, [R][Hq][d] storage) into coef (layer l at coef +
// l * coef_layer_stride floats, [R][Hkv][2d]: N then P), for the active requests.
cudaError_t launch_coef(const Geom& G, const int32_t* active, int32_t n_active, int32_t layers, const void* draft,
                        int64_t draft_layer_stride, float* coef, int64_t coef_layer_stride, cudaStream_t s);
cudaError_t launch_stage(const Geom& G, const LayerState& S, const ReqTables& T, int32_t n_active,
                         int32_t max_nb, const float* coef, uint32_t* scores, int32_t* arrivals,
                         int32_t cap_blocks, int32_t step, Counters* ctr, int32_t* err, cudaStream_t s,
                         int* n_launches, int32_t* pred_ids = nullptr, int32_t* pred_n = nullptr);
// `work`: two int32 counters of this layer that start at zero and are left at zero.
cudaError_t launch_gather(const Geom& G, const LayerState& S, const ReqTables& T, int32_t n_active,
                          int32_t layer, int32_t max_fetch, int32_t* work, int32_t* err, cudaStream_t s);
// Attention: decides between the tensor-core path (bf16, d = 128, g <= 8) and the CUDA-core
// path; `partials` is a workspace of at least attend_workspace_bytes() bytes.
size_t attend_workspace_bytes(const Geom& G, int32_t n_active);
// `arrivals`: [n_active * Hkv] int32 split arrival counters that start at zero and are left at
// zero; the last CTA of a split unit merges the partials. `ws_bytes` is the size of `partials`:
// a launch never splits a unit more than its partials fit.
// With a draft query `dq` (look-ahead attention), its heads attend over the same resident set and
// write `dout`: in the same pass when 2g <= 8, else in a second pass.
cudaError_t launch_attend(const Geom& G, const LayerState& S, const ReqTables& T, int32_t n_active,
                          int32_t layer, const void* q, void* out, const void* dq, void* dout,
                          const CUtensorMap* pool_map, void* partials, size_t ws_bytes, int32_t* arrivals,
                          Counters* ctr, int32_t* err, cudaStream_t s, int* n_launches, int* used_split);
bool attend_uses_tensor_cores(const Geom& G);

}  // namespace okv
