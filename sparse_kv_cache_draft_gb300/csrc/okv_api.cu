// C ABI of the okv library: context, requests, the per-layer staging pipeline, inspection and
// timing. Declarations and contracts are in include/okv.h.
//
// Stream layout (OasisKV, paperlayer.ai/abs/2608.08097v1, "4 System Design": the per-layer
// background chain of top-K prediction, KV selection and KV transfer runs on independent
// workers overlapped across layers and steps; the foreground waits only for that layer's
// transfer):
//   caller stream : [wait staged(l)] attend(l)      (okv_append: [wait staged(l)] append(l))
//   select stream : [wait caller] [wait staged(l)] score+top-K(l) -> select(l) -> selected(l)
//   copy stream   : [wait selected(l)] gather(l) -> staged(l)
//   append stream : okv_step's appends, all enqueued up front: [wait staged(l)] append(l) -> appended(l)
// Staging of layer l at step t starts after the work the caller enqueued before it (its
// attention of layer l at step t, which reads the slots the gather may overwrite), and the
// attention of layer l at step t+1 waits only for staged(l) (and, in okv_step, appended(l)).
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <chrono>
#include <thread>

#include "okv_internal.h"

using okv::Counters;
using okv::Geom;
using okv::LayerState;
using okv::ReqTables;

struct TimedLaunch {
  int kind;
  cudaEvent_t a, b;
};

struct okv_ctx {
  okv_config cfg{};
  Geom G{};
  int device = 0;
  std::string last_error;

  // device state, [layers] x per-layer block
  uint8_t* summ = nullptr;
  uint8_t* pool = nullptr;
  int32_t* slot_block = nullptr;
  int32_t* stamp = nullptr;
  int32_t* sel_ids = nullptr;
  float* sel_scores = nullptr;
  int32_t* n_sel = nullptr;
  int32_t* fetch = nullptr;
  int32_t* n_fetch = nullptr;
  int32_t* len = nullptr;
  int32_t* len_active = nullptr;   // [layers][R]: the lengths by position in the active list
  int32_t* active_dev = nullptr;
  uint64_t* host_kv_dev = nullptr;
  int32_t* cap_dev = nullptr;
  int32_t* local_of = nullptr;     // [layers][R][Hkv][nb_max]
  int32_t* local_used = nullptr;   // [layers][R][Hkv]
  int32_t* route = nullptr;        // [layers][R][Hkv][kb]
  uint64_t* local_kv_dev = nullptr;  // [R]
  int32_t* local_cap_dev = nullptr;  // [R], -1 for a request that holds its full KV
  int32_t* err_dev = nullptr;
  Counters* ctr_dev = nullptr;
  void* partials = nullptr;
  size_t partials_bytes = 0;
  float* coef_buf = nullptr;     // [layers][R][Hkv][2d]: okv_stage's scoring coefficients of each layer
  float* pred_coef = nullptr;    // [R][Hkv][2d]: okv_predict's
  uint32_t* scores = nullptr;    // [R][Hkv][nb_max]: block score images of the layer being staged
  int32_t* stage_arrivals = nullptr;   // [R * Hkv]: scoring CTAs finished per unit (kept at zero)
  // second staging lane (odd layers), when OKV_STAGE_LANES=2: its own stream and workspace
  uint32_t* scores2 = nullptr;
  int32_t* stage_arrivals2 = nullptr;
  int32_t* attend_arrivals = nullptr;  // [R * Hkv]: attention split CTAs finished per unit
  int32_t* append_arrivals = nullptr;  // [layers][R]: append CTAs finished per request (kept at zero)
  int32_t* gather_work = nullptr;      // [layers][2]: gather work and exit counters (kept at zero)
  float* step_coef = nullptr;          // [2][layers][R][Hkv][2d]: okv_step's coefficients of its drafts
  int step_parity = 0;                 // which half of step_coef the next okv_step fills
  cudaEvent_t ev_step_read[2] = {nullptr, nullptr};  // the stagings of the last step using each half
  cudaEvent_t ev_step_read2[2] = {nullptr, nullptr}; // ... on the second staging lane
  bool step_used[2] = {false, false};
  bool stage_on_caller = false;  // run scoring/selection on the caller's stream (see okv_create)
  CUtensorMap pool_map;  // 64-byte aligned by its type
  bool have_map = false;

  // host mirrors
  std::vector<int> active;             // [R] 0/1
  std::vector<int32_t> active_list;    // compact
  std::vector<void*> host_ptr;         // [R]
  std::vector<int32_t> cap_blocks;     // [R]
  std::vector<void*> local_ptr;        // [R] decode-side tier of a partially staged request
  std::vector<int32_t> local_cap;      // [R] its entries per unit (-1: full-KV request)
  std::vector<int32_t> len_host;       // [L][R]
  std::vector<int> shared_buf;         // [R] host buffer shared with another active request

  // streams and events
  cudaStream_t sel_stream = nullptr, copy_stream = nullptr;
  cudaStream_t sel_stream2 = nullptr;        // the second staging lane, or NULL
  cudaStream_t att_stream = nullptr;         // okv_step's coefficients and attentions, or NULL: the caller's stream
  cudaStream_t app_stream = nullptr;         // okv_step's appends, ahead of the caller's stream
  std::vector<cudaEvent_t> ev_appended;      // [layers]: the last append of each layer
  cudaEvent_t ev_in = nullptr;
  std::vector<cudaEvent_t> ev_selected, ev_staged;
  std::vector<char> staged_once;

  // timing
  bool timing = false;
  std::vector<TimedLaunch> pending;
  std::vector<cudaEvent_t> event_pool;
  double ms[OKV_K_COUNT] = {};
  int64_t n_launch_kind[OKV_K_COUNT] = {};
  int64_t launches = 0;

  // sizes
  int64_t per_layer_units = 0;
  int64_t summ_layer_bytes = 0, pool_layer_bytes = 0;
};

namespace {

okv_status fail(okv_ctx* ctx, okv_status st, const char* fmt, ...) {
  if (ctx) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    ctx->last_error = buf;
  }
  return st;
}

#define OKV_CUDA(ctx, call)                                                                    \
  do {                                                                                         \
    cudaError_t e_ = (call);                                                                   \
    if (e_ != cudaSuccess)                                                                     \
      return fail(ctx, e_ == cudaErrorMemoryAllocation ? OKV_ENOMEM : OKV_ECUDA, "%s: %s (%s:%d)", \
                  #call, cudaGetErrorString(e_), __FILE__, __LINE__);                          \
  } while (0)

LayerState layer_state(const okv_ctx* c, int32_t layer) {
  const Geom& G = c->G;
  const int64_t U = c->per_layer_units;
  LayerState S;
  S.summ = c->summ + layer * c->summ_layer_bytes;
  S.pool = c->pool + layer * c->pool_layer_bytes;
  S.slot_block = c->slot_block + layer * U * G.kb;
  S.stamp = c->stamp + layer * U * G.kb;
  S.sel_ids = c->sel_ids + layer * U * G.kb;
  S.sel_scores = c->sel_scores + layer * U * G.kb;
  S.n_sel = c->n_sel + layer * U;
  S.fetch = c->fetch + layer * U * G.kb * 2;
  S.n_fetch = c->n_fetch + layer * U;
  S.len = c->len + (int64_t)layer * G.R;
  S.len_act = c->len_active + (int64_t)layer * G.R;
  S.local_of = c->local_of + layer * U * G.nb_max;
  S.local_used = c->local_used + layer * U;
  S.route = c->route + layer * U * G.kb;
  return S;
}

ReqTables req_tables(const okv_ctx* c) {
  ReqTables T;
  T.active = c->active_dev;
  T.host_kv = c->host_kv_dev;
  T.cap_blocks = c->cap_dev;
  T.local_kv = c->local_kv_dev;
  T.local_cap = c->local_cap_dev;
  return T;
}

int32_t cap_to_blocks(float cap, int32_t kb) {
  double c = floor((double)cap * (double)kb);
  if (c < 1.0) c = 1.0;
  if (c > kb) c = kb;
  return (int32_t)c;
}

// Timing: a pair of events around one launch on `s`.
struct Timer {
  okv_ctx* c;
  int kind;
  cudaStream_t s;
  cudaEvent_t a = nullptr, b = nullptr;
  Timer(okv_ctx* c_, int k, cudaStream_t s_) : c(c_), kind(k), s(s_) {
    if (!c->timing) return;
    a = take();
    b = take();
    if (a && b) cudaEventRecord(a, s);
  }
  cudaEvent_t take() {
    if (!c->event_pool.empty()) {
      cudaEvent_t e = c->event_pool.back();
      c->event_pool.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
  }
  void stop(int n_launches) {
    c->launches += n_launches;
    c->n_launch_kind[kind] += n_launches;
    if (!c->timing || !a || !b) return;
    cudaEventRecord(b, s);
    c->pending.push_back({kind, a, b});
  }
};

okv_status check_device_error(okv_ctx* c) {
  int32_t e[4];
  OKV_CUDA(c, cudaMemcpy(e, c->err_dev, sizeof(e), cudaMemcpyDeviceToHost));
  if (e[0] != 0) {
    static const int32_t zero[4] = {0, 0, 0, 0};
    cudaMemcpy(c->err_dev, zero, sizeof(zero), cudaMemcpyHostToDevice);
    static const char* names[] = {"none", "block id out of range", "slot out of range",
                                  "append past capacity", "context length out of range",
                                  "asynchronous copy wait timed out", "decode-side entry out of range"};
    const char* n = (e[0] >= 0 && e[0] <= 6) ? names[e[0]] : "unknown";
    return fail(c, OKV_EDEVICE, "device error %d (%s): layer/site %d, request %d, value %d", e[0], n,
                e[1], e[2], e[3]);
  }
  return OKV_OK;
}

okv_status sync_internal(okv_ctx* c) {
  OKV_CUDA(c, cudaStreamSynchronize(c->app_stream));
  OKV_CUDA(c, cudaStreamSynchronize(c->sel_stream));
  if (c->sel_stream2) OKV_CUDA(c, cudaStreamSynchronize(c->sel_stream2));
  if (c->att_stream) OKV_CUDA(c, cudaStreamSynchronize(c->att_stream));
  OKV_CUDA(c, cudaStreamSynchronize(c->copy_stream));
  return OKV_OK;
}

okv_status upload_active(okv_ctx* c) {
  c->active_list.clear();
  for (int32_t r = 0; r < c->G.R; ++r)
    if (c->active[r]) c->active_list.push_back(r);
  if (!c->active_list.empty()) {
    OKV_CUDA(c, cudaMemcpy(c->active_dev, c->active_list.data(), c->active_list.size() * sizeof(int32_t),
                           cudaMemcpyHostToDevice));
    // the lengths by active position (the staging reads a unit's length without first reading its
    // request id; the append kernel keeps both copies advancing together)
    std::vector<int32_t> la((size_t)c->G.L * c->G.R, 0);
    for (int32_t l = 0; l < c->G.L; ++l)
      for (size_t a = 0; a < c->active_list.size(); ++a)
        la[(size_t)l * c->G.R + a] = c->len_host[(size_t)l * c->G.R + c->active_list[a]];
    OKV_CUDA(c, cudaMemcpy(c->len_active, la.data(), la.size() * sizeof(int32_t), cudaMemcpyHostToDevice));
  }
  // shared host buffers among active requests
  for (int32_t r = 0; r < c->G.R; ++r) c->shared_buf[r] = 0;
  for (size_t i = 0; i < c->active_list.size(); ++i)
    for (size_t j = i + 1; j < c->active_list.size(); ++j)
      if (c->host_ptr[c->active_list[i]] == c->host_ptr[c->active_list[j]])
        c->shared_buf[c->active_list[i]] = c->shared_buf[c->active_list[j]] = 1;
  return OKV_OK;
}

int32_t max_blocks_at(const okv_ctx* c, int32_t layer) {
  int32_t m = 0;
  for (int32_t r : c->active_list) {
    const int32_t nb = (c->len_host[(size_t)layer * c->G.R + r] + c->G.bs - 1) / c->G.bs;
    if (nb > m) m = nb;
  }
  return m;
}

}  // namespace

extern "C" {

const char* okv_status_string(okv_status s) {
  switch (s) {
    case OKV_OK: return "ok";
    case OKV_EINVAL: return "invalid argument";
    case OKV_ENOMEM: return "out of memory";
    case OKV_ECUDA: return "CUDA error";
    case OKV_EDEVICE: return "device error";
    case OKV_ETIMEOUT: return "timeout";
    case OKV_ESTATE: return "invalid state";
  }
  return "unknown status";
}

const char* okv_last_error(const okv_ctx* ctx) { return ctx ? ctx->last_error.c_str() : ""; }

okv_status okv_host_alloc(int64_t bytes, void** out) {
  if (!out || bytes <= 0) return OKV_EINVAL;
  *out = nullptr;
  cudaError_t e = cudaHostAlloc(out, (size_t)bytes, cudaHostAllocMapped | cudaHostAllocPortable);
  if (e != cudaSuccess) {
    *out = nullptr;
    return e == cudaErrorMemoryAllocation ? OKV_ENOMEM : OKV_ECUDA;
  }
  return OKV_OK;
}

okv_status okv_host_free(void* p) {
  if (!p) return OKV_OK;
  return cudaFreeHost(p) == cudaSuccess ? OKV_OK : OKV_ECUDA;
}

void okv_destroy(okv_ctx* c) {
  if (!c) return;
  if (c->sel_stream) cudaStreamSynchronize(c->sel_stream);
  if (c->sel_stream2) cudaStreamSynchronize(c->sel_stream2);
  if (c->att_stream) cudaStreamSynchronize(c->att_stream);
  if (c->copy_stream) cudaStreamSynchronize(c->copy_stream);
  if (c->app_stream) cudaStreamSynchronize(c->app_stream);
  for (auto& t : c->pending) {
    cudaEventDestroy(t.a);
    cudaEventDestroy(t.b);
  }
  for (auto e : c->event_pool) cudaEventDestroy(e);
  for (auto e : c->ev_selected) if (e) cudaEventDestroy(e);
  for (auto e : c->ev_staged) if (e) cudaEventDestroy(e);
  for (auto e : c->ev_appended) if (e) cudaEventDestroy(e);
  if (c->ev_in) cudaEventDestroy(c->ev_in);
  for (auto e : c->ev_step_read) if (e) cudaEventDestroy(e);
  for (auto e : c->ev_step_read2) if (e) cudaEventDestroy(e);
  if (c->sel_stream) cudaStreamDestroy(c->sel_stream);
  if (c->sel_stream2) cudaStreamDestroy(c->sel_stream2);
  if (c->att_stream) cudaStreamDestroy(c->att_stream);
  if (c->copy_stream) cudaStreamDestroy(c->copy_stream);
  if (c->app_stream) cudaStreamDestroy(c->app_stream);
  void* bufs[] = {c->summ, c->pool, c->slot_block, c->stamp, c->sel_ids, c->sel_scores,
                  c->n_sel, c->fetch, c->n_fetch, c->len, c->len_active, c->active_dev, c->host_kv_dev, c->cap_dev,
                  c->err_dev, c->ctr_dev, c->partials, c->coef_buf, c->pred_coef, c->scores, c->stage_arrivals, c->attend_arrivals,
                  c->scores2, c->stage_arrivals2,
                  c->local_of, c->local_used, c->route, c->local_kv_dev, c->local_cap_dev,
                  c->append_arrivals, c->step_coef, c->gather_work};
  for (void* p : bufs)
    if (p) cudaFree(p);
  delete c;
}

okv_status okv_create(const okv_config* cfg, okv_ctx** out) {
  if (!cfg || !out) return OKV_EINVAL;
  *out = nullptr;
  const okv_config& k = *cfg;
  okv_ctx* c = new okv_ctx();
  auto bad = [&](const char* why) {
    okv_status st = fail(c, OKV_EINVAL, "okv_create: %s", why);
    fprintf(stderr, "okv_create: %s\n", why);
    delete c;
    return st;
  };
  if (k.layers <= 0 || k.q_heads <= 0 || k.kv_heads <= 0 || k.q_heads % k.kv_heads) return bad("heads");
  if (k.head_dim <= 0 || k.head_dim % 32 || k.head_dim > 256) return bad("head_dim must be a multiple of 32, at most 256");
  if (k.q_heads / k.kv_heads > 8) return bad("GQA group larger than 8");
  if (k.block_size <= 0 || k.block_size > 64) return bad("block_size must be in 1..64");
  if (k.budget_tokens < k.block_size || k.budget_tokens % k.block_size) return bad("budget must be a multiple of block_size");
  if (k.budget_tokens / k.block_size > 1024) return bad("at most 1024 slots per unit");
  if (k.max_requests <= 0 || k.max_blocks_per_request <= 0) return bad("sizes");
  if ((int64_t)k.max_blocks_per_request * k.block_size > INT32_MAX)
    return bad("max_blocks_per_request * block_size must fit in 32 bits (token positions)");
  if (!(k.fetch_cap > 0.f) || k.fetch_cap > 1.f) return bad("fetch_cap must be in (0, 1]");
  if (k.dtype != OKV_F32 && k.dtype != OKV_BF16) return bad("dtype");
  c->cfg = k;
  Geom& G = c->G;
  G.L = k.layers;
  G.Hq = k.q_heads;
  G.Hkv = k.kv_heads;
  G.g = k.q_heads / k.kv_heads;
  G.d = k.head_dim;
  G.bs = k.block_size;
  G.kb = k.budget_tokens / k.block_size;
  G.R = k.max_requests;
  G.nb_max = k.max_blocks_per_request;
  G.dtype = k.dtype;
  G.elem = k.dtype == OKV_F32 ? 4 : 2;
  G.block_bytes = (int64_t)2 * G.bs * G.d * G.elem;
  if ((G.bs * G.d * G.elem) % 16) return bad("block rows must be a multiple of 16 bytes");
  {
    // the selection of a unit runs in one CTA with the unit's per-block arrays on chip
    int dev = 0, optin = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) optin = 0;
    const size_t need = okv::stage_smem_bytes(G, G.nb_max);
    if (optin > 0 && need > (size_t)optin) {
      int32_t fits = G.nb_max;
      while (fits > 1 && okv::stage_smem_bytes(G, fits) > (size_t)optin) fits -= fits > 4096 ? 64 : 1;
      char why[256];
      snprintf(why, sizeof(why),
               "max_blocks_per_request %d needs %zu bytes of shared memory per staging CTA; this device "
               "allows %d (at most about %d blocks at this budget)",
               G.nb_max, need, optin, fits);
      return bad(why);
    }
  }

  okv_status st = OKV_OK;
  auto alloc = [&](void** p, size_t bytes) -> bool {
    cudaError_t e = cudaMalloc(p, bytes ? bytes : 16);
    if (e != cudaSuccess) {
      st = fail(c, e == cudaErrorMemoryAllocation ? OKV_ENOMEM : OKV_ECUDA, "cudaMalloc(%zu): %s", bytes,
                cudaGetErrorString(e));
      return false;
    }
    return true;
  };
  cudaGetDevice(&c->device);
  const int64_t U = (int64_t)G.R * G.Hkv;
  c->per_layer_units = U;
  c->summ_layer_bytes = U * G.nb_max * 2 * G.d * G.elem;
  c->pool_layer_bytes = U * G.kb * G.block_bytes;
  const int64_t L = G.L;
  bool ok = alloc((void**)&c->summ, L * c->summ_layer_bytes) && alloc((void**)&c->pool, L * c->pool_layer_bytes) &&
            alloc((void**)&c->slot_block, L * U * G.kb * 4) && alloc((void**)&c->stamp, L * U * G.kb * 4) &&
            alloc((void**)&c->sel_ids, L * U * G.kb * 4) && alloc((void**)&c->sel_scores, L * U * G.kb * 4) &&
            alloc((void**)&c->n_sel, L * U * 4) && alloc((void**)&c->fetch, L * U * G.kb * 8) &&
            alloc((void**)&c->n_fetch, L * U * 4) && alloc((void**)&c->len, L * G.R * 4) &&
            alloc((void**)&c->len_active, L * G.R * 4) &&
            alloc((void**)&c->active_dev, G.R * 4) && alloc((void**)&c->host_kv_dev, G.R * 8) &&
            alloc((void**)&c->cap_dev, G.R * 4) && alloc((void**)&c->err_dev, 16) &&
            alloc((void**)&c->ctr_dev, sizeof(Counters)) &&
            alloc((void**)&c->coef_buf, (size_t)L * U * 2 * G.d * sizeof(float)) &&
            alloc((void**)&c->pred_coef, (size_t)U * 2 * G.d * sizeof(float)) &&
            alloc((void**)&c->scores, (size_t)U * G.nb_max * sizeof(uint32_t)) &&
            alloc((void**)&c->stage_arrivals, (size_t)U * 4) && alloc((void**)&c->attend_arrivals, (size_t)U * 4) &&
            alloc((void**)&c->local_of, (size_t)L * U * G.nb_max * 4) && alloc((void**)&c->local_used, (size_t)L * U * 4) &&
            alloc((void**)&c->route, (size_t)L * U * G.kb * 4) && alloc((void**)&c->local_kv_dev, G.R * 8) &&
            alloc((void**)&c->local_cap_dev, G.R * 4) && alloc((void**)&c->append_arrivals, (size_t)L * G.R * 4) &&
            alloc((void**)&c->step_coef, (size_t)2 * L * U * 2 * G.d * sizeof(float)) &&
            alloc((void**)&c->gather_work, (size_t)L * 2 * 4);
  // Staging lanes: odd layers stage on a second stream with a workspace of its own, so one layer's
  // per-unit selection tails overlap the next layer's scoring (measured on GB300: +3% decode
  // tok/s at the 32B-class shapes, the same at Qwen3-8B batch 128). OKV_STAGE_LANES=1 keeps one.
  const char* plane = getenv("OKV_STAGE_LANES");
  const bool two_lanes = !(plane && strcmp(plane, "1") == 0);
  if (ok && two_lanes)
    ok = alloc((void**)&c->scores2, (size_t)U * G.nb_max * sizeof(uint32_t)) &&
         alloc((void**)&c->stage_arrivals2, (size_t)U * 4);
  if (ok) {
    size_t ws = 0;
    for (int32_t n = 1; n <= G.R; ++n) {
      const size_t w = okv::attend_workspace_bytes(G, n);
      if (w > ws) ws = w;
    }
    c->partials_bytes = ws;
    ok = alloc(&c->partials, ws);
  }
  if (!ok) {
    fprintf(stderr, "okv_create: %s\n", c->last_error.c_str());
    okv_destroy(c);
    return st;
  }
  auto ck = [&](cudaError_t e) {
    if (e != cudaSuccess && st == OKV_OK) st = fail(c, OKV_ECUDA, "okv_create: %s", cudaGetErrorString(e));
  };
  ck(cudaMemset(c->slot_block, 0xFF, L * U * G.kb * 4));
  ck(cudaMemset(c->stamp, 0xFF, L * U * G.kb * 4));
  ck(cudaMemset(c->n_sel, 0, L * U * 4));
  ck(cudaMemset(c->n_fetch, 0, L * U * 4));
  ck(cudaMemset(c->len, 0, L * G.R * 4));
  ck(cudaMemset(c->len_active, 0, L * G.R * 4));
  ck(cudaMemset(c->err_dev, 0, 16));
  ck(cudaMemset(c->stage_arrivals, 0, U * 4));
  if (c->stage_arrivals2) ck(cudaMemset(c->stage_arrivals2, 0, U * 4));
  ck(cudaMemset(c->attend_arrivals, 0, U * 4));
  ck(cudaMemset(c->ctr_dev, 0, sizeof(Counters)));
  ck(cudaMemset(c->host_kv_dev, 0, G.R * 8));
  ck(cudaMemset(c->cap_dev, 0, G.R * 4));
  ck(cudaMemset(c->local_of, 0xFF, (size_t)L * U * G.nb_max * 4));
  ck(cudaMemset(c->local_used, 0, (size_t)L * U * 4));
  ck(cudaMemset(c->route, 0xFF, (size_t)L * U * G.kb * 4));
  ck(cudaMemset(c->local_kv_dev, 0, G.R * 8));
  ck(cudaMemset(c->local_cap_dev, 0xFF, G.R * 4));
  ck(cudaMemset(c->append_arrivals, 0, (size_t)L * G.R * 4));
  ck(cudaMemset(c->gather_work, 0, (size_t)L * 2 * 4));
  int lo = 0, hi = 0;
  ck(cudaDeviceGetStreamPriorityRange(&lo, &hi));
  // Three priority levels. Scoring and selection run on the internal select streams at the least
  // priority. The gather (copy stream) and okv_step's appends run at the greatest: the host link
  // is the longest pole of a step, so the gather must never wait for SMs. okv_step's own work
  // (the coefficients of every layer, then the attentions) runs on an internal stream between
  // the two, joined back to the caller's stream at the end of the step: the attention of a layer
  // then takes SMs before the background staging but after the gather. Measured on GB300
  // (interleaved pairs, median of three timed regions each):
  //   - 16K / b128: the same tok/s (12.37K against 12.43K median over four pairs), e2e higher in
  //     every pair (+1.4% to +8.2%), the attention's in-step share of the HBM peak 0.73-0.76
  //     against 0.56-0.58 on the caller's stream;
  //   - 32K / b32: +1.6% to +9.3% tok/s in three of three pairs;
  //   - at the greatest priority, beside the gather: the same tok/s but e2e 15-20% lower.
  // Alternatives: OKV_ATTEND_PRIORITY=caller (okv_step's work on the caller's stream),
  // OKV_ATTEND_PRIORITY=high (the greatest priority), OKV_STAGE_STREAM=caller (staging on the
  // caller's stream after the attention: 9.4K against 10.2K tok/s in an earlier build),
  // OKV_STAGE_PRIORITY=high (staging at the greatest priority: 8.2K).
  const char* pe = getenv("OKV_STAGE_PRIORITY");
  const int prio = (pe && strcmp(pe, "high") == 0) ? hi : lo;  // of the select stream
  const char* ps = getenv("OKV_STAGE_STREAM");
  c->stage_on_caller = ps && strcmp(ps, "caller") == 0;
  ck(cudaStreamCreateWithPriority(&c->sel_stream, cudaStreamNonBlocking, prio));
  if (c->scores2) ck(cudaStreamCreateWithPriority(&c->sel_stream2, cudaStreamNonBlocking, prio));
  const char* pa = getenv("OKV_ATTEND_PRIORITY");
  if (!(pa && strcmp(pa, "caller") == 0)) {
    const int mid = (pa && strcmp(pa, "high") == 0) ? hi : (lo + hi) / 2;  // e.g. -2 in [-5, 0]
    ck(cudaStreamCreateWithPriority(&c->att_stream, cudaStreamNonBlocking, mid));
  }
  ck(cudaStreamCreateWithPriority(&c->copy_stream, cudaStreamNonBlocking, hi));
  ck(cudaStreamCreateWithPriority(&c->app_stream, cudaStreamNonBlocking, hi));
  ck(cudaEventCreateWithFlags(&c->ev_in, cudaEventDisableTiming));
  for (auto& e : c->ev_step_read) ck(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
  for (auto& e : c->ev_step_read2) ck(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
  c->ev_selected.assign(G.L, nullptr);
  c->ev_staged.assign(G.L, nullptr);
  c->ev_appended.assign(G.L, nullptr);
  c->staged_once.assign(G.L, 0);
  for (int32_t l = 0; l < G.L; ++l) {
    ck(cudaEventCreateWithFlags(&c->ev_selected[l], cudaEventDisableTiming));
    ck(cudaEventCreateWithFlags(&c->ev_staged[l], cudaEventDisableTiming));
    ck(cudaEventCreateWithFlags(&c->ev_appended[l], cudaEventDisableTiming));
  }
  c->active.assign(G.R, 0);
  c->host_ptr.assign(G.R, nullptr);
  c->cap_blocks.assign(G.R, 0);
  c->local_ptr.assign(G.R, nullptr);
  c->local_cap.assign(G.R, -1);
  c->len_host.assign((size_t)G.L * G.R, 0);
  c->shared_buf.assign(G.R, 0);

  if (st == OKV_OK && okv::attend_uses_tensor_cores(G)) {
    // pool as rows of 256 bytes: dims {64 elements, 2 halves, rows}, box = one slot (32 rows)
    const uint64_t rows = (uint64_t)L * U * G.kb * 32;
    if (rows >= (1ull << 31)) {
      st = fail(c, OKV_EINVAL, "okv_create: slot pool too large for 32-bit TMA row coordinates");
    } else {
      typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess || !fn || q != cudaDriverEntryPointSuccess) {
        st = fail(c, OKV_ECUDA, "okv_create: cuTensorMapEncodeTiled unavailable");
      } else {
        const cuuint64_t dims[3] = {64, 2, rows};
        const cuuint64_t strides[2] = {128, 256};
        const cuuint32_t box[3] = {64, 2, 32};
        const cuuint32_t estr[3] = {1, 1, 1};
        CUresult r = ((EncodeFn)fn)(&c->pool_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, c->pool, dims, strides, box,
                                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS)
          st = fail(c, OKV_ECUDA, "okv_create: cuTensorMapEncodeTiled failed (%d)", (int)r);
        else
          c->have_map = true;
      }
    }
  }
  if (st == OKV_OK) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) st = fail(c, OKV_ECUDA, "okv_create: %s", cudaGetErrorString(e));
  }
  if (st != OKV_OK) {
    fprintf(stderr, "okv_create: %s\n", c->last_error.c_str());
    okv_destroy(c);
    return st;
  }
  *out = c;
  return OKV_OK;
}

}  // extern "C"

namespace {

// Device address of page-locked, device-mapped host memory, or nullptr.
void* mapped_device_pointer(void* p) {
  cudaPointerAttributes attr{};
  void* dptr = nullptr;
  // page-locked host memory only (on address-translation systems pageable memory would also be
  // reachable, but at the mercy of the OS pager)
  if (cudaPointerGetAttributes(&attr, p) != cudaSuccess || attr.type != cudaMemoryTypeHost ||
      cudaHostGetDevicePointer(&dptr, p, 0) != cudaSuccess || !dptr) {
    cudaGetLastError();
    return nullptr;
  }
  return dptr;
}

bool overlaps(const void* a, int64_t na, const void* b, int64_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + (uintptr_t)nb && y < x + (uintptr_t)na;
}

// local_cap < 0: a request that holds its full KV (okv_add_request); else partial staging.
okv_status add_request_impl(okv_ctx* c, const char* who, int32_t req, void* host_kv, int32_t capacity_blocks,
                            void* local_kv, int32_t local_cap, int32_t n_tokens, void* stream) {
  const Geom& G = c->G;
  cudaStream_t s = (cudaStream_t)stream;
  if (req < 0 || req >= G.R) return fail(c, OKV_EINVAL, "%s: request id %d out of range", who, req);
  if (c->active[req]) return fail(c, OKV_ESTATE, "%s: request %d is already active", who, req);
  if (!host_kv) return fail(c, OKV_EINVAL, "%s: host_kv is NULL", who);
  if (capacity_blocks <= 0 || capacity_blocks > G.nb_max)
    return fail(c, OKV_EINVAL, "%s: capacity_blocks %d not in 1..%d", who, capacity_blocks, G.nb_max);
  if (n_tokens < 0 || (int64_t)n_tokens > (int64_t)capacity_blocks * G.bs)
    return fail(c, OKV_EINVAL, "%s: n_tokens %d exceeds the capacity", who, n_tokens);
  void* dptr = mapped_device_pointer(host_kv);
  if (!dptr) return fail(c, OKV_EINVAL, "%s: host_kv is not page-locked, device-mapped memory", who);
  if ((reinterpret_cast<uintptr_t>(dptr) & 15) != 0) return fail(c, OKV_EINVAL, "%s: host_kv must be 16-byte aligned", who);
  const int64_t unit_bytes = (int64_t)G.L * G.Hkv * G.block_bytes;
  void* lptr = nullptr;
  if (local_cap >= 0) {
    if (local_cap > capacity_blocks)
      return fail(c, OKV_EINVAL, "%s: local_capacity_blocks %d not in 0..%d", who, local_cap, capacity_blocks);
    if (local_cap > 0) {
      if (!local_kv) return fail(c, OKV_EINVAL, "%s: local_kv is NULL", who);
      lptr = mapped_device_pointer(local_kv);
      if (!lptr) return fail(c, OKV_EINVAL, "%s: local_kv is not page-locked, device-mapped memory", who);
      if ((reinterpret_cast<uintptr_t>(lptr) & 15) != 0)
        return fail(c, OKV_EINVAL, "%s: local_kv must be 16-byte aligned", who);
      const int64_t lbytes = unit_bytes * local_cap;
      bool clash = overlaps(local_kv, lbytes, host_kv, unit_bytes * capacity_blocks);
      for (int32_t r : c->active_list) {
        clash = clash || overlaps(local_kv, lbytes, c->host_ptr[r], unit_bytes * c->cap_blocks[r]);
        if (c->local_cap[r] > 0) clash = clash || overlaps(local_kv, lbytes, c->local_ptr[r], unit_bytes * c->local_cap[r]);
      }
      if (clash) return fail(c, OKV_EINVAL, "%s: local_kv overlaps a buffer of an active request", who);
    }
  }
  for (int32_t r : c->active_list)
    if (c->local_cap[r] > 0 && overlaps(host_kv, unit_bytes * capacity_blocks, c->local_ptr[r], unit_bytes * c->local_cap[r]))
      return fail(c, OKV_EINVAL, "%s: host_kv overlaps the decode-side tier of request %d", who, r);
  // every earlier use of the context's tables must be complete before they are reset
  if (okv_status st = sync_internal(c)) return st;
  OKV_CUDA(c, cudaStreamSynchronize(s));

  // an active request registered with the same buffer and length has identical summaries
  int32_t twin = -1;
  for (int32_t r : c->active_list) {
    if (c->host_ptr[r] != host_kv || c->cap_blocks[r] != capacity_blocks) continue;
    bool same = true;
    for (int32_t l = 0; l < G.L && same; ++l) same = c->len_host[(size_t)l * G.R + r] == n_tokens;
    if (same) {
      twin = r;
      break;
    }
  }
  okv::StateBase B;
  B.slot_block = c->slot_block;
  B.stamp = c->stamp;
  B.n_sel = c->n_sel;
  B.n_fetch = c->n_fetch;
  B.len = c->len;
  B.local_of = c->local_of;
  B.local_used = c->local_used;
  B.host_kv_tab = c->host_kv_dev;
  B.local_kv_tab = c->local_kv_dev;
  B.cap_tab = c->cap_dev;
  B.local_cap_tab = c->local_cap_dev;
  okv::RequestInit q;
  q.req = req;
  q.n_tok = n_tokens;
  q.cap = capacity_blocks;
  q.local_cap = local_cap;
  q.host_kv = (uint64_t)(uintptr_t)dptr;
  q.local_kv = (uint64_t)(uintptr_t)lptr;
  OKV_CUDA(c, okv::launch_reset_request(G, B, q, s));
  c->launches += 1;
  if (twin >= 0) {
    const size_t bytes = (size_t)G.Hkv * G.nb_max * 2 * G.d * G.elem;
    for (int32_t l = 0; l < G.L; ++l) {
      uint8_t* base = c->summ + l * c->summ_layer_bytes;
      OKV_CUDA(c, cudaMemcpyAsync(base + (size_t)req * bytes, base + (size_t)twin * bytes, bytes,
                                  cudaMemcpyDeviceToDevice, s));
    }
  } else {
    Timer t(c, OKV_K_SUMMARY, s);
    OKV_CUDA(c, okv::launch_summary_build(G, 0, G.L, req, (uint64_t)(uintptr_t)dptr, capacity_blocks, n_tokens,
                                          c->summ, c->err_dev, s));
    t.stop(n_tokens > 0 ? 1 : 0);
  }
  OKV_CUDA(c, cudaStreamSynchronize(s));
  c->active[req] = 1;
  c->host_ptr[req] = host_kv;
  c->cap_blocks[req] = capacity_blocks;
  c->local_ptr[req] = local_cap > 0 ? local_kv : nullptr;
  c->local_cap[req] = local_cap;
  for (int32_t l = 0; l < G.L; ++l) c->len_host[(size_t)l * G.R + req] = n_tokens;
  if (okv_status st = upload_active(c)) return st;
  return check_device_error(c);
}

}  // namespace

extern "C" {

okv_status okv_add_request(okv_ctx* c, int32_t req, void* host_kv, int32_t capacity_blocks,
                           int32_t n_tokens, void* stream) {
  if (!c) return OKV_EINVAL;
  return add_request_impl(c, "okv_add_request", req, host_kv, capacity_blocks, nullptr, -1, n_tokens, stream);
}

okv_status okv_add_request_partial(okv_ctx* c, int32_t req, void* full_kv, int32_t capacity_blocks,
                                   void* local_kv, int32_t local_capacity_blocks, int32_t n_tokens, void* stream) {
  if (!c) return OKV_EINVAL;
  if (local_capacity_blocks < 0)
    return fail(c, OKV_EINVAL, "okv_add_request_partial: local_capacity_blocks %d is negative", local_capacity_blocks);
  return add_request_impl(c, "okv_add_request_partial", req, full_kv, capacity_blocks, local_kv,
                          local_capacity_blocks, n_tokens, stream);
}

okv_status okv_remove_request(okv_ctx* c, int32_t req) {
  if (!c) return OKV_EINVAL;
  if (req < 0 || req >= c->G.R) return fail(c, OKV_EINVAL, "okv_remove_request: request id %d out of range", req);
  if (!c->active[req]) return fail(c, OKV_ESTATE, "okv_remove_request: request %d is not active", req);
  if (okv_status st = sync_internal(c)) return st;
  OKV_CUDA(c, cudaDeviceSynchronize());
  c->active[req] = 0;
  c->host_ptr[req] = nullptr;
  c->local_ptr[req] = nullptr;
  c->local_cap[req] = -1;
  for (int32_t l = 0; l < c->G.L; ++l) c->len_host[(size_t)l * c->G.R + req] = 0;
  return upload_active(c);
}

}  // extern "C"

namespace {

okv_status append_check(okv_ctx* c, int32_t layer) {
  const Geom& G = c->G;
  if (layer < 0 || layer >= G.L) return fail(c, OKV_EINVAL, "okv_append: layer %d out of range", layer);
  for (int32_t r : c->active_list) {
    if (c->shared_buf[r])
      return fail(c, OKV_EINVAL, "okv_append: request %d shares its host buffer with another active request", r);
    const int32_t n = c->len_host[(size_t)layer * G.R + r];
    if ((int64_t)n >= (int64_t)c->cap_blocks[r] * G.bs)
      return fail(c, OKV_EINVAL, "okv_append: request %d is full at layer %d", r, layer);
  }
  return OKV_OK;
}

// Enqueue the append of one layer on `s`, after the layer's last staging (its gather may have
// written the tail block's slot and read the host block the append writes).
okv_status append_enqueue(okv_ctx* c, int32_t layer, const void* k_new, const void* v_new, cudaStream_t s) {
  const Geom& G = c->G;
  const int32_t n_active = (int32_t)c->active_list.size();
  if (n_active == 0) return OKV_OK;
  if (c->staged_once[layer]) OKV_CUDA(c, cudaStreamWaitEvent(s, c->ev_staged[layer], 0));
  const LayerState S = layer_state(c, layer);
  const ReqTables T = req_tables(c);
  Timer t(c, OKV_K_APPEND, s);
  OKV_CUDA(c, okv::launch_append(G, S, T, n_active, layer, k_new, v_new, c->append_arrivals + (size_t)layer * G.R,
                                 c->err_dev, s));
  t.stop(1);
  for (int32_t r : c->active_list) c->len_host[(size_t)layer * G.R + r] += 1;
  return OKV_OK;
}

}  // namespace

extern "C" {

okv_status okv_append(okv_ctx* c, int32_t layer, const void* k_new, const void* v_new, void* stream) {
  if (!c) return OKV_EINVAL;
  if (!k_new || !v_new) return fail(c, OKV_EINVAL, "okv_append: NULL input");
  if (okv_status st = append_check(c, layer)) return st;
  return append_enqueue(c, layer, k_new, v_new, (cudaStream_t)stream);
}

}  // extern "C"

namespace {

// `coef_ready`: the layer's scoring coefficients, already computed from the draft by okv_step
// (for every layer at once); NULL: compute them here from draft_q, on the caller's stream, so the
// caller may reuse its draft buffer. Only the caller's work so far is waited for.
okv_status stage_impl(okv_ctx* c, int32_t layer, const void* draft_q, const float* coef_ready, int32_t step,
                      float fetch_cap, void* stream) {
  const Geom& G = c->G;
  if (layer < 0 || layer >= G.L) return fail(c, OKV_EINVAL, "okv_stage: layer %d out of range", layer);
  if (!draft_q && !coef_ready) return fail(c, OKV_EINVAL, "okv_stage: NULL draft query");
  const float cap = fetch_cap < 0.f ? c->cfg.fetch_cap : fetch_cap;
  if (!(cap > 0.f) || cap > 1.f) return fail(c, OKV_EINVAL, "okv_stage: fetch cap %g not in (0, 1]", cap);
  const int32_t C = cap_to_blocks(cap, G.kb);
  const int32_t n_active = (int32_t)c->active_list.size();
  if (n_active == 0) return OKV_OK;
  cudaStream_t s = (cudaStream_t)stream;
  const LayerState S = layer_state(c, layer);
  const ReqTables T = req_tables(c);
  const bool lane2 = c->sel_stream2 && (layer & 1);
  cudaStream_t ss = lane2 ? c->sel_stream2 : c->sel_stream;
  uint32_t* scores_ws = lane2 ? c->scores2 : c->scores;
  int32_t* arrivals_ws = lane2 ? c->stage_arrivals2 : c->stage_arrivals;
  const float* coef = coef_ready;
  if (!coef_ready) {
    // the coefficients of this layer's draft, on the caller's stream after the previous staging of
    // this layer has read the layer's coefficient buffer
    float* dst = c->coef_buf + (size_t)layer * c->per_layer_units * 2 * G.d;
    if (c->staged_once[layer] && !c->stage_on_caller) OKV_CUDA(c, cudaStreamWaitEvent(s, c->ev_selected[layer], 0));
    {
      Timer t(c, OKV_K_COEF, s);
      OKV_CUDA(c, okv::launch_coef(G, c->active_dev, n_active, 1, draft_q, 0, dst, 0, s));
      t.stop(1);
    }
    coef = dst;
  }
  if (c->stage_on_caller) {
    // scoring and selection follow the caller's attention of this layer on its own stream
    ss = s;
    if (c->staged_once[layer]) OKV_CUDA(c, cudaStreamWaitEvent(s, c->ev_staged[layer], 0));
  } else {
    // scoring and selection follow the caller's work so far (its attention of this layer and the
    // coefficients)
    OKV_CUDA(c, cudaEventRecord(c->ev_in, s));
    OKV_CUDA(c, cudaStreamWaitEvent(ss, c->ev_in, 0));
    if (c->staged_once[layer]) OKV_CUDA(c, cudaStreamWaitEvent(ss, c->ev_staged[layer], 0));
  }
  {
    Timer t(c, OKV_K_SCORE_TOPK, ss);
    int n = 0;
    OKV_CUDA(c, okv::launch_stage(G, S, T, n_active, max_blocks_at(c, layer), coef, scores_ws, arrivals_ws, C,
                                  step, c->ctr_dev, c->err_dev, ss, &n));
    t.stop(n);
  }
  OKV_CUDA(c, cudaEventRecord(c->ev_selected[layer], ss));
  OKV_CUDA(c, cudaStreamWaitEvent(c->copy_stream, c->ev_selected[layer], 0));
  {
    Timer t(c, OKV_K_GATHER, c->copy_stream);
    OKV_CUDA(c, okv::launch_gather(G, S, T, n_active, layer, C, c->gather_work + 2 * layer, c->err_dev,
                                   c->copy_stream));
    t.stop(1);
  }
  OKV_CUDA(c, cudaEventRecord(c->ev_staged[layer], c->copy_stream));
  c->staged_once[layer] = 1;
  return OKV_OK;
}

}  // namespace

extern "C" {

okv_status okv_stage(okv_ctx* c, int32_t layer, const void* draft_q, int32_t step, float fetch_cap,
                     void* stream) {
  if (!c) return OKV_EINVAL;
  return stage_impl(c, layer, draft_q, nullptr, step, fetch_cap, stream);
}

namespace {

okv_status attend_impl(okv_ctx* c, const char* who, int32_t layer, const void* q, void* out, const void* dq,
                       void* dout, void* stream) {
  if (!c) return OKV_EINVAL;
  const Geom& G = c->G;
  if (layer < 0 || layer >= G.L) return fail(c, OKV_EINVAL, "%s: layer %d out of range", who, layer);
  if (!q || !out) return fail(c, OKV_EINVAL, "%s: NULL pointer", who);
  const int32_t n_active = (int32_t)c->active_list.size();
  if (n_active == 0) return OKV_OK;
  cudaStream_t s = (cudaStream_t)stream;
  if (c->staged_once[layer]) OKV_CUDA(c, cudaStreamWaitEvent(s, c->ev_staged[layer], 0));
  const LayerState S = layer_state(c, layer);
  const ReqTables T = req_tables(c);
  int n_launch = 0, split = 0;
  Timer t(c, OKV_K_ATTEND, s);
  OKV_CUDA(c, okv::launch_attend(G, S, T, n_active, layer, q, out, dq, dout, c->have_map ? &c->pool_map : nullptr,
                                 c->partials, c->partials_bytes, c->attend_arrivals, c->ctr_dev, c->err_dev, s,
                                 &n_launch, &split));
  t.stop(n_launch);
  return OKV_OK;
}

}  // namespace

okv_status okv_predict(okv_ctx* c, int32_t layer, const void* query, int32_t* counts, int32_t* ids, void* stream) {
  if (!c) return OKV_EINVAL;
  const Geom& G = c->G;
  if (layer < 0 || layer >= G.L) return fail(c, OKV_EINVAL, "okv_predict: layer %d out of range", layer);
  if (!query || !counts || !ids) return fail(c, OKV_EINVAL, "okv_predict: NULL pointer");
  const int32_t n_active = (int32_t)c->active_list.size();
  if (n_active == 0) return OKV_OK;
  cudaStream_t s = (cudaStream_t)stream;
  // the scoring workspace is shared with staging: run where staging runs, after the caller's work
  cudaStream_t ss = c->stage_on_caller ? s : c->sel_stream;
  if (!c->stage_on_caller) {
    OKV_CUDA(c, cudaEventRecord(c->ev_in, s));
    OKV_CUDA(c, cudaStreamWaitEvent(ss, c->ev_in, 0));
  }
  const LayerState S = layer_state(c, layer);
  const ReqTables T = req_tables(c);
  {
    Timer t(c, OKV_K_COEF, ss);
    OKV_CUDA(c, okv::launch_coef(G, c->active_dev, n_active, 1, query, 0, c->pred_coef, 0, ss));
    t.stop(1);
  }
  {
    Timer t(c, OKV_K_SCORE_TOPK, ss);
    int n = 0;
    OKV_CUDA(c, okv::launch_stage(G, S, T, n_active, max_blocks_at(c, layer), c->pred_coef, c->scores,
                                  c->stage_arrivals, 1, 0, c->ctr_dev, c->err_dev, ss, &n, ids, counts));
    t.stop(n);
  }
  if (!c->stage_on_caller) {
    OKV_CUDA(c, cudaEventRecord(c->ev_in, ss));
    OKV_CUDA(c, cudaStreamWaitEvent(s, c->ev_in, 0));
  }
  return OKV_OK;
}

okv_status okv_attend(okv_ctx* c, int32_t layer, const void* q, void* out, void* stream) {
  return attend_impl(c, "okv_attend", layer, q, out, nullptr, nullptr, stream);
}

okv_status okv_attend_lookahead(okv_ctx* c, int32_t layer, const void* q, const void* draft_q, void* out,
                                void* draft_out, void* stream) {
  if (c && (!draft_q || !draft_out)) return fail(c, OKV_EINVAL, "okv_attend_lookahead: NULL draft pointer");
  return attend_impl(c, "okv_attend_lookahead", layer, q, out, draft_q, draft_out, stream);
}

okv_status okv_step(okv_ctx* c, const void* q, const void* draft_q, void* out, const void* k_new,
                    const void* v_new, int32_t step, float fetch_cap, void* stream) {
  if (!c) return OKV_EINVAL;
  if (!q || !draft_q || !out) return fail(c, OKV_EINVAL, "okv_step: NULL pointer");
  if ((k_new == nullptr) != (v_new == nullptr)) return fail(c, OKV_EINVAL, "okv_step: k_new and v_new go together");
  const Geom& G = c->G;
  const size_t qbytes = (size_t)G.R * G.Hq * G.d * G.elem;
  const size_t kvbytes = (size_t)G.R * G.Hkv * G.d * G.elem;
  cudaStream_t s = (cudaStream_t)stream;
  // The scoring coefficients of every layer's draft in one launch, into the half of step_coef
  // the step before last used (its stagings have read it long since), instead of one launch per
  // layer on the caller's stream; the caller may then reuse draft_q.
  // The step's own work (coefficients, attentions, the staging's waits on them) runs on the
  // internal attention stream (above the staging, below the gather), which first takes up the
  // caller's work so far and which the caller's stream waits for at the end; with
  // OKV_ATTEND_PRIORITY=caller it runs on the caller's stream itself.
  cudaStream_t as = s;
  if (c->att_stream) {
    OKV_CUDA(c, cudaEventRecord(c->ev_in, s));
    OKV_CUDA(c, cudaStreamWaitEvent(c->att_stream, c->ev_in, 0));
    as = c->att_stream;
  }
  const int p = c->step_parity;
  const size_t cstride = (size_t)c->per_layer_units * 2 * G.d;  // floats of one layer
  float* coefs = c->step_coef + (size_t)p * G.L * cstride;
  if (c->step_used[p]) {
    OKV_CUDA(c, cudaStreamWaitEvent(as, c->ev_step_read[p], 0));
    if (c->sel_stream2) OKV_CUDA(c, cudaStreamWaitEvent(as, c->ev_step_read2[p], 0));
  }
  {
    Timer t(c, OKV_K_COEF, as);
    OKV_CUDA(c, okv::launch_coef(G, c->active_dev, (int32_t)c->active_list.size(), G.L, draft_q,
                                 (int64_t)G.R * G.Hq * G.d, coefs, (int64_t)cstride, as));
    t.stop(c->active_list.empty() ? 0 : 1);
  }
  c->step_parity ^= 1;
  const uint8_t* drafts = (const uint8_t*)draft_q;
  if (k_new) {
    // Every layer's append goes on the append stream at once, each after its layer's last
    // staging; the caller's stream waits for a layer's append only before that layer's attention.
    for (int32_t l = 0; l < G.L; ++l)
      if (okv_status st = append_check(c, l)) return st;
    OKV_CUDA(c, cudaEventRecord(c->ev_in, as));  // k_new / v_new are ready
    OKV_CUDA(c, cudaStreamWaitEvent(c->app_stream, c->ev_in, 0));
    for (int32_t l = 0; l < G.L; ++l) {
      okv_status st = append_enqueue(c, l, (const uint8_t*)k_new + l * kvbytes, (const uint8_t*)v_new + l * kvbytes,
                                     c->app_stream);
      if (st != OKV_OK) return st;
      OKV_CUDA(c, cudaEventRecord(c->ev_appended[l], c->app_stream));
    }
  }
  for (int32_t l = 0; l < G.L; ++l) {
    if (k_new) OKV_CUDA(c, cudaStreamWaitEvent(as, c->ev_appended[l], 0));
    okv_status st = okv_attend(c, l, (const uint8_t*)q + l * qbytes, (uint8_t*)out + l * qbytes, as);
    if (st != OKV_OK) return st;
    st = stage_impl(c, l, drafts + l * qbytes, coefs + (size_t)l * cstride, step, fetch_cap, as);
    if (st != OKV_OK) return st;
  }
  if (c->att_stream) {
    OKV_CUDA(c, cudaEventRecord(c->ev_in, as));
    OKV_CUDA(c, cudaStreamWaitEvent(s, c->ev_in, 0));
  }
  OKV_CUDA(c, cudaEventRecord(c->ev_step_read[p], c->sel_stream));
  if (c->sel_stream2) OKV_CUDA(c, cudaEventRecord(c->ev_step_read2[p], c->sel_stream2));
  c->step_used[p] = true;
  return OKV_OK;
}

okv_status okv_join(okv_ctx* c, void* stream) {
  if (!c) return OKV_EINVAL;
  cudaStream_t s = (cudaStream_t)stream;
  OKV_CUDA(c, cudaEventRecord(c->ev_in, c->app_stream));
  OKV_CUDA(c, cudaStreamWaitEvent(s, c->ev_in, 0));
  OKV_CUDA(c, cudaEventRecord(c->ev_in, c->sel_stream));
  OKV_CUDA(c, cudaStreamWaitEvent(s, c->ev_in, 0));
  if (c->sel_stream2) {
    OKV_CUDA(c, cudaEventRecord(c->ev_in, c->sel_stream2));
    OKV_CUDA(c, cudaStreamWaitEvent(s, c->ev_in, 0));
  }
  if (c->att_stream) {
    OKV_CUDA(c, cudaEventRecord(c->ev_in, c->att_stream));
    OKV_CUDA(c, cudaStreamWaitEvent(s, c->ev_in, 0));
  }
  OKV_CUDA(c, cudaEventRecord(c->ev_in, c->copy_stream));
  OKV_CUDA(c, cudaStreamWaitEvent(s, c->ev_in, 0));
  return OKV_OK;
}

okv_status okv_sync(okv_ctx* c, int64_t timeout_ms) {
  if (!c) return OKV_EINVAL;
  // one event at the end of each internal stream (staging, gather, appends of okv_step)
  cudaStream_t streams[5] = {c->sel_stream, c->copy_stream, c->app_stream, nullptr, nullptr};
  int ns = 3;
  if (c->sel_stream2) streams[ns++] = c->sel_stream2;
  if (c->att_stream) streams[ns++] = c->att_stream;
  cudaEvent_t ev[5] = {nullptr, nullptr, nullptr, nullptr, nullptr};
  for (int i = 0; i < ns; ++i) {
    OKV_CUDA(c, cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming));
    OKV_CUDA(c, cudaEventRecord(ev[i], streams[i]));
  }
  const auto t0 = std::chrono::steady_clock::now();
  okv_status st = OKV_OK;
  for (;;) {
    bool done = true;
    cudaError_t bad = cudaSuccess;
    for (int i = 0; i < ns; ++i) {
      const cudaError_t q = cudaEventQuery(ev[i]);
      if (q == cudaErrorNotReady) done = false;
      else if (q != cudaSuccess) bad = q;
    }
    if (bad != cudaSuccess) {
      st = fail(c, OKV_ECUDA, "okv_sync: %s", cudaGetErrorString(bad));
      break;
    }
    if (done) break;
    const auto ms = std::chrono::duration_cast<std::chrono::milliseconds>(std::chrono::steady_clock::now() - t0).count();
    if (timeout_ms >= 0 && ms > timeout_ms) {
      st = fail(c, OKV_ETIMEOUT, "okv_sync: work still running after %lld ms", (long long)timeout_ms);
      break;
    }
    std::this_thread::sleep_for(std::chrono::microseconds(50));
  }
  for (auto e : ev)
    if (e) cudaEventDestroy(e);
  if (st != OKV_OK) return st;
  return check_device_error(c);
}

okv_status okv_read_summaries(okv_ctx* c, int32_t layer, int32_t req, void* out) {
  if (!c || !out) return OKV_EINVAL;
  const Geom& G = c->G;
  if (layer < 0 || layer >= G.L || req < 0 || req >= G.R) return fail(c, OKV_EINVAL, "okv_read_summaries: range");
  if (okv_status st = sync_internal(c)) return st;
  const size_t bytes = (size_t)G.Hkv * G.nb_max * 2 * G.d * G.elem;
  OKV_CUDA(c, cudaMemcpy(out, c->summ + layer * c->summ_layer_bytes + (size_t)req * bytes, bytes, cudaMemcpyDeviceToHost));
  return check_device_error(c);
}

okv_status okv_read_selection(okv_ctx* c, int32_t layer, int32_t* counts, int32_t* ids, float* scores) {
  if (!c) return OKV_EINVAL;
  const Geom& G = c->G;
  if (layer < 0 || layer >= G.L) return fail(c, OKV_EINVAL, "okv_read_selection: layer out of range");
  if (okv_status st = sync_internal(c)) return st;
  const LayerState S = layer_state(c, layer);
  const int64_t U = c->per_layer_units;
  if (counts) OKV_CUDA(c, cudaMemcpy(counts, S.n_sel, U * 4, cudaMemcpyDeviceToHost));
  if (ids) OKV_CUDA(c, cudaMemcpy(ids, S.sel_ids, U * G.kb * 4, cudaMemcpyDeviceToHost));
  if (scores) OKV_CUDA(c, cudaMemcpy(scores, S.sel_scores, U * G.kb * 4, cudaMemcpyDeviceToHost));
  return check_device_error(c);
}

okv_status okv_read_slot_table(okv_ctx* c, int32_t layer, int32_t* slot_block, int32_t* stamps) {
  if (!c) return OKV_EINVAL;
  const Geom& G = c->G;
  if (layer < 0 || layer >= G.L) return fail(c, OKV_EINVAL, "okv_read_slot_table: layer out of range");
  if (okv_status st = sync_internal(c)) return st;
  const LayerState S = layer_state(c, layer);
  const int64_t U = c->per_layer_units;
  if (slot_block) OKV_CUDA(c, cudaMemcpy(slot_block, S.slot_block, U * G.kb * 4, cudaMemcpyDeviceToHost));
  if (stamps) OKV_CUDA(c, cudaMemcpy(stamps, S.stamp, U * G.kb * 4, cudaMemcpyDeviceToHost));
  return check_device_error(c);
}

okv_status okv_read_fetch_list(okv_ctx* c, int32_t layer, int32_t* counts, int32_t* entries) {
  if (!c) return OKV_EINVAL;
  const Geom& G = c->G;
  if (layer < 0 || layer >= G.L) return fail(c, OKV_EINVAL, "okv_read_fetch_list: layer out of range");
  if (okv_status st = sync_internal(c)) return st;
  const LayerState S = layer_state(c, layer);
  const int64_t U = c->per_layer_units;
  if (counts) OKV_CUDA(c, cudaMemcpy(counts, S.n_fetch, U * 4, cudaMemcpyDeviceToHost));
  if (entries) OKV_CUDA(c, cudaMemcpy(entries, S.fetch, U * G.kb * 8, cudaMemcpyDeviceToHost));
  return check_device_error(c);
}

okv_status okv_read_pool(okv_ctx* c, int32_t layer, int32_t req, int32_t kv_head, void* out) {
  if (!c || !out) return OKV_EINVAL;
  const Geom& G = c->G;
  if (layer < 0 || layer >= G.L || req < 0 || req >= G.R || kv_head < 0 || kv_head >= G.Hkv)
    return fail(c, OKV_EINVAL, "okv_read_pool: range");
  if (okv_status st = sync_internal(c)) return st;
  const LayerState S = layer_state(c, layer);
  const size_t bytes = (size_t)G.kb * G.block_bytes;
  OKV_CUDA(c, cudaMemcpy(out, S.pool + ((size_t)req * G.Hkv + kv_head) * bytes, bytes, cudaMemcpyDeviceToHost));
  return check_device_error(c);
}

okv_status okv_read_lengths(okv_ctx* c, int32_t layer, int32_t* lengths) {
  if (!c || !lengths) return OKV_EINVAL;
  const Geom& G = c->G;
  if (layer < 0 || layer >= G.L) return fail(c, OKV_EINVAL, "okv_read_lengths: layer out of range");
  if (okv_status st = sync_internal(c)) return st;
  OKV_CUDA(c, cudaMemcpy(lengths, c->len + (size_t)layer * G.R, G.R * 4, cudaMemcpyDeviceToHost));
  for (int32_t r = 0; r < G.R; ++r)
    if (!c->active[r]) lengths[r] = 0;
  return check_device_error(c);
}

okv_status okv_read_local(okv_ctx* c, int32_t layer, int32_t* local_used, int32_t* local_of, int32_t* routes) {
  if (!c) return OKV_EINVAL;
  const Geom& G = c->G;
  if (layer < 0 || layer >= G.L) return fail(c, OKV_EINVAL, "okv_read_local: layer out of range");
  if (okv_status st = sync_internal(c)) return st;
  const LayerState S = layer_state(c, layer);
  const int64_t U = c->per_layer_units;
  if (local_used) OKV_CUDA(c, cudaMemcpy(local_used, S.local_used, U * 4, cudaMemcpyDeviceToHost));
  if (local_of) OKV_CUDA(c, cudaMemcpy(local_of, S.local_of, U * G.nb_max * 4, cudaMemcpyDeviceToHost));
  if (routes) OKV_CUDA(c, cudaMemcpy(routes, S.route, U * G.kb * 4, cudaMemcpyDeviceToHost));
  return check_device_error(c);
}

okv_status okv_set_timing(okv_ctx* c, int32_t enable) {
  if (!c) return OKV_EINVAL;
  if (okv_status st = sync_internal(c)) return st;
  OKV_CUDA(c, cudaDeviceSynchronize());
  for (auto& t : c->pending) {
    c->event_pool.push_back(t.a);
    c->event_pool.push_back(t.b);
  }
  c->pending.clear();
  for (int k = 0; k < OKV_K_COUNT; ++k) {
    c->ms[k] = 0.0;
    c->n_launch_kind[k] = 0;
  }
  OKV_CUDA(c, cudaMemset(c->ctr_dev, 0, sizeof(Counters)));
  c->timing = enable != 0;
  return OKV_OK;
}

okv_status okv_read_timing(okv_ctx* c, okv_timing* out) {
  if (!c || !out) return OKV_EINVAL;
  for (auto& t : c->pending) {
    OKV_CUDA(c, cudaEventSynchronize(t.b));
    float ms = 0.f;
    OKV_CUDA(c, cudaEventElapsedTime(&ms, t.a, t.b));
    c->ms[t.kind] += ms;
    c->event_pool.push_back(t.a);
    c->event_pool.push_back(t.b);
  }
  c->pending.clear();
  Counters h{};
  OKV_CUDA(c, cudaMemcpy(&h, c->ctr_dev, sizeof(h), cudaMemcpyDeviceToHost));
  for (int k = 0; k < OKV_K_COUNT; ++k) {
    out->ms[k] = c->ms[k];
    out->launches[k] = c->n_launch_kind[k];
  }
  out->fetched_blocks = (int64_t)h.fetched_blocks;
  out->attended_slots = (int64_t)h.attended_slots;
  out->local_hits = (int64_t)h.local_hits;
  out->local_fills = (int64_t)h.local_fills;
  out->full_reads = (int64_t)h.full_reads;
  return OKV_OK;
}

int64_t okv_launch_count(const okv_ctx* c) { return c ? c->launches : 0; }

}  // extern "C"
