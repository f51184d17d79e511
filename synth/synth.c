/*
 * Seeded synthetic workload for the lookahead sparse KV staging path.
 * See synth.h for the definitions. Plain C99 + pthreads; no architecture-specific code.
 */
#include "synth.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

enum { ST_K = 1, ST_V = 2, ST_DIR = 3, ST_QNOISE = 4, ST_DNOISE = 5, ST_PLANT = 6, ST_TEST = 7 };

/* SplitMix64 output function applied to one counter value. */
static uint64_t sm64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static uint64_t chain(uint64_t seed, uint64_t stream, uint64_t a, uint64_t b, uint64_t c,
                      uint64_t d) {
  uint64_t k = sm64(seed);
  k = sm64(k ^ stream);
  k = sm64(k ^ a);
  k = sm64(k ^ b);
  k = sm64(k ^ c);
  k = sm64(k ^ d);
  return k;
}

/* Two standard normals from one 64-bit hash (Box-Muller on two 24-bit uniforms). */
static void normal_pair(uint64_t w, double* z0, double* z1) {
  /* binary32 arithmetic: the values are stored as binary32 or bfloat16 */
  const float inv24 = 1.0f / 16777216.0f;
  float u1 = ((float)(uint32_t)(w >> 40) + 0.5f) * inv24; /* (0, 1) */
  float u2 = (float)(uint32_t)(w & 0xFFFFFFull) * inv24;  /* [0, 1) */
  float r = sqrtf(-2.0f * logf(u1));
  float a = 6.2831853071795864769f * u2;
  *z0 = (double)(r * cosf(a));
  *z1 = (double)(r * sinf(a));
}

static double normal_at(uint64_t base, int64_t c) {
  double z0, z1;
  normal_pair(sm64(base ^ (uint64_t)(c >> 1)), &z0, &z1);
  return (c & 1) ? z1 : z0;
}

int synth_dtype_size(int32_t dtype) {
  return dtype == SYNTH_F32 ? 4 : (dtype == SYNTH_BF16 ? 2 : 0);
}

static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

static void store(void* base, int32_t dtype, int64_t i, double x) {
  float f = (float)x;
  if (dtype == SYNTH_F32)
    ((float*)base)[i] = f;
  else
    ((uint16_t*)base)[i] = f32_to_bf16_rne(f);
}

static int check_params(const synth_params* p) {
  if (!p) return -1;
  if (p->layers <= 0 || p->q_heads <= 0 || p->kv_heads <= 0 || p->head_dim <= 0 ||
      p->block_size <= 0 || p->q_heads % p->kv_heads != 0)
    return -1;
  if (synth_dtype_size(p->dtype) == 0) return -1;
  if (p->n_dirs <= 0 || p->n_active < 0 || p->active_period <= 0) return -1;
  if (p->plant_mode != SYNTH_PLANT_MOD && p->plant_mode != SYNTH_PLANT_COUNT) return -1;
  if (p->plant_mode == SYNTH_PLANT_COUNT && (p->n_plant < 0 || p->plant_blocks < 0)) return -1;
  return 0;
}

int synth_direction(double* out, const synth_params* p, int32_t layer, int32_t req_key,
                    int32_t kv_head, int32_t j) {
  if (check_params(p) || !out) return -1;
  const int d = p->head_dim;
  uint64_t base = chain(p->seed, ST_DIR, (uint64_t)layer, (uint64_t)req_key, (uint64_t)kv_head,
                        (uint64_t)j);
  double nrm = 0.0;
  for (int c = 0; c < d; ++c) {
    out[c] = normal_at(base, c);
    nrm += out[c] * out[c];
  }
  nrm = sqrt(nrm);
  for (int c = 0; c < d; ++c) out[c] /= nrm;
  return 0;
}

/* Per-block direction table of one (layer, req_key, kv_head): dirs[b] for b < nb. */
static void block_directions(const synth_params* p, int32_t layer, int32_t req_key,
                             int32_t kv_head, int32_t nb, int32_t* dirs) {
  if (p->plant_mode == SYNTH_PLANT_MOD) {
    for (int32_t b = 0; b < nb; ++b) dirs[b] = b % p->n_dirs;
    return;
  }
  for (int32_t b = 0; b < nb; ++b) dirs[b] = -1;
  const int32_t pb = p->plant_blocks;
  if (pb <= 0 || p->n_plant <= 0) return;
  /* rank of each candidate block by (hash, block) ascending */
  uint64_t* h = (uint64_t*)malloc(sizeof(uint64_t) * (size_t)pb);
  for (int32_t b = 0; b < pb; ++b)
    h[b] = chain(p->seed, ST_PLANT, (uint64_t)layer, (uint64_t)req_key, (uint64_t)kv_head,
                 (uint64_t)b);
  for (int32_t b = 0; b < pb && b < nb; ++b) {
    int32_t rank = 0;
    for (int32_t o = 0; o < pb; ++o)
      if (h[o] < h[b] || (h[o] == h[b] && o < b)) ++rank;
    if (rank < p->n_plant) dirs[b] = (int32_t)(sm64(h[b]) % (uint64_t)p->n_dirs);
  }
  free(h);
}

int32_t synth_block_direction(const synth_params* p, int32_t layer, int32_t req_key,
                              int32_t kv_head, int32_t block) {
  if (check_params(p) || block < 0) return -1;
  if (p->plant_mode == SYNTH_PLANT_MOD) return block % p->n_dirs;
  int32_t nb = block + 1;
  int32_t* dirs = (int32_t*)malloc(sizeof(int32_t) * (size_t)nb);
  block_directions(p, layer, req_key, kv_head, nb, dirs);
  int32_t j = dirs[block];
  free(dirs);
  return j;
}

/* ---- KV fill --------------------------------------------------------------------------- */

typedef struct {
  void* buf;
  const synth_params* p;
  int32_t req_key, tok_begin, tok_end, cap_blocks;
  int32_t layer_begin; /* first layer written; buf starts at that layer */
  int32_t n_items;     /* (layers written) * kv_heads */
  int32_t tid, n_threads;
} fill_job;

static void fill_unit(const fill_job* J, int32_t layer, int32_t h) {
  const synth_params* p = J->p;
  const int d = p->head_dim, bs = p->block_size;
  const int64_t unit_elems = (int64_t)J->cap_blocks * 2 * bs * d;
  const int64_t unit_off = ((int64_t)(layer - J->layer_begin) * p->kv_heads + h) * unit_elems;
  const int32_t nb_used = (J->tok_end + bs - 1) / bs;
  int32_t* dirs = (int32_t*)malloc(sizeof(int32_t) * (size_t)(nb_used > 0 ? nb_used : 1));
  block_directions(p, layer, J->req_key, h, nb_used, dirs);
  double* u = (double*)malloc(sizeof(double) * (size_t)p->n_dirs * d);
  for (int j = 0; j < p->n_dirs; ++j) synth_direction(u + (size_t)j * d, p, layer, J->req_key, h, j);
  for (int32_t t = J->tok_begin; t < J->tok_end; ++t) {
    const int32_t b = t / bs, i = t % bs;
    const int32_t j = dirs[b];
    uint64_t bk = chain(p->seed, ST_K, (uint64_t)layer, (uint64_t)J->req_key, (uint64_t)h, (uint64_t)t);
    uint64_t bv = chain(p->seed, ST_V, (uint64_t)layer, (uint64_t)J->req_key, (uint64_t)h, (uint64_t)t);
    int64_t ko = unit_off + (((int64_t)b * 2 + 0) * bs + i) * d;
    int64_t vo = unit_off + (((int64_t)b * 2 + 1) * bs + i) * d;
    for (int c = 0; c < d; c += 2) {
      double k0, k1, v0, v1;
      normal_pair(sm64(bk ^ (uint64_t)(c >> 1)), &k0, &k1);
      normal_pair(sm64(bv ^ (uint64_t)(c >> 1)), &v0, &v1);
      if (j >= 0) {
        k0 += p->amplitude * u[(size_t)j * d + c];
        if (c + 1 < d) k1 += p->amplitude * u[(size_t)j * d + c + 1];
      }
      store(J->buf, p->dtype, ko + c, k0);
      store(J->buf, p->dtype, vo + c, v0);
      if (c + 1 < d) {
        store(J->buf, p->dtype, ko + c + 1, k1);
        store(J->buf, p->dtype, vo + c + 1, v1);
      }
    }
  }
  free(u);
  free(dirs);
}

static void* fill_worker(void* arg) {
  fill_job* J = (fill_job*)arg;
  for (int32_t it = J->tid; it < J->n_items; it += J->n_threads)
    fill_unit(J, J->layer_begin + it / J->p->kv_heads, it % J->p->kv_heads);
  return NULL;
}

static int fill_layers(void* buf, const synth_params* p, int32_t req_key, int32_t layer_begin,
                       int32_t n_layers, int32_t tok_begin, int32_t tok_end, int32_t cap_blocks,
                       int32_t n_threads) {
  if (check_params(p) || !buf || tok_begin < 0 || tok_end < tok_begin ||
      (int64_t)cap_blocks * p->block_size < tok_end)
    return -1;
  if (n_threads < 1) n_threads = 1;
  const int32_t n_items = n_layers * p->kv_heads;
  if (n_threads > n_items) n_threads = n_items;
  fill_job* jobs = (fill_job*)malloc(sizeof(fill_job) * (size_t)n_threads);
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)n_threads);
  for (int t = 0; t < n_threads; ++t) {
    fill_job J = {buf, p, req_key, tok_begin, tok_end, cap_blocks, layer_begin, n_items, t, n_threads};
    jobs[t] = J;
  }
  for (int t = 1; t < n_threads; ++t) pthread_create(&th[t], NULL, fill_worker, &jobs[t]);
  fill_worker(&jobs[0]);
  for (int t = 1; t < n_threads; ++t) pthread_join(th[t], NULL);
  free(th);
  free(jobs);
  return 0;
}

int synth_fill_kv(void* buf, const synth_params* p, int32_t req_key, int32_t tok_begin,
                  int32_t tok_end, int32_t cap_blocks, int32_t n_threads) {
  if (check_params(p)) return -1;
  return fill_layers(buf, p, req_key, 0, p->layers, tok_begin, tok_end, cap_blocks, n_threads);
}

int synth_fill_kv_layer(void* buf, const synth_params* p, int32_t req_key, int32_t layer,
                        int32_t tok_begin, int32_t tok_end, int32_t cap_blocks, int32_t n_threads) {
  if (check_params(p) || layer < 0 || layer >= p->layers) return -1;
  return fill_layers(buf, p, req_key, layer, 1, tok_begin, tok_end, cap_blocks, n_threads);
}

/* ---- queries ----------------------------------------------------------------------------- */

static int64_t floor_div(int64_t a, int64_t b) {
  int64_t q = a / b;
  if ((a % b != 0) && ((a < 0) != (b < 0))) --q;
  return q;
}

/* normalize(sum of the active directions of step s) into dir[d] */
static void active_direction(const synth_params* p, int32_t layer, int32_t req_key, int32_t h,
                             int32_t s, double* dir, double* tmp) {
  const int d = p->head_dim;
  for (int c = 0; c < d; ++c) dir[c] = 0.0;
  int64_t w = floor_div(s, p->active_period);
  for (int i = 0; i < p->n_active; ++i) {
    int64_t j = (w + i) % p->n_dirs;
    if (j < 0) j += p->n_dirs;
    synth_direction(tmp, p, layer, req_key, h, (int32_t)j);
    for (int c = 0; c < d; ++c) dir[c] += tmp[c];
  }
  double nrm = 0.0;
  for (int c = 0; c < d; ++c) nrm += dir[c] * dir[c];
  nrm = sqrt(nrm);
  if (nrm > 0.0)
    for (int c = 0; c < d; ++c) dir[c] /= nrm;
}

typedef struct {
  void* out;
  const synth_params* p;
  int32_t layer, step, kind, batch;
  const int32_t *req_ids, *req_keys;
  int32_t tid, n_threads;
} query_job;

static void* query_worker(void* arg) {
  query_job* J = (query_job*)arg;
  const synth_params* p = J->p;
  const int d = p->head_dim, hq_n = p->q_heads, g = p->q_heads / p->kv_heads;
  double* dir = (double*)malloc(sizeof(double) * (size_t)d);
  double* tmp = (double*)malloc(sizeof(double) * (size_t)d);
  const int32_t qstep = J->kind == 0 ? J->step : J->step + 1;
  for (int32_t i = J->tid; i < J->batch; i += J->n_threads) {
    const int32_t rid = J->req_ids[i], rkey = J->req_keys[i];
    for (int hq = 0; hq < hq_n; ++hq) {
      const int h = hq / g;
      active_direction(p, J->layer, rkey, h, qstep, dir, tmp);
      uint64_t bq = chain(p->seed, ST_QNOISE, (uint64_t)(int64_t)qstep, (uint64_t)J->layer,
                          (uint64_t)rid, (uint64_t)hq);
      uint64_t bd = chain(p->seed, ST_DNOISE, (uint64_t)(int64_t)J->step, (uint64_t)J->layer,
                          (uint64_t)rid, (uint64_t)hq);
      const int64_t o = ((int64_t)i * hq_n + hq) * d;
      for (int c = 0; c < d; ++c) {
        double x = dir[c] + p->sigma_q * normal_at(bq, c);
        if (J->kind == 1) x += p->sigma_d * normal_at(bd, c);
        store(J->out, p->dtype, o + c, x);
      }
    }
  }
  free(tmp);
  free(dir);
  return NULL;
}

int synth_queries(void* out, const synth_params* p, int32_t layer, int32_t step, int32_t kind,
                  int32_t batch, const int32_t* req_ids, const int32_t* req_keys,
                  int32_t n_threads) {
  if (check_params(p) || !out || !req_ids || !req_keys || batch < 0 || (kind != 0 && kind != 1))
    return -1;
  if (n_threads < 1) n_threads = 1;
  if (n_threads > batch) n_threads = batch > 0 ? batch : 1;
  query_job* jobs = (query_job*)malloc(sizeof(query_job) * (size_t)n_threads);
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)n_threads);
  for (int t = 0; t < n_threads; ++t) {
    query_job J = {out, p, layer, step, kind, batch, req_ids, req_keys, t, n_threads};
    jobs[t] = J;
  }
  for (int t = 1; t < n_threads; ++t) pthread_create(&th[t], NULL, query_worker, &jobs[t]);
  query_worker(&jobs[0]);
  for (int t = 1; t < n_threads; ++t) pthread_join(th[t], NULL);
  free(th);
  free(jobs);
  return 0;
}

int synth_token_kv(void* out_k, void* out_v, const synth_params* p, int32_t layer,
                   int32_t batch, const int32_t* req_keys, const int32_t* positions) {
  if (check_params(p) || !out_k || !out_v || !req_keys || !positions || batch < 0) return -1;
  const int d = p->head_dim, bs = p->block_size;
  double* u = (double*)malloc(sizeof(double) * (size_t)d);
  for (int32_t i = 0; i < batch; ++i) {
    const int32_t t = positions[i];
    if (t < 0) { free(u); return -1; }
    for (int h = 0; h < p->kv_heads; ++h) {
      const int32_t j = synth_block_direction(p, layer, req_keys[i], h, t / bs);
      if (j >= 0) synth_direction(u, p, layer, req_keys[i], h, j);
      uint64_t bk = chain(p->seed, ST_K, (uint64_t)layer, (uint64_t)req_keys[i], (uint64_t)h, (uint64_t)t);
      uint64_t bv = chain(p->seed, ST_V, (uint64_t)layer, (uint64_t)req_keys[i], (uint64_t)h, (uint64_t)t);
      const int64_t o = ((int64_t)i * p->kv_heads + h) * d;
      for (int c = 0; c < d; ++c) {
        double k = normal_at(bk, c) + (j >= 0 ? p->amplitude * u[c] : 0.0);
        store(out_k, p->dtype, o + c, k);
        store(out_v, p->dtype, o + c, normal_at(bv, c));
      }
    }
  }
  free(u);
  return 0;
}

int synth_normals(double* out, int64_t n, uint64_t seed, uint64_t stream, uint64_t a, uint64_t b) {
  if (!out || n < 0) return -1;
  uint64_t base = chain(seed, ST_TEST + stream, a, b, 0, 0);
  for (int64_t i = 0; i < n; ++i) out[i] = normal_at(base, i);
  return 0;
}
