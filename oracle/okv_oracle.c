/*
 * ORACLE: test infrastructure, not product code (see okv_oracle.h).
 *
 * Plain binary64 restatement of one decode step of OasisKV's lookahead sparse KV
 * staging, following "4 System Design" of paperlayer.ai/abs/2608.08097v1 and the
 * sizing of "2 Background". Where the pages leave a step open, the plainest reading
 * is taken and named at the function.
 */
#include "okv_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ---- storage access ----------------------------------------------------------------------- */

static double load(const void* base, int32_t dtype, int64_t i) {
  if (dtype == ORACLE_F32) return (double)((const float*)base)[i];
  uint32_t u = (uint32_t)((const uint16_t*)base)[i] << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* copy one stored element's bit pattern (min and max pick one of their inputs) */
static void copy_elem(void* dst, int64_t di, const void* src, int64_t si, int32_t dtype) {
  if (dtype == ORACLE_F32)
    ((float*)dst)[di] = ((const float*)src)[si];
  else
    ((uint16_t*)dst)[di] = ((const uint16_t*)src)[si];
}

/* element offsets inside one unit's host region [cap_blocks][2][bs][d] */
static int64_t k_off(int32_t b, int32_t t, int32_t c, int32_t bs, int32_t d) {
  return (((int64_t)b * 2 + 0) * bs + t) * d + c;
}
static int64_t v_off(int32_t b, int32_t t, int32_t c, int32_t bs, int32_t d) {
  return (((int64_t)b * 2 + 1) * bs + t) * d + c;
}

static int32_t n_blocks(int32_t n_tok, int32_t bs) { return (n_tok + bs - 1) / bs; }

/* valid tokens of block b of a context of n_tok tokens */
static int32_t valid_in_block(int32_t b, int32_t n_tok, int32_t bs) {
  int32_t n = n_tok - b * bs;
  return n < 0 ? 0 : (n > bs ? bs : n);
}

/* ---- sizing ("2 Background", KV-cache pressure) ------------------------------------------- */

/* One token stores a K and a V vector per layer and KV head. */
int64_t oracle_kv_bytes_per_token(int64_t layers, int64_t kv_heads, int64_t head_dim,
                                  int64_t elem_bytes) {
  return 2 * layers * kv_heads * head_dim * elem_bytes;
}

/* "At most C blocks per KV head are transferred per layer" ("4 System Design"); the cap is a
 * fraction of the budget. Reading: C = floor(cap * budget_blocks), at least one block. */
int32_t oracle_fetch_cap_blocks(float cap, int32_t budget_blocks) {
  double c = floor((double)cap * (double)budget_blocks);
  if (c < 1.0) c = 1.0;
  if (c > budget_blocks) c = budget_blocks;
  return (int32_t)c;
}

/* ---- S1: block summaries ("4 System Design": coordinate-wise minimum and maximum keys,
 *      two vectors per block) ---------------------------------------------------------------- */

void oracle_block_summary(const void* host_unit, int32_t dtype, int32_t n_tok, int32_t bs,
                          int32_t d, void* summ) {
  const int32_t nb = n_blocks(n_tok, bs);
  for (int32_t b = 0; b < nb; ++b) {
    const int32_t nv = valid_in_block(b, n_tok, bs);
    for (int32_t c = 0; c < d; ++c) {
      /* start from the block's first token; a later token replaces the running minimum
       * (maximum) only when strictly smaller (larger) */
      int64_t imin = k_off(b, 0, c, bs, d), imax = imin;
      for (int32_t t = 1; t < nv; ++t) {
        int64_t i = k_off(b, t, c, bs, d);
        if (load(host_unit, dtype, i) < load(host_unit, dtype, imin)) imin = i;
        if (load(host_unit, dtype, i) > load(host_unit, dtype, imax)) imax = i;
      }
      copy_elem(summ, ((int64_t)b * 2 + 0) * d + c, host_unit, imin, dtype);
      copy_elem(summ, ((int64_t)b * 2 + 1) * d + c, host_unit, imax, dtype);
    }
  }
}

/* ---- S2: block scores ("4 System Design": the draft query scans the compressed per-block
 *      key summaries to rank blocks). Reading: per query head, the largest value q.k can take
 *      over the box [kmin, kmax] is sum_c max(q_c kmin_c, q_c kmax_c); the KV head's score is
 *      the sum over the query heads of its group. ------------------------------------------- */

void oracle_block_scores(const void* summ, int32_t dtype, int32_t nb, int32_t d, const void* q,
                         int32_t g, float* scores) {
  for (int32_t b = 0; b < nb; ++b) {
    double s = 0.0;
    for (int32_t h = 0; h < g; ++h) {
      for (int32_t c = 0; c < d; ++c) {
        double x = load(q, dtype, (int64_t)h * d + c);
        double lo = x * load(summ, dtype, ((int64_t)b * 2 + 0) * d + c);
        double hi = x * load(summ, dtype, ((int64_t)b * 2 + 1) * d + c);
        s += lo > hi ? lo : hi;
      }
    }
    scores[b] = (float)s;
  }
}

/* ---- S3: per-head top-K ("4 System Design": top-K prediction). Order: score descending,
 *      equal scores by lower block id. -------------------------------------------------------- */

typedef struct {
  float s;
  int32_t id;
} scored;

static int cmp_scored(const void* a, const void* b) {
  const scored* x = (const scored*)a;
  const scored* y = (const scored*)b;
  if (x->s > y->s) return -1;
  if (x->s < y->s) return 1;
  return (x->id > y->id) - (x->id < y->id);
}

int32_t oracle_topk(const float* scores, int32_t nb, int32_t kb, int32_t* ids) {
  scored* v = (scored*)malloc(sizeof(scored) * (size_t)(nb > 0 ? nb : 1));
  for (int32_t b = 0; b < nb; ++b) {
    v[b].s = scores[b];
    v[b].id = b;
  }
  qsort(v, (size_t)nb, sizeof(scored), cmp_scored);
  const int32_t n = nb < kb ? nb : kb;
  for (int32_t i = 0; i < n; ++i) ids[i] = v[i].id;
  free(v);
  return n;
}

/* ---- S4: KV selection ("4 System Design": at most C blocks per KV head move per layer;
 *      resident predicted blocks stay; admitted non-resident blocks are paired with
 *      least-recently-selected eviction targets).
 * Readings:
 *  - hits (selected and resident) get stamp = step and are never evicted this step;
 *  - misses are taken in selection order and the first min(C, #misses) are admitted;
 *  - eviction targets: free slots by ascending slot first, then resident blocks not selected
 *    this step by (stamp ascending, block id ascending);
 *  - an admitted block gets stamp = step; the fetch list is in admission order. ------------- */

typedef struct {
  int32_t cls, stamp, block, slot;
} target;

static int cmp_target(const void* a, const void* b) {
  const target* x = (const target*)a;
  const target* y = (const target*)b;
  if (x->cls != y->cls) return x->cls - y->cls;
  if (x->cls == 0) return (x->slot > y->slot) - (x->slot < y->slot);
  if (x->stamp != y->stamp) return (x->stamp > y->stamp) - (x->stamp < y->stamp);
  return (x->block > y->block) - (x->block < y->block);
}

int32_t oracle_select_update(int32_t* resident, int32_t* slot_block, int32_t* stamp, int32_t kb,
                             const int32_t* sel, int32_t n_sel, int32_t cap_blocks, int32_t step,
                             int32_t* fetch) {
  int32_t* hit_slot = (int32_t*)calloc((size_t)kb, sizeof(int32_t));
  int32_t* miss = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n_sel > 0 ? n_sel : 1));
  int32_t n_miss = 0;
  for (int32_t i = 0; i < n_sel; ++i) {
    const int32_t b = sel[i];
    const int32_t s = resident[b];
    if (s >= 0) {
      stamp[s] = step;
      hit_slot[s] = 1;
    } else {
      miss[n_miss++] = b;
    }
  }
  const int32_t n_admit = n_miss < cap_blocks ? n_miss : cap_blocks;

  target* t = (target*)malloc(sizeof(target) * (size_t)kb);
  int32_t n_t = 0;
  for (int32_t s = 0; s < kb; ++s) {
    if (slot_block[s] < 0) {
      target x = {0, 0, -1, s};
      t[n_t++] = x;
    } else if (!hit_slot[s]) {
      target x = {1, stamp[s], slot_block[s], s};
      t[n_t++] = x;
    }
  }
  qsort(t, (size_t)n_t, sizeof(target), cmp_target);

  for (int32_t i = 0; i < n_admit; ++i) {
    const int32_t s = t[i].slot;
    const int32_t old = slot_block[s];
    if (old >= 0) resident[old] = -1;
    slot_block[s] = miss[i];
    resident[miss[i]] = s;
    stamp[s] = step;
    fetch[2 * i + 0] = miss[i];
    fetch[2 * i + 1] = s;
  }
  free(t);
  free(miss);
  free(hit_slot);
  return n_admit;
}

/* ---- Decode-side tier of a request admitted with partial staging ("4 System Design", last
 *      bullet: the full KV cache of a request stays in the prefill side's host memory until the
 *      request completes, and the decode side keeps only the subset that decoding has asked for).
 *      Reading: the fetch list is walked in order; a block the decode side already holds is read
 *      from its kept copy; a block fetched for the first time is read from the full copy and kept
 *      in the next unused entry of the decode-side tier; kept blocks stay until the request ends;
 *      once the tier's `local_cap` entries are used, first-time blocks are read from the full copy
 *      and not kept. route[i] = 2 * entry (read the kept copy), 2 * entry + 1 (read the full copy
 *      and keep it in that entry), or -1 (read the full copy only). Returns the number of fetch
 *      entries read from the full copy. --------------------------------------------------------- */

int32_t oracle_local_route(int32_t* local_of, int32_t* local_used, int32_t local_cap,
                           const int32_t* fetch, int32_t n_fetch, int32_t* route) {
  int32_t from_full = 0;
  for (int32_t i = 0; i < n_fetch; ++i) {
    const int32_t b = fetch[2 * i + 0];
    if (local_of[b] >= 0) {
      route[i] = 2 * local_of[b];
      continue;
    }
    ++from_full;
    if (*local_used < local_cap) {
      local_of[b] = *local_used;
      *local_used += 1;
      route[i] = 2 * local_of[b] + 1;
    } else {
      route[i] = -1;
    }
  }
  return from_full;
}

/* ---- S6: attention over the resident set ("4 System Design": attention runs over the
 *      resident KV). Reading: every valid token of every occupied slot; scale 1/sqrt(d);
 *      keys already carry their positions; an empty set yields zeros. ----------------------- */

static void softmax_attend(const void* host_unit, int32_t dtype, const int32_t* blocks,
                           int32_t n_blocks_listed, int32_t n_tok, int32_t bs, int32_t d,
                           const void* q, int32_t g, double* out) {
  const double scale = 1.0 / sqrt((double)d);
  int64_t n_keys = 0;
  for (int32_t i = 0; i < n_blocks_listed; ++i) n_keys += valid_in_block(blocks[i], n_tok, bs);
  double* z = (double*)malloc(sizeof(double) * (size_t)(n_keys > 0 ? n_keys : 1));
  for (int32_t h = 0; h < g; ++h) {
    int64_t k = 0;
    double m = -INFINITY;
    for (int32_t i = 0; i < n_blocks_listed; ++i) {
      const int32_t b = blocks[i];
      const int32_t nv = valid_in_block(b, n_tok, bs);
      for (int32_t t = 0; t < nv; ++t) {
        double dot = 0.0;
        for (int32_t c = 0; c < d; ++c)
          dot += load(q, dtype, (int64_t)h * d + c) * load(host_unit, dtype, k_off(b, t, c, bs, d));
        z[k] = dot * scale;
        if (z[k] > m) m = z[k];
        ++k;
      }
    }
    double denom = 0.0;
    for (int64_t i = 0; i < n_keys; ++i) {
      z[i] = exp(z[i] - m);
      denom += z[i];
    }
    for (int32_t c = 0; c < d; ++c) out[(int64_t)h * d + c] = 0.0;
    k = 0;
    for (int32_t i = 0; i < n_blocks_listed; ++i) {
      const int32_t b = blocks[i];
      const int32_t nv = valid_in_block(b, n_tok, bs);
      for (int32_t t = 0; t < nv; ++t) {
        for (int32_t c = 0; c < d; ++c)
          out[(int64_t)h * d + c] += z[k] * load(host_unit, dtype, v_off(b, t, c, bs, d));
        ++k;
      }
    }
    if (n_keys > 0)
      for (int32_t c = 0; c < d; ++c) out[(int64_t)h * d + c] /= denom;
  }
  free(z);
}

void oracle_attend(const void* host_unit, int32_t dtype, const int32_t* slot_block, int32_t kb,
                   int32_t n_tok, int32_t bs, int32_t d, const void* q, int32_t g, double* out) {
  int32_t* blocks = (int32_t*)malloc(sizeof(int32_t) * (size_t)(kb > 0 ? kb : 1));
  int32_t n = 0;
  for (int32_t s = 0; s < kb; ++s)
    if (slot_block[s] >= 0) blocks[n++] = slot_block[s];
  softmax_attend(host_unit, dtype, blocks, n, n_tok, bs, d, q, g, out);
  free(blocks);
}

void oracle_dense_attend(const void* host_unit, int32_t dtype, int32_t n_tok, int32_t bs,
                         int32_t d, const void* q, int32_t g, double* out) {
  const int32_t nb = n_blocks(n_tok, bs);
  int32_t* blocks = (int32_t*)malloc(sizeof(int32_t) * (size_t)(nb > 0 ? nb : 1));
  for (int32_t b = 0; b < nb; ++b) blocks[b] = b;
  softmax_attend(host_unit, dtype, blocks, nb, n_tok, bs, d, q, g, out);
  free(blocks);
}

/* ---- S8: append ("2 Background": the cache must remain available throughout generation;
 *      "4 System Design": the summaries stay in HBM). Reading: the host copy is written, and
 *      the tail block's min/max absorb the new key (a new block starts from it). ------------ */

void oracle_append(void* host_unit, void* summ, int32_t dtype, int32_t n_tok, int32_t bs,
                   int32_t d, const void* k_new, const void* v_new) {
  const int32_t b = n_tok / bs, t = n_tok % bs;
  for (int32_t c = 0; c < d; ++c) {
    copy_elem(host_unit, k_off(b, t, c, bs, d), k_new, c, dtype);
    copy_elem(host_unit, v_off(b, t, c, bs, d), v_new, c, dtype);
    const int64_t mn = ((int64_t)b * 2 + 0) * d + c, mx = ((int64_t)b * 2 + 1) * d + c;
    if (t == 0) {
      copy_elem(summ, mn, k_new, c, dtype);
      copy_elem(summ, mx, k_new, c, dtype);
    } else {
      const double x = load(k_new, dtype, c);
      if (x < load(summ, dtype, mn)) copy_elem(summ, mn, k_new, c, dtype);
      if (x > load(summ, dtype, mx)) copy_elem(summ, mx, k_new, c, dtype);
    }
  }
}

/* ---- batched driver ------------------------------------------------------------------------ */

static void run_unit(oracle_unit* u, const oracle_dims* D, int32_t what) {
  const int32_t nb = n_blocks(u->n_tok, D->bs);
  if (what & ORACLE_DO_SUMMARY) oracle_block_summary(u->host_unit, D->dtype, u->n_tok, D->bs, D->d, u->summ);
  if (what & ORACLE_DO_SCORE) {
    float* sc = u->scores ? u->scores : (float*)malloc(sizeof(float) * (size_t)(nb > 0 ? nb : 1));
    oracle_block_scores(u->summ, D->dtype, nb, D->d, u->q, D->g, sc);
    const int32_t n = oracle_topk(sc, nb, D->kb, u->sel_ids);
    *u->n_sel = n;
    if (u->sel_scores)
      for (int32_t i = 0; i < n; ++i) u->sel_scores[i] = sc[u->sel_ids[i]];
    if (!u->scores) free(sc);
  }
  if (what & ORACLE_DO_SELECT) {
    const int32_t* sel = u->n_sel_override >= 0 ? u->sel_override : u->sel_ids;
    const int32_t n = u->n_sel_override >= 0 ? u->n_sel_override : *u->n_sel;
    *u->n_fetch = oracle_select_update(u->resident, u->slot_block, u->stamp, D->kb, sel, n,
                                       D->cap_blocks, D->step, u->fetch);
    if (u->route) {
      if (u->local_cap >= 0)
        oracle_local_route(u->local_of, u->local_used, u->local_cap, u->fetch, *u->n_fetch, u->route);
      else
        for (int32_t i = 0; i < *u->n_fetch; ++i) u->route[i] = -1;
    }
  }
  if (what & ORACLE_DO_ATTEND)
    oracle_attend(u->host_unit, D->dtype, u->slot_block, D->kb, u->n_tok, D->bs, D->d, u->q, D->g,
                  u->out);
  if (what & ORACLE_DO_DENSE)
    oracle_dense_attend(u->host_unit, D->dtype, u->n_tok, D->bs, D->d, u->q, D->g, u->out);
}

typedef struct {
  oracle_unit* units;
  int32_t n_units, what, tid, n_threads;
  const oracle_dims* D;
} run_job;

static void* run_worker(void* arg) {
  run_job* J = (run_job*)arg;
  for (int32_t i = J->tid; i < J->n_units; i += J->n_threads) run_unit(&J->units[i], J->D, J->what);
  return NULL;
}

int oracle_run_units(oracle_unit* units, int32_t n_units, const oracle_dims* dims, int32_t what,
                     int32_t n_threads) {
  if (!units || !dims || n_units < 0) return -1;
  if (n_threads < 1) n_threads = 1;
  if (n_threads > n_units) n_threads = n_units > 0 ? n_units : 1;
  run_job* jobs = (run_job*)malloc(sizeof(run_job) * (size_t)n_threads);
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)n_threads);
  for (int32_t t = 0; t < n_threads; ++t) {
    run_job J = {units, n_units, what, t, n_threads, dims};
    jobs[t] = J;
  }
  for (int32_t t = 1; t < n_threads; ++t) pthread_create(&th[t], NULL, run_worker, &jobs[t]);
  run_worker(&jobs[0]);
  for (int32_t t = 1; t < n_threads; ++t) pthread_join(th[t], NULL);
  free(th);
  free(jobs);
  return 0;
}
