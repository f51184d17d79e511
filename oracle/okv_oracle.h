/*
 * ORACLE: test infrastructure, not product code.
 *
 * A plain, slow, obviously correct CPU restatement of the per-decode-step path of
 * OasisKV ("OasisKV: Scaling In-Decode KV Cache Beyond HBM with Lookahead Sparse
 * Prefetching", arXiv 2608.08097; summary page paperlayer.ai/abs/2608.08097v1,
 * section "4 System Design"). Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load it. It shares no code with the CUDA library.
 *
 * Arithmetic is binary64 throughout; values are read from their storage type
 * (binary32 or bfloat16) exactly. Scores are rounded once to binary32 for ranking.
 *
 * Pins (tests/test_oracle_*.py): closed-form KV sizing from "2 Background";
 * brute-force min/max; the score's upper-bound property and its one-token special
 * case; brute-force sorting for top-K; the selection rules of "4 System Design"
 * checked as invariants plus hand-worked scenarios; the decode-side tier against a
 * first-demand set computation and a hand-worked scenario; sparse attention equal to a
 * textbook dense softmax attention when the budget covers the context; one-token
 * and equal-score special cases; appends equal to a rebuild.
 */
#ifndef OKV_ORACLE_H
#define OKV_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };

/* Bytes of K and V per token: 2 * layers * kv_heads * head_dim * elem_bytes. */
int64_t oracle_kv_bytes_per_token(int64_t layers, int64_t kv_heads, int64_t head_dim,
                                  int64_t elem_bytes);

/* Fetch cap in blocks: C = max(1, floor(cap * budget_blocks)). */
int32_t oracle_fetch_cap_blocks(float cap, int32_t budget_blocks);

/* Summaries of one (layer, request, kv head). host_unit: [cap_blocks][2][bs][d] (K then V);
 * summ: [nb][2][d], nb = ceil(n_tok / bs); [b][0] = coordinate-wise min, [b][1] = max of the
 * block's valid keys. */
void oracle_block_summary(const void* host_unit, int32_t dtype, int32_t n_tok, int32_t bs,
                          int32_t d, void* summ);

/* Score of every block against the g draft query heads of the group:
 * s_b = sum_h sum_c max(q[h][c] * kmin[b][c], q[h][c] * kmax[b][c]), rounded to binary32. */
void oracle_block_scores(const void* summ, int32_t dtype, int32_t nb, int32_t d, const void* q,
                         int32_t g, float* scores);

/* Top-K: ids of the min(kb, nb) blocks first in (score desc, id asc). Returns that count. */
int32_t oracle_topk(const float* scores, int32_t nb, int32_t kb, int32_t* ids);

/* Diff / admit / evict for one unit (see the .c file for the rules). resident: [nb] block->slot
 * or -1; slot_block: [kb] slot->block or -1; stamp: [kb]; fetch: [kb][2] (block, slot).
 * Returns the number of fetch entries. */
int32_t oracle_select_update(int32_t* resident, int32_t* slot_block, int32_t* stamp, int32_t kb,
                             const int32_t* sel, int32_t n_sel, int32_t cap_blocks, int32_t step,
                             int32_t* fetch);

/* Decode-side tier of a partially staged request (see the .c file): walks the fetch list
 * ([n_fetch][2] (block, slot)) in order and writes route[i] = 2*entry (read the kept copy),
 * 2*entry + 1 (read the full copy, keep it in that entry) or -1 (read the full copy only);
 * local_of: [nb] block -> kept entry or -1; *local_used: entries in use (at most local_cap).
 * Returns how many entries read the full copy. */
int32_t oracle_local_route(int32_t* local_of, int32_t* local_used, int32_t local_cap,
                           const int32_t* fetch, int32_t n_fetch, int32_t* route);

/* Softmax attention of g query heads over every valid token of every block named in
 * slot_block (entries >= 0), reading K and V from host_unit. out: [g][d]. */
void oracle_attend(const void* host_unit, int32_t dtype, const int32_t* slot_block, int32_t kb,
                   int32_t n_tok, int32_t bs, int32_t d, const void* q, int32_t g, double* out);

/* Dense softmax attention over all n_tok tokens (the special case budget >= context). */
void oracle_dense_attend(const void* host_unit, int32_t dtype, int32_t n_tok, int32_t bs,
                         int32_t d, const void* q, int32_t g, double* out);

/* Append one token at position n_tok: writes K and V into host_unit and updates the tail
 * block's summary (a new block starts with min = max = k). */
void oracle_append(void* host_unit, void* summ, int32_t dtype, int32_t n_tok, int32_t bs,
                   int32_t d, const void* k_new, const void* v_new);

/* ---- batched driver over independent units -------------------------------------------- */

enum {
  ORACLE_DO_SUMMARY = 1,  /* build summ from host_unit */
  ORACLE_DO_SCORE = 2,    /* scores + top-K from summ and q */
  ORACLE_DO_SELECT = 4,   /* diff / admit / evict */
  ORACLE_DO_ATTEND = 8,   /* sparse attention over the slot table */
  ORACLE_DO_DENSE = 16    /* dense attention */
};

typedef struct {
  const void* host_unit;    /* [cap_blocks][2][bs][d] */
  void* summ;               /* [nb][2][d] */
  const void* q;            /* [g][d]: draft query for SCORE, query for ATTEND/DENSE */
  int32_t n_tok;
  int32_t n_sel_override;   /* >= 0: SELECT uses sel_override instead of this unit's top-K */
  const int32_t* sel_override;
  int32_t* resident;        /* [nb] */
  int32_t* slot_block;      /* [kb] */
  int32_t* stamp;           /* [kb] */
  float* scores;            /* [nb] or NULL */
  int32_t* sel_ids;         /* [kb] */
  float* sel_scores;        /* [kb] or NULL */
  int32_t* n_sel;
  int32_t* fetch;           /* [kb][2] */
  int32_t* n_fetch;
  double* out;              /* [g][d] */
  int32_t local_cap;        /* < 0: the request holds its full KV; else decode-side tier entries */
  int32_t* local_of;        /* [nb] block -> decode-side entry or -1 (local_cap >= 0) */
  int32_t* local_used;      /* entries in use (local_cap >= 0) */
  int32_t* route;           /* [kb] or NULL: SELECT also routes its fetch list (-1 for full KV) */
} oracle_unit;

typedef struct {
  int32_t dtype, bs, d, g, kb, cap_blocks, step;
} oracle_dims;

/* Run the steps named in `what` for every unit, spread over n_threads host threads. */
int oracle_run_units(oracle_unit* units, int32_t n_units, const oracle_dims* dims, int32_t what,
                     int32_t n_threads);

#ifdef __cplusplus
}
#endif
#endif
