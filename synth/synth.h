/*
 * Seeded synthetic inputs for the lookahead sparse KV staging path.
 *
 * This module generates the workload only: host KV cache contents, per-step
 * queries and draft queries, and the K/V of appended tokens. It holds none of
 * the method's arithmetic (no summaries, scores, selection or attention), so the
 * CPU oracle and the GPU path can both read what it writes without sharing any
 * of the computation under test.
 *
 * Workload shape (OasisKV, paperlayer.ai/abs/2608.08097v1, "4 System Design"
 * and the evaluation's Qwen3-8B / 32B-class GQA shapes): keys and values are
 * N(0,1); some blocks carry a planted key direction (+A*u_j on every key of the
 * block); the query of every head is normalize(sum of the active directions)
 * plus N(0, sigma_q^2) noise per dimension, and the draft (lookahead) query of
 * step t is the query of step t+1 plus N(0, sigma_d^2) noise.
 *
 * Random numbers: SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014) used as a counter-based hash of
 * (seed, stream, fields...), 24-bit uniforms, and the Box-Muller transform
 * (Box & Muller 1958) for normals.
 *
 * Storage dtypes: SYNTH_F32 (IEEE binary32) or SYNTH_BF16 (bfloat16, the upper
 * 16 bits of binary32 after round-to-nearest-even).
 */
#ifndef OKV_SYNTH_H
#define OKV_SYNTH_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { SYNTH_F32 = 0, SYNTH_BF16 = 1 };
enum { SYNTH_PLANT_MOD = 0, SYNTH_PLANT_COUNT = 1 };

typedef struct {
  uint64_t seed;
  int32_t layers, q_heads, kv_heads, head_dim, block_size;
  int32_t dtype;          /* SYNTH_F32 or SYNTH_BF16 */
  int32_t plant_mode;     /* MOD: block b carries direction b mod P (every block planted);
                             COUNT: the n_plant blocks (of plant_blocks) with the smallest
                             hash carry direction hash mod P */
  int32_t n_dirs;         /* P, size of the direction dictionary of one (layer, request, kv head) */
  int32_t n_plant;        /* COUNT mode: how many blocks are planted */
  int32_t plant_blocks;   /* COUNT mode: blocks [0, plant_blocks) are candidates */
  int32_t n_active;       /* directions active in one step's query */
  int32_t active_period;  /* the active window advances by one direction every active_period steps */
  double amplitude;       /* A: planted keys get +A*u_j */
  double sigma_q;         /* query noise std per dimension */
  double sigma_d;         /* draft noise std per dimension */
} synth_params;

/* Element size in bytes of a storage dtype (4 or 2), 0 for an unknown dtype. */
int synth_dtype_size(int32_t dtype);

/*
 * Fill tokens [tok_begin, tok_end) of one request's host KV buffer.
 * Layout of buf: [layers][kv_heads][cap_blocks][2][block_size][head_dim]; index 0
 * of the "2" axis is K, 1 is V. req_key selects the content (two requests with the
 * same req_key hold identical KV). Positions outside [tok_begin, tok_end) are not
 * written. Returns 0, or -1 on bad arguments.
 */
int synth_fill_kv(void* buf, const synth_params* p, int32_t req_key, int32_t tok_begin,
                  int32_t tok_end, int32_t cap_blocks, int32_t n_threads);

/*
 * The same contents as synth_fill_kv writes for one layer: tokens [tok_begin, tok_end) of
 * layer `layer` into buf laid out [kv_heads][cap_blocks][2][block_size][head_dim].
 * Returns 0, or -1 on bad arguments.
 */
int synth_fill_kv_layer(void* buf, const synth_params* p, int32_t req_key, int32_t layer,
                        int32_t tok_begin, int32_t tok_end, int32_t cap_blocks, int32_t n_threads);

/*
 * One layer's query (kind 0) or draft query (kind 1) of step `step` for `batch`
 * requests. out: [batch][q_heads][head_dim] in the storage dtype.
 * req_ids[i] is the request id (drives the noise); req_keys[i] its KV content key
 * (drives the directions). The draft of step t equals query(t+1) + sigma_d noise.
 */
int synth_queries(void* out, const synth_params* p, int32_t layer, int32_t step, int32_t kind,
                  int32_t batch, const int32_t* req_ids, const int32_t* req_keys,
                  int32_t n_threads);

/*
 * K and V of one token per request for one layer: out_k, out_v [batch][kv_heads][head_dim],
 * token position positions[i] of request content req_keys[i]; identical to what
 * synth_fill_kv writes at that position.
 */
int synth_token_kv(void* out_k, void* out_v, const synth_params* p, int32_t layer,
                   int32_t batch, const int32_t* req_keys, const int32_t* positions);

/* The direction u_j of (layer, req_key, kv_head) as doubles, out[head_dim]. */
int synth_direction(double* out, const synth_params* p, int32_t layer, int32_t req_key,
                    int32_t kv_head, int32_t j);

/* Direction index planted in block `block` of (layer, req_key, kv_head), or -1. */
int32_t synth_block_direction(const synth_params* p, int32_t layer, int32_t req_key,
                              int32_t kv_head, int32_t block);

/* n standard normals from (seed, stream, a, b, c, d) into out (for statistics tests). */
int synth_normals(double* out, int64_t n, uint64_t seed, uint64_t stream, uint64_t a, uint64_t b);

#ifdef __cplusplus
}
#endif
#endif
