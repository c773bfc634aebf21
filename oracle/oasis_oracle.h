/*
 * oasis_oracle.h -- CPU oracle for the OasisKV decode hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  This header and oasis_oracle.c are the slow,
 * plain, single-threaded reference that the GPU library is checked against.
 * Only the test suite, the package smoke check and the benchmark's CPU
 * baseline leg load it.  The GPU library neither includes nor links it, and
 * this code shares no source with the GPU library.
 *
 * [OasisKV] below means the page "OasisKV: Scaling In-Decode KV Cache Beyond
 * HBM with Lookahead Sparse Prefetching" (arXiv:2608.08097, summary page that
 * carries the paper's figure and table captions).
 *
 * Every function here is pinned by the CPU tests to hand-computed cases,
 * closed forms, brute force or invariants.  Parity unpinned: multi-step
 * trajectories (the functions chained over many steps); the page prints
 * none.
 *
 * Layouts (row-major, all sizes in elements):
 *   K, V (host full cache) : [B][Hkv][NB][bs][D]      bf16 bit patterns
 *   summ                   : [B][Hkv][NB][D]          fp32
 *   q_draft                : [B][L][Hq][D]            bf16 bit patterns
 *   scores                 : [B][Hkv][NB]             fp32
 *   topk_ids               : [B][Hkv][K]              int32
 *   slot_of_block          : [B][Hkv][NB]             int32, -1 = not resident
 *   block_of_slot          : [B][Hkv][S]              int32, -1 = empty slot
 *   last_used              : [B][Hkv][S]              int32, -1 = never
 *   fetch_block/fetch_slot/evict_block : [B][Hkv][cap] int32, -1 past the count
 *   n_fetch, n_evict       : [B][Hkv]                 int32
 *   pool K, V              : [B][Hkv][S][bs][D]       bf16 bit patterns
 *   q                      : [B][Hq][D]               bf16 bit patterns
 *   out                    : [B][Hq][D]               fp32 (oracle keeps fp32)
 * with S = kv_budget_tokens / block_size and query head hq = h*G + g,
 * G = Hq / Hkv.
 */
#ifndef OASIS_ORACLE_H
#define OASIS_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int32_t batch;            /* B */
    int32_t num_q_heads;      /* Hq */
    int32_t num_kv_heads;     /* Hkv */
    int32_t head_dim;         /* D */
    int32_t block_size;       /* bs, tokens per KV block */
    int32_t num_blocks;       /* NB, context blocks per (request, KV head) */
    int32_t kv_budget_tokens; /* S * bs */
    int32_t lookahead;        /* L draft tokens */
    int32_t top_k;            /* K predicted blocks per KV head */
    float   fetch_ratio;      /* cap = ceil(ratio*S); <0 or >=1 means cap = K */
    int32_t sink_blocks;      /* blocks [0, sink) always selected */
    int32_t local_blocks;     /* last `local` blocks always selected */
} orc_cfg;

/* 0 when the configuration is consistent, otherwise a negative code. */
int orc_check_cfg(const orc_cfg* c);
int orc_fetch_cap(const orc_cfg* c);

void orc_build_summaries(const orc_cfg* c, const uint16_t* k, float* summ);
void orc_score_blocks(const orc_cfg* c, const uint16_t* q_draft, const float* summ,
                      float* scores);
void orc_build_summaries_minmax(const orc_cfg* c, const uint16_t* k, uint16_t* summ_mm);
void orc_score_blocks_minmax(const orc_cfg* c, const uint16_t* q_draft, const uint16_t* summ_mm,
                             float* scores);
int  orc_select_topk(const orc_cfg* c, const float* scores, int32_t* topk_ids);
int  orc_select_topk_ctx(const orc_cfg* c, const float* scores, const int32_t* ctx_len,
                         int32_t* topk_ids);
int  orc_append_kv(const orc_cfg* c, const uint16_t* k_new, const uint16_t* v_new,
                   int32_t* ctx_len, const int32_t* clock, int32_t step, uint16_t* host_k,
                   uint16_t* host_v, int32_t* slot_of_block, int32_t* block_of_slot,
                   int32_t* last_used, uint16_t* pool_k, uint16_t* pool_v);
void orc_refresh_summaries(const orc_cfg* c, const int32_t* ctx_len, const uint16_t* host_k,
                           float* summ, uint16_t* summ_mm);
int  orc_plan_fetch(const orc_cfg* c, const int32_t* topk_ids, int32_t step,
                    int32_t* slot_of_block, int32_t* block_of_slot, int32_t* last_used,
                    int32_t* fetch_block, int32_t* fetch_slot, int32_t* evict_block,
                    int32_t* n_fetch, int32_t* n_evict);
int  orc_fetch_blocks(const orc_cfg* c, const uint16_t* host_k, const uint16_t* host_v,
                      const int32_t* fetch_block, const int32_t* fetch_slot,
                      const int32_t* n_fetch, uint16_t* pool_k, uint16_t* pool_v);
void orc_sparse_decode_attn(const orc_cfg* c, const uint16_t* q, const uint16_t* pool_k,
                            const uint16_t* pool_v, const int32_t* block_of_slot,
                            const int32_t* ctx_len, double scale, float* out);
void orc_dense_decode_attn(const orc_cfg* c, const uint16_t* q, const uint16_t* k,
                           const uint16_t* v, const int32_t* ctx_len, double scale,
                           float* out);

#ifdef __cplusplus
}
#endif

#endif /* OASIS_ORACLE_H */
