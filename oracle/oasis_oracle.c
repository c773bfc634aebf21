/*
 * oasis_oracle.c -- CPU oracle for the OasisKV decode hot path.
 *
 * TEST INFRASTRUCTURE ONLY: plain, slow, single-threaded C11, used to check
 * the GPU library.  Nothing in the GPU library includes, links or calls it.
 *
 * [OasisKV] = "OasisKV: Scaling In-Decode KV Cache Beyond HBM with Lookahead
 * Sparse Prefetching" (arXiv:2608.08097, summary page with the paper's figure
 * and table captions).  Every function below follows the step of the method
 * named in its comment, in the order the page gives: look-ahead scoring of
 * compressed keys and top-K prediction (Fig. 7), selection against the GPU
 * working set with capped eviction (explanatory diagram step 3; Tab. 2,
 * "LRU eviction"), the head-wise block map (Fig. 9), the transfer (Fig. 8),
 * and sparse attention over the working set (Fig. 7).
 *
 * Where the page leaves a step open, the reading used here is stated at the
 * function.  Floating-point sums accumulate in double; fp32 results are the
 * double result rounded once.
 */
#include "oasis_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* bf16 -> double: a bf16 value is the upper half of an fp32 bit pattern. */
static double bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static int slots_of(const orc_cfg* c) { return c->kv_budget_tokens / c->block_size; }

int orc_check_cfg(const orc_cfg* c)
{
    if (c->batch < 1 || c->num_kv_heads < 1 || c->num_q_heads < 1) return -1;
    if (c->num_q_heads % c->num_kv_heads != 0) return -2;
    if (c->head_dim < 1 || c->block_size < 1 || c->num_blocks < 1) return -3;
    if (c->kv_budget_tokens < c->block_size || c->kv_budget_tokens % c->block_size) return -4;
    if (c->lookahead < 1) return -5;
    if (c->top_k < 1 || c->top_k > c->num_blocks || c->top_k > slots_of(c)) return -6;
    if (c->sink_blocks < 0 || c->local_blocks < 0) return -7;
    return 0;
}

/*
 * Fetch cap per (request, KV head) and step: [OasisKV] Tab. 2 caption -- the
 * cap bounds the blocks fetched per step by a fetch ratio; the "Fetch all" row
 * has no cap.  Reading: the ratio applies to the budget in blocks S, so
 * cap = ceil(ratio * S), computed in double with a 1e-6 allowance so that a
 * ratio whose product with S is an integer up to float rounding gives that
 * integer; clamped to [0, K].  A ratio < 0 or >= 1 means "fetch all": cap = K.
 */
int orc_fetch_cap(const orc_cfg* c)
{
    double r = (double)c->fetch_ratio;
    int cap;
    if (r < 0.0 || r >= 1.0) return c->top_k;
    cap = (int)ceil(r * (double)slots_of(c) - 1e-6);
    if (cap < 0) cap = 0;
    if (cap > c->top_k) cap = c->top_k;
    return cap;
}

/*
 * Compressed keys, [OasisKV] Fig. 7 (left): one summary vector per KV block,
 * kept on the GPU for every block of the context.  The page pools each block;
 * the pooling used here is the fp32 mean of the block's keys:
 *   summ[b,h,j,d] = fp32( (sum_{t<bs} K[b,h,j*bs+t,d]) / bs ).
 */
void orc_build_summaries(const orc_cfg* c, const uint16_t* k, float* summ)
{
    const int B = c->batch, H = c->num_kv_heads, NB = c->num_blocks;
    const int bs = c->block_size, D = c->head_dim;
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
            for (int j = 0; j < NB; ++j)
                for (int d = 0; d < D; ++d) {
                    double sum = 0.0;
                    for (int t = 0; t < bs; ++t) {
                        size_t idx = ((((size_t)b * H + h) * NB + j) * bs + t) * D + d;
                        sum += bf16_to_double(k[idx]);
                    }
                    summ[(((size_t)b * H + h) * NB + j) * D + d] = (float)(sum / (double)bs);
                }
}

/*
 * Look-ahead block scoring, [OasisKV] Fig. 7 (right) and 'What they did'
 * item 2: the draft (preview) tokens' queries scan the compressed keys of all
 * blocks.  For KV head h, the queries of its GQA group g < G and of every
 * draft token l < L are dotted with each block summary; the block's score is
 * the maximum over (l, g).  No 1/sqrt(D) factor: a positive scale does not
 * change the ranking.  Stored as fp32 (the double maximum rounded once).
 */
void orc_score_blocks(const orc_cfg* c, const uint16_t* q_draft, const float* summ,
                      float* scores)
{
    const int B = c->batch, H = c->num_kv_heads, Hq = c->num_q_heads;
    const int G = Hq / H, L = c->lookahead, NB = c->num_blocks, D = c->head_dim;
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
            for (int j = 0; j < NB; ++j) {
                const float* s = summ + (((size_t)b * H + h) * NB + j) * D;
                double best = -INFINITY;
                for (int l = 0; l < L; ++l)
                    for (int g = 0; g < G; ++g) {
                        const uint16_t* q = q_draft + (((size_t)b * L + l) * Hq + (size_t)h * G + g) * D;
                        double dot = 0.0;
                        for (int d = 0; d < D; ++d) dot += bf16_to_double(q[d]) * (double)s[d];
                        if (dot > best) best = dot;
                    }
                scores[((size_t)b * H + h) * NB + j] = (float)best;
            }
}

/*
 * Min/max compressed keys, [OasisKV] Fig. 7 (left): the page pools each block
 * by its minimum and maximum.  Per dimension d of block j, the largest and
 * the smallest of the block's bs key values, kept as the bf16 key value
 * itself; row 0 of the block's pair is the max, row 1 the min.  Reading: where
 * several tokens hold the extreme value, the first in token order gives the
 * stored bit pattern (this only decides between +0 and -0).
 */
void orc_build_summaries_minmax(const orc_cfg* c, const uint16_t* k, uint16_t* summ_mm)
{
    const int B = c->batch, H = c->num_kv_heads, NB = c->num_blocks;
    const int bs = c->block_size, D = c->head_dim;
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
            for (int j = 0; j < NB; ++j)
                for (int d = 0; d < D; ++d) {
                    const size_t blk = ((size_t)b * H + h) * NB + j;
                    uint16_t hi = k[(blk * bs) * D + d], lo = hi;
                    for (int t = 1; t < bs; ++t) {
                        uint16_t x = k[(blk * bs + t) * D + d];
                        if (bf16_to_double(x) > bf16_to_double(hi)) hi = x;
                        if (bf16_to_double(x) < bf16_to_double(lo)) lo = x;
                    }
                    summ_mm[(blk * 2 + 0) * D + d] = hi;
                    summ_mm[(blk * 2 + 1) * D + d] = lo;
                }
}

/*
 * Look-ahead scoring against min/max compressed keys ([OasisKV] Fig. 7): for
 * each draft query q (every l < L, g < G of KV head h) the block's bound
 *   sum_d max(q_d * min_d, q_d * max_d),
 * the largest q . k any key k inside the block's per-dimension box can give;
 * the block's score is the maximum over (l, g), as for the mean keys.
 */
void orc_score_blocks_minmax(const orc_cfg* c, const uint16_t* q_draft, const uint16_t* summ_mm,
                             float* scores)
{
    const int B = c->batch, H = c->num_kv_heads, Hq = c->num_q_heads;
    const int G = Hq / H, L = c->lookahead, NB = c->num_blocks, D = c->head_dim;
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
            for (int j = 0; j < NB; ++j) {
                const uint16_t* mx = summ_mm + ((((size_t)b * H + h) * NB + j) * 2 + 0) * D;
                const uint16_t* mn = summ_mm + ((((size_t)b * H + h) * NB + j) * 2 + 1) * D;
                double best = -INFINITY;
                for (int l = 0; l < L; ++l)
                    for (int g = 0; g < G; ++g) {
                        const uint16_t* q = q_draft + (((size_t)b * L + l) * Hq + (size_t)h * G + g) * D;
                        double bound = 0.0;
                        for (int d = 0; d < D; ++d) {
                            double qd = bf16_to_double(q[d]);
                            double lo = qd * bf16_to_double(mn[d]), hi = qd * bf16_to_double(mx[d]);
                            bound += lo > hi ? lo : hi;
                        }
                        if (bound > best) best = bound;
                    }
                scores[((size_t)b * H + h) * NB + j] = (float)best;
            }
}

/* Forced blocks: the sink [0, sink) and the local window, the last `local`
 * blocks of the context.  They are always selected and count toward K. */
static int is_forced(const orc_cfg* c, int j)
{
    return j < c->sink_blocks || j >= c->num_blocks - c->local_blocks;
}

typedef struct { float s; int32_t id; } scored_id;

/* Order: higher score first; equal scores by lower block id first. */
static int cmp_score_desc_id_asc(const void* pa, const void* pb)
{
    const scored_id* a = (const scored_id*)pa;
    const scored_id* b = (const scored_id*)pb;
    if (a->s > b->s) return -1;
    if (a->s < b->s) return 1;
    return (a->id > b->id) - (a->id < b->id);
}

/*
 * Per-KV-head top-K block prediction, [OasisKV] explanatory diagram step 2
 * ("top-K prediction") and Fig. 4 (top-20 blocks): the K blocks with the
 * highest scores.  Readings: equal scores go to the lower block id; forced
 * blocks (sink and local window) are always selected and count toward K.
 * Output order per (b, h): forced blocks by ascending id, then the others by
 * (score descending, id ascending).  This order is the fetch priority.
 * Returns 0, or -1 when the forced blocks alone exceed K.
 */
int orc_select_topk(const orc_cfg* c, const float* scores, int32_t* topk_ids)
{
    const int B = c->batch, H = c->num_kv_heads, NB = c->num_blocks, K = c->top_k;
    scored_id* rest = (scored_id*)malloc(sizeof(scored_id) * (size_t)NB);
    int rc = 0;
    if (!rest) return -2;
    for (int b = 0; b < B && rc == 0; ++b)
        for (int h = 0; h < H; ++h) {
            const float* sc = scores + ((size_t)b * H + h) * NB;
            int32_t* out = topk_ids + ((size_t)b * H + h) * K;
            int nf = 0, nr = 0;
            for (int j = 0; j < NB; ++j) {
                if (is_forced(c, j)) {
                    if (nf >= K) { rc = -1; break; }
                    out[nf++] = j;
                } else {
                    rest[nr].s = sc[j];
                    rest[nr].id = j;
                    ++nr;
                }
            }
            if (rc) break;
            qsort(rest, (size_t)nr, sizeof(scored_id), cmp_score_desc_id_asc);
            for (int i = 0; nf + i < K; ++i) out[nf + i] = rest[i].id;
        }
    free(rest);
    return rc;
}

/*
 * Top-K over a growing context.  Reading of 'What they did' item 4 (the
 * local window of recent tokens stays in the working set) once decoding
 * appends tokens: with n = ceil(ctx_len[b] / bs) blocks in the context (at
 * most NB), the forced blocks are the sink [0, min(sink, n)) and the last
 * `local` blocks of the context [max(n - local, 0), n); the other blocks of
 * the context compete by score, and blocks at or beyond n (not yet written)
 * rank as if scored -infinity, so they are picked only when the context has
 * fewer than K blocks.  Ties: lower id first.  With ctx_len = NB * bs this
 * is orc_select_topk.
 */
int orc_select_topk_ctx(const orc_cfg* c, const float* scores, const int32_t* ctx_len,
                        int32_t* topk_ids)
{
    const int B = c->batch, H = c->num_kv_heads, NB = c->num_blocks, K = c->top_k;
    const int bs = c->block_size;
    scored_id* rest = (scored_id*)malloc(sizeof(scored_id) * (size_t)NB);
    int rc = 0;
    if (!rest) return -2;
    for (int b = 0; b < B && rc == 0; ++b) {
        long long nb = ctx_len[b] <= 0 ? 0 : ((long long)ctx_len[b] + bs - 1) / bs;
        const int n = nb > NB ? NB : (int)nb;
        const int sink_end = c->sink_blocks < n ? c->sink_blocks : n;
        const int win_begin = n - c->local_blocks > 0 ? n - c->local_blocks : 0;
        for (int h = 0; h < H; ++h) {
            const float* sc = scores + ((size_t)b * H + h) * NB;
            int32_t* out = topk_ids + ((size_t)b * H + h) * K;
            int nf = 0, nr = 0;
            for (int j = 0; j < NB; ++j) {
                const int forced = j < sink_end || (j >= win_begin && j < n);
                if (forced) {
                    if (nf >= K) { rc = -1; break; }
                    out[nf++] = j;
                } else {
                    rest[nr].s = j < n ? sc[j] : -INFINITY;
                    rest[nr].id = j;
                    ++nr;
                }
            }
            if (rc) break;
            qsort(rest, (size_t)nr, sizeof(scored_id), cmp_score_desc_id_asc);
            for (int i = 0; nf + i < K; ++i) out[nf + i] = rest[i].id;
        }
    }
    free(rest);
    return rc;
}

typedef struct { int32_t last; int32_t blk; int32_t slot; } lru_entry;

/* LRU order: least recently used first; equal times by lower block id. */
static int cmp_lru(const void* pa, const void* pb)
{
    const lru_entry* a = (const lru_entry*)pa;
    const lru_entry* b = (const lru_entry*)pb;
    if (a->last != b->last) return (a->last > b->last) - (a->last < b->last);
    return (a->blk > b->blk) - (a->blk < b->blk);
}

static int cmp_int32(const void* pa, const void* pb)
{
    int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
    return (a > b) - (a < b);
}

/*
 * KV selection with capped eviction, [OasisKV] explanatory diagram step 3:
 * the predicted set P is compared with the set R resident in the GPU working
 * set and only the missing blocks are fetched, at most `cap` per step
 * (Tab. 2); victims are chosen by LRU (Tab. 2 caption).  The head-wise map
 * between GPU working-set slots and CPU blocks is Fig. 9: slot_of_block and
 * block_of_slot are that map, per (request, KV head).
 *
 * Steps for each (b, h), with t = step:
 *  1. M = P minus R, in topk_ids order (the fetch priority).  Blocks of P
 *     already resident are "used" at t: last_used[slot] = t.
 *  2. Fetch the first n = min(|M|, cap) blocks of M.
 *  3. Evict e = max(0, |R| + n - S) blocks of R minus P, least recently used
 *     first, ties by lower block id.
 *  4. Free slots = empty slots and the victims' slots, ascending slot index;
 *     the fetched blocks in ascending block id take the first n of them.
 *  5. Update both maps; fetched blocks get last_used = t.
 * Outputs: fetch_block/fetch_slot sorted by block id, evict_block sorted by
 * block id, entries past n (resp. e) set to -1; n_fetch = n, n_evict = e.
 * Returns 0, or a negative code when the state is inconsistent.
 */
int orc_plan_fetch(const orc_cfg* c, const int32_t* topk_ids, int32_t step,
                   int32_t* slot_of_block, int32_t* block_of_slot, int32_t* last_used,
                   int32_t* fetch_block, int32_t* fetch_slot, int32_t* evict_block,
                   int32_t* n_fetch, int32_t* n_evict)
{
    const int B = c->batch, H = c->num_kv_heads, NB = c->num_blocks, K = c->top_k;
    const int S = slots_of(c);
    const int cap = orc_fetch_cap(c);
    const int capw = cap > 0 ? cap : 1; /* row width of the output lists */
    int32_t* missing = (int32_t*)malloc(sizeof(int32_t) * (size_t)K);
    int32_t* fetched = (int32_t*)malloc(sizeof(int32_t) * (size_t)K);
    char* in_p = (char*)malloc((size_t)S);
    lru_entry* cand = (lru_entry*)malloc(sizeof(lru_entry) * (size_t)S);
    int32_t* freed = (int32_t*)malloc(sizeof(int32_t) * (size_t)S);
    int32_t* evicted = (int32_t*)malloc(sizeof(int32_t) * (size_t)S);
    char* seen = (char*)malloc((size_t)NB);
    int rc = 0;
    if (!missing || !fetched || !in_p || !cand || !freed || !evicted || !seen) rc = -9;

    for (int b = 0; b < B && rc == 0; ++b)
        for (int h = 0; h < H && rc == 0; ++h) {
            const size_t u = (size_t)b * H + h;
            const int32_t* P = topk_ids + u * K;
            int32_t* sob = slot_of_block + u * NB;
            int32_t* bos = block_of_slot + u * S;
            int32_t* lu = last_used + u * S;
            int32_t* fb = fetch_block + u * capw;
            int32_t* fs = fetch_slot + u * capw;
            int32_t* eb = evict_block + u * capw;
            int nm = 0, nres = 0, nc = 0, nfree = 0, n, e;

            memset(in_p, 0, (size_t)S);
            memset(seen, 0, (size_t)NB);
            /* step 1: hits are used at t; misses keep the priority order */
            for (int i = 0; i < K; ++i) {
                int32_t p = P[i];
                if (p < 0 || p >= NB) { rc = -1; break; }
                if (seen[p]) { rc = -4; break; }
                seen[p] = 1;
                int32_t s = sob[p];
                if (s >= 0) {
                    if (s >= S || bos[s] != p) { rc = -2; break; }
                    lu[s] = step;
                    in_p[s] = 1;
                } else {
                    missing[nm++] = p;
                }
            }
            if (rc) break;
            /* step 2 */
            n = nm < cap ? nm : cap;
            /* step 3: victims among R minus P */
            for (int s = 0; s < S; ++s) {
                if (bos[s] < 0) continue;
                ++nres;
                if (!in_p[s]) {
                    cand[nc].last = lu[s];
                    cand[nc].blk = bos[s];
                    cand[nc].slot = s;
                    ++nc;
                }
            }
            e = nres + n - S;
            if (e < 0) e = 0;
            if (e > nc) { rc = -3; break; }
            qsort(cand, (size_t)nc, sizeof(lru_entry), cmp_lru);
            /* step 4: free slots in ascending slot index */
            for (int s = 0; s < S; ++s) {
                int free_slot = bos[s] < 0;
                for (int v = 0; v < e && !free_slot; ++v) free_slot = (cand[v].slot == s);
                if (free_slot) freed[nfree++] = s;
            }
            memcpy(fetched, missing, sizeof(int32_t) * (size_t)n);
            qsort(fetched, (size_t)n, sizeof(int32_t), cmp_int32);
            for (int v = 0; v < e; ++v) evicted[v] = cand[v].blk;
            qsort(evicted, (size_t)e, sizeof(int32_t), cmp_int32);
            /* step 5: apply */
            for (int v = 0; v < e; ++v) {
                sob[cand[v].blk] = -1;
                bos[cand[v].slot] = -1;
            }
            for (int r = 0; r < n; ++r) {
                int32_t s = freed[r];
                bos[s] = fetched[r];
                sob[fetched[r]] = s;
                lu[s] = step;
            }
            for (int r = 0; r < capw; ++r) {
                fb[r] = r < n ? fetched[r] : -1;
                fs[r] = r < n ? freed[r] : -1;
                eb[r] = r < e ? evicted[r] : -1;
            }
            n_fetch[u] = n;
            n_evict[u] = e;
        }
    free(missing); free(fetched); free(in_p); free(cand); free(freed); free(evicted); free(seen);
    return rc;
}

/*
 * KV transfer, [OasisKV] Fig. 8 and explanatory diagram step 4: the selected
 * blocks' keys and values are copied from the CPU full cache into their
 * working-set slots.  A plain byte copy per block.
 * Returns 0, or -1 on an out-of-range block id or slot.
 */
int orc_fetch_blocks(const orc_cfg* c, const uint16_t* host_k, const uint16_t* host_v,
                     const int32_t* fetch_block, const int32_t* fetch_slot,
                     const int32_t* n_fetch, uint16_t* pool_k, uint16_t* pool_v)
{
    const int B = c->batch, H = c->num_kv_heads, NB = c->num_blocks, S = slots_of(c);
    const int cap = orc_fetch_cap(c), capw = cap > 0 ? cap : 1;
    const size_t blk_elems = (size_t)c->block_size * c->head_dim;
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            const size_t u = (size_t)b * H + h;
            if (n_fetch[u] < 0 || n_fetch[u] > cap) return -1;
            for (int r = 0; r < n_fetch[u]; ++r) {
                int32_t j = fetch_block[u * capw + r], s = fetch_slot[u * capw + r];
                if (j < 0 || j >= NB || s < 0 || s >= S) return -1;
                memcpy(pool_k + (u * S + s) * blk_elems, host_k + (u * NB + j) * blk_elems,
                       blk_elems * sizeof(uint16_t));
                memcpy(pool_v + (u * S + s) * blk_elems, host_v + (u * NB + j) * blk_elems,
                       blk_elems * sizeof(uint16_t));
            }
        }
    return 0;
}

/*
 * Decode-time append (the decode loop of [OasisKV] Fig. 8 advances one token
 * per step; the page leaves the bookkeeping open, these are the readings):
 * for each request b the new token sits at position p = ctx_len[b], in block
 * j = p / bs, row t = p % bs, for every KV head h.
 *  1. The full cache gets the token: host K/V [b,h,j,t,:] = k_new/v_new [b,h,:].
 *  2. The working set holds the newest block, so that the token attends to
 *     itself and to the tokens just before it: if block j is not resident it
 *     takes a slot now -- the lowest empty slot, else the least recently used
 *     resident block that is not forced in the grown context (sink and local
 *     window of n = j + 1 blocks, as in orc_select_topk_ctx), ties by lower
 *     block id -- with last_used = the step, and rows 0..t-1 of the block are
 *     copied in from the full cache.  Row t of the slot gets the token.
 *  3. ctx_len[b] = p + 1.
 * The block's compressed keys follow with orc_refresh_summaries.
 * The step is clock[b*H+h] when clock is given, else `step`.  A request whose
 * context is full (p >= NB*bs) or negative is left unchanged and the call
 * returns -1; a head with no slot to give (every resident block forced, none
 * empty) gets row 1 only and the call returns -2.  Returns 0 otherwise.
 */
int orc_append_kv(const orc_cfg* c, const uint16_t* k_new, const uint16_t* v_new,
                  int32_t* ctx_len, const int32_t* clock, int32_t step, uint16_t* host_k,
                  uint16_t* host_v, int32_t* slot_of_block, int32_t* block_of_slot,
                  int32_t* last_used, uint16_t* pool_k, uint16_t* pool_v)
{
    const int B = c->batch, H = c->num_kv_heads, NB = c->num_blocks;
    const int bs = c->block_size, D = c->head_dim, S = slots_of(c);
    int rc = 0;
    for (int b = 0; b < B; ++b) {
        const int32_t p = ctx_len[b];
        if (p < 0 || (long long)p >= (long long)NB * bs) { rc = -1; continue; }
        const int j = p / bs, t = p % bs;
        const int n = j + 1;
        const int sink_end = c->sink_blocks < n ? c->sink_blocks : n;
        const int win_begin = n - c->local_blocks > 0 ? n - c->local_blocks : 0;
        for (int h = 0; h < H; ++h) {
            const size_t u = (size_t)b * H + h;
            const size_t row = ((u * NB + j) * bs + t) * D;
            int32_t* sob = slot_of_block + u * NB;
            int32_t* bos = block_of_slot + u * S;
            int32_t* lu = last_used + u * S;
            /* 1 */
            memcpy(host_k + row, k_new + u * D, sizeof(uint16_t) * D);
            memcpy(host_v + row, v_new + u * D, sizeof(uint16_t) * D);
            /* 2 */
            int32_t s = sob[j];
            if (s < 0) {
                int best = -1;
                for (int q = 0; q < S && best < 0; ++q)
                    if (bos[q] < 0) best = q;
                if (best < 0)
                    for (int q = 0; q < S; ++q) {
                        const int32_t blk = bos[q];
                        if (blk < sink_end || (blk >= win_begin && blk < n)) continue;
                        if (best < 0 || lu[q] < lu[best] || (lu[q] == lu[best] && blk < bos[best]))
                            best = q;
                    }
                if (best < 0) {
                    rc = rc ? rc : -2;
                } else {
                    if (bos[best] >= 0) sob[bos[best]] = -1;
                    bos[best] = j;
                    sob[j] = best;
                    lu[best] = clock ? clock[u] : step;
                    s = best;
                    for (int r = 0; r < t; ++r) {
                        memcpy(pool_k + ((u * S + s) * bs + r) * D, host_k + ((u * NB + j) * bs + r) * D,
                               sizeof(uint16_t) * D);
                        memcpy(pool_v + ((u * S + s) * bs + r) * D, host_v + ((u * NB + j) * bs + r) * D,
                               sizeof(uint16_t) * D);
                    }
                }
            }
            if (s >= 0) {
                memcpy(pool_k + ((u * S + s) * bs + t) * D, k_new + u * D, sizeof(uint16_t) * D);
                memcpy(pool_v + ((u * S + s) * bs + t) * D, v_new + u * D, sizeof(uint16_t) * D);
            }
        }
        /* 3 */
        ctx_len[b] = p + 1;
    }
    return rc;
}

/*
 * Compressed keys of each context's newest block after an append ([OasisKV]
 * Fig. 7 left, over a growing context).  Reading: a block's summary covers
 * its tokens inside the context.  For request b the last token is
 * p = ctx_len[b] - 1 (nothing to do for an empty context); its block
 * j = p / bs holds rows 0..t, t = p % bs, and for every KV head:
 *   summ[b,h,j,:]  = the mean of those rows (summed in double in row order,
 *                    divided by t + 1, rounded once to fp32);
 *   summ_mm        (if given) their elementwise max and min, first row first
 *                    on equal values, as orc_build_summaries_minmax.
 * With a full block this is the summary orc_build_summaries gives.
 */
void orc_refresh_summaries(const orc_cfg* c, const int32_t* ctx_len, const uint16_t* host_k,
                           float* summ, uint16_t* summ_mm)
{
    const int B = c->batch, H = c->num_kv_heads, NB = c->num_blocks;
    const int bs = c->block_size, D = c->head_dim;
    for (int b = 0; b < B; ++b) {
        const long long p = (long long)ctx_len[b] - 1;
        if (p < 0) continue;
        const int j = (int)(p / bs), t = (int)(p % bs);
        if (j >= NB) continue;
        for (int h = 0; h < H; ++h) {
            const size_t u = (size_t)b * H + h;
            for (int d = 0; d < D; ++d) {
                const uint16_t* kb = host_k + (u * NB + j) * bs * D + d;
                double sum = 0.0;
                uint16_t hi = kb[0], lo = kb[0];
                for (int r = 0; r <= t; ++r) {
                    sum += bf16_to_double(kb[(size_t)r * D]);
                    if (bf16_to_double(kb[(size_t)r * D]) > bf16_to_double(hi)) hi = kb[(size_t)r * D];
                    if (bf16_to_double(kb[(size_t)r * D]) < bf16_to_double(lo)) lo = kb[(size_t)r * D];
                }
                summ[(u * NB + j) * D + d] = (float)(sum / (double)(t + 1));
                if (summ_mm) {
                    summ_mm[((u * NB + j) * 2 + 0) * D + d] = hi;
                    summ_mm[((u * NB + j) * 2 + 1) * D + d] = lo;
                }
            }
        }
    }
}

/*
 * Sparse decode attention over the working set, [OasisKV] Fig. 7 (right):
 * each query head attends to the keys and values held in the bounded GPU
 * working set of its KV head (GQA: query head h*G+g reads KV head h).
 * Reading: every valid slot (block_of_slot >= 0) is attended, and token
 * j*bs+t of block j takes part only if it is below ctx_len[b] (all tokens
 * when ctx_len is NULL).  Exact softmax in double, two passes (maximum, then
 * weights); a head with no visible token outputs zeros.
 */
void orc_sparse_decode_attn(const orc_cfg* c, const uint16_t* q, const uint16_t* pool_k,
                            const uint16_t* pool_v, const int32_t* block_of_slot,
                            const int32_t* ctx_len, double scale, float* out)
{
    const int B = c->batch, H = c->num_kv_heads, Hq = c->num_q_heads, G = Hq / H;
    const int S = slots_of(c), bs = c->block_size, D = c->head_dim;
    double* acc = (double*)malloc(sizeof(double) * (size_t)D);
    if (!acc) return;
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
            for (int g = 0; g < G; ++g) {
                const int hq = h * G + g;
                const uint16_t* qv = q + ((size_t)b * Hq + hq) * D;
                const size_t u = (size_t)b * H + h;
                double mx = -INFINITY, den = 0.0;
                /* pass 1: maximum logit */
                for (int s = 0; s < S; ++s) {
                    int32_t j = block_of_slot[u * S + s];
                    if (j < 0) continue;
                    for (int t = 0; t < bs; ++t) {
                        if (ctx_len && (int64_t)j * bs + t >= ctx_len[b]) continue;
                        const uint16_t* kv = pool_k + ((u * S + s) * bs + t) * D;
                        double x = 0.0;
                        for (int d = 0; d < D; ++d) x += bf16_to_double(qv[d]) * bf16_to_double(kv[d]);
                        x *= scale;
                        if (x > mx) mx = x;
                    }
                }
                for (int d = 0; d < D; ++d) acc[d] = 0.0;
                /* pass 2: weights and weighted values */
                if (mx > -INFINITY) {
                    for (int s = 0; s < S; ++s) {
                        int32_t j = block_of_slot[u * S + s];
                        if (j < 0) continue;
                        for (int t = 0; t < bs; ++t) {
                            if (ctx_len && (int64_t)j * bs + t >= ctx_len[b]) continue;
                            const uint16_t* kv = pool_k + ((u * S + s) * bs + t) * D;
                            const uint16_t* vv = pool_v + ((u * S + s) * bs + t) * D;
                            double x = 0.0;
                            for (int d = 0; d < D; ++d) x += bf16_to_double(qv[d]) * bf16_to_double(kv[d]);
                            double w = exp(x * scale - mx);
                            den += w;
                            for (int d = 0; d < D; ++d) acc[d] += w * bf16_to_double(vv[d]);
                        }
                    }
                }
                float* o = out + ((size_t)b * Hq + hq) * D;
                for (int d = 0; d < D; ++d) o[d] = den > 0.0 ? (float)(acc[d] / den) : 0.0f;
            }
    free(acc);
}

/*
 * Dense decode attention over the full context (the "Full" anchor of
 * [OasisKV] Tab. 1): textbook softmax(q k^T * scale) v over every token
 * n < ctx_len[b] (all NB*bs tokens when ctx_len is NULL) of the host cache.
 * Used to pin the sparse path: with every block resident the two agree.
 */
void orc_dense_decode_attn(const orc_cfg* c, const uint16_t* q, const uint16_t* k,
                           const uint16_t* v, const int32_t* ctx_len, double scale,
                           float* out)
{
    const int B = c->batch, H = c->num_kv_heads, Hq = c->num_q_heads, G = Hq / H;
    const int NB = c->num_blocks, bs = c->block_size, D = c->head_dim;
    const int64_t ntok_all = (int64_t)NB * bs;
    double* logit = (double*)malloc(sizeof(double) * (size_t)ntok_all);
    double* acc = (double*)malloc(sizeof(double) * (size_t)D);
    if (!logit || !acc) { free(logit); free(acc); return; }
    for (int b = 0; b < B; ++b) {
        int64_t ntok = ctx_len ? ctx_len[b] : ntok_all;
        if (ntok > ntok_all) ntok = ntok_all;
        for (int hq = 0; hq < Hq; ++hq) {
            const int h = hq / G;
            const uint16_t* qv = q + ((size_t)b * Hq + hq) * D;
            const uint16_t* kb = k + ((size_t)b * H + h) * (size_t)ntok_all * D;
            const uint16_t* vb = v + ((size_t)b * H + h) * (size_t)ntok_all * D;
            double mx = -INFINITY, den = 0.0;
            for (int64_t n = 0; n < ntok; ++n) {
                double x = 0.0;
                for (int d = 0; d < D; ++d) x += bf16_to_double(qv[d]) * bf16_to_double(kb[n * D + d]);
                logit[n] = x * scale;
                if (logit[n] > mx) mx = logit[n];
            }
            for (int d = 0; d < D; ++d) acc[d] = 0.0;
            for (int64_t n = 0; n < ntok; ++n) {
                double w = exp(logit[n] - mx);
                den += w;
                for (int d = 0; d < D; ++d) acc[d] += w * bf16_to_double(vb[n * D + d]);
            }
            float* o = out + ((size_t)b * Hq + hq) * D;
            for (int d = 0; d < D; ++d) o[d] = den > 0.0 ? (float)(acc[d] / den) : 0.0f;
        }
    }
    free(logit);
    free(acc);
}
