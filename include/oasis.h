/*
 * oasis.h -- C ABI of liboasis, the GB300 (sm_103a) decode hot path of
 * look-ahead sparse KV prefetching.
 *
 * Method: "OasisKV: Scaling In-Decode KV Cache Beyond HBM with Lookahead
 * Sparse Prefetching" (arXiv:2608.08097; cited below as [OasisKV] with the
 * figure, table or step of its summary page).  The full KV cache of every
 * layer lives in pinned host memory; each (request, KV head) keeps a bounded
 * working set of S = kv_budget_tokens / block_size KV blocks in HBM
 * ([OasisKV] Fig. 7 left, Fig. 9).  Once per layer and decode step:
 *
 *   oasis_sparse_decode_attn   attention over the working set      (Fig. 7 right)
 *   oasis_attend_and_score     attention of one layer + scoring of another in one launch (Fig. 8)
 *     (_minmax: the same with min/max-pooled keys)
 *   oasis_sparse_decode_attn_joint  decoded + draft tokens in one pass of the working set (Fig. 7 right)
 *   oasis_score_blocks         draft queries scan compressed keys  (Fig. 7 right)
 *   oasis_score_blocks_minmax  the same against min/max-pooled keys (Fig. 7 left)
 *   oasis_select_topk          top-K blocks per KV head            (diagram step 2)
 *     (_ctx, and oasis_predict_select_ctx: local window at each context's end)
 *   oasis_predict_chain        scoring + top-K + plan in one launch (diagram steps 2-3)
 *   oasis_plan_fetch           diff vs. working set, capped LRU    (diagram step 3, Tab. 2)
 *   oasis_fetch_blocks         host -> HBM transfer, copy stream   (diagram step 4, Fig. 8)
 *   oasis_append_kv            the decoded token joins cache and working set (Fig. 8)
 *   oasis_refresh_summaries    the newest block's compressed keys follow (Fig. 7 left)
 *
 * Conventions
 *   - All pointers except `cfg` and the outputs of the query functions are
 *     DEVICE-accessible addresses.  `host_k`/`host_v` point to pinned host
 *     memory mapped into the device address space (cudaHostAlloc with
 *     cudaHostAllocMapped, or cudaHostRegister + cudaHostGetDevicePointer).
 *   - bf16 tensors are passed as `uint16_t*` holding bf16 bit patterns.
 *   - Streams are `cudaStream_t` values passed as `void*` (NULL = legacy
 *     default stream).  Every call only enqueues work on the stream it is
 *     given and returns; ordering across streams is the caller's (events).
 *   - The caller owns every buffer.  The library allocates no device or host
 *     memory, except a few bytes of per-device state (a device error word)
 *     created on the first call on each device.
 *   - Arguments are validated before anything is launched.  Invalid ones
 *     return OASIS_ERR_INVALID_ARG (or OASIS_ERR_UNSUPPORTED for legal but
 *     unimplemented shapes) and launch nothing.  A failed launch returns
 *     OASIS_ERR_CUDA.  Problems only visible on the device (an out-of-range
 *     id inside a device array, a bounded wait that ran out) never trap: the
 *     kernel skips the offending access and sets a bit in the per-device
 *     error word, read with oasis_device_errors().
 *
 * Layouts (row-major; B batch, Hq query heads, Hkv KV heads, G = Hq/Hkv,
 * D = head_dim = 128, bs = block_size = 16, NB = num_blocks, L = lookahead,
 * K = top_k, S = slots, cap = oasis_fetch_cap(cfg); query head h*G+g reads
 * KV head h):
 *   host K, V       [B][Hkv][NB][bs][D]  bf16  full cache, pinned host
 *   summ            [B][Hkv][NB][D]      fp32  compressed keys (block means)
 *   summ_mm         [B][Hkv][NB][2][D]   bf16  min/max compressed keys (max row, min row)
 *   q_draft         [B][L][Hq][D]        bf16  draft-token queries
 *   scores          [B][Hkv][NB]         fp32
 *   topk_ids        [B][Hkv][K]          int32 in priority order
 *   slot_of_block   [B][Hkv][NB]         int32 working-set slot, -1 = absent
 *   block_of_slot   [B][Hkv][S]          int32 block in the slot, -1 = empty
 *   last_used       [B][Hkv][S]          int32 step of last use, -1 = never
 *   fetch_block, fetch_slot, evict_block [B][Hkv][max(cap,1)] int32, -1 padded
 *   n_fetch, n_evict [B][Hkv]            int32
 *   pool K, V       [B][Hkv][S][bs][D]   bf16  working set in HBM
 *   q               [B][Hq][D]           bf16  decode query
 *   out             [B][Hq][D]           bf16
 */
#ifndef OASIS_H
#define OASIS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    OASIS_OK = 0,
    OASIS_ERR_INVALID_ARG = 1,  /* bad pointer, size, alignment or configuration */
    OASIS_ERR_UNSUPPORTED = 2,  /* legal shape this build does not implement */
    OASIS_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
    OASIS_ERR_TIMEOUT = 4       /* oasis_stream_wait ran out of time */
} oasis_status_t;

/* Bits of the per-device error word (oasis_device_errors). */
#define OASIS_DEVERR_FETCH_RANGE  0x1u  /* fetch list entry out of range; copy skipped */
#define OASIS_DEVERR_PLAN_STATE   0x2u  /* inconsistent working-set map; (b,h) left unchanged */
#define OASIS_DEVERR_TOPK_IDS     0x4u  /* top-K id out of range or repeated; (b,h) left unchanged */
#define OASIS_DEVERR_WAIT_TIMEOUT 0x8u  /* a bounded device wait gave up; outputs invalid */
#define OASIS_DEVERR_SLOT_RANGE   0x10u /* block_of_slot entry >= NB; slot skipped */
#define OASIS_DEVERR_CTX_FULL     0x20u /* append: context at capacity (NB*bs) or negative; request skipped */
#define OASIS_DEVERR_NO_SLOT      0x40u /* append: newest block not resident and every slot forced; pool not written */

/* Per-layer problem description ([OasisKV] diagram steps 2-3, Tab. 1-2):
 * block size, KV budget, look-ahead tokens, top-K and fetch ratio. */
typedef struct {
    int32_t batch;             /* B requests */
    int32_t num_q_heads;       /* Hq */
    int32_t num_kv_heads;      /* Hkv; Hq % Hkv == 0 */
    int32_t head_dim;          /* D; this build: 128 */
    int32_t block_size;        /* tokens per KV block; this build: 16 */
    int32_t num_blocks;        /* NB context blocks per (request, KV head) */
    int32_t kv_budget_tokens;  /* working-set budget; S = kv_budget_tokens / block_size */
    int32_t lookahead;         /* L draft tokens */
    int32_t top_k;             /* K predicted blocks per KV head, K <= S, K <= NB */
    float   fetch_ratio;       /* per-step fetch cap = ceil(ratio*S); <0 or >=1: cap = K */
    int32_t sink_blocks;       /* blocks [0, sink) are always predicted */
    int32_t local_blocks;      /* the last `local` blocks are always predicted */
} oasis_config_t;

/* Checks a configuration without launching anything.  OASIS_OK,
 * OASIS_ERR_INVALID_ARG or OASIS_ERR_UNSUPPORTED.  Limits of this build:
 * head_dim 128, block_size 16, G <= 8, L*G <= 64, S <= 1024, K <= 1024,
 * NB <= 32768, B*Hkv <= 65535, (sink + local) <= K. */
oasis_status_t oasis_validate_config(const oasis_config_t* cfg);

/* Blocks fetched at most per (request, KV head) and step ([OasisKV] Tab. 2:
 * the fetch ratio bounds the blocks fetched per step).  The ratio applies to
 * the budget in blocks: cap = ceil(ratio * S - 1e-6) in double, clamped to
 * [0, K]; a ratio < 0 or >= 1 ("fetch all") gives K.  Returns -1 for an
 * invalid configuration. */
int32_t oasis_fetch_cap(const oasis_config_t* cfg);

/* Compressed keys ([OasisKV] Fig. 7 left): summ[b,h,j,:] = fp32 mean of the
 * bs keys of block j, the sum taken exactly and rounded once.  Set-up work
 * (admission), not part of the per-step path.  `k` may be a device buffer or
 * mapped pinned host memory, 16-byte aligned; `summ` 16-byte aligned. */
oasis_status_t oasis_build_summaries(const oasis_config_t* cfg, const uint16_t* k,
                                     float* summ, void* stream);

/* Look-ahead scoring ([OasisKV] Fig. 7 right; 'What they did' item 2):
 * scores[b,h,j] = max over l < L, g < G of  q_draft[b,l,h*G+g,:] . summ[b,h,j,:].
 * Tensor-core contraction with fp32 accumulation; the fp32 summary enters as
 * a two-term tf32 split (tf32 head plus tf32-rounded residual, about 2^-22
 * relative per term), so the result is within a few fp32 ulps of the exact
 * value.  q_draft and summ 16-byte aligned. */
oasis_status_t oasis_score_blocks(const oasis_config_t* cfg, const uint16_t* q_draft,
                                  const float* summ, float* scores, void* stream);

/* Min/max compressed keys, the pooling [OasisKV] Fig. 7 (left) names:
 *   summ_mm[b,h,j,0,:] = elementwise max of the bs keys of block j,
 *   summ_mm[b,h,j,1,:] = elementwise min,
 * bf16 values copied from the keys (exact; on equal values the earlier
 * token's bit pattern, which decides +0 / -0).  Layout [B][Hkv][NB][2][D]
 * bf16: 512 bytes per block, as many as the fp32 mean.  Set-up work, like
 * oasis_build_summaries; k and summ_mm 16-byte aligned. */
oasis_status_t oasis_build_summaries_minmax(const oasis_config_t* cfg, const uint16_t* k,
                                            uint16_t* summ_mm, void* stream);

/* Look-ahead scoring against min/max compressed keys:
 *   scores[b,h,j] = max over l < L, g < G of
 *                   sum_d max(q_d * min_d, q_d * max_d),  q = q_draft[b,l,h*G+g,:],
 * an upper bound of q . k for every key k of the block.  Computed as the dot
 * product of [max(q,0) | min(q,0)] with [max | min] on bf16 tensor cores:
 * exact products, fp32 accumulation of 256 terms (error at most about
 * 256 * 2^-23 of sum_d |q_d| * max(|min_d|, |max_d|)).  Same scores layout as
 * oasis_score_blocks, so oasis_select_topk and the planning follow unchanged.
 * L*G <= 32 (else OASIS_ERR_UNSUPPORTED).  q_draft and summ_mm 16-byte
 * aligned, scores 8-byte aligned. */
oasis_status_t oasis_score_blocks_minmax(const oasis_config_t* cfg, const uint16_t* q_draft,
                                         const uint16_t* summ_mm, float* scores, void* stream);

/* Per-KV-head top-K ([OasisKV] diagram step 2, Fig. 4).  Forced blocks (sink
 * and local window) come first in ascending id and count toward K; the other
 * K - |forced| are the highest scores, equal scores to the lower id, listed
 * by (score descending, id ascending).  The list order is the fetch priority
 * used by oasis_plan_fetch.  Scores must not be NaN (-0.0 equals +0.0). */
oasis_status_t oasis_select_topk(const oasis_config_t* cfg, const float* scores,
                                 int32_t* topk_ids, void* stream);

/* Top-K over a growing context ([OasisKV] 'What they did' item 4 as decoding
 * appends tokens): as oasis_select_topk, with n = ceil(ctx_len[b] / bs) (at
 * most NB) blocks in request b's context: the forced blocks are the sink
 * [0, min(sink, n)) and the local window [max(n - local, 0), n), and blocks
 * at or beyond n rank as if scored -infinity (picked, lowest id first, only
 * when the context has fewer than K blocks).  ctx_len [B] int32 on the device.
 * With ctx_len[b] = NB*bs for every b the result is oasis_select_topk's. */
oasis_status_t oasis_select_topk_ctx(const oasis_config_t* cfg, const float* scores,
                                     const int32_t* ctx_len, int32_t* topk_ids, void* stream);

/* Selection with capped eviction ([OasisKV] diagram step 3; Tab. 2 "LRU
 * eviction"; Fig. 9 head-wise block map).  Per (b,h), with P = topk_ids and R
 * the resident blocks:
 *   1. blocks of P already in R are used at `step` (last_used = step);
 *   2. the first n = min(|P \ R|, cap) missing blocks in list order are fetched;
 *   3. e = max(0, |R| + n - S) victims leave R \ P, least recently used first,
 *      equal times by lower block id;
 *   4. free slots (empty, then freed; ascending slot index) are paired with
 *      the fetched blocks in ascending block id; they get last_used = step.
 * The three state arrays are updated in place.  Outputs are sorted by block
 * id and padded with -1.  The caller must not run this while an attention
 * call still reads the same block_of_slot, nor fetch into the pool until the
 * attention over the old working set has finished (victim slots are reused). */
oasis_status_t oasis_plan_fetch(const oasis_config_t* cfg, const int32_t* topk_ids,
                                int32_t step, int32_t* slot_of_block,
                                int32_t* block_of_slot, int32_t* last_used,
                                int32_t* fetch_block, int32_t* fetch_slot,
                                int32_t* evict_block, int32_t* n_fetch,
                                int32_t* n_evict, void* stream);

/* oasis_plan_fetch with the step kept in device memory: clock is [B][Hkv]
 * int32; each (b,h) plans at step clock[b,h] and the call then advances it by
 * one.  With every clock equal to t on entry the result is that of
 * oasis_plan_fetch(..., step = t, ...).  No host value changes from one
 * decode step to the next, so a captured CUDA graph of the layer step can be
 * replayed step after step. */
oasis_status_t oasis_plan_fetch_clocked(const oasis_config_t* cfg, const int32_t* topk_ids,
                                        int32_t* clock, int32_t* slot_of_block,
                                        int32_t* block_of_slot, int32_t* last_used,
                                        int32_t* fetch_block, int32_t* fetch_slot,
                                        int32_t* evict_block, int32_t* n_fetch,
                                        int32_t* n_evict, void* stream);

/* Top-K and planning of one layer-step in one launch ([OasisKV] explanatory
 * diagram steps 2-3): the result is exactly that of oasis_select_topk
 * followed by oasis_plan_fetch (or oasis_plan_fetch_clocked when `clock` is
 * not NULL, in which case `step` is ignored), with the top-K list of each
 * (request, KV head) kept on chip in between.  topk_ids is still written. */
oasis_status_t oasis_predict_select(const oasis_config_t* cfg, const float* scores,
                                    int32_t step, int32_t* clock, int32_t* topk_ids,
                                    int32_t* slot_of_block, int32_t* block_of_slot,
                                    int32_t* last_used, int32_t* fetch_block,
                                    int32_t* fetch_slot, int32_t* evict_block,
                                    int32_t* n_fetch, int32_t* n_evict, void* stream);

/* The whole prediction chain in one launch ([OasisKV] Fig. 7 right, diagram
 * steps 2-3): oasis_score_blocks(cfg, q_draft, summ, scores) followed by
 * oasis_predict_select(cfg, scores, step, clock, ...), with the same results
 * bit for bit (scores are written too).  The CTAs scoring one (request, KV
 * head) form a thread-block cluster; after a cluster barrier the unit's first
 * CTA selects and plans.  Supported: L*G <= 32, S <= 256, K <= 256,
 * NB <= 8192 (else OASIS_ERR_UNSUPPORTED).  Alignment as for the two calls. */
oasis_status_t oasis_predict_chain(const oasis_config_t* cfg, const uint16_t* q_draft,
                                   const float* summ, float* scores, int32_t step, int32_t* clock,
                                   int32_t* topk_ids, int32_t* slot_of_block,
                                   int32_t* block_of_slot, int32_t* last_used,
                                   int32_t* fetch_block, int32_t* fetch_slot, int32_t* evict_block,
                                   int32_t* n_fetch, int32_t* n_evict, void* stream);

/* oasis_predict_select with the top-K of oasis_select_topk_ctx (the window
 * follows each request's context length ctx_len [B]). */
oasis_status_t oasis_predict_select_ctx(const oasis_config_t* cfg, const float* scores,
                                        const int32_t* ctx_len, int32_t step, int32_t* clock,
                                        int32_t* topk_ids, int32_t* slot_of_block,
                                        int32_t* block_of_slot, int32_t* last_used,
                                        int32_t* fetch_block, int32_t* fetch_slot,
                                        int32_t* evict_block, int32_t* n_fetch, int32_t* n_evict,
                                        void* stream);

/* Decode-time append ([OasisKV] Fig. 8: the decode loop advances a token per
 * step) of one token per request, at position p = ctx_len[b] (row t = p % bs
 * of block j = p / bs), for every KV head h:
 *   1. host K/V [b,h,j,t,:] = k_new/v_new [b,h,:] (host_k/host_v: mapped
 *      pinned memory, their device addresses);
 *   2. the working set holds the newest block: if block j is not resident it
 *      takes the lowest empty slot, else the slot of the least recently used
 *      resident block that is not forced in the grown context (sink and
 *      local window of j + 1 blocks), ties by lower block id; the maps are
 *      updated, last_used = clock[b*Hkv+h] (clock given) or `step`, and rows
 *      0..t-1 are copied in from the host cache.  Row t of the slot gets the
 *      token;
 *   3. ctx_len[b] = p + 1.
 * The block's compressed keys follow with oasis_refresh_summaries, which may
 * run on another stream beside the attention.  k_new, v_new [B][Hkv][D] bf16
 * (8-byte aligned); ctx_len [B] int32, read and advanced on the device.  A
 * request whose context is at capacity (p >= NB*bs) is skipped and flags
 * OASIS_DEVERR_CTX_FULL.  A head whose newest block finds no slot (every
 * resident block forced) would write the cache only and flag
 * OASIS_DEVERR_NO_SLOT; with a valid configuration this cannot happen (at
 * most K <= S forced blocks, the newest one among them), so the flag marks a
 * broken working set.  Hkv <= 32.  Order it after the step's reads of the
 * same slots (attention) and before the next planning of the same layer. */
oasis_status_t oasis_append_kv(const oasis_config_t* cfg, const uint16_t* k_new,
                               const uint16_t* v_new, int32_t* ctx_len, const int32_t* clock,
                               int32_t step, uint16_t* host_k, uint16_t* host_v,
                               int32_t* slot_of_block, int32_t* block_of_slot, int32_t* last_used,
                               uint16_t* pool_k, uint16_t* pool_v, void* stream);

/* Compressed keys of each context's newest block over its rows inside the
 * context ([OasisKV] Fig. 7 left, as the context grows): with p = ctx_len[b]
 * - 1 (nothing for an empty context), block j = p / bs, rows 0..t, t = p % bs:
 *   summ[b,h,j,:]   = fp32 mean of the rows (double sum in row order,
 *                     divided by t+1, rounded once), for every KV head h;
 *   summ_mm         (may be NULL) their max and min rows, bf16.
 * For a full block this equals oasis_build_summaries(_minmax).  The rows are
 * read from the working set when the block is resident (pool_k), else from
 * the host cache; the two hold the same keys.  Call after oasis_append_kv
 * (ordered after it), before the layer's next scoring. */
oasis_status_t oasis_refresh_summaries(const oasis_config_t* cfg, const int32_t* ctx_len,
                                       const uint16_t* host_k, const int32_t* slot_of_block,
                                       const uint16_t* pool_k, float* summ, uint16_t* summ_mm,
                                       void* stream);

/* KV transfer ([OasisKV] diagram step 4, Fig. 8): for every r < n_fetch[b,h],
 * copies block fetch_block[b,h,r] of host K and V into slot fetch_slot[b,h,r]
 * of the pools.  A gather kernel reads the mapped pinned host memory directly
 * (zero-copy over the host link); meant for a dedicated copy stream so that it
 * overlaps compute.  All of host_k, host_v, pool_k, pool_v 16-byte aligned. */
oasis_status_t oasis_fetch_blocks(const oasis_config_t* cfg, const uint16_t* host_k,
                                  const uint16_t* host_v, const int32_t* fetch_block,
                                  const int32_t* fetch_slot, const int32_t* n_fetch,
                                  uint16_t* pool_k, uint16_t* pool_v, void* copy_stream);

/* Sparse decode attention over the working set ([OasisKV] Fig. 7 right):
 * out[b,h*G+g,:] = softmax over every token t of every valid slot s
 * (block_of_slot >= 0, block*bs + t < ctx_len[b]) of scale * q.k, times v.
 * One pass, online softmax, fp32 accumulation, bf16 output; a head with no
 * visible token outputs zeros.  ctx_len is [B] int32 or NULL (no mask).
 * The kernel keeps all of its scratch in shared memory (each unit's CTAs merge
 * through distributed shared memory); `workspace` is accepted for
 * compatibility and never touched: at least oasis_attn_workspace_bytes(cfg)
 * bytes, 256-byte aligned.  q, pools and out 16-byte aligned; scale > 0. */
oasis_status_t oasis_sparse_decode_attn(const oasis_config_t* cfg, const uint16_t* q,
                                        const uint16_t* pool_k, const uint16_t* pool_v,
                                        const int32_t* block_of_slot, const int32_t* ctx_len,
                                        float scale, uint16_t* out, void* workspace,
                                        size_t workspace_bytes, void* stream);

/* Scratch bytes oasis_sparse_decode_attn needs for `cfg` (0 on invalid cfg). */
size_t oasis_attn_workspace_bytes(const oasis_config_t* cfg);

/* oasis_sparse_decode_attn for callers that cannot allocate device memory --
 * for example code running inside another framework's memory pool or
 * allocator hooks, under a device-memory quota, or on a latency-critical path
 * where a cudaMalloc (which may synchronize) is not acceptable.  The method's
 * pages have no counterpart: this is a deployment convenience.
 * Same arguments and result as oasis_sparse_decode_attn, without the
 * workspace: its scratch is a fixed 8 MiB array in device memory that every
 * GPU that loads this library holds until the process exits.  The caller
 * still owns q, the pools, block_of_slot, ctx_len and out.  Nothing is
 * allocated: no cudaMalloc, no cudaFree, no allocating library call.
 * Configurations needing more scratch than 8 MiB (see
 * oasis_attn_workspace_bytes) return OASIS_ERR_UNSUPPORTED and launch
 * nothing.  The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call before
 * any stream capture.  The current attention kernel keeps all its scratch in
 * shared memory, so the array is passed but not written, and calls on
 * different streams do not interfere. */
oasis_status_t oasis_sparse_decode_attn_static(const oasis_config_t* cfg, const uint16_t* q,
                                               const uint16_t* pool_k, const uint16_t* pool_v,
                                               const int32_t* block_of_slot,
                                               const int32_t* ctx_len, float scale,
                                               uint16_t* out, void* stream);

/* The attention of one layer and the look-ahead scoring of another, with the
 * same configuration, in one launch: exactly oasis_sparse_decode_attn(cfg, q,
 * pool_k, pool_v, block_of_slot, ctx_len, scale, out) and
 * oasis_score_blocks(cfg, q_draft, summ, scores), bit for bit, with the SMs
 * shared between the two by construction ([OasisKV] Fig. 8: a layer's
 * prediction runs in the background of the following layers' compute).  The
 * two must not share output memory.  Same argument rules as the two calls.
 * Launched as a programmatic dependent of the previous kernel in `stream`:
 * it may start while that kernel finishes, and reads nothing before that
 * kernel's results are visible, so stream order holds as for any launch. */
oasis_status_t oasis_attend_and_score(const oasis_config_t* cfg, const uint16_t* q,
                                      const uint16_t* pool_k, const uint16_t* pool_v,
                                      const int32_t* block_of_slot, const int32_t* ctx_len,
                                      float scale, uint16_t* out, const uint16_t* q_draft,
                                      const float* summ, float* scores, void* stream);

/* oasis_attend_and_score with the min/max compressed keys:
 * oasis_sparse_decode_attn(cfg, q, ...) and oasis_score_blocks_minmax(cfg,
 * q_draft, summ_mm, scores) in one launch, bit for bit.  L*G <= 32. */
oasis_status_t oasis_attend_and_score_minmax(const oasis_config_t* cfg, const uint16_t* q,
                                             const uint16_t* pool_k, const uint16_t* pool_v,
                                             const int32_t* block_of_slot, const int32_t* ctx_len,
                                             float scale, uint16_t* out, const uint16_t* q_draft,
                                             const uint16_t* summ_mm, float* scores,
                                             void* stream);

/* Joint attention of the decoded token and the L draft tokens over the same
 * working set, in one pass over its K and V ([OasisKV] Fig. 7 right: the
 * attention kernel processes the normal and the draft queries together).
 *   out[b, 0, n, :] = the oasis_sparse_decode_attn output for q[b, n, :]
 *   out[b, l, n, :] = the same attention with q_draft[b, l-1, n, :] as the
 *                     query, 1 <= l <= L
 * with the same slots, context mask and scale for all 1 + L rows (the draft
 * tokens' own keys are not in the cache).
 *   q        [B][Hq][D]         bf16
 *   q_draft  [B][L][Hq][D]      bf16
 *   out      [B][1+L][Hq][D]    bf16 (written in full; every row of a unit
 *                               whose slots are all empty or masked is 0)
 * Pools, block_of_slot, ctx_len and scale as for oasis_sparse_decode_attn.
 * Needs no workspace.  q, q_draft, pools and out 16-byte aligned; scale > 0.
 * Any group size G: the G*(1+L) rows of a KV head are taken 24 at a time,
 * and each further 24 rows stream the head's slots once more. */
oasis_status_t oasis_sparse_decode_attn_joint(const oasis_config_t* cfg, const uint16_t* q,
                                              const uint16_t* q_draft, const uint16_t* pool_k,
                                              const uint16_t* pool_v, const int32_t* block_of_slot,
                                              const int32_t* ctx_len, float scale, uint16_t* out,
                                              void* stream);

/* Pins and maps `bytes` of existing host memory at `host` (cudaHostRegister,
 * mapped) and returns in *dev_ptr the address kernels use to read it: the
 * form oasis_fetch_blocks expects for host_k / host_v.  Not for the per-step
 * path (it blocks and may be slow for large ranges). */
oasis_status_t oasis_host_register(void* host, size_t bytes, void** dev_ptr);
/* Undoes oasis_host_register. */
oasis_status_t oasis_host_unregister(void* host);

/* Reads the current device's error word into *flags (OASIS_DEVERR_* bits)
 * and clears it when `clear` is non-zero.  Synchronizes the device. */
oasis_status_t oasis_device_errors(uint32_t* flags, int32_t clear);

/* Waits for `stream` with a time limit: OASIS_OK once its work is done,
 * OASIS_ERR_TIMEOUT after `timeout_ms`, OASIS_ERR_CUDA on a CUDA error. */
oasis_status_t oasis_stream_wait(void* stream, int32_t timeout_ms);

/* Human-readable name of a status code (static string). */
const char* oasis_status_string(oasis_status_t status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int32_t oasis_version(void);

#ifdef __cplusplus
}
#endif

#endif /* OASIS_H */
