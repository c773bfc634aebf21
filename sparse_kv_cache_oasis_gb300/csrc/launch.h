// Internal launchers of the liboasis kernels.  The C ABI (api.cu) validates
// every argument before calling these; the launchers only size grids and
// launch.  Each returns the cudaError_t of its launch.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/oasis.h"

namespace oasis {

// Per-device facts the launchers need (filled once per device by api.cu).
struct DeviceInfo {
  int sm_count = 0;
  int score_ctas_per_sm = 0;
  int attn_ctas_per_sm = 0;
  uint32_t* err = nullptr;  // device error word
};

// Derived sizes of one configuration.
struct Shape {
  int B, Hq, Hkv, G, D, bs, NB, S, L, K, cap, sink, local;
  int units() const { return B * Hkv; }
};

cudaError_t launch_build_summaries(const Shape& s, const uint16_t* k, float* summ,
                                   cudaStream_t st, const DeviceInfo& di);
cudaError_t launch_score_blocks(const Shape& s, const uint16_t* q_draft, const float* summ,
                                float* scores, cudaStream_t st, const DeviceInfo& di);
cudaError_t launch_build_summaries_minmax(const Shape& s, const uint16_t* k, uint16_t* summ_mm,
                                          cudaStream_t st, const DeviceInfo& di);
cudaError_t launch_score_blocks_minmax(const Shape& s, const uint16_t* q_draft,
                                       const uint16_t* summ_mm, float* scores, cudaStream_t st,
                                       const DeviceInfo& di);
cudaError_t launch_select_topk(const Shape& s, const float* scores, const int32_t* ctx_len,
                               int32_t* topk_ids, cudaStream_t st, const DeviceInfo& di);
cudaError_t launch_plan_fetch(const Shape& s, const int32_t* topk_ids, int32_t step,
                              int32_t* clock, int32_t* slot_of_block, int32_t* block_of_slot,
                              int32_t* last_used, int32_t* fetch_block, int32_t* fetch_slot,
                              int32_t* evict_block, int32_t* n_fetch, int32_t* n_evict,
                              cudaStream_t st, const DeviceInfo& di);
cudaError_t launch_select_and_plan(const Shape& s, const float* scores, const int32_t* ctx_len,
                                   int32_t* topk_ids,
                                   int32_t step, int32_t* clock, int32_t* slot_of_block,
                                   int32_t* block_of_slot, int32_t* last_used,
                                   int32_t* fetch_block, int32_t* fetch_slot,
                                   int32_t* evict_block, int32_t* n_fetch, int32_t* n_evict,
                                   cudaStream_t st, const DeviceInfo& di);
cudaError_t launch_fetch_blocks(const Shape& s, const uint16_t* host_k, const uint16_t* host_v,
                                const int32_t* fetch_block, const int32_t* fetch_slot,
                                const int32_t* n_fetch, uint16_t* pool_k, uint16_t* pool_v,
                                cudaStream_t st, const DeviceInfo& di);

// Decode-time append of one token per request (write-allocate of the newest block).
cudaError_t launch_append_kv(const Shape& s, const uint16_t* k_new, const uint16_t* v_new,
                             int32_t* ctx_len, const int32_t* clock, int32_t step,
                             uint16_t* host_k, uint16_t* host_v, int32_t* slot_of_block,
                             int32_t* block_of_slot, int32_t* last_used, uint16_t* pool_k,
                             uint16_t* pool_v, cudaStream_t st, const DeviceInfo& di);
cudaError_t launch_refresh_summaries(const Shape& s, const int32_t* ctx_len,
                                     const uint16_t* host_k, const int32_t* slot_of_block,
                                     const uint16_t* pool_k, float* summ, uint16_t* summ_mm,
                                     cudaStream_t st, const DeviceInfo& di);

// Attention: the pools are read by TMA through these two tensor maps.
size_t attn_workspace_bytes(const Shape& s);
size_t attn_counter_offset(const Shape& s);  // arrival counters inside the workspace
size_t attn_counter_bytes(const Shape& s);
cudaError_t attn_configure(int device);  // one-time function attributes
int attn_ctas_per_sm();
cudaError_t launch_sparse_decode_attn(const Shape& s, const uint16_t* q,
                                      const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                      const int32_t* block_of_slot, const int32_t* ctx_len,
                                      float scale, uint16_t* out, void* workspace,
                                      cudaStream_t st, const DeviceInfo& di);
int attn_split(const Shape& s, int sm_count);  // CTAs per unit (cluster size)

// Scoring, top-K and plan of every unit in one launch (clusters per unit).
bool chain_supported(const Shape& s);
cudaError_t chain_configure();  // one-time function attributes
cudaError_t launch_predict_chain(const Shape& s, const uint16_t* q_draft, const float* summ,
                                 float* scores, int32_t step, int32_t* clock, int32_t* topk_ids,
                                 int32_t* slot_of_block, int32_t* block_of_slot,
                                 int32_t* last_used, int32_t* fetch_block, int32_t* fetch_slot,
                                 int32_t* evict_block, int32_t* n_fetch, int32_t* n_evict,
                                 cudaStream_t st, const DeviceInfo& di);

// Joint attention of the decoded and the draft tokens: row tiles per CTA,
// row groups per unit and CTAs per (unit, row group).
struct JointSplit {
  int nt, groups, P;
};
JointSplit joint_split(const Shape& s, int sm_count);
cudaError_t joint_configure();  // one-time function attributes
cudaError_t launch_sparse_decode_attn_joint(const Shape& s, const uint16_t* q,
                                            const uint16_t* q_draft, const CUtensorMap& tm_k,
                                            const CUtensorMap& tm_v,
                                            const int32_t* block_of_slot, const int32_t* ctx_len,
                                            float scale, uint16_t* out, cudaStream_t st,
                                            const DeviceInfo& di);

// Attention of one layer and scoring of another in one launch (same shapes).
cudaError_t fused_configure();  // one-time function attributes
cudaError_t launch_attend_and_score(const Shape& s, const CUtensorMap& tm_k,
                                    const CUtensorMap& tm_v, const uint16_t* q,
                                    const int32_t* block_of_slot, const int32_t* ctx_len,
                                    float scale, uint16_t* out, const uint16_t* q_draft,
                                    const void* summ, bool minmax, float* scores,
                                    cudaStream_t st, const DeviceInfo& di);
int score_ctas_per_sm();
cudaError_t score_configure();  // one-time function attributes
cudaError_t pred_configure();   // one-time function attributes (top-K / plan kernels)
cudaError_t fetch_configure();  // one-time function attributes

}  // namespace oasis
