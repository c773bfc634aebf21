// C ABI of liboasis (declarations and contracts in include/oasis.h).
//
// Every entry point validates its arguments on the host before launching
// anything: configuration limits, null pointers and alignment.  Launch
// errors come back as OASIS_ERR_CUDA; anomalies only visible on the device
// set bits in a per-device error word (OASIS_DEVERR_*), never a trap.
#include <cuda.h>
#include <cuda_runtime.h>

#include <chrono>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <thread>

#include "../../include/oasis.h"
#include "common.cuh"
#include "launch.h"

namespace oasis {

__device__ uint32_t g_device_error;  // one per device context

namespace {

constexpr int kMaxDevices = 64;

struct DeviceSlot {
  bool ready = false;
  DeviceInfo info;
};
std::mutex g_mu;
DeviceSlot g_dev[kMaxDevices];

oasis_status_t device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return OASIS_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceSlot& d = g_dev[dev];
  if (!d.ready) {
    DeviceInfo di;
    if (cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return OASIS_ERR_CUDA;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return OASIS_ERR_CUDA;
    di.err = static_cast<uint32_t*>(p);
    if (attn_configure(dev) != cudaSuccess) return OASIS_ERR_CUDA;
    if (score_configure() != cudaSuccess) return OASIS_ERR_CUDA;
    if (pred_configure() != cudaSuccess) return OASIS_ERR_CUDA;
    if (fetch_configure() != cudaSuccess) return OASIS_ERR_CUDA;
    if (fused_configure() != cudaSuccess) return OASIS_ERR_CUDA;
    if (joint_configure() != cudaSuccess) return OASIS_ERR_CUDA;
    if (chain_configure() != cudaSuccess) return OASIS_ERR_CUDA;
    di.score_ctas_per_sm = score_ctas_per_sm();
    di.attn_ctas_per_sm = attn_ctas_per_sm();
    d.info = di;
    d.ready = true;
  }
  *out = d.info;
  return OASIS_OK;
}

int forced_count(int NB, int sink, int local) {
  const int a = sink < NB ? sink : NB;
  const int b0 = NB - local > 0 ? NB - local : 0;
  const int lo = a > b0 ? a : b0;
  return a + (NB - lo);
}

int cap_of(const oasis_config_t* c, int S) {
  const double r = static_cast<double>(c->fetch_ratio);
  if (r < 0.0 || r >= 1.0) return c->top_k;
  int cap = static_cast<int>(std::ceil(r * static_cast<double>(S) - 1e-6));
  if (cap < 0) cap = 0;
  if (cap > c->top_k) cap = c->top_k;
  return cap;
}

// Checks shared by every entry point; fills the derived shape.
oasis_status_t make_shape(const oasis_config_t* c, Shape* s) {
  if (!c) return OASIS_ERR_INVALID_ARG;
  if (c->batch < 1 || c->num_q_heads < 1 || c->num_kv_heads < 1 || c->num_blocks < 1 ||
      c->lookahead < 1 || c->top_k < 1 || c->head_dim < 1 || c->block_size < 1)
    return OASIS_ERR_INVALID_ARG;
  if (c->num_q_heads % c->num_kv_heads != 0) return OASIS_ERR_INVALID_ARG;
  if (c->kv_budget_tokens < c->block_size || c->kv_budget_tokens % c->block_size != 0)
    return OASIS_ERR_INVALID_ARG;
  if (c->sink_blocks < 0 || c->local_blocks < 0) return OASIS_ERR_INVALID_ARG;
  if (!std::isfinite(c->fetch_ratio)) return OASIS_ERR_INVALID_ARG;
  const int S = c->kv_budget_tokens / c->block_size;
  if (c->top_k > S || c->top_k > c->num_blocks) return OASIS_ERR_INVALID_ARG;
  if (forced_count(c->num_blocks, c->sink_blocks, c->local_blocks) > c->top_k)
    return OASIS_ERR_INVALID_ARG;
  if (c->head_dim != kHeadDim || c->block_size != kBlockSize) return OASIS_ERR_UNSUPPORTED;
  if (S > 1024 || c->top_k > 1024 || c->num_blocks > 32768) return OASIS_ERR_UNSUPPORTED;
  const int64_t units = static_cast<int64_t>(c->batch) * c->num_kv_heads;
  if (units > 65535) return OASIS_ERR_UNSUPPORTED;
  if (units * S * kBlockSize >= (int64_t(1) << 31)) return OASIS_ERR_UNSUPPORTED;
  s->B = c->batch;
  s->Hq = c->num_q_heads;
  s->Hkv = c->num_kv_heads;
  s->G = c->num_q_heads / c->num_kv_heads;
  s->D = c->head_dim;
  s->bs = c->block_size;
  s->NB = c->num_blocks;
  s->S = S;
  s->L = c->lookahead;
  s->K = c->top_k;
  s->cap = cap_of(c, S);
  s->sink = c->sink_blocks;
  s->local = c->local_blocks;
  return OASIS_OK;
}

bool aligned(const void* p, uintptr_t a) { return p && (reinterpret_cast<uintptr_t>(p) % a) == 0; }

oasis_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? OASIS_OK : OASIS_ERR_CUDA; }

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// A pool [rows = B*Hkv*S*16][128] bf16 read as 16-row x 64-column boxes, 128B swizzle.
oasis_status_t encode_pool(CUtensorMap* tm, const void* pool, const Shape& s) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return OASIS_ERR_CUDA;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim),
                              static_cast<cuuint64_t>(s.units()) * s.S * kBlockSize};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kHeadDim) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kBlockSize)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pool), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? OASIS_OK : OASIS_ERR_INVALID_ARG;
}

// Scratch of oasis_sparse_decode_attn_static: a fixed array in device memory
// that exists on every GPU this library is loaded on, so that call needs no
// allocation.  In host code the name is only a stand-in; the device address is
// looked up once per device with cudaGetSymbolAddress.
constexpr size_t kStaticAttnScratchBytes = 8u << 20;  // 8 MiB
static __device__ __align__(256) unsigned char g_static_attn_scratch[kStaticAttnScratchBytes];
void* g_static_scratch_addr[kMaxDevices];

oasis_status_t static_attn_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return OASIS_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_static_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_attn_scratch) != cudaSuccess || !p) return OASIS_ERR_CUDA;
    g_static_scratch_addr[dev] = p;
  }
  *out = g_static_scratch_addr[dev];
  return OASIS_OK;
}

}  // namespace
}  // namespace oasis

using namespace oasis;

extern "C" {

oasis_status_t oasis_validate_config(const oasis_config_t* cfg) {
  Shape s;
  oasis_status_t st = make_shape(cfg, &s);
  if (st != OASIS_OK) return st;
  if (s.G > kMaxAttnGroup) return OASIS_ERR_UNSUPPORTED;
  if (s.L * s.G > 64) return OASIS_ERR_UNSUPPORTED;
  return OASIS_OK;
}

int32_t oasis_fetch_cap(const oasis_config_t* cfg) {
  Shape s;
  if (make_shape(cfg, &s) != OASIS_OK) return -1;
  return s.cap;
}

oasis_status_t oasis_build_summaries(const oasis_config_t* cfg, const uint16_t* k, float* summ,
                                     void* stream) {
  Shape s;
  oasis_status_t st = make_shape(cfg, &s);
  if (st != OASIS_OK) return st;
  if (!aligned(k, 16) || !aligned(summ, 16)) return OASIS_ERR_INVALID_ARG;
  DeviceInfo di;
  if ((st = device_info(&di)) != OASIS_OK) return st;
  return from_cuda(launch_build_summaries(s, k, summ, static_cast<cudaStream_t>(stream), di));
}

oasis_status_t oasis_score_blocks(const oasis_config_t* cfg, const uint16_t* q_draft,
                                  const float* summ, float* scores, void* stream) {
  Shape s;
  oasis_status_t st = make_shape(cfg, &s);
  if (st != OASIS_OK) return st;
  if (s.L * s.G > 64) return OASIS_ERR_UNSUPPORTED;
  if (!aligned(q_draft, 16) || !aligned(summ, 16) || !aligned(scores, 8)) return OASIS_ERR_INVALID_ARG;
  DeviceInfo di;
  if ((st = device_info(&di)) != OASIS_OK) return st;
  return from_cuda(launch_score_blocks(s, q_draft, summ, scores, static_cast<cudaStream_t>(stream), di));
}

oasis_status_t oasis_build_summaries_minmax(const oasis_config_t* cfg, const uint16_t* k,
                                            uint16_t* summ_mm, void* stream) {
  Shape s;
  oasis_status_t st = make_shape(cfg, &s);
  if (st != OASIS_OK) return st;
  if (!aligned(k, 16) || !aligned(summ_mm, 16)) return OASIS_ERR_INVALID_ARG;
  DeviceInfo di;
  if ((st = device_info(&di)) != OASIS_OK) return st;
  return from_cuda(
      launch_build_summaries_minmax(s, k, summ_mm, static_cast<cudaStream_t>(stream), di));
}

oasis_status_t oasis_score_blocks_minmax(const oasis_config_t* cfg, const uint16_t* q_draft,
                                         const uint16_t* summ_mm, float* scores, void* stream) {
  Shape s;
  oasis_status_t st = make_shape(cfg, &s);
  if (st != OASIS_OK) return st;
  if (s.L * s.G > 32) return OASIS_ERR_UNSUPPORTED;
  if (!aligned(q_draft, 16) || !aligned(summ_mm, 16) || !aligned(scores, 8))
    return OASIS_ERR_INVALID_ARG;
  DeviceInfo di;
  if ((st = device_info(&di)) != OASIS_OK) return st;
  return from_cuda(
      launch_score_blocks_minmax(s, q_draft, summ_mm, scores, static_cast<cudaStream_t>(stream), di));
}

oasis_status_t oasis_select_topk(const oasis_config_t* cfg, const float* scores,
                                 int32_t* topk_ids, void* stream) {
  Shape s;
  oasis_status_t st = make_shape(cfg, &s);
  if (st != OASIS_OK) return st;
  if (!aligned(scores, 4) || !aligned(topk_ids, 4)) return OASIS_ERR_INVALID_ARG;
  DeviceInfo di;
  if ((st = device_info(&di)) != OASIS_OK) return st;
  return from_cuda(
      launch_select_topk(s, scores, nullptr, topk_ids, static_cast<cudaStream_t>(stream), di));
}

oasis_status_t oasis_select_topk_ctx(const oasis_config_t* cfg, const float* scores,
                                     const int32_t* ctx_len, int32_t* topk_ids, void* stream) {
  Shape s;
  oasis_status_t st = make_shape(cfg, &s);
  if (st != OASIS_OK) return st;
  if (!aligned(scores, 4) || !aligned(topk_ids, 4) || !aligned(ctx_len, 4))
    return OASIS_ERR_INVALID_ARG;
  DeviceInfo di;
  if ((st = device_info(&di)) != OASIS_OK) return st;
  return from_cuda(
      launch_select_topk(s, scores, ctx_len, topk_ids, static_cast<cudaStream_t>(stream), di));
}

oasis_status_t oasis_plan_fetch(const oasis_config_t* cfg, const int32_t* topk_ids, int32_t step,
                                int32_t* slot_of_block, int32_t* block_of_slot,
                                int32_t* last_used, int32_t* fetch_block, int32_t* fetch_slot,
                                int32_t* evict_block, int32_t* n_fetch, int32_t* n_evict,
                                void* stream) {
  Shape s;
  oasis_status_t st = make_shape(cfg, &s);
  if (st != OASIS_OK) return st;
  const void* ptrs[] = {topk_ids, slot_of_block, block_of_slot, last_used, fetch_block,
                        fetch_slot, evict_block, n_fetch, n_evict};
  for (const void* p : ptrs)
    if (!aligned(p, 4)) return OASIS_ERR_INVALID_ARG;
  DeviceInfo di;
  if ((st = device_info(&di)) != OASIS_OK) return st;
  return from_cuda(launch_plan_fetch(s, topk_ids, step, nullptr, slot_of_block, block_of_slot,
                                     last_used, fetch_block, fetch_slot, evict_block, n_fetch,
                                     n_evict, static_cast<cudaStream_t>(stream), di));
}

oasis_status_t oasis_plan_fetch_clocked(const oasis_config_t* cfg, const int32_t* topk_ids,
                                        int32_t* clock, int32_t* slot_of_block,
                                        int32_t* block_of_slot, int32_t* last_used,
                                        int32_t* fetch_block, int32_t* fetch_slot,
                                        int32_t* evict_block, int32_t* n_fetch, int32_t* n_evict,
                                        void* stream) {
  Shape s;
  oasis_status_t st = make_shape(cfg, &s);
  if (st != OASIS_OK) return st;
  const void* ptrs[] = {topk_ids, clock, slot_of_block, block_of_slot, last_used, fetch_block,
                        fetch_slot, evict_block, n_fetch, n_evict};
  for (const void* p : ptrs)
    if (!aligned(p, 4)) return OASIS_ERR_INVALID_ARG;
  DeviceInfo di;
  if ((st = device_info(&di)) != OASIS_OK) return st;
  return from_cuda(launch_plan_fetch(s, topk_ids, 0, clock, slot_of_block, block_of_slot,
                                     last_used, fetch_block, fetch_slot, evict_block, n_fetch,
                                     n_evict, static_cast<cudaStream_t>(stream), di));
}

oasis_status_t oasis_predict_select(const oasis_config_t* cfg, const float* scores,
                                    int32_t step, int32_t* clock, int32_t* topk_ids,
                                    int32_t* slot_of_block, int32_t* block_of_slot,
                                    int32_t* last_used, int32_t* fetch_block,
                                    int32_t* fetch_slot, int32_t* evict_block,
                                    int32_t* n_fetch, int32_t* n_evict, void* stream) {
  Shape s;
  oasis_status_t st = make_shape(cfg, &s);
  if (st != OASIS_OK) return st;
  const void* ptrs[] = {scores, topk_ids, slot_of_block, block_of_slot, last_used,
                        fetch_block, fetch_slot, evict_block, n_fetch, n_evict};
  for (const void* p : ptrs)
    if (!aligned(p, 4)) return OASIS_ERR_INVALID_ARG;
  if (clock && !aligned(clock, 4)) return OASIS_ERR_INVALID_ARG;
  DeviceInfo di;
  if ((st = device_info(&di)) != OASIS_OK) return st;
  return from_cuda(launch_select_and_plan(s, scores, nullptr, topk_ids, step, clock, slot_of_block,
                                          block_of_slot, last_used, fetch_block, fetch_slot,
                                          evict_block, n_fetch, n_evict,
                                          static_cast<cudaStream_t>(stream), di));
}

oasis_status_t oasis_predict_chain(const oasis_config_t* cfg, const uint16_t* q_draft,
                                   const float* summ, float* scores, int32_t step, int32_t* clock,
                                   int32_t* topk_ids, int32_t* slot_of_block,
                                   int32_t* block_of_slot, int32_t* last_used,
                                   int32_t* fetch_block, int32_t* fetch_slot, int32_t* evict_block,
                                   int32_t* n_fetch, int32_t* n_evict, void* stream) {
  Shape s;
  oasis_status_t st = make_shape(cfg, &s);
  if (st != OASIS_OK) return st;
  if (!chain_supported(s)) return OASIS_ERR_UNSUPPORTED;
  if (!aligned(q_draft, 16) || !aligned(summ, 16) || !aligned(scores, 8))
    return OASIS_ERR_INVALID_ARG;
  const void* ptrs[] = {topk_ids, slot_of_block, block_of_slot, last_used,
                        fetch_block, fetch_slot, evict_block, n_fetch, n_evict};
  for (const void* p : ptrs)
    if (!aligned(p, 4)) return OASIS_ERR_INVALID_ARG;
  if (clock && !aligned(clock, 4)) return OASIS_ERR_INVALID_ARG;
  DeviceInfo di;
  if ((st = device_info(&di)) != OASIS_OK) return st;
  return from_cuda(launch_predict_chain(s, q_draft, summ, scores, step, clock, topk_ids,
                                        slot_of_block, block_of_slot, last_used, fetch_block,
                                        fetch_slot, evict_block, n_fetch, n_evict,
                                        static_cast<cudaStream_t>(stream), di));
}

oasis_status_t oasis_predict_select_ctx(const oasis_config_t* cfg, const float* scores,
                                        const int32_t* ctx_len, int32_t step, int32_t* clock,
                                        int32_t* topk_ids, int32_t* slot_of_block,
                                        int32_t* block_of_slot, int32_t* last_used,
                                        int32_t* fetch_block, int32_t* fetch_slot,
                                        int32_t* evict_block, int32_t* n_fetch, int32_t* n_evict,
                                        void* stream) {
  Shape s;
  oasis_status_t st = make_shape(cfg, &s);
  if (st != OASIS_OK) return st;
  const void* ptrs[] = {scores, ctx_len, topk_ids, slot_of_block, block_of_slot, last_used,
                        fetch_block, fetch_slot, evict_block, n_fetch, n_evict};
  for (const void* p : ptrs)
    if (!aligned(p, 4)) return OASIS_ERR_INVALID_ARG;
  if (clock && !aligned(clock, 4)) return OASIS_ERR_INVALID_ARG;
  DeviceInfo di;
  if ((st = device_info(&di)) != OASIS_OK) return st;
  return from_cuda(launch_select_and_plan(s, scores, ctx_len, topk_ids, step, clock, slot_of_block,
                                          block_of_slot, last_used, fetch_block, fetch_slot,
                                          evict_block, n_fetch, n_evict,
                                          static_cast<cudaStream_t>(stream), di));
}

oasis_status_t oasis_append_kv(const oasis_config_t* cfg, const uint16_t* k_new,
                               const uint16_t* v_new, int32_t* ctx_len, const int32_t* clock,
                               int32_t step, uint16_t* host_k, uint16_t* host_v,
                               int32_t* slot_of_block, int32_t* block_of_slot, int32_t* last_used,
                               uint16_t* pool_k, uint16_t* pool_v, void* stream) {
  Shape s;
  oasis_status_t st = make_shape(cfg, &s);
  if (st != OASIS_OK) return st;
  if (s.Hkv > 32) return OASIS_ERR_UNSUPPORTED;
  if (!aligned(k_new, 8) || !aligned(v_new, 8) || !aligned(host_k, 16) || !aligned(host_v, 16) ||
      !aligned(pool_k, 16) || !aligned(pool_v, 16) || !aligned(ctx_len, 4) ||
      !aligned(slot_of_block, 4) || !aligned(block_of_slot, 4) || !aligned(last_used, 4))
    return OASIS_ERR_INVALID_ARG;
  if (clock && !aligned(clock, 4)) return OASIS_ERR_INVALID_ARG;
  DeviceInfo di;
  if ((st = device_info(&di)) != OASIS_OK) return st;
  return from_cuda(launch_append_kv(s, k_new, v_new, ctx_len, clock, step, host_k, host_v,
                                    slot_of_block, block_of_slot, last_used, pool_k, pool_v,
                                    static_cast<cudaStream_t>(stream), di));
}

oasis_status_t oasis_refresh_summaries(const oasis_config_t* cfg, const int32_t* ctx_len,
                                       const uint16_t* host_k, const int32_t* slot_of_block,
                                       const uint16_t* pool_k, float* summ, uint16_t* summ_mm,
                                       void* stream) {
  Shape s;
  oasis_status_t st = make_shape(cfg, &s);
  if (st != OASIS_OK) return st;
  if (!aligned(ctx_len, 4) || !aligned(host_k, 16) || !aligned(slot_of_block, 4) ||
      !aligned(pool_k, 16) || !aligned(summ, 16))
    return OASIS_ERR_INVALID_ARG;
  if (summ_mm && !aligned(summ_mm, 16)) return OASIS_ERR_INVALID_ARG;
  DeviceInfo di;
  if ((st = device_info(&di)) != OASIS_OK) return st;
  return from_cuda(launch_refresh_summaries(s, ctx_len, host_k, slot_of_block, pool_k, summ,
                                            summ_mm, static_cast<cudaStream_t>(stream), di));
}

oasis_status_t oasis_fetch_blocks(const oasis_config_t* cfg, const uint16_t* host_k,
                                  const uint16_t* host_v, const int32_t* fetch_block,
                                  const int32_t* fetch_slot, const int32_t* n_fetch,
                                  uint16_t* pool_k, uint16_t* pool_v, void* copy_stream) {
  Shape s;
  oasis_status_t st = make_shape(cfg, &s);
  if (st != OASIS_OK) return st;
  if (!aligned(host_k, 16) || !aligned(host_v, 16) || !aligned(pool_k, 16) || !aligned(pool_v, 16))
    return OASIS_ERR_INVALID_ARG;
  if (!aligned(fetch_block, 4) || !aligned(fetch_slot, 4) || !aligned(n_fetch, 4))
    return OASIS_ERR_INVALID_ARG;
  DeviceInfo di;
  if ((st = device_info(&di)) != OASIS_OK) return st;
  return from_cuda(launch_fetch_blocks(s, host_k, host_v, fetch_block, fetch_slot, n_fetch, pool_k,
                                       pool_v, static_cast<cudaStream_t>(copy_stream), di));
}

size_t oasis_attn_workspace_bytes(const oasis_config_t* cfg) {
  Shape s;
  if (make_shape(cfg, &s) != OASIS_OK) return 0;
  return attn_workspace_bytes(s);
}

oasis_status_t oasis_sparse_decode_attn(const oasis_config_t* cfg, const uint16_t* q,
                                        const uint16_t* pool_k, const uint16_t* pool_v,
                                        const int32_t* block_of_slot, const int32_t* ctx_len,
                                        float scale, uint16_t* out, void* workspace,
                                        size_t workspace_bytes, void* stream) {
  Shape s;
  oasis_status_t st = make_shape(cfg, &s);
  if (st != OASIS_OK) return st;
  if (s.G > kMaxAttnGroup) return OASIS_ERR_UNSUPPORTED;
  if (!std::isfinite(scale) || !(scale > 0.f)) return OASIS_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(pool_k, 16) || !aligned(pool_v, 16) || !aligned(out, 16) ||
      !aligned(block_of_slot, 4))
    return OASIS_ERR_INVALID_ARG;
  if (ctx_len && !aligned(ctx_len, 4)) return OASIS_ERR_INVALID_ARG;
  if (!aligned(workspace, 256) || workspace_bytes < attn_workspace_bytes(s)) return OASIS_ERR_INVALID_ARG;
  DeviceInfo di;
  if ((st = device_info(&di)) != OASIS_OK) return st;
  CUtensorMap tk, tv;
  if ((st = encode_pool(&tk, pool_k, s)) != OASIS_OK) return st;
  if ((st = encode_pool(&tv, pool_v, s)) != OASIS_OK) return st;
  return from_cuda(launch_sparse_decode_attn(s, q, tk, tv, block_of_slot, ctx_len, scale, out,
                                             workspace, static_cast<cudaStream_t>(stream), di));
}

oasis_status_t oasis_sparse_decode_attn_joint(const oasis_config_t* cfg, const uint16_t* q,
                                              const uint16_t* q_draft, const uint16_t* pool_k,
                                              const uint16_t* pool_v, const int32_t* block_of_slot,
                                              const int32_t* ctx_len, float scale, uint16_t* out,
                                              void* stream) {
  Shape s;
  oasis_status_t st = make_shape(cfg, &s);
  if (st != OASIS_OK) return st;
  if (!std::isfinite(scale) || !(scale > 0.f)) return OASIS_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(q_draft, 16) || !aligned(pool_k, 16) || !aligned(pool_v, 16) ||
      !aligned(out, 16) || !aligned(block_of_slot, 4))
    return OASIS_ERR_INVALID_ARG;
  if (ctx_len && !aligned(ctx_len, 4)) return OASIS_ERR_INVALID_ARG;
  DeviceInfo di;
  if ((st = device_info(&di)) != OASIS_OK) return st;
  const JointSplit j = joint_split(s, di.sm_count);
  if (static_cast<int64_t>(s.units()) * j.groups * j.P > 0x7fffffff) return OASIS_ERR_UNSUPPORTED;
  CUtensorMap tk, tv;
  if ((st = encode_pool(&tk, pool_k, s)) != OASIS_OK) return st;
  if ((st = encode_pool(&tv, pool_v, s)) != OASIS_OK) return st;
  return from_cuda(launch_sparse_decode_attn_joint(s, q, q_draft, tk, tv, block_of_slot, ctx_len,
                                                   scale, out, static_cast<cudaStream_t>(stream),
                                                   di));
}

oasis_status_t oasis_attend_and_score(const oasis_config_t* cfg, const uint16_t* q,
                                      const uint16_t* pool_k, const uint16_t* pool_v,
                                      const int32_t* block_of_slot, const int32_t* ctx_len,
                                      float scale, uint16_t* out, const uint16_t* q_draft,
                                      const float* summ, float* scores, void* stream) {
  Shape s;
  oasis_status_t st = make_shape(cfg, &s);
  if (st != OASIS_OK) return st;
  if (s.G > kMaxAttnGroup || s.L * s.G > 64) return OASIS_ERR_UNSUPPORTED;
  if (!std::isfinite(scale) || !(scale > 0.f)) return OASIS_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(pool_k, 16) || !aligned(pool_v, 16) || !aligned(out, 16) ||
      !aligned(block_of_slot, 4))
    return OASIS_ERR_INVALID_ARG;
  if (ctx_len && !aligned(ctx_len, 4)) return OASIS_ERR_INVALID_ARG;
  if (!aligned(q_draft, 16) || !aligned(summ, 16) || !aligned(scores, 8)) return OASIS_ERR_INVALID_ARG;
  DeviceInfo di;
  if ((st = device_info(&di)) != OASIS_OK) return st;
  CUtensorMap tk, tv;
  if ((st = encode_pool(&tk, pool_k, s)) != OASIS_OK) return st;
  if ((st = encode_pool(&tv, pool_v, s)) != OASIS_OK) return st;
  return from_cuda(launch_attend_and_score(s, tk, tv, q, block_of_slot, ctx_len, scale, out, q_draft,
                                           summ, false, scores, static_cast<cudaStream_t>(stream),
                                           di));
}

oasis_status_t oasis_attend_and_score_minmax(const oasis_config_t* cfg, const uint16_t* q,
                                             const uint16_t* pool_k, const uint16_t* pool_v,
                                             const int32_t* block_of_slot, const int32_t* ctx_len,
                                             float scale, uint16_t* out, const uint16_t* q_draft,
                                             const uint16_t* summ_mm, float* scores,
                                             void* stream) {
  Shape s;
  oasis_status_t st = make_shape(cfg, &s);
  if (st != OASIS_OK) return st;
  if (s.G > kMaxAttnGroup || s.L * s.G > 32) return OASIS_ERR_UNSUPPORTED;
  if (!std::isfinite(scale) || !(scale > 0.f)) return OASIS_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(pool_k, 16) || !aligned(pool_v, 16) || !aligned(out, 16) ||
      !aligned(block_of_slot, 4))
    return OASIS_ERR_INVALID_ARG;
  if (ctx_len && !aligned(ctx_len, 4)) return OASIS_ERR_INVALID_ARG;
  if (!aligned(q_draft, 16) || !aligned(summ_mm, 16) || !aligned(scores, 8))
    return OASIS_ERR_INVALID_ARG;
  DeviceInfo di;
  if ((st = device_info(&di)) != OASIS_OK) return st;
  CUtensorMap tk, tv;
  if ((st = encode_pool(&tk, pool_k, s)) != OASIS_OK) return st;
  if ((st = encode_pool(&tv, pool_v, s)) != OASIS_OK) return st;
  return from_cuda(launch_attend_and_score(s, tk, tv, q, block_of_slot, ctx_len, scale, out, q_draft,
                                           summ_mm, true, scores, static_cast<cudaStream_t>(stream),
                                           di));
}

oasis_status_t oasis_host_register(void* host, size_t bytes, void** dev_ptr) {
  if (!host || !dev_ptr || bytes == 0) return OASIS_ERR_INVALID_ARG;
  if (cudaHostRegister(host, bytes, cudaHostRegisterMapped | cudaHostRegisterPortable) != cudaSuccess)
    return OASIS_ERR_CUDA;
  if (cudaHostGetDevicePointer(dev_ptr, host, 0) != cudaSuccess) {
    cudaHostUnregister(host);
    return OASIS_ERR_CUDA;
  }
  return OASIS_OK;
}

oasis_status_t oasis_host_unregister(void* host) {
  if (!host) return OASIS_ERR_INVALID_ARG;
  return from_cuda(cudaHostUnregister(host));
}

oasis_status_t oasis_sparse_decode_attn_static(const oasis_config_t* cfg, const uint16_t* q,
                                               const uint16_t* pool_k, const uint16_t* pool_v,
                                               const int32_t* block_of_slot,
                                               const int32_t* ctx_len, float scale,
                                               uint16_t* out, void* stream) {
  Shape s;
  oasis_status_t st = make_shape(cfg, &s);
  if (st != OASIS_OK) return st;
  if (s.G > kMaxAttnGroup) return OASIS_ERR_UNSUPPORTED;
  if (attn_workspace_bytes(s) > kStaticAttnScratchBytes) return OASIS_ERR_UNSUPPORTED;
  if (!std::isfinite(scale) || !(scale > 0.f)) return OASIS_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(pool_k, 16) || !aligned(pool_v, 16) || !aligned(out, 16) ||
      !aligned(block_of_slot, 4))
    return OASIS_ERR_INVALID_ARG;
  if (ctx_len && !aligned(ctx_len, 4)) return OASIS_ERR_INVALID_ARG;
  DeviceInfo di;
  if ((st = device_info(&di)) != OASIS_OK) return st;
  void* scratch = nullptr;
  if ((st = static_attn_scratch(&scratch)) != OASIS_OK) return st;
  CUtensorMap tk, tv;
  if ((st = encode_pool(&tk, pool_k, s)) != OASIS_OK) return st;
  if ((st = encode_pool(&tv, pool_v, s)) != OASIS_OK) return st;
  // the array keeps whatever the previous call left; the arrival counters must start at zero
  const size_t cnt = attn_counter_bytes(s);
  if (cnt && cudaMemsetAsync(static_cast<unsigned char*>(scratch) + attn_counter_offset(s), 0, cnt,
                             static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return OASIS_ERR_CUDA;
  return from_cuda(launch_sparse_decode_attn(s, q, tk, tv, block_of_slot, ctx_len, scale, out,
                                             scratch, static_cast<cudaStream_t>(stream), di));
}

oasis_status_t oasis_device_errors(uint32_t* flags, int32_t clear) {
  if (!flags) return OASIS_ERR_INVALID_ARG;
  DeviceInfo di;
  oasis_status_t st = device_info(&di);
  if (st != OASIS_OK) return st;
  if (cudaDeviceSynchronize() != cudaSuccess) return OASIS_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, di.err, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return OASIS_ERR_CUDA;
  *flags = v;
  if (clear) {
    const uint32_t zero = 0;
    if (cudaMemcpy(di.err, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
      return OASIS_ERR_CUDA;
  }
  return OASIS_OK;
}

oasis_status_t oasis_stream_wait(void* stream, int32_t timeout_ms) {
  const auto t0 = std::chrono::steady_clock::now();
  for (;;) {
    const cudaError_t e = cudaStreamQuery(static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) return OASIS_OK;
    if (e != cudaErrorNotReady) return OASIS_ERR_CUDA;
    const auto ms = std::chrono::duration_cast<std::chrono::milliseconds>(
                        std::chrono::steady_clock::now() - t0).count();
    if (ms >= timeout_ms) return OASIS_ERR_TIMEOUT;
    std::this_thread::sleep_for(std::chrono::microseconds(50));
  }
}

const char* oasis_status_string(oasis_status_t status) {
  switch (status) {
    case OASIS_OK: return "OASIS_OK";
    case OASIS_ERR_INVALID_ARG: return "OASIS_ERR_INVALID_ARG";
    case OASIS_ERR_UNSUPPORTED: return "OASIS_ERR_UNSUPPORTED";
    case OASIS_ERR_CUDA: return "OASIS_ERR_CUDA";
    case OASIS_ERR_TIMEOUT: return "OASIS_ERR_TIMEOUT";
  }
  return "OASIS_UNKNOWN_STATUS";
}

int32_t oasis_version(void) { return 100; }

}  // extern "C"
