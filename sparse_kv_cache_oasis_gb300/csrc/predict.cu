// Top-K block prediction and capped-eviction planning ("OasisKV: Scaling
// In-Decode KV Cache Beyond HBM with Lookahead Sparse Prefetching",
// explanatory diagram steps 2-3; Fig. 4; Tab. 2 fetch cap and LRU eviction;
// Fig. 9 head-wise GPU-slot <-> CPU-block map).
//
// Both steps are small integer work per (request, KV head) and bound by
// latency, so each unit is one CTA and the code is organised to keep the
// chain of dependent memory round trips and barriers short:
//
// Top-K (topk_unit): scores stay in registers as order-preserving 32-bit
// keys (-0.0 folded onto +0.0, so the order is the fp32 order); a 4-pass MSB
// radix select with warp-aggregated shared histograms finds the threshold;
// equal keys are taken by ascending id; the selected blocks are compacted with
// one atomic per warp and placed by counting larger 64-bit keys
// (score_key << 32 | ~id), several threads per key.  Forced blocks (sink and
// local window) come first in ascending id.  Output order: score descending,
// id ascending -- the fetch priority.
//
// Plan (plan_unit): the working-set map entries are loaded up front; ids are
// checked with a shared bitmap; LRU victims are ranked by counting smaller
// 64-bit (last_used, block) keys; prefix sums give the fetch set and the free
// slots; fetched blocks in ascending id take the free slots in ascending
// order.  Results equal the plain sequential definition exactly.  Bad input
// (id out of range or repeated, map directions disagreeing) leaves the unit
// unchanged, reports n = e = 0 and sets an error bit.
//
// Three kernels: top-K alone, plan alone, and both fused in one CTA (the
// top-K list never leaves shared memory before the plan uses it, and the map
// loads overlap the selection).
#include "predict_body.cuh"

namespace oasis {

// ---------------------------------------------------------------- kernels
template <int ITEMS, bool CTX>
__global__ void __launch_bounds__(kPredThreads) topk_kernel(const float* __restrict__ scores,
                                                            const int32_t* __restrict__ ctx_len,
                                                            int32_t* __restrict__ topk_ids,
                                                            int NB, int K, int sink, int local,
                                                            int Hkv, int bs, PredLayout lay) {
  extern __shared__ __align__(16) unsigned char pred_smem[];
  int* sP;
  TopkSmem tk;
  PlanSmem pl;
  lay.carve(pred_smem, &sP, &tk, &pl);
  const int64_t u = blockIdx.x;
  const int nblk = CTX ? context_blocks(ctx_len, static_cast<int>(u / Hkv), bs, NB) : NB;
  topk_unit<ITEMS, CTX>(scores + u * NB, NB, nblk, K, sink, local, sP, topk_ids + u * K, tk);
}

__global__ void __launch_bounds__(kPredThreads) plan_kernel(
    const int32_t* __restrict__ topk_ids, int32_t step, int32_t* __restrict__ clock,
    int32_t* __restrict__ slot_of_block, int32_t* __restrict__ block_of_slot,
    int32_t* __restrict__ last_used, int32_t* __restrict__ fetch_block,
    int32_t* __restrict__ fetch_slot, int32_t* __restrict__ evict_block,
    int32_t* __restrict__ n_fetch, int32_t* __restrict__ n_evict, int NB, int S, int K, int cap,
    int capw, uint32_t* err, PredLayout lay) {
  extern __shared__ __align__(16) unsigned char pred_smem[];
  int* sP;
  TopkSmem tk;
  PlanSmem pl;
  lay.carve(pred_smem, &sP, &tk, &pl);
  const int64_t u = blockIdx.x;
  const int32_t st = clock ? clock[u] : step;
  int32_t* sob = slot_of_block + u * NB;
  const SlotView v = load_slot_view(sob, block_of_slot + u * S, last_used + u * S, S, NB);
  for (int i = threadIdx.x; i < K; i += blockDim.x) sP[i] = topk_ids[u * K + i];
  __syncthreads();
  plan_unit(sP, v, st, clock ? clock + u : nullptr, sob, block_of_slot + u * S, last_used + u * S,
            fetch_block + u * capw, fetch_slot + u * capw, evict_block + u * capw, n_fetch + u,
            n_evict + u, NB, S, K, cap, capw, err, pl);
}

// Top-K and plan of one unit in one CTA; the map loads overlap the selection.
template <int ITEMS, bool CTX>
__global__ void __launch_bounds__(kPredThreads) topk_plan_kernel(
    const float* __restrict__ scores, const int32_t* __restrict__ ctx_len,
    int32_t* __restrict__ topk_ids, int32_t step,
    int32_t* __restrict__ clock, int32_t* __restrict__ slot_of_block,
    int32_t* __restrict__ block_of_slot, int32_t* __restrict__ last_used,
    int32_t* __restrict__ fetch_block, int32_t* __restrict__ fetch_slot,
    int32_t* __restrict__ evict_block, int32_t* __restrict__ n_fetch,
    int32_t* __restrict__ n_evict, int NB, int S, int K, int cap, int capw, int sink, int local,
    int Hkv, int bs, uint32_t* err, PredLayout lay) {
  extern __shared__ __align__(16) unsigned char pred_smem[];
  int* sP;
  TopkSmem tk;
  PlanSmem pl;
  lay.carve(pred_smem, &sP, &tk, &pl);
  const int64_t u = blockIdx.x;
  const int32_t st = clock ? clock[u] : step;
  int32_t* sob = slot_of_block + u * NB;
  const SlotView v = load_slot_view(sob, block_of_slot + u * S, last_used + u * S, S, NB);
  const int nblk = CTX ? context_blocks(ctx_len, static_cast<int>(u / Hkv), bs, NB) : NB;
  topk_unit<ITEMS, CTX>(scores + u * NB, NB, nblk, K, sink, local, sP, topk_ids + u * K, tk);
  plan_unit(sP, v, st, clock ? clock + u : nullptr, sob, block_of_slot + u * S, last_used + u * S,
            fetch_block + u * capw, fetch_slot + u * capw, evict_block + u * capw, n_fetch + u,
            n_evict + u, NB, S, K, cap, capw, err, pl);
}

// Largest shared-memory carve-out for the top-K / plan kernels: they run on
// SMs that also host the attention and scoring kernels of the step.
template <int N>
static cudaError_t pred_configure_n() {
  const int c = cudaSharedmemCarveoutMaxShared;
  cudaError_t e = cudaFuncSetAttribute(topk_kernel<N, false>, cudaFuncAttributePreferredSharedMemoryCarveout, c);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(topk_kernel<N, true>, cudaFuncAttributePreferredSharedMemoryCarveout, c);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(topk_plan_kernel<N, false>, cudaFuncAttributePreferredSharedMemoryCarveout, c);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(topk_plan_kernel<N, true>, cudaFuncAttributePreferredSharedMemoryCarveout, c);
  return e;
}

cudaError_t pred_configure() {
  cudaError_t e = cudaFuncSetAttribute(plan_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                       cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess) e = pred_configure_n<1>();
  if (e == cudaSuccess) e = pred_configure_n<2>();
  if (e == cudaSuccess) e = pred_configure_n<4>();
  if (e == cudaSuccess) e = pred_configure_n<8>();
  if (e == cudaSuccess) e = pred_configure_n<16>();
  if (e == cudaSuccess) e = pred_configure_n<32>();
  return e;
}

#define OASIS_ITEMS_SWITCH(items, CALL) \
  do {                                  \
    if ((items) <= 1) CALL(1);          \
    if ((items) <= 2) CALL(2);          \
    if ((items) <= 4) CALL(4);          \
    if ((items) <= 8) CALL(8);          \
    if ((items) <= 16) CALL(16);        \
    if ((items) <= 32) CALL(32);        \
    return cudaErrorInvalidValue;       \
  } while (0)

cudaError_t launch_select_topk(const Shape& s, const float* scores, const int32_t* ctx_len,
                               int32_t* topk_ids, cudaStream_t st, const DeviceInfo&) {
  const int T = pred_threads(s.K, s.NB);
  const int items = (s.NB + T - 1) / T;
  const PredLayout lay = pred_layout(s);
#define OASIS_TOPK(N)                                                                              \
  {                                                                                                \
    if (ctx_len)                                                                                   \
      topk_kernel<N, true><<<s.units(), T, lay.bytes(), st>>>(scores, ctx_len, topk_ids, s.NB, s.K,   \
                                                              s.sink, s.local, s.Hkv, s.bs, lay);   \
    else                                                                                           \
      topk_kernel<N, false><<<s.units(), T, lay.bytes(), st>>>(scores, ctx_len, topk_ids, s.NB, s.K,  \
                                                               s.sink, s.local, s.Hkv, s.bs, lay);  \
    return cudaGetLastError();                                                                     \
  }
  OASIS_ITEMS_SWITCH(items, OASIS_TOPK);
#undef OASIS_TOPK
}

cudaError_t launch_plan_fetch(const Shape& s, const int32_t* topk_ids, int32_t step,
                              int32_t* clock, int32_t* slot_of_block, int32_t* block_of_slot,
                              int32_t* last_used, int32_t* fetch_block, int32_t* fetch_slot,
                              int32_t* evict_block, int32_t* n_fetch, int32_t* n_evict,
                              cudaStream_t st, const DeviceInfo& di) {
  const int capw = s.cap > 0 ? s.cap : 1;
  const PredLayout lay = pred_layout(s);
  const int need = s.S > s.K ? s.S : s.K;
  plan_kernel<<<s.units(), pred_threads(need, 0), lay.bytes(), st>>>(
      topk_ids, step, clock, slot_of_block, block_of_slot, last_used, fetch_block, fetch_slot,
      evict_block, n_fetch, n_evict, s.NB, s.S, s.K, s.cap, capw, di.err, lay);
  return cudaGetLastError();
}

cudaError_t launch_select_and_plan(const Shape& s, const float* scores, const int32_t* ctx_len,
                                   int32_t* topk_ids,
                                   int32_t step, int32_t* clock, int32_t* slot_of_block,
                                   int32_t* block_of_slot, int32_t* last_used,
                                   int32_t* fetch_block, int32_t* fetch_slot,
                                   int32_t* evict_block, int32_t* n_fetch, int32_t* n_evict,
                                   cudaStream_t st, const DeviceInfo& di) {
  const int capw = s.cap > 0 ? s.cap : 1;
  const int need = s.S > s.K ? s.S : s.K;
  const int T = pred_threads(need, s.NB);
  const int items = (s.NB + T - 1) / T;
  const PredLayout lay = pred_layout(s);
#define OASIS_TP(N)                                                                             \
  {                                                                                             \
    if (ctx_len)                                                                                \
      topk_plan_kernel<N, true><<<s.units(), T, lay.bytes(), st>>>(                             \
          scores, ctx_len, topk_ids, step, clock, slot_of_block, block_of_slot, last_used,      \
          fetch_block, fetch_slot, evict_block, n_fetch, n_evict, s.NB, s.S, s.K, s.cap, capw,   \
          s.sink, s.local, s.Hkv, s.bs, di.err, lay);                                           \
    else                                                                                        \
      topk_plan_kernel<N, false><<<s.units(), T, lay.bytes(), st>>>(                            \
          scores, ctx_len, topk_ids, step, clock, slot_of_block, block_of_slot, last_used,      \
          fetch_block, fetch_slot, evict_block, n_fetch, n_evict, s.NB, s.S, s.K, s.cap, capw,   \
          s.sink, s.local, s.Hkv, s.bs, di.err, lay);                                           \
    return cudaGetLastError();                                                                  \
  }
  OASIS_ITEMS_SWITCH(items, OASIS_TP);
#undef OASIS_TP
}

}  // namespace oasis
