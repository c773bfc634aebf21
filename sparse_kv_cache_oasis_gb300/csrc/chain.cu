// The prediction chain in one launch ("OasisKV: Scaling In-Decode KV Cache
// Beyond HBM with Lookahead Sparse Prefetching", Fig. 7 right and the
// explanatory diagram steps 2-3): a (request, KV head) unit's look-ahead
// scoring, its top-K and its capped-eviction plan without kernel boundaries
// between them.  Same arithmetic as oasis_score_blocks followed by
// oasis_predict_select, bit for bit.
//
// GB300 design: the P CTAs of a unit form a thread-block cluster.  Every CTA
// scores a contiguous share of the unit's 8-block tiles with the scoring body
// (per-warp cp.async rings, tensor-core contraction) and writes its scores to
// global memory, where they stay in L2; one cluster barrier (release / acquire
// at cluster scope) publishes them; the unit's first CTA then runs the top-K
// and plan bodies over them (map loads first, so that they overlap the
// selection) while the other CTAs of the cluster are done.  256 threads per
// CTA serve both roles: 8 scoring warps, then the top-K's 256 threads.
#include <cooperative_groups.h>

#include "launch.h"
#include "predict_body.cuh"
#include "score_body.cuh"

namespace oasis {

namespace cg = cooperative_groups;

constexpr int kChainThreads = 256;
constexpr int kChainWarps = kChainThreads / 32;
constexpr size_t kChainRingBytes =
    static_cast<size_t>(kChainWarps) * kScoreStages * 8 * 32 * sizeof(float4);

template <int MT, int ITEMS>
__global__ void __launch_bounds__(kChainThreads, 1) chain_kernel(
    const uint16_t* __restrict__ q_draft, const float4* __restrict__ summ,
    float* __restrict__ scores, int32_t step, int32_t* __restrict__ clock,
    int32_t* __restrict__ topk_ids, int32_t* __restrict__ slot_of_block,
    int32_t* __restrict__ block_of_slot, int32_t* __restrict__ last_used,
    int32_t* __restrict__ fetch_block, int32_t* __restrict__ fetch_slot,
    int32_t* __restrict__ evict_block, int32_t* __restrict__ n_fetch,
    int32_t* __restrict__ n_evict, int L, int Hq, int Hkv, int G, int NB, int S, int K, int cap,
    int capw, int sink, int local, int P, uint32_t* err, PredLayout lay) {
  extern __shared__ __align__(16) unsigned char chain_smem[];
  const int u = blockIdx.x / P, r = blockIdx.x - u * P;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // this CTA's tiles of the unit, a contiguous share of them per warp
  const int ntiles = (NB + 7) >> 3;
  const int t_lo = u * ntiles + (r * ntiles) / P, t_hi = u * ntiles + ((r + 1) * ntiles) / P;
  const int qw = (t_hi - t_lo + kChainWarps - 1) / kChainWarps;
  const int w_lo = t_lo + warp * qw < t_hi ? t_lo + warp * qw : t_hi;
  const int tpw = w_lo + qw < t_hi ? qw : t_hi - w_lo;
  score_warp_range<MT>(q_draft, summ, scores, L, Hq, Hkv, G, NB, w_lo, tpw,
                       reinterpret_cast<float4*>(chain_smem) + warp * kScoreStages * 8 * 32, lane);
  if (P > 1)
    cg::this_cluster().sync();  // every CTA's scores are visible to the unit's first CTA
  else
    __syncthreads();
  if (r != 0) return;
  int* sP;
  TopkSmem tk;
  PlanSmem pl;
  lay.carve(chain_smem + kChainRingBytes, &sP, &tk, &pl);
  const int32_t st = clock ? clock[u] : step;
  int32_t* sob = slot_of_block + static_cast<int64_t>(u) * NB;
  int32_t* bos = block_of_slot + static_cast<int64_t>(u) * S;
  int32_t* lu = last_used + static_cast<int64_t>(u) * S;
  const SlotView v = load_slot_view(sob, bos, lu, S, NB);
  topk_unit<ITEMS, false>(scores + static_cast<int64_t>(u) * NB, NB, NB, K, sink, local, sP,
                          topk_ids + static_cast<int64_t>(u) * K, tk);
  plan_unit(sP, v, st, clock ? clock + u : nullptr, sob, bos, lu, fetch_block + u * capw,
            fetch_slot + u * capw, evict_block + u * capw, n_fetch + u, n_evict + u, NB, S, K, cap,
            capw, err, pl);
}

static int chain_split(const Shape& s, int sm_count) {
  const int ntiles = (s.NB + 7) / 8;
  int p = (sm_count > 0 ? sm_count : 148) / s.units();
  if (p > 8) p = 8;
  if (p > ntiles) p = ntiles;
  return p < 1 ? 1 : p;
}

bool chain_supported(const Shape& s) {
  return s.L * s.G <= 32 && s.S <= kChainThreads && s.K <= kChainThreads &&
         s.NB <= 32 * kChainThreads;
}

template <int MT, int ITEMS>
static cudaError_t chain_configure_one() {
  const auto fn = chain_kernel<MT, ITEMS>;
  // the largest layout the supported shapes need
  PredLayout lay;
  lay.K = kChainThreads;
  lay.S = kChainThreads;
  lay.NB = 32 * kChainThreads;
  lay.capw = kChainThreads;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kChainRingBytes + lay.bytes()));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  return e;
}

template <int MT>
static cudaError_t chain_configure_mt() {
  cudaError_t e = chain_configure_one<MT, 1>();
  if (e == cudaSuccess) e = chain_configure_one<MT, 2>();
  if (e == cudaSuccess) e = chain_configure_one<MT, 4>();
  if (e == cudaSuccess) e = chain_configure_one<MT, 8>();
  if (e == cudaSuccess) e = chain_configure_one<MT, 16>();
  if (e == cudaSuccess) e = chain_configure_one<MT, 32>();
  return e;
}

cudaError_t chain_configure() {
  cudaError_t e = chain_configure_mt<1>();
  if (e == cudaSuccess) e = chain_configure_mt<2>();
  return e;
}

template <int MT, int ITEMS>
static cudaError_t launch_one(const Shape& s, const uint16_t* q_draft, const float* summ,
                              float* scores, int32_t step, int32_t* clock, int32_t* topk_ids,
                              int32_t* slot_of_block, int32_t* block_of_slot, int32_t* last_used,
                              int32_t* fetch_block, int32_t* fetch_slot, int32_t* evict_block,
                              int32_t* n_fetch, int32_t* n_evict, cudaStream_t st,
                              const DeviceInfo& di) {
  const int P = chain_split(s, di.sm_count);
  const PredLayout lay = pred_layout(s);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(s.units() * P));
  cfg.blockDim = dim3(kChainThreads);
  cfg.dynamicSmemBytes = kChainRingBytes + lay.bytes();
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(P);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = P > 1 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, chain_kernel<MT, ITEMS>, q_draft,
                            reinterpret_cast<const float4*>(summ), scores, step, clock, topk_ids,
                            slot_of_block, block_of_slot, last_used, fetch_block, fetch_slot,
                            evict_block, n_fetch, n_evict, s.L, s.Hq, s.Hkv, s.G, s.NB, s.S, s.K,
                            s.cap, s.cap > 0 ? s.cap : 1, s.sink, s.local, P, di.err, lay);
}

template <int MT>
static cudaError_t launch_mt(const Shape& s, const uint16_t* q_draft, const float* summ,
                             float* scores, int32_t step, int32_t* clock, int32_t* topk_ids,
                             int32_t* slot_of_block, int32_t* block_of_slot, int32_t* last_used,
                             int32_t* fetch_block, int32_t* fetch_slot, int32_t* evict_block,
                             int32_t* n_fetch, int32_t* n_evict, cudaStream_t st,
                             const DeviceInfo& di) {
  const int items = (s.NB + kChainThreads - 1) / kChainThreads;
#define OASIS_CHAIN(N)                                                                          \
  return launch_one<MT, N>(s, q_draft, summ, scores, step, clock, topk_ids, slot_of_block,     \
                           block_of_slot, last_used, fetch_block, fetch_slot, evict_block,      \
                           n_fetch, n_evict, st, di)
  if (items <= 1) OASIS_CHAIN(1);
  if (items <= 2) OASIS_CHAIN(2);
  if (items <= 4) OASIS_CHAIN(4);
  if (items <= 8) OASIS_CHAIN(8);
  if (items <= 16) OASIS_CHAIN(16);
  if (items <= 32) OASIS_CHAIN(32);
#undef OASIS_CHAIN
  return cudaErrorInvalidValue;
}

cudaError_t launch_predict_chain(const Shape& s, const uint16_t* q_draft, const float* summ,
                                 float* scores, int32_t step, int32_t* clock, int32_t* topk_ids,
                                 int32_t* slot_of_block, int32_t* block_of_slot,
                                 int32_t* last_used, int32_t* fetch_block, int32_t* fetch_slot,
                                 int32_t* evict_block, int32_t* n_fetch, int32_t* n_evict,
                                 cudaStream_t st, const DeviceInfo& di) {
  if ((s.L * s.G + 15) / 16 <= 1)
    return launch_mt<1>(s, q_draft, summ, scores, step, clock, topk_ids, slot_of_block,
                        block_of_slot, last_used, fetch_block, fetch_slot, evict_block, n_fetch,
                        n_evict, st, di);
  return launch_mt<2>(s, q_draft, summ, scores, step, clock, topk_ids, slot_of_block,
                      block_of_slot, last_used, fetch_block, fetch_slot, evict_block, n_fetch,
                      n_evict, st, di);
}

}  // namespace oasis
