// One layer-step's two HBM streams in one launch: the block-sparse attention
// of one layer and the look-ahead scoring of another ("OasisKV: Scaling
// In-Decode KV Cache Beyond HBM with Lookahead Sparse Prefetching", Fig. 8:
// a layer's prediction runs in the background of the following layers'
// compute).  The two are independent; fusing them fixes how they share the
// SMs instead of leaving it to the block scheduler.
//
// GB300 design: one CTA per SM with 4 attention warps and 4 scoring warps
// (measured per Llama layer-step with 3/4/5/6/7/8 scoring warps:
// 28.1/26.0/26.5/26.9/27.3/27.4 us).
// The attention CTAs (P per unit, in clusters of P, exactly as the attention
// kernel) come first; the rest of the grid is scoring-only and there all eight
// warps score.  The scoring tiles are spread evenly over the scoring warps.
// Both roles are the bodies of the separate kernels; the attention warps
// synchronise on named barrier 1, the scoring warps never wait for them.
// The launch is a programmatic dependent of the stream's previous kernel:
// its CTAs start while that kernel drains and wait (griddepcontrol) for its
// results before reading anything, so back-to-back steps overlap launch and
// tail (27.65 -> 27.2 us per pipelined Llama layer-step).
#include "attn_body.cuh"
#include "launch.h"
#include "score_body.cuh"

namespace oasis {

constexpr int kFusedScoreWarps = 4;
constexpr int kFusedThreads = (kAttnWarps + kFusedScoreWarps) * 32;
constexpr size_t kFusedScoreRing = static_cast<size_t>(kScoreStages) * 8 * 32 * sizeof(float4);
constexpr size_t kFusedSmem = kAttnSmem + kFusedScoreWarps * kFusedScoreRing;
// Tiles of a scoring warp in a CTA that also attends, relative to one in a
// scoring-only CTA (measured best at an equal share; 0.8 and 1.2-1.5 slower).
constexpr double kAttendingWarpShare = 1.0;

__device__ __forceinline__ void attn_warps_barrier() {
  asm volatile("bar.sync 1, %0;\n" ::"n"(kAttnThreads) : "memory");
}

template <int MT, int KIND>
__device__ __forceinline__ void attn_score_body(
    const CUtensorMap* tm_k, const CUtensorMap* tm_v,
    const uint16_t* __restrict__ q, const int32_t* __restrict__ block_of_slot,
    const int32_t* __restrict__ ctx_len, float scale_log2, uint16_t* __restrict__ out,
    const uint16_t* __restrict__ q_draft, const float4* __restrict__ summ,
    float* __restrict__ scores, int Hq, int Hkv, int G, int S, int NB, int L, int P, int nA,
    int T, int Ra, int Rs, uint32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  // launched as a programmatic dependent of the stream's previous kernel:
  // let the next one launch, then wait for the previous one's results
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  if (c < nA && warp < kAttnWarps) {
    const int u = c / P, b = u / Hkv, h = u - b * Hkv;
    const GroupRows rows{q, out, (static_cast<int64_t>(b) * Hq + h * G) * kHeadDim};
    attn_cta<1>(tm_k, tm_v, rows, G, block_of_slot, ctx_len, scale_log2, Hkv, S, NB, P, err, smem,
                u, c % P, warp, lane, [] { attn_warps_barrier(); });
    return;
  }
  // scoring warps (all eight in a scoring-only CTA): this CTA's tiles, then a
  // contiguous share of them per warp
  const bool attends = c < nA;
  const int nsw = attends ? kFusedScoreWarps : kFusedScoreWarps + kAttnWarps;
  const int sw = attends ? warp - kAttnWarps : warp;
  const int64_t lo = attends ? static_cast<int64_t>(c) * Ra
                             : static_cast<int64_t>(nA) * Ra + static_cast<int64_t>(c - nA) * Rs;
  const int n = attends ? Ra : Rs;
  const int t_lo = lo < T ? static_cast<int>(lo) : T;
  const int t_hi = t_lo + n < T ? t_lo + n : T;
  const int qw = (t_hi - t_lo + nsw - 1) / nsw;
  const int w_lo = t_lo + sw * qw < t_hi ? t_lo + sw * qw : t_hi;
  const int tpw = w_lo + qw < t_hi ? qw : t_hi - w_lo;
  float4* ring = reinterpret_cast<float4*>(smem + (attends ? kAttnSmemBody : 0)) +
                 sw * kScoreStages * 8 * 32;
  score_warp_range<MT, KIND>(q_draft, summ, scores, L, Hq, Hkv, G, NB, w_lo, tpw, ring, lane);
}

#define OASIS_FUSED_PARAMS                                                                       \
  const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,            \
      const uint16_t *__restrict__ q, const int32_t *__restrict__ block_of_slot,                 \
      const int32_t *__restrict__ ctx_len, float scale_log2, uint16_t *__restrict__ out,         \
      const uint16_t *__restrict__ q_draft, const float4 *__restrict__ summ,                     \
      float *__restrict__ scores, int Hq, int Hkv, int G, int S, int NB, int L, int P, int nA,    \
      int T, int Ra, int Rs, uint32_t *err
#define OASIS_FUSED_ARGS                                                                         \
  &tm_k, &tm_v, q, block_of_slot, ctx_len, scale_log2, out, q_draft, summ, scores, Hq, Hkv, G, S, \
      NB, L, P, nA, T, Ra, Rs, err

// At most 128 registers a thread (up to 16 scoring rows, and 32 with the mean
// keys).  With the CTA's warps at 128 the SM's four register banks keep room for the
// step's top-K + plan CTA beside this one; at 130 (the 16-row min/max-key
// instantiation uncapped) that CTA no longer fits and waits for the whole
// launch (43 instead of 27 us per Llama layer-step).
template <int MT, int KIND>
__global__ void __maxnreg__(128) attn_score_kernel(OASIS_FUSED_PARAMS) {
  attn_score_body<MT, KIND>(OASIS_FUSED_ARGS);
}

// Wider query tiles (48 or 64 rows; 32 with min/max keys, whose query
// fragments stay unpacked): the registers they need.
template <int MT, int KIND>
__global__ void __launch_bounds__(kFusedThreads) attn_score_kernel_wide(OASIS_FUSED_PARAMS) {
  attn_score_body<MT, KIND>(OASIS_FUSED_ARGS);
}

template <int MT, int KIND>
constexpr auto fused_kernel() {
  if constexpr (MT == 1 || (MT == 2 && KIND == kSummMean))
    return attn_score_kernel<MT, KIND>;
  else
    return attn_score_kernel_wide<MT, KIND>;
}

template <int MT, int KIND>
static cudaError_t fused_configure_mt() {
  const auto fn = fused_kernel<MT, KIND>();
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kFusedSmem));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  return e;
}

cudaError_t fused_configure() {
  cudaError_t e = fused_configure_mt<1, kSummMean>();
  if (e == cudaSuccess) e = fused_configure_mt<2, kSummMean>();
  if (e == cudaSuccess) e = fused_configure_mt<3, kSummMean>();
  if (e == cudaSuccess) e = fused_configure_mt<4, kSummMean>();
  if (e == cudaSuccess) e = fused_configure_mt<1, kSummMinMax>();
  if (e == cudaSuccess) e = fused_configure_mt<2, kSummMinMax>();
  return e;
}

template <int MT, int KIND>
static cudaError_t launch_fused_mt(const Shape& s, const CUtensorMap& tm_k,
                                   const CUtensorMap& tm_v, const uint16_t* q,
                                   const int32_t* block_of_slot, const int32_t* ctx_len,
                                   float scale, uint16_t* out, const uint16_t* q_draft,
                                   const void* summ, float* scores, cudaStream_t st,
                                   const DeviceInfo& di) {
  const int sms = di.sm_count > 0 ? di.sm_count : 148;
  const int P = attn_split(s, sms);
  const int nA = s.units() * P;
  const int ntiles = (s.NB + 7) / 8;
  const int64_t T = static_cast<int64_t>(s.units()) * ntiles;
  // the grid: the attention CTAs, then whole clusters of scoring-only CTAs up to one per SM
  const int C = nA < sms ? nA + (sms - nA) / P * P : nA;
  // scoring tiles per scoring warp: kAttendingWarpShare as many in a CTA that
  // also attends (4 scoring warps) as in a scoring-only one (8); the scoring
  // warps are bound by their own instruction latency, not by the SM's bytes
  int64_t Ra, Rs = 0;
  if (C > nA) {
    const double wa = kFusedScoreWarps * kAttendingWarpShare, ws = kFusedScoreWarps + kAttnWarps;
    Ra = static_cast<int64_t>(static_cast<double>(T) * wa / (wa * nA + ws * (C - nA)));
    Rs = (T - nA * Ra + (C - nA) - 1) / (C - nA);
    if (Rs < 0) Rs = 0;
  } else {
    Ra = (T + nA - 1) / nA;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(C));
  cfg.blockDim = dim3(kFusedThreads);
  cfg.dynamicSmemBytes = kFusedSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(P);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = P > 1 ? 2 : 1;
  const float scale_log2 = scale * 1.4426950408889634f;
  return cudaLaunchKernelEx(&cfg, fused_kernel<MT, KIND>(), tm_k, tm_v, q, block_of_slot,
                            ctx_len, scale_log2, out, q_draft, static_cast<const float4*>(summ),
                            scores, s.Hq, s.Hkv, s.G, s.S, s.NB,
                            s.L, P, nA, static_cast<int>(T), static_cast<int>(Ra),
                            static_cast<int>(Rs), di.err);
}

cudaError_t launch_attend_and_score(const Shape& s, const CUtensorMap& tm_k,
                                    const CUtensorMap& tm_v, const uint16_t* q,
                                    const int32_t* block_of_slot, const int32_t* ctx_len,
                                    float scale, uint16_t* out, const uint16_t* q_draft,
                                    const void* summ, bool minmax, float* scores,
                                    cudaStream_t st, const DeviceInfo& di) {
  const int mt = (s.L * s.G + 15) / 16;
#define OASIS_FUSED(M, K)                                                                        \
  return launch_fused_mt<M, K>(s, tm_k, tm_v, q, block_of_slot, ctx_len, scale, out, q_draft,  \
                               summ, scores, st, di)
  if (minmax) {
    if (mt == 1) OASIS_FUSED(1, kSummMinMax);
    if (mt == 2) OASIS_FUSED(2, kSummMinMax);
    return cudaErrorInvalidValue;  // rejected earlier by validation (L*G <= 32)
  }
  if (mt == 1) OASIS_FUSED(1, kSummMean);
  if (mt == 2) OASIS_FUSED(2, kSummMean);
  if (mt == 3) OASIS_FUSED(3, kSummMean);
  if (mt == 4) OASIS_FUSED(4, kSummMean);
#undef OASIS_FUSED
  return cudaErrorInvalidValue;  // rejected earlier by validation (L*G <= 64)
}

}  // namespace oasis
