// Look-ahead block scoring ("OasisKV: Scaling In-Decode KV Cache Beyond HBM
// with Lookahead Sparse Prefetching", Fig. 7 right; 'What they did' item 2):
// the draft tokens' queries scan the compressed key of every block,
//   score[b,h,j] = max over (l, g) of q_draft[b,l,h*G+g,:] . summ[b,h,j,:].
//
// This is a dense contraction per (request, KV head): Q (L*G x 128) times
// the summaries (128 x NB), then a max over the L*G rows.  It reads 512 B of
// summary per block and does L*G*128 multiply-adds on it (8-16 flop/B at the
// workloads' shapes), which is at or above the fp32 CUDA-core rate at full
// HBM bandwidth, so it runs on the tensor cores:
//   - A = queries: bf16 values are exact in tf32;
//   - B = summaries: fp32 split as hi = x with its 13 low mantissa bits
//     cleared (exactly a tf32 value) and lo = x - hi (exact in fp32; the
//     tensor core reads it as tf32, dropping at most 2^-11 of it), two MMA
//     passes; the product error is ~2^-21 relative, far below the fp32 result
//     rounding that ranking depends on;
//   - mma.sync m16n8k8 tf32 with fp32 accumulation, one 16-row tile per 16
//     query rows.
// Memory path: summaries are streamed once with 16-byte cp.async copies into
// a per-warp ring of kScoreStages tiles in shared memory (L1 bypassed); each
// lane copies exactly the 8 x 16 bytes its B fragments need and reads them back
// itself, so the ring layout [p][lane] is bank-conflict free and needs no
// barrier.  The contraction index is permuted so that thread (g, t) of a warp
// loads 16 contiguous bytes of block g: dims 16p+4t..16p+4t+3 serve k-steps
// 2p and 2p+1 (A uses the same permutation, so the dot products are unchanged).
// Each lane keeps its A fragments of the current unit in registers as the
// queries' own bf16 pairs (a bf16 value is a tf32 value with zero low bits, so
// unpacking is a shift or a mask); only the summaries pass through shared
// memory, which halves the kernel's shared-memory traffic against staging the
// queries there, and leaves the SM's shared-memory bandwidth to the attention
// kernel running beside it.
// Balance: the tiles of 8 consecutive blocks of all (request, KV head) units
// form one list of T tiles; CTA c (two per SM) takes the contiguous range
// [c*Rt, (c+1)*Rt) and each warp a contiguous sixth of it, so every SM
// streams the same number of bytes whatever NB and the unit count, and a
// warp reloads its query fragments only where its tiles cross into the next
// unit.  Two CTAs per SM (72 KiB of rings each) took 16.4 us at the Llama
// layer against 18.9 us for one: the kernel is bound by each warp's latency
// per tile, and twice the warps hide more of it.  A caller that wants the
// attention and the scoring at once uses the fused launch (stream.cu), which
// shares every SM between the two roles.
#include "launch.h"
#include "score_body.cuh"

namespace oasis {

constexpr int kScoreThreads = 192;
constexpr int kScoreWarps = kScoreThreads / 32;
constexpr int kMinTilesPerCta = 16;
constexpr int kScoreCtasPerSm = 2;  // resident CTAs of this kernel per SM

template <int MT, int KIND>
__global__ void __launch_bounds__(kScoreThreads) score_kernel(
    const uint16_t* __restrict__ q_draft, const float4* __restrict__ summ,
    float* __restrict__ scores, int L, int Hq, int Hkv, int G, int NB, int T, int Rt) {
  // shared memory: one ring per warp of kScoreStages tiles, each [p][lane]
  // float4 (a lane reads back what it copied)
  extern __shared__ float4 smem4[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t_lo = blockIdx.x * Rt;
  const int t_hi = t_lo + Rt < T ? t_lo + Rt : T;
  // this warp's tiles: the contiguous [w_lo, w_lo + tpw)
  const int qw = (t_hi - t_lo + kScoreWarps - 1) / kScoreWarps;
  const int w_lo = t_lo + warp * qw < t_hi ? t_lo + warp * qw : t_hi;
  const int tpw = w_lo + qw < t_hi ? qw : t_hi - w_lo;
  score_warp_range<MT, KIND>(q_draft, summ, scores, L, Hq, Hkv, G, NB, w_lo, tpw,
                             smem4 + warp * kScoreStages * 8 * 32, lane);
}

static size_t score_smem_bytes(int) {
  return sizeof(float4) * static_cast<size_t>(kScoreWarps) * kScoreStages * 8 * 32;
}

template <int MT, int KIND>
static cudaError_t launch_mt(const Shape& s, const uint16_t* q_draft, const void* summ,
                             float* scores, cudaStream_t st, const DeviceInfo& di) {
  // kScoreCtasPerSm CTAs per SM over equal contiguous tile ranges
  const int ntiles = (s.NB + 7) / 8;
  const int64_t T = static_cast<int64_t>(s.units()) * ntiles;
  int64_t C = static_cast<int64_t>(kScoreCtasPerSm) * (di.sm_count > 0 ? di.sm_count : 148);
  const int64_t cap = (T + kMinTilesPerCta - 1) / kMinTilesPerCta;
  if (C > cap) C = cap;
  if (C < 1) C = 1;
  const int64_t Rt = (T + C - 1) / C;
  const int64_t grid = (T + Rt - 1) / Rt;
  score_kernel<MT, KIND><<<static_cast<unsigned>(grid), kScoreThreads, score_smem_bytes(MT), st>>>(
      q_draft, static_cast<const float4*>(summ), scores, s.L, s.Hq, s.Hkv, s.G, s.NB,
      static_cast<int>(T), static_cast<int>(Rt));
  return cudaGetLastError();
}

cudaError_t launch_score_blocks(const Shape& s, const uint16_t* q_draft, const float* summ,
                                float* scores, cudaStream_t st, const DeviceInfo& di) {
  const int mt = (s.L * s.G + 15) / 16;
  switch (mt) {
    case 1: return launch_mt<1, kSummMean>(s, q_draft, summ, scores, st, di);
    case 2: return launch_mt<2, kSummMean>(s, q_draft, summ, scores, st, di);
    case 3: return launch_mt<3, kSummMean>(s, q_draft, summ, scores, st, di);
    case 4: return launch_mt<4, kSummMean>(s, q_draft, summ, scores, st, di);
    default: return cudaErrorInvalidValue;  // rejected earlier by validation (L*G <= 64)
  }
}

cudaError_t launch_score_blocks_minmax(const Shape& s, const uint16_t* q_draft,
                                       const uint16_t* summ_mm, float* scores, cudaStream_t st,
                                       const DeviceInfo& di) {
  const int mt = (s.L * s.G + 15) / 16;
  switch (mt) {
    case 1: return launch_mt<1, kSummMinMax>(s, q_draft, summ_mm, scores, st, di);
    case 2: return launch_mt<2, kSummMinMax>(s, q_draft, summ_mm, scores, st, di);
    default: return cudaErrorInvalidValue;  // rejected earlier by validation (L*G <= 32)
  }
}

template <int MT, int KIND>
static cudaError_t score_configure_mt() {
  const auto fn = score_kernel<MT, KIND>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(score_smem_bytes(MT)));
  if (e == cudaSuccess)  // largest carve-out: the step's other kernels share the SM
    e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  return e;
}

cudaError_t score_configure() {
  cudaError_t e = score_configure_mt<1, kSummMean>();
  if (e == cudaSuccess) e = score_configure_mt<2, kSummMean>();
  if (e == cudaSuccess) e = score_configure_mt<3, kSummMean>();
  if (e == cudaSuccess) e = score_configure_mt<4, kSummMean>();
  if (e == cudaSuccess) e = score_configure_mt<1, kSummMinMax>();
  if (e == cudaSuccess) e = score_configure_mt<2, kSummMinMax>();
  return e;
}

int score_ctas_per_sm() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, score_kernel<1, kSummMean>, kScoreThreads,
                                                    score_smem_bytes(1)) != cudaSuccess)
    return 2;
  return n > 0 ? n : 1;
}

}  // namespace oasis
