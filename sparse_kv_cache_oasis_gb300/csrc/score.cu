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
//   - B = summaries: fp32 split as hi = tf32(x), lo = tf32(x - hi) (x - hi is
//     exact), two MMA passes; the product error is ~2^-22 relative, far
//     below the fp32 result rounding that ranking depends on;
//   - mma.sync m16n8k8 tf32 with fp32 accumulation, one 16-row tile per 16
//     query rows.
// Memory path: summaries are streamed once with 16-byte evict-first loads
// straight into the MMA fragment registers (no shared-memory staging).  The
// contraction index is permuted so that thread (g, t) of a warp loads 16
// contiguous bytes of block g: dims 16p+4t..16p+4t+3 serve k-steps 2p and
// 2p+1 (A uses the same permutation, so the dot products are unchanged).
// Each warp handles tiles of 8 consecutive blocks; the grid is sized to one
// wave of resident CTAs.
#include "common.cuh"
#include "launch.h"

namespace oasis {

constexpr int kScoreThreads = 256;
constexpr int kScoreWarps = kScoreThreads / 32;

template <int MT>
__global__ void __launch_bounds__(kScoreThreads) score_kernel(
    const uint16_t* __restrict__ q_draft, const float* __restrict__ summ,
    float* __restrict__ scores, int L, int Hq, int Hkv, int G, int NB, int tpw) {
  // A fragments, laid out [mt][p][half][lane] so each warp read is contiguous
  extern __shared__ float4 sQ[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int u = blockIdx.y;
  const int b = u / Hkv, h = u - b * Hkv;
  const int M = L * G;

  for (int idx = tid; idx < MT * 8 * 2 * 32; idx += kScoreThreads) {
    const int ln = idx & 31, half = (idx >> 5) & 1, p = (idx >> 6) & 7, mt = idx >> 9;
    const int row = 16 * mt + (ln >> 2) + 8 * half;
    const int col = 16 * p + 4 * (ln & 3);
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (row < M) {
      const int l = row / G, gq = row - l * G;
      const uint2 w = *reinterpret_cast<const uint2*>(
          q_draft + ((static_cast<int64_t>(b) * L + l) * Hq + h * G + gq) * kHeadDim + col);
      v = make_float4(bf16lo_to_f32(w.x), bf16hi_to_f32(w.x), bf16lo_to_f32(w.y),
                      bf16hi_to_f32(w.y));
    }
    sQ[idx] = v;
  }
  __syncthreads();

  const int ntiles = (NB + 7) >> 3;
  const int tile_base = blockIdx.x * kScoreWarps * tpw;
  const float* base = summ + static_cast<int64_t>(u) * NB * kHeadDim;
  float* out = scores + static_cast<int64_t>(u) * NB;

#pragma unroll 1
  for (int i = 0; i < tpw; ++i) {
    const int tile = tile_base + warp + kScoreWarps * i;
    if (tile >= ntiles) break;
    const int n0 = tile * 8;
    const int blk = n0 + g;
    float4 v[8];
    if (blk < NB) {
      const float4* src = reinterpret_cast<const float4*>(base + static_cast<int64_t>(blk) * kHeadDim) + t;
#pragma unroll
      for (int p = 0; p < 8; ++p) v[p] = __ldcs(src + 4 * p);
    } else {
#pragma unroll
      for (int p = 0; p < 8; ++p) v[p] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float acc[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      const uint32_t hx = to_tf32(v[p].x), hy = to_tf32(v[p].y);
      const uint32_t hz = to_tf32(v[p].z), hw = to_tf32(v[p].w);
      const uint32_t lx = to_tf32(v[p].x - __uint_as_float(hx));
      const uint32_t ly = to_tf32(v[p].y - __uint_as_float(hy));
      const uint32_t lz = to_tf32(v[p].z - __uint_as_float(hz));
      const uint32_t lw = to_tf32(v[p].w - __uint_as_float(hw));
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const float4 qa = sQ[((mt * 8 + p) * 2 + 0) * 32 + lane];
        const float4 qb = sQ[((mt * 8 + p) * 2 + 1) * 32 + lane];
        const uint32_t a0 = __float_as_uint(qa.x), a1 = __float_as_uint(qb.x);
        const uint32_t a2 = __float_as_uint(qa.y), a3 = __float_as_uint(qb.y);
        const uint32_t c0 = __float_as_uint(qa.z), c1 = __float_as_uint(qb.z);
        const uint32_t c2 = __float_as_uint(qa.w), c3 = __float_as_uint(qb.w);
        mma_tf32_1688(acc[mt], a0, a1, a2, a3, hx, hy);  // k-step 2p, hi
        mma_tf32_1688(acc[mt], a0, a1, a2, a3, lx, ly);  // k-step 2p, lo
        mma_tf32_1688(acc[mt], c0, c1, c2, c3, hz, hw);  // k-step 2p+1, hi
        mma_tf32_1688(acc[mt], c0, c1, c2, c3, lz, lw);  // k-step 2p+1, lo
      }
    }
    // max over the valid query rows (rows >= L*G are padding)
    float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      if (16 * mt + g < M) {
        m0 = fmaxf(m0, acc[mt][0]);
        m1 = fmaxf(m1, acc[mt][1]);
      }
      if (16 * mt + g + 8 < M) {
        m0 = fmaxf(m0, acc[mt][2]);
        m1 = fmaxf(m1, acc[mt][3]);
      }
    }
    m0 = warp_max_xor_g(m0);
    m1 = warp_max_xor_g(m1);
    if (g == 0) {
      const int col = n0 + 2 * t;
      if (col + 1 < NB) {
        __stcs(reinterpret_cast<float2*>(out + col), make_float2(m0, m1));
      } else if (col < NB) {
        out[col] = m0;
      }
    }
  }
}

template <int MT>
static cudaError_t launch_mt(const Shape& s, const uint16_t* q_draft, const float* summ,
                             float* scores, cudaStream_t st, const DeviceInfo& di) {
  const int ntiles = (s.NB + 7) / 8;
  const int64_t total_tiles = static_cast<int64_t>(ntiles) * s.units();
  int per_sm = di.score_ctas_per_sm > 0 ? di.score_ctas_per_sm : 2;
  const int64_t warps_resident = static_cast<int64_t>(di.sm_count > 0 ? di.sm_count : 148) * per_sm * kScoreWarps;
  int tpw = static_cast<int>((total_tiles + warps_resident - 1) / warps_resident);
  if (tpw < 1) tpw = 1;
  const int ctas_per_unit = (ntiles + kScoreWarps * tpw - 1) / (kScoreWarps * tpw);
  dim3 grid(ctas_per_unit, s.units());
  const size_t smem = sizeof(float4) * MT * 8 * 2 * 32;
  score_kernel<MT><<<grid, kScoreThreads, smem, st>>>(q_draft, summ, scores, s.L, s.Hq, s.Hkv,
                                                      s.G, s.NB, tpw);
  return cudaGetLastError();
}

cudaError_t launch_score_blocks(const Shape& s, const uint16_t* q_draft, const float* summ,
                                float* scores, cudaStream_t st, const DeviceInfo& di) {
  const int mt = (s.L * s.G + 15) / 16;
  switch (mt) {
    case 1: return launch_mt<1>(s, q_draft, summ, scores, st, di);
    case 2: return launch_mt<2>(s, q_draft, summ, scores, st, di);
    case 3: return launch_mt<3>(s, q_draft, summ, scores, st, di);
    case 4: return launch_mt<4>(s, q_draft, summ, scores, st, di);
    default: return cudaErrorInvalidValue;  // rejected earlier by validation (L*G <= 64)
  }
}

int score_ctas_per_sm() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, score_kernel<1>, kScoreThreads,
                                                    sizeof(float4) * 8 * 2 * 32) != cudaSuccess)
    return 2;
  return n > 0 ? n : 1;
}

}  // namespace oasis
