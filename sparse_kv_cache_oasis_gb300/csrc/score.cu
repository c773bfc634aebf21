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
// form one list of T tiles; CTA c (one per SM) takes the contiguous range
// [c*Rt, (c+1)*Rt) and each warp a contiguous eighth of it, so every SM
// streams the same number of bytes whatever NB and the unit count, a warp
// reloads its query fragments only where its tiles cross into the next unit,
// and one CTA per SM leaves room for the attention kernel's CTA beside it.
#include "common.cuh"
#include "launch.h"

namespace oasis {

constexpr int kScoreThreads = 192;
constexpr int kScoreWarps = kScoreThreads / 32;
constexpr int kScoreStages = 3;  // tiles of 8 blocks in flight per warp (4 KiB each)
constexpr int kMinTilesPerCta = 16;

// 16-byte asynchronous global->shared copy (bypasses L1) and its group fences.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

constexpr uint32_t kTf32Mask = 0xFFFFE000u;  // sign, exponent, 10 mantissa bits

// Words per (16-row tile, k-step pair) of a lane's A fragments: the four
// bf16-pair words they come in, unpacked at each use.  (Keeping them unpacked
// saves ~64 instructions per tile but needs ~30 more registers per thread,
// and the kernel must leave room in each SM sub-partition's register file for
// the attention and top-K kernels that run beside it.)
__host__ __device__ constexpr int frag_words(int) { return 4; }

// Scores of 8 blocks (one tile) from their summaries in v; writes them out.
template <int MT>
__device__ __forceinline__ void score_tile(const float4 (&v)[8], const uint32_t (&wq)[MT][8][frag_words(MT)], int lane, int g,
                                           int t, int M, int n0, int NB, int64_t out_off,
                                           float* out) {
  // four independent accumulator chains (hi/lo x even/odd k-step) keep the
  // MMA dependency chains short; they are summed at the end
  float acc[MT][4], acc1[MT][4], acc2[MT][4], acc3[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[mt][r] = acc1[mt][r] = acc2[mt][r] = acc3[mt][r] = 0.f;
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    const uint32_t hx = __float_as_uint(v[p].x) & kTf32Mask, hy = __float_as_uint(v[p].y) & kTf32Mask;
    const uint32_t hz = __float_as_uint(v[p].z) & kTf32Mask, hw = __float_as_uint(v[p].w) & kTf32Mask;
    const uint32_t lx = __float_as_uint(v[p].x - __uint_as_float(hx));
    const uint32_t ly = __float_as_uint(v[p].y - __uint_as_float(hy));
    const uint32_t lz = __float_as_uint(v[p].z - __uint_as_float(hz));
    const uint32_t lw = __float_as_uint(v[p].w - __uint_as_float(hw));
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      // rows g and g+8, dims 16p+4t..+3 as bf16 pairs -> tf32 bit patterns
      const uint32_t a0 = wq[mt][p][0] << 16, a1 = wq[mt][p][2] << 16;
      const uint32_t a2 = wq[mt][p][0] & 0xFFFF0000u, a3 = wq[mt][p][2] & 0xFFFF0000u;
      const uint32_t c0 = wq[mt][p][1] << 16, c1 = wq[mt][p][3] << 16;
      const uint32_t c2 = wq[mt][p][1] & 0xFFFF0000u, c3 = wq[mt][p][3] & 0xFFFF0000u;
      mma_tf32_1688(acc[mt], a0, a1, a2, a3, hx, hy);   // k-step 2p, hi
      mma_tf32_1688(acc1[mt], a0, a1, a2, a3, lx, ly);  // k-step 2p, lo
      mma_tf32_1688(acc2[mt], c0, c1, c2, c3, hz, hw);  // k-step 2p+1, hi
      mma_tf32_1688(acc3[mt], c0, c1, c2, c3, lz, lw);  // k-step 2p+1, lo
    }
  }
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[mt][r] = (acc[mt][r] + acc2[mt][r]) + (acc1[mt][r] + acc3[mt][r]);
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
    // a float2 store needs an even element offset (out_off + col); odd NB breaks it
    const bool even = ((out_off + col) & 1) == 0;
    if (col + 1 < NB && even) {
      __stcs(reinterpret_cast<float2*>(out + col), make_float2(m0, m1));
    } else {
      if (col < NB) out[col] = m0;
      if (col + 1 < NB) out[col + 1] = m1;
    }
  }
}

template <int MT>
__global__ void __launch_bounds__(kScoreThreads) score_kernel(
    const uint16_t* __restrict__ q_draft, const float* __restrict__ summ,
    float* __restrict__ scores, int L, int Hq, int Hkv, int G, int NB, int T, int Rt) {
  // shared memory: one ring per warp of kScoreStages tiles, each [p][lane]
  // float4 (a lane reads back what it copied)
  extern __shared__ float4 smem4[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  float4* ring = smem4 + warp * kScoreStages * 8 * 32;
  const uint32_t ring_s = smem_u32(ring);
  const int M = L * G;
  const int ntiles = (NB + 7) >> 3;
  const int t_lo = blockIdx.x * Rt;
  const int t_hi = t_lo + Rt < T ? t_lo + Rt : T;
  // this warp's tiles: the contiguous [w_lo, w_lo + tpw)
  const int qw = (t_hi - t_lo + kScoreWarps - 1) / kScoreWarps;
  const int w_lo = t_lo + warp * qw < t_hi ? t_lo + warp * qw : t_hi;
  const int tpw = w_lo + qw < t_hi ? qw : t_hi - w_lo;

  int u_iss = w_lo / ntiles;  // unit of the last tile issued (tiles only move forward)
  // copies tile i of this warp into stage i % kScoreStages (one commit group per call)
  auto issue = [&](int i) {
    if (i < tpw) {
      const int tile = w_lo + i;
      while (tile >= (u_iss + 1) * ntiles) ++u_iss;
      const int u = u_iss;
      const int blk = (tile - u * ntiles) * 8 + g;
      const int st = i % kScoreStages;
      if (blk < NB) {
        const float4* src = reinterpret_cast<const float4*>(
                                summ + (static_cast<int64_t>(u) * NB + blk) * kHeadDim) + t;
#pragma unroll
        for (int p = 0; p < 8; ++p)
          cp_async16(ring_s + static_cast<uint32_t>(((st * 8 + p) * 32 + lane) * 16), src + 4 * p);
      } else {
#pragma unroll
        for (int p = 0; p < 8; ++p) ring[(st * 8 + p) * 32 + lane] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    cp_async_commit();
  };
#pragma unroll
  for (int i = 0; i < kScoreStages - 1; ++i) issue(i);

  // A fragments of unit u: rows 16mt+g (+8), dims 16p+4t..+3, as bf16 pairs
  // (rows >= L*G are padding and stay zero)
  uint32_t wq[MT][8][frag_words(MT)];
  auto load_q = [&](int u) {
    const int b = u / Hkv, h = u - b * Hkv;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int row = 16 * mt + g + 8 * half;
        const int l = row / G, gq = row - l * G;
        const uint2* src = reinterpret_cast<const uint2*>(
            q_draft + ((static_cast<int64_t>(b) * L + l) * Hq + h * G + gq) * kHeadDim + 4 * t);
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          const uint2 w = row < M ? __ldg(src + 4 * p) : make_uint2(0u, 0u);
          wq[mt][p][2 * half] = w.x;
          wq[mt][p][2 * half + 1] = w.y;
        }
      }
    }
  };
  int u_use = -1;  // unit whose fragments are loaded
#pragma unroll 1
  for (int i = 0; i < tpw; ++i) {
    const int tile = w_lo + i;
    int u = u_use < 0 ? tile / ntiles : u_use;
    while (tile >= (u + 1) * ntiles) ++u;
    if (u != u_use) {
      load_q(u);
      u_use = u;
    }
    issue(i + kScoreStages - 1);
    cp_async_wait<kScoreStages - 1>();  // tile i has landed (this lane's copies)
    const int st = i % kScoreStages;
    float4 v[8];
#pragma unroll
    for (int p = 0; p < 8; ++p) v[p] = ring[(st * 8 + p) * 32 + lane];
    const int64_t out_off = static_cast<int64_t>(u) * NB;
    score_tile<MT>(v, wq, lane, g, t, M, (tile - u * ntiles) * 8, NB, out_off, scores + out_off);
  }
  cp_async_wait<0>();
}

static size_t score_smem_bytes(int) {
  return sizeof(float4) * static_cast<size_t>(kScoreWarps) * kScoreStages * 8 * 32;
}

template <int MT>
static cudaError_t launch_mt(const Shape& s, const uint16_t* q_draft, const float* summ,
                             float* scores, cudaStream_t st, const DeviceInfo& di) {
  // one CTA per SM over equal contiguous tile ranges
  const int ntiles = (s.NB + 7) / 8;
  const int64_t T = static_cast<int64_t>(s.units()) * ntiles;
  int64_t C = di.sm_count > 0 ? di.sm_count : 148;
  const int64_t cap = (T + kMinTilesPerCta - 1) / kMinTilesPerCta;
  if (C > cap) C = cap;
  if (C < 1) C = 1;
  const int64_t Rt = (T + C - 1) / C;
  const int64_t grid = (T + Rt - 1) / Rt;
  score_kernel<MT><<<static_cast<unsigned>(grid), kScoreThreads, score_smem_bytes(MT), st>>>(
      q_draft, summ, scores, s.L, s.Hq, s.Hkv, s.G, s.NB, static_cast<int>(T), static_cast<int>(Rt));
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

template <int MT>
static cudaError_t score_configure_mt() {
  cudaError_t e = cudaFuncSetAttribute(score_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(score_smem_bytes(MT)));
  if (e == cudaSuccess)  // largest carve-out: the step's other kernels share the SM
    e = cudaFuncSetAttribute(score_kernel<MT>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  return e;
}

cudaError_t score_configure() {
  cudaError_t e = score_configure_mt<1>();
  if (e == cudaSuccess) e = score_configure_mt<2>();
  if (e == cudaSuccess) e = score_configure_mt<3>();
  if (e == cudaSuccess) e = score_configure_mt<4>();
  return e;
}

int score_ctas_per_sm() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, score_kernel<1>, kScoreThreads,
                                                    score_smem_bytes(1)) != cudaSuccess)
    return 2;
  return n > 0 ? n : 1;
}

}  // namespace oasis
