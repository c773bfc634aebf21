// Body of the look-ahead block scoring ("OasisKV: Scaling In-Decode KV Cache
// Beyond HBM with Lookahead Sparse Prefetching", Fig. 7 right), shared by the
// scoring kernel and the fused attention + scoring kernel.  The design is
// described in score.cu.
#pragma once

#include "common.cuh"

namespace oasis {


constexpr int kScoreStages = 3;  // tiles of 8 blocks in flight per warp (4 KiB each)

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

// Words per (16-row tile, k-step pair) of a lane's A fragments: with one row
// tile they are kept unpacked (eight tf32 bit patterns, 64 instructions per
// tile fewer), with more as the four bf16-pair words they come in, unpacked at
// each use (to bound the registers).
__host__ __device__ constexpr int frag_words(int mt) { return mt == 1 ? 8 : 4; }

// Compressed-key kinds: the fp32 mean key of a block, or its elementwise max
// and min keys (bf16, [max(D) | min(D)] per block).  Both are 512 bytes per
// block, so the streaming below is the same; only the contraction differs.
constexpr int kSummMean = 0;
constexpr int kSummMinMax = 1;
constexpr int kMaxMinMaxTiles = 2;  // min/max scoring keeps every A fragment unpacked

// Words per (16-row tile, chunk p) of a lane's A fragments.
__host__ __device__ constexpr int q_words(int mt, int kind) {
  return kind == kSummMinMax ? 8 : frag_words(mt);
}

// Max over the valid query rows of a tile's accumulators (rows >= M are
// padding), then the 8 block scores are written out.
template <int MT>
__device__ __forceinline__ void score_store(const float (&acc)[MT][4], int g, int t, int M, int n0,
                                            int NB, int64_t out_off, float* out) {
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

// Min/max scores of 8 blocks (one tile).  Per dimension
//   max(q*mn, q*mx) = max(q, 0)*mx + min(q, 0)*mn     (mx >= mn),
// so a block's score is one 256-long dot product of [q+ | q-] with
// [mx | mn]: every operand is a bf16 value (a sign mask splits q), the
// products are exact in fp32, and bf16 MMAs (m16n8k16, fp32 accumulation)
// take it.  Lane (g, t)'s 16 bytes of chunk p hold k-steps 2p and 2p+1.
template <int MT>
__device__ __forceinline__ void score_tile_minmax(const float4 (&v)[8],
                                                  const uint32_t (&wq)[MT][8][8], int g, int t,
                                                  int M, int n0, int NB, int64_t out_off,
                                                  float* out) {
  float acc[MT][4], acc1[MT][4], acc2[MT][4], acc3[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[mt][r] = acc1[mt][r] = acc2[mt][r] = acc3[mt][r] = 0.f;
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    const uint32_t x = __float_as_uint(v[p].x), y = __float_as_uint(v[p].y);
    const uint32_t z = __float_as_uint(v[p].z), w = __float_as_uint(v[p].w);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      // rows g and g+8: words 0-3 of the chunk are wq[..][0-3] and [4-7]
      const uint32_t a[4] = {wq[mt][p][0], wq[mt][p][4], wq[mt][p][1], wq[mt][p][5]};
      const uint32_t c[4] = {wq[mt][p][2], wq[mt][p][6], wq[mt][p][3], wq[mt][p][7]};
      mma_bf16_16816((p & 1) ? acc2[mt] : acc[mt], a, x, y);   // k-step 2p
      mma_bf16_16816((p & 1) ? acc3[mt] : acc1[mt], c, z, w);  // k-step 2p+1
    }
  }
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[mt][r] = (acc[mt][r] + acc2[mt][r]) + (acc1[mt][r] + acc3[mt][r]);
  score_store<MT>(acc, g, t, M, n0, NB, out_off, out);
}

// Scores of 8 blocks (one tile) from their summaries in v; writes them out.
template <int MT>
__device__ __forceinline__ void score_tile(const float4 (&v)[8],
                                           const uint32_t (&wq)[MT][8][frag_words(MT)], int g,
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
      uint32_t a0, a1, a2, a3, c0, c1, c2, c3;
      if constexpr (MT == 1) {
        a0 = wq[mt][p][0]; a1 = wq[mt][p][1]; a2 = wq[mt][p][2]; a3 = wq[mt][p][3];
        c0 = wq[mt][p][4]; c1 = wq[mt][p][5]; c2 = wq[mt][p][6]; c3 = wq[mt][p][7];
      } else {
        a0 = wq[mt][p][0] << 16; a1 = wq[mt][p][2] << 16;
        a2 = wq[mt][p][0] & 0xFFFF0000u; a3 = wq[mt][p][2] & 0xFFFF0000u;
        c0 = wq[mt][p][1] << 16; c1 = wq[mt][p][3] << 16;
        c2 = wq[mt][p][1] & 0xFFFF0000u; c3 = wq[mt][p][3] & 0xFFFF0000u;
      }
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
  score_store<MT>(acc, g, t, M, n0, NB, out_off, out);
}

// One warp's share of the scoring: the contiguous tiles [w_lo, w_lo + tpw) of
// the global tile list (8 blocks per tile), streamed through `ring`
// (kScoreStages x 8 x 32 float4 of shared memory owned by this warp).  `summ`
// holds one 512-byte row (32 float4) of compressed key per block, of kind KIND.
template <int MT, int KIND = kSummMean>
__device__ __forceinline__ void score_warp_range(const uint16_t* __restrict__ q_draft,
                                                 const float4* __restrict__ summ,
                                                 float* __restrict__ scores, int L, int Hq, int Hkv,
                                                 int G, int NB, int w_lo, int tpw, float4* ring,
                                                 int lane) {
  static_assert(KIND == kSummMean || MT <= kMaxMinMaxTiles, "min/max row tiles");
  const int g = lane >> 2, t = lane & 3;
  const uint32_t ring_s = smem_u32(ring);
  const int M = L * G;
  const int ntiles = (NB + 7) >> 3;
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
        const float4* src = summ + (static_cast<int64_t>(u) * NB + blk) * 32 + t;
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

  // A fragments of unit u, rows 16mt+g (+8) (rows >= L*G are padding and stay
  // zero).  Mean: dims 16p+4t..+3 as bf16 pairs.  Min/max: chunk p < 4 holds
  // q+ of dims 8(t+4p)..+7 and chunk p+4 q- of the same dims.
  uint32_t wq[MT][8][q_words(MT, KIND)];
  auto load_q = [&](int u) {
    const int b = u / Hkv, h = u - b * Hkv;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int row = 16 * mt + g + 8 * half;
        const int l = row / G, gq = row - l * G;
        const uint16_t* qrow = q_draft + ((static_cast<int64_t>(b) * L + l) * Hq + h * G + gq) * kHeadDim;
        if constexpr (KIND == kSummMinMax) {
          const uint4* src = reinterpret_cast<const uint4*>(qrow + 8 * t);
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            const uint4 w = row < M ? __ldg(src + 4 * p) : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t neg = ((ws[i] & 0x80008000u) >> 15) * 0xFFFFu;  // negative halves
              wq[mt][p][4 * half + i] = ws[i] & ~neg;
              wq[mt][p + 4][4 * half + i] = ws[i] & neg;
            }
          }
        } else {
          const uint2* src = reinterpret_cast<const uint2*>(qrow + 4 * t);
#pragma unroll
          for (int p = 0; p < 8; ++p) {
            const uint2 w = row < M ? __ldg(src + 4 * p) : make_uint2(0u, 0u);
            if constexpr (MT == 1) {
              wq[mt][p][half] = w.x << 16;
              wq[mt][p][2 + half] = w.x & 0xFFFF0000u;
              wq[mt][p][4 + half] = w.y << 16;
              wq[mt][p][6 + half] = w.y & 0xFFFF0000u;
            } else {
              wq[mt][p][2 * half] = w.x;
              wq[mt][p][2 * half + 1] = w.y;
            }
          }
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
    if constexpr (KIND == kSummMinMax)
      score_tile_minmax<MT>(v, wq, g, t, M, (tile - u * ntiles) * 8, NB, out_off,
                            scores + out_off);
    else
      score_tile<MT>(v, wq, g, t, M, (tile - u * ntiles) * 8, NB, out_off, scores + out_off);
  }
  cp_async_wait<0>();
}

}  // namespace oasis
