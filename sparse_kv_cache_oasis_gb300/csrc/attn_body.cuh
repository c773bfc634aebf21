// Body of the block-sparse paged GQA decode attention ("OasisKV: Scaling
// In-Decode KV Cache Beyond HBM with Lookahead Sparse Prefetching", Fig. 7
// right), shared by the attention kernel and the fused attention + scoring
// kernel.  The design is described in attn.cu.
#pragma once

#include <cooperative_groups.h>
#include <cuda.h>

#include "common.cuh"

namespace oasis {

namespace cg = cooperative_groups;


constexpr int kAttnWarps = 4;
constexpr int kAttnThreads = kAttnWarps * 32;
constexpr int kStages = 3;
constexpr int kStageBytes = 2 * kBlockSize * kHeadDim * 2;  // K + V of one slot: 8 KiB
constexpr int kHalfTileBytes = kBlockSize * 64 * 2;         // 16 rows x 128 B
constexpr int kRingBytes = kStages * kStageBytes;
constexpr int kPartStride = 4 + kHeadDim;  // floats per head row: m, l, pad, pad, O[128]
constexpr int kMaxGroup = kMaxAttnGroup;
constexpr int kPartFloats = kMaxGroup * kPartStride;  // one partial (all heads)
constexpr int kMaxSplit = 8;                           // CTAs per unit = cluster size
constexpr int kMinSlotsPerCta = 16;
// rings | the CTA's partial | ring barriers (plus 1 KiB for the alignment)
constexpr size_t kAttnSmemBody = static_cast<size_t>(kAttnWarps) * kRingBytes +
                                 static_cast<size_t>(kPartFloats) * sizeof(float) +
                                 static_cast<size_t>(kAttnWarps) * kStages * 8;
constexpr size_t kAttnSmem = 1024 + kAttnSmemBody;

// byte offset of 16-byte chunk `chunk` (0..7) of row `row` in a 128B-swizzled 16x64 bf16 box
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

template <bool V>
struct Bool {
  static constexpr bool value = V;
};

// Folds n partials (the head row at ptr(k) of each) into (m, l, O[4*lane..+3]):
// two passes, the max first, then the weighted sums.
template <typename Ptr>
__device__ __forceinline__ void fold_partials(int n, Ptr ptr, int lane, float* m_out, float* l_out,
                                              float4* o_out) {
  float mx = -INFINITY;
  for (int k = 0; k < n; ++k) mx = fmaxf(mx, ptr(k)[0]);
  float l = 0.f;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k = 0; k < n; ++k) {
    const float* p = ptr(k);
    const float m = p[0];
    if (m == -INFINITY) continue;  // an empty partial
    const float w = exp2f(m - mx);
    const float4 v = *reinterpret_cast<const float4*>(p + 4 + 4 * lane);
    l += w * p[1];
    o.x += w * v.x;
    o.y += w * v.y;
    o.z += w * v.z;
    o.w += w * v.w;
  }
  *m_out = mx;
  *l_out = l;
  *o_out = o;
}

// One CTA's share of the attention: unit u, rank r of the P CTAs of its
// cluster; `smem` is 1 KiB aligned and kAttnSmemBody bytes long, `warp` is
// 0..3, and `cta_bar()` synchronises the four attention warps of the CTA.
template <typename CtaBar>
__device__ __forceinline__ void attn_cta(
    const CUtensorMap* tm_k, const CUtensorMap* tm_v, const uint16_t* __restrict__ q,
    const int32_t* __restrict__ block_of_slot, const int32_t* __restrict__ ctx_len,
    float scale_log2, uint16_t* __restrict__ out, int Hq, int Hkv, int G, int S, int NB, int P,
    uint32_t* err, uint8_t* smem, int u, int r, int warp, int lane, CtaBar cta_bar) {
  const int g = lane >> 2, t = lane & 3;
  const int b = u / Hkv, h = u - b * Hkv;
  // this CTA's slots [ca, cb) of the unit, this warp's quarter [wa, wb)
  const int ca = u * S + (r * S) / P, cb = u * S + ((r + 1) * S) / P;
  const int qn = (cb - ca + kAttnWarps - 1) / kAttnWarps;
  const int wa = ca + warp * qn < cb ? ca + warp * qn : cb;
  const int wb = wa + qn < cb ? wa + qn : cb;

  uint8_t* ring = smem + static_cast<size_t>(warp) * kRingBytes;
  const uint32_t ring_s = smem_u32(ring);
  float* cta_part = reinterpret_cast<float*>(smem + static_cast<size_t>(kAttnWarps) * kRingBytes);
  const uint32_t bar0 = smem_u32(cta_part + kPartFloats) + 8 * kStages * warp;

  if (lane == 0) {
    prefetch_tmap(tm_k);
    prefetch_tmap(tm_v);
    for (int st = 0; st < kStages; ++st) mbar_init(bar0 + 8 * st, 1);
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  __syncwarp();

  // ---- issue cursor over the valid slots of [wa, wb), 32 slots at a time
  int cur_base = wa - 32, cur_blk = -1;
  unsigned cur_mask = 0u;
  bool exhausted = wa >= wb;
  int issued = 0, rb = -1;  // lane k keeps the block of the entries k mod kStages
  auto try_issue = [&]() {
    while (cur_mask == 0u) {
      cur_base += 32;
      if (cur_base >= wb) {
        exhausted = true;
        return;
      }
      const int j = cur_base + lane;
      cur_blk = -1;
      if (j < wb) {
        cur_blk = block_of_slot[j];
        if (cur_blk >= NB) {
          set_error(err, OASIS_DEVERR_SLOT_RANGE);
          cur_blk = -1;
        }
      }
      cur_mask = __ballot_sync(0xffffffffu, cur_blk >= 0);
    }
    const int l = __ffs(cur_mask) - 1;
    cur_mask &= cur_mask - 1;
    const int j = cur_base + l;
    const int blk = __shfl_sync(0xffffffffu, cur_blk, l);
    const int st = issued % kStages;
    if (lane == st) rb = blk;
    if (lane == 0) {
      const uint32_t dst = ring_s + st * kStageBytes;
      const uint32_t bar = bar0 + 8 * st;
      const int row = j * kBlockSize;
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(bar, kStageBytes);
      tma_load_2d(dst, tm_k, 0, row, bar);
      tma_load_2d(dst + kHalfTileBytes, tm_k, 64, row, bar);
      tma_load_2d(dst + 2 * kHalfTileBytes, tm_v, 0, row, bar);
      tma_load_2d(dst + 3 * kHalfTileBytes, tm_v, 64, row, bar);
    }
    ++issued;
  };
  while (issued < kStages && !exhausted) try_issue();

  // ---- the unit's queries (rows h*G + g of request b; rows >= G are padding)
  const int k_row = (lane & 7) + 8 * ((lane >> 3) & 1);
  const int k_hi = lane >> 4;
  const int v_row = (lane & 7) + 8 * (lane >> 4);
  const int v_hi = (lane >> 3) & 1;
  const int ctx = ctx_len ? ctx_len[b] : 0x7fffffff;
  uint32_t qf[8][2];
  {
    const uint32_t* q32 = reinterpret_cast<const uint32_t*>(q);
    const int64_t row = (static_cast<int64_t>(b) * Hq + h * G + g) * (kHeadDim / 2);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      qf[kk][0] = g < G ? q32[row + 8 * kk + t] : 0u;
      qf[kk][1] = g < G ? q32[row + 8 * kk + 4 + t] : 0u;
    }
  }
  float o[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  float m_e = -INFINITY, m_o = -INFINITY, l_e = 0.f, l_o = 0.f;

  // One step folds one slot, or two slots (32 tokens) when the next one has
  // been issued: the two S^T products and O^T updates are independent MMA
  // chains, and the softmax bookkeeping (running max, rescale) is shared.
  auto step = [&](auto pair_tag, uint32_t kA, int bA, uint32_t kB, int bB) {
    constexpr bool kPair = decltype(pair_tag)::value;
    const uint32_t vA = kA + 2 * kHalfTileBytes, vB = kB + 2 * kHalfTileBytes;
    float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint32_t off = (kk >> 2) * kHalfTileBytes + swz(k_row, 2 * (kk & 3) + k_hi);
      uint32_t af[4];
      ldmatrix_x4(af, kA + off);
      if constexpr (kPair) {
        uint32_t bf[4];
        ldmatrix_x4(bf, kB + off);
        mma_bf16_16816(sb, bf, qf[kk][0], qf[kk][1]);
      }
      mma_bf16_16816(sa, af, qf[kk][0], qf[kk][1]);
    }
    // tokens at or beyond the context length take no part
    const int ta = bA * kBlockSize + g, tb = bB * kBlockSize + g;
    const float a0 = ta < ctx ? sa[0] * scale_log2 : -INFINITY;
    const float a1 = ta < ctx ? sa[1] * scale_log2 : -INFINITY;
    const float a2 = ta + 8 < ctx ? sa[2] * scale_log2 : -INFINITY;
    const float a3 = ta + 8 < ctx ? sa[3] * scale_log2 : -INFINITY;
    const float b0 = kPair && tb < ctx ? sb[0] * scale_log2 : -INFINITY;
    const float b1 = kPair && tb < ctx ? sb[1] * scale_log2 : -INFINITY;
    const float b2 = kPair && tb + 8 < ctx ? sb[2] * scale_log2 : -INFINITY;
    const float b3 = kPair && tb + 8 < ctx ? sb[3] * scale_log2 : -INFINITY;
    const float mn_e = fmaxf(m_e, warp_max_xor_g(fmaxf(fmaxf(a0, a2), fmaxf(b0, b2))));
    const float mn_o = fmaxf(m_o, warp_max_xor_g(fmaxf(fmaxf(a1, a3), fmaxf(b1, b3))));
    const float mu_e = mn_e == -INFINITY ? 0.f : mn_e;
    const float mu_o = mn_o == -INFINITY ? 0.f : mn_o;
    const float al_e = ex2_approx(m_e - mu_e), al_o = ex2_approx(m_o - mu_o);
    const float pa0 = ex2_approx(a0 - mu_e), pa2 = ex2_approx(a2 - mu_e);
    const float pa1 = ex2_approx(a1 - mu_o), pa3 = ex2_approx(a3 - mu_o);
    float pb0 = 0.f, pb1 = 0.f, pb2 = 0.f, pb3 = 0.f;
    if constexpr (kPair) {
      pb0 = ex2_approx(b0 - mu_e);
      pb2 = ex2_approx(b2 - mu_e);
      pb1 = ex2_approx(b1 - mu_o);
      pb3 = ex2_approx(b3 - mu_o);
    }
    l_e = l_e * al_e + ((pa0 + pa2) + (pb0 + pb2));
    l_o = l_o * al_o + ((pa1 + pa3) + (pb1 + pb3));
    m_e = mn_e;
    m_o = mn_o;
    if (__any_sync(0xffffffffu, al_e != 1.f || al_o != 1.f)) {  // a running max moved
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        o[mt][0] *= al_e;
        o[mt][1] *= al_o;
        o[mt][2] *= al_e;
        o[mt][3] *= al_o;
      }
    }
    const uint32_t qa0 = movmatrix_trans(pack_bf16x2(pa0, pa1));  // tokens 0-7
    const uint32_t qa1 = movmatrix_trans(pack_bf16x2(pa2, pa3));  // tokens 8-15
    uint32_t qb0 = 0u, qb1 = 0u;
    if constexpr (kPair) {
      qb0 = movmatrix_trans(pack_bf16x2(pb0, pb1));
      qb1 = movmatrix_trans(pack_bf16x2(pb2, pb3));
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const uint32_t off = (mt >> 2) * kHalfTileBytes + swz(v_row, 2 * (mt & 3) + v_hi);
      uint32_t af[4];
      ldmatrix_x4_trans(af, vA + off);
      if constexpr (kPair) {
        uint32_t bf[4];
        ldmatrix_x4_trans(bf, vB + off);
        mma_bf16_16816(o[mt], bf, qb0, qb1);
      }
      mma_bf16_16816(o[mt], af, qa0, qa1);
    }
  };

  bool ok = true;
  int consumed = 0;
#pragma unroll 1
  while (consumed < issued) {
    const int stA = consumed % kStages;
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar0 + 8 * stA, (consumed / kStages) & 1))) {
      ok = false;
      break;
    }
    const int bA = __shfl_sync(0xffffffffu, rb, stA);
    const int stB = (consumed + 1) % kStages;
    const int bB = __shfl_sync(0xffffffffu, rb, stB);
    const bool pair = consumed + 1 < issued;
    if (pair) {
      if (!__all_sync(0xffffffffu,
                      mbar_wait_bounded(bar0 + 8 * stB, ((consumed + 1) / kStages) & 1))) {
        ok = false;
        break;
      }
      step(Bool<true>(), ring_s + stA * kStageBytes, bA, ring_s + stB * kStageBytes, bB);
    } else {
      step(Bool<false>(), ring_s + stA * kStageBytes, bA, 0u, 0);
    }
    __syncwarp();
    consumed += pair ? 2 : 1;
    if (!exhausted) try_issue();  // refill the stages just consumed
    if (pair && !exhausted) try_issue();
  }
  if (!ok) {
    if (lane == 0) set_error(err, OASIS_DEVERR_WAIT_TIMEOUT);
    // let the copies still in flight land before the ring is reused or released
    for (int i = consumed; i < issued; ++i)
      (void)mbar_wait_bounded(bar0 + 8 * (i % kStages), (i / kStages) & 1);
  }

  // ---- park this warp's partial (every warp, an empty one too) in its ring
  {
    const float le = warp_sum_xor_g(l_e), lo = warp_sum_xor_g(l_o);
    float* pe = reinterpret_cast<float*>(ring) + (2 * t) * kPartStride;
    float* po = pe + kPartStride;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      pe[4 + 16 * mt + g] = o[mt][0];
      po[4 + 16 * mt + g] = o[mt][1];
      pe[4 + 16 * mt + g + 8] = o[mt][2];
      po[4 + 16 * mt + g + 8] = o[mt][3];
    }
    if (g == 0) {
      pe[0] = m_e;
      pe[1] = le;
      po[0] = m_o;
      po[1] = lo;
    }
  }
  cta_bar();

  // ---- fold the four warps' partials, a head per warp at a time: the output
  //      itself when the CTA holds the whole unit, else the CTA's partial
  const float* rings = reinterpret_cast<const float*>(smem);
  constexpr int kRingFloats = kRingBytes / static_cast<int>(sizeof(float));
  uint16_t* out_u = out + (static_cast<int64_t>(b) * Hq + h * G) * kHeadDim;
  auto write_out = [&](int hd, float l, float4 v) {
    const float inv = l > 0.f ? 1.f / l : 0.f;
    uint2 pk;
    pk.x = pack_bf16x2(v.x * inv, v.y * inv);
    pk.y = pack_bf16x2(v.z * inv, v.w * inv);
    *reinterpret_cast<uint2*>(out_u + hd * kHeadDim + 4 * lane) = pk;
  };
  for (int hd = warp; hd < G; hd += kAttnWarps) {
    float m, l;
    float4 v;
    fold_partials(
        kAttnWarps, [&](int k) { return rings + k * kRingFloats + hd * kPartStride; }, lane, &m,
        &l, &v);
    if (P == 1) {
      write_out(hd, l, v);
    } else {
      float* cp = cta_part + hd * kPartStride;
      *reinterpret_cast<float4*>(cp + 4 + 4 * lane) = v;
      if (lane == 0) {
        cp[0] = m;
        cp[1] = l;
      }
    }
  }
  if (P == 1) return;

  // ---- the unit's first CTA folds the cluster's partials through distributed
  //      shared memory; the second barrier keeps every CTA's shared memory
  //      alive until it has been read
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  if (r == 0) {
    for (int hd = warp; hd < G; hd += kAttnWarps) {
      float m, l;
      float4 v;
      fold_partials(
          P,
          [&](int k) {
            return static_cast<const float*>(cluster.map_shared_rank(cta_part, k)) +
                   hd * kPartStride;
          },
          lane, &m, &l, &v);
      write_out(hd, l, v);
    }
  }
  cluster.sync();
}

}  // namespace oasis
