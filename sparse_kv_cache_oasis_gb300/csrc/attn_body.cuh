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
constexpr int kMaxRowTiles = 3;  // query rows per CTA: at most 8 per tile, 24 in all
constexpr int kMaxSplit = 8;     // CTAs per unit = cluster size
constexpr int kMinSlotsPerCta = 16;
// floats of one partial (m, l, O of every row of NT row tiles)
__host__ __device__ constexpr int part_floats(int nt) { return 8 * nt * kPartStride; }
// rings | the CTA's partial | ring barriers (plus 1 KiB for the alignment)
__host__ __device__ constexpr size_t attn_smem_body(int nt) {
  return static_cast<size_t>(kAttnWarps) * kRingBytes +
         static_cast<size_t>(part_floats(nt)) * sizeof(float) +
         static_cast<size_t>(kAttnWarps) * kStages * 8;
}
constexpr size_t kAttnSmemBody = attn_smem_body(1);  // one row tile: up to 8 query heads
constexpr size_t kAttnSmem = 1024 + kAttnSmemBody;
static_assert(kMaxAttnGroup <= 8, "one row tile holds a GQA group");
static_assert(part_floats(kMaxRowTiles) * sizeof(float) <= kRingBytes,
              "a warp's partial fits its ring");

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

// The query rows of one CTA: row r (0 <= r < the CTA's row count) has its
// query at query(r) and its output at output(r), D bf16 values each.
struct GroupRows {  // the G query heads h*G + r of KV head h of request b
  const uint16_t* q;
  uint16_t* out;
  int64_t base;  // (b*Hq + h*G) * D
  __device__ __forceinline__ const uint16_t* query(int r) const {
    return q + base + static_cast<int64_t>(r) * kHeadDim;
  }
  __device__ __forceinline__ uint16_t* output(int r) const {
    return out + base + static_cast<int64_t>(r) * kHeadDim;
  }
};

// Joint rows of one unit: row0 + r = l*G + g is query head h*G + g of token
// l of request b, l = 0 the decoded token (q), l >= 1 draft token l-1
// (q_draft); the output has the rows of all 1 + L tokens.
struct JointRows {
  const uint16_t* q;
  const uint16_t* q_draft;
  uint16_t* out;
  int b, h, Hq, G, L, row0;
  __device__ __forceinline__ void split(int r, int* l, int* head) const {
    const int rr = row0 + r;
    *l = rr / G;
    *head = h * G + (rr - *l * G);
  }
  __device__ __forceinline__ const uint16_t* query(int r) const {
    int l, hd;
    split(r, &l, &hd);
    return l == 0 ? q + (static_cast<int64_t>(b) * Hq + hd) * kHeadDim
                  : q_draft + ((static_cast<int64_t>(b) * L + (l - 1)) * Hq + hd) * kHeadDim;
  }
  __device__ __forceinline__ uint16_t* output(int r) const {
    int l, hd;
    split(r, &l, &hd);
    return out + ((static_cast<int64_t>(b) * (L + 1) + l) * Hq + hd) * kHeadDim;
  }
};

// One CTA's share of the attention: unit u, rank r of the P CTAs of its
// cluster, query rows 0..n_rows-1 of `rows` (n_rows <= 8*NT) as the N
// dimension of the MMAs in NT tiles of 8 columns; `smem` is 1 KiB aligned and
// attn_smem_body<NT>() bytes long, `warp` is 0..3, and `cta_bar()`
// synchronises the four attention warps of the CTA.
template <int NT, typename Rows, typename CtaBar>
__device__ __forceinline__ void attn_cta(
    const CUtensorMap* tm_k, const CUtensorMap* tm_v, const Rows& rows, int n_rows,
    const int32_t* __restrict__ block_of_slot, const int32_t* __restrict__ ctx_len,
    float scale_log2, int Hkv, int S, int NB, int P, uint32_t* err, uint8_t* smem, int u, int r,
    int warp, int lane, CtaBar cta_bar) {
  static_assert(NT >= 1 && NT <= kMaxRowTiles, "row tiles");
  // two slots per step where one row tile leaves the registers for it
  constexpr bool kPairSteps = NT == 1;
  const int g = lane >> 2, t = lane & 3;
  const int b = u / Hkv;
  // this CTA's slots [ca, cb) of the unit, this warp's quarter [wa, wb)
  const int ca = u * S + (r * S) / P, cb = u * S + ((r + 1) * S) / P;
  const int qn = (cb - ca + kAttnWarps - 1) / kAttnWarps;
  const int wa = ca + warp * qn < cb ? ca + warp * qn : cb;
  const int wb = wa + qn < cb ? wa + qn : cb;

  uint8_t* ring = smem + static_cast<size_t>(warp) * kRingBytes;
  const uint32_t ring_s = smem_u32(ring);
  float* cta_part = reinterpret_cast<float*>(smem + static_cast<size_t>(kAttnWarps) * kRingBytes);
  const uint32_t bar0 = smem_u32(cta_part + part_floats(NT)) + 8 * kStages * warp;

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

  // ---- the query fragments: column g of tile nt is row 8*nt + g (rows at or
  //      beyond n_rows are zero padding)
  const int k_row = (lane & 7) + 8 * ((lane >> 3) & 1);
  const int k_hi = lane >> 4;
  const int v_row = (lane & 7) + 8 * (lane >> 4);
  const int v_hi = (lane >> 3) & 1;
  const int ctx = ctx_len ? ctx_len[b] : 0x7fffffff;
  uint32_t qf[8][NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int c = 8 * nt + g;
    const uint32_t* q32 = c < n_rows ? reinterpret_cast<const uint32_t*>(rows.query(c)) : nullptr;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      qf[kk][nt][0] = q32 ? q32[8 * kk + t] : 0u;
      qf[kk][nt][1] = q32 ? q32[8 * kk + 4 + t] : 0u;
    }
  }
  float o[8][NT][4];
  float m_e[NT], m_o[NT], l_e[NT], l_o[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.f;
    m_e[nt] = m_o[nt] = -INFINITY;
    l_e[nt] = l_o[nt] = 0.f;
  }

  // One step folds one slot, or two slots (32 tokens) when the next one has
  // been issued: the two S^T products and O^T updates are independent MMA
  // chains, and the softmax bookkeeping (running max, rescale) is shared.
  // K and V^T fragments are loaded once per step and serve every row tile.
  auto step = [&](auto pair_tag, uint32_t kA, int bA, uint32_t kB, int bB) {
    constexpr bool kPair = decltype(pair_tag)::value;
    const uint32_t vA = kA + 2 * kHalfTileBytes, vB = kB + 2 * kHalfTileBytes;
    float sa[NT][4], sb[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) sa[nt][i] = sb[nt][i] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint32_t off = (kk >> 2) * kHalfTileBytes + swz(k_row, 2 * (kk & 3) + k_hi);
      uint32_t af[4];
      ldmatrix_x4(af, kA + off);
      if constexpr (kPair) {
        uint32_t bf[4];
        ldmatrix_x4(bf, kB + off);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(sb[nt], bf, qf[kk][nt][0], qf[kk][nt][1]);
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(sa[nt], af, qf[kk][nt][0], qf[kk][nt][1]);
    }
    // tokens at or beyond the context length take no part
    const int ta = bA * kBlockSize + g, tb = bB * kBlockSize + g;
    const bool inA0 = ta < ctx, inA8 = ta + 8 < ctx;
    const bool inB0 = kPair && tb < ctx, inB8 = kPair && tb + 8 < ctx;
    float al_e[NT], al_o[NT];
    uint32_t pk_a0[NT], pk_a1[NT], pk_b0[NT], pk_b1[NT];  // P rounded to bf16, token-major
    bool moved = false;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float a0 = inA0 ? sa[nt][0] * scale_log2 : -INFINITY;
      const float a1 = inA0 ? sa[nt][1] * scale_log2 : -INFINITY;
      const float a2 = inA8 ? sa[nt][2] * scale_log2 : -INFINITY;
      const float a3 = inA8 ? sa[nt][3] * scale_log2 : -INFINITY;
      const float b0 = inB0 ? sb[nt][0] * scale_log2 : -INFINITY;
      const float b1 = inB0 ? sb[nt][1] * scale_log2 : -INFINITY;
      const float b2 = inB8 ? sb[nt][2] * scale_log2 : -INFINITY;
      const float b3 = inB8 ? sb[nt][3] * scale_log2 : -INFINITY;
      const float mn_e = fmaxf(m_e[nt], warp_max_xor_g(fmaxf(fmaxf(a0, a2), fmaxf(b0, b2))));
      const float mn_o = fmaxf(m_o[nt], warp_max_xor_g(fmaxf(fmaxf(a1, a3), fmaxf(b1, b3))));
      const float mu_e = mn_e == -INFINITY ? 0.f : mn_e;
      const float mu_o = mn_o == -INFINITY ? 0.f : mn_o;
      al_e[nt] = ex2_approx(m_e[nt] - mu_e);
      al_o[nt] = ex2_approx(m_o[nt] - mu_o);
      const float pa0 = ex2_approx(a0 - mu_e), pa2 = ex2_approx(a2 - mu_e);
      const float pa1 = ex2_approx(a1 - mu_o), pa3 = ex2_approx(a3 - mu_o);
      float pb0 = 0.f, pb1 = 0.f, pb2 = 0.f, pb3 = 0.f;
      if constexpr (kPair) {
        pb0 = ex2_approx(b0 - mu_e);
        pb2 = ex2_approx(b2 - mu_e);
        pb1 = ex2_approx(b1 - mu_o);
        pb3 = ex2_approx(b3 - mu_o);
      }
      l_e[nt] = l_e[nt] * al_e[nt] + ((pa0 + pa2) + (pb0 + pb2));
      l_o[nt] = l_o[nt] * al_o[nt] + ((pa1 + pa3) + (pb1 + pb3));
      m_e[nt] = mn_e;
      m_o[nt] = mn_o;
      moved = moved || al_e[nt] != 1.f || al_o[nt] != 1.f;
      pk_a0[nt] = pack_bf16x2(pa0, pa1);
      pk_a1[nt] = pack_bf16x2(pa2, pa3);
      pk_b0[nt] = pack_bf16x2(pb0, pb1);
      pk_b1[nt] = pack_bf16x2(pb2, pb3);
    }
    if (__any_sync(0xffffffffu, moved)) {  // a running max moved
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          o[mt][nt][0] *= al_e[nt];
          o[mt][nt][1] *= al_o[nt];
          o[mt][nt][2] *= al_e[nt];
          o[mt][nt][3] *= al_o[nt];
        }
    }
    uint32_t qa0[NT], qa1[NT], qb0[NT], qb1[NT];  // P^T fragments
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      qa0[nt] = movmatrix_trans(pk_a0[nt]);  // tokens 0-7
      qa1[nt] = movmatrix_trans(pk_a1[nt]);  // tokens 8-15
      qb0[nt] = qb1[nt] = 0u;
      if constexpr (kPair) {
        qb0[nt] = movmatrix_trans(pk_b0[nt]);
        qb1[nt] = movmatrix_trans(pk_b1[nt]);
      }
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const uint32_t off = (mt >> 2) * kHalfTileBytes + swz(v_row, 2 * (mt & 3) + v_hi);
      uint32_t af[4];
      ldmatrix_x4_trans(af, vA + off);
      if constexpr (kPair) {
        uint32_t bf[4];
        ldmatrix_x4_trans(bf, vB + off);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(o[mt][nt], bf, qb0[nt], qb1[nt]);
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(o[mt][nt], af, qa0[nt], qa1[nt]);
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
    const bool pair = kPairSteps && consumed + 1 < issued;
    if (pair) {
      if (!__all_sync(0xffffffffu,
                      mbar_wait_bounded(bar0 + 8 * stB, ((consumed + 1) / kStages) & 1))) {
        ok = false;
        break;
      }
      if constexpr (kPairSteps)
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
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const float le = warp_sum_xor_g(l_e[nt]), lo = warp_sum_xor_g(l_o[nt]);
    float* pe = reinterpret_cast<float*>(ring) + (8 * nt + 2 * t) * kPartStride;
    float* po = pe + kPartStride;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      pe[4 + 16 * mt + g] = o[mt][nt][0];
      po[4 + 16 * mt + g] = o[mt][nt][1];
      pe[4 + 16 * mt + g + 8] = o[mt][nt][2];
      po[4 + 16 * mt + g + 8] = o[mt][nt][3];
    }
    if (g == 0) {
      pe[0] = m_e[nt];
      pe[1] = le;
      po[0] = m_o[nt];
      po[1] = lo;
    }
  }
  cta_bar();

  // ---- fold the four warps' partials, a row per warp at a time: the output
  //      itself when the CTA holds the whole unit, else the CTA's partial
  const float* rings = reinterpret_cast<const float*>(smem);
  constexpr int kRingFloats = kRingBytes / static_cast<int>(sizeof(float));
  auto write_out = [&](int hd, float l, float4 v) {
    const float inv = l > 0.f ? 1.f / l : 0.f;
    uint2 pk;
    pk.x = pack_bf16x2(v.x * inv, v.y * inv);
    pk.y = pack_bf16x2(v.z * inv, v.w * inv);
    *reinterpret_cast<uint2*>(rows.output(hd) + 4 * lane) = pk;
  };
  for (int hd = warp; hd < n_rows; hd += kAttnWarps) {
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
    for (int hd = warp; hd < n_rows; hd += kAttnWarps) {
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
