// Block-sparse paged GQA decode attention over the working set ("OasisKV:
// Scaling In-Decode KV Cache Beyond HBM with Lookahead Sparse Prefetching",
// Fig. 7 right): for every query head, softmax(scale * q.k) v over the tokens
// of the valid slots of its KV head's working set.
//
// GB300 design
//   - Split: each (request, KV head) unit's S slots are split over P CTAs
//     (P = SMs / units, at most 8), the P CTAs of a unit forming one thread
//     block cluster; with 64 units on 152 SMs that is 2 CTAs (128 SMs), each
//     streaming 64 slots.  Each of the 4 warps of a CTA owns a contiguous
//     quarter of the CTA's slots.  (Equal ranges of one global slot list, one
//     CTA per SM, were measured too: they stream faster but need a merge
//     through global memory whose fences, counters and L2 round trips left a
//     ~6 us tail; the cluster merge below has none of them.)
//   - Each warp streams its valid slots through its own ring of kStages
//     shared-memory stages.  Lane 0 issues TMA tile loads (four 16x64 bf16
//     boxes per slot: K and V, two halves each) with 128-byte swizzle; an
//     mbarrier per stage counts the 8 KiB of each slot.  All waits are bounded.
//   - Tensor cores (mma.sync m16n8k16 bf16, fp32 accumulate) with the GQA
//     group as the N dimension:  S^T = K Q^T  (M = 16 tokens of the slot,
//     K = 128 dims, N = 8 query heads, G of them real) and O^T += V^T P^T
//     (M = 128 dims in 8 tiles, K = 16 tokens, N = heads).  K and V^T
//     fragments come from the swizzled tiles with ldmatrix / ldmatrix.trans;
//     P^T is the S^T accumulator rounded to bf16 and transposed in registers
//     with movmatrix.  Online softmax in base 2, fp32 state (max m, sum l).
//     A step folds two slots (32 tokens) whenever the next one has landed:
//     two independent MMA chains, one shared softmax update.
//   - Merging (online-softmax partials (m, l, O) in fp32): each warp parks its
//     partial in its idle ring; after one CTA barrier the warps fold the four
//     partials head by head; with P = 1 that is the output, otherwise each
//     CTA leaves one partial in its shared memory, and after a cluster barrier
//     the unit's first CTA reads the P partials through distributed shared
//     memory and writes the output.  No workspace, no global partials.
#include <cooperative_groups.h>
#include <cuda.h>

#include "common.cuh"
#include "launch.h"

namespace cg = cooperative_groups;

namespace oasis {

constexpr int kAttnWarps = 4;
constexpr int kAttnThreads = kAttnWarps * 32;
constexpr int kStages = 4;
constexpr int kStageBytes = 2 * kBlockSize * kHeadDim * 2;  // K + V of one slot: 8 KiB
constexpr int kHalfTileBytes = kBlockSize * 64 * 2;         // 16 rows x 128 B
constexpr int kRingBytes = kStages * kStageBytes;
constexpr int kPartStride = 4 + kHeadDim;  // floats per head row: m, l, pad, pad, O[128]
constexpr int kMaxGroup = kMaxAttnGroup;
constexpr int kPartFloats = kMaxGroup * kPartStride;  // one partial (all heads)
constexpr int kMaxSplit = 8;                           // CTAs per unit = cluster size
constexpr int kMinSlotsPerCta = 16;
// rings | the CTA's partial | ring barriers
constexpr size_t kAttnSmem = 1024 + static_cast<size_t>(kAttnWarps) * kRingBytes +
                             static_cast<size_t>(kPartFloats) * sizeof(float) +
                             static_cast<size_t>(kAttnWarps) * kStages * 8;

static int current_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return 148;
  }
  return n;
}

// CTAs per unit: as many as fill the SMs once, at most the cluster limit, and
// at least kMinSlotsPerCta slots each.
static int split_of(const Shape& s, int sm_count) {
  int p = (sm_count > 0 ? sm_count : 148) / s.units();
  if (p > kMaxSplit) p = kMaxSplit;
  if (p > s.S / kMinSlotsPerCta) p = s.S / kMinSlotsPerCta;
  return p < 1 ? 1 : p;
}

// The kernel needs no workspace; the C ABI keeps the argument, and asks for a
// token 256 bytes so that existing callers stay valid.
size_t attn_workspace_bytes(const Shape&) { return 256; }
size_t attn_counter_offset(const Shape&) { return 0; }
size_t attn_counter_bytes(const Shape&) { return 0; }

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

__global__ void __launch_bounds__(kAttnThreads) attn_kernel(
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
    const uint16_t* __restrict__ q, const int32_t* __restrict__ block_of_slot,
    const int32_t* __restrict__ ctx_len, float scale_log2, uint16_t* __restrict__ out, int Hq,
    int Hkv, int G, int S, int NB, int P, uint32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int u = blockIdx.x / P, r = blockIdx.x - u * P;  // unit, rank in its cluster
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
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
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
      tma_load_2d(dst, &tm_k, 0, row, bar);
      tma_load_2d(dst + kHalfTileBytes, &tm_k, 64, row, bar);
      tma_load_2d(dst + 2 * kHalfTileBytes, &tm_v, 0, row, bar);
      tma_load_2d(dst + 3 * kHalfTileBytes, &tm_v, 64, row, bar);
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
  __syncthreads();

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

cudaError_t attn_configure(int) {
  cudaError_t e = cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kAttnSmem));
  if (e == cudaSuccess)  // largest carve-out: the step's other kernels share the SM
    e = cudaFuncSetAttribute(attn_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  return e;
}

int attn_ctas_per_sm() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_kernel, kAttnThreads, kAttnSmem) !=
      cudaSuccess)
    return 1;
  return n > 0 ? n : 1;
}

cudaError_t launch_sparse_decode_attn(const Shape& s, const uint16_t* q,
                                      const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                      const int32_t* block_of_slot, const int32_t* ctx_len,
                                      float scale, uint16_t* out, void*, cudaStream_t st,
                                      const DeviceInfo& di) {
  const int P = split_of(s, di.sm_count > 0 ? di.sm_count : current_sm_count());
  const float scale_log2 = scale * 1.4426950408889634f;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(s.units() * P));
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = kAttnSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(P);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = P > 1 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, attn_kernel, tm_k, tm_v, q, block_of_slot, ctx_len, scale_log2,
                            out, s.Hq, s.Hkv, s.G, s.S, s.NB, P, di.err);
}

}  // namespace oasis
