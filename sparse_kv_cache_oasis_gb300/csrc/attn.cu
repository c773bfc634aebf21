// Block-sparse paged GQA decode attention over the working set ("OasisKV:
// Scaling In-Decode KV Cache Beyond HBM with Lookahead Sparse Prefetching",
// Fig. 7 right): for every query head, softmax(scale * q.k) v over the tokens
// of the valid slots of its KV head's working set.
//
// GB300 design
//   - Work unit: a warp owns kSlotsPerWarp consecutive slots of one
//     (request, KV head); a CTA is kAttnWarps such warps of the same unit.
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
//     with movmatrix.
//   - Online softmax in base 2, fp32 state (max m, sum l) per head column.
//   - Warps of a CTA are merged in shared memory; CTAs of a unit write fp32
//     partials (m, l, O) to the workspace and the last CTA to arrive (atomic
//     counter, reset after use) merges them and writes bf16 out.
#include <cuda.h>

#include "common.cuh"
#include "launch.h"

namespace oasis {

constexpr int kAttnWarps = 4;
constexpr int kAttnThreads = kAttnWarps * 32;
constexpr int kSlotsPerWarp = 8;
constexpr int kStages = 3;
constexpr int kStageBytes = 2 * kBlockSize * kHeadDim * 2;  // K + V of one slot: 8 KiB
constexpr int kHalfTileBytes = kBlockSize * 64 * 2;         // 16 rows x 128 B
constexpr int kPartStride = 4 + kHeadDim;                   // m, l, pad, pad, O[128]
constexpr int kMaxGroup = kMaxAttnGroup;
constexpr size_t kAttnSmem = 1024 + static_cast<size_t>(kAttnWarps) * kStages * kStageBytes +
                             static_cast<size_t>(kAttnWarps) * kStages * 8;

static int ctas_per_unit_of(int S) {
  const int per_cta = kAttnWarps * kSlotsPerWarp;
  return (S + per_cta - 1) / per_cta;
}

size_t attn_workspace_bytes(const Shape& s) {
  const int ncta = ctas_per_unit_of(s.S);
  if (ncta <= 1) return 256;
  const size_t part = static_cast<size_t>(s.units()) * ncta * kMaxGroup * kPartStride * sizeof(float);
  const size_t cnt = static_cast<size_t>(s.units()) * sizeof(int);
  return ((part + 255) / 256) * 256 + ((cnt + 255) / 256) * 256;
}

// Where the per-unit arrival counters sit in the workspace, and their size
// (none when a unit fits one CTA); they must be zero before a call.
size_t attn_counter_offset(const Shape& s) {
  const size_t part = static_cast<size_t>(s.units()) * ctas_per_unit_of(s.S) * kMaxGroup *
                      kPartStride * sizeof(float);
  return ((part + 255) / 256) * 256;
}
size_t attn_counter_bytes(const Shape& s) {
  return ctas_per_unit_of(s.S) > 1 ? static_cast<size_t>(s.units()) * sizeof(int) : 0;
}

// byte offset of 16-byte chunk `chunk` (0..7) of row `row` in a 128B-swizzled 16x64 bf16 box
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__global__ void __launch_bounds__(kAttnThreads) attn_kernel(
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
    const uint16_t* __restrict__ q, const int32_t* __restrict__ block_of_slot,
    const int32_t* __restrict__ ctx_len, float scale_log2, uint16_t* __restrict__ out,
    float* __restrict__ ws_part, int* __restrict__ ws_cnt, int Hq, int Hkv, int G, int S, int NB,
    int ncta, uint32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ int sLast;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int u = blockIdx.x / ncta, cc = blockIdx.x - u * ncta;
  const int b = u / Hkv, h = u - b * Hkv;
  const int slot0 = (cc * kAttnWarps + warp) * kSlotsPerWarp;

  uint8_t* ring = smem + static_cast<size_t>(warp) * kStages * kStageBytes;
  const uint32_t ring_s = smem_u32(ring);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(kAttnWarps) * kStages * kStageBytes) +
                   warp * kStages;
  const uint32_t bar0 = smem_u32(bars);

  // valid slots of this warp's chunk
  int blk_lane = -1;
  if (lane < kSlotsPerWarp && slot0 + lane < S) {
    blk_lane = block_of_slot[static_cast<int64_t>(u) * S + slot0 + lane];
    if (blk_lane >= NB) {
      set_error(err, OASIS_DEVERR_SLOT_RANGE);
      blk_lane = -1;
    }
  }
  const unsigned vmask = __ballot_sync(0xffffffffu, blk_lane >= 0);
  const int nvalid = __popc(vmask);
  const int ctx = ctx_len ? ctx_len[b] : 0x7fffffff;

  if (lane == 0) {
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    for (int st = 0; st < kStages; ++st) mbar_init(bar0 + 8 * st, 1);
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  __syncwarp();

  auto nth_valid = [&](int i) {  // lane index of the i-th valid slot
    unsigned m = vmask;
    for (int k = 0; k < i; ++k) m &= m - 1;
    return __ffs(m) - 1;
  };
  auto issue = [&](int i) {  // lane 0 only
    const int st = i % kStages;
    const int s = slot0 + nth_valid(i);
    const int row = (u * S + s) * kBlockSize;
    const uint32_t dst = ring_s + st * kStageBytes;
    const uint32_t bar = bar0 + 8 * st;
    mbar_arrive_expect_tx(bar, kStageBytes);
    tma_load_2d(dst, &tm_k, 0, row, bar);
    tma_load_2d(dst + kHalfTileBytes, &tm_k, 64, row, bar);
    tma_load_2d(dst + 2 * kHalfTileBytes, &tm_v, 0, row, bar);
    tma_load_2d(dst + 3 * kHalfTileBytes, &tm_v, 64, row, bar);
  };
  int issued = nvalid < kStages ? nvalid : kStages;
  if (lane == 0)
    for (int i = 0; i < issued; ++i) issue(i);

  // Q^T as the B operand: k = dims, n = query head g of this KV head
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

  // per-lane ldmatrix offsets inside a slot's tiles
  const int k_row = (lane & 7) + 8 * ((lane >> 3) & 1);
  const int k_hi = lane >> 4;                 // second 8-dim chunk of the 16-dim k-step
  const int v_row = (lane & 7) + 8 * (lane >> 4);
  const int v_hi = (lane >> 3) & 1;

  bool ok = true;
  int consumed = 0;
#pragma unroll 1
  for (int i = 0; i < nvalid; ++i) {
    const int st = i % kStages;
    const bool done = mbar_wait_bounded(bar0 + 8 * st, (i / kStages) & 1);
    if (!__all_sync(0xffffffffu, done)) {
      ok = false;
      break;
    }
    consumed = i + 1;
    const int blk = __shfl_sync(0xffffffffu, blk_lane, nth_valid(i));
    const uint32_t kt = ring_s + st * kStageBytes;
    const uint32_t vt = kt + 2 * kHalfTileBytes;

    float sacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t a[4];
      const int chunk = 2 * (kk & 3) + k_hi;
      ldmatrix_x4(a, kt + (kk >> 2) * kHalfTileBytes + swz(k_row, chunk));
      mma_bf16_16816(sacc, a, qf[kk][0], qf[kk][1]);
    }
    // tokens at or beyond the context length take no part
    const int tok0 = blk * kBlockSize + g;
    float x0 = tok0 < ctx ? sacc[0] * scale_log2 : -INFINITY;
    float x1 = tok0 < ctx ? sacc[1] * scale_log2 : -INFINITY;
    float x2 = tok0 + 8 < ctx ? sacc[2] * scale_log2 : -INFINITY;
    float x3 = tok0 + 8 < ctx ? sacc[3] * scale_log2 : -INFINITY;
    const float mn_e = fmaxf(m_e, warp_max_xor_g(fmaxf(x0, x2)));
    const float mn_o = fmaxf(m_o, warp_max_xor_g(fmaxf(x1, x3)));
    const float mu_e = mn_e == -INFINITY ? 0.f : mn_e;
    const float mu_o = mn_o == -INFINITY ? 0.f : mn_o;
    const float al_e = exp2f(m_e - mu_e), al_o = exp2f(m_o - mu_o);
    const float p0 = exp2f(x0 - mu_e), p2 = exp2f(x2 - mu_e);
    const float p1 = exp2f(x1 - mu_o), p3 = exp2f(x3 - mu_o);
    l_e = l_e * al_e + p0 + p2;
    l_o = l_o * al_o + p1 + p3;
    m_e = mn_e;
    m_o = mn_o;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      o[mt][0] *= al_e;
      o[mt][1] *= al_o;
      o[mt][2] *= al_e;
      o[mt][3] *= al_o;
    }
    const uint32_t pb0 = movmatrix_trans(pack_bf16x2(p0, p1));  // tokens 0-7
    const uint32_t pb1 = movmatrix_trans(pack_bf16x2(p2, p3));  // tokens 8-15
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      uint32_t a[4];
      const int chunk = 2 * (mt & 3) + v_hi;
      ldmatrix_x4_trans(a, vt + (mt >> 2) * kHalfTileBytes + swz(v_row, chunk));
      mma_bf16_16816(o[mt], a, pb0, pb1);
    }
    __syncwarp();
    if (lane == 0 && issued < nvalid) {
      fence_proxy_async_smem();
      issue(issued);
    }
    issued = __shfl_sync(0xffffffffu, issued + (issued < nvalid ? 1 : 0), 0);
  }
  if (!ok) {
    if (lane == 0) set_error(err, OASIS_DEVERR_WAIT_TIMEOUT);
    // let the copies still in flight land before the shared memory is released
    for (int i = consumed; i < issued; ++i) (void)mbar_wait_bounded(bar0 + 8 * (i % kStages), (i / kStages) & 1);
  }

  l_e = warp_sum_xor_g(l_e);
  l_o = warp_sum_xor_g(l_o);

  // ---- merge the warps of this CTA in shared memory (reuses the rings)
  __syncthreads();
  float* part = reinterpret_cast<float*>(smem);  // [warp][head][kPartStride]
  {
    float* pe = part + (warp * kMaxGroup + 2 * t) * kPartStride;
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
      pe[1] = l_e;
      po[0] = m_o;
      po[1] = l_o;
    }
  }
  __syncthreads();

  const int64_t out_row0 = (static_cast<int64_t>(b) * Hq + h * G);
  for (int it = tid; it < G * 32; it += kAttnThreads) {
    const int hd = it >> 5, dq = it & 31;
    float mw[kAttnWarps], M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) {
      mw[w] = part[(w * kMaxGroup + hd) * kPartStride];
      M = fmaxf(M, mw[w]);
    }
    float Lsum = 0.f;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kAttnWarps; ++w) {
        const float* pw = part + (w * kMaxGroup + hd) * kPartStride;
        const float c = exp2f(mw[w] - M);
        Lsum += c * pw[1];
        const float4 ov = *reinterpret_cast<const float4*>(pw + 4 + 4 * dq);
        O.x += c * ov.x;
        O.y += c * ov.y;
        O.z += c * ov.z;
        O.w += c * ov.w;
      }
    }
    if (ncta == 1) {
      const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
      uint2 pk;
      pk.x = pack_bf16x2(O.x * inv, O.y * inv);
      pk.y = pack_bf16x2(O.z * inv, O.w * inv);
      *reinterpret_cast<uint2*>(out + (out_row0 + hd) * kHeadDim + 4 * dq) = pk;
    } else {
      float* wp = ws_part + ((static_cast<int64_t>(u) * ncta + cc) * kMaxGroup + hd) * kPartStride;
      if (dq == 0) {
        wp[0] = M;
        wp[1] = Lsum;
      }
      *reinterpret_cast<float4*>(wp + 4 + 4 * dq) = O;
    }
  }
  if (ncta == 1) return;

  // ---- the last CTA of this (request, KV head) merges the partials
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const int prev = atomicAdd(ws_cnt + u, 1);
    sLast = prev == ncta - 1;
  }
  __syncthreads();
  if (!sLast) return;
  __threadfence();
  for (int it = tid; it < G * 32; it += kAttnThreads) {
    const int hd = it >> 5, dq = it & 31;
    const float* base = ws_part + (static_cast<int64_t>(u) * ncta * kMaxGroup + hd) * kPartStride;
    float M = -INFINITY;
    for (int c = 0; c < ncta; ++c) M = fmaxf(M, __ldcg(base + c * kMaxGroup * kPartStride));
    float Lsum = 0.f;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
      for (int c = 0; c < ncta; ++c) {
        const float* pc = base + c * kMaxGroup * kPartStride;
        const float w = exp2f(__ldcg(pc) - M);
        Lsum += w * __ldcg(pc + 1);
        const float4 ov = __ldcg(reinterpret_cast<const float4*>(pc + 4 + 4 * dq));
        O.x += w * ov.x;
        O.y += w * ov.y;
        O.z += w * ov.z;
        O.w += w * ov.w;
      }
    }
    const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
    uint2 pk;
    pk.x = pack_bf16x2(O.x * inv, O.y * inv);
    pk.y = pack_bf16x2(O.z * inv, O.w * inv);
    *reinterpret_cast<uint2*>(out + (out_row0 + hd) * kHeadDim + 4 * dq) = pk;
  }
  if (tid == 0) ws_cnt[u] = 0;
}

cudaError_t attn_configure(int) {
  return cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(kAttnSmem));
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
                                      float scale, uint16_t* out, void* workspace,
                                      cudaStream_t st, const DeviceInfo& di) {
  const int ncta = ctas_per_unit_of(s.S);
  float* ws_part = reinterpret_cast<float*>(workspace);
  int* ws_cnt = nullptr;
  if (ncta > 1) {
    const size_t part = static_cast<size_t>(s.units()) * ncta * kMaxGroup * kPartStride * sizeof(float);
    ws_cnt = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(workspace) + ((part + 255) / 256) * 256);
  }
  const float scale_log2 = scale * 1.4426950408889634f;
  attn_kernel<<<s.units() * ncta, kAttnThreads, kAttnSmem, st>>>(
      tm_k, tm_v, q, block_of_slot, ctx_len, scale_log2, out, ws_part, ws_cnt, s.Hq, s.Hkv, s.G,
      s.S, s.NB, ncta, di.err);
  return cudaGetLastError();
}

}  // namespace oasis
