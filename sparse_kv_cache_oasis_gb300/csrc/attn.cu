// Block-sparse paged GQA decode attention over the working set ("OasisKV:
// Scaling In-Decode KV Cache Beyond HBM with Lookahead Sparse Prefetching",
// Fig. 7 right): for every query head, softmax(scale * q.k) v over the tokens
// of the valid slots of its KV head's working set.
//
// GB300 design
//   - Balance: the (request, KV head) units' slots form one list of N = U*S
//     slots.  CTA c owns the contiguous range [c*R, (c+1)*R), R = ceil(N/C),
//     with C = one CTA per SM, so every SM streams the same number of bytes
//     whatever the unit boundaries (and one CTA per SM leaves room for the
//     scoring kernel's CTA beside it).  Each of the 4 warps owns a contiguous
//     quarter of the CTA's range and works on its own from there on.
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
//   - Merging (split slot ranges, online-softmax partials (m, l, O) in fp32):
//     a unit whose slots all lie in one warp's range is finished by that warp
//     from its registers.  Otherwise each warp parks its partial for the unit
//     in its own ring (idle once its copies have landed); after one CTA
//     barrier the warps fold the parked partials, one (unit, head) pair per
//     warp at a time: a unit inside the CTA's range is finished there, a unit
//     crossing the range's edge (at most the first and the last) leaves one
//     CTA partial in the workspace.  Each CTA then adds the number of such a
//     unit's slots it covered to the unit's counter; the CTA that brings it to
//     S folds the unit's CTA partials from L2, writes bf16 out and puts the
//     counter back to zero for the next call.  The workspace is two partials
//     per CTA plus one counter per unit, whatever the shape.
#include <cuda.h>

#include "common.cuh"
#include "launch.h"

namespace oasis {

constexpr int kAttnWarps = 4;
constexpr int kAttnThreads = kAttnWarps * 32;
constexpr int kStages = 3;
constexpr int kStageBytes = 2 * kBlockSize * kHeadDim * 2;  // K + V of one slot: 8 KiB
constexpr int kHalfTileBytes = kBlockSize * 64 * 2;         // 16 rows x 128 B
constexpr int kRingBytes = kStages * kStageBytes;
constexpr int kPartStride = 4 + kHeadDim;  // floats per head row: m, l, pad, pad, O[128]
constexpr int kMaxGroup = kMaxAttnGroup;
constexpr int kPartFloats = kMaxGroup * kPartStride;  // one partial (all heads)
constexpr int kMinSlotsPerCta = 16;
constexpr size_t kAttnSmem = 1024 + static_cast<size_t>(kAttnWarps) * kRingBytes +
                             static_cast<size_t>(kAttnWarps) * kStages * 8;

// ------------------------------------------------------------ static partition
struct Part {
  int N;  // slots in the list (U * S)
  int R;  // slots per CTA range
  __host__ __device__ int start(int c) const { return c * R < N ? c * R : N; }
  __host__ __device__ int quarter() const { return (R + kAttnWarps - 1) / kAttnWarps; }
  // slots of warp w of CTA c: [*lo, *hi)
  __host__ __device__ void warp_range(int c, int w, int* lo, int* hi) const {
    const int b = start(c + 1);
    const int a = start(c) + w * quarter();
    *lo = a < b ? a : b;
    *hi = *lo + quarter() < b ? *lo + quarter() : b;
  }
};

static Part make_part(int64_t N, int sm_count) {
  int64_t c = sm_count > 0 ? sm_count : 148;
  const int64_t cap = (N + kMinSlotsPerCta - 1) / kMinSlotsPerCta;
  if (c > cap) c = cap;
  if (c < 1) c = 1;
  Part pt;
  pt.N = static_cast<int>(N);
  pt.R = static_cast<int>((N + c - 1) / c);
  return pt;
}
static int part_ctas(const Part& pt) { return (pt.N + pt.R - 1) / pt.R; }

static int current_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return 192;  // no device: size for a large part
  }
  return n;
}

// two partials (the units crossing the range's left and right edges) per CTA
static size_t partial_bytes(const Part& pt) {
  return static_cast<size_t>(part_ctas(pt)) * 2 * kPartFloats * sizeof(float);
}
static size_t align256(size_t x) { return (x + 255) / 256 * 256; }

size_t attn_workspace_bytes(const Shape& s) {
  const Part pt = make_part(static_cast<int64_t>(s.units()) * s.S, current_sm_count());
  return align256(partial_bytes(pt)) + align256(static_cast<size_t>(s.units()) * sizeof(int));
}

// Where the per-unit arrival counters sit in the workspace, and their size;
// they must be zero before a call (every call leaves them at zero).
size_t attn_counter_offset(const Shape& s) {
  const Part pt = make_part(static_cast<int64_t>(s.units()) * s.S, current_sm_count());
  return align256(partial_bytes(pt));
}
size_t attn_counter_bytes(const Shape& s) { return static_cast<size_t>(s.units()) * sizeof(int); }

// byte offset of 16-byte chunk `chunk` (0..7) of row `row` in a 128B-swizzled 16x64 bf16 box
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ uint16_t bf16_bits(float x) {
  return static_cast<uint16_t>(pack_bf16x2(x, 0.f) & 0xFFFFu);
}

__global__ void __launch_bounds__(kAttnThreads) attn_kernel(
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
    const uint16_t* __restrict__ q, const int32_t* __restrict__ block_of_slot,
    const int32_t* __restrict__ ctx_len, float scale_log2, uint16_t* __restrict__ out,
    float* __restrict__ ws_part, int* __restrict__ ws_cnt, int Hq, int Hkv, int G, int S, int NB,
    int N, int R, uint32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const Part pt{N, R};
  const int c = blockIdx.x;
  int wa, wb;
  pt.warp_range(c, warp, &wa, &wb);
  const bool has_work = wa < wb;  // a quarter can be empty for tiny ranges

  uint8_t* ring = smem + static_cast<size_t>(warp) * kRingBytes;
  const uint32_t ring_s = smem_u32(ring);
  const uint32_t bars = smem_u32(smem + static_cast<size_t>(kAttnWarps) * kRingBytes);
  const uint32_t bar0 = bars + 8 * kStages * warp;

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
  bool exhausted = !has_work;
  int issued = 0, rj = -1, rb = -1;  // lane k keeps (slot, block) of the entries k mod kStages
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
    if (lane == st) {
      rj = j;
      rb = blk;
    }
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

  // ---- per-unit online-softmax state
  const int uf = wa / S, ul = has_work ? (wb - 1) / S : uf - 1;  // first and last unit of the range
  auto owned = [&](int u) { return u * S >= wa && u * S + S <= wb; };
  const int k_row = (lane & 7) + 8 * ((lane >> 3) & 1);
  const int k_hi = lane >> 4;
  const int v_row = (lane & 7) + 8 * (lane >> 4);
  const int v_hi = (lane >> 3) & 1;
  uint32_t qf[8][2];
  float o[8][4];
  float m_e = -INFINITY, m_o = -INFINITY, l_e = 0.f, l_o = 0.f;
  int cur_u = -1, ctx = 0;

  auto begin_unit = [&](int u) {
    cur_u = u;
    const int b = u / Hkv, h = u - b * Hkv;
    ctx = ctx_len ? ctx_len[b] : 0x7fffffff;
    const uint32_t* q32 = reinterpret_cast<const uint32_t*>(q);
    const int64_t row = (static_cast<int64_t>(b) * Hq + h * G + g) * (kHeadDim / 2);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      qf[kk][0] = g < G ? q32[row + 8 * kk + t] : 0u;
      qf[kk][1] = g < G ? q32[row + 8 * kk + 4 + t] : 0u;
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    m_e = m_o = -INFINITY;
    l_e = l_o = 0.f;
  };
  // A shared first unit is finished mid-stream, while copies are still landing
  // in the ring: its partial is held in registers until the stream is done.
  float ho_[8][4];
  float hm_e = -INFINITY, hm_o = -INFINITY, hl_e = 0.f, hl_o = 0.f;
  bool held = false;
  // parks a partial in slot `side` of this warp's ring (free once the stream is done)
  auto park = [&](int side, const float (&ov)[8][4], float me, float mo, float le, float lo) {
    float* pe = reinterpret_cast<float*>(ring) + side * kPartFloats + (2 * t) * kPartStride;
    float* po = pe + kPartStride;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      pe[4 + 16 * mt + g] = ov[mt][0];
      po[4 + 16 * mt + g] = ov[mt][1];
      pe[4 + 16 * mt + g + 8] = ov[mt][2];
      po[4 + 16 * mt + g + 8] = ov[mt][3];
    }
    if (g == 0) {
      pe[0] = me;
      pe[1] = le;
      po[0] = mo;
      po[1] = lo;
    }
  };
  // Hands on the state of cur_u: the output itself when this warp owns the
  // whole unit, else the warp's partial for it (held, or parked when it is
  // the last unit, which is only finished after the stream).
  auto flush = [&]() {
    const float le = warp_sum_xor_g(l_e), lo_ = warp_sum_xor_g(l_o);
    const int he = 2 * t, hoo = 2 * t + 1;  // the two heads of this lane's columns
    if (owned(cur_u)) {
      const int b = cur_u / Hkv, h = cur_u - b * Hkv;
      const float ie = le > 0.f ? 1.f / le : 0.f, io = lo_ > 0.f ? 1.f / lo_ : 0.f;
      uint16_t* oe = out + (static_cast<int64_t>(b) * Hq + h * G + he) * kHeadDim;
      uint16_t* oo = oe + kHeadDim;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        if (he < G) {
          oe[16 * mt + g] = bf16_bits(o[mt][0] * ie);
          oe[16 * mt + g + 8] = bf16_bits(o[mt][2] * ie);
        }
        if (hoo < G) {
          oo[16 * mt + g] = bf16_bits(o[mt][1] * io);
          oo[16 * mt + g + 8] = bf16_bits(o[mt][3] * io);
        }
      }
    } else if (cur_u == uf) {
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        ho_[mt][0] = o[mt][0];
        ho_[mt][1] = o[mt][1];
        ho_[mt][2] = o[mt][2];
        ho_[mt][3] = o[mt][3];
      }
      hm_e = m_e;
      hm_o = m_o;
      hl_e = le;
      hl_o = lo_;
      held = true;
    } else {
      park(1, o, m_e, m_o, le, lo_);
    }
  };

  bool ok = true;
  int consumed = 0;
  if (has_work) begin_unit(uf);
#pragma unroll 1
  while (consumed < issued) {
    const int st = consumed % kStages;
    const bool done = mbar_wait_bounded(bar0 + 8 * st, (consumed / kStages) & 1);
    if (!__all_sync(0xffffffffu, done)) {
      ok = false;
      break;
    }
    const int j = __shfl_sync(0xffffffffu, rj, st);
    const int blk = __shfl_sync(0xffffffffu, rb, st);
    while (j >= (cur_u + 1) * S) {  // units of this range before j's are complete (possibly empty)
      flush();
      begin_unit(cur_u + 1);
    }
    const uint32_t kt = ring_s + st * kStageBytes;
    const uint32_t vt = kt + 2 * kHalfTileBytes;

    // S^T in two independent accumulator chains (even / odd k-steps)
    float sacc[4] = {0.f, 0.f, 0.f, 0.f}, sac2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < 8; kk += 2) {
      uint32_t af[4], ag[4];
      ldmatrix_x4(af, kt + (kk >> 2) * kHalfTileBytes + swz(k_row, 2 * (kk & 3) + k_hi));
      ldmatrix_x4(ag, kt + ((kk + 1) >> 2) * kHalfTileBytes + swz(k_row, 2 * ((kk + 1) & 3) + k_hi));
      mma_bf16_16816(sacc, af, qf[kk][0], qf[kk][1]);
      mma_bf16_16816(sac2, ag, qf[kk + 1][0], qf[kk + 1][1]);
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) sacc[r] += sac2[r];
    // V^T fragments into registers: the stage is then free and is refilled
    // before the softmax and the O update, one slot's compute earlier
    uint32_t vf[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
      ldmatrix_x4_trans(vf[mt], vt + (mt >> 2) * kHalfTileBytes + swz(v_row, 2 * (mt & 3) + v_hi));
    __syncwarp();
    ++consumed;
    if (!exhausted) try_issue();  // refills the stage just read
    // tokens at or beyond the context length take no part
    const int tok0 = blk * kBlockSize + g;
    const float x0 = tok0 < ctx ? sacc[0] * scale_log2 : -INFINITY;
    const float x1 = tok0 < ctx ? sacc[1] * scale_log2 : -INFINITY;
    const float x2 = tok0 + 8 < ctx ? sacc[2] * scale_log2 : -INFINITY;
    const float x3 = tok0 + 8 < ctx ? sacc[3] * scale_log2 : -INFINITY;
    const float mn_e = fmaxf(m_e, warp_max_xor_g(fmaxf(x0, x2)));
    const float mn_o = fmaxf(m_o, warp_max_xor_g(fmaxf(x1, x3)));
    const float mu_e = mn_e == -INFINITY ? 0.f : mn_e;
    const float mu_o = mn_o == -INFINITY ? 0.f : mn_o;
    const float al_e = ex2_approx(m_e - mu_e), al_o = ex2_approx(m_o - mu_o);
    const float p0 = ex2_approx(x0 - mu_e), p2 = ex2_approx(x2 - mu_e);
    const float p1 = ex2_approx(x1 - mu_o), p3 = ex2_approx(x3 - mu_o);
    l_e = l_e * al_e + p0 + p2;
    l_o = l_o * al_o + p1 + p3;
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
    const uint32_t pb0 = movmatrix_trans(pack_bf16x2(p0, p1));  // tokens 0-7
    const uint32_t pb1 = movmatrix_trans(pack_bf16x2(p2, p3));  // tokens 8-15
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) mma_bf16_16816(o[mt], vf[mt], pb0, pb1);
  }
  if (!ok) {
    if (lane == 0) set_error(err, OASIS_DEVERR_WAIT_TIMEOUT);
    // let the copies still in flight land before the ring is reused or released
    for (int i = consumed; i < issued; ++i)
      (void)mbar_wait_bounded(bar0 + 8 * (i % kStages), (i / kStages) & 1);
  } else if (has_work) {
    // the last unit, and any trailing units without a valid slot (all
    // streaming copies have landed, so the ring is free for the partials)
    while (true) {
      flush();
      if (cur_u >= ul) break;
      begin_unit(cur_u + 1);
    }
    if (held) park(0, ho_, hm_e, hm_o, hl_e, hl_o);
  }

  // ---- CTA level: fold the warps' parked partials unit by unit.  A unit that
  //      lies inside the CTA's range is finished here; one that crosses its
  //      edge (at most the first and the last) leaves one CTA partial in the
  //      workspace.  Tasks are (unit, head) pairs, spread over the warps.
  __syncthreads();
  const int ca = pt.start(c), cb = pt.start(c + 1);
  const int ua = ca / S, ub = (cb - 1) / S;
  const float* rings = reinterpret_cast<const float*>(smem);
  constexpr int kRingFloats = kRingBytes / static_cast<int>(sizeof(float));
  const int nu = ub - ua + 1;
#pragma unroll 1
  for (int task = warp; task < nu * G; task += kAttnWarps) {
    const int u = ua + task / G, hd = task - (task / G) * G;
    const int us = u * S, ue = us + S;
    unsigned wm = 0u;
    bool warp_done = false;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) {
      int lo, hi;
      pt.warp_range(c, w, &lo, &hi);
      if (lo < hi && lo < ue && hi > us) {
        wm |= 1u << w;
        warp_done = lo <= us && ue <= hi;  // that warp owned the unit and wrote it out
      }
    }
    if (warp_done) continue;
    // two-pass fold over at most kAttnWarps partials: max, weights, sums
    float mw[kAttnWarps], lw[kAttnWarps];
    float4 ow[kAttnWarps];
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) {
      mw[w] = -INFINITY;
      lw[w] = 0.f;
      ow[w] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (wm & (1u << w)) {
        int lo, hi;
        pt.warp_range(c, w, &lo, &hi);
        const float* p = rings + w * kRingFloats + (lo / S == u ? 0 : kPartFloats) + hd * kPartStride;
        mw[w] = p[0];
        lw[w] = p[1];
        ow[w] = *reinterpret_cast<const float4*>(p + 4 + 4 * lane);
        mx = fmaxf(mx, mw[w]);
      }
    }
    float ls = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) {
      const float wt = mw[w] == -INFINITY ? 0.f : exp2f(mw[w] - mx);
      ls += wt * lw[w];
      acc.x += wt * ow[w].x;
      acc.y += wt * ow[w].y;
      acc.z += wt * ow[w].z;
      acc.w += wt * ow[w].w;
    }
    if (us >= ca && ue <= cb) {  // inside the CTA's range: final
      const int b = u / Hkv, h = u - b * Hkv;
      const float inv = ls > 0.f ? 1.f / ls : 0.f;
      uint2 pk;
      pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
      pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
      *reinterpret_cast<uint2*>(out + (static_cast<int64_t>(b) * Hq + h * G + hd) * kHeadDim +
                                4 * lane) = pk;
    } else {
      float* q_ = ws_part + (static_cast<int64_t>(c) * 2 + (u == ua ? 0 : 1)) * kPartFloats +
                  hd * kPartStride;
      *reinterpret_cast<float4*>(q_ + 4 + 4 * lane) = acc;
      if (lane == 0) {
        q_[0] = mx;
        q_[1] = ls;
      }
    }
  }

  // ---- count in for the edge units (lanes 0 and 1 of warp 0): each CTA adds
  //      the number of the unit's slots it covered; the CTA that brings the
  //      count to S merges the unit and puts the counter back to zero.  A CTA
  //      counts in even after a timed-out wait (the error word is set) so that
  //      the counters return to zero.
  __shared__ int sMerge[2];
  __threadfence();  // this CTA's partials, before its count
  __syncthreads();
  if (warp == 0) {
    int u = -1;
    if (lane == 0 && ua * S < ca) u = ua;
    if (lane == 1 && (ub + 1) * S > cb && (ub != ua || ua * S >= ca)) u = ub;
    bool last = false;
    if (u >= 0) {
      const int lo = ca > u * S ? ca : u * S;
      const int hi = cb < u * S + S ? cb : u * S + S;
      last = atomicAdd(ws_cnt + u, hi - lo) + (hi - lo) == S;
    }
    if (lane < 2) sMerge[lane] = last ? u : -1;
  }
  __syncthreads();
  const int m0 = sMerge[0], m1 = sMerge[1];
  if (m0 < 0 && m1 < 0) return;
  __threadfence();  // the other CTAs' partials, after their counts
  const int nm = (m0 >= 0) + (m1 >= 0);
#pragma unroll 1
  for (int task = warp; task < nm * G; task += kAttnWarps) {
    const int u = (task / G == 0 && m0 >= 0) ? m0 : m1;
    const int hd = task - (task / G) * G;
    const int b = u / Hkv, h = u - b * Hkv;
    const int c_lo = (u * S) / R, c_hi = (u * S + S - 1) / R;
    float M = -INFINITY, L = 0.f;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    constexpr int kBatch = 8;
#pragma unroll 1
    for (int c0 = c_lo; c0 <= c_hi; c0 += kBatch) {
      float mv[kBatch], lv[kBatch];
      float4 ov[kBatch];
      float bm = M;
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        mv[k] = -INFINITY;
        lv[k] = 0.f;
        ov[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        const int cc = c0 + k;
        if (cc <= c_hi) {
          const float* p = ws_part +
                           (static_cast<int64_t>(cc) * 2 + (pt.start(cc) / S == u ? 0 : 1)) * kPartFloats +
                           hd * kPartStride;
          mv[k] = __ldcg(p);
          lv[k] = __ldcg(p + 1);
          ov[k] = __ldcg(reinterpret_cast<const float4*>(p + 4 + 4 * lane));
        }
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) bm = fmaxf(bm, mv[k]);
      if (bm != -INFINITY) {
        const float r = exp2f(M - bm);  // 0 while M is -inf
        L *= r;
        O.x *= r;
        O.y *= r;
        O.z *= r;
        O.w *= r;
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          const float wt = mv[k] == -INFINITY ? 0.f : exp2f(mv[k] - bm);
          L += wt * lv[k];
          O.x += wt * ov[k].x;
          O.y += wt * ov[k].y;
          O.z += wt * ov[k].z;
          O.w += wt * ov[k].w;
        }
        M = bm;
      }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    uint2 pk;
    pk.x = pack_bf16x2(O.x * inv, O.y * inv);
    pk.y = pack_bf16x2(O.z * inv, O.w * inv);
    *reinterpret_cast<uint2*>(out + (static_cast<int64_t>(b) * Hq + h * G + hd) * kHeadDim +
                              4 * lane) = pk;
  }
  if (threadIdx.x == 0) {
    if (m0 >= 0) ws_cnt[m0] = 0;
    if (m1 >= 0) ws_cnt[m1] = 0;
  }
}

cudaError_t attn_configure(int) {
  cudaError_t e = cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kAttnSmem));
  if (e == cudaSuccess)
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
                                      float scale, uint16_t* out, void* workspace,
                                      cudaStream_t st, const DeviceInfo& di) {
  const Part pt = make_part(static_cast<int64_t>(s.units()) * s.S, di.sm_count);
  float* ws_part = reinterpret_cast<float*>(workspace);
  int* ws_cnt = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(workspace) +
                                       align256(partial_bytes(pt)));
  const float scale_log2 = scale * 1.4426950408889634f;
  attn_kernel<<<part_ctas(pt), kAttnThreads, kAttnSmem, st>>>(
      tm_k, tm_v, q, block_of_slot, ctx_len, scale_log2, out, ws_part, ws_cnt, s.Hq, s.Hkv, s.G,
      s.S, s.NB, pt.N, pt.R, di.err);
  return cudaGetLastError();
}

}  // namespace oasis
