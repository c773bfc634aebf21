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
//   - A unit whose slots all lie in one warp's range is finished by that warp
//     straight from its registers.  A unit shared by several warps (at most
//     the first and the last unit of a warp's range) gets one fp32 partial
//     (m, l, O) per warp; each warp then adds the number of the unit's slots it
//     covered to the unit's counter, and the warp that brings it to S merges
//     the unit: bulk copies of the partials into its own (now idle) ring, then
//     per head a warp-wide max, one weight per partial and a weighted sum of
//     the O columns in shared memory, bf16 out, and the counter back to zero
//     for the next call.  The workspace is therefore two partials
//     per warp plus one counter per unit, whatever the shape.
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
                             static_cast<size_t>(kAttnWarps) * (kStages + 1) * 8;

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

// two partials (first and last unit of the range) per warp
static size_t partial_bytes(const Part& pt) {
  return static_cast<size_t>(part_ctas(pt)) * kAttnWarps * 2 * kPartFloats * sizeof(float);
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
  if (wa >= wb) return;  // an empty quarter (tiny ranges only): nothing to stream or count

  uint8_t* ring = smem + static_cast<size_t>(warp) * kRingBytes;
  const uint32_t ring_s = smem_u32(ring);
  const uint32_t bars = smem_u32(smem + static_cast<size_t>(kAttnWarps) * kRingBytes);
  const uint32_t bar0 = bars + 8 * kStages * warp;
  const uint32_t mbar = bars + 8 * kStages * kAttnWarps + 8 * warp;  // merge copies

  if (lane == 0) {
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    for (int st = 0; st < kStages; ++st) mbar_init(bar0 + 8 * st, 1);
    mbar_init(mbar, 1);
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  __syncwarp();

  // ---- issue cursor over the valid slots of [wa, wb), 32 slots at a time
  int cur_base = wa - 32, cur_blk = -1;
  unsigned cur_mask = 0u;
  bool exhausted = false;
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
  const int uf = wa / S, ul = (wb - 1) / S;  // first and last unit of the range
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
  // Hands on the state of cur_u: the output itself when this warp owns the
  // whole unit, else the warp's partial for it.
  auto flush = [&]() {
    const float le = warp_sum_xor_g(l_e), lo_ = warp_sum_xor_g(l_o);
    const int he = 2 * t, ho = 2 * t + 1;  // the two heads of this lane's columns
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
        if (ho < G) {
          oo[16 * mt + g] = bf16_bits(o[mt][1] * io);
          oo[16 * mt + g + 8] = bf16_bits(o[mt][3] * io);
        }
      }
      return;
    }
    const int side = cur_u == uf ? 0 : 1;
    float* pe = ws_part + ((static_cast<int64_t>(c) * kAttnWarps + warp) * 2 + side) * kPartFloats +
                he * kPartStride;
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
      po[1] = lo_;
    }
  };

  bool ok = true;
  int consumed = 0;
  begin_unit(uf);
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
    const int u = j / S;
    while (cur_u < u) {  // units of this range before u are complete (possibly empty)
      flush();
      begin_unit(cur_u + 1);
    }
    const uint32_t kt = ring_s + st * kStageBytes;
    const uint32_t vt = kt + 2 * kHalfTileBytes;

    float sacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t af[4];
      ldmatrix_x4(af, kt + (kk >> 2) * kHalfTileBytes + swz(k_row, 2 * (kk & 3) + k_hi));
      mma_bf16_16816(sacc, af, qf[kk][0], qf[kk][1]);
    }
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
      uint32_t af[4];
      ldmatrix_x4_trans(af, vt + (mt >> 2) * kHalfTileBytes + swz(v_row, 2 * (mt & 3) + v_hi));
      mma_bf16_16816(o[mt], af, pb0, pb1);
    }
    __syncwarp();
    ++consumed;
    if (!exhausted) try_issue();  // refills the stage just consumed
  }
  if (!ok) {
    if (lane == 0) set_error(err, OASIS_DEVERR_WAIT_TIMEOUT);
    // let the copies still in flight land before the ring is reused or released
    for (int i = consumed; i < issued; ++i)
      (void)mbar_wait_bounded(bar0 + 8 * (i % kStages), (i / kStages) & 1);
  } else {
    while (true) {  // the last unit, and any trailing units without a valid slot
      flush();
      if (cur_u >= ul) break;
      begin_unit(cur_u + 1);
    }
  }

  // ---- count in for the shared first and last units (lanes 0 and 1).  A warp
  //      counts in even after a timed-out wait (the error word is set) so that
  //      the counters return to zero.
  __threadfence();  // the partials above, before the count
  __syncwarp();
  int mine = -1;
  bool last = false;
  if ((lane == 0 && !owned(uf)) || (lane == 1 && ul != uf && !owned(ul))) {
    mine = lane == 0 ? uf : ul;
    const int lo = wa > mine * S ? wa : mine * S;
    const int hi = wb < mine * S + S ? wb : mine * S + S;
    last = atomicAdd(ws_cnt + mine, hi - lo) + (hi - lo) == S;
  }
  unsigned lm = __ballot_sync(0xffffffffu, last);
  int phase = 0;
#pragma unroll 1
  while (lm) {
    const int u = __shfl_sync(0xffffffffu, mine, __ffs(lm) - 1);
    lm &= lm - 1;
    __threadfence();          // the other warps' partials, after their counts
    fence_proxy_async_all();  // ... and before the bulk copies read them
    const int b = u / Hkv, h = u - b * Hkv;
    const int ua = u * S, ub = ua + S;
    const int c_lo = ua / R, c_hi = (ub - 1) / R;
    const int ncand = (c_hi - c_lo + 1) * kAttnWarps;
    // Rounds of bulk copies into this warp's ring: slot 0 keeps the merge of
    // the rounds before (in the partial's own format), the other slots take
    // new partials.  Each round folds all its slots at once: a warp-wide max
    // and weight per partial, then a weighted sum of the O columns.
    const int row_floats = G * kPartStride;
    const uint32_t row_bytes = static_cast<uint32_t>(row_floats) * sizeof(float);
    const int cap = kRingBytes / static_cast<int>(row_bytes);  // partials the ring holds (>= 5)
    float* ring_f = reinterpret_cast<float*>(ring);
    int held = 0;
    bool merge_ok = true;
#pragma unroll 1
    for (int base = 0; base < ncand && merge_ok; base += 32) {
      // lane i looks at candidate warp base+i of the CTAs meeting the unit
      const int i = base + lane;
      int off = -1;
      if (i < ncand) {
        const int cc = c_lo + i / kAttnWarps, ww = i % kAttnWarps;
        int lo, hi;
        pt.warp_range(cc, ww, &lo, &hi);
        if (lo < hi && lo < ub && hi > ua)
          off = ((cc * kAttnWarps + ww) * 2 + (lo / S == u ? 0 : 1)) * kPartFloats;
      }
      unsigned cm = __ballot_sync(0xffffffffu, off >= 0);
#pragma unroll 1
      while (cm) {
        unsigned take = 0u;
        int n = 0;
        for (unsigned rest = cm; rest && n < cap - held; rest &= rest - 1, ++n)
          take |= rest & (~rest + 1u);
        cm &= ~take;
        __syncwarp();
        if (lane == 0) {
          fence_proxy_async_smem();  // earlier reads of the ring, before the copies
          mbar_arrive_expect_tx(mbar, n * row_bytes);
        }
        __syncwarp();
        if (take & (1u << lane)) {
          const int rank = __popc(take & ((1u << lane) - 1u));
          bulk_load(ring_s + (held + rank) * row_bytes, ws_part + off, row_bytes, mbar);
        }
        const bool landed = mbar_wait_bounded(mbar, phase & 1);
        ++phase;
        if (!__all_sync(0xffffffffu, landed)) {
          if (lane == 0) set_error(err, OASIS_DEVERR_WAIT_TIMEOUT);
          (void)mbar_wait_bounded(mbar, (phase - 1) & 1);
          merge_ok = false;
          break;
        }
        const int nn = held + n;
        const bool final_round = cm == 0u && base + 32 >= ncand;
#pragma unroll 1
        for (int hd = 0; hd < G; ++hd) {
          float* ph = ring_f + hd * kPartStride;  // row hd of slot 0; slot k is k * row_floats on
          const float mk = lane < nn ? ph[lane * row_floats] : -INFINITY;
          const float lk = lane < nn ? ph[lane * row_floats + 1] : 0.f;
          float mx = mk;
#pragma unroll
          for (int d = 16; d > 0; d >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, d));
          const float wk = mk == -INFINITY ? 0.f : exp2f(mk - mx);
          float ls = wk * lk;
#pragma unroll
          for (int d = 16; d > 0; d >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, d);
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int k = 0; k < nn; ++k) {
            const float w = __shfl_sync(0xffffffffu, wk, k);
            const float4 v = *reinterpret_cast<const float4*>(ph + k * row_floats + 4 + 4 * lane);
            acc.x += w * v.x;
            acc.y += w * v.y;
            acc.z += w * v.z;
            acc.w += w * v.w;
          }
          if (final_round) {
            const float inv = ls > 0.f ? 1.f / ls : 0.f;
            uint2 pk;
            pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
            pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
            *reinterpret_cast<uint2*>(out + (static_cast<int64_t>(b) * Hq + h * G + hd) * kHeadDim +
                                      4 * lane) = pk;
          } else {  // each lane rewrites only what it alone read: its column and, lane 0, m and l
            *reinterpret_cast<float4*>(ph + 4 + 4 * lane) = acc;
            if (lane == 0) {
              ph[0] = mx;
              ph[1] = ls;
            }
          }
        }
        held = 1;
      }
    }
    if (lane == 0) ws_cnt[u] = 0;
  }
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
