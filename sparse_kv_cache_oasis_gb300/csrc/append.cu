// Decode-time append: the new token of every request joins the caches
// ("OasisKV: Scaling In-Decode KV Cache Beyond HBM with Lookahead Sparse
// Prefetching", Fig. 8: the decode loop advances one token per step).  For
// request b the token sits at p = ctx_len[b], row t = p % bs of block
// j = p / bs, for every KV head:
//   1. the full cache in (mapped) host memory gets the K and V rows;
//   2. the working set keeps the newest block: if block j is not resident it
//      takes the lowest empty slot, else the slot of the least recently used
//      resident block that is not forced in the grown context (sink and local
//      window of j + 1 blocks), ties by lower block id; the slot's rows
//      0..t-1 come in from the full cache and row t gets the token;
//   3. ctx_len[b] = p + 1.
// Then, off the attention's critical path, the refresh recomputes the
// compressed keys of each context's newest block over its rows inside the
// context (the mean: double sum in row order, divided by t + 1, rounded once;
// the max and min rows when given).
//
// GB300 design: the append is latency-bound and sits between a layer's QKV
// and its attention, so it does no arithmetic: one warp per KV head (lane l
// owns dims 4l..4l+3, 8-byte accesses), each in a one-warp CTA, the request's
// Hkv CTAs forming a thread-block cluster (Hkv <= 8; more heads share one CTA
// per request).  The context length is read by every warp before one cluster
// barrier and advanced after it.  The victim search is a warp-wide minimum
// over 64-bit keys (class, last use, block id); rows copied into a newly
// taken slot are loaded eight at a time before they are stored.  The
// attention that follows is a programmatic dependent: it may launch while
// this grid runs and waits for its results.  The exact mean needs
// double arithmetic, which GB300 runs at a small fraction of its fp32 rate
// (one CTA per request with the mean inside took ~8 us); the refresh runs it
// one warp per SM on a stream beside the attention.
#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"

namespace oasis {

namespace cg = cooperative_groups;

constexpr int kMaxSpreadHeads = 8;  // portable cluster size

__device__ __forceinline__ void bf16x4_to_f32(uint2 v, float (&f)[4], uint16_t (&bits)[4]) {
  bits[0] = static_cast<uint16_t>(v.x & 0xFFFFu);
  bits[1] = static_cast<uint16_t>(v.x >> 16);
  bits[2] = static_cast<uint16_t>(v.y & 0xFFFFu);
  bits[3] = static_cast<uint16_t>(v.y >> 16);
#pragma unroll
  for (int i = 0; i < 4; ++i) f[i] = __uint_as_float(static_cast<uint32_t>(bits[i]) << 16);
}

// SPREAD: one CTA (one warp) per KV head, the request's Hkv CTAs forming a
// thread-block cluster; else one CTA per request with a warp per head.
template <bool SPREAD>
__global__ void __launch_bounds__(SPREAD ? 32 : 1024) append_kernel(
    const uint16_t* __restrict__ k_new, const uint16_t* __restrict__ v_new,
    int32_t* __restrict__ ctx_len, const int32_t* __restrict__ clock, int32_t step,
    uint16_t* __restrict__ host_k, uint16_t* __restrict__ host_v,
    int32_t* __restrict__ slot_of_block, int32_t* __restrict__ block_of_slot,
    int32_t* __restrict__ last_used, uint16_t* __restrict__ pool_k, uint16_t* __restrict__ pool_v,
    int Hkv, int NB, int S, int sink, int local, uint32_t* err) {
  const int b = SPREAD ? blockIdx.x / Hkv : blockIdx.x;
  const int h = SPREAD ? blockIdx.x - b * Hkv : threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // the attention that follows may launch now (it waits for this grid's results)
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  const int64_t u = static_cast<int64_t>(b) * Hkv + h;
  // the token's rows do not depend on the context length: load them first
  const uint2 kn = reinterpret_cast<const uint2*>(k_new + u * kHeadDim)[lane];
  const uint2 vn = reinterpret_cast<const uint2*>(v_new + u * kHeadDim)[lane];
  const int p = ctx_len[b];
  const bool full = p < 0 || static_cast<int64_t>(p) >= static_cast<int64_t>(NB) * kBlockSize;
  if (!full) {
    const int j = p / kBlockSize, t = p - j * kBlockSize;
    const int64_t row0 = (u * NB + j) * kBlockSize;  // token 0 of block j in the full cache
    int32_t* sob = slot_of_block + u * NB;
    int32_t* bos = block_of_slot + u * S;
    int32_t* lu = last_used + u * S;
    int s = sob[j];
    // 1. the full cache
    reinterpret_cast<uint2*>(host_k + (row0 + t) * kHeadDim)[lane] = kn;
    reinterpret_cast<uint2*>(host_v + (row0 + t) * kHeadDim)[lane] = vn;
    // 2. the working set
    bool fill = false;  // the slot is new to the block: rows 0..t-1 go in too
    if (s >= S) {       // a broken map: leave the working set alone
      if (lane == 0) set_error(err, OASIS_DEVERR_PLAN_STATE);
      s = -1;
    } else if (s < 0) {
      const int n = j + 1;
      const int sink_end = sink < n ? sink : n;
      const int win_begin = n - local > 0 ? n - local : 0;
      unsigned long long best = ~0ull;
      int best_slot = -1;
#pragma unroll 4
      for (int q = lane; q < S; q += 32) {
        const int blk = bos[q];
        const int last = lu[q];
        unsigned long long key = ~0ull;
        if (blk < 0) {
          key = static_cast<unsigned long long>(q);  // empty slots first, lowest index
        } else if (blk < NB && !(blk < sink_end || (blk >= win_begin && blk < n))) {
          // an unforced resident block: least recently used, then lower id
          const uint32_t lb = static_cast<uint32_t>(last) ^ 0x80000000u;  // signed order
          key = (1ull << 63) | (static_cast<unsigned long long>(lb) << 31) |
                static_cast<unsigned long long>(blk);
        }
        if (key < best) {
          best = key;
          best_slot = q;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long ok = __shfl_xor_sync(0xffffffffu, best, o);
        const int os = __shfl_xor_sync(0xffffffffu, best_slot, o);
        if (ok < best) {
          best = ok;
          best_slot = os;
        }
      }
      if (best_slot < 0) {
        if (lane == 0) set_error(err, OASIS_DEVERR_NO_SLOT);
      } else {
        s = best_slot;
        fill = true;
        if (lane == 0) {
          const int victim = bos[s];
          if (victim >= 0) sob[victim] = -1;
          bos[s] = j;
          sob[j] = s;
          lu[s] = clock ? clock[u] : step;
        }
      }
    }
    if (s >= 0) {
      uint16_t* pk = pool_k + (u * S + s) * kBlockSize * kHeadDim;
      uint16_t* pv = pool_v + (u * S + s) * kBlockSize * kHeadDim;
      reinterpret_cast<uint2*>(pk + t * kHeadDim)[lane] = kn;
      reinterpret_cast<uint2*>(pv + t * kHeadDim)[lane] = vn;
      // a newly taken slot: rows 0..t-1 from the cache, eight rows in flight at a time
      for (int r0 = 0; fill && r0 < t; r0 += 8) {
        uint2 rk[8], rv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (r0 + i < t) {
            rk[i] = reinterpret_cast<const uint2*>(host_k + (row0 + r0 + i) * kHeadDim)[lane];
            rv[i] = reinterpret_cast<const uint2*>(host_v + (row0 + r0 + i) * kHeadDim)[lane];
          }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (r0 + i < t) {
            reinterpret_cast<uint2*>(pk + (r0 + i) * kHeadDim)[lane] = rk[i];
            reinterpret_cast<uint2*>(pv + (r0 + i) * kHeadDim)[lane] = rv[i];
          }
        }
      }
    }
  }
  // every warp of the request has read the old length before it advances
  if constexpr (SPREAD)
    cg::this_cluster().sync();
  else
    __syncthreads();
  if (threadIdx.x == 0 && h == 0) {
    if (full)
      set_error(err, OASIS_DEVERR_CTX_FULL);
    else
      ctx_len[b] = p + 1;
  }
}

cudaError_t launch_append_kv(const Shape& s, const uint16_t* k_new, const uint16_t* v_new,
                             int32_t* ctx_len, const int32_t* clock, int32_t step,
                             uint16_t* host_k, uint16_t* host_v, int32_t* slot_of_block,
                             int32_t* block_of_slot, int32_t* last_used, uint16_t* pool_k,
                             uint16_t* pool_v, cudaStream_t st, const DeviceInfo& di) {
  if (s.Hkv > kMaxSpreadHeads) {
    append_kernel<false><<<s.B, 32 * s.Hkv, 0, st>>>(
        k_new, v_new, ctx_len, clock, step, host_k, host_v, slot_of_block, block_of_slot,
        last_used, pool_k, pool_v, s.Hkv, s.NB, s.S, s.sink, s.local, di.err);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(s.B * s.Hkv));
  cfg.blockDim = dim3(32);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(s.Hkv);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, append_kernel<true>, k_new, v_new, ctx_len, clock, step, host_k,
                            host_v, slot_of_block, block_of_slot, last_used, pool_k, pool_v, s.Hkv,
                            s.NB, s.S, s.sink, s.local, di.err);
}

// Compressed keys of each context's newest block, over its rows inside the
// context: one warp per (request, KV head), each in a CTA of its own so that
// the double arithmetic of the exact mean spreads over the SMs.  The rows are
// read from the working set when the block is resident (HBM; the append keeps
// it there), else from the cache, all 16 loads in flight at once.
__global__ void __launch_bounds__(32) refresh_kernel(const int32_t* __restrict__ ctx_len,
                                                     const uint16_t* __restrict__ host_k,
                                                     const int32_t* __restrict__ slot_of_block,
                                                     const uint16_t* __restrict__ pool_k,
                                                     float* __restrict__ summ,
                                                     uint16_t* __restrict__ summ_mm, int Hkv,
                                                     int NB, int S) {
  const int64_t u = blockIdx.x;
  const int b = static_cast<int>(u / Hkv), lane = threadIdx.x;
  const int64_t p = static_cast<int64_t>(ctx_len[b]) - 1;
  if (p < 0) return;  // an empty context has no block
  const int j = static_cast<int>(p / kBlockSize), t = static_cast<int>(p % kBlockSize);
  if (j >= NB) return;
  const int s = slot_of_block[u * NB + j];
  const uint16_t* src = s >= 0 && s < S ? pool_k + (u * S + s) * kBlockSize * kHeadDim
                                        : host_k + (u * NB + j) * kBlockSize * kHeadDim;
  uint2 rk[kBlockSize];
#pragma unroll
  for (int r = 0; r < kBlockSize; ++r)
    rk[r] = r <= t ? reinterpret_cast<const uint2*>(src + r * kHeadDim)[lane] : make_uint2(0u, 0u);
  double acc[4] = {0.0, 0.0, 0.0, 0.0};
  float hi[4], lo[4];
  uint16_t hib[4], lob[4];
#pragma unroll
  for (int r = 0; r < kBlockSize; ++r) {
    if (r > t) break;
    float f[4];
    uint16_t bits[4];
    bf16x4_to_f32(rk[r], f, bits);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[i] += static_cast<double>(f[i]);  // in row order, as the definition
      if (r == 0 || f[i] > hi[i]) {
        hi[i] = f[i];
        hib[i] = bits[i];
      }
      if (r == 0 || f[i] < lo[i]) {
        lo[i] = f[i];
        lob[i] = bits[i];
      }
    }
  }
  const double cnt = static_cast<double>(t + 1);
  float4 m;
  m.x = __double2float_rn(acc[0] / cnt);
  m.y = __double2float_rn(acc[1] / cnt);
  m.z = __double2float_rn(acc[2] / cnt);
  m.w = __double2float_rn(acc[3] / cnt);
  reinterpret_cast<float4*>(summ + (u * NB + j) * kHeadDim)[lane] = m;
  if (summ_mm) {
    uint16_t* d = summ_mm + (u * NB + j) * 2 * kHeadDim + 4 * lane;
    *reinterpret_cast<uint2*>(d) = make_uint2(hib[0] | (static_cast<uint32_t>(hib[1]) << 16),
                                              hib[2] | (static_cast<uint32_t>(hib[3]) << 16));
    *reinterpret_cast<uint2*>(d + kHeadDim) =
        make_uint2(lob[0] | (static_cast<uint32_t>(lob[1]) << 16),
                   lob[2] | (static_cast<uint32_t>(lob[3]) << 16));
  }
}

cudaError_t launch_refresh_summaries(const Shape& s, const int32_t* ctx_len,
                                     const uint16_t* host_k, const int32_t* slot_of_block,
                                     const uint16_t* pool_k, float* summ, uint16_t* summ_mm,
                                     cudaStream_t st, const DeviceInfo&) {
  refresh_kernel<<<s.units(), 32, 0, st>>>(ctx_len, host_k, slot_of_block, pool_k, summ, summ_mm,
                                           s.Hkv, s.NB, s.S);
  return cudaGetLastError();
}

}  // namespace oasis
