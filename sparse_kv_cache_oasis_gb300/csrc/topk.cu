// Per-KV-head top-K block prediction ("OasisKV: Scaling In-Decode KV Cache
// Beyond HBM with Lookahead Sparse Prefetching", explanatory diagram step 2,
// Fig. 4).
//
// One CTA of 1024 threads per (request, KV head); the scores stay in
// registers.  Forced blocks (sink and local window) are written first in
// ascending id.  The remaining K - |forced| blocks are found by a 4-pass MSB
// radix select over order-preserving 32-bit keys of the fp32 scores (-0.0 is
// folded onto +0.0 so that the order is exactly the fp32 order); blocks equal
// to the threshold are taken by ascending id.  The selected blocks are then
// placed by counting, for each, how many selected 64-bit keys
// (score_key << 32 | ~id) are larger: the output is the unique order by score
// descending, id ascending.  Histograms use warp-aggregated shared atomics
// (__match_any_sync) because the first digit of similar scores collides.
#include "common.cuh"
#include "launch.h"

namespace oasis {

constexpr int kTopkThreads = 1024;

__device__ __forceinline__ uint32_t orderable(float f) {
  uint32_t b = __float_as_uint(f);
  if (b == 0x80000000u) b = 0u;  // -0.0 == +0.0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

template <int ITEMS>
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const float* __restrict__ scores,
                                                            int32_t* __restrict__ topk_ids,
                                                            int NB, int K, int sink, int local) {
  __shared__ int hist[256];
  __shared__ int sDigit, sGreater, sEqual, sCount;
  __shared__ int sScan[33];
  __shared__ unsigned long long sKeys[1024];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t u = blockIdx.x;
  const float* sc = scores + u * NB;
  int32_t* out = topk_ids + u * K;

  // forced blocks: [0, a) and [lo, NB), ascending
  const int a = sink < NB ? sink : NB;
  const int b0 = NB - local > 0 ? NB - local : 0;
  const int lo = a > b0 ? a : b0;
  const int F = a + (NB - lo);
  const int need = K - F;
  for (int i = tid; i < F && i < K; i += kTopkThreads) out[i] = i < a ? i : lo + (i - a);
  if (need <= 0) return;

  uint32_t key[ITEMS];
  bool valid[ITEMS];
#pragma unroll
  for (int it = 0; it < ITEMS; ++it) {
    const int j = tid + it * kTopkThreads;
    valid[it] = j < NB && !(j < a || j >= lo);
    key[it] = valid[it] ? orderable(sc[j]) : 0u;
  }

  uint32_t prefix = 0u, mask = 0u;
  int remaining = need;
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    if (tid < 256) hist[tid] = 0;
    __syncthreads();
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
      const bool part = valid[it] && (key[it] & mask) == prefix;
      const int bin = part ? static_cast<int>((key[it] >> shift) & 255u) : 256;
      const unsigned peers = __match_any_sync(0xffffffffu, bin);
      if (part && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
    }
    __syncthreads();
    if (warp == 0) {
      int c[8], local_sum = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        c[k] = hist[lane * 8 + k];
        local_sum += c[k];
      }
      int incl = local_sum;  // suffix sum over lanes >= lane
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl += y;
      }
      int running = incl - local_sum;  // elements with a larger digit
#pragma unroll
      for (int k = 7; k >= 0; --k) {
        if (running < remaining && running + c[k] >= remaining) {
          sDigit = lane * 8 + k;
          sGreater = running;
          sEqual = c[k];
        }
        running += c[k];
      }
    }
    __syncthreads();
    prefix |= static_cast<uint32_t>(sDigit) << shift;
    mask |= 255u << shift;
    remaining -= sGreater;
    __syncthreads();
  }
  const int n_equal = sEqual;  // elements whose key equals the threshold

  // equal keys are taken by ascending id; rank them only when it matters
  int eq_rank[ITEMS];
#pragma unroll
  for (int it = 0; it < ITEMS; ++it) eq_rank[it] = 0;
  if (n_equal > remaining) {
    int base = 0;
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
      int tot;
      const int e = valid[it] && key[it] == prefix;
      eq_rank[it] = base + block_exclusive_scan(e, sScan, &tot);
      base += tot;
    }
  }
  if (tid == 0) sCount = 0;
  __syncthreads();
#pragma unroll
  for (int it = 0; it < ITEMS; ++it) {
    const int j = tid + it * kTopkThreads;
    const bool sel = valid[it] && (key[it] > prefix || (key[it] == prefix && eq_rank[it] < remaining));
    if (sel) {
      const int pos = atomicAdd(&sCount, 1);
      if (pos < 1024) sKeys[pos] = (static_cast<unsigned long long>(key[it]) << 32) |
                   static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(j));
    }
  }
  __syncthreads();
  for (int i = tid; i < need; i += kTopkThreads) {
    const unsigned long long my = sKeys[i];
    int r = 0;
    for (int k = 0; k < need; ++k) r += sKeys[k] > my;
    out[F + r] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(my & 0xFFFFFFFFull));
  }
}

template <int ITEMS>
static cudaError_t launch_items(const Shape& s, const float* scores, int32_t* topk_ids,
                                cudaStream_t st) {
  topk_kernel<ITEMS><<<s.units(), kTopkThreads, 0, st>>>(scores, topk_ids, s.NB, s.K, s.sink,
                                                         s.local);
  return cudaGetLastError();
}

cudaError_t launch_select_topk(const Shape& s, const float* scores, int32_t* topk_ids,
                               cudaStream_t st, const DeviceInfo&) {
  const int items = (s.NB + kTopkThreads - 1) / kTopkThreads;
  if (items <= 1) return launch_items<1>(s, scores, topk_ids, st);
  if (items <= 2) return launch_items<2>(s, scores, topk_ids, st);
  if (items <= 4) return launch_items<4>(s, scores, topk_ids, st);
  if (items <= 8) return launch_items<8>(s, scores, topk_ids, st);
  if (items <= 16) return launch_items<16>(s, scores, topk_ids, st);
  if (items <= 32) return launch_items<32>(s, scores, topk_ids, st);
  return cudaErrorInvalidValue;  // rejected earlier by validation (NB <= 32768)
}

}  // namespace oasis
