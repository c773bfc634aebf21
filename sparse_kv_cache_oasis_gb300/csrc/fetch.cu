// KV transfer ("OasisKV: Scaling In-Decode KV Cache Beyond HBM with Lookahead
// Sparse Prefetching", explanatory diagram step 4 and Fig. 8): the blocks
// chosen by the planner are copied from the pinned host cache into their HBM
// working-set slots, on a copy stream that overlaps compute.
//
// GB300 design: a zero-copy gather.  The host cache is mapped into the device
// address space and read directly over NVLink-C2C with 16-byte loads; there is
// no staging copy and no per-block copy-engine call.  The planned (request,
// KV head, list entry) items are split in equal contiguous shares over a
// small fixed number of CTAs; a CTA first gathers the counts of its units and
// the block and slot of its valid entries (loads in flight together, empty
// entries skipped), then 128 threads move one entry's 4 KiB K block and 4 KiB
// V block after another, all four 16-byte loads of a thread issued before
// any store.  The CTA count bounds the
// link requests in flight: the transfer runs beside the HBM-bound attention
// and scoring kernels, and an unbounded burst of long-latency host reads
// slows their streams more than it speeds the transfer (measured on the 32K /
// 2K-budget Llama layer step, µs per step for 48/64/96/128/192/448 CTAs:
// 33.5/32.6/32.6/33.4/38.0/44.0).
#include "common.cuh"
#include "launch.h"

namespace oasis {

constexpr int kFetchThreads = 128;
constexpr int kVecPerBlock = kBlockSize * kHeadDim * 2 / 16;  // 256 int4 per K (or V) block
constexpr int kVecPerThread = kVecPerBlock / kFetchThreads;   // 2
constexpr int kFetchCtas = 64;  // CTAs of the grid-stride gather (bounds the link requests in flight)

__global__ void __launch_bounds__(kFetchThreads) fetch_kernel(
    const int4* __restrict__ host_k, const int4* __restrict__ host_v,
    const int32_t* __restrict__ fetch_block, const int32_t* __restrict__ fetch_slot,
    const int32_t* __restrict__ n_fetch, int4* __restrict__ pool_k, int4* __restrict__ pool_v,
    int NB, int S, int capw, int64_t items, uint32_t* err) {
  // this CTA's contiguous share [a, b) of the units x capw list entries, its
  // units taken kFetchThreads at a time: their counts and an exclusive scan
  // number the valid entries; then, kFetchThreads entries at a time, the
  // entries' block and slot are loaded together and the blocks copied one
  // after another (each copy one host round trip; stores never wait)
  __shared__ int s_lo[kFetchThreads], s_c[kFetchThreads], s_off[kFetchThreads];
  __shared__ int s_u[kFetchThreads], s_j[kFetchThreads], s_s[kFetchThreads];
  __shared__ int s_warp[kFetchThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t per = (items + gridDim.x - 1) / gridDim.x;
  const int64_t a = static_cast<int64_t>(blockIdx.x) * per;
  const int64_t b = a + per < items ? a + per : items;
  if (a >= b) return;
  const int64_t u_first = a / capw, u_last = (b - 1) / capw;
  for (int64_t ub = u_first; ub <= u_last; ub += kFetchThreads) {
    // entries [lo, lo + c) of unit ub + tid lie in [a, b) and below its count
    int lo = 0, c = 0;
    const int64_t u = ub + tid;
    if (u <= u_last) {
      int n = n_fetch[u];
      if (n < 0 || n > capw) {
        if (u * capw >= a) set_error(err, OASIS_DEVERR_FETCH_RANGE);
        n = n < 0 ? 0 : capw;
      }
      const int64_t r_lo = a > u * capw ? a - u * capw : 0;
      const int64_t r_hi = b < (u + 1) * capw ? b - u * capw : capw;
      lo = static_cast<int>(r_lo);
      const int hi = static_cast<int>(r_hi < n ? r_hi : n);
      c = hi > lo ? hi - lo : 0;
    }
    // exclusive scan of c over the CTA
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    __syncthreads();  // the previous chunk's shared arrays are no longer read
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    int base = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kFetchThreads / 32; ++w) {
      if (w < warp) base += s_warp[w];
      total += s_warp[w];
    }
    s_lo[tid] = lo;
    s_c[tid] = c;
    s_off[tid] = base + incl - c;
    __syncthreads();
    for (int k0 = 0; k0 < total; k0 += kFetchThreads) {
      const int kn = total - k0 < kFetchThreads ? total - k0 : kFetchThreads;
      if (k0 > 0) __syncthreads();  // the previous batch's copies read s_j / s_s / s_u
      if (tid < kn) {
        const int k = k0 + tid;
        int lo_i = 0, hi_i = kFetchThreads - 1;  // last unit with s_off <= k and c > 0
        while (lo_i < hi_i) {
          const int mid = (lo_i + hi_i + 1) >> 1;
          if (s_off[mid] <= k) lo_i = mid; else hi_i = mid - 1;
        }
        while (lo_i > 0 && (s_c[lo_i] == 0 || k >= s_off[lo_i] + s_c[lo_i])) --lo_i;  // empty units
        const int r = s_lo[lo_i] + (k - s_off[lo_i]);
        const int64_t idx = (ub + lo_i) * capw + r;
        s_u[tid] = lo_i;
        s_j[tid] = fetch_block[idx];
        s_s[tid] = fetch_slot[idx];
      }
      __syncthreads();
      for (int k = 0; k < kn; ++k) {
        const int64_t uu = ub + s_u[k];
        const int j = s_j[k], sl = s_s[k];
        if (j < 0 || j >= NB || sl < 0 || sl >= S) {
          if (tid == 0) set_error(err, OASIS_DEVERR_FETCH_RANGE);
          continue;
        }
        const int64_t src = (uu * NB + j) * kVecPerBlock;
        const int64_t dst = (uu * S + sl) * kVecPerBlock;
        int4 kv[kVecPerThread], vv[kVecPerThread];
#pragma unroll
        for (int i = 0; i < kVecPerThread; ++i) {
          kv[i] = host_k[src + tid + i * kFetchThreads];
          vv[i] = host_v[src + tid + i * kFetchThreads];
        }
#pragma unroll
        for (int i = 0; i < kVecPerThread; ++i) {
          pool_k[dst + tid + i * kFetchThreads] = kv[i];
          pool_v[dst + tid + i * kFetchThreads] = vv[i];
        }
      }
    }
  }
}

// Largest shared-memory carve-out (the transfer shares SMs with the attention
// and scoring kernels of the step).
cudaError_t fetch_configure() {
  return cudaFuncSetAttribute(fetch_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                              cudaSharedmemCarveoutMaxShared);
}

cudaError_t launch_fetch_blocks(const Shape& s, const uint16_t* host_k, const uint16_t* host_v,
                                const int32_t* fetch_block, const int32_t* fetch_slot,
                                const int32_t* n_fetch, uint16_t* pool_k, uint16_t* pool_v,
                                cudaStream_t st, const DeviceInfo& di) {
  const int capw = s.cap > 0 ? s.cap : 1;
  const int64_t items = static_cast<int64_t>(capw) * s.units();
  const int grid = items < kFetchCtas ? static_cast<int>(items) : kFetchCtas;
  fetch_kernel<<<grid, kFetchThreads, 0, st>>>(
      reinterpret_cast<const int4*>(host_k), reinterpret_cast<const int4*>(host_v), fetch_block,
      fetch_slot, n_fetch, reinterpret_cast<int4*>(pool_k), reinterpret_cast<int4*>(pool_v), s.NB,
      s.S, capw, items, di.err);
  return cudaGetLastError();
}

}  // namespace oasis
