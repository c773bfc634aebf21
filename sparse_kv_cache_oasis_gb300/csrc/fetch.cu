// KV transfer ("OasisKV: Scaling In-Decode KV Cache Beyond HBM with Lookahead
// Sparse Prefetching", explanatory diagram step 4 and Fig. 8): the blocks
// chosen by the planner are copied from the pinned host cache into their HBM
// working-set slots, on a copy stream that overlaps compute.
//
// GB300 design: a zero-copy gather.  The host cache is mapped into the device
// address space and read directly over NVLink-C2C with 16-byte loads; there is
// no staging copy and no per-block copy-engine call.  The planned (request,
// KV head, list entry) items are taken grid-stride by a small fixed number of
// CTAs; 128 threads move an item's 4 KiB K block and 4 KiB V block, all four
// 16-byte loads of a thread issued before any store.  The CTA count bounds the
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
    int NB, int S, int capw, int items, uint32_t* err) {
  // items = units x capw list entries, taken grid-stride
  for (int it = blockIdx.x; it < items; it += gridDim.x) {
    const int u = it / capw;  // (request, KV head) unit
    const int r = it - u * capw;  // entry of the fetch list
    const int n = n_fetch[u];
    if (r == 0 && threadIdx.x == 0 && (n < 0 || n > capw)) set_error(err, OASIS_DEVERR_FETCH_RANGE);
    if (r >= n) continue;
    const int j = fetch_block[static_cast<int64_t>(u) * capw + r];
    const int s = fetch_slot[static_cast<int64_t>(u) * capw + r];
    if (j < 0 || j >= NB || s < 0 || s >= S) {
      if (threadIdx.x == 0) set_error(err, OASIS_DEVERR_FETCH_RANGE);
      continue;
    }
    const int64_t src = (static_cast<int64_t>(u) * NB + j) * kVecPerBlock;
    const int64_t dst = (static_cast<int64_t>(u) * S + s) * kVecPerBlock;
    int4 kv[kVecPerThread], vv[kVecPerThread];
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i) {
      kv[i] = host_k[src + threadIdx.x + i * kFetchThreads];
      vv[i] = host_v[src + threadIdx.x + i * kFetchThreads];
    }
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i) {
      pool_k[dst + threadIdx.x + i * kFetchThreads] = kv[i];
      pool_v[dst + threadIdx.x + i * kFetchThreads] = vv[i];
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
  const int items = capw * s.units();
  const int grid = items < kFetchCtas ? items : kFetchCtas;
  fetch_kernel<<<grid, kFetchThreads, 0, st>>>(
      reinterpret_cast<const int4*>(host_k), reinterpret_cast<const int4*>(host_v), fetch_block,
      fetch_slot, n_fetch, reinterpret_cast<int4*>(pool_k), reinterpret_cast<int4*>(pool_v), s.NB,
      s.S, capw, items, di.err);
  return cudaGetLastError();
}

}  // namespace oasis
