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
#include "attn_body.cuh"
#include "launch.h"

namespace oasis {

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
int attn_split(const Shape& s, int sm_count) {
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

__global__ void __launch_bounds__(kAttnThreads) attn_kernel(
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
    const uint16_t* __restrict__ q, const int32_t* __restrict__ block_of_slot,
    const int32_t* __restrict__ ctx_len, float scale_log2, uint16_t* __restrict__ out, int Hq,
    int Hkv, int G, int S, int NB, int P, uint32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int u = blockIdx.x / P, r = blockIdx.x - u * P;  // unit, rank in its cluster
  const int b = u / Hkv, h = u - b * Hkv;
  const GroupRows rows{q, out, (static_cast<int64_t>(b) * Hq + h * G) * kHeadDim};
  attn_cta<1>(&tm_k, &tm_v, rows, G, block_of_slot, ctx_len, scale_log2, Hkv, S, NB, P, err, smem,
              u, r, threadIdx.x >> 5, threadIdx.x & 31, [] { __syncthreads(); });
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
  const int P = attn_split(s, di.sm_count > 0 ? di.sm_count : current_sm_count());
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
