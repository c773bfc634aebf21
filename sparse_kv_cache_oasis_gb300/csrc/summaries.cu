// Compressed keys ("OasisKV: Scaling In-Decode KV Cache Beyond HBM with
// Lookahead Sparse Prefetching", Fig. 7 left): the fp32 mean key of every
// 16-token block, kept in HBM for the whole context.
//
// One warp per block; lane l owns dims 4l..4l+3.  The 16 keys are summed in
// double in token order (exact for bf16 inputs) and divided by 16, then
// rounded once to fp32.  Set-up work at admission, not on the per-step path.
#include "common.cuh"
#include "launch.h"

namespace oasis {

__global__ void __launch_bounds__(256) summaries_kernel(const uint16_t* __restrict__ k,
                                                        float* __restrict__ summ,
                                                        int64_t nblocks_total) {
  const int64_t blk = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (blk >= nblocks_total) return;
  // keys of this block: 16 rows of 128 bf16 = 16 x 32 uint2
  const uint2* src = reinterpret_cast<const uint2*>(k + blk * (kBlockSize * kHeadDim)) + lane;
  double a0 = 0.0, a1 = 0.0, a2 = 0.0, a3 = 0.0;
#pragma unroll
  for (int t = 0; t < kBlockSize; ++t) {
    const uint2 v = src[t * (kHeadDim / 4)];
    a0 += static_cast<double>(bf16lo_to_f32(v.x));
    a1 += static_cast<double>(bf16hi_to_f32(v.x));
    a2 += static_cast<double>(bf16lo_to_f32(v.y));
    a3 += static_cast<double>(bf16hi_to_f32(v.y));
  }
  const double inv = 1.0 / kBlockSize;  // power of two: exact
  float4 o;
  o.x = __double2float_rn(a0 * inv);
  o.y = __double2float_rn(a1 * inv);
  o.z = __double2float_rn(a2 * inv);
  o.w = __double2float_rn(a3 * inv);
  reinterpret_cast<float4*>(summ + blk * kHeadDim)[lane] = o;
}

cudaError_t launch_build_summaries(const Shape& s, const uint16_t* k, float* summ,
                                   cudaStream_t st, const DeviceInfo&) {
  const int64_t nblk = static_cast<int64_t>(s.units()) * s.NB;
  const int64_t threads = nblk * 32;
  const int64_t grid = (threads + 255) / 256;
  summaries_kernel<<<static_cast<unsigned>(grid), 256, 0, st>>>(k, summ, nblk);
  return cudaGetLastError();
}

}  // namespace oasis
