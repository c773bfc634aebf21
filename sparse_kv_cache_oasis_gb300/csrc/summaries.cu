// Compressed keys ("OasisKV: Scaling In-Decode KV Cache Beyond HBM with
// Lookahead Sparse Prefetching", Fig. 7 left): the fp32 mean key of every
// 16-token block (or its min/max keys, below), kept in HBM for the whole
// context.
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

// Min/max compressed keys (the pooling Fig. 7 left names): per block the
// elementwise max and min of its 16 keys, kept as the bf16 values themselves
// in one 512-byte row [max(D) | min(D)].  One warp per block, lane l owns dims
// 4l..4l+3; on equal values the earlier token's bits are kept (so +0 and -0
// resolve by token order).
__global__ void __launch_bounds__(256) summaries_minmax_kernel(const uint16_t* __restrict__ k,
                                                               uint16_t* __restrict__ summ_mm,
                                                               int64_t nblocks_total) {
  const int64_t blk = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (blk >= nblocks_total) return;
  const uint16_t* src = k + blk * (kBlockSize * kHeadDim) + 4 * lane;
  uint16_t mxb[4], mnb[4];
  float mx[4], mn[4];
#pragma unroll
  for (int t = 0; t < kBlockSize; ++t) {
    const uint2 v = *reinterpret_cast<const uint2*>(src + t * kHeadDim);
    const uint16_t bits[4] = {static_cast<uint16_t>(v.x & 0xFFFFu), static_cast<uint16_t>(v.x >> 16),
                              static_cast<uint16_t>(v.y & 0xFFFFu), static_cast<uint16_t>(v.y >> 16)};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float f = __uint_as_float(static_cast<uint32_t>(bits[i]) << 16);
      if (t == 0 || f > mx[i]) {
        mx[i] = f;
        mxb[i] = bits[i];
      }
      if (t == 0 || f < mn[i]) {
        mn[i] = f;
        mnb[i] = bits[i];
      }
    }
  }
  uint16_t* dst = summ_mm + blk * (2 * kHeadDim) + 4 * lane;
  *reinterpret_cast<uint2*>(dst) =
      make_uint2(mxb[0] | (static_cast<uint32_t>(mxb[1]) << 16), mxb[2] | (static_cast<uint32_t>(mxb[3]) << 16));
  *reinterpret_cast<uint2*>(dst + kHeadDim) =
      make_uint2(mnb[0] | (static_cast<uint32_t>(mnb[1]) << 16), mnb[2] | (static_cast<uint32_t>(mnb[3]) << 16));
}

cudaError_t launch_build_summaries_minmax(const Shape& s, const uint16_t* k, uint16_t* summ_mm,
                                          cudaStream_t st, const DeviceInfo&) {
  const int64_t nblk = static_cast<int64_t>(s.units()) * s.NB;
  const int64_t grid = (nblk * 32 + 255) / 256;
  summaries_minmax_kernel<<<static_cast<unsigned>(grid), 256, 0, st>>>(k, summ_mm, nblk);
  return cudaGetLastError();
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
