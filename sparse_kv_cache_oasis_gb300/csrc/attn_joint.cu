// Joint attention of the decoded token and the L draft tokens over one pass of
// the working set ("OasisKV: Scaling In-Decode KV Cache Beyond HBM with
// Lookahead Sparse Prefetching", Fig. 7 right: the attention kernel takes the
// normal and the draft queries together).  Every one of the T = 1 + L tokens'
// G query heads of a KV head is a row of that head's unit: T*G rows that all
// read the same K and V tiles.
//
// GB300 design: the attention body of attn.cu with the rows as the N
// dimension of the MMAs in NT tiles of 8 (NT <= 3: up to 24 rows per CTA).
// Each K / V^T fragment loaded from shared memory now feeds NT MMAs, so the
// KV bytes and the shared-memory traffic per slot stay those of the single
// query while the tensor work grows with the rows.  Units with more than 24
// rows are split into row groups of 8*NT rows, each a cluster of its own that
// streams the unit's slots again; the groups of a unit are adjacent in the
// grid and run together, so the repeated reads mostly hit L2.
#include "attn_body.cuh"
#include "launch.h"

namespace oasis {

template <int NT>
__global__ void __launch_bounds__(kAttnThreads) attn_joint_kernel(
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
    const uint16_t* __restrict__ q, const uint16_t* __restrict__ q_draft,
    const int32_t* __restrict__ block_of_slot, const int32_t* __restrict__ ctx_len,
    float scale_log2, uint16_t* __restrict__ out, int Hq, int Hkv, int G, int L, int S, int NB,
    int P, int n_groups, uint32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int c = blockIdx.x / P, r = blockIdx.x - c * P;  // (unit, row group), rank in cluster
  const int u = c / n_groups, grp = c - u * n_groups;
  const int b = u / Hkv, h = u - b * Hkv;
  const int row0 = grp * 8 * NT;
  const int rest = G * (L + 1) - row0;
  const JointRows rows{q, q_draft, out, b, h, Hq, G, L, row0};
  attn_cta<NT>(&tm_k, &tm_v, rows, rest < 8 * NT ? rest : 8 * NT, block_of_slot, ctx_len,
               scale_log2, Hkv, S, NB, P, err, smem, u, r, threadIdx.x >> 5, threadIdx.x & 31,
               [] { __syncthreads(); });
}

JointSplit joint_split(const Shape& s, int sm_count) {
  JointSplit j;
  const int rows = s.G * (s.L + 1);
  j.nt = (rows + 7) / 8 < kMaxRowTiles ? (rows + 7) / 8 : kMaxRowTiles;
  j.groups = (rows + 8 * j.nt - 1) / (8 * j.nt);
  // two CTAs per SM fit (at most 112 KB of shared memory, 128 threads of at
  // most 236 registers): P fills them.  Llama layer, 20 rows: 25.4 us at one
  // CTA per SM (P = 2), 23.3 us at two (P = 4), 36.2 us at P = 8.
  int p = 2 * (sm_count > 0 ? sm_count : 148) / (s.units() * j.groups);
  if (p > kMaxSplit) p = kMaxSplit;
  if (p > s.S / kMinSlotsPerCta) p = s.S / kMinSlotsPerCta;
  j.P = p < 1 ? 1 : p;
  return j;
}

template <int NT>
static cudaError_t joint_configure_nt() {
  const auto fn = attn_joint_kernel<NT>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(1024 + attn_smem_body(NT)));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  return e;
}

cudaError_t joint_configure() {
  cudaError_t e = joint_configure_nt<1>();
  if (e == cudaSuccess) e = joint_configure_nt<2>();
  if (e == cudaSuccess) e = joint_configure_nt<3>();
  return e;
}

template <int NT>
static cudaError_t launch_nt(const Shape& s, const JointSplit& j, const uint16_t* q,
                             const uint16_t* q_draft, const CUtensorMap& tm_k,
                             const CUtensorMap& tm_v, const int32_t* block_of_slot,
                             const int32_t* ctx_len, float scale_log2, uint16_t* out,
                             cudaStream_t st, const DeviceInfo& di) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(s.units() * j.groups * j.P));
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = 1024 + attn_smem_body(NT);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(j.P);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = j.P > 1 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, attn_joint_kernel<NT>, tm_k, tm_v, q, q_draft, block_of_slot,
                            ctx_len, scale_log2, out, s.Hq, s.Hkv, s.G, s.L, s.S, s.NB, j.P,
                            j.groups, di.err);
}

cudaError_t launch_sparse_decode_attn_joint(const Shape& s, const uint16_t* q,
                                            const uint16_t* q_draft, const CUtensorMap& tm_k,
                                            const CUtensorMap& tm_v,
                                            const int32_t* block_of_slot, const int32_t* ctx_len,
                                            float scale, uint16_t* out, cudaStream_t st,
                                            const DeviceInfo& di) {
  const JointSplit j = joint_split(s, di.sm_count);
  const float scale_log2 = scale * 1.4426950408889634f;
  switch (j.nt) {
    case 1:
      return launch_nt<1>(s, j, q, q_draft, tm_k, tm_v, block_of_slot, ctx_len, scale_log2, out,
                          st, di);
    case 2:
      return launch_nt<2>(s, j, q, q_draft, tm_k, tm_v, block_of_slot, ctx_len, scale_log2, out,
                          st, di);
    default:
      return launch_nt<3>(s, j, q, q_draft, tm_k, tm_v, block_of_slot, ctx_len, scale_log2, out,
                          st, di);
  }
}

}  // namespace oasis
