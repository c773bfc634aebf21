// KV selection with capped eviction ("OasisKV: Scaling In-Decode KV Cache
// Beyond HBM with Lookahead Sparse Prefetching", explanatory diagram step 3;
// Tab. 2, fetch cap and LRU eviction; Fig. 9, head-wise GPU-slot <-> CPU-block
// map).
//
// One CTA per (request, KV head) with one thread per top-K entry and per
// working-set slot.  Everything is integer work on a few hundred entries held
// in shared memory; ranks come from block-wide prefix sums and from counting
// comparisons, so the result is the same on every run and equals the plain
// sequential definition:
//   1. predicted blocks already resident are used at `step`;
//   2. the first n = min(#missing, cap) missing blocks, in list (priority)
//      order, are fetched;
//   3. e = max(0, |R| + n - S) residents outside the prediction are evicted,
//      least recently used first, ties to the lower block id;
//   4. free slots (empty or freed) in ascending order receive the fetched
//      blocks in ascending block id, and are marked used at `step`.
// An id out of range, a repeated id or a map whose two directions disagree
// leaves the (request, KV head) untouched, reports n = e = 0 and sets an error
// bit.
#include "common.cuh"
#include "launch.h"

namespace oasis {

constexpr int kInP = 1;

__global__ void plan_kernel(const int32_t* __restrict__ topk_ids, int32_t step_arg,
                            int32_t* __restrict__ clock, int32_t* __restrict__ slot_of_block, int32_t* __restrict__ block_of_slot,
                            int32_t* __restrict__ last_used, int32_t* __restrict__ fetch_block,
                            int32_t* __restrict__ fetch_slot, int32_t* __restrict__ evict_block,
                            int32_t* __restrict__ n_fetch, int32_t* __restrict__ n_evict, int NB,
                            int S, int K, int cap, int capw, uint32_t* err) {
  extern __shared__ int smem[];
  int* sP = smem;               // [K]   predicted blocks, priority order
  int* sBos = sP + K;           // [S]   block of slot
  int* sLu = sBos + S;          // [S]   last used
  int* sFlag = sLu + S;         // [S]   kInP
  int* sFetch = sFlag + S;      // [capw] fetched blocks, priority order
  int* sFreeSlot = sFetch + capw;    // [capw] free slots, ascending
  int* sVictim = sFreeSlot + capw;   // [capw] victim blocks, LRU order
  int* sScan = sVictim + capw;       // [33]
  __shared__ int sBad;

  const int tid = threadIdx.x, T = blockDim.x;
  const int64_t u = blockIdx.x;
  // the step is a value, or the unit's clock in device memory (advanced at the end)
  const int32_t step = clock ? clock[u] : step_arg;
  const int32_t* P = topk_ids + u * K;
  int32_t* sob = slot_of_block + u * NB;
  int32_t* bos = block_of_slot + u * S;
  int32_t* lu = last_used + u * S;

  if (tid == 0) sBad = 0;
  for (int i = tid; i < K; i += T) sP[i] = P[i];
  for (int s = tid; s < S; s += T) {
    sBos[s] = bos[s];
    sLu[s] = lu[s];
    sFlag[s] = 0;
  }
  __syncthreads();

  // ---- validation: ids in range and distinct; both map directions agree
  if (tid < K) {
    const int p = sP[tid];
    if (p < 0 || p >= NB) {
      atomicOr(&sBad, OASIS_DEVERR_TOPK_IDS);
    } else {
      for (int i = 0; i < tid; ++i)
        if (sP[i] == p) atomicOr(&sBad, OASIS_DEVERR_TOPK_IDS);
    }
  }
  if (tid < S) {
    const int j = sBos[tid];
    if (j >= NB || (j >= 0 && sob[j] != tid)) atomicOr(&sBad, OASIS_DEVERR_PLAN_STATE);
  }
  __syncthreads();
  int hit_slot = -1, miss = 0;
  if (sBad == 0 && tid < K) {
    const int p = sP[tid];
    const int s = sob[p];
    if (s >= 0) {
      if (s >= S || sBos[s] != p) atomicOr(&sBad, OASIS_DEVERR_PLAN_STATE);
      else hit_slot = s;
    } else {
      miss = 1;
    }
  }
  __syncthreads();
  const int bad = sBad;
  if (bad) {
    if (tid == 0) {
      set_error(err, static_cast<uint32_t>(bad));
      n_fetch[u] = 0;
      n_evict[u] = 0;
      if (clock) clock[u] = step + 1;
    }
    for (int r = tid; r < capw; r += T) {
      fetch_block[u * capw + r] = -1;
      fetch_slot[u * capw + r] = -1;
      evict_block[u * capw + r] = -1;
    }
    return;
  }

  // ---- step 1: hits are used now
  if (hit_slot >= 0) {
    sFlag[hit_slot] = kInP;
    sLu[hit_slot] = step;
  }
  // ---- step 2: the first n misses in priority order
  int nmiss;
  const int mrank = block_exclusive_scan(miss, sScan, &nmiss);
  const int n = nmiss < cap ? nmiss : cap;
  if (miss && mrank < n) sFetch[mrank] = sP[tid];

  // ---- step 3: LRU victims among residents outside the prediction
  const int resident = (tid < S) && sBos[tid] >= 0;
  const int cand = resident && !(sFlag[tid] & kInP);
  int nres;
  (void)block_exclusive_scan(resident, sScan, &nres);
  int e = nres + n - S;
  if (e < 0) e = 0;
  int victim = 0;
  if (cand) {
    const int my_lu = sLu[tid], my_blk = sBos[tid];
    int rank = 0;
    for (int s2 = 0; s2 < S; ++s2) {
      const int b2 = sBos[s2];
      if (b2 < 0 || (sFlag[s2] & kInP)) continue;
      const int l2 = sLu[s2];
      rank += (l2 < my_lu) || (l2 == my_lu && b2 < my_blk);
    }
    if (rank < e) {
      victim = 1;
      sVictim[rank] = my_blk;
    }
  }
  // ---- step 4: free slots in ascending order
  const int is_free = (tid < S) && (sBos[tid] < 0 || victim);
  int nfree;
  const int frank = block_exclusive_scan(is_free, sScan, &nfree);
  if (is_free && frank < n) sFreeSlot[frank] = tid;
  __syncthreads();

  // fetched blocks in ascending id take the free slots in ascending order
  int my_fetch_blk = -1, my_fetch_slot = -1;
  if (tid < n) {
    my_fetch_blk = sFetch[tid];
    int r = 0;
    for (int i = 0; i < n; ++i) r += sFetch[i] < my_fetch_blk;
    my_fetch_slot = sFreeSlot[r];
    fetch_block[u * capw + r] = my_fetch_blk;
    fetch_slot[u * capw + r] = my_fetch_slot;
  }
  if (tid < e) {
    const int vb = sVictim[tid];
    int r = 0;
    for (int i = 0; i < e; ++i) r += sVictim[i] < vb;
    evict_block[u * capw + r] = vb;
  }
  for (int r = tid; r < capw; r += T) {
    if (r >= n) {
      fetch_block[u * capw + r] = -1;
      fetch_slot[u * capw + r] = -1;
    }
    if (r >= e) evict_block[u * capw + r] = -1;
  }
  // ---- apply: victims leave, fetched blocks enter
  if (victim) {
    sob[sBos[tid]] = -1;
    sBos[tid] = -1;
  }
  __syncthreads();
  if (tid < n) {
    sBos[my_fetch_slot] = my_fetch_blk;
    sLu[my_fetch_slot] = step;
    sob[my_fetch_blk] = my_fetch_slot;
  }
  __syncthreads();
  for (int s = tid; s < S; s += T) {
    bos[s] = sBos[s];
    lu[s] = sLu[s];
  }
  if (tid == 0) {
    n_fetch[u] = n;
    n_evict[u] = e;
    if (clock) clock[u] = step + 1;
  }
}

cudaError_t launch_plan_fetch(const Shape& s, const int32_t* topk_ids, int32_t step,
                              int32_t* clock, int32_t* slot_of_block, int32_t* block_of_slot,
                              int32_t* last_used, int32_t* fetch_block, int32_t* fetch_slot,
                              int32_t* evict_block, int32_t* n_fetch, int32_t* n_evict,
                              cudaStream_t st, const DeviceInfo& di) {
  const int capw = s.cap > 0 ? s.cap : 1;
  const int need = s.S > s.K ? s.S : s.K;
  const int threads = ((need + 31) / 32) * 32;
  const size_t smem = sizeof(int) * (static_cast<size_t>(s.K) + 3 * s.S + 3 * capw + 33);
  plan_kernel<<<s.units(), threads, smem, st>>>(topk_ids, step, clock, slot_of_block, block_of_slot,
                                                last_used, fetch_block, fetch_slot, evict_block,
                                                n_fetch, n_evict, s.NB, s.S, s.K, s.cap, capw,
                                                di.err);
  return cudaGetLastError();
}

}  // namespace oasis
