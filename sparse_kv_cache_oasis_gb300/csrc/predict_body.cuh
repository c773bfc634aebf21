// Bodies of the top-K block prediction and the capped-eviction planning
// ("OasisKV: Scaling In-Decode KV Cache Beyond HBM with Lookahead Sparse
// Prefetching", explanatory diagram steps 2-3), shared by the prediction
// kernels and the fused prediction chain.  The design is described in
// predict.cu.
#pragma once

#include "common.cuh"
#include "launch.h"

namespace oasis {

constexpr int kPredThreads = 1024;

__device__ __forceinline__ uint32_t orderable(float f) {
  uint32_t b = __float_as_uint(f);
  if (b == 0x80000000u) b = 0u;  // -0.0 == +0.0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Shared-memory views, carved from dynamic shared memory sized to the shape
// (top-K and plan scratch share one region: the plan starts after the top-K
// list is final).
struct TopkSmem {
  unsigned long long* keys;  // [K]
  int* hist;                 // [256]
  int* digit;
  int* greater;
  int* equal;
  int* count;
  int* scan;                 // [33]
};

struct PlanSmem {
  unsigned long long* lru_key;  // [S] per slot: candidate key or ~0
  int* bos;                     // [S] block of slot (updated in place)
  int* lu;                      // [S] last used (updated in place)
  int* inp;                     // [S] slot holds a predicted block
  unsigned int* seen;           // [ceil(NB/32)] bitmap of predicted ids
  int* fetch;                   // [capw] fetched blocks, priority order
  int* free_slot;               // [capw] free slots, ascending
  int* victim;                  // [capw] victim blocks, LRU order
  int* scan;                    // [33]
  int* bad;
};

struct PredLayout {
  int K, S, NB, capw;
  __host__ __device__ size_t list_bytes() const { return ((static_cast<size_t>(K) * 4 + 7) / 8) * 8; }
  __host__ __device__ size_t topk_bytes() const { return static_cast<size_t>(K) * 8 + (256 + 4 + 33) * 4; }
  __host__ __device__ size_t plan_bytes() const {
    return static_cast<size_t>(S) * 8 + static_cast<size_t>(S) * 12 + static_cast<size_t>((NB + 31) / 32) * 4 +
           static_cast<size_t>(capw) * 12 + (33 + 1) * 4;
  }
  __host__ __device__ size_t bytes() const {
    const size_t t = topk_bytes(), q = plan_bytes();
    return list_bytes() + (t > q ? t : q);
  }
  __device__ void carve(unsigned char* base, int** list, TopkSmem* tk, PlanSmem* pl) const {
    *list = reinterpret_cast<int*>(base);
    unsigned char* r = base + list_bytes();
    tk->keys = reinterpret_cast<unsigned long long*>(r);
    int* ti = reinterpret_cast<int*>(r + static_cast<size_t>(K) * 8);
    tk->hist = ti;
    tk->digit = ti + 256;
    tk->greater = ti + 257;
    tk->equal = ti + 258;
    tk->count = ti + 259;
    tk->scan = ti + 260;
    pl->lru_key = reinterpret_cast<unsigned long long*>(r);
    int* pi = reinterpret_cast<int*>(r + static_cast<size_t>(S) * 8);
    pl->bos = pi;
    pl->lu = pi + S;
    pl->inp = pi + 2 * S;
    pl->seen = reinterpret_cast<unsigned int*>(pi + 3 * S);
    int* after = pi + 3 * S + (NB + 31) / 32;
    pl->fetch = after;
    pl->free_slot = after + capw;
    pl->victim = after + 2 * capw;
    pl->scan = after + 3 * capw;
    pl->bad = after + 3 * capw + 33;
  }
};

// Blocks in the context of request b: ceil(ctx_len[b] / bs), at most NB
// (all NB without a context length).
__device__ __forceinline__ int context_blocks(const int32_t* ctx_len, int b, int bs, int NB) {
  if (!ctx_len) return NB;
  const int c = ctx_len[b];
  if (c <= 0) return 0;
  const long long n = (static_cast<long long>(c) + bs - 1) / bs;
  return n < NB ? static_cast<int>(n) : NB;
}

// Writes the unit's top-K list (priority order) to `out_smem` (K ints) and,
// if out_global is not null, to global memory.  All threads must call it.
// `nblk` blocks are in the context: the local window ends there, and blocks at
// or beyond it rank as if scored -infinity (nblk = NB: the whole cache).
template <int ITEMS, bool CTX>
__device__ void topk_unit(const float* __restrict__ sc, int NB, int nblk_arg, int K, int sink,
                          int local, int* out_smem, int32_t* __restrict__ out_global,
                          const TopkSmem& sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = blockDim.x;
  // with a context length: the scores are loaded first, before anything that
  // depends on the length, so that their loads overlap its load
  float raw[ITEMS];
  if constexpr (CTX) {
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
      const int j = tid + it * T;
      raw[it] = j < NB ? __ldcg(sc + j) : 0.f;
    }
  }
  const int nblk = CTX ? nblk_arg : NB;  // without a context length: the whole cache
  const int a = sink < nblk ? sink : nblk;
  const int b0 = nblk - local > 0 ? nblk - local : 0;
  const int lo = a > b0 ? a : b0;
  const int F = a + (nblk - lo);
  const int need = K - F;
  for (int i = tid; i < F && i < K; i += T) {
    const int id = i < a ? i : lo + (i - a);
    out_smem[i] = id;
    if (out_global) out_global[i] = id;
  }
  if (need <= 0) {
    __syncthreads();
    return;
  }
  uint32_t key[ITEMS];
  bool valid[ITEMS];
#pragma unroll
  for (int it = 0; it < ITEMS; ++it) {
    const int j = tid + it * T;
    if constexpr (CTX) {
      valid[it] = j < NB && !(j < a || (j >= lo && j < nblk));
      key[it] = valid[it] ? orderable(j < nblk ? raw[it] : -INFINITY) : 0u;
    } else {
      valid[it] = j < NB && !(j < a || j >= lo);
      key[it] = valid[it] ? orderable(__ldcg(sc + j)) : 0u;
    }
  }
  uint32_t prefix = 0u, mask = 0u;
  int remaining = need;
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += T) sm.hist[i] = 0;
    __syncthreads();
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
      const bool part = valid[it] && (key[it] & mask) == prefix;
      const int bin = part ? static_cast<int>((key[it] >> shift) & 255u) : 256;
      const unsigned peers = __match_any_sync(0xffffffffu, bin);
      if (part && lane == __ffs(peers) - 1) atomicAdd(&sm.hist[bin], __popc(peers));
    }
    __syncthreads();
    if (warp == 0) {
      int c[8], lsum = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        c[k] = sm.hist[lane * 8 + k];
        lsum += c[k];
      }
      int incl = lsum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl += y;
      }
      int running = incl - lsum;
#pragma unroll
      for (int k = 7; k >= 0; --k) {
        if (running < remaining && running + c[k] >= remaining) {
          *sm.digit = lane * 8 + k;
          *sm.greater = running;
          *sm.equal = c[k];
        }
        running += c[k];
      }
    }
    __syncthreads();
    prefix |= static_cast<uint32_t>(*sm.digit) << shift;
    mask |= 255u << shift;
    remaining -= *sm.greater;
  }
  const int n_equal = *sm.equal;
  int eq_rank[ITEMS];
#pragma unroll
  for (int it = 0; it < ITEMS; ++it) eq_rank[it] = 0;
  if (n_equal > remaining) {  // ties at the threshold: lowest ids first
    int base = 0;
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
      int tot;
      const int e = valid[it] && key[it] == prefix;
      eq_rank[it] = base + block_exclusive_scan(e, sm.scan, &tot);
      base += tot;
    }
  }
  if (tid == 0) *sm.count = 0;
  __syncthreads();
#pragma unroll
  for (int it = 0; it < ITEMS; ++it) {
    const int j = tid + it * T;
    const bool sel =
        valid[it] && (key[it] > prefix || (key[it] == prefix && eq_rank[it] < remaining));
    const unsigned bal = __ballot_sync(0xffffffffu, sel);
    int base = 0;
    if (lane == 0 && bal) base = atomicAdd(sm.count, __popc(bal));
    base = __shfl_sync(0xffffffffu, base, 0);
    if (sel) {
      const int pos = base + __popc(bal & ((1u << lane) - 1u));
      if (pos < K)
        sm.keys[pos] = (static_cast<unsigned long long>(key[it]) << 32) |
                       static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(j));
    }
  }
  __syncthreads();
  // rank = number of larger keys; tpk threads per key share the comparisons
  int tpk = 1;
  while (tpk < 32 && need * tpk * 2 <= T) tpk *= 2;
  for (int i0 = 0; i0 < need; i0 += T / tpk) {
    const int i = i0 + tid / tpk, sub = tid % tpk;
    unsigned long long my = 0ull;
    int r = 0;
    if (i < need) {
      my = sm.keys[i];
      for (int k = sub; k < need; k += tpk) r += sm.keys[k] > my;
    }
    for (int o = 1; o < tpk; o <<= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
    if (i < need && sub == 0) {
      const int id = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(my & 0xFFFFFFFFull));
      out_smem[F + r] = id;
      if (out_global) out_global[F + r] = id;
    }
  }
  __syncthreads();
}

// Per-thread view of the unit's working-set map, loaded before the plan.
struct SlotView {
  int bos;   // block in slot tid (tid < S), else -1
  int lu;    // last used of slot tid
  int chk;   // slot_of_block[bos] when the slot is valid, for the map check
};

__device__ __forceinline__ SlotView load_slot_view(const int32_t* __restrict__ sob,
                                                   const int32_t* __restrict__ bos,
                                                   const int32_t* __restrict__ lu, int S, int NB) {
  SlotView v{-1, -1, static_cast<int>(threadIdx.x)};
  if (static_cast<int>(threadIdx.x) < S) {
    v.bos = bos[threadIdx.x];
    v.lu = lu[threadIdx.x];
    if (v.bos >= 0 && v.bos < NB) v.chk = sob[v.bos];
  }
  return v;
}

// Plans one unit from the priority list P (shared memory, K ints).  Needs
// blockDim.x >= max(S, K).  All threads must call it.
static __device__ void plan_unit(const int* P, const SlotView v, int32_t step, int32_t* __restrict__ clock_u,
                          int32_t* __restrict__ sob, int32_t* __restrict__ bos,
                          int32_t* __restrict__ lu, int32_t* __restrict__ fetch_block,
                          int32_t* __restrict__ fetch_slot, int32_t* __restrict__ evict_block,
                          int32_t* __restrict__ n_fetch_u, int32_t* __restrict__ n_evict_u,
                          int NB, int S, int K, int cap, int capw, uint32_t* err, const PlanSmem& sm) {
  const int tid = threadIdx.x, T = blockDim.x;
  if (tid == 0) *sm.bad = 0;
  for (int w = tid; w < (NB + 31) / 32; w += T) sm.seen[w] = 0u;
  if (tid < S) sm.inp[tid] = 0;
  __syncthreads();
  // ids in range and distinct; both directions of the map agree
  int p = -1, sp = -1;
  if (tid < K) {
    p = P[tid];
    if (p < 0 || p >= NB) {
      atomicOr(sm.bad, OASIS_DEVERR_TOPK_IDS);
    } else {
      const unsigned bit = 1u << (p & 31);
      if (atomicOr(&sm.seen[p >> 5], bit) & bit) atomicOr(sm.bad, OASIS_DEVERR_TOPK_IDS);
      sp = sob[p];
    }
  }
  if (tid < S && (v.bos >= NB || (v.bos >= 0 && v.chk != tid)))
    atomicOr(sm.bad, OASIS_DEVERR_PLAN_STATE);
  if (tid < S) sm.bos[tid] = v.bos;
  __syncthreads();
  if (tid < K && sp >= 0 && (sp >= S || sm.bos[sp] != p)) atomicOr(sm.bad, OASIS_DEVERR_PLAN_STATE);
  __syncthreads();
  const int bad = *sm.bad;
  if (bad) {
    if (tid == 0) {
      set_error(err, static_cast<uint32_t>(bad));
      *n_fetch_u = 0;
      *n_evict_u = 0;
      if (clock_u) *clock_u = step + 1;
    }
    for (int r = tid; r < capw; r += T) {
      fetch_block[r] = -1;
      fetch_slot[r] = -1;
      evict_block[r] = -1;
    }
    return;
  }
  // 1. predicted blocks already resident are used at `step`
  if (tid < K && sp >= 0) sm.inp[sp] = 1;
  // 2. the first n misses in priority order are fetched
  const int miss = (tid < K) && sp < 0;
  int nmiss;
  const int mrank = block_exclusive_scan(miss, sm.scan, &nmiss);  // its barriers publish inp
  const int n = nmiss < cap ? nmiss : cap;
  if (miss && mrank < n) sm.fetch[mrank] = p;
  // 3. LRU victims among residents outside the prediction
  const bool resident = tid < S && v.bos >= 0;
  const bool cand = resident && sm.inp[tid] == 0;
  const int nres = __syncthreads_count(resident);
  int e = nres + n - S;
  if (e < 0) e = 0;
  unsigned long long mykey = ~0ull;
  if (cand)
    mykey = (static_cast<unsigned long long>(static_cast<uint32_t>(v.lu) ^ 0x80000000u) << 32) |
            static_cast<uint32_t>(v.bos);
  if (tid < S) sm.lru_key[tid] = mykey;
  __syncthreads();
  int victim = 0;
  if (cand && e > 0) {
    int rank = 0;
#pragma unroll 8
    for (int s2 = 0; s2 < S; ++s2) rank += sm.lru_key[s2] < mykey;
    if (rank < e) {
      victim = 1;
      sm.victim[rank] = v.bos;
    }
  }
  // 4. free slots (empty or freed) in ascending order
  const int is_free = (tid < S) && (v.bos < 0 || victim);
  int nfree;
  const int frank = block_exclusive_scan(is_free, sm.scan, &nfree);
  if (is_free && frank < n) sm.free_slot[frank] = tid;
  __syncthreads();
  // fetched blocks in ascending id take the free slots in ascending order
  int my_blk = -1, my_slot = -1;
  if (tid < n) {
    my_blk = sm.fetch[tid];
    int r = 0;
    for (int i = 0; i < n; ++i) r += sm.fetch[i] < my_blk;
    my_slot = sm.free_slot[r];
    fetch_block[r] = my_blk;
    fetch_slot[r] = my_slot;
  }
  if (tid < e) {
    const int vb = sm.victim[tid];
    int r = 0;
    for (int i = 0; i < e; ++i) r += sm.victim[i] < vb;
    evict_block[r] = vb;
  }
  for (int r = tid; r < capw; r += T) {
    if (r >= n) {
      fetch_block[r] = -1;
      fetch_slot[r] = -1;
    }
    if (r >= e) evict_block[r] = -1;
  }
  // apply: victims leave, fetched blocks enter; predicted residents are used now
  int new_bos = v.bos, new_lu = (tid < S && sm.inp[tid]) ? step : v.lu;
  if (victim) {
    sob[v.bos] = -1;
    new_bos = -1;
  }
  if (tid < S) {
    sm.bos[tid] = new_bos;
    sm.lu[tid] = new_lu;
  }
  __syncthreads();
  if (tid < n) {
    sm.bos[my_slot] = my_blk;
    sm.lu[my_slot] = step;
    sob[my_blk] = my_slot;
  }
  __syncthreads();
  if (tid < S) {
    bos[tid] = sm.bos[tid];
    lu[tid] = sm.lu[tid];
  }
  if (tid == 0) {
    *n_fetch_u = n;
    *n_evict_u = e;
    if (clock_u) *clock_u = step + 1;
  }
}

// Threads per CTA: 256 unless the slots, the list or the scores (at most 32
// per thread in registers, 16 where possible) need more.
inline int pred_threads(int need, int NB) {
  int t = 256;
  while (t < kPredThreads && (t < need || (NB + t - 1) / t > 16)) t *= 2;
  return t;
}

inline PredLayout pred_layout(const Shape& s) {
  PredLayout lay;
  lay.K = s.K;
  lay.S = s.S;
  lay.NB = s.NB;
  lay.capw = s.cap > 0 ? s.cap : 1;
  return lay;
}

}  // namespace oasis
