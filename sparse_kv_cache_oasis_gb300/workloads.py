"""Synthetic decode workloads and their seeded input generators.

This module holds shapes, seeds and random inputs only -- none of the
method's arithmetic (no scoring, selection, planning or attention).  Both the
GPU library's tests and the CPU oracle's tests draw their inputs from here,
so the two sides always see the same bytes.

Every random array comes from its own numpy ``Philox`` stream, keyed by
``(seed, layer, tensor, request, kv_head)``; the result does not depend on the
number of threads used to fill it.  bf16 values are produced by
round-to-nearest-even from fp32 and handled as uint16 bit patterns.

Shapes follow the workloads of "OasisKV: Scaling In-Decode KV Cache Beyond HBM
with Lookahead Sparse Prefetching": a 2,048-token KV budget (Tab. 1 caption,
'What they did' item 4), fetch ratios of Tab. 2, Qwen3-8B / Qwen3-32B /
Llama-3.1-8B head shapes (Tab. 1, Fig. 2, Fig. 11), at 16K-128K contexts.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, replace

import numpy as np

# tensor ids of the random streams
_T_KEYS, _T_VALUES, _T_QUERIES, _T_RESIDENT, _T_STRUCT = 0, 1, 2, 3, 4

PLANTED_BLOCKS = 8        # planted blocks per (request, KV head) in the tiny workload
PLANT_SHIFT = 0.5         # shift of a planted key along the query direction
ZIPF_S = 1.1              # exponent of the heavy-hitter profile
WALK_SIGMA = 0.1          # per-step drift of the decode queries


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    ctx_tokens: int
    kv_budget_tokens: int
    lookahead: int
    top_k: int
    fetch_ratio: float
    seed: int
    head_dim: int = 128
    block_size: int = 16
    sink_blocks: int = 0
    local_blocks: int = 0
    layers: int = 1
    steps: int = 1
    structure: str = "walk"          # "planted" | "walk" | "zipf"
    key_std: float = 1.0 / math.sqrt(128.0)

    @property
    def num_blocks(self) -> int:
        return self.ctx_tokens // self.block_size

    @property
    def slots(self) -> int:
        return self.kv_budget_tokens // self.block_size

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def config(self) -> dict:
        """Fields of the per-layer configuration, in the order of the C structs."""
        return dict(batch=self.batch, num_q_heads=self.num_q_heads,
                    num_kv_heads=self.num_kv_heads, head_dim=self.head_dim,
                    block_size=self.block_size, num_blocks=self.num_blocks,
                    kv_budget_tokens=self.kv_budget_tokens, lookahead=self.lookahead,
                    top_k=self.top_k, fetch_ratio=float(self.fetch_ratio),
                    sink_blocks=self.sink_blocks, local_blocks=self.local_blocks)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# Tiny single-layer step: GQA 4, 4,096-token context, 8 planted blocks per
# KV head, budget 64 blocks, top-32, fetch cap 4 (= ratio 4/64).
TINY = Workload(name="tiny-gqa4-ctx4k", batch=1, num_q_heads=16, num_kv_heads=4,
                ctx_tokens=4096, kv_budget_tokens=64 * 16, lookahead=2, top_k=32,
                fetch_ratio=4.0 / 64.0, seed=1001, steps=1, structure="planted")

# Llama-3.1-8B-shaped decode layer: 32 q / 8 KV heads, batch 8, 32K context,
# 2,048-token budget, L=4, top-128, ratio 0.05, 20 random-walk decode steps.
LLAMA8B_LAYER = Workload(name="llama3.1-8b-layer-ctx32k-b8", batch=8, num_q_heads=32,
                         num_kv_heads=8, ctx_tokens=32768, kv_budget_tokens=2048,
                         lookahead=4, top_k=128, fetch_ratio=0.05, seed=1002, steps=20,
                         structure="walk")

# Qwen3-8B-shaped full decode step: 36 layers, batch 32, 32K context, keys
# N(0,1) with Zipf(1.1) heavy-hitter blocks, 64 steps.
QWEN3_8B_STEP = Workload(name="qwen3-8b-36layer-ctx32k-b32", batch=32, num_q_heads=32,
                         num_kv_heads=8, ctx_tokens=32768, kv_budget_tokens=2048,
                         lookahead=4, top_k=128, fetch_ratio=0.05, seed=1003, layers=36,
                         steps=64, structure="zipf", key_std=1.0)

# Long context: 8 layers of Qwen3-32B shape (64 q / 8 KV heads), batch 8,
# 131,072-token context, ratio 0.02, sink block 0 and the last 4 blocks forced.
LONG_CTX = Workload(name="qwen3-32b-8layer-ctx128k-b8", batch=8, num_q_heads=64,
                    num_kv_heads=8, ctx_tokens=131072, kv_budget_tokens=2048, lookahead=4,
                    top_k=128, fetch_ratio=0.02, seed=1004, sink_blocks=1, local_blocks=4,
                    layers=8, steps=20, structure="walk")

# Fetch-ratio x batch sweep on the Qwen3-8B layer shape (Tab. 2 columns).
SWEEP_RATIOS = (0.01, 0.02, 0.05, 0.10, 0.20, -1.0)   # -1: fetch all
SWEEP_BATCHES = (1, 8, 32, 64)


def sweep_point(ratio: float, batch: int) -> Workload:
    tag = "all" if ratio < 0 else f"{ratio:.2f}"
    return Workload(name=f"qwen3-8b-layer-sweep-r{tag}-b{batch}", batch=batch,
                    num_q_heads=32, num_kv_heads=8, ctx_tokens=32768,
                    kv_budget_tokens=2048, lookahead=4, top_k=128, fetch_ratio=ratio,
                    seed=1005, steps=32, structure="walk")


PRESETS = {w.name: w for w in (TINY, LLAMA8B_LAYER, QWEN3_8B_STEP, LONG_CTX)}


# --------------------------------------------------------------------------
# random streams and bf16 bit patterns
# --------------------------------------------------------------------------
def rng(seed: int, layer: int, tensor: int, b: int = 0, h: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, layer, tensor, b, h])))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


# --------------------------------------------------------------------------
# queries
# --------------------------------------------------------------------------
def query_sequence(wl: Workload, layer: int = 0) -> np.ndarray:
    """fp32 queries [T, B, Hq, D] with T = steps + lookahead + 1.

    "walk"/"zipf": q_0 ~ N(0,1)/sqrt(D); q_{t+1} = q_t + sigma * N(0,1)/sqrt(D)
    with sigma = 0.1.  "planted": T independent N(0,1)/sqrt(D) draws.
    The decode query of step t is q_t; its draft queries are q_{t+1..t+L}.
    """
    T = wl.steps + wl.lookahead + 1
    D = wl.head_dim
    out = np.empty((T, wl.batch, wl.num_q_heads, D), dtype=np.float32)
    for b in range(wl.batch):
        g = rng(wl.seed, layer, _T_QUERIES, b)
        eps = g.standard_normal((T, wl.num_q_heads, D)) / math.sqrt(D)
        if wl.structure == "planted":
            seq = eps
        else:
            seq = np.empty_like(eps)
            seq[0] = eps[0]
            for t in range(1, T):
                seq[t] = seq[t - 1] + WALK_SIGMA * eps[t]
        out[:, b] = seq.astype(np.float32)
    return out


def step_queries(wl: Workload, qseq: np.ndarray, step: int):
    """(q [B,Hq,D], q_draft [B,L,Hq,D]) as bf16 bit patterns for one step."""
    q = to_bf16_bits(qseq[step])
    qd = to_bf16_bits(np.ascontiguousarray(qseq[step + 1:step + 1 + wl.lookahead].transpose(1, 0, 2, 3)))
    return q, qd


def query_direction(wl: Workload, qseq: np.ndarray) -> np.ndarray:
    """u[b,h]: unit vector of the mean of the G*L step-0 draft queries of KV head h."""
    G, L = wl.group, wl.lookahead
    dr = qseq[1:1 + L].astype(np.float64)                       # [L, B, Hq, D]
    dr = dr.reshape(L, wl.batch, wl.num_kv_heads, G, wl.head_dim)
    m = dr.mean(axis=(0, 3))                                    # [B, Hkv, D]
    return (m / np.linalg.norm(m, axis=-1, keepdims=True)).astype(np.float32)


# --------------------------------------------------------------------------
# keys and values of the full (host) cache
# --------------------------------------------------------------------------
def planted_blocks(wl: Workload, layer: int, b: int, h: int) -> np.ndarray:
    g = rng(wl.seed, layer, _T_STRUCT, b, h)
    return np.sort(g.choice(wl.num_blocks, size=PLANTED_BLOCKS, replace=False)).astype(np.int32)


def zipf_ranking(wl: Workload, layer: int, b: int, h: int) -> np.ndarray:
    """Block at position r-1 of the returned permutation has heavy-hitter rank r."""
    return rng(wl.seed, layer, _T_STRUCT, b, h).permutation(wl.num_blocks).astype(np.int32)


def _fill_unit(wl, layer, tensor, b, h, u_bh, out_unit):
    NB, bs, D = wl.num_blocks, wl.block_size, wl.head_dim
    g = rng(wl.seed, layer, tensor, b, h)
    x = g.standard_normal((NB, bs, D), dtype=np.float32)
    if tensor == _T_KEYS:
        x *= np.float32(wl.key_std)
        if wl.structure == "planted":
            x[planted_blocks(wl, layer, b, h)] += np.float32(PLANT_SHIFT) * u_bh
        elif wl.structure == "zipf":
            perm = zipf_ranking(wl, layer, b, h)
            w = (PLANT_SHIFT * np.arange(1, NB + 1, dtype=np.float64) ** (-ZIPF_S)).astype(np.float32)
            x[perm] += w[:, None, None] * u_bh[None, None, :]
    else:
        x *= np.float32(1.0 / math.sqrt(D))
    out_unit[...] = to_bf16_bits(x)


def gen_kv(wl: Workload, layer: int = 0, qseq: np.ndarray | None = None,
           out_k: np.ndarray | None = None, out_v: np.ndarray | None = None):
    """Host cache K and V, bf16 bit patterns [B, Hkv, NB, bs, D] each.

    Values are N(0,1)/sqrt(D).  Keys are N(0,1) * key_std, plus the
    workload's structure along u[b,h] (query_direction): "planted" shifts every
    key of PLANTED_BLOCKS seeded blocks by 0.5*u; "zipf" shifts every key of
    the block of heavy-hitter rank r by 0.5 * r**-1.1 * u.
    """
    if qseq is None:
        qseq = query_sequence(wl, layer)
    u = query_direction(wl, qseq)
    shape = (wl.batch, wl.num_kv_heads, wl.num_blocks, wl.block_size, wl.head_dim)
    k = np.empty(shape, dtype=np.uint16) if out_k is None else out_k
    v = np.empty(shape, dtype=np.uint16) if out_v is None else out_v
    jobs = []
    with ThreadPoolExecutor(_threads()) as ex:
        for b in range(wl.batch):
            for h in range(wl.num_kv_heads):
                jobs.append(ex.submit(_fill_unit, wl, layer, _T_KEYS, b, h, u[b, h], k[b, h]))
                jobs.append(ex.submit(_fill_unit, wl, layer, _T_VALUES, b, h, None, v[b, h]))
        for j in jobs:
            j.result()
    return k, v


# --------------------------------------------------------------------------
# initial working set
# --------------------------------------------------------------------------
def initial_resident(wl: Workload, layer: int = 0):
    """(slot_of_block [B,Hkv,NB], block_of_slot [B,Hkv,S], last_used [B,Hkv,S]).

    min(S, NB) distinct seeded blocks per (request, KV head), forced blocks
    (sink and local window) first, in seeded slot order; last_used = -1.
    """
    B, H, NB, S = wl.batch, wl.num_kv_heads, wl.num_blocks, wl.slots
    sob = np.full((B, H, NB), -1, dtype=np.int32)
    bos = np.full((B, H, S), -1, dtype=np.int32)
    lu = np.full((B, H, S), -1, dtype=np.int32)
    forced = [j for j in range(NB) if j < wl.sink_blocks or j >= NB - wl.local_blocks]
    nres = min(S, NB)
    for b in range(B):
        for h in range(H):
            g = rng(wl.seed, layer, _T_RESIDENT, b, h)
            others = np.setdiff1d(np.arange(NB), np.asarray(forced, dtype=np.int64))
            pick = g.choice(others, size=nres - len(forced), replace=False)
            chosen = np.concatenate([np.asarray(forced, dtype=np.int64), pick])
            slots = g.permutation(S)[:nres]
            bos[b, h, slots] = chosen
            sob[b, h, chosen] = slots
    return sob, bos, lu


def initial_pool(wl: Workload, k: np.ndarray, v: np.ndarray, block_of_slot: np.ndarray):
    """Working-set pools [B,Hkv,S,bs,D] holding the initially resident blocks (zeros in empty slots)."""
    B, H, S = block_of_slot.shape
    shape = (B, H, S, wl.block_size, wl.head_dim)
    pk = np.zeros(shape, dtype=np.uint16)
    pv = np.zeros(shape, dtype=np.uint16)
    for b in range(B):
        for h in range(H):
            sel = block_of_slot[b, h]
            ok = sel >= 0
            pk[b, h, ok] = k[b, h, sel[ok]]
            pv[b, h, ok] = v[b, h, sel[ok]]
    return pk, pv
