"""CPU oracle for the OasisKV decode hot path -- TEST INFRASTRUCTURE ONLY.

A thin ctypes wrapper over ``oasis_oracle.c`` (plain single-threaded C,
double accumulation).  Only the tests, the package smoke check and the
benchmark's CPU-baseline leg may import this package.  The GPU library does
not import, link or call it, and it imports nothing from the GPU library.

Arrays are numpy: bf16 tensors travel as uint16 bit patterns, layouts are
the ones documented in ``oasis_oracle.h``.  Configurations are plain dicts
with the fields of ``orc_cfg``.

Method source: "OasisKV: Scaling In-Decode KV Cache Beyond HBM with Lookahead
Sparse Prefetching" (arXiv:2608.08097 summary page); each C function cites the
figure, table or step of the page it follows.

Parity unpinned: multi-step trajectories (``Stepper`` run over many steps).
Each step's functions are pinned on their own; the page prints no trajectory
that would pin the chain of steps as a whole.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oasis_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboasis_oracle.so")
_lock = threading.Lock()
_lib = None


class OrcCfg(C.Structure):
    _fields_ = [("batch", C.c_int32), ("num_q_heads", C.c_int32), ("num_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("block_size", C.c_int32), ("num_blocks", C.c_int32),
                ("kv_budget_tokens", C.c_int32), ("lookahead", C.c_int32), ("top_k", C.c_int32),
                ("fetch_ratio", C.c_float), ("sink_blocks", C.c_int32), ("local_blocks", C.c_int32)]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (a checker, not part of the product)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "oasis_oracle.h"))):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-Wall", "-shared", "-fPIC",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = C.CDLL(_LIB_PATH)
            P = C.c_void_p
            cfgp = C.POINTER(OrcCfg)
            sig = {
                "orc_check_cfg": (C.c_int, [cfgp]),
                "orc_fetch_cap": (C.c_int, [cfgp]),
                "orc_build_summaries": (None, [cfgp, P, P]),
                "orc_score_blocks": (None, [cfgp, P, P, P]),
                "orc_build_summaries_minmax": (None, [cfgp, P, P]),
                "orc_score_blocks_minmax": (None, [cfgp, P, P, P]),
                "orc_select_topk": (C.c_int, [cfgp, P, P]),
                "orc_select_topk_ctx": (C.c_int, [cfgp, P, P, P]),
                "orc_append_kv": (C.c_int, [cfgp, P, P, P, P, C.c_int32, P, P, P, P, P, P, P]),
                "orc_refresh_summaries": (None, [cfgp, P, P, P, P]),
                "orc_plan_fetch": (C.c_int, [cfgp, P, C.c_int32, P, P, P, P, P, P, P, P]),
                "orc_fetch_blocks": (C.c_int, [cfgp, P, P, P, P, P, P, P]),
                "orc_sparse_decode_attn": (None, [cfgp, P, P, P, P, P, C.c_double, P]),
                "orc_dense_decode_attn": (None, [cfgp, P, P, P, P, C.c_double, P]),
            }
            for name, (res, args) in sig.items():
                f = getattr(_lib, name)
                f.restype = res
                f.argtypes = args
    return _lib


class using_library:
    """Context manager: route every call to another build of the oracle
    (used by the test that checks the pins catch planted mistakes)."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        lib()
        self.saved = _lib
        other = C.CDLL(self.path)
        for name in ("orc_check_cfg", "orc_fetch_cap", "orc_build_summaries", "orc_score_blocks",
                     "orc_select_topk", "orc_plan_fetch", "orc_fetch_blocks",
                     "orc_sparse_decode_attn", "orc_dense_decode_attn"):
            f, g = getattr(other, name), getattr(self.saved, name)
            f.restype, f.argtypes = g.restype, g.argtypes
        _lib = other
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def _cfg(cfg: dict) -> OrcCfg:
    c = OrcCfg(**{k: cfg[k] for k, _ in OrcCfg._fields_})
    rc = lib().orc_check_cfg(C.byref(c))
    if rc != 0:
        raise ValueError(f"oracle: inconsistent configuration (code {rc}): {cfg}")
    return c


def _p(a: np.ndarray, dtype) -> C.c_void_p:
    if a.dtype != dtype or not a.flags.c_contiguous:
        raise TypeError(f"oracle: expected C-contiguous {np.dtype(dtype)}, got {a.dtype}")
    return C.c_void_p(a.ctypes.data)


def _sizes(cfg):
    B, H, Hq = cfg["batch"], cfg["num_kv_heads"], cfg["num_q_heads"]
    NB, bs, D = cfg["num_blocks"], cfg["block_size"], cfg["head_dim"]
    S = cfg["kv_budget_tokens"] // bs
    return B, H, Hq, NB, bs, D, S


def _check(a, shape, name):
    if tuple(a.shape) != tuple(shape):
        raise ValueError(f"oracle: {name} has shape {a.shape}, expected {shape}")


def fetch_cap(cfg: dict) -> int:
    return int(lib().orc_fetch_cap(C.byref(_cfg(cfg))))


def build_summaries(cfg: dict, k: np.ndarray) -> np.ndarray:
    B, H, Hq, NB, bs, D, S = _sizes(cfg)
    _check(k, (B, H, NB, bs, D), "k")
    out = np.empty((B, H, NB, D), dtype=np.float32)
    lib().orc_build_summaries(C.byref(_cfg(cfg)), _p(k, np.uint16), _p(out, np.float32))
    return out


def score_blocks(cfg: dict, q_draft: np.ndarray, summ: np.ndarray) -> np.ndarray:
    B, H, Hq, NB, bs, D, S = _sizes(cfg)
    _check(q_draft, (B, cfg["lookahead"], Hq, D), "q_draft")
    _check(summ, (B, H, NB, D), "summ")
    out = np.empty((B, H, NB), dtype=np.float32)
    lib().orc_score_blocks(C.byref(_cfg(cfg)), _p(q_draft, np.uint16), _p(summ, np.float32),
                           _p(out, np.float32))
    return out


def build_summaries_minmax(cfg: dict, k: np.ndarray) -> np.ndarray:
    """[B, H, NB, 2, D] bf16 bits: per block the elementwise max (row 0) and
    min (row 1) of its keys."""
    B, H, Hq, NB, bs, D, S = _sizes(cfg)
    _check(k, (B, H, NB, bs, D), "k")
    out = np.empty((B, H, NB, 2, D), dtype=np.uint16)
    lib().orc_build_summaries_minmax(C.byref(_cfg(cfg)), _p(k, np.uint16), _p(out, np.uint16))
    return out


def score_blocks_minmax(cfg: dict, q_draft: np.ndarray, summ_mm: np.ndarray) -> np.ndarray:
    B, H, Hq, NB, bs, D, S = _sizes(cfg)
    _check(q_draft, (B, cfg["lookahead"], Hq, D), "q_draft")
    _check(summ_mm, (B, H, NB, 2, D), "summ_mm")
    out = np.empty((B, H, NB), dtype=np.float32)
    lib().orc_score_blocks_minmax(C.byref(_cfg(cfg)), _p(q_draft, np.uint16),
                                  _p(summ_mm, np.uint16), _p(out, np.float32))
    return out


def select_topk(cfg: dict, scores: np.ndarray) -> np.ndarray:
    B, H, Hq, NB, bs, D, S = _sizes(cfg)
    _check(scores, (B, H, NB), "scores")
    out = np.empty((B, H, cfg["top_k"]), dtype=np.int32)
    rc = lib().orc_select_topk(C.byref(_cfg(cfg)), _p(scores, np.float32), _p(out, np.int32))
    if rc != 0:
        raise ValueError(f"oracle: select_topk failed (code {rc})")
    return out


def select_topk_ctx(cfg: dict, scores: np.ndarray, ctx_len: np.ndarray) -> np.ndarray:
    """Top-K over a growing context: blocks past ceil(ctx_len/bs) rank last,
    the local window ends at the context's last block."""
    B, H, Hq, NB, bs, D, S = _sizes(cfg)
    _check(scores, (B, H, NB), "scores")
    cl = np.ascontiguousarray(ctx_len, dtype=np.int32)
    _check(cl, (B,), "ctx_len")
    out = np.empty((B, H, cfg["top_k"]), dtype=np.int32)
    rc = lib().orc_select_topk_ctx(C.byref(_cfg(cfg)), _p(scores, np.float32), _p(cl, np.int32),
                                   _p(out, np.int32))
    if rc != 0:
        raise ValueError(f"oracle: select_topk_ctx failed (code {rc})")
    return out


def append_kv(cfg: dict, k_new, v_new, ctx_len, step, host_k, host_v, slot_of_block,
              block_of_slot, last_used, pool_k, pool_v, clock=None) -> int:
    """Appends one token per request, in place on every array passed (ctx_len
    included).  Returns the oracle's code: 0, -1 (a full context) or -2 (a
    head with no slot to give).  Summaries: refresh_summaries."""
    B, H, Hq, NB, bs, D, S = _sizes(cfg)
    _check(k_new, (B, H, D), "k_new")
    _check(v_new, (B, H, D), "v_new")
    _check(ctx_len, (B,), "ctx_len")
    _check(host_k, (B, H, NB, bs, D), "host_k")
    _check(host_v, (B, H, NB, bs, D), "host_v")
    _check(slot_of_block, (B, H, NB), "slot_of_block")
    _check(block_of_slot, (B, H, S), "block_of_slot")
    _check(last_used, (B, H, S), "last_used")
    _check(pool_k, (B, H, S, bs, D), "pool_k")
    _check(pool_v, (B, H, S, bs, D), "pool_v")
    ck = None
    if clock is not None:
        _check(clock, (B, H), "clock")
        ck = _p(clock, np.int32)
    return int(lib().orc_append_kv(
        C.byref(_cfg(cfg)), _p(k_new, np.uint16), _p(v_new, np.uint16), _p(ctx_len, np.int32), ck,
        int(step), _p(host_k, np.uint16), _p(host_v, np.uint16), _p(slot_of_block, np.int32),
        _p(block_of_slot, np.int32), _p(last_used, np.int32), _p(pool_k, np.uint16),
        _p(pool_v, np.uint16)))


def refresh_summaries(cfg: dict, ctx_len, host_k, summ, summ_mm=None) -> None:
    """Recomputes, in place, the summaries of each context's newest block over
    its rows inside the context."""
    B, H, Hq, NB, bs, D, S = _sizes(cfg)
    _check(ctx_len, (B,), "ctx_len")
    _check(host_k, (B, H, NB, bs, D), "host_k")
    _check(summ, (B, H, NB, D), "summ")
    mm = None
    if summ_mm is not None:
        _check(summ_mm, (B, H, NB, 2, D), "summ_mm")
        mm = _p(summ_mm, np.uint16)
    lib().orc_refresh_summaries(C.byref(_cfg(cfg)), _p(ctx_len, np.int32), _p(host_k, np.uint16),
                                _p(summ, np.float32), mm)


def plan_fetch(cfg: dict, topk_ids: np.ndarray, step: int, slot_of_block: np.ndarray,
               block_of_slot: np.ndarray, last_used: np.ndarray) -> dict:
    """Runs one planning step.  The three state arrays are updated in place."""
    B, H, Hq, NB, bs, D, S = _sizes(cfg)
    _check(topk_ids, (B, H, cfg["top_k"]), "topk_ids")
    _check(slot_of_block, (B, H, NB), "slot_of_block")
    _check(block_of_slot, (B, H, S), "block_of_slot")
    _check(last_used, (B, H, S), "last_used")
    capw = max(fetch_cap(cfg), 1)
    fb = np.empty((B, H, capw), dtype=np.int32)
    fs = np.empty_like(fb)
    eb = np.empty_like(fb)
    nf = np.empty((B, H), dtype=np.int32)
    ne = np.empty_like(nf)
    rc = lib().orc_plan_fetch(C.byref(_cfg(cfg)), _p(topk_ids, np.int32), int(step),
                              _p(slot_of_block, np.int32), _p(block_of_slot, np.int32),
                              _p(last_used, np.int32), _p(fb, np.int32), _p(fs, np.int32),
                              _p(eb, np.int32), _p(nf, np.int32), _p(ne, np.int32))
    if rc != 0:
        raise ValueError(f"oracle: plan_fetch failed (code {rc})")
    return dict(fetch_block=fb, fetch_slot=fs, evict_block=eb, n_fetch=nf, n_evict=ne)


def fetch_blocks(cfg: dict, host_k, host_v, fetch_block, fetch_slot, n_fetch, pool_k, pool_v):
    """Copies the planned blocks into the pools (in place)."""
    rc = lib().orc_fetch_blocks(C.byref(_cfg(cfg)), _p(host_k, np.uint16), _p(host_v, np.uint16),
                                _p(fetch_block, np.int32), _p(fetch_slot, np.int32),
                                _p(n_fetch, np.int32), _p(pool_k, np.uint16), _p(pool_v, np.uint16))
    if rc != 0:
        raise ValueError(f"oracle: fetch_blocks failed (code {rc})")


def sparse_decode_attn(cfg: dict, q, pool_k, pool_v, block_of_slot, ctx_len=None,
                       scale: float | None = None) -> np.ndarray:
    B, H, Hq, NB, bs, D, S = _sizes(cfg)
    _check(q, (B, Hq, D), "q")
    _check(pool_k, (B, H, S, bs, D), "pool_k")
    _check(pool_v, (B, H, S, bs, D), "pool_v")
    _check(block_of_slot, (B, H, S), "block_of_slot")
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    cl = None
    if ctx_len is not None:
        ctx_keep = np.ascontiguousarray(ctx_len, dtype=np.int32)
        cl = _p(ctx_keep, np.int32)
    out = np.empty((B, Hq, D), dtype=np.float32)
    lib().orc_sparse_decode_attn(C.byref(_cfg(cfg)), _p(q, np.uint16), _p(pool_k, np.uint16),
                                 _p(pool_v, np.uint16), _p(block_of_slot, np.int32), cl,
                                 float(scale), _p(out, np.float32))
    return out


def sparse_decode_attn_joint(cfg: dict, q, q_draft, pool_k, pool_v, block_of_slot, ctx_len=None,
                             scale: float | None = None) -> np.ndarray:
    """Attention of the decoded token and of each draft token over the same
    working set ([OasisKV] Fig. 7 right: the attention kernel takes the normal
    and the draft queries together).  Reading: every one of the 1 + L query
    rows sees the same resident slots under the same context mask, since the
    draft tokens' own keys are not in the cache.  Output [B, 1+L, Hq, D]
    fp32: row 0 from q, row l from q_draft[:, l-1]."""
    B, H, Hq, NB, bs, D, S = _sizes(cfg)
    L = cfg["lookahead"]
    _check(q_draft, (B, L, Hq, D), "q_draft")
    rows = [q] + [np.ascontiguousarray(q_draft[:, l]) for l in range(L)]
    return np.stack([sparse_decode_attn(cfg, r, pool_k, pool_v, block_of_slot, ctx_len, scale)
                     for r in rows], axis=1)


def dense_decode_attn(cfg: dict, q, k, v, ctx_len=None, scale: float | None = None) -> np.ndarray:
    B, H, Hq, NB, bs, D, S = _sizes(cfg)
    _check(q, (B, Hq, D), "q")
    _check(k, (B, H, NB, bs, D), "k")
    _check(v, (B, H, NB, bs, D), "v")
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    cl = None
    if ctx_len is not None:
        ctx_keep = np.ascontiguousarray(ctx_len, dtype=np.int32)
        cl = _p(ctx_keep, np.int32)
    out = np.empty((B, Hq, D), dtype=np.float32)
    lib().orc_dense_decode_attn(C.byref(_cfg(cfg)), _p(q, np.uint16), _p(k, np.uint16),
                                _p(v, np.uint16), cl, float(scale), _p(out, np.float32))
    return out


def unit_cfg(cfg: dict) -> dict:
    """Configuration of a single (request, KV head) unit of `cfg`."""
    G = cfg["num_q_heads"] // cfg["num_kv_heads"]
    return dict(cfg, batch=1, num_kv_heads=1, num_q_heads=G)


class Stepper:
    """Runs the whole hot path of one layer-step on the CPU, step by step.

    Order of one layer-step t: attention over the current working set with
    q_t, then scoring with the draft queries, top-K, planning at step t and
    the transfer that produces the next working set ([OasisKV] Fig. 8: the
    draft query of step t drives prediction, selection and transfer before
    the same layer's attention at step t+1).  Parity unpinned over many
    steps: only the per-step functions it calls are pinned.
    """

    def __init__(self, cfg, host_k, host_v, summ, slot_of_block, block_of_slot, last_used,
                 pool_k, pool_v, ctx_len=None, scale=None):
        self.cfg = cfg
        self.host_k, self.host_v, self.summ = host_k, host_v, summ
        self.sob, self.bos, self.lu = slot_of_block, block_of_slot, last_used
        self.pool_k, self.pool_v = pool_k, pool_v
        self.ctx_len, self.scale = ctx_len, scale

    def step(self, t, q, q_draft):
        out = sparse_decode_attn(self.cfg, q, self.pool_k, self.pool_v, self.bos, self.ctx_len, self.scale)
        scores = score_blocks(self.cfg, q_draft, self.summ)
        topk = select_topk(self.cfg, scores)
        plan = plan_fetch(self.cfg, topk, t, self.sob, self.bos, self.lu)
        fetch_blocks(self.cfg, self.host_k, self.host_v, plan["fetch_block"], plan["fetch_slot"],
                     plan["n_fetch"], self.pool_k, self.pool_v)
        return dict(out=out, scores=scores, topk=topk, **plan)
