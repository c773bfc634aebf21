"""ctypes binding of liboasis (include/oasis.h), one Python function per C entry point.

Argument marshalling only: shapes, dtypes, devices and contiguity of torch
tensors are checked, raw pointers and the current CUDA stream are passed to
the C function, and a non-OK status raises OasisError.  Every computation
runs in the library's CUDA kernels; there is no fallback: if liboasis.so is
missing or CUDA is unavailable, the call raises.
"""
from __future__ import annotations

import ctypes as C
import os
import re
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liboasis.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "oasis.h")

OASIS_OK, OASIS_ERR_INVALID_ARG, OASIS_ERR_UNSUPPORTED, OASIS_ERR_CUDA, OASIS_ERR_TIMEOUT = range(5)
DEVERR_FETCH_RANGE, DEVERR_PLAN_STATE, DEVERR_TOPK_IDS, DEVERR_WAIT_TIMEOUT, DEVERR_SLOT_RANGE = (
    0x1, 0x2, 0x4, 0x8, 0x10)
DEVERR_CTX_FULL, DEVERR_NO_SLOT = 0x20, 0x40


class OasisError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {_status_name(status)}")


class OasisConfig(C.Structure):
    _fields_ = [("batch", C.c_int32), ("num_q_heads", C.c_int32), ("num_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("block_size", C.c_int32), ("num_blocks", C.c_int32),
                ("kv_budget_tokens", C.c_int32), ("lookahead", C.c_int32), ("top_k", C.c_int32),
                ("fetch_ratio", C.c_float), ("sink_blocks", C.c_int32), ("local_blocks", C.c_int32)]

    @classmethod
    def make(cls, cfg) -> "OasisConfig":
        if isinstance(cfg, OasisConfig):
            return cfg
        if not isinstance(cfg, dict):
            cfg = cfg.config()
        return cls(**{k: cfg[k] for k, _ in cls._fields_})

    def as_dict(self) -> dict:
        return {k: getattr(self, k) for k, _ in self._fields_}


_P = C.c_void_p
_SIGS = {
    "oasis_validate_config": (C.c_int, [C.POINTER(OasisConfig)]),
    "oasis_fetch_cap": (C.c_int32, [C.POINTER(OasisConfig)]),
    "oasis_build_summaries": (C.c_int, [C.POINTER(OasisConfig), _P, _P, _P]),
    "oasis_score_blocks": (C.c_int, [C.POINTER(OasisConfig), _P, _P, _P, _P]),
    "oasis_select_topk": (C.c_int, [C.POINTER(OasisConfig), _P, _P, _P]),
    "oasis_plan_fetch": (C.c_int, [C.POINTER(OasisConfig), _P, C.c_int32] + [_P] * 9),
    "oasis_plan_fetch_clocked": (C.c_int, [C.POINTER(OasisConfig)] + [_P] * 11),
    "oasis_predict_select": (C.c_int, [C.POINTER(OasisConfig), _P, C.c_int32] + [_P] * 11),
    "oasis_fetch_blocks": (C.c_int, [C.POINTER(OasisConfig)] + [_P] * 8),
    "oasis_sparse_decode_attn": (C.c_int, [C.POINTER(OasisConfig), _P, _P, _P, _P, _P, C.c_float,
                                           _P, _P, C.c_size_t, _P]),
    "oasis_attn_workspace_bytes": (C.c_size_t, [C.POINTER(OasisConfig)]),
    "oasis_sparse_decode_attn_static": (C.c_int, [C.POINTER(OasisConfig), _P, _P, _P, _P, _P,
                                                  C.c_float, _P, _P]),
    "oasis_attend_and_score": (C.c_int, [C.POINTER(OasisConfig), _P, _P, _P, _P, _P, C.c_float,
                                         _P, _P, _P, _P, _P]),
    "oasis_sparse_decode_attn_joint": (C.c_int, [C.POINTER(OasisConfig), _P, _P, _P, _P, _P, _P,
                                                 C.c_float, _P, _P]),
    "oasis_build_summaries_minmax": (C.c_int, [C.POINTER(OasisConfig), _P, _P, _P]),
    "oasis_score_blocks_minmax": (C.c_int, [C.POINTER(OasisConfig), _P, _P, _P, _P]),
    "oasis_select_topk_ctx": (C.c_int, [C.POINTER(OasisConfig), _P, _P, _P, _P]),
    "oasis_predict_select_ctx": (C.c_int, [C.POINTER(OasisConfig), _P, _P, C.c_int32, _P, _P, _P,
                                           _P, _P, _P, _P, _P, _P, _P, _P]),
    "oasis_append_kv": (C.c_int, [C.POINTER(OasisConfig), _P, _P, _P, _P, C.c_int32, _P, _P, _P,
                                  _P, _P, _P, _P, _P]),
    "oasis_refresh_summaries": (C.c_int, [C.POINTER(OasisConfig), _P, _P, _P, _P, _P, _P, _P]),
    "oasis_predict_chain": (C.c_int, [C.POINTER(OasisConfig), _P, _P, _P, C.c_int32, _P, _P, _P,
                                      _P, _P, _P, _P, _P, _P, _P, _P]),
    "oasis_attend_and_score_minmax": (C.c_int, [C.POINTER(OasisConfig), _P, _P, _P, _P, _P,
                                                C.c_float, _P, _P, _P, _P, _P]),
    "oasis_host_register": (C.c_int, [_P, C.c_size_t, C.POINTER(C.c_void_p)]),
    "oasis_host_unregister": (C.c_int, [_P]),
    "oasis_device_errors": (C.c_int, [C.POINTER(C.c_uint32), C.c_int32]),
    "oasis_stream_wait": (C.c_int, [_P, C.c_int32]),
    "oasis_status_string": (C.c_char_p, [C.c_int]),
    "oasis_version": (C.c_int32, []),
}

_lib = None
_lock = threading.Lock()


def header_symbols() -> list[str]:
    """Names of the functions declared in include/oasis.h."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(oasis_[a-z_0-9]+)\s*\(", text)))


def lib() -> C.CDLL:
    """Loads liboasis.so (built by build.py); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise OSError(f"liboasis.so is not built ({LIB_PATH}); run "
                              "`python -m sparse_kv_cache_oasis_gb300.build`")
            handle = C.CDLL(LIB_PATH)
            for name, (res, args) in _SIGS.items():
                f = getattr(handle, name)
                f.restype = res
                f.argtypes = args
            _lib = handle
    return _lib


def _status_name(st: int) -> str:
    try:
        return lib().oasis_status_string(st).decode()
    except Exception:
        return f"status {st}"


def _check(fn: str, st: int) -> None:
    if st != OASIS_OK:
        raise OasisError(fn, st)


def _stream(stream) -> C.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return C.c_void_p(stream.cuda_stream)
    return C.c_void_p(int(stream))


def _ptr(t, dtype, shape, name, device=True):
    if isinstance(t, int):  # a raw address (e.g. mapped host memory)
        return C.c_void_p(t)
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor or an address")
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if device and t.device.type != "cuda":
        raise ValueError(f"{name}: must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    return C.c_void_p(t.data_ptr())


def _dims(c: OasisConfig):
    S = c.kv_budget_tokens // c.block_size
    return c.batch, c.num_kv_heads, c.num_q_heads, c.num_blocks, c.block_size, c.head_dim, S


# ------------------------------------------------------------------ entry points
def oasis_validate_config(cfg) -> int:
    return lib().oasis_validate_config(C.byref(OasisConfig.make(cfg)))


def oasis_fetch_cap(cfg) -> int:
    return int(lib().oasis_fetch_cap(C.byref(OasisConfig.make(cfg))))


def cap_width(cfg) -> int:
    cap = oasis_fetch_cap(cfg)
    if cap < 0:
        raise OasisError("oasis_fetch_cap", OASIS_ERR_INVALID_ARG)
    return max(cap, 1)


def oasis_build_summaries(cfg, k, summ, stream=None) -> None:
    c = OasisConfig.make(cfg)
    B, H, Hq, NB, bs, D, S = _dims(c)
    kp = _ptr(k, torch.bfloat16, (B, H, NB, bs, D), "k", device=False)
    sp = _ptr(summ, torch.float32, (B, H, NB, D), "summ")
    _check("oasis_build_summaries", lib().oasis_build_summaries(C.byref(c), kp, sp, _stream(stream)))


def oasis_score_blocks(cfg, q_draft, summ, scores, stream=None) -> None:
    c = OasisConfig.make(cfg)
    B, H, Hq, NB, bs, D, S = _dims(c)
    _check("oasis_score_blocks", lib().oasis_score_blocks(
        C.byref(c), _ptr(q_draft, torch.bfloat16, (B, c.lookahead, Hq, D), "q_draft"),
        _ptr(summ, torch.float32, (B, H, NB, D), "summ"),
        _ptr(scores, torch.float32, (B, H, NB), "scores"), _stream(stream)))


def oasis_build_summaries_minmax(cfg, k, summ_mm, stream=None) -> None:
    """Per-block elementwise max and min keys, [B, Hkv, NB, 2, D] bf16."""
    c = OasisConfig.make(cfg)
    B, H, Hq, NB, bs, D, S = _dims(c)
    kp = _ptr(k, torch.bfloat16, (B, H, NB, bs, D), "k", device=False)
    sp = _ptr(summ_mm, torch.bfloat16, (B, H, NB, 2, D), "summ_mm")
    _check("oasis_build_summaries_minmax",
           lib().oasis_build_summaries_minmax(C.byref(c), kp, sp, _stream(stream)))


def oasis_score_blocks_minmax(cfg, q_draft, summ_mm, scores, stream=None) -> None:
    c = OasisConfig.make(cfg)
    B, H, Hq, NB, bs, D, S = _dims(c)
    _check("oasis_score_blocks_minmax", lib().oasis_score_blocks_minmax(
        C.byref(c), _ptr(q_draft, torch.bfloat16, (B, c.lookahead, Hq, D), "q_draft"),
        _ptr(summ_mm, torch.bfloat16, (B, H, NB, 2, D), "summ_mm"),
        _ptr(scores, torch.float32, (B, H, NB), "scores"), _stream(stream)))


def oasis_select_topk(cfg, scores, topk_ids, stream=None) -> None:
    c = OasisConfig.make(cfg)
    B, H, Hq, NB, bs, D, S = _dims(c)
    _check("oasis_select_topk", lib().oasis_select_topk(
        C.byref(c), _ptr(scores, torch.float32, (B, H, NB), "scores"),
        _ptr(topk_ids, torch.int32, (B, H, c.top_k), "topk_ids"), _stream(stream)))


def oasis_plan_fetch(cfg, topk_ids, step, slot_of_block, block_of_slot, last_used, fetch_block,
                     fetch_slot, evict_block, n_fetch, n_evict, stream=None) -> None:
    c = OasisConfig.make(cfg)
    B, H, Hq, NB, bs, D, S = _dims(c)
    w = cap_width(c)
    i32 = torch.int32
    _check("oasis_plan_fetch", lib().oasis_plan_fetch(
        C.byref(c), _ptr(topk_ids, i32, (B, H, c.top_k), "topk_ids"), int(step),
        _ptr(slot_of_block, i32, (B, H, NB), "slot_of_block"),
        _ptr(block_of_slot, i32, (B, H, S), "block_of_slot"),
        _ptr(last_used, i32, (B, H, S), "last_used"),
        _ptr(fetch_block, i32, (B, H, w), "fetch_block"), _ptr(fetch_slot, i32, (B, H, w), "fetch_slot"),
        _ptr(evict_block, i32, (B, H, w), "evict_block"), _ptr(n_fetch, i32, (B, H), "n_fetch"),
        _ptr(n_evict, i32, (B, H), "n_evict"), _stream(stream)))


def oasis_plan_fetch_clocked(cfg, topk_ids, clock, slot_of_block, block_of_slot, last_used,
                             fetch_block, fetch_slot, evict_block, n_fetch, n_evict,
                             stream=None) -> None:
    c = OasisConfig.make(cfg)
    B, H, Hq, NB, bs, D, S = _dims(c)
    w = cap_width(c)
    i32 = torch.int32
    _check("oasis_plan_fetch_clocked", lib().oasis_plan_fetch_clocked(
        C.byref(c), _ptr(topk_ids, i32, (B, H, c.top_k), "topk_ids"),
        _ptr(clock, i32, (B, H), "clock"),
        _ptr(slot_of_block, i32, (B, H, NB), "slot_of_block"),
        _ptr(block_of_slot, i32, (B, H, S), "block_of_slot"),
        _ptr(last_used, i32, (B, H, S), "last_used"),
        _ptr(fetch_block, i32, (B, H, w), "fetch_block"), _ptr(fetch_slot, i32, (B, H, w), "fetch_slot"),
        _ptr(evict_block, i32, (B, H, w), "evict_block"), _ptr(n_fetch, i32, (B, H), "n_fetch"),
        _ptr(n_evict, i32, (B, H), "n_evict"), _stream(stream)))


def oasis_predict_select(cfg, scores, step, clock, topk_ids, slot_of_block, block_of_slot,
                         last_used, fetch_block, fetch_slot, evict_block, n_fetch, n_evict,
                         stream=None) -> None:
    """Top-K then plan in one launch; `clock` ([B, Hkv] int32 tensor) or None."""
    c = OasisConfig.make(cfg)
    B, H, Hq, NB, bs, D, S = _dims(c)
    w = cap_width(c)
    i32 = torch.int32
    ck = C.c_void_p(0) if clock is None else _ptr(clock, i32, (B, H), "clock")
    _check("oasis_predict_select", lib().oasis_predict_select(
        C.byref(c), _ptr(scores, torch.float32, (B, H, NB), "scores"), int(step), ck,
        _ptr(topk_ids, i32, (B, H, c.top_k), "topk_ids"),
        _ptr(slot_of_block, i32, (B, H, NB), "slot_of_block"),
        _ptr(block_of_slot, i32, (B, H, S), "block_of_slot"),
        _ptr(last_used, i32, (B, H, S), "last_used"),
        _ptr(fetch_block, i32, (B, H, w), "fetch_block"), _ptr(fetch_slot, i32, (B, H, w), "fetch_slot"),
        _ptr(evict_block, i32, (B, H, w), "evict_block"), _ptr(n_fetch, i32, (B, H), "n_fetch"),
        _ptr(n_evict, i32, (B, H), "n_evict"), _stream(stream)))


def oasis_predict_chain(cfg, q_draft, summ, scores, step, clock, topk_ids, slot_of_block,
                        block_of_slot, last_used, fetch_block, fetch_slot, evict_block, n_fetch,
                        n_evict, stream=None) -> None:
    """Scoring, top-K and plan in one launch; `clock` ([B, Hkv] int32) or None."""
    c = OasisConfig.make(cfg)
    B, H, Hq, NB, bs, D, S = _dims(c)
    w = cap_width(c)
    i32 = torch.int32
    ck = C.c_void_p(0) if clock is None else _ptr(clock, i32, (B, H), "clock")
    _check("oasis_predict_chain", lib().oasis_predict_chain(
        C.byref(c), _ptr(q_draft, torch.bfloat16, (B, c.lookahead, Hq, D), "q_draft"),
        _ptr(summ, torch.float32, (B, H, NB, D), "summ"),
        _ptr(scores, torch.float32, (B, H, NB), "scores"), int(step), ck,
        _ptr(topk_ids, i32, (B, H, c.top_k), "topk_ids"),
        _ptr(slot_of_block, i32, (B, H, NB), "slot_of_block"),
        _ptr(block_of_slot, i32, (B, H, S), "block_of_slot"),
        _ptr(last_used, i32, (B, H, S), "last_used"),
        _ptr(fetch_block, i32, (B, H, w), "fetch_block"), _ptr(fetch_slot, i32, (B, H, w), "fetch_slot"),
        _ptr(evict_block, i32, (B, H, w), "evict_block"), _ptr(n_fetch, i32, (B, H), "n_fetch"),
        _ptr(n_evict, i32, (B, H), "n_evict"), _stream(stream)))


def oasis_select_topk_ctx(cfg, scores, ctx_len, topk_ids, stream=None) -> None:
    """Top-K with the local window at each request's context end (ctx_len [B])."""
    c = OasisConfig.make(cfg)
    B, H, Hq, NB, bs, D, S = _dims(c)
    _check("oasis_select_topk_ctx", lib().oasis_select_topk_ctx(
        C.byref(c), _ptr(scores, torch.float32, (B, H, NB), "scores"),
        _ptr(ctx_len, torch.int32, (B,), "ctx_len"),
        _ptr(topk_ids, torch.int32, (B, H, c.top_k), "topk_ids"), _stream(stream)))


def oasis_predict_select_ctx(cfg, scores, ctx_len, step, clock, topk_ids, slot_of_block,
                             block_of_slot, last_used, fetch_block, fetch_slot, evict_block,
                             n_fetch, n_evict, stream=None) -> None:
    """oasis_predict_select over a growing context (ctx_len [B])."""
    c = OasisConfig.make(cfg)
    B, H, Hq, NB, bs, D, S = _dims(c)
    w = cap_width(c)
    i32 = torch.int32
    ck = C.c_void_p(0) if clock is None else _ptr(clock, i32, (B, H), "clock")
    _check("oasis_predict_select_ctx", lib().oasis_predict_select_ctx(
        C.byref(c), _ptr(scores, torch.float32, (B, H, NB), "scores"),
        _ptr(ctx_len, i32, (B,), "ctx_len"), int(step), ck,
        _ptr(topk_ids, i32, (B, H, c.top_k), "topk_ids"),
        _ptr(slot_of_block, i32, (B, H, NB), "slot_of_block"),
        _ptr(block_of_slot, i32, (B, H, S), "block_of_slot"),
        _ptr(last_used, i32, (B, H, S), "last_used"),
        _ptr(fetch_block, i32, (B, H, w), "fetch_block"), _ptr(fetch_slot, i32, (B, H, w), "fetch_slot"),
        _ptr(evict_block, i32, (B, H, w), "evict_block"), _ptr(n_fetch, i32, (B, H), "n_fetch"),
        _ptr(n_evict, i32, (B, H), "n_evict"), _stream(stream)))


def oasis_append_kv(cfg, k_new, v_new, ctx_len, step, clock, host_k, host_v, slot_of_block,
                    block_of_slot, last_used, pool_k, pool_v, stream=None) -> None:
    """Appends one token per request (k_new, v_new [B, Hkv, D] bf16) at
    ctx_len [B] and advances it.  host_k / host_v: device addresses of the
    mapped pinned cache (ints) or device tensors."""
    c = OasisConfig.make(cfg)
    B, H, Hq, NB, bs, D, S = _dims(c)
    i32, bf = torch.int32, torch.bfloat16
    ck = C.c_void_p(0) if clock is None else _ptr(clock, i32, (B, H), "clock")
    _check("oasis_append_kv", lib().oasis_append_kv(
        C.byref(c), _ptr(k_new, bf, (B, H, D), "k_new"), _ptr(v_new, bf, (B, H, D), "v_new"),
        _ptr(ctx_len, i32, (B,), "ctx_len"), ck, int(step),
        _ptr(host_k, bf, (B, H, NB, bs, D), "host_k", device=False),
        _ptr(host_v, bf, (B, H, NB, bs, D), "host_v", device=False),
        _ptr(slot_of_block, i32, (B, H, NB), "slot_of_block"),
        _ptr(block_of_slot, i32, (B, H, S), "block_of_slot"),
        _ptr(last_used, i32, (B, H, S), "last_used"),
        _ptr(pool_k, bf, (B, H, S, bs, D), "pool_k"), _ptr(pool_v, bf, (B, H, S, bs, D), "pool_v"),
        _stream(stream)))


def oasis_refresh_summaries(cfg, ctx_len, host_k, slot_of_block, pool_k, summ, summ_mm=None,
                            stream=None) -> None:
    """Summaries of each context's newest block over its rows in the context."""
    c = OasisConfig.make(cfg)
    B, H, Hq, NB, bs, D, S = _dims(c)
    bf = torch.bfloat16
    mm = C.c_void_p(0) if summ_mm is None else _ptr(summ_mm, bf, (B, H, NB, 2, D), "summ_mm")
    _check("oasis_refresh_summaries", lib().oasis_refresh_summaries(
        C.byref(c), _ptr(ctx_len, torch.int32, (B,), "ctx_len"),
        _ptr(host_k, bf, (B, H, NB, bs, D), "host_k", device=False),
        _ptr(slot_of_block, torch.int32, (B, H, NB), "slot_of_block"),
        _ptr(pool_k, bf, (B, H, S, bs, D), "pool_k"),
        _ptr(summ, torch.float32, (B, H, NB, D), "summ"), mm, _stream(stream)))


def oasis_fetch_blocks(cfg, host_k, host_v, fetch_block, fetch_slot, n_fetch, pool_k, pool_v,
                       stream=None) -> None:
    """host_k / host_v: device addresses of mapped pinned memory (ints), or
    pinned CPU tensors (their address is used directly, valid under UVA)."""
    c = OasisConfig.make(cfg)
    B, H, Hq, NB, bs, D, S = _dims(c)
    w = cap_width(c)
    i32 = torch.int32
    for name, t in (("host_k", host_k), ("host_v", host_v)):
        if isinstance(t, torch.Tensor) and t.device.type == "cpu" and not t.is_pinned():
            raise ValueError(f"{name}: host tensor must be pinned")
    _check("oasis_fetch_blocks", lib().oasis_fetch_blocks(
        C.byref(c), _ptr(host_k, torch.bfloat16, (B, H, NB, bs, D), "host_k", device=False),
        _ptr(host_v, torch.bfloat16, (B, H, NB, bs, D), "host_v", device=False),
        _ptr(fetch_block, i32, (B, H, w), "fetch_block"), _ptr(fetch_slot, i32, (B, H, w), "fetch_slot"),
        _ptr(n_fetch, i32, (B, H), "n_fetch"),
        _ptr(pool_k, torch.bfloat16, (B, H, S, bs, D), "pool_k"),
        _ptr(pool_v, torch.bfloat16, (B, H, S, bs, D), "pool_v"), _stream(stream)))


def oasis_attn_workspace_bytes(cfg) -> int:
    return int(lib().oasis_attn_workspace_bytes(C.byref(OasisConfig.make(cfg))))


def oasis_sparse_decode_attn(cfg, q, pool_k, pool_v, block_of_slot, ctx_len, scale, out,
                             workspace, stream=None) -> None:
    c = OasisConfig.make(cfg)
    B, H, Hq, NB, bs, D, S = _dims(c)
    ws = _ptr(workspace, torch.uint8, None, "workspace")
    nbytes = workspace.numel() if isinstance(workspace, torch.Tensor) else 0
    cl = None if ctx_len is None else _ptr(ctx_len, torch.int32, (B,), "ctx_len")
    _check("oasis_sparse_decode_attn", lib().oasis_sparse_decode_attn(
        C.byref(c), _ptr(q, torch.bfloat16, (B, Hq, D), "q"),
        _ptr(pool_k, torch.bfloat16, (B, H, S, bs, D), "pool_k"),
        _ptr(pool_v, torch.bfloat16, (B, H, S, bs, D), "pool_v"),
        _ptr(block_of_slot, torch.int32, (B, H, S), "block_of_slot"), cl, float(scale),
        _ptr(out, torch.bfloat16, (B, Hq, D), "out"), ws, nbytes, _stream(stream)))


def oasis_sparse_decode_attn_static(cfg, q, pool_k, pool_v, block_of_slot, ctx_len, scale, out,
                                    stream=None) -> None:
    """oasis_sparse_decode_attn without a workspace argument: the library's
    fixed device scratch is used instead, so the call allocates nothing."""
    c = OasisConfig.make(cfg)
    B, H, Hq, NB, bs, D, S = _dims(c)
    cl = None if ctx_len is None else _ptr(ctx_len, torch.int32, (B,), "ctx_len")
    _check("oasis_sparse_decode_attn_static", lib().oasis_sparse_decode_attn_static(
        C.byref(c), _ptr(q, torch.bfloat16, (B, Hq, D), "q"),
        _ptr(pool_k, torch.bfloat16, (B, H, S, bs, D), "pool_k"),
        _ptr(pool_v, torch.bfloat16, (B, H, S, bs, D), "pool_v"),
        _ptr(block_of_slot, torch.int32, (B, H, S), "block_of_slot"), cl, float(scale),
        _ptr(out, torch.bfloat16, (B, Hq, D), "out"), _stream(stream)))


def oasis_attend_and_score(cfg, q, pool_k, pool_v, block_of_slot, ctx_len, scale, out,
                           q_draft, summ, scores, stream=None) -> None:
    """oasis_sparse_decode_attn(q, pools, ...) and oasis_score_blocks(q_draft,
    summ, scores) -- usually of two different layers -- in one launch."""
    c = OasisConfig.make(cfg)
    B, H, Hq, NB, bs, D, S = _dims(c)
    cl = None if ctx_len is None else _ptr(ctx_len, torch.int32, (B,), "ctx_len")
    _check("oasis_attend_and_score", lib().oasis_attend_and_score(
        C.byref(c), _ptr(q, torch.bfloat16, (B, Hq, D), "q"),
        _ptr(pool_k, torch.bfloat16, (B, H, S, bs, D), "pool_k"),
        _ptr(pool_v, torch.bfloat16, (B, H, S, bs, D), "pool_v"),
        _ptr(block_of_slot, torch.int32, (B, H, S), "block_of_slot"), cl, float(scale),
        _ptr(out, torch.bfloat16, (B, Hq, D), "out"),
        _ptr(q_draft, torch.bfloat16, (B, c.lookahead, Hq, D), "q_draft"),
        _ptr(summ, torch.float32, (B, H, NB, D), "summ"),
        _ptr(scores, torch.float32, (B, H, NB), "scores"), _stream(stream)))


def oasis_sparse_decode_attn_joint(cfg, q, q_draft, pool_k, pool_v, block_of_slot, ctx_len, scale,
                                   out, stream=None) -> None:
    """Attention of the decoded token (q) and the L draft tokens (q_draft) in
    one pass over the working set; out is [B, 1+L, Hq, D]."""
    c = OasisConfig.make(cfg)
    B, H, Hq, NB, bs, D, S = _dims(c)
    L = c.lookahead
    cl = None if ctx_len is None else _ptr(ctx_len, torch.int32, (B,), "ctx_len")
    _check("oasis_sparse_decode_attn_joint", lib().oasis_sparse_decode_attn_joint(
        C.byref(c), _ptr(q, torch.bfloat16, (B, Hq, D), "q"),
        _ptr(q_draft, torch.bfloat16, (B, L, Hq, D), "q_draft"),
        _ptr(pool_k, torch.bfloat16, (B, H, S, bs, D), "pool_k"),
        _ptr(pool_v, torch.bfloat16, (B, H, S, bs, D), "pool_v"),
        _ptr(block_of_slot, torch.int32, (B, H, S), "block_of_slot"), cl, float(scale),
        _ptr(out, torch.bfloat16, (B, L + 1, Hq, D), "out"), _stream(stream)))


def oasis_attend_and_score_minmax(cfg, q, pool_k, pool_v, block_of_slot, ctx_len, scale, out,
                                  q_draft, summ_mm, scores, stream=None) -> None:
    """oasis_attend_and_score with min/max compressed keys (summ_mm)."""
    c = OasisConfig.make(cfg)
    B, H, Hq, NB, bs, D, S = _dims(c)
    cl = None if ctx_len is None else _ptr(ctx_len, torch.int32, (B,), "ctx_len")
    _check("oasis_attend_and_score_minmax", lib().oasis_attend_and_score_minmax(
        C.byref(c), _ptr(q, torch.bfloat16, (B, Hq, D), "q"),
        _ptr(pool_k, torch.bfloat16, (B, H, S, bs, D), "pool_k"),
        _ptr(pool_v, torch.bfloat16, (B, H, S, bs, D), "pool_v"),
        _ptr(block_of_slot, torch.int32, (B, H, S), "block_of_slot"), cl, float(scale),
        _ptr(out, torch.bfloat16, (B, Hq, D), "out"),
        _ptr(q_draft, torch.bfloat16, (B, c.lookahead, Hq, D), "q_draft"),
        _ptr(summ_mm, torch.bfloat16, (B, H, NB, 2, D), "summ_mm"),
        _ptr(scores, torch.float32, (B, H, NB), "scores"), _stream(stream)))


def oasis_host_register(tensor: torch.Tensor) -> int:
    """Pins and maps a CPU tensor in place; returns its device address."""
    if tensor.device.type != "cpu" or not tensor.is_contiguous():
        raise ValueError("oasis_host_register: expects a contiguous CPU tensor")
    dev = C.c_void_p()
    _check("oasis_host_register", lib().oasis_host_register(
        C.c_void_p(tensor.data_ptr()), tensor.numel() * tensor.element_size(), C.byref(dev)))
    return int(dev.value)


def oasis_host_unregister(tensor: torch.Tensor) -> None:
    _check("oasis_host_unregister", lib().oasis_host_unregister(C.c_void_p(tensor.data_ptr())))


def oasis_device_errors(clear: bool = True) -> int:
    v = C.c_uint32()
    _check("oasis_device_errors", lib().oasis_device_errors(C.byref(v), int(bool(clear))))
    return int(v.value)


def oasis_stream_wait(stream=None, timeout_ms: int = 10000) -> int:
    return int(lib().oasis_stream_wait(_stream(stream), int(timeout_ms)))


def oasis_status_string(status: int) -> str:
    return lib().oasis_status_string(int(status)).decode()


def oasis_version() -> int:
    return int(lib().oasis_version())
