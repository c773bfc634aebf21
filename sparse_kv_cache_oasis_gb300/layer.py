"""Device state of one attention layer and its decode step, over the C ABI.

``LayerState`` owns the buffers of one layer of one workload: the full K/V
cache in pinned, mapped host memory, the compressed keys, the HBM working
set (pools and the head-wise slot/block map with LRU times) and the per-step
scratch.  ``step`` enqueues the hot path of one layer for one decode step,
in the order of "OasisKV: Scaling In-Decode KV Cache Beyond HBM with Lookahead
Sparse Prefetching", Fig. 8: attention over the current working set, draft
scoring, top-K, planning, then the transfer on the copy stream that must end
before the same layer's attention of the next step.

PyTorch here only allocates memory and provides streams and events; every
step of the path is a liboasis kernel.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from . import binding as ob


def bits_to_bf16(a: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bit patterns (numpy) -> bf16 CPU tensor sharing the memory."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def bf16_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


class LayerState:
    def __init__(self, cfg, host_k: torch.Tensor, host_v: torch.Tensor, slot_of_block: np.ndarray,
                 block_of_slot: np.ndarray, last_used: np.ndarray, device: str = "cuda",
                 ctx_len: np.ndarray | None = None, register_host: bool = True):
        self.cfg = ob.OasisConfig.make(cfg)
        c = self.cfg
        st = ob.oasis_validate_config(c)
        if st != ob.OASIS_OK:
            raise ob.OasisError("oasis_validate_config", st)
        B, H, Hq, NB = c.batch, c.num_kv_heads, c.num_q_heads, c.num_blocks
        bs, D, L, K = c.block_size, c.head_dim, c.lookahead, c.top_k
        S = c.kv_budget_tokens // bs
        self.S = S
        self.capw = ob.cap_width(c)
        dev = torch.device(device)
        # full cache: pinned + mapped host memory, read by the GPU over the host link
        self.host_k, self.host_v = host_k.contiguous(), host_v.contiguous()
        self._registered = False
        if register_host:
            self.host_k_dev = ob.oasis_host_register(self.host_k)
            self.host_v_dev = ob.oasis_host_register(self.host_v)
            self._registered = True
        else:
            self.host_k_dev = self.host_k.data_ptr()
            self.host_v_dev = self.host_v.data_ptr()
        f32, i32, bf = torch.float32, torch.int32, torch.bfloat16
        self.summ = torch.empty((B, H, NB, D), dtype=f32, device=dev)
        ob.oasis_build_summaries(c, self.host_k_dev, self.summ)
        self.slot_of_block = torch.from_numpy(np.ascontiguousarray(slot_of_block, np.int32)).to(dev)
        self.block_of_slot = torch.from_numpy(np.ascontiguousarray(block_of_slot, np.int32)).to(dev)
        self.last_used = torch.from_numpy(np.ascontiguousarray(last_used, np.int32)).to(dev)
        # initial working set (admission): copy the resident blocks into the pools
        self.pool_k = torch.zeros((B, H, S, bs, D), dtype=bf, device=dev)
        self.pool_v = torch.zeros((B, H, S, bs, D), dtype=bf, device=dev)
        bos = torch.from_numpy(np.ascontiguousarray(block_of_slot, np.int64))
        hk = self.host_k.view(B * H, NB, bs * D)
        hv = self.host_v.view(B * H, NB, bs * D)
        pk = self.pool_k.view(B * H, S, bs * D)
        pv = self.pool_v.view(B * H, S, bs * D)
        for u in range(B * H):
            row = bos.view(B * H, S)[u]
            slots = torch.nonzero(row >= 0).flatten()
            if slots.numel():
                pk[u, slots.to(dev)] = hk[u, row[slots]].to(dev)
                pv[u, slots.to(dev)] = hv[u, row[slots]].to(dev)
        self.ctx_len = None if ctx_len is None else torch.from_numpy(
            np.ascontiguousarray(ctx_len, np.int32)).to(dev)
        # per-step buffers
        self.scores = torch.empty((B, H, NB), dtype=f32, device=dev)
        self.topk = torch.empty((B, H, K), dtype=i32, device=dev)
        self.fetch_block = torch.full((B, H, self.capw), -1, dtype=i32, device=dev)
        self.fetch_slot = torch.full((B, H, self.capw), -1, dtype=i32, device=dev)
        self.evict_block = torch.full((B, H, self.capw), -1, dtype=i32, device=dev)
        self.n_fetch = torch.zeros((B, H), dtype=i32, device=dev)
        self.n_evict = torch.zeros((B, H), dtype=i32, device=dev)
        self.out = torch.empty((B, Hq, D), dtype=bf, device=dev)
        self.out_joint = torch.empty((B, L + 1, Hq, D), dtype=bf, device=dev)  # decoded + drafts
        self.clock = torch.zeros((B, H), dtype=i32, device=dev)  # device step per (b, h)
        self.workspace = torch.zeros(max(ob.oasis_attn_workspace_bytes(c), 256), dtype=torch.uint8,
                                     device=dev)
        self.scale = 1.0 / math.sqrt(D)
        self.fetch_done = torch.cuda.Event()
        self.fetch_done.record(torch.cuda.current_stream(dev))

    def build_minmax_summaries(self):
        """Min/max compressed keys beside the mean ones: self.summ_mm
        [B, Hkv, NB, 2, D] bf16 (max row, min row)."""
        c = self.cfg
        self.summ_mm = torch.empty((c.batch, c.num_kv_heads, c.num_blocks, 2, c.head_dim),
                                   dtype=torch.bfloat16, device=self.summ.device)
        ob.oasis_build_summaries_minmax(c, self.host_k_dev, self.summ_mm)

    # -- the five calls -----------------------------------------------------
    def attention(self, q, stream=None):
        ob.oasis_sparse_decode_attn(self.cfg, q, self.pool_k, self.pool_v, self.block_of_slot,
                                    self.ctx_len, self.scale, self.out, self.workspace, stream)

    def attention_joint(self, q, q_draft, stream=None):
        """Attention of the decoded token and the draft tokens in one pass:
        self.out_joint[:, 0] for q, self.out_joint[:, l] for q_draft[:, l-1]."""
        ob.oasis_sparse_decode_attn_joint(self.cfg, q, q_draft, self.pool_k, self.pool_v,
                                          self.block_of_slot, self.ctx_len, self.scale,
                                          self.out_joint, stream)

    def attention_and_score(self, q, other, q_draft, stream=None):
        """This layer's attention and `other` layer's scoring in one launch."""
        ob.oasis_attend_and_score(self.cfg, q, self.pool_k, self.pool_v, self.block_of_slot,
                                  self.ctx_len, self.scale, self.out, q_draft, other.summ,
                                  other.scores, stream)

    def attention_and_score_minmax(self, q, other, q_draft, stream=None):
        """This layer's attention and `other` layer's min/max-key scoring in one launch."""
        ob.oasis_attend_and_score_minmax(self.cfg, q, self.pool_k, self.pool_v, self.block_of_slot,
                                         self.ctx_len, self.scale, self.out, q_draft, other.summ_mm,
                                         other.scores, stream)

    def predict(self, q_draft, step, stream=None):
        ob.oasis_score_blocks(self.cfg, q_draft, self.summ, self.scores, stream)
        ob.oasis_select_topk(self.cfg, self.scores, self.topk, stream)
        ob.oasis_plan_fetch(self.cfg, self.topk, step, self.slot_of_block, self.block_of_slot,
                            self.last_used, self.fetch_block, self.fetch_slot, self.evict_block,
                            self.n_fetch, self.n_evict, stream)

    def score_minmax(self, q_draft, stream=None):
        """Scoring against the min/max compressed keys into self.scores."""
        ob.oasis_score_blocks_minmax(self.cfg, q_draft, self.summ_mm, self.scores, stream)

    def append(self, k_new, v_new, stream=None):
        """Decode-time append of one token per request at self.ctx_len (which
        it advances): cache and working set (newest block kept resident, LRU
        time from the device clock).  refresh_summaries follows."""
        ob.oasis_append_kv(self.cfg, k_new, v_new, self.ctx_len, 0, self.clock, self.host_k_dev,
                           self.host_v_dev, self.slot_of_block, self.block_of_slot, self.last_used,
                           self.pool_k, self.pool_v, stream)

    def refresh_summaries(self, stream=None):
        """The newest block's summaries (min/max too when built) after an append."""
        ob.oasis_refresh_summaries(self.cfg, self.ctx_len, self.host_k_dev, self.slot_of_block,
                                   self.pool_k, self.summ, getattr(self, "summ_mm", None), stream)

    def select_ctx(self, stream=None):
        """Top-K with the local window at each context's end, then the plan,
        in one launch (device clock)."""
        ob.oasis_predict_select_ctx(self.cfg, self.scores, self.ctx_len, 0, self.clock, self.topk,
                                    self.slot_of_block, self.block_of_slot, self.last_used,
                                    self.fetch_block, self.fetch_slot, self.evict_block,
                                    self.n_fetch, self.n_evict, stream)

    def predict_chain(self, q_draft, stream=None):
        """Scoring, top-K and planning in one launch (device clock)."""
        ob.oasis_predict_chain(self.cfg, q_draft, self.summ, self.scores, 0, self.clock,
                               self.topk, self.slot_of_block, self.block_of_slot, self.last_used,
                               self.fetch_block, self.fetch_slot, self.evict_block, self.n_fetch,
                               self.n_evict, stream)

    def predict_clocked(self, q_draft, stream=None):
        """predict() with the step taken from (and advanced in) self.clock."""
        ob.oasis_score_blocks(self.cfg, q_draft, self.summ, self.scores, stream)
        ob.oasis_select_topk(self.cfg, self.scores, self.topk, stream)
        ob.oasis_plan_fetch_clocked(self.cfg, self.topk, self.clock, self.slot_of_block,
                                    self.block_of_slot, self.last_used, self.fetch_block,
                                    self.fetch_slot, self.evict_block, self.n_fetch, self.n_evict,
                                    stream)

    def predict_fused(self, q_draft, stream=None):
        """Scoring, then top-K and planning fused in one launch (device clock)."""
        ob.oasis_score_blocks(self.cfg, q_draft, self.summ, self.scores, stream)
        ob.oasis_predict_select(self.cfg, self.scores, 0, self.clock, self.topk,
                                self.slot_of_block, self.block_of_slot, self.last_used,
                                self.fetch_block, self.fetch_slot, self.evict_block,
                                self.n_fetch, self.n_evict, stream)

    def fetch(self, stream=None):
        ob.oasis_fetch_blocks(self.cfg, self.host_k_dev, self.host_v_dev, self.fetch_block,
                              self.fetch_slot, self.n_fetch, self.pool_k, self.pool_v, stream)

    def step(self, step, q, q_draft, compute=None, copy=None):
        """One layer-step.  Attention waits for the previous transfer of this
        layer; the transfer runs on `copy` after the plan and records
        `fetch_done`."""
        compute = compute or torch.cuda.current_stream()
        copy = copy or compute
        torch.cuda.nvtx.range_push(f"oasis layer-step {step}")
        compute.wait_event(self.fetch_done)
        self.attention(q, compute)
        self.predict(q_draft, step, compute)
        planned = torch.cuda.Event()
        planned.record(compute)
        copy.wait_event(planned)
        self.fetch(copy)
        self.fetch_done.record(copy)
        torch.cuda.nvtx.range_pop()
        return self.out

    def close(self):
        if self._registered:
            torch.cuda.synchronize()
            ob.oasis_host_unregister(self.host_k)
            ob.oasis_host_unregister(self.host_v)
            self._registered = False

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- host views for checks ------------------------------------------------
    def state_numpy(self):
        return (self.slot_of_block.cpu().numpy(), self.block_of_slot.cpu().numpy(),
                self.last_used.cpu().numpy())

    _STATE = ("slot_of_block", "block_of_slot", "last_used", "clock", "pool_k", "pool_v", "summ")

    def dump(self, path):
        """Writes the layer's device state (working-set maps, LRU times, step
        clock, pools, summaries, context lengths) to an .npz file, e.g. to
        replay a step on the oracle from exactly this state."""
        arrays = {}
        for name in self._STATE:
            t = getattr(self, name).detach().cpu().contiguous()
            arrays[name] = t.view(torch.int16).numpy() if t.dtype == torch.bfloat16 else t.numpy()
        if self.ctx_len is not None:
            arrays["ctx_len"] = self.ctx_len.cpu().numpy()
        np.savez(path, **arrays)

    def restore(self, path):
        """Loads a state written by dump() into this layer's buffers (same shapes)."""
        with np.load(path) as z:
            for name in self._STATE:
                dst = getattr(self, name)
                src = torch.from_numpy(z[name])
                if dst.dtype == torch.bfloat16:
                    src = src.view(torch.bfloat16)
                if tuple(src.shape) != tuple(dst.shape):
                    raise ValueError(f"{name}: shape {tuple(src.shape)} in {path}, expected {tuple(dst.shape)}")
                dst.copy_(src)
            if "ctx_len" in z.files:
                if self.ctx_len is None:
                    self.ctx_len = torch.from_numpy(z["ctx_len"]).to(self.summ.device)
                else:
                    self.ctx_len.copy_(torch.from_numpy(z["ctx_len"]))
