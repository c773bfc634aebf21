"""Min/max compressed keys on the GPU against the oracle.

The pooling "OasisKV: Scaling In-Decode KV Cache Beyond HBM with Lookahead
Sparse Prefetching", Fig. 7 (left) names: per block the elementwise max and
min keys, and a block score sum_d max(q_d min_d, q_d max_d) maximised over
the draft tokens and the GQA group.

Tolerances: summaries bit-exact (they are key values); scores within
4e-5 * max_(l,g) sum_d |q_d| max(|min_d|, |max_d|): the products are exact
on the bf16 tensor cores and 256 of them are accumulated in fp32, at most
256 * 2^-23 (3.05e-5) of that sum even with truncating adds; top-K lists
equal to the oracle's from the oracle's scores, up to near ties (1e-4
relative, as for the mean keys).
"""
import numpy as np
import pytest
import torch

import oracle
from sparse_kv_cache_oasis_gb300 import binding as ob
from sparse_kv_cache_oasis_gb300 import workloads as W

from gpu_helpers import check_topk, dev_bits

pytestmark = pytest.mark.gpu

MINMAX_REL = 4e-5


def _wl(**kw):
    base = dict(name="minmax", batch=2, num_q_heads=8, num_kv_heads=2, ctx_tokens=16 * 203,
                kv_budget_tokens=16 * 48, lookahead=3, top_k=40, fetch_ratio=0.1, seed=79)
    base.update(kw)
    return W.Workload(**base)


def _bound(qd_bits, mm_bits, G):
    qd = W.bf16_bits_to_f32(qd_bits).astype(np.float64)                    # [B, L, Hq, D]
    B, L, Hq, D = qd.shape
    ext = np.abs(W.bf16_bits_to_f32(mm_bits).astype(np.float64)).max(axis=3)  # [B, H, NB, D]
    qa = np.abs(qd).reshape(B, L, Hq // G, G, D)
    s = np.einsum("blhgd,bhjd->blhgj", qa, ext)                           # [B, L, H, G, NB]
    return MINMAX_REL * s.max(axis=(1, 3)) + 1e-30


def _case(wl, step=0, full_topk=True):
    cfg = wl.config()
    qseq = W.query_sequence(wl, 0)
    k, _ = W.gen_kv(wl, 0, qseq)
    _, qd = W.step_queries(wl, qseq, step)
    B, H, NB, D = wl.batch, wl.num_kv_heads, wl.num_blocks, 128
    gk = dev_bits(k)
    mm = torch.empty((B, H, NB, 2, D), dtype=torch.bfloat16, device="cuda")
    ob.oasis_build_summaries_minmax(cfg, gk, mm)
    torch.cuda.synchronize()
    ref_mm = oracle.build_summaries_minmax(cfg, k)
    got_mm = mm.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got_mm, ref_mm)
    del gk
    scores = torch.full((B, H, NB), float("nan"), dtype=torch.float32, device="cuda")
    ob.oasis_score_blocks_minmax(cfg, dev_bits(qd), mm, scores)
    torch.cuda.synchronize()
    ref = oracle.score_blocks_minmax(cfg, qd, ref_mm)
    got = scores.cpu().numpy()
    bound = _bound(qd, ref_mm, wl.group)
    err = np.abs(got.astype(np.float64) - ref)
    assert (err <= bound).all(), f"max err {err.max():.3g}, worst ratio {(err / bound).max():.3g}"
    if full_topk:  # the top-K of the GPU scores against the oracle's, near ties allowed
        topk = torch.empty((B, H, wl.top_k), dtype=torch.int32, device="cuda")
        ob.oasis_select_topk(cfg, scores, topk)
        ref_ids = oracle.select_topk(cfg, ref)
        gids = topk.cpu().numpy()
        for b in range(B):  # equal, or different only where the oracle has a near tie
            for h in range(H):
                check_topk(gids[b, h], ref_ids[b, h], ref[b, h], cfg)
    assert ob.oasis_device_errors() == 0


@pytest.mark.parametrize("wl", [
    W.TINY,                                              # L*G = 8, planted blocks
    _wl(),                                               # L*G = 12, NB = 203 (ragged tile)
    _wl(num_q_heads=16, lookahead=4, seed=80),           # L*G = 32: two row tiles
    _wl(num_q_heads=2, num_kv_heads=2, lookahead=1, seed=81),  # L*G = 1
    _wl(key_std=3.0, seed=82),                           # wider keys
])
def test_minmax_summaries_scores_topk(wl):
    _case(wl)
    _case(wl, step=1, full_topk=False)


def test_minmax_llama_layer_full_size():
    _case(W.LLAMA8B_LAYER, full_topk=True)


def test_minmax_rejects_more_than_32_rows():
    wl = _wl(num_q_heads=16, lookahead=5)                # L*G = 40
    B, H, NB = wl.batch, wl.num_kv_heads, wl.num_blocks
    mm = torch.zeros((B, H, NB, 2, 128), dtype=torch.bfloat16, device="cuda")
    qd = torch.zeros((B, 5, 16, 128), dtype=torch.bfloat16, device="cuda")
    sc = torch.zeros((B, H, NB), dtype=torch.float32, device="cuda")
    with pytest.raises(ob.OasisError):
        ob.oasis_score_blocks_minmax(wl.config(), qd, mm, sc)
