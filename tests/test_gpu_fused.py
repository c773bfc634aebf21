"""The fused attention + scoring call against the two separate calls.

oasis_attend_and_score runs the attention of one layer and the scoring of
another in one launch; both halves are the same arithmetic as
oasis_sparse_decode_attn and oasis_score_blocks (which the other GPU tests pin
to the oracle), so the outputs must agree with those calls bit for bit.
The shapes cover a unit split over a cluster of CTAs (Llama layer), one CTA
per unit with more units than SMs (Qwen3-8B batch 32), G = 8 with two
16-row query tiles, ragged context lengths and empty slots; the same with the
min/max compressed keys against oasis_score_blocks_minmax.
"""
import math

import pytest
import torch

from sparse_kv_cache_oasis_gb300 import binding as ob
from sparse_kv_cache_oasis_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _rand(shape, gen, dtype=torch.bfloat16, scale=1.0):
    return (torch.randn(shape, generator=gen, device="cuda") * scale).to(dtype)


def _case(wl, seed, ctx=None, empty_frac=0.0):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    B, H, Hq, S, NB, L = wl.batch, wl.num_kv_heads, wl.num_q_heads, wl.slots, wl.num_blocks, wl.lookahead
    q = _rand((B, Hq, 128), g)
    pk = _rand((B, H, S, 16, 128), g, scale=0.7)
    pv = _rand((B, H, S, 16, 128), g)
    bos = torch.stack([torch.randperm(NB, generator=g, device="cuda")[:S] for _ in range(B * H)])
    bos = bos.reshape(B, H, S).to(torch.int32)
    if empty_frac:
        bos[torch.rand((B, H, S), generator=g, device="cuda") < empty_frac] = -1
    qd = _rand((B, L, Hq, 128), g)
    summ = torch.randn((B, H, NB, 128), generator=g, device="cuda") * 0.05
    cl = None if ctx is None else torch.tensor(ctx, dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(128)

    out_a = torch.empty((B, Hq, 128), dtype=torch.bfloat16, device="cuda")
    sc_a = torch.empty((B, H, NB), dtype=torch.float32, device="cuda")
    ws = torch.zeros(ob.oasis_attn_workspace_bytes(wl), dtype=torch.uint8, device="cuda")
    ob.oasis_sparse_decode_attn(wl, q, pk, pv, bos, cl, scale, out_a, ws)
    ob.oasis_score_blocks(wl, qd, summ, sc_a)

    out_b = torch.full_like(out_a, float("nan"))
    sc_b = torch.full_like(sc_a, float("nan"))
    for _ in range(2):  # twice: the call leaves nothing behind that changes the next one
        ob.oasis_attend_and_score(wl, q, pk, pv, bos, cl, scale, out_b, qd, summ, sc_b)
        torch.cuda.synchronize()
        assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
        assert torch.equal(sc_a.view(torch.int32), sc_b.view(torch.int32))
    assert ob.oasis_device_errors() == 0


def test_fused_llama_layer_cluster_split():
    _case(W.LLAMA8B_LAYER, seed=21)


def test_fused_more_units_than_sms():
    _case(W.QWEN3_8B_STEP.with_(layers=1), seed=22)


def test_fused_group8_ragged_and_empty():
    wl = W.Workload(name="g8", batch=3, num_q_heads=32, num_kv_heads=4, ctx_tokens=16 * 203,
                    kv_budget_tokens=16 * 77, lookahead=4, top_k=40, fetch_ratio=0.1, seed=5)
    _case(wl, seed=23, ctx=[16 * 203, 999, 40], empty_frac=0.2)


def test_fused_tiny_units():
    wl = W.Workload(name="tiny-units", batch=40, num_q_heads=32, num_kv_heads=8,
                    ctx_tokens=16 * 203, kv_budget_tokens=16 * 3, lookahead=2, top_k=3,
                    fetch_ratio=0.1, seed=6)
    _case(wl, seed=24, empty_frac=0.1)


def _case_minmax(wl, seed, ctx=None, empty_frac=0.0):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    B, H, Hq, S, NB, L = wl.batch, wl.num_kv_heads, wl.num_q_heads, wl.slots, wl.num_blocks, wl.lookahead
    q = _rand((B, Hq, 128), g)
    pk = _rand((B, H, S, 16, 128), g, scale=0.7)
    pv = _rand((B, H, S, 16, 128), g)
    bos = torch.stack([torch.randperm(NB, generator=g, device="cuda")[:S] for _ in range(B * H)])
    bos = bos.reshape(B, H, S).to(torch.int32)
    if empty_frac:
        bos[torch.rand((B, H, S), generator=g, device="cuda") < empty_frac] = -1
    qd = _rand((B, L, Hq, 128), g)
    mm = _rand((B, H, NB, 2, 128), g, scale=0.3)
    cl = None if ctx is None else torch.tensor(ctx, dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(128)
    out_a = torch.empty((B, Hq, 128), dtype=torch.bfloat16, device="cuda")
    sc_a = torch.empty((B, H, NB), dtype=torch.float32, device="cuda")
    ws = torch.zeros(ob.oasis_attn_workspace_bytes(wl), dtype=torch.uint8, device="cuda")
    ob.oasis_sparse_decode_attn(wl, q, pk, pv, bos, cl, scale, out_a, ws)
    ob.oasis_score_blocks_minmax(wl, qd, mm, sc_a)
    out_b = torch.full_like(out_a, float("nan"))
    sc_b = torch.full_like(sc_a, float("nan"))
    ob.oasis_attend_and_score_minmax(wl, q, pk, pv, bos, cl, scale, out_b, qd, mm, sc_b)
    torch.cuda.synchronize()
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    assert torch.equal(sc_a.view(torch.int32), sc_b.view(torch.int32))
    assert ob.oasis_device_errors() == 0


def test_fused_minmax_llama_layer():
    _case_minmax(W.LLAMA8B_LAYER, seed=31)


def test_fused_minmax_two_row_tiles_ragged():
    wl = W.Workload(name="g8mm", batch=3, num_q_heads=32, num_kv_heads=4, ctx_tokens=16 * 203,
                    kv_budget_tokens=16 * 77, lookahead=4, top_k=40, fetch_ratio=0.1, seed=5)
    _case_minmax(wl, seed=32, ctx=[16 * 203, 999, 40], empty_frac=0.2)
