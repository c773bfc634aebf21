"""Kernel-by-kernel parity of the GPU library (through the C ABI) with the CPU
oracle on identical seeded inputs.  Tolerances are defined in gpu_helpers."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (ATOL, RTOL, assert_attn_close, check_topk, dev_bits, score_bound,
                         setup_layer)
from sparse_kv_cache_oasis_gb300 import binding as ob
from sparse_kv_cache_oasis_gb300 import workloads as W
from sparse_kv_cache_oasis_gb300.layer import LayerState, bf16_to_bits, bits_to_bf16

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def small_wl(**kw):
    base = dict(name="small", batch=2, num_q_heads=8, num_kv_heads=2, ctx_tokens=16 * 203,
                kv_budget_tokens=16 * 48, lookahead=3, top_k=40, fetch_ratio=0.1, seed=77)
    base.update(kw)
    return W.Workload(**base)


# --------------------------------------------------------------------- summaries
@pytest.mark.parametrize("wl", [W.TINY, small_wl(), small_wl(key_std=3.0, seed=5)])
def test_summaries_bit_exact(wl):
    st, k, v, _ = setup_layer(wl)
    torch.cuda.synchronize()
    ref = oracle.build_summaries(wl.config(), k)
    assert np.array_equal(st.summ.cpu().numpy(), ref)
    assert ob.oasis_device_errors() == 0
    st.close()


# --------------------------------------------------------------------- scores
@pytest.mark.parametrize("wl", [
    W.TINY,                                                   # L*G = 8  (one 16-row tile, padded)
    small_wl(),                                               # L*G = 12, NB = 203 (ragged tile)
    small_wl(num_q_heads=16, lookahead=4, seed=9),            # L*G = 32 (two tiles)
    small_wl(num_q_heads=16, lookahead=3, seed=10),           # L*G = 24
    small_wl(num_q_heads=16, num_kv_heads=2, lookahead=6, seed=11, top_k=8, kv_budget_tokens=16 * 8),  # 48
    small_wl(num_q_heads=16, lookahead=8, seed=12),           # L*G = 64 (four tiles)
    small_wl(num_q_heads=2, num_kv_heads=2, lookahead=1, seed=13),  # L*G = 1
])
def test_scores_within_bound(wl):
    st, k, v, qseq = setup_layer(wl)
    _, qd = W.step_queries(wl, qseq, 0)
    ob.oasis_score_blocks(wl, dev_bits(qd), st.summ, st.scores)
    torch.cuda.synchronize()
    summ = st.summ.cpu().numpy()
    ref = oracle.score_blocks(wl.config(), qd, summ)
    got = st.scores.cpu().numpy()
    bound = score_bound(qd, summ, wl.group)
    assert (np.abs(got.astype(np.float64) - ref) <= bound).all(), np.abs(got - ref).max()
    st.close()


# --------------------------------------------------------------------- top-K
def _topk_case(NB, K, scores, sink=0, local=0, B=1, H=1):
    cfg = dict(batch=B, num_q_heads=H, num_kv_heads=H, head_dim=128, block_size=16, num_blocks=NB,
               kv_budget_tokens=16 * max(K, 1), lookahead=1, top_k=K, fetch_ratio=0.5,
               sink_blocks=sink, local_blocks=local)
    s = np.ascontiguousarray(scores.reshape(B, H, NB), np.float32)
    dev = torch.from_numpy(s).cuda()
    out = torch.full((B, H, K), -7, dtype=torch.int32, device="cuda")
    ob.oasis_select_topk(cfg, dev, out)
    torch.cuda.synchronize()
    ref = oracle.select_topk(cfg, s)
    assert np.array_equal(out.cpu().numpy(), ref)


def test_topk_bit_exact_random_and_ties():
    rs = np.random.default_rng(21)
    _topk_case(2048, 128, rs.standard_normal(2048 * 8), B=2, H=4)
    _topk_case(203, 40, rs.standard_normal(203))
    _topk_case(2048, 128, rs.integers(-3, 4, 2048).astype(np.float32))          # heavy ties
    _topk_case(2048, 128, np.zeros(2048, np.float32))                           # all equal
    _topk_case(1000, 1, rs.standard_normal(1000))
    _topk_case(64, 64, rs.standard_normal(64))                                  # K = NB
    z = np.where(rs.random(512) < 0.5, -0.0, 0.0).astype(np.float32)            # -0.0 == +0.0
    z[::7] = rs.standard_normal(len(z[::7]))
    _topk_case(512, 100, z)
    _topk_case(4096, 300, -np.abs(rs.standard_normal(4096)).astype(np.float32))  # all negative
    tiny = (rs.standard_normal(3000) * 1e-39).astype(np.float32)                 # denormals
    _topk_case(3000, 50, tiny)
    big = rs.choice([1e30, -1e30, np.inf, -np.inf, 5.0], 3000).astype(np.float32)
    _topk_case(3000, 200, big)


def test_topk_forced_blocks_and_sizes():
    rs = np.random.default_rng(22)
    _topk_case(8192, 128, rs.standard_normal(8192 * 2), sink=1, local=4, B=1, H=2)
    _topk_case(32768, 128, rs.standard_normal(32768))
    _topk_case(16384, 1024, rs.standard_normal(16384), sink=3, local=5)
    _topk_case(100, 10, rs.standard_normal(100), sink=10, local=0)              # forced fills K
    _topk_case(100, 20, rs.standard_normal(100), sink=8, local=8)               # overlap-free forced
    _topk_case(10, 10, rs.standard_normal(10), sink=6, local=6)                 # sink/local overlap


# --------------------------------------------------------------------- plan
def _random_state(rs, B, H, NB, S, full=True):
    sob = np.full((B, H, NB), -1, np.int32)
    bos = np.full((B, H, S), -1, np.int32)
    lu = np.full((B, H, S), -1, np.int32)
    for b in range(B):
        for h in range(H):
            n = S if full else int(rs.integers(0, S + 1))
            blocks = rs.choice(NB, size=n, replace=False)
            slots = rs.choice(S, size=n, replace=False)
            bos[b, h, slots] = blocks
            sob[b, h, blocks] = slots
            lu[b, h, slots] = rs.integers(-3, 5, size=n)
    return sob, bos, lu


@pytest.mark.parametrize("NB,S,K,ratio,sink,local,full", [
    (2048, 128, 128, 0.05, 0, 0, True),
    (256, 64, 32, 4 / 64, 0, 0, True),
    (8192, 128, 128, 0.02, 1, 4, True),
    (300, 40, 30, -1.0, 0, 0, False),
    (300, 40, 30, 0.5, 2, 2, False),
    (1000, 1024, 1000, 0.01, 0, 0, False),
    (64, 8, 8, 0.0, 0, 0, True),
])
def test_plan_bit_exact(NB, S, K, ratio, sink, local, full):
    rs = np.random.default_rng(NB + S + K)
    B, H = 3, 2
    cfg = dict(batch=B, num_q_heads=H, num_kv_heads=H, head_dim=128, block_size=16, num_blocks=NB,
               kv_budget_tokens=16 * S, lookahead=1, top_k=K, fetch_ratio=ratio, sink_blocks=sink,
               local_blocks=local)
    sob, bos, lu = _random_state(rs, B, H, NB, S, full)
    d = {n: torch.from_numpy(a.copy()).cuda() for n, a in (("sob", sob), ("bos", bos), ("lu", lu))}
    w = max(oracle.fetch_cap(cfg), 1)
    outs = {n: torch.full((B, H, w), -9, dtype=torch.int32, device="cuda") for n in ("fb", "fs", "eb")}
    nf = torch.full((B, H), -9, dtype=torch.int32, device="cuda")
    ne = torch.full((B, H), -9, dtype=torch.int32, device="cuda")
    for step in range(5):
        scores = rs.standard_normal((B, H, NB)).astype(np.float32)
        topk = oracle.select_topk(cfg, scores)
        ob.oasis_plan_fetch(cfg, torch.from_numpy(topk).cuda(), step, d["sob"], d["bos"], d["lu"],
                            outs["fb"], outs["fs"], outs["eb"], nf, ne)
        ref = oracle.plan_fetch(cfg, topk, step, sob, bos, lu)
        torch.cuda.synchronize()
        assert np.array_equal(nf.cpu().numpy(), ref["n_fetch"])
        assert np.array_equal(ne.cpu().numpy(), ref["n_evict"])
        assert np.array_equal(outs["fb"].cpu().numpy(), ref["fetch_block"])
        assert np.array_equal(outs["fs"].cpu().numpy(), ref["fetch_slot"])
        assert np.array_equal(outs["eb"].cpu().numpy(), ref["evict_block"])
        assert np.array_equal(d["sob"].cpu().numpy(), sob)
        assert np.array_equal(d["bos"].cpu().numpy(), bos)
        assert np.array_equal(d["lu"].cpu().numpy(), lu)
    assert ob.oasis_device_errors() == 0


def test_plan_rejects_bad_state_with_error_flag():
    cfg = dict(batch=1, num_q_heads=1, num_kv_heads=1, head_dim=128, block_size=16, num_blocks=16,
               kv_budget_tokens=64, lookahead=1, top_k=2, fetch_ratio=0.5, sink_blocks=0, local_blocks=0)
    ob.oasis_device_errors(clear=True)
    sob = torch.full((1, 1, 16), -1, dtype=torch.int32, device="cuda")
    bos = torch.tensor([[[3, -1, -1, -1]]], dtype=torch.int32, device="cuda")  # map disagrees
    lu = torch.zeros((1, 1, 4), dtype=torch.int32, device="cuda")
    fb, fs, eb = (torch.zeros((1, 1, 2), dtype=torch.int32, device="cuda") for _ in range(3))
    nf, ne = (torch.full((1, 1), 5, dtype=torch.int32, device="cuda") for _ in range(2))
    topk = torch.tensor([[[1, 2]]], dtype=torch.int32, device="cuda")
    ob.oasis_plan_fetch(cfg, topk, 0, sob, bos, lu, fb, fs, eb, nf, ne)
    flags = ob.oasis_device_errors(clear=True)
    assert flags & ob.DEVERR_PLAN_STATE
    assert nf.item() == 0 and ne.item() == 0 and (fb == -1).all()
    assert bos.cpu().tolist() == [[[3, -1, -1, -1]]]
    sob[0, 0, 3] = 0
    topk = torch.tensor([[[7, 7]]], dtype=torch.int32, device="cuda")          # repeated id
    ob.oasis_plan_fetch(cfg, topk, 0, sob, bos, lu, fb, fs, eb, nf, ne)
    assert ob.oasis_device_errors(clear=True) & ob.DEVERR_TOPK_IDS
    topk = torch.tensor([[[1, 99]]], dtype=torch.int32, device="cuda")         # out of range
    ob.oasis_plan_fetch(cfg, topk, 0, sob, bos, lu, fb, fs, eb, nf, ne)
    assert ob.oasis_device_errors(clear=True) & ob.DEVERR_TOPK_IDS


# --------------------------------------------------------------------- fetch
def test_fetch_bytes_and_range_checks():
    wl = small_wl(fetch_ratio=-1.0)
    cfg = wl.config()
    B, H, NB, S = wl.batch, wl.num_kv_heads, wl.num_blocks, wl.slots
    rs = np.random.default_rng(4)
    hk = rs.integers(0, 65535, size=(B, H, NB, 16, 128), dtype=np.uint16)
    hv = rs.integers(0, 65535, size=(B, H, NB, 16, 128), dtype=np.uint16)
    tk, tv = bits_to_bf16(hk), bits_to_bf16(hv)
    dk, dv = ob.oasis_host_register(tk), ob.oasis_host_register(tv)
    try:
        w = max(oracle.fetch_cap(cfg), 1)
        fb = np.full((B, H, w), -1, np.int32)
        fs = np.full((B, H, w), -1, np.int32)
        nf = rs.integers(0, w + 1, size=(B, H)).astype(np.int32)
        for b in range(B):
            for h in range(H):
                fb[b, h, :nf[b, h]] = np.sort(rs.choice(NB, nf[b, h], replace=False))
                fs[b, h, :nf[b, h]] = rs.choice(S, nf[b, h], replace=False)
        pk = np.zeros((B, H, S, 16, 128), np.uint16)
        pv = np.zeros_like(pk)
        gk, gv = dev_bits(pk), dev_bits(pv)
        ob.oasis_fetch_blocks(cfg, dk, dv, torch.from_numpy(fb).cuda(), torch.from_numpy(fs).cuda(),
                              torch.from_numpy(nf).cuda(), gk, gv)
        oracle.fetch_blocks(cfg, hk, hv, fb, fs, nf, pk, pv)
        torch.cuda.synchronize()
        assert np.array_equal(bf16_to_bits(gk), pk) and np.array_equal(bf16_to_bits(gv), pv)
        assert ob.oasis_device_errors() == 0
        # an out-of-range entry is skipped and flagged; the others still land
        fb2, fs2 = fb.copy(), fs.copy()
        nf2 = np.full((B, H), 2, np.int32)
        fb2[:, :, 0], fs2[:, :, 0] = NB, 0
        fb2[:, :, 1], fs2[:, :, 1] = 5, S - 1
        ob.oasis_fetch_blocks(cfg, dk, dv, torch.from_numpy(fb2).cuda(), torch.from_numpy(fs2).cuda(),
                              torch.from_numpy(nf2).cuda(), gk, gv)
        flags = ob.oasis_device_errors(clear=True)
        assert flags & ob.DEVERR_FETCH_RANGE
        got = bf16_to_bits(gk)
        assert np.array_equal(got[:, :, S - 1], hk[:, :, 5])
        assert np.array_equal(got[:, :, 0], pk[:, :, 0])
    finally:
        torch.cuda.synchronize()
        ob.oasis_host_unregister(tk)
        ob.oasis_host_unregister(tv)


@pytest.mark.parametrize("B,H,NB,S,ratio,full", [
    (32, 8, 160, 128, -1.0, True),     # 256 units, every list full: 512 entries per CTA, 4 batches
    (1100, 8, 6, 4, 0.5, False),       # 8800 units: more than 128 units per CTA
    (3, 2, 64, 16, 0.2, False),        # fewer items than CTAs
])
def test_fetch_many_entries_and_units(B, H, NB, S, ratio, full):
    cfg = dict(batch=B, num_q_heads=H, num_kv_heads=H, head_dim=128, block_size=16, num_blocks=NB,
               kv_budget_tokens=16 * S, lookahead=1, top_k=S, fetch_ratio=ratio, sink_blocks=0,
               local_blocks=0)
    rs = np.random.default_rng(B + NB)
    hk = rs.integers(0, 65535, size=(B, H, NB, 16, 128), dtype=np.uint16)
    hv = rs.integers(0, 65535, size=(B, H, NB, 16, 128), dtype=np.uint16)
    tk, tv = bits_to_bf16(hk), bits_to_bf16(hv)
    dk, dv = ob.oasis_host_register(tk), ob.oasis_host_register(tv)
    try:
        w = max(oracle.fetch_cap(cfg), 1)
        fb = np.full((B, H, w), -1, np.int32)
        fs = np.full((B, H, w), -1, np.int32)
        nf = (np.full((B, H), w) if full else rs.integers(0, w + 1, size=(B, H))).astype(np.int32)
        for b in range(B):
            for h in range(H):
                fb[b, h, :nf[b, h]] = np.sort(rs.choice(NB, nf[b, h], replace=False))
                fs[b, h, :nf[b, h]] = rs.choice(S, nf[b, h], replace=False)
        pk = rs.integers(0, 65535, size=(B, H, S, 16, 128), dtype=np.uint16)
        pv = rs.integers(0, 65535, size=(B, H, S, 16, 128), dtype=np.uint16)
        gk, gv = dev_bits(pk), dev_bits(pv)
        ob.oasis_fetch_blocks(cfg, dk, dv, torch.from_numpy(fb).cuda(), torch.from_numpy(fs).cuda(),
                              torch.from_numpy(nf).cuda(), gk, gv)
        oracle.fetch_blocks(cfg, hk, hv, fb, fs, nf, pk, pv)
        torch.cuda.synchronize()
        assert np.array_equal(bf16_to_bits(gk), pk) and np.array_equal(bf16_to_bits(gv), pv)
        assert ob.oasis_device_errors() == 0
    finally:
        torch.cuda.synchronize()
        ob.oasis_host_unregister(tk)
        ob.oasis_host_unregister(tv)


# --------------------------------------------------------------------- attention
def _attn_case(wl, ctx_len=None, empty_frac=0.0, seed=0, scale=None):
    cfg = wl.config()
    B, H, Hq, S = wl.batch, wl.num_kv_heads, wl.num_q_heads, wl.slots
    rs = np.random.default_rng(seed)
    pk = W.to_bf16_bits(rs.standard_normal((B, H, S, 16, 128)).astype(np.float32) * 0.7)
    pv = W.to_bf16_bits(rs.standard_normal((B, H, S, 16, 128)).astype(np.float32))
    q = W.to_bf16_bits(rs.standard_normal((B, Hq, 128)).astype(np.float32))
    bos = np.stack([np.stack([rs.permutation(wl.num_blocks)[:S] for _ in range(H)]) for _ in range(B)]).astype(np.int32)
    bos[rs.random(bos.shape) < empty_frac] = -1
    scale = scale if scale is not None else 1 / math.sqrt(128)
    out = torch.empty((B, Hq, 128), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(ob.oasis_attn_workspace_bytes(cfg), dtype=torch.uint8, device="cuda")
    cl = None if ctx_len is None else torch.from_numpy(np.asarray(ctx_len, np.int32)).cuda()
    for rep in range(2):  # the workspace must be reusable call after call
        ob.oasis_sparse_decode_attn(cfg, dev_bits(q), dev_bits(pk), dev_bits(pv),
                                    torch.from_numpy(bos).cuda(), cl, scale, out, ws)
        torch.cuda.synchronize()
        ref = oracle.sparse_decode_attn(cfg, q, pk, pv, bos, None if ctx_len is None else np.asarray(ctx_len, np.int32), scale)
        assert_attn_close(bf16_to_bits(out), ref, f"{wl.name} rep {rep}")
    assert ob.oasis_device_errors() == 0
    return bf16_to_bits(out), ref


def test_attention_llama_layer_full_size():
    _attn_case(W.LLAMA8B_LAYER, seed=1)


def test_attention_shapes_masks_and_empty_slots():
    _attn_case(W.TINY, seed=2)                                             # S = 64, one CTA per unit
    _attn_case(W.LONG_CTX.with_(layers=1), seed=3)                         # G = 8
    _attn_case(small_wl(kv_budget_tokens=16 * 37, top_k=20), seed=4, empty_frac=0.3)  # ragged S
    wl = small_wl(batch=3)
    _attn_case(wl, ctx_len=[16 * 203, 1000, 37], seed=5)                  # ragged context lengths
    _attn_case(small_wl(num_q_heads=2, num_kv_heads=2, top_k=8, kv_budget_tokens=16 * 8), seed=6)  # G = 1
    _attn_case(small_wl(num_q_heads=6, num_kv_heads=2), seed=7, scale=0.5)                       # G = 3


def test_attention_units_inside_one_warp_and_long_units():
    # many short units: several lie wholly inside one warp's slot range and are
    # finished from registers, others straddle two warps and are merged
    _attn_case(small_wl(batch=40, num_q_heads=32, num_kv_heads=8, kv_budget_tokens=16 * 3, top_k=3),
               seed=10, empty_frac=0.2)
    _attn_case(small_wl(batch=64, num_q_heads=16, num_kv_heads=8, kv_budget_tokens=16 * 2, top_k=2), seed=11)
    # one unit spread over hundreds of warps (G = 8): merged in several rounds
    _attn_case(small_wl(batch=1, num_q_heads=16, num_kv_heads=2, ctx_tokens=16 * 2048,
                        kv_budget_tokens=16 * 1024, top_k=64), seed=12, empty_frac=0.1)


def test_attention_empty_and_fully_masked_give_zeros():
    wl = small_wl()
    out, ref = _attn_case(wl, seed=8, empty_frac=1.0)
    assert not W.bf16_bits_to_f32(out).any() and not ref.any()
    out, ref = _attn_case(wl, ctx_len=[0, 0], seed=9)
    assert not W.bf16_bits_to_f32(out).any()


# --------------------------------------------------------------------- worked example
def test_worked_example_on_gpu():
    with open(os.path.join(GOLDEN, "worked_example_4block.json")) as f:
        ex = json.load(f)
    cfg = ex["config"]
    NB, D = cfg["num_blocks"], 128
    k = np.zeros((1, 1, NB, 16, D), np.float32)
    v = np.zeros((1, 1, NB, 16, D), np.float32)
    for j, key in enumerate(ex["block_keys"]):
        k[0, 0, j, :, :len(key)] = key
    for j, val in enumerate(ex["block_values"]):
        v[0, 0, j, :, :len(val)] = val
    qd = np.zeros((1, 2, 2, D), np.float32)
    for l in range(2):
        for g in range(2):
            vec = ex["draft_queries_l_g"][l][g]
            qd[0, l, g, :len(vec)] = vec
    q = np.zeros((1, 2, D), np.float32)
    for g, vec in enumerate(ex["decode_queries"]):
        q[0, g, :len(vec)] = vec
    kb, vb = W.to_bf16_bits(k), W.to_bf16_bits(v)
    bos0 = np.asarray(ex["initial_block_of_slot"], np.int32).reshape(1, 1, 2)
    sob0 = np.full((1, 1, NB), -1, np.int32)
    for s, j in enumerate(bos0[0, 0]):
        sob0[0, 0, j] = s
    lu0 = np.asarray(ex["initial_last_used"], np.int32).reshape(1, 1, 2)
    st = LayerState(cfg, bits_to_bf16(kb), bits_to_bf16(vb), sob0, bos0, lu0)
    st.scale = math.log(3.0)
    st.predict(dev_bits(W.to_bf16_bits(qd)), ex["step"])
    st.fetch()
    st.attention(dev_bits(W.to_bf16_bits(q)))
    torch.cuda.synchronize()
    assert st.summ.cpu().numpy()[0, 0, :, :2].tolist() == ex["expected_summaries"]
    assert st.scores.cpu().numpy()[0, 0].tolist() == ex["expected_scores"]
    assert st.topk.cpu().numpy()[0, 0].tolist() == ex["expected_topk"]
    assert st.fetch_block.cpu().numpy()[0, 0].tolist() == ex["expected_fetch_block"]
    assert st.fetch_slot.cpu().numpy()[0, 0].tolist() == ex["expected_fetch_slot"]
    assert st.evict_block.cpu().numpy()[0, 0].tolist() == ex["expected_evict_block"]
    assert st.block_of_slot.cpu().numpy()[0, 0].tolist() == ex["expected_block_of_slot"]
    assert st.slot_of_block.cpu().numpy()[0, 0].tolist() == ex["expected_slot_of_block"]
    assert st.last_used.cpu().numpy()[0, 0].tolist() == ex["expected_last_used"]
    out = W.bf16_bits_to_f32(bf16_to_bits(st.out))[0, :, :4]
    assert np.allclose(out, np.asarray(ex["expected_attention_out"]), atol=ATOL, rtol=RTOL)
    st.close()


def test_plan_clocked_equals_plan_with_step():
    rs = np.random.default_rng(31)
    B, H, NB, S, K = 2, 3, 512, 64, 48
    cfg = dict(batch=B, num_q_heads=H, num_kv_heads=H, head_dim=128, block_size=16, num_blocks=NB,
               kv_budget_tokens=16 * S, lookahead=1, top_k=K, fetch_ratio=0.1, sink_blocks=0,
               local_blocks=0)
    sob, bos, lu = _random_state(rs, B, H, NB, S, True)
    a = [torch.from_numpy(x.copy()).cuda() for x in (sob, bos, lu)]
    b = [torch.from_numpy(x.copy()).cuda() for x in (sob, bos, lu)]
    w = max(oracle.fetch_cap(cfg), 1)
    oa = [torch.zeros((B, H, w), dtype=torch.int32, device="cuda") for _ in range(3)] + \
         [torch.zeros((B, H), dtype=torch.int32, device="cuda") for _ in range(2)]
    obuf = [torch.zeros_like(x) for x in oa]
    clock = torch.full((B, H), 7, dtype=torch.int32, device="cuda")
    for t in range(7, 12):
        topk = torch.from_numpy(oracle.select_topk(cfg, rs.standard_normal((B, H, NB)).astype(np.float32))).cuda()
        ob.oasis_plan_fetch(cfg, topk, t, *a, *oa)
        ob.oasis_plan_fetch_clocked(cfg, topk, clock, *b, *obuf)
        torch.cuda.synchronize()
        for x, y in zip(a + oa, b + obuf):
            assert torch.equal(x, y)
        assert (clock == t + 1).all()


@pytest.mark.parametrize("NB,S,K,ratio,sink,local", [
    (2048, 128, 128, 0.05, 0, 0), (8192, 128, 128, 0.02, 1, 4), (300, 40, 30, 0.5, 2, 2),
    (5000, 1024, 1000, -1.0, 0, 0), (64, 8, 8, 0.0, 0, 0)])
def test_predict_select_fused_equals_separate(NB, S, K, ratio, sink, local):
    rs = np.random.default_rng(NB + K)
    B, H = 2, 3
    cfg = dict(batch=B, num_q_heads=H, num_kv_heads=H, head_dim=128, block_size=16, num_blocks=NB,
               kv_budget_tokens=16 * S, lookahead=1, top_k=K, fetch_ratio=ratio, sink_blocks=sink,
               local_blocks=local)
    sob, bos, lu = _random_state(rs, B, H, NB, S, full=(S <= NB))
    w = max(oracle.fetch_cap(cfg), 1)

    def bufs():
        st = [torch.from_numpy(x.copy()).cuda() for x in (sob, bos, lu)]
        out = [torch.full((B, H, w), -9, dtype=torch.int32, device="cuda") for _ in range(3)] + \
              [torch.full((B, H), -9, dtype=torch.int32, device="cuda") for _ in range(2)]
        return st, out, torch.full((B, H, K), -9, dtype=torch.int32, device="cuda")

    a_st, a_out, a_topk = bufs()
    b_st, b_out, b_topk = bufs()
    clock = torch.full((B, H), 3, dtype=torch.int32, device="cuda")
    for t in range(3, 7):
        scores = torch.from_numpy(rs.standard_normal((B, H, NB)).astype(np.float32)).cuda()
        ob.oasis_select_topk(cfg, scores, a_topk)
        ob.oasis_plan_fetch(cfg, a_topk, t, *a_st, *a_out)
        if t % 2:
            ob.oasis_predict_select(cfg, scores, 0, clock, b_topk, *b_st, *b_out)
        else:
            ob.oasis_predict_select(cfg, scores, t, None, b_topk, *b_st, *b_out)
            clock += 1
        torch.cuda.synchronize()
        assert torch.equal(a_topk, b_topk)
        for x, y in zip(a_st + a_out, b_st + b_out):
            assert torch.equal(x, y)
        # and the oracle agrees on the plan
    assert ob.oasis_device_errors() == 0
