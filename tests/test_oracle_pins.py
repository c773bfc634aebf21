"""Pins for the CPU oracle: each check ties the oracle to something other than
itself -- the hand-computed worked example, closed forms, textbook special
cases computed by scipy, brute force on tiny inputs, and the invariants that
"OasisKV: Scaling In-Decode KV Cache Beyond HBM with Lookahead Sparse
Prefetching" fixes (per-step fetch cap, Tab. 2; bounded working set, Fig. 9).

Every ``test_*`` here takes no arguments so that the mutant check
(test_oracle_mutants.py) can rerun the whole set against a deliberately
broken oracle build.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
from scipy.special import softmax

import oracle
from sparse_kv_cache_oasis_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def bf(x):
    return W.to_bf16_bits(np.asarray(x, dtype=np.float32))


def f32(b):
    return W.bf16_bits_to_f32(b)


def small_cfg(**kw):
    base = dict(batch=1, num_q_heads=2, num_kv_heads=1, head_dim=128, block_size=16,
                num_blocks=8, kv_budget_tokens=64, lookahead=2, top_k=4, fetch_ratio=0.5,
                sink_blocks=0, local_blocks=0)
    base.update(kw)
    return base


# ----------------------------------------------------------------------------
# worked example (tests/golden/worked_example_4block.json)
# ----------------------------------------------------------------------------
def _worked():
    with open(os.path.join(GOLDEN, "worked_example_4block.json")) as f:
        ex = json.load(f)
    cfg = ex["config"]
    NB, bs, D = cfg["num_blocks"], cfg["block_size"], cfg["head_dim"]
    k = np.zeros((1, 1, NB, bs, D), np.float32)
    v = np.zeros((1, 1, NB, bs, D), np.float32)
    for j, key in enumerate(ex["block_keys"]):
        k[0, 0, j, :, :len(key)] = key
    for j, val in enumerate(ex["block_values"]):
        v[0, 0, j, :, :len(val)] = val
    L, G = cfg["lookahead"], cfg["num_q_heads"]
    qd = np.zeros((1, L, G, D), np.float32)
    for l in range(L):
        for g in range(G):
            vec = ex["draft_queries_l_g"][l][g]
            qd[0, l, g, :len(vec)] = vec
    q = np.zeros((1, G, D), np.float32)
    for g, vec in enumerate(ex["decode_queries"]):
        q[0, g, :len(vec)] = vec
    return ex, cfg, bf(k), bf(v), bf(qd), bf(q)


def test_worked_example_summaries_scores_topk():
    ex, cfg, k, v, qd, q = _worked()
    summ = oracle.build_summaries(cfg, k)
    for j, exp in enumerate(ex["expected_summaries"]):
        assert np.array_equal(summ[0, 0, j, :len(exp)], np.asarray(exp, np.float32))
        assert not summ[0, 0, j, len(exp):].any()
    scores = oracle.score_blocks(cfg, qd, summ)
    assert np.array_equal(scores[0, 0], np.asarray(ex["expected_scores"], np.float32))
    topk = oracle.select_topk(cfg, scores)
    assert topk[0, 0].tolist() == ex["expected_topk"]
    assert oracle.fetch_cap(cfg) == ex["expected_fetch_cap"]


def test_worked_example_plan_fetch_attention():
    ex, cfg, k, v, qd, q = _worked()
    NB = cfg["num_blocks"]
    S = cfg["kv_budget_tokens"] // cfg["block_size"]
    bos = np.asarray(ex["initial_block_of_slot"], np.int32).reshape(1, 1, S)
    sob = np.full((1, 1, NB), -1, np.int32)
    for s, j in enumerate(bos[0, 0]):
        sob[0, 0, j] = s
    lu = np.asarray(ex["initial_last_used"], np.int32).reshape(1, 1, S)
    topk = np.asarray(ex["expected_topk"], np.int32).reshape(1, 1, -1)
    plan = oracle.plan_fetch(cfg, topk, ex["step"], sob, bos, lu)
    assert plan["n_fetch"][0, 0] == len(ex["expected_fetch_block"])
    assert plan["n_evict"][0, 0] == len(ex["expected_evict_block"])
    assert plan["fetch_block"][0, 0].tolist() == ex["expected_fetch_block"]
    assert plan["fetch_slot"][0, 0].tolist() == ex["expected_fetch_slot"]
    assert plan["evict_block"][0, 0].tolist() == ex["expected_evict_block"]
    assert bos[0, 0].tolist() == ex["expected_block_of_slot"]
    assert sob[0, 0].tolist() == ex["expected_slot_of_block"]
    assert lu[0, 0].tolist() == ex["expected_last_used"]
    # pool as it was before the step, then the transfer
    pk, pv = W.initial_pool(dict_to_wl(cfg), k, v, np.asarray(ex["initial_block_of_slot"], np.int32).reshape(1, 1, S))
    oracle.fetch_blocks(cfg, k, v, plan["fetch_block"], plan["fetch_slot"], plan["n_fetch"], pk, pv)
    for s, j in enumerate(bos[0, 0]):
        assert np.array_equal(pk[0, 0, s], k[0, 0, j]) and np.array_equal(pv[0, 0, s], v[0, 0, j])
    out = oracle.sparse_decode_attn(cfg, q, pk, pv, bos, None, math.log(3.0))
    exp = np.asarray(ex["expected_attention_out"], np.float32)
    assert np.allclose(out[0, :, :exp.shape[1]], exp, atol=1e-6, rtol=0)
    assert not out[0, :, exp.shape[1]:].any()


def dict_to_wl(cfg):
    return W.Workload(name="cfg", batch=cfg["batch"], num_q_heads=cfg["num_q_heads"],
                      num_kv_heads=cfg["num_kv_heads"], ctx_tokens=cfg["num_blocks"] * cfg["block_size"],
                      kv_budget_tokens=cfg["kv_budget_tokens"], lookahead=cfg["lookahead"],
                      top_k=cfg["top_k"], fetch_ratio=cfg["fetch_ratio"], seed=0,
                      head_dim=cfg["head_dim"], block_size=cfg["block_size"],
                      sink_blocks=cfg["sink_blocks"], local_blocks=cfg["local_blocks"])


# ----------------------------------------------------------------------------
# summaries: closed forms and exact rounding
# ----------------------------------------------------------------------------
def test_summary_closed_forms():
    cfg = small_cfg(num_blocks=4, num_kv_heads=2, num_q_heads=2, batch=2)
    D, bs = 128, 16
    k = np.zeros((2, 2, 4, bs, D), np.float32)
    # constant block -> that constant
    k[0, 0, 0] = np.linspace(-3, 3, D, dtype=np.float32)
    # half the tokens at 2, half at 0 -> 1
    k[0, 1, 1, :8, 0] = 2.0
    # token t holds t -> mean 7.5
    k[1, 0, 2, :, 5] = np.arange(bs, dtype=np.float32)
    # a single token of 1 -> 1/16, only in block 3 of (b=1, h=1)
    k[1, 1, 3, 11, 7] = 1.0
    kb = bf(k)
    summ = oracle.build_summaries(cfg, kb)
    assert np.array_equal(summ[0, 0, 0], f32(kb[0, 0, 0, 0]))
    assert summ[0, 1, 1, 0] == 1.0 and np.count_nonzero(summ[0, 1]) == 1
    assert summ[1, 0, 2, 5] == 7.5 and np.count_nonzero(summ[1, 0]) == 1
    assert summ[1, 1, 3, 7] == 1.0 / 16 and np.count_nonzero(summ[1, 1]) == 1
    assert np.count_nonzero(summ[0, 0, 1:]) == 0


def test_summary_rounding_is_exact_mean_rounded_once():
    cfg = small_cfg(num_blocks=1, top_k=1)
    rs = np.random.default_rng(11)
    k = bf(rs.standard_normal((1, 1, 1, 16, 128)).astype(np.float32) * 3)
    summ = oracle.build_summaries(cfg, k)
    kf = f32(k)
    for d in range(128):
        exact = sum(Fraction(float(kf[0, 0, 0, t, d])) for t in range(16)) / 16
        # the exact mean of 16 bf16 values fits a double, so this rounds once
        assert summ[0, 0, 0, d] == np.float32(float(exact))


# ----------------------------------------------------------------------------
# scoring: special cases and the GQA / draft-token index structure
# ----------------------------------------------------------------------------
def test_score_single_query_is_a_dot_product():
    cfg = small_cfg(num_q_heads=1, lookahead=1, num_blocks=16, top_k=4)
    rs = np.random.default_rng(3)
    qd = bf(rs.standard_normal((1, 1, 1, 128)).astype(np.float32))
    summ = rs.standard_normal((1, 1, 16, 128)).astype(np.float32)
    sc = oracle.score_blocks(cfg, qd, summ)
    ref = summ[0, 0].astype(np.float64) @ f32(qd[0, 0, 0]).astype(np.float64)
    assert np.array_equal(sc[0, 0], ref.astype(np.float32))


def test_score_gqa_group_and_draft_index():
    # Hkv = 2, G = 2, L = 2, B = 2.  Only query heads of KV head 0 point along
    # +e0 in request 0; KV head 1's group points along -e0.  In request 1 only
    # draft token 1 is non-zero.
    cfg = small_cfg(batch=2, num_q_heads=4, num_kv_heads=2, lookahead=2, num_blocks=3, top_k=2)
    qd = np.zeros((2, 2, 4, 128), np.float32)
    qd[0, :, 0:2, 0] = 1.0
    qd[0, :, 2:4, 0] = -1.0
    qd[1, 1, 3, 1] = 3.0
    summ = np.zeros((2, 2, 3, 128), np.float32)
    summ[:, :, :, 0] = 1.0
    summ[:, :, :, 1] = [1.0, 2.0, -1.0]
    sc = oracle.score_blocks(cfg, bf(qd), summ)
    assert sc[0, 0].tolist() == [1.0, 1.0, 1.0]
    assert sc[0, 1].tolist() == [-1.0, -1.0, -1.0]
    assert sc[1, 0].tolist() == [0.0, 0.0, 0.0]
    assert sc[1, 1].tolist() == [3.0, 6.0, 0.0]   # max(0 from zero rows, 3*summ)


def test_score_is_max_not_sum_and_homogeneous():
    cfg = small_cfg(num_q_heads=2, lookahead=2, num_blocks=32, top_k=4)
    rs = np.random.default_rng(5)
    qd = bf(rs.standard_normal((1, 2, 2, 128)).astype(np.float32))
    summ = rs.standard_normal((1, 1, 32, 128)).astype(np.float32)
    sc = oracle.score_blocks(cfg, qd, summ)
    # each query row alone bounds the score from below, and one row attains it
    rows = [oracle.score_blocks(small_cfg(num_q_heads=1, lookahead=1, num_blocks=32, top_k=4),
                                np.ascontiguousarray(qd[:, l:l + 1, g:g + 1]), summ)[0, 0]
            for l in range(2) for g in range(2)]
    rows = np.stack(rows)
    assert np.array_equal(sc[0, 0], rows.max(axis=0))
    # permuting draft tokens and group members leaves the score unchanged
    sc2 = oracle.score_blocks(cfg, np.ascontiguousarray(qd[:, ::-1, ::-1]), summ)
    assert np.array_equal(sc, sc2)
    # doubling the summaries doubles the score exactly
    sc3 = oracle.score_blocks(cfg, qd, summ * 2)
    assert np.array_equal(sc3, sc * 2)


# ----------------------------------------------------------------------------
# top-K: brute force over all subsets, ties, forced blocks
# ----------------------------------------------------------------------------
def _dominates(a, b, s):
    return s[a] > s[b] or (s[a] == s[b] and a < b)


def test_topk_brute_force_with_ties():
    rs = np.random.default_rng(7)
    for trial in range(60):
        NB = int(rs.integers(4, 9))
        K = int(rs.integers(1, NB + 1))
        cfg = small_cfg(num_blocks=NB, top_k=K, kv_budget_tokens=16 * max(K, 1))
        s = rs.integers(-2, 3, size=NB).astype(np.float32) * 0.5   # many ties
        ids = oracle.select_topk(cfg, s.reshape(1, 1, NB))[0, 0].tolist()
        winners = [T for T in itertools.combinations(range(NB), K)
                   if all(_dominates(a, b, s) for a in T for b in range(NB) if b not in T)]
        assert len(winners) == 1
        assert sorted(ids) == list(winners[0])
        # output order: score descending, then id ascending
        assert all(_dominates(ids[i], ids[i + 1], s) for i in range(K - 1))


def test_topk_all_equal_scores_pick_lowest_ids():
    cfg = small_cfg(num_blocks=8, top_k=3)
    ids = oracle.select_topk(cfg, np.zeros((1, 1, 8), np.float32))
    assert ids[0, 0].tolist() == [0, 1, 2]


def test_topk_forced_blocks_first_and_counted():
    cfg = small_cfg(num_blocks=10, top_k=5, kv_budget_tokens=80, sink_blocks=1, local_blocks=2)
    s = np.asarray([-5, 1, 9, 3, 8, 2, 7, 0, -1, -2], np.float32).reshape(1, 1, 10)
    ids = oracle.select_topk(cfg, s)[0, 0].tolist()
    assert ids == [0, 8, 9, 2, 4]
    with pytest.raises(ValueError):
        oracle.select_topk(small_cfg(num_blocks=10, top_k=2, kv_budget_tokens=80, sink_blocks=1,
                                     local_blocks=2), s)


# ----------------------------------------------------------------------------
# fetch cap: Tab. 2 ratios on a 128-block budget
# ----------------------------------------------------------------------------
def test_fetch_cap_tab2_ratios():
    base = small_cfg(num_blocks=2048, kv_budget_tokens=2048, top_k=128)
    expect = {0.01: 2, 0.02: 3, 0.05: 7, 0.10: 13, 0.20: 26, -1.0: 128, 1.0: 128, 0.0: 0}
    for r, cap in expect.items():
        assert oracle.fetch_cap(dict(base, fetch_ratio=r)) == cap
    assert oracle.fetch_cap(dict(base, kv_budget_tokens=1024, top_k=32, fetch_ratio=4 / 64)) == 4
    assert oracle.fetch_cap(dict(base, kv_budget_tokens=130 * 16, top_k=128, fetch_ratio=0.1)) == 13


# ----------------------------------------------------------------------------
# plan: invariants over random multi-step trajectories
# ----------------------------------------------------------------------------
def _check_plan_step(cfg, topk, step, sob0, bos0, lu0, sob, bos, lu, plan):
    NB, S, K = cfg["num_blocks"], cfg["kv_budget_tokens"] // cfg["block_size"], cfg["top_k"]
    cap = oracle.fetch_cap(cfg)
    for b in range(cfg["batch"]):
        for h in range(cfg["num_kv_heads"]):
            P = topk[b, h].tolist()
            R0 = {int(j) for j in bos0[b, h] if j >= 0}
            R1 = {int(j) for j in bos[b, h] if j >= 0}
            n, e = int(plan["n_fetch"][b, h]), int(plan["n_evict"][b, h])
            fb = plan["fetch_block"][b, h][:n].tolist()
            fs = plan["fetch_slot"][b, h][:n].tolist()
            eb = plan["evict_block"][b, h][:e].tolist()
            missing = [p for p in P if p not in R0]
            assert n == min(len(missing), cap) and n <= cap            # cap (Tab. 2)
            assert len(R1) <= S                                        # budget (Fig. 9)
            assert sorted(fb) == fb and set(fb) == set(missing[:n])    # highest priority first
            assert sorted(eb) == eb and set(eb) <= R0 - set(P)         # victims outside P
            assert R1 == (R0 - set(eb)) | set(fb)
            assert e == max(0, len(R0) + n - S)
            # LRU: every victim is older (or equal and lower id) than every kept candidate
            kept = [(int(lu0[b, h, s]), int(bos0[b, h, s])) for s in range(S)
                    if bos0[b, h, s] >= 0 and bos0[b, h, s] not in P and bos0[b, h, s] not in eb]
            vict = [(int(lu0[b, h, sob0[b, h, j]]), j) for j in eb]
            assert all(v < kk for v in vict for kk in kept)
            # slots: ascending free slots paired with ascending block ids
            free = sorted([s for s in range(S) if bos0[b, h, s] < 0] + [int(sob0[b, h, j]) for j in eb])
            assert fs == free[:n]
            # maps are mutual inverses
            for s in range(S):
                if bos[b, h, s] >= 0:
                    assert sob[b, h, bos[b, h, s]] == s
            assert np.count_nonzero(sob[b, h] >= 0) == len(R1)
            # last_used: predicted-resident and fetched blocks are used at `step`
            for s in range(S):
                j = bos[b, h, s]
                if j >= 0 and (j in P):
                    assert lu[b, h, s] == step
                elif j >= 0:
                    assert lu[b, h, s] == lu0[b, h, s]
            if len(missing) <= cap:
                assert set(P) <= R1
            # forced blocks are never evicted
            forced = [j for j in range(NB) if j < cfg["sink_blocks"] or j >= NB - cfg["local_blocks"]]
            assert not (set(eb) & set(forced))


def test_plan_invariants_random_trajectories():
    rs = np.random.default_rng(13)
    for trial in range(12):
        NB = int(rs.integers(16, 48))
        S = int(rs.integers(4, 12))
        K = int(rs.integers(2, S + 1))
        ratio = float(rs.choice([0.1, 0.25, 0.5, -1.0]))
        sink, local = (1, 2) if trial % 3 == 0 else (0, 0)
        K = max(K, sink + local + 1)
        S = max(S, K)
        cfg = small_cfg(batch=2, num_kv_heads=2, num_q_heads=2, num_blocks=NB,
                        kv_budget_tokens=16 * S, top_k=K, fetch_ratio=ratio,
                        sink_blocks=sink, local_blocks=local)
        sob = np.full((2, 2, NB), -1, np.int32)
        bos = np.full((2, 2, S), -1, np.int32)
        lu = np.full((2, 2, S), -1, np.int32)
        for b in range(2):
            for h in range(2):
                nres = int(rs.integers(0, S + 1))
                blocks = rs.choice(NB, size=nres, replace=False)
                slots = rs.choice(S, size=nres, replace=False)
                bos[b, h, slots] = blocks
                sob[b, h, blocks] = slots
        for step in range(8):
            scores = rs.standard_normal((2, 2, NB)).astype(np.float32)
            topk = oracle.select_topk(cfg, scores)
            sob0, bos0, lu0 = sob.copy(), bos.copy(), lu.copy()
            plan = oracle.plan_fetch(cfg, topk, step, sob, bos, lu)
            _check_plan_step(cfg, topk, step, sob0, bos0, lu0, sob, bos, lu, plan)


def test_plan_rejects_inconsistent_state():
    cfg = small_cfg(num_blocks=8, kv_budget_tokens=32, top_k=2)
    sob = np.full((1, 1, 8), -1, np.int32)
    bos = np.asarray([[[3, -1]]], np.int32)        # slot 0 claims block 3, map disagrees
    sob[0, 0, 3] = 1
    lu = np.full((1, 1, 2), -1, np.int32)
    with pytest.raises(ValueError):
        oracle.plan_fetch(cfg, np.asarray([[[3, 4]]], np.int32), 0, sob, bos, lu)
    with pytest.raises(ValueError):
        oracle.plan_fetch(cfg, np.asarray([[[5, 5]]], np.int32), 0,
                          np.full((1, 1, 8), -1, np.int32), np.full((1, 1, 2), -1, np.int32), lu)


# ----------------------------------------------------------------------------
# fetch: byte copies, range checks
# ----------------------------------------------------------------------------
def test_fetch_copies_bytes_and_checks_ranges():
    cfg = small_cfg(batch=1, num_kv_heads=2, num_q_heads=2, num_blocks=6, kv_budget_tokens=48,
                    top_k=3, fetch_ratio=-1.0)
    rs = np.random.default_rng(2)
    hk = rs.integers(0, 65535, size=(1, 2, 6, 16, 128), dtype=np.uint16)
    hv = rs.integers(0, 65535, size=(1, 2, 6, 16, 128), dtype=np.uint16)
    pk = np.zeros((1, 2, 3, 16, 128), np.uint16)
    pv = np.zeros_like(pk)
    fb = np.asarray([[[1, 4, -1], [0, -1, -1]]], np.int32)
    fs = np.asarray([[[2, 0, -1], [1, -1, -1]]], np.int32)
    nf = np.asarray([[2, 1]], np.int32)
    oracle.fetch_blocks(cfg, hk, hv, fb, fs, nf, pk, pv)
    assert np.array_equal(pk[0, 0, 2], hk[0, 0, 1]) and np.array_equal(pv[0, 0, 0], hv[0, 0, 4])
    assert np.array_equal(pk[0, 1, 1], hk[0, 1, 0]) and not pk[0, 0, 1].any() and not pk[0, 1, 0].any()
    with pytest.raises(ValueError):
        oracle.fetch_blocks(cfg, hk, hv, np.asarray([[[6, -1, -1], [0, -1, -1]]], np.int32), fs, nf, pk, pv)


# ----------------------------------------------------------------------------
# attention: textbook softmax attention (scipy), closed forms, masking
# ----------------------------------------------------------------------------
def _scipy_attention(q, k, v, scale):
    """softmax(q k^T * scale) v with scipy, float64; q [Hq,D], k/v [Hkv,T,D]."""
    Hq, Hkv = q.shape[0], k.shape[0]
    G = Hq // Hkv
    out = np.zeros((Hq, q.shape[1]))
    for hq in range(Hq):
        w = softmax(k[hq // G] @ q[hq] * scale)
        out[hq] = w @ v[hq // G]
    return out


def test_dense_attention_matches_scipy_softmax():
    cfg = small_cfg(batch=2, num_q_heads=4, num_kv_heads=2, num_blocks=5, kv_budget_tokens=80, top_k=2)
    rs = np.random.default_rng(17)
    q = bf(rs.standard_normal((2, 4, 128)).astype(np.float32))
    k = bf(rs.standard_normal((2, 2, 5, 16, 128)).astype(np.float32))
    v = bf(rs.standard_normal((2, 2, 5, 16, 128)).astype(np.float32))
    ctx = np.asarray([80, 37], np.int32)
    out = oracle.dense_decode_attn(cfg, q, k, v, ctx, 0.125)
    for b in range(2):
        T = int(ctx[b])
        kk = f32(k[b]).reshape(2, 80, 128)[:, :T].astype(np.float64)
        vv = f32(v[b]).reshape(2, 80, 128)[:, :T].astype(np.float64)
        ref = _scipy_attention(f32(q[b]).astype(np.float64), kk, vv, 0.125)
        assert np.allclose(out[b], ref, rtol=1e-6, atol=1e-7)


def test_sparse_equals_dense_when_every_block_is_resident():
    # all NB blocks resident in a shuffled slot order: sparse attention == dense
    wl = W.TINY.with_(kv_budget_tokens=W.TINY.ctx_tokens, top_k=W.TINY.num_blocks)
    cfg = wl.config()
    qs = W.query_sequence(wl)
    k, v = W.gen_kv(wl, 0, qs)
    q, _ = W.step_queries(wl, qs, 0)
    sob, bos, lu = W.initial_resident(wl)
    assert (bos >= 0).all()
    pk, pv = W.initial_pool(wl, k, v, bos)
    sparse = oracle.sparse_decode_attn(cfg, q, pk, pv, bos)
    dense = oracle.dense_decode_attn(cfg, q, k, v)
    assert np.allclose(sparse, dense, rtol=1e-5, atol=1e-7)


def test_attention_closed_forms_and_masking():
    cfg = small_cfg(batch=2, num_q_heads=2, num_kv_heads=1, num_blocks=4, kv_budget_tokens=48, top_k=3)
    rs = np.random.default_rng(23)
    q = bf(rs.standard_normal((2, 2, 128)).astype(np.float32))
    pk = np.zeros((2, 1, 3, 16, 128), np.float32)
    pk[:] = rs.standard_normal(128).astype(np.float32)            # identical keys -> uniform weights
    pv = rs.standard_normal((2, 1, 3, 16, 128)).astype(np.float32)
    pkb, pvb = bf(pk), bf(pv)
    bos = np.asarray([[[2, -1, 0]], [[1, 3, 0]]], np.int32)
    out = oracle.sparse_decode_attn(cfg, q, pkb, pvb, bos)
    vf = f32(pvb)
    assert np.allclose(out[0, 0], vf[0, 0, [0, 2]].reshape(-1, 128).mean(0), rtol=1e-6, atol=1e-7)
    assert np.allclose(out[1, 1], vf[1, 0].reshape(-1, 128).mean(0), rtol=1e-6, atol=1e-7)
    # ctx_len: request 1 sees tokens < 17 -> block 0 (slot 2, 16 tokens) + token 16 (block 1, slot 0, t=0)
    ctx = np.asarray([64, 17], np.int32)
    out = oracle.sparse_decode_attn(cfg, q, pkb, pvb, bos, ctx)
    vis = np.concatenate([vf[1, 0, 2], vf[1, 0, 0, :1]])
    assert np.allclose(out[1, 0], vis.mean(0), rtol=1e-6, atol=1e-7)
    # nothing visible -> zeros; empty working set -> zeros
    out = oracle.sparse_decode_attn(cfg, q, pkb, pvb, np.full((2, 1, 3), -1, np.int32))
    assert not out.any()
    out = oracle.sparse_decode_attn(cfg, q, pkb, pvb, bos, np.asarray([0, 0], np.int32))
    assert not out.any()


# ----------------------------------------------------------------------------
# min/max compressed keys
# ----------------------------------------------------------------------------
def test_minmax_summaries_are_columnwise_extremes():
    cfg = small_cfg(batch=2, num_q_heads=4, num_kv_heads=2, num_blocks=3, top_k=2)
    rs = np.random.default_rng(41)
    k = bf(rs.standard_normal((2, 2, 3, 16, 128)).astype(np.float32))
    # +0 / -0 ties: block (0,0,0) dim 0 holds -0 first, then +0 (all else positive)
    k[0, 0, 0, :, 0] = bf(np.full(16, 1.5, np.float32))
    k[0, 0, 0, 3, 0], k[0, 0, 0, 9, 0] = 0x8000, 0x0000
    mm = oracle.build_summaries_minmax(cfg, k)
    kf = f32(k)
    assert np.array_equal(f32(mm[:, :, :, 0]), kf.max(axis=3))
    assert np.array_equal(f32(mm[:, :, :, 1]), kf.min(axis=3))
    assert mm[0, 0, 0, 1, 0] == 0x8000 and mm[0, 0, 0, 0, 0] == bf(1.5)
    # every stored value is one of the block's own key values (bit for bit)
    for idx in [(1, 1, 2, 0, 17), (0, 1, 1, 1, 100)]:
        b, h, j, r, d = idx
        assert mm[idx] in set(k[b, h, j, :, d].tolist())


def test_minmax_score_is_the_box_bound():
    """sum_d max(q_d mn_d, q_d mx_d) is the largest q.x over the box
    [mn, mx]: with D = 4 the 16 corners give it by brute force."""
    cfg = small_cfg(head_dim=4, num_blocks=5, lookahead=3, num_q_heads=2, num_kv_heads=1)
    rs = np.random.default_rng(42)
    k = bf(rs.standard_normal((1, 1, 5, 16, 4)).astype(np.float32))
    qd = bf(rs.standard_normal((1, 3, 2, 4)).astype(np.float32))
    mm = oracle.build_summaries_minmax(cfg, k)
    sc = oracle.score_blocks_minmax(cfg, qd, mm)
    mx, mn = f32(mm[0, 0, :, 0]).astype(np.float64), f32(mm[0, 0, :, 1]).astype(np.float64)
    q = f32(qd[0]).astype(np.float64).reshape(6, 4)
    for j in range(5):
        corners = np.array([[mx[j, d] if (c >> d) & 1 else mn[j, d] for d in range(4)]
                            for c in range(16)])
        want = (q @ corners.T).max()
        assert sc[0, 0, j] == np.float32(want)
        # an upper bound of every key of the block, for every draft query
        assert sc[0, 0, j] >= (q @ f32(k[0, 0, j]).astype(np.float64).T).max() - 1e-6


def test_minmax_score_closed_forms():
    cfg = small_cfg(num_blocks=4, lookahead=1, num_q_heads=1, num_kv_heads=1)
    rs = np.random.default_rng(43)
    k = bf(rs.standard_normal((1, 1, 4, 16, 128)).astype(np.float32))
    # block 3: all 16 keys equal -> min = max = the key -> the plain dot product
    k[0, 0, 3] = k[0, 0, 3, 5]
    mm = oracle.build_summaries_minmax(cfg, k)
    kf = f32(k).astype(np.float64)
    qpos = bf(np.abs(rs.standard_normal((1, 1, 1, 128))).astype(np.float32))
    qneg = bf(-np.abs(rs.standard_normal((1, 1, 1, 128))).astype(np.float32))
    qp, qn = f32(qpos[0, 0, 0]).astype(np.float64), f32(qneg[0, 0, 0]).astype(np.float64)
    sp = oracle.score_blocks_minmax(cfg, qpos, mm)[0, 0]
    sn = oracle.score_blocks_minmax(cfg, qneg, mm)[0, 0]
    for j in range(4):
        assert sp[j] == np.float32(qp @ kf[0, 0, j].max(axis=0))   # q >= 0 picks the max row
        assert sn[j] == np.float32(qn @ kf[0, 0, j].min(axis=0))   # q <= 0 picks the min row
    assert sp[3] == np.float32(qp @ kf[0, 0, 3, 0])
    # a constant block scores as its mean key does (the mean is that key)
    summ = oracle.build_summaries(cfg, k)
    assert oracle.score_blocks(cfg, qpos, summ)[0, 0, 3] == sp[3]


def test_minmax_score_max_over_drafts_and_group():
    # the block's score is the best (l, g) bound; head h reads only its own group
    cfg = small_cfg(num_blocks=3, lookahead=2, num_q_heads=4, num_kv_heads=2, top_k=2)
    rs = np.random.default_rng(44)
    k = bf(rs.standard_normal((1, 2, 3, 16, 128)).astype(np.float32))
    qd = bf(rs.standard_normal((1, 2, 4, 128)).astype(np.float32))
    mm = oracle.build_summaries_minmax(cfg, k)
    sc = oracle.score_blocks_minmax(cfg, qd, mm)
    for h in range(2):
        single = []
        for l in range(2):
            for g in range(2):
                c1 = small_cfg(num_blocks=3, lookahead=1, num_q_heads=1, num_kv_heads=1, top_k=2)
                q1 = np.ascontiguousarray(qd[:, l:l + 1, h * 2 + g:h * 2 + g + 1])
                single.append(oracle.score_blocks_minmax(c1, q1, np.ascontiguousarray(mm[:, h:h + 1]))[0, 0])
        assert np.array_equal(sc[0, h], np.max(single, axis=0))


# ----------------------------------------------------------------------------
# growing context: top-K with a sliding local window, and the append
# ----------------------------------------------------------------------------
def test_topk_ctx_hand_cases():
    # NB = 8, K = 4, sink 1, local 2; scores favour high ids except block 1
    cfg = small_cfg(num_blocks=8, kv_budget_tokens=16 * 4, top_k=4, sink_blocks=1, local_blocks=2)
    sc = np.asarray([[[0.1, 5.0, 0.2, 0.3, 7.0, 8.0, 9.0, 10.0]]], np.float32)
    def ids(ctx):
        return oracle.select_topk_ctx(cfg, sc, np.asarray([ctx], np.int32))[0, 0].tolist()
    assert ids(50) == [0, 2, 3, 1]        # 4 blocks: sink 0, window {2, 3}, then block 1 by score
    assert ids(17) == [0, 1, 2, 3]        # 2 blocks, both forced; the rest rank -inf -> lowest ids
    assert ids(0) == [0, 1, 2, 3]         # empty context: nothing forced, all -inf
    assert ids(16 * 5) == [0, 3, 4, 1]    # 5 blocks: window {3, 4}; block 1 beats block 2
    assert ids(16 * 8) == [0, 6, 7, 5]    # full context: as the plain top-K
    assert ids(16 * 8) == oracle.select_topk(cfg, sc)[0, 0].tolist()


def test_topk_ctx_full_context_is_plain_topk():
    cfg = small_cfg(batch=2, num_q_heads=4, num_kv_heads=2, num_blocks=40, kv_budget_tokens=16 * 12,
                    top_k=12, sink_blocks=2, local_blocks=3)
    sc = np.random.default_rng(45).standard_normal((2, 2, 40)).astype(np.float32)
    full = np.asarray([40 * 16, 40 * 16], np.int32)
    assert np.array_equal(oracle.select_topk_ctx(cfg, sc, full), oracle.select_topk(cfg, sc))


def _append_setup():
    B, H, NB, S = 2, 2, 6, 3
    cfg = small_cfg(batch=B, num_q_heads=H, num_kv_heads=H, num_blocks=NB, kv_budget_tokens=16 * S,
                    top_k=3, sink_blocks=1, local_blocks=1)
    rs = np.random.default_rng(46)
    hk = bf(rs.standard_normal((B, H, NB, 16, 128)).astype(np.float32))
    hv = bf(rs.standard_normal((B, H, NB, 16, 128)).astype(np.float32))
    kn = bf(rs.standard_normal((B, H, 128)).astype(np.float32))
    vn = bf(rs.standard_normal((B, H, 128)).astype(np.float32))
    bos = np.asarray([[[0, 1, -1], [0, 3, 1]], [[0, 2, 4], [0, 4, 5]]], np.int32)
    lu = np.asarray([[[4, 4, -1], [5, 2, 2]], [[1, 1, 1], [1, 3, 0]]], np.int32)
    sob = np.full((B, H, NB), -1, np.int32)
    for b in range(B):
        for h in range(H):
            for q in range(S):
                if bos[b, h, q] >= 0:
                    sob[b, h, bos[b, h, q]] = q
    pk = bf(rs.standard_normal((B, H, S, 16, 128)).astype(np.float32))
    pv = bf(rs.standard_normal((B, H, S, 16, 128)).astype(np.float32))
    summ = rs.standard_normal((B, H, NB, 128)).astype(np.float32)
    mm = bf(rs.standard_normal((B, H, NB, 2, 128)).astype(np.float32))
    return cfg, hk, hv, kn, vn, sob, bos, lu, pk, pv, summ, mm


def test_append_writes_token_summary_and_working_set():
    cfg, hk, hv, kn, vn, sob, bos, lu, pk, pv, summ, mm = _append_setup()
    hk0, pk0, pv0 = hk.copy(), pk.copy(), pv.copy()
    ctx = np.asarray([32, 40], np.int32)       # request 0 starts block 2; request 1 is at row 8 of it
    rc = oracle.append_kv(cfg, kn, vn, ctx, 9, hk, hv, sob, bos, lu, pk, pv)
    assert rc == 0 and ctx.tolist() == [33, 41]
    summ0 = summ.copy()
    oracle.refresh_summaries(cfg, ctx, hk, summ, mm)
    for b, t in ((0, 0), (1, 8)):
        for h in range(2):
            assert np.array_equal(hk[b, h, 2, t], kn[b, h]) and np.array_equal(hv[b, h, 2, t], vn[b, h])
            rows = f32(hk[b, h, 2, :t + 1]).astype(np.float64)
            assert np.array_equal(summ[b, h, 2], np.float32([math.fsum(c) / (t + 1) for c in rows.T]))
            assert np.array_equal(f32(mm[b, h, 2, 0]), rows.max(0).astype(np.float32))
            assert np.array_equal(f32(mm[b, h, 2, 1]), rows.min(0).astype(np.float32))
    # (0,0): empty slot 2 takes block 2
    assert bos[0, 0].tolist() == [0, 1, 2] and sob[0, 0, 2] == 2 and lu[0, 0, 2] == 9
    # (0,1): no empty slot; blocks 3 and 1 tie at last use 2 -> block 1 (lower id) leaves slot 2
    assert bos[0, 1].tolist() == [0, 3, 2] and sob[0, 1, 1] == -1 and lu[0, 1].tolist() == [5, 2, 9]
    # (1,0): block 2 already resident in slot 1 -> only row 8 of slot 1 changes
    assert bos[1, 0].tolist() == [0, 2, 4] and lu[1, 0].tolist() == [1, 1, 1]
    assert np.array_equal(pk[1, 0, 1, 8], kn[1, 0])
    changed = np.argwhere((pk[1, 0] != pk0[1, 0]).any(axis=-1))
    assert changed.tolist() == [[1, 8]]
    # (1,1): LRU block 5 (last use 0) leaves slot 2; rows 0-7 of block 2 come in from the cache
    assert bos[1, 1].tolist() == [0, 4, 2] and sob[1, 1, 5] == -1 and lu[1, 1, 2] == 9
    assert np.array_equal(pk[1, 1, 2, :8], hk0[1, 1, 2, :8]) and np.array_equal(pk[1, 1, 2, 8], kn[1, 1])
    assert np.array_equal(pk[1, 1, 2, 9:], pk0[1, 1, 2, 9:])      # rows past the context untouched
    # blocks other than 2 keep their summaries and cache rows
    assert np.array_equal(np.delete(hk, 2, axis=2), np.delete(hk0, 2, axis=2))
    assert np.array_equal(np.delete(summ, 2, axis=2), np.delete(summ0, 2, axis=2))


def test_refresh_of_a_full_block_is_the_build():
    cfg, hk, hv, kn, vn, sob, bos, lu, pk, pv, summ, mm = _append_setup()
    full = np.asarray([16 * 6, 16 * 3], np.int32)  # last blocks 5 and 2, both complete
    oracle.refresh_summaries(cfg, full, hk, summ, mm)
    ref, ref_mm = oracle.build_summaries(cfg, hk), oracle.build_summaries_minmax(cfg, hk)
    assert np.array_equal(summ[0, :, 5], ref[0, :, 5]) and np.array_equal(summ[1, :, 2], ref[1, :, 2])
    assert np.array_equal(mm[0, :, 5], ref_mm[0, :, 5]) and np.array_equal(mm[1, :, 2], ref_mm[1, :, 2])
    # an empty context changes nothing
    before = summ.copy()
    oracle.refresh_summaries(cfg, np.asarray([0, 0], np.int32), hk, summ, mm)
    assert np.array_equal(summ, before)


def test_append_full_context_and_no_free_slot():
    cfg, hk, hv, kn, vn, sob, bos, lu, pk, pv, summ, mm = _append_setup()
    full = dict(cfg, local_blocks=3)   # window of 3 blocks: every resident block of (0,1) is forced
    ctx = np.asarray([16 * 6, 16 * 4], np.int32)   # request 0 full; request 1 starts block 4
    bos[1, 1] = [0, 2, 3]
    lu[1, 1] = [0, 0, 0]
    sob[1, 1] = -1
    sob[1, 1, 0], sob[1, 1, 2], sob[1, 1, 3] = 0, 1, 2
    hk0, pk0, bos0, sob0 = hk.copy(), pk.copy(), bos.copy(), sob.copy()
    rc = oracle.append_kv(full, kn, vn, ctx, 3, hk, hv, sob, bos, lu, pk, pv)
    assert rc == -1 and ctx.tolist() == [96, 65]
    oracle.refresh_summaries(full, ctx, hk, summ, mm)
    assert np.array_equal(hk[0], hk0[0]) and np.array_equal(pk[0], pk0[0])   # request 0 untouched
    # (1,1): blocks 0 (sink), 2 and 3 (window of block 4) are forced: no slot, pool untouched
    assert np.array_equal(bos[1, 1], bos0[1, 1]) and np.array_equal(pk[1, 1], pk0[1, 1])
    assert np.array_equal(hk[1, 1, 4, 0], kn[1, 1])
    assert np.array_equal(summ[1, 1, 4], f32(kn[1, 1]))
    # (1,0): block 4 resident in slot 2 -> row 0 written there
    assert np.array_equal(pk[1, 0, 2, 0], kn[1, 0])
    rc = oracle.append_kv(full, kn, vn, np.asarray([5, 70], np.int32), 3, hk, hv, sob, bos, lu, pk, pv)
    assert rc == -2


def test_joint_attention_rows_follow_their_tokens():
    """Joint attention: output row l of request b, head n attends with draft
    token l-1's query (row 0: the decoded token's).  Keys are one-hot per
    token and every query points hard at one token, so each output row is
    that token's value row; a masked target falls back to the mean of the
    visible values."""
    B, G, Hkv, L, S = 2, 2, 2, 3, 4
    Hq = G * Hkv
    cfg = small_cfg(batch=B, num_q_heads=Hq, num_kv_heads=Hkv, num_blocks=6,
                    kv_budget_tokens=16 * S, lookahead=L, top_k=4)
    rs = np.random.default_rng(31)
    pk = np.zeros((B, Hkv, S, 16, 128), np.float32)
    for s_ in range(S):
        for t in range(16):
            pk[:, :, s_, t, 16 * s_ + t] = 1.0                      # token (slot s_, t) -> e_{16 s_ + t}
    pvb = bf(rs.standard_normal((B, Hkv, S, 16, 128)).astype(np.float32))
    pkb = bf(pk)
    bos = np.asarray([[[3, 0, 5, 1], [2, 4, 1, 0]], [[0, 1, 2, 3], [5, 4, 3, 2]]], np.int32)
    target = rs.integers(0, 16 * S, size=(B, L + 1, Hq))             # token index 16*slot + t
    qrows = np.zeros((B, L + 1, Hq, 128), np.float32)
    for b, l, n in itertools.product(range(B), range(L + 1), range(Hq)):
        qrows[b, l, n, target[b, l, n]] = 40.0
    q, qd = bf(qrows[:, 0]), bf(qrows[:, 1:])
    out = oracle.sparse_decode_attn_joint(cfg, q, qd, pkb, pvb, bos, None, 1.0)
    assert out.shape == (B, L + 1, Hq, 128)
    vf = f32(pvb).reshape(B, Hkv, 16 * S, 128)
    for b, l, n in itertools.product(range(B), range(L + 1), range(Hq)):
        assert np.allclose(out[b, l, n], vf[b, n // G, target[b, l, n]], atol=1e-12)
    # row 0 is the plain attention of q
    assert np.array_equal(out[:, 0], oracle.sparse_decode_attn(cfg, q, pkb, pvb, bos, None, 1.0))
    # one context length for all rows: request 0 sees blocks 0 and 1 only
    # (positions < 32), i.e. slots holding blocks 0, 1 of each KV head
    ctx = np.asarray([32, 96], np.int32)
    out = oracle.sparse_decode_attn_joint(cfg, q, qd, pkb, pvb, bos, ctx, 1.0)
    for h in range(Hkv):
        vis = [16 * s_ + t for s_ in range(S) if bos[0, h, s_] < 2 for t in range(16)]
        for l, g in itertools.product(range(L + 1), range(G)):
            n = h * G + g
            want = vf[0, h, target[0, l, n]] if target[0, l, n] in vis else vf[0, h, vis].mean(0)
            assert np.allclose(out[0, l, n], want, atol=1e-12)


# ----------------------------------------------------------------------------
# planted recovery on the tiny workload (seeded expectation)
# ----------------------------------------------------------------------------
def test_planted_blocks_are_recovered():
    wl = W.TINY
    cfg = wl.config()
    qs = W.query_sequence(wl)
    k, v = W.gen_kv(wl, 0, qs)
    _, qd = W.step_queries(wl, qs, 0)
    summ = oracle.build_summaries(cfg, k)
    topk = oracle.select_topk(cfg, oracle.score_blocks(cfg, qd, summ))
    for h in range(wl.num_kv_heads):
        assert set(W.planted_blocks(wl, 0, 0, h).tolist()) <= set(topk[0, h].tolist())
