"""The seeded synthetic inputs follow their stated recipe.

The workloads stand in for those of "OasisKV: Scaling In-Decode KV Cache
Beyond HBM with Lookahead Sparse Prefetching" (Tab. 1 and Tab. 2 shapes):
random-walk decode queries whose draft tokens are the next L queries of the
same walk, keys N(0, key_std^2) with planted or Zipf(1.1) heavy-hitter blocks
shifted along the drafts' mean direction, values N(0,1)/sqrt(D), a seeded
initial working set with the forced blocks in it, and bf16 round-to-nearest-
even.  Each property is checked against an independent computation (torch's
bf16 conversion, the same draw without structure, sample statistics).
"""
import math

import numpy as np
import pytest
import torch

from sparse_kv_cache_oasis_gb300 import workloads as W


def _small(**kw):
    base = dict(name="recipe", batch=2, num_q_heads=8, num_kv_heads=2, ctx_tokens=16 * 64,
                kv_budget_tokens=16 * 16, lookahead=3, top_k=8, fetch_ratio=0.25, seed=321,
                steps=6)
    base.update(kw)
    return W.Workload(**base)


def test_bf16_rounding_matches_torch():
    rs = np.random.default_rng(5)
    x = np.concatenate([
        rs.standard_normal(20000).astype(np.float32) * 10.0 ** rs.integers(-20, 20, 20000),
        # exact ties: halfway between two bf16 values, both parities of the kept bit
        (np.arange(1, 2000, dtype=np.uint32) << 16 | np.uint32(0x8000)).view(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, 3.4e38, -3.4e38, 1e-45], dtype=np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(W.to_bf16_bits(x), want)
    back = W.bf16_bits_to_f32(want)
    assert np.array_equal(W.to_bf16_bits(back), want)        # bf16 values are fixed points


def test_streams_are_keyed_not_sequential():
    wl = _small(structure="planted")
    k2, v2 = W.gen_kv(wl, 0)
    k2b, v2b = W.gen_kv(wl, 0)
    assert np.array_equal(k2, k2b) and np.array_equal(v2, v2b)
    k1, v1 = W.gen_kv(wl.with_(batch=1), 0)                  # request 0 alone: the same bytes
    assert np.array_equal(k1[0], k2[0]) and np.array_equal(v1[0], v2[0])
    kl, _ = W.gen_kv(wl, 1)                                  # another layer: other bytes
    assert not np.array_equal(kl, k2)
    assert not np.array_equal(k2[0, 0], k2[0, 1]) and not np.array_equal(k2[0], k2[1])


def test_random_walk_queries_and_drafts():
    wl = _small(batch=4, num_q_heads=16, steps=40, lookahead=4)
    q = W.query_sequence(wl).astype(np.float64)              # [T, B, Hq, D]
    assert q.shape == (wl.steps + wl.lookahead + 1, 4, 16, 128)
    D = 128
    assert abs(q[0].std() * math.sqrt(D) - 1.0) < 0.03
    inc = np.diff(q, axis=0)
    assert abs(inc.std() * math.sqrt(D) / W.WALK_SIGMA - 1.0) < 0.02
    assert abs(inc.mean()) < 1e-3
    for t in (0, 7, wl.steps - 1):
        qb, qd = W.step_queries(wl, q.astype(np.float32), t)
        assert np.array_equal(qb, W.to_bf16_bits(q[t].astype(np.float32)))
        assert qd.shape == (4, wl.lookahead, 16, 128)
        for l in range(wl.lookahead):
            assert np.array_equal(qd[:, l], W.to_bf16_bits(q[t + 1 + l].astype(np.float32)))
    planted = W.query_sequence(wl.with_(structure="planted")).astype(np.float64)
    assert abs(np.corrcoef(planted[1].ravel(), planted[0].ravel())[0, 1]) < 0.05   # independent draws


def test_values_and_unstructured_keys_statistics():
    wl = _small(batch=1, num_kv_heads=1, num_q_heads=4, ctx_tokens=16 * 512, key_std=0.3)
    k, v = W.gen_kv(wl)
    kf = W.bf16_bits_to_f32(k).astype(np.float64)
    vf = W.bf16_bits_to_f32(v).astype(np.float64)
    assert abs(vf.std() * math.sqrt(128) - 1.0) < 0.01 and abs(vf.mean()) < 2e-3
    assert abs(kf.std() / 0.3 - 1.0) < 0.01 and abs(kf.mean()) < 2e-3


def test_planted_blocks_shift_along_the_draft_direction():
    wl = W.TINY
    qseq = W.query_sequence(wl)
    u = W.query_direction(wl, qseq).astype(np.float64)       # [B, Hkv, D]
    assert np.allclose(np.linalg.norm(u, axis=-1), 1.0, atol=1e-6)
    # u is the normalised mean of the G*L step-0 draft queries of the KV head
    G, L = wl.group, wl.lookahead
    for h in range(wl.num_kv_heads):
        m = qseq[1:1 + L, 0, h * G:(h + 1) * G].astype(np.float64).reshape(-1, 128).mean(axis=0)
        assert np.allclose(u[0, h], m / np.linalg.norm(m), atol=1e-6)
    k, _ = W.gen_kv(wl, 0, qseq)
    kf = W.bf16_bits_to_f32(k).astype(np.float64)
    for h in range(wl.num_kv_heads):
        proj = kf[0, h].mean(axis=1) @ u[0, h]              # block mean along u
        pb = W.planted_blocks(wl, 0, 0, h)
        assert len(set(pb.tolist())) == W.PLANTED_BLOCKS
        rest = np.setdiff1d(np.arange(wl.num_blocks), pb)
        assert np.all(np.abs(proj[pb] - W.PLANT_SHIFT) < 0.1)
        assert np.all(np.abs(proj[rest]) < 0.1)


def test_zipf_heavy_hitters_follow_the_rank_profile():
    wl = _small(batch=1, num_kv_heads=2, num_q_heads=8, ctx_tokens=16 * 128, structure="zipf",
                key_std=1.0)
    qseq = W.query_sequence(wl)
    u = W.query_direction(wl, qseq).astype(np.float64)
    kz, vz = W.gen_kv(wl, 0, qseq)
    kw, vw = W.gen_kv(wl.with_(structure="walk"), 0, qseq)  # same draws, no structure
    assert np.array_equal(vz, vw)
    diff = W.bf16_bits_to_f32(kz).astype(np.float64) - W.bf16_bits_to_f32(kw).astype(np.float64)
    ranks = np.arange(1, wl.num_blocks + 1)
    want = W.PLANT_SHIFT * ranks ** (-W.ZIPF_S)
    for h in range(2):
        perm = W.zipf_ranking(wl, 0, 0, h)
        assert np.array_equal(np.sort(perm), np.arange(wl.num_blocks))
        shift = diff[0, h].mean(axis=1) @ u[0, h]           # per block, along u
        # block perm[r-1] carries 0.5 * r**-1.1, up to bf16 rounding of keys ~N(0,1)
        assert np.allclose(shift[perm], want, atol=4e-3)
        # and nothing off the direction u (beyond rounding)
        resid = diff[0, h].mean(axis=1) - np.outer(shift, u[0, h])
        assert np.abs(resid).max() < 4e-3


@pytest.mark.parametrize("wl", [
    _small(),
    _small(sink_blocks=1, local_blocks=4),
    _small(ctx_tokens=16 * 10, kv_budget_tokens=16 * 16),     # fewer blocks than slots
    W.LONG_CTX.with_(batch=1, num_kv_heads=2, num_q_heads=16, ctx_tokens=16 * 300),
])
def test_initial_working_set(wl):
    sob, bos, lu = W.initial_resident(wl)
    B, H, NB, S = wl.batch, wl.num_kv_heads, wl.num_blocks, wl.slots
    assert sob.shape == (B, H, NB) and bos.shape == (B, H, S) and lu.shape == (B, H, S)
    assert (lu == -1).all()
    forced = [j for j in range(NB) if j < wl.sink_blocks or j >= NB - wl.local_blocks]
    for b in range(B):
        for h in range(H):
            res = bos[b, h][bos[b, h] >= 0]
            assert len(res) == min(S, NB) and len(set(res.tolist())) == len(res)
            assert set(forced) <= set(res.tolist())
            for s in range(S):                              # mutual inverses
                if bos[b, h, s] >= 0:
                    assert sob[b, h, bos[b, h, s]] == s
            assert (sob[b, h] >= 0).sum() == len(res)
    sob2, bos2, _ = W.initial_resident(wl)
    assert np.array_equal(sob, sob2) and np.array_equal(bos, bos2)


def test_initial_pool_holds_the_resident_blocks():
    wl = _small(ctx_tokens=16 * 12)                          # 12 blocks, 16 slots: 4 empty
    k, v = W.gen_kv(wl)
    sob, bos, _ = W.initial_resident(wl)
    pk, pv = W.initial_pool(wl, k, v, bos)
    for b in range(wl.batch):
        for h in range(wl.num_kv_heads):
            for s in range(wl.slots):
                j = bos[b, h, s]
                if j >= 0:
                    assert np.array_equal(pk[b, h, s], k[b, h, j])
                    assert np.array_equal(pv[b, h, s], v[b, h, j])
                else:
                    assert not pk[b, h, s].any() and not pv[b, h, s].any()
