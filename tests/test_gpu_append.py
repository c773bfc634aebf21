"""A growing context on the GPU against the oracle, step by step, bit for bit.

Each step appends one token per request ("OasisKV: Scaling In-Decode KV Cache
Beyond HBM with Lookahead Sparse Prefetching", Fig. 8: the decode loop
advances a token per step) and refreshes the newest blocks' summaries, then
selects with the local window at the context's end and plans and transfers
as in the fixed-context path.  Scores
are seeded inputs shared by both sides, so every output is integer or a
bf16 / fp32 value computed by the same rounding: the host cache, the pools,
both maps, the LRU times, the mean and min/max summaries, the context
lengths, the top-K lists and the transfer lists must all match exactly.
Covered: appends inside a block and across block boundaries, a newest block
taking an empty slot or evicting the least recently used unforced block,
requests reaching capacity (flagged, skipped).  (A head with no slot to give
cannot arise under a valid configuration: the forced blocks number at most
K <= S, one of them the newest block itself.)
"""
import numpy as np
import pytest
import torch

import oracle
from sparse_kv_cache_oasis_gb300 import binding as ob
from sparse_kv_cache_oasis_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _dev(a, dtype=None):
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).cuda()
    return torch.from_numpy(a.copy()).cuda()


class Loop:
    def __init__(self, cfg, ctx0, seed):
        self.cfg = cfg
        B, H, NB, S = cfg["batch"], cfg["num_kv_heads"], cfg["num_blocks"], cfg["kv_budget_tokens"] // 16
        self.B, self.H, self.NB, self.S = B, H, NB, S
        rs = np.random.default_rng(seed)
        self.rs = rs
        hk = W.to_bf16_bits(rs.standard_normal((B, H, NB, 16, 128)).astype(np.float32))
        hv = W.to_bf16_bits(rs.standard_normal((B, H, NB, 16, 128)).astype(np.float32))
        self.ctx = np.asarray(ctx0, np.int32)
        bos = np.full((B, H, S), -1, np.int32)
        for b in range(B):
            n = min(NB, -(-int(self.ctx[b]) // 16))
            for h in range(H):
                k = min(S - (h % 2), n)          # every other head keeps an empty slot
                bos[b, h, :k] = rs.permutation(n)[:k]
        sob = np.full((B, H, NB), -1, np.int32)
        for b in range(B):
            for h in range(H):
                for q in range(S):
                    if bos[b, h, q] >= 0:
                        sob[b, h, bos[b, h, q]] = q
        lu = np.where(bos >= 0, rs.integers(0, 4, bos.shape), -1).astype(np.int32)
        pk = np.zeros((B, H, S, 16, 128), np.uint16)
        pv = np.zeros_like(pk)
        for b in range(B):
            for h in range(H):
                for q in range(S):
                    if bos[b, h, q] >= 0:
                        pk[b, h, q], pv[b, h, q] = hk[b, h, bos[b, h, q]], hv[b, h, bos[b, h, q]]
        summ = oracle.build_summaries(cfg, hk)
        mm = oracle.build_summaries_minmax(cfg, hk)
        # oracle state
        self.o = dict(hk=hk.copy(), hv=hv.copy(), sob=sob.copy(), bos=bos.copy(), lu=lu.copy(),
                      pk=pk.copy(), pv=pv.copy(), summ=summ.copy(), mm=mm.copy(), ctx=self.ctx.copy())
        # GPU state: the cache in pinned, mapped host memory
        self.hk_t = torch.from_numpy(hk.view(np.int16).copy()).view(torch.bfloat16)
        self.hv_t = torch.from_numpy(hv.view(np.int16).copy()).view(torch.bfloat16)
        self.hk_dev = ob.oasis_host_register(self.hk_t)
        self.hv_dev = ob.oasis_host_register(self.hv_t)
        self.g = dict(sob=_dev(sob), bos=_dev(bos), lu=_dev(lu), pk=_dev(pk), pv=_dev(pv),
                      summ=_dev(summ), mm=_dev(mm), ctx=_dev(self.ctx))
        w = ob.cap_width(cfg)
        i32 = torch.int32
        self.g.update(topk=torch.zeros((B, H, cfg["top_k"]), dtype=i32, device="cuda"),
                      fb=torch.zeros((B, H, w), dtype=i32, device="cuda"),
                      fs=torch.zeros((B, H, w), dtype=i32, device="cuda"),
                      eb=torch.zeros((B, H, w), dtype=i32, device="cuda"),
                      nf=torch.zeros((B, H), dtype=i32, device="cuda"),
                      ne=torch.zeros((B, H), dtype=i32, device="cuda"))

    def step(self, t, plan=True):
        cfg, o, g, rs = self.cfg, self.o, self.g, self.rs
        B, H, NB = self.B, self.H, self.NB
        kn = W.to_bf16_bits(rs.standard_normal((B, H, 128)).astype(np.float32))
        vn = W.to_bf16_bits(rs.standard_normal((B, H, 128)).astype(np.float32))
        ob.oasis_append_kv(cfg, _dev(kn), _dev(vn), g["ctx"], t, None, self.hk_dev, self.hv_dev,
                           g["sob"], g["bos"], g["lu"], g["pk"], g["pv"])
        ob.oasis_refresh_summaries(cfg, g["ctx"], self.hk_dev, g["sob"], g["pk"], g["summ"], g["mm"])
        rc = oracle.append_kv(cfg, kn, vn, o["ctx"], t, o["hk"], o["hv"], o["sob"], o["bos"], o["lu"],
                              o["pk"], o["pv"])
        oracle.refresh_summaries(cfg, o["ctx"], o["hk"], o["summ"], o["mm"])
        torch.cuda.synchronize()
        flags = ob.oasis_device_errors(clear=True)
        if plan:
            sc = rs.standard_normal((B, H, NB)).astype(np.float32)
            ob.oasis_predict_select_ctx(cfg, _dev(sc), g["ctx"], t, None, g["topk"], g["sob"], g["bos"],
                                        g["lu"], g["fb"], g["fs"], g["eb"], g["nf"], g["ne"])
            ob.oasis_fetch_blocks(cfg, self.hk_dev, self.hv_dev, g["fb"], g["fs"], g["nf"], g["pk"], g["pv"])
            ids = oracle.select_topk_ctx(cfg, sc, o["ctx"])
            pl = oracle.plan_fetch(cfg, ids, t, o["sob"], o["bos"], o["lu"])
            oracle.fetch_blocks(cfg, o["hk"], o["hv"], pl["fetch_block"], pl["fetch_slot"],
                                pl["n_fetch"], o["pk"], o["pv"])
            torch.cuda.synchronize()
            assert np.array_equal(g["topk"].cpu().numpy(), ids)
            assert np.array_equal(g["fb"].cpu().numpy(), pl["fetch_block"])
            assert np.array_equal(g["fs"].cpu().numpy(), pl["fetch_slot"])
            assert np.array_equal(g["nf"].cpu().numpy(), pl["n_fetch"])
            flags |= ob.oasis_device_errors(clear=True)
        self.compare()
        return rc, flags

    def compare(self):
        o, g = self.o, self.g
        assert np.array_equal(g["ctx"].cpu().numpy(), o["ctx"])
        assert np.array_equal(_bits(self.hk_t), o["hk"]) and np.array_equal(_bits(self.hv_t), o["hv"])
        for k in ("sob", "bos", "lu"):
            assert np.array_equal(g[k].cpu().numpy(), o[k]), k
        assert np.array_equal(_bits(g["pk"]), o["pk"]) and np.array_equal(_bits(g["pv"]), o["pv"])
        assert np.array_equal(g["summ"].cpu().numpy().view(np.uint32), o["summ"].view(np.uint32))
        assert np.array_equal(_bits(g["mm"]), o["mm"])

    def close(self):
        torch.cuda.synchronize()
        ob.oasis_host_unregister(self.hk_t)
        ob.oasis_host_unregister(self.hv_t)


def _cfg(**kw):
    base = dict(batch=3, num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16, num_blocks=12,
                kv_budget_tokens=16 * 5, lookahead=2, top_k=5, fetch_ratio=0.4, sink_blocks=1,
                local_blocks=2)
    base.update(kw)
    return base


def test_growing_context_loop_bit_exact():
    # mid-block, at a block boundary, and two tokens short of capacity
    loop = Loop(_cfg(), [16 * 6 - 3, 16 * 4, 16 * 12 - 2], seed=61)
    try:
        for t in range(24):
            rc, flags = loop.step(t)
            if t < 2:
                assert rc == 0 and flags == 0
            else:  # request 2 is full from its third append on: flagged and skipped
                assert rc == -1 and flags == ob.DEVERR_CTX_FULL
        assert loop.o["ctx"].tolist() == [16 * 6 - 3 + 24, 16 * 4 + 24, 16 * 12]
    finally:
        loop.close()


def test_append_many_heads_sparse_planning():
    # 8 KV heads (8 warps per request); planning only every third step, so
    # several appends in a row allocate and evict without the planner
    cfg = _cfg(batch=2, num_q_heads=8, num_kv_heads=8, kv_budget_tokens=16 * 4, top_k=4,
               fetch_ratio=0.5)
    loop = Loop(cfg, [16 * 3 - 1, 16 * 5 + 7], seed=62)
    try:
        for t in range(40):
            rc, flags = loop.step(t, plan=(t % 3 == 0))
            assert rc == 0 and flags == 0
    finally:
        loop.close()


def test_append_sixteen_heads_share_one_cta():
    # more than 8 KV heads: one CTA per request with a warp per head
    cfg = _cfg(batch=2, num_q_heads=16, num_kv_heads=16, kv_budget_tokens=16 * 4, top_k=4,
               fetch_ratio=0.5)
    loop = Loop(cfg, [16 * 4 - 2, 16 * 7], seed=64)
    try:
        for t in range(20):
            rc, flags = loop.step(t, plan=(t % 2 == 0))
            assert rc == 0 and flags == 0
    finally:
        loop.close()


def test_append_full_context_flag_and_hand_state():
    # the hand-made state of the oracle's append pins, with pools made
    # consistent with the cache (as the planner keeps them)
    import test_oracle_pins as pins
    cfg, hk, hv, kn, vn, sob, bos, lu, pk, pv, summ, mm = pins._append_setup()
    for b in range(2):
        for h in range(2):
            for q in range(3):
                if bos[b, h, q] >= 0:
                    pk[b, h, q], pv[b, h, q] = hk[b, h, bos[b, h, q]], hv[b, h, bos[b, h, q]]
    hk_t = torch.from_numpy(hk.view(np.int16).copy()).view(torch.bfloat16)
    hv_t = torch.from_numpy(hv.view(np.int16).copy()).view(torch.bfloat16)
    hk_d, hv_d = ob.oasis_host_register(hk_t), ob.oasis_host_register(hv_t)
    try:
        g = [_dev(x) for x in (sob, bos, lu, pk, pv, summ, mm)]
        for ctx, want_rc, want_flag in (([32, 40], 0, 0), ([16 * 6, 16 * 4], -1, ob.DEVERR_CTX_FULL),
                                        ([5, 70], 0, 0)):
            cl = np.asarray(ctx, np.int32)
            gcl = _dev(cl)
            ob.oasis_append_kv(cfg, _dev(kn), _dev(vn), gcl, 3, None, hk_d, hv_d, *g[:5])
            ob.oasis_refresh_summaries(cfg, gcl, hk_d, g[0], g[3], g[5], g[6])
            rc = oracle.append_kv(cfg, kn, vn, cl, 3, hk, hv, sob, bos, lu, pk, pv)
            oracle.refresh_summaries(cfg, cl, hk, summ, mm)
            torch.cuda.synchronize()
            assert rc == want_rc and ob.oasis_device_errors(clear=True) == want_flag
            assert np.array_equal(gcl.cpu().numpy(), cl)
            assert np.array_equal(_bits(hk_t), hk) and np.array_equal(_bits(hv_t), hv)
            for got, want in zip(g, (sob, bos, lu, pk, pv, summ, mm)):
                if got.dtype == torch.bfloat16:
                    assert np.array_equal(_bits(got), want)
                elif got.dtype == torch.float32:
                    assert np.array_equal(got.cpu().numpy().view(np.uint32), want.view(np.uint32))
                else:
                    assert np.array_equal(got.cpu().numpy(), want)
    finally:
        torch.cuda.synchronize()
        ob.oasis_host_unregister(hk_t)
        ob.oasis_host_unregister(hv_t)


def test_topk_ctx_matches_oracle_and_full_context():
    cfg = _cfg(batch=4, num_blocks=300, kv_budget_tokens=16 * 40, top_k=40, sink_blocks=2,
               local_blocks=5)
    rs = np.random.default_rng(63)
    sc = rs.standard_normal((4, 2, 300)).astype(np.float32)
    sc[0, 0, 10:20] = sc[0, 0, 10]                  # ties: lower ids first
    for ctx in ([0, 17, 16 * 37, 16 * 300], [16 * 300] * 4, [5, 16 * 41 + 1, 4000, 16 * 299]):
        cl = np.asarray(ctx, np.int32)
        out = torch.empty((4, 2, 40), dtype=torch.int32, device="cuda")
        ob.oasis_select_topk_ctx(cfg, _dev(sc), _dev(cl), out)
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy(), oracle.select_topk_ctx(cfg, sc, cl))
    plain = torch.empty((4, 2, 40), dtype=torch.int32, device="cuda")
    ob.oasis_select_topk(cfg, _dev(sc), plain)
    torch.cuda.synchronize()
    full = np.asarray([16 * 300] * 4, np.int32)
    assert np.array_equal(plain.cpu().numpy(), oracle.select_topk_ctx(cfg, sc, full))
    assert ob.oasis_device_errors() == 0
