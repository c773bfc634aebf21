"""The prediction chain in one launch against the separate calls.

oasis_predict_chain runs the look-ahead scoring, the top-K and the capped
planning of "OasisKV: Scaling In-Decode KV Cache Beyond HBM with Lookahead
Sparse Prefetching" (Fig. 7 right; explanatory diagram steps 2-3) in one
launch.  Its arithmetic is that of oasis_score_blocks followed by
oasis_predict_select, which the other GPU tests pin to the oracle, so every
output (scores, top-K lists, maps, LRU times, transfer lists, clock) must be
equal bit for bit, step after step.  Shapes: the Llama layer (a unit split
over a cluster of two CTAs), more units than SMs (one CTA per unit), two
16-row query tiles, ragged block counts, forced blocks, partly empty
working sets, a fetch-all cap.
"""
import numpy as np
import pytest
import torch

from sparse_kv_cache_oasis_gb300 import binding as ob
from sparse_kv_cache_oasis_gb300 import workloads as W

from test_gpu_kernels import _random_state

pytestmark = pytest.mark.gpu


def _case(B, Hq, H, NB, S, K, L, ratio, sink, local, full, seed, steps=4):
    rs = np.random.default_rng(seed)
    cfg = dict(batch=B, num_q_heads=Hq, num_kv_heads=H, head_dim=128, block_size=16, num_blocks=NB,
               kv_budget_tokens=16 * S, lookahead=L, top_k=K, fetch_ratio=ratio, sink_blocks=sink,
               local_blocks=local)
    sob, bos, lu = _random_state(rs, B, H, NB, S, full=full)
    w = ob.cap_width(cfg)
    summ = torch.from_numpy((rs.standard_normal((B, H, NB, 128)) * 0.1).astype(np.float32)).cuda()

    def bufs():
        st = [torch.from_numpy(x.copy()).cuda() for x in (sob, bos, lu)]
        out = [torch.full((B, H, w), -9, dtype=torch.int32, device="cuda") for _ in range(3)] + \
              [torch.full((B, H), -9, dtype=torch.int32, device="cuda") for _ in range(2)]
        return (st, out, torch.full((B, H, K), -9, dtype=torch.int32, device="cuda"),
                torch.full((B, H, NB), float("nan"), dtype=torch.float32, device="cuda"),
                torch.full((B, H), 5, dtype=torch.int32, device="cuda"))

    a_st, a_out, a_topk, a_sc, a_clock = bufs()
    b_st, b_out, b_topk, b_sc, b_clock = bufs()
    for t in range(steps):
        qd = torch.from_numpy(W.to_bf16_bits(rs.standard_normal((B, L, Hq, 128)).astype(np.float32))
                              .view(np.int16)).view(torch.bfloat16).cuda()
        clocked = t % 2 == 0
        ob.oasis_score_blocks(cfg, qd, summ, a_sc)
        ob.oasis_predict_select(cfg, a_sc, 40 + t, a_clock if clocked else None, a_topk, *a_st, *a_out)
        ob.oasis_predict_chain(cfg, qd, summ, b_sc, 40 + t, b_clock if clocked else None, b_topk,
                               *b_st, *b_out)
        torch.cuda.synchronize()
        assert torch.equal(a_sc.view(torch.int32), b_sc.view(torch.int32))
        assert torch.equal(a_topk, b_topk)
        for x, y in zip(a_st + a_out + [a_clock], b_st + b_out + [b_clock]):
            assert torch.equal(x, y)
    assert ob.oasis_device_errors() == 0


def test_chain_llama_layer():
    _case(8, 32, 8, 2048, 128, 128, 4, 0.05, 0, 0, True, seed=71)


def test_chain_more_units_than_sms_and_two_row_tiles():
    _case(32, 64, 8, 520, 64, 48, 4, 0.1, 1, 2, False, seed=72, steps=3)   # 256 units, L*G = 32


@pytest.mark.parametrize("NB,S,K,ratio,sink,local,full", [
    (300, 40, 30, 0.5, 2, 2, False), (8192, 128, 128, 0.02, 1, 4, True),
    (64, 8, 8, -1.0, 0, 0, True), (13, 4, 4, 0.25, 0, 1, False)])
def test_chain_shapes(NB, S, K, ratio, sink, local, full):
    _case(2, 6, 3, NB, S, K, 3, ratio, sink, local, full, seed=NB + K)


def test_chain_rejects_unsupported_shapes():
    cfg = dict(batch=1, num_q_heads=8, num_kv_heads=1, head_dim=128, block_size=16, num_blocks=600,
               kv_budget_tokens=16 * 300, lookahead=2, top_k=300, fetch_ratio=0.1, sink_blocks=0,
               local_blocks=0)                                          # K > 256
    z = lambda *s, dt=torch.int32: torch.zeros(s, dtype=dt, device="cuda")
    with pytest.raises(ob.OasisError):
        ob.oasis_predict_chain(cfg, z(1, 2, 8, 128, dt=torch.bfloat16), z(1, 1, 600, 128, dt=torch.float32),
                               z(1, 1, 600, dt=torch.float32), 0, None, z(1, 1, 300), z(1, 1, 600),
                               z(1, 1, 300), z(1, 1, 300), z(1, 1, 30), z(1, 1, 30), z(1, 1, 30),
                               z(1, 1), z(1, 1))
