"""Joint attention of the decoded token and the draft tokens against the oracle.

oasis_sparse_decode_attn_joint attends with the 1 + L query rows of every
query head (the decoded token, then the L draft tokens) in one pass over the
working set ("OasisKV: Scaling In-Decode KV Cache Beyond HBM with Lookahead
Sparse Prefetching", Fig. 7 right).  Each output row is compared with the
oracle's attention for that row's query, within the attention tolerance of
the other GPU tests.  The shapes cover one, two and three 8-row tiles per
CTA, units of 40 rows taken in two row groups, a unit split over a cluster of
CTAs, ragged context lengths, empty slots and fully masked requests.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from sparse_kv_cache_oasis_gb300 import binding as ob
from sparse_kv_cache_oasis_gb300 import workloads as W

from gpu_helpers import assert_attn_close, bf16_to_bits, dev_bits

pytestmark = pytest.mark.gpu


def _wl(**kw):
    base = dict(name="joint", batch=2, num_q_heads=8, num_kv_heads=2, ctx_tokens=16 * 203,
                kv_budget_tokens=16 * 48, lookahead=3, top_k=40, fetch_ratio=0.1, seed=78)
    base.update(kw)
    return W.Workload(**base)


def _joint_case(wl, seed, ctx_len=None, empty_frac=0.0, scale=None, check_row0=True):
    cfg = wl.config()
    B, H, Hq, S, L = wl.batch, wl.num_kv_heads, wl.num_q_heads, wl.slots, wl.lookahead
    rs = np.random.default_rng(seed)
    pk = W.to_bf16_bits(rs.standard_normal((B, H, S, 16, 128)).astype(np.float32) * 0.7)
    pv = W.to_bf16_bits(rs.standard_normal((B, H, S, 16, 128)).astype(np.float32))
    q = W.to_bf16_bits(rs.standard_normal((B, Hq, 128)).astype(np.float32))
    qd = W.to_bf16_bits(rs.standard_normal((B, L, Hq, 128)).astype(np.float32))
    bos = np.stack([np.stack([rs.permutation(wl.num_blocks)[:S] for _ in range(H)])
                    for _ in range(B)]).astype(np.int32)
    bos[rs.random(bos.shape) < empty_frac] = -1
    scale = scale if scale is not None else 1 / math.sqrt(128)
    cl_np = None if ctx_len is None else np.asarray(ctx_len, np.int32)
    cl = None if cl_np is None else torch.from_numpy(cl_np).cuda()
    gq, gqd, gk, gv = dev_bits(q), dev_bits(qd), dev_bits(pk), dev_bits(pv)
    gbos = torch.from_numpy(bos).cuda()
    out = torch.full((B, L + 1, Hq, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    ref = oracle.sparse_decode_attn_joint(cfg, q, qd, pk, pv, bos, cl_np, scale)
    for rep in range(2):  # nothing left behind changes the next call
        ob.oasis_sparse_decode_attn_joint(cfg, gq, gqd, gk, gv, gbos, cl, scale, out)
        torch.cuda.synchronize()
        assert_attn_close(bf16_to_bits(out), ref, f"{wl.name} rep {rep}")
    if check_row0:  # row 0 against the single-query kernel, same tolerance
        single = torch.empty((B, Hq, 128), dtype=torch.bfloat16, device="cuda")
        ws = torch.zeros(ob.oasis_attn_workspace_bytes(cfg), dtype=torch.uint8, device="cuda")
        ob.oasis_sparse_decode_attn(cfg, gq, gk, gv, gbos, cl, scale, single, ws)
        torch.cuda.synchronize()
        assert_attn_close(bf16_to_bits(out[:, 0]), W.bf16_bits_to_f32(bf16_to_bits(single)),
                          f"{wl.name} row 0 vs single-query kernel")
    assert ob.oasis_device_errors() == 0
    return bf16_to_bits(out), ref


def test_joint_llama_layer_full_size():
    # G = 4, L = 4: 20 rows in three tiles; 64 units over a cluster of CTAs each
    _joint_case(W.LLAMA8B_LAYER, seed=41)


def test_joint_group8_two_row_groups():
    # G = 8, L = 4: 40 rows per unit in two row groups (24 + 16)
    _joint_case(W.LONG_CTX.with_(layers=1, batch=2), seed=42)


@pytest.mark.parametrize("hq,hkv,L,tiles", [(2, 2, 1, 1), (8, 2, 1, 1), (8, 2, 2, 2), (6, 2, 3, 2),
                                           (8, 2, 5, 3), (16, 2, 8, 3)])
def test_joint_row_tiles(hq, hkv, L, tiles):
    wl = _wl(num_q_heads=hq, num_kv_heads=hkv, lookahead=L)
    G = hq // hkv
    assert min(3, -(-G * (L + 1) // 8)) == tiles
    _joint_case(wl, seed=43 + hq + L)


def test_joint_ragged_context_and_empty_slots():
    _joint_case(_wl(batch=3, kv_budget_tokens=16 * 37, top_k=20), seed=50, empty_frac=0.3,
                ctx_len=[16 * 203, 1000, 37], scale=0.5)


def test_joint_short_and_long_units():
    _joint_case(_wl(batch=40, num_q_heads=32, num_kv_heads=8, kv_budget_tokens=16 * 3, top_k=3,
                    lookahead=2), seed=51, empty_frac=0.2)
    _joint_case(_wl(batch=1, num_q_heads=16, num_kv_heads=2, ctx_tokens=16 * 2048,
                    kv_budget_tokens=16 * 1024, top_k=64, lookahead=2), seed=52, empty_frac=0.1)


def test_joint_empty_and_fully_masked_give_zeros():
    out, ref = _joint_case(_wl(), seed=53, empty_frac=1.0)
    assert not W.bf16_bits_to_f32(out).any() and not ref.any()
    out, _ = _joint_case(_wl(), seed=54, ctx_len=[0, 0])
    assert not W.bf16_bits_to_f32(out).any()
