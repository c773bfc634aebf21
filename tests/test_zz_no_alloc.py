"""The attention call that allocates nothing (oasis_sparse_decode_attn_static).

Some callers cannot allocate device memory at all -- code running inside
another framework's memory pool or allocator hooks, under a device-memory
quota, or on a latency-critical path where a cudaMalloc (which may
synchronize the device) is not acceptable.  For them the library keeps a fixed
device scratch array and offers a variant of the attention call that uses it
instead of a caller-provided workspace.

This test calls that variant through the C ABI twice in a row, on different
inputs, and checks each output against the ordinary call with its own
workspace, within the attention tolerance the other GPU tests use.  It must
pass both on its own in a fresh process and after every other test.
"""
import math

import numpy as np
import pytest
import torch

from gpu_helpers import ATOL, RTOL, dev_bits
from sparse_kv_cache_oasis_gb300 import binding as ob
from sparse_kv_cache_oasis_gb300 import workloads as W
from sparse_kv_cache_oasis_gb300.layer import bf16_to_bits

pytestmark = pytest.mark.gpu


def _inputs(wl, seed, empty_frac=0.0):
    B, H, Hq, S = wl.batch, wl.num_kv_heads, wl.num_q_heads, wl.slots
    rs = np.random.default_rng(seed)
    pk = W.to_bf16_bits(rs.standard_normal((B, H, S, 16, 128)).astype(np.float32) * 0.7)
    pv = W.to_bf16_bits(rs.standard_normal((B, H, S, 16, 128)).astype(np.float32))
    q = W.to_bf16_bits(rs.standard_normal((B, Hq, 128)).astype(np.float32))
    bos = np.stack([np.stack([rs.permutation(wl.num_blocks)[:S] for _ in range(H)])
                    for _ in range(B)]).astype(np.int32)
    bos[rs.random(bos.shape) < empty_frac] = -1
    return dev_bits(q), dev_bits(pk), dev_bits(pv), torch.from_numpy(bos).cuda()


def _with_workspace(wl, q, pk, pv, bos, ctx, scale):
    out = torch.empty((wl.batch, wl.num_q_heads, 128), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(ob.oasis_attn_workspace_bytes(wl), dtype=torch.uint8, device="cuda")
    ob.oasis_sparse_decode_attn(wl, q, pk, pv, bos, ctx, scale, out, ws)
    torch.cuda.synchronize()
    return W.bf16_bits_to_f32(bf16_to_bits(out)).astype(np.float64)


@pytest.mark.parametrize("wl", [
    W.LLAMA8B_LAYER,
    W.Workload(name="ragged", batch=3, num_q_heads=12, num_kv_heads=2, ctx_tokens=16 * 203,
               kv_budget_tokens=16 * 77, lookahead=2, top_k=40, fetch_ratio=0.1, seed=5),
])
def test_no_alloc_attention_matches_workspace_call_twice(wl):
    scale = 1.0 / math.sqrt(128)
    ctx = None
    if wl.batch == 3:
        ctx = torch.tensor([16 * 203, 999, 40], dtype=torch.int32, device="cuda")
    for call, seed in enumerate((11, 12)):
        q, pk, pv, bos = _inputs(wl, seed, empty_frac=0.2 * call)
        ref = _with_workspace(wl, q, pk, pv, bos, ctx, scale)
        out = torch.full((wl.batch, wl.num_q_heads, 128), float("nan"), dtype=torch.bfloat16,
                         device="cuda")
        ob.oasis_sparse_decode_attn_static(wl, q, pk, pv, bos, ctx, scale, out)
        torch.cuda.synchronize()
        got = W.bf16_bits_to_f32(bf16_to_bits(out)).astype(np.float64)
        err = np.abs(got - ref)
        assert np.isfinite(got).all(), f"call {call}: non-finite output"
        assert (err <= ATOL + RTOL * np.abs(ref)).all(), f"call {call}: max err {err.max():.3g}"
    assert ob.oasis_device_errors() == 0


def test_no_alloc_scratch_covers_the_largest_valid_shape():
    """The scratch holds two partials per warp of one CTA per SM plus one
    counter per unit, so the largest shape the library accepts fits in the
    fixed 8 MiB; the call's size guard (OASIS_ERR_UNSUPPORTED) never fires
    for a valid configuration on this part."""
    big = W.Workload(name="largest", batch=8191, num_q_heads=64, num_kv_heads=8,
                     ctx_tokens=16 * 32768, kv_budget_tokens=16 * 1024, lookahead=1, top_k=1024,
                     fetch_ratio=0.05, seed=1)
    assert ob.oasis_validate_config(big) == ob.OASIS_OK
    assert big.batch * big.num_kv_heads <= 65535
    assert ob.oasis_attn_workspace_bytes(big) <= 8 << 20
