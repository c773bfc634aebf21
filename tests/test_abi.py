"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, and rejects bad arguments before launching anything."""
import ctypes as C
import math
import os
import subprocess

import pytest
import torch

from sparse_kv_cache_oasis_gb300 import binding as ob
from sparse_kv_cache_oasis_gb300 import workloads as W

import oracle


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(ob.LIB_PATH):
        from sparse_kv_cache_oasis_gb300 import build
        build.build()
    return ob.lib()


def test_exports_every_header_symbol(lib):
    names = ob.header_symbols()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", ob.LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    assert set(names) <= exported
    # the hot-path entry points named by the method's pipeline
    for n in ("oasis_score_blocks", "oasis_select_topk", "oasis_plan_fetch", "oasis_fetch_blocks",
              "oasis_sparse_decode_attn"):
        assert n in names


def test_library_links_no_oracle_and_no_torch(lib):
    out = subprocess.run(["nm", "-D", ob.LIB_PATH], capture_output=True, text=True).stdout
    assert "orc_" not in out
    deps = subprocess.run(["ldd", ob.LIB_PATH], capture_output=True, text=True).stdout
    assert "torch" not in deps and "oracle" not in deps


def test_status_strings_and_version(lib):
    assert ob.oasis_status_string(ob.OASIS_OK) == "OASIS_OK"
    assert ob.oasis_status_string(ob.OASIS_ERR_TIMEOUT) == "OASIS_ERR_TIMEOUT"
    assert ob.oasis_version() >= 100


@pytest.mark.parametrize("wl", [W.TINY, W.LLAMA8B_LAYER, W.QWEN3_8B_STEP, W.LONG_CTX]
                         + [W.sweep_point(r, b) for r in W.SWEEP_RATIOS for b in (1, 64)])
def test_workloads_validate_and_cap_matches_oracle(lib, wl):
    assert ob.oasis_validate_config(wl) == ob.OASIS_OK
    assert ob.oasis_fetch_cap(wl) == oracle.fetch_cap(wl.config())
    assert ob.oasis_attn_workspace_bytes(wl) > 0


def test_cap_matches_oracle_over_ratios(lib):
    base = W.LLAMA8B_LAYER.config()
    for S in (16, 64, 128, 130, 1024):
        for r in (0.0, 0.001, 0.01, 0.02, 0.05, 0.0625, 0.1, 0.2, 0.5, 0.999, 1.0, -1.0, -0.5):
            cfg = dict(base, kv_budget_tokens=16 * S, top_k=min(128, S), fetch_ratio=r)
            assert ob.oasis_fetch_cap(cfg) == oracle.fetch_cap(cfg), (S, r)


def _bad_configs():
    good = W.TINY.config()
    yield dict(good, batch=0), ob.OASIS_ERR_INVALID_ARG
    yield dict(good, num_q_heads=15), ob.OASIS_ERR_INVALID_ARG
    yield dict(good, kv_budget_tokens=1000), ob.OASIS_ERR_INVALID_ARG
    yield dict(good, top_k=65), ob.OASIS_ERR_INVALID_ARG          # K > S
    yield dict(good, top_k=300, kv_budget_tokens=16 * 512), ob.OASIS_ERR_INVALID_ARG  # K > NB
    yield dict(good, sink_blocks=20, local_blocks=20), ob.OASIS_ERR_INVALID_ARG  # forced > K
    yield dict(good, fetch_ratio=float("nan")), ob.OASIS_ERR_INVALID_ARG
    yield dict(good, head_dim=64), ob.OASIS_ERR_UNSUPPORTED
    yield dict(good, block_size=32, kv_budget_tokens=2048), ob.OASIS_ERR_UNSUPPORTED
    yield dict(good, num_q_heads=64), ob.OASIS_ERR_UNSUPPORTED     # G = 16
    yield dict(good, num_blocks=40000), ob.OASIS_ERR_UNSUPPORTED
    yield dict(good, lookahead=0), ob.OASIS_ERR_INVALID_ARG


@pytest.mark.parametrize("cfg,status", list(_bad_configs()))
def test_bad_configs_rejected(lib, cfg, status):
    assert ob.oasis_validate_config(cfg) == status


def test_entry_points_reject_bad_arguments_before_launch(lib):
    """Null and misaligned pointers and bad configurations come back as
    OASIS_ERR_INVALID_ARG without touching the GPU (none is present here)."""
    c = ob.OasisConfig.make(W.TINY)
    P = C.c_void_p
    null = P(0)
    odd = P(0x1001)
    ok = P(0x10000)
    L = lib
    assert L.oasis_build_summaries(C.byref(c), null, ok, null) == ob.OASIS_ERR_INVALID_ARG
    assert L.oasis_score_blocks(C.byref(c), odd, ok, ok, null) == ob.OASIS_ERR_INVALID_ARG
    assert L.oasis_select_topk(C.byref(c), ok, null, null) == ob.OASIS_ERR_INVALID_ARG
    assert L.oasis_plan_fetch(C.byref(c), ok, 0, ok, ok, ok, ok, ok, ok, ok, P(2), null) == ob.OASIS_ERR_INVALID_ARG
    assert L.oasis_fetch_blocks(C.byref(c), odd, ok, ok, ok, ok, ok, ok, null) == ob.OASIS_ERR_INVALID_ARG
    ws = ob.oasis_attn_workspace_bytes(c)
    # scale must be positive and finite; workspace large enough and 256-byte aligned
    assert L.oasis_sparse_decode_attn(C.byref(c), ok, ok, ok, ok, null, -1.0, ok, ok, ws, null) == ob.OASIS_ERR_INVALID_ARG
    assert L.oasis_sparse_decode_attn(C.byref(c), ok, ok, ok, ok, null, 0.1, ok, P(0x10010), ws, null) == ob.OASIS_ERR_INVALID_ARG
    assert L.oasis_sparse_decode_attn(C.byref(c), ok, ok, ok, ok, null, 0.1, ok, ok, ws - 1, null) == ob.OASIS_ERR_INVALID_ARG
    # joint attention: the draft queries and the output are checked like q
    assert L.oasis_sparse_decode_attn_joint(C.byref(c), ok, odd, ok, ok, ok, null, 0.1, ok, null) == ob.OASIS_ERR_INVALID_ARG
    assert L.oasis_sparse_decode_attn_joint(C.byref(c), ok, ok, ok, ok, ok, null, 0.1, null, null) == ob.OASIS_ERR_INVALID_ARG
    assert L.oasis_sparse_decode_attn_joint(C.byref(c), ok, ok, ok, ok, ok, null, math.inf, ok, null) == ob.OASIS_ERR_INVALID_ARG
    # min/max scoring: at most 32 query rows per KV head, alignment as for the mean keys
    wide = ob.OasisConfig.make(dict(W.TINY.config(), lookahead=9))  # L*G = 36
    assert L.oasis_score_blocks_minmax(C.byref(wide), ok, ok, ok, null) == ob.OASIS_ERR_UNSUPPORTED
    assert L.oasis_score_blocks_minmax(C.byref(c), odd, ok, ok, null) == ob.OASIS_ERR_INVALID_ARG
    assert L.oasis_build_summaries_minmax(C.byref(c), ok, odd, null) == ob.OASIS_ERR_INVALID_ARG
    # the one-launch prediction chain: at most 256 slots / top-K
    big = ob.OasisConfig.make(dict(W.TINY.config(), kv_budget_tokens=16 * 300, top_k=300, num_blocks=600))
    assert L.oasis_predict_chain(C.byref(big), ok, ok, ok, 0, null, ok, ok, ok, ok, ok, ok, ok, ok, ok,
                                 null) == ob.OASIS_ERR_UNSUPPORTED
    assert L.oasis_predict_chain(C.byref(c), odd, ok, ok, 0, null, ok, ok, ok, ok, ok, ok, ok, ok, ok,
                                 null) == ob.OASIS_ERR_INVALID_ARG
    bad = ob.OasisConfig.make(dict(W.TINY.config(), head_dim=64))
    assert L.oasis_score_blocks(C.byref(bad), ok, ok, ok, null) == ob.OASIS_ERR_UNSUPPORTED
    assert L.oasis_select_topk(None, ok, ok, null) == ob.OASIS_ERR_INVALID_ARG
    assert ob.oasis_fetch_cap(dict(W.TINY.config(), batch=0)) == -1
    assert ob.oasis_attn_workspace_bytes(dict(W.TINY.config(), batch=0)) == 0


def test_binding_checks_tensors(lib):
    wl = W.TINY
    with pytest.raises(ValueError):  # CPU tensors are refused for device arguments
        ob.oasis_select_topk(wl, torch.zeros(1, 4, 256), torch.zeros(1, 4, 32, dtype=torch.int32))
    with pytest.raises(TypeError):
        ob.oasis_select_topk(wl, torch.zeros(1, 4, 256, dtype=torch.float64),
                             torch.zeros(1, 4, 32, dtype=torch.int32))


def test_header_layout_and_constants_match_the_binding(tmp_path):
    """A C program built against include/oasis.h prints the struct layout, the
    status codes and the device error bits; the ctypes binding must agree."""
    fields = [n for n, _ in ob.OasisConfig._fields_]
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "oasis.h"', 'int main(void) {',
             '  printf("sizeof %zu\\n", sizeof(oasis_config_t));']
    lines += [f'  printf("off_{n} %zu\\n", offsetof(oasis_config_t, {n}));' for n in fields]
    status = ["OASIS_OK", "OASIS_ERR_INVALID_ARG", "OASIS_ERR_UNSUPPORTED", "OASIS_ERR_CUDA",
              "OASIS_ERR_TIMEOUT"]
    deverr = ["FETCH_RANGE", "PLAN_STATE", "TOPK_IDS", "WAIT_TIMEOUT", "SLOT_RANGE", "CTX_FULL",
              "NO_SLOT"]
    lines += [f'  printf("{s} %d\\n", (int){s});' for s in status]
    lines += [f'  printf("DEVERR_{d} %u\\n", (unsigned)OASIS_DEVERR_{d});' for d in deverr]
    lines += ['  return 0;', '}']
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-std=c11", "-Wall", "-Werror", "-I",
                           os.path.dirname(ob.HEADER), str(src), "-o", str(exe)])
    got = dict(line.split() for line in subprocess.check_output([str(exe)], text=True).splitlines())
    assert int(got["sizeof"]) == C.sizeof(ob.OasisConfig)
    for n in fields:
        assert int(got[f"off_{n}"]) == getattr(ob.OasisConfig, n).offset, n
    for s in status:
        assert int(got[s]) == getattr(ob, s), s
    for d in deverr:
        assert int(got[f"DEVERR_{d}"]) == getattr(ob, f"DEVERR_{d}"), d


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the behaviour without a device")
def test_without_a_device_waits_and_queries_fail_fast(lib):
    """No device: the bounded stream wait and the error-word query return
    OASIS_ERR_CUDA at once instead of waiting or reporting success."""
    import time
    t0 = time.monotonic()
    assert ob.oasis_stream_wait(0, 2000) == ob.OASIS_ERR_CUDA
    assert time.monotonic() - t0 < 1.0
    with pytest.raises(ob.OasisError) as e:
        ob.oasis_device_errors()
    assert e.value.status == ob.OASIS_ERR_CUDA
