#!/usr/bin/env python
"""Benchmark of the look-ahead sparse-KV decode hot path on one GB300.

Workload: the Llama-3.1-8B-shaped decode layer of "OasisKV: Scaling In-Decode
KV Cache Beyond HBM with Lookahead Sparse Prefetching" workloads -- 32 query
/ 8 KV heads, head_dim 128, batch 8, 32,768-token context (2,048 blocks of
16 per KV head), 2,048-token KV budget (128 blocks), L = 4 draft tokens,
top-K = 128, fetch ratio 0.05 (cap 7 blocks per head and step), the full
KV cache (1 GiB) in pinned host memory, random-walk queries (sigma 0.1).

One step = one pass of the whole hot path for one layer: sparse attention,
draft scoring, top-K, capped LRU planning and the host->HBM transfer.  Four
independent copies of the layer (distinct seeds) are cycled step after step,
as consecutive layers of a model would be: the working set touched between
two visits of the same copy (4 x 134 MB) is larger than L2, and the transfer
of one layer overlaps the next layer's compute (copy stream), as in Fig. 8.
Each step replays a CUDA graph: attention of copy s beside scoring of copy
s-1, top-K + plan of copy s-2 and the transfer of copy s-3 (a software
pipeline over layers); the LRU step lives in device memory, so replays
advance it.

Prints one JSON line (rank 0).  Beside the headline (`value`, `roofline` of
the fused attention + scoring launch, `step_roofline`, `e2e` with the
queries copied in and the output copied out every step, `cpu_baseline`,
`clocks`), it carries each kernel timed alone (`kernels_ms`) and the rows
beyond the hot path, each on the same layer: `joint_attention` (decoded and
draft tokens in one KV pass), `minmax_scoring` and `minmax_step` (min/max
compressed keys), `predict_chain` (scoring + top-K + plan in one launch) and
`growing_context` (a token appended per step, the local window following the
context).  --impl reference times the CPU oracle on the same workload
instead; --sweep runs the fetch-ratio x batch sweep on the Qwen3-8B layer
shape (one JSON line per point, not the benchmark line).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_kv_cache_oasis_gb300 import workloads as W  # noqa: E402

METRIC = "decode tok/s at 32K ctx, 2K-token KV budget; % of HBM+host-link roofline"
UNIT = "tok/s"
WORKLOAD = W.LLAMA8B_LAYER
INSTANCES = 4
QUERY_SETS = 20          # the workload's 20 consecutive decode steps, cycled
GROW_ROOM = 1024         # tokens of room left in each context for the growing-context run


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["oasis", "reference"], default="oasis")
    ap.add_argument("--instances", type=int, default=INSTANCES)
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the CPU-oracle sample")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-grow", action="store_true", help="skip the growing-context run")
    ap.add_argument("--no-minmax-step", action="store_true", help="skip the min/max-key step run")
    ap.add_argument("--sweep", action="store_true",
                    help="instead of the benchmark: the fetch-ratio x batch sweep (one JSON line per point)")
    ap.add_argument("--sweep-batches", default="1,8,32,64")
    ap.add_argument("--profile-chain", type=int, default=0,
                    help="with --profile-steps: then this many prediction-chain launches")
    ap.add_argument("--profile-grow", action="store_true",
                    help="with --profile-steps: run the growing-context form of the step")
    ap.add_argument("--profile-steps", type=int, default=0,
                    help="only run this many untimed graph steps (for ncu launch lists)")
    ap.add_argument("--profile-joint", type=int, default=0,
                    help="with --profile-steps: then this many joint-attention launches")
    ap.add_argument("--profile-minmax", type=int, default=0,
                    help="with --profile-steps: then this many min/max-key scoring launches")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest `value` over the ranks: the slowest replica sets the job's
    time.  One all-reduce of one number (the replicas share no data)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, batch: int, ms_per_step: float) -> float:
    """Decode tokens per second of the whole job: every rank decodes `batch`
    sequences per layer-step (weak scaling)."""
    return world * batch / (ms_per_step * 1e-3)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "of measured: hbm_gbs (copy) of MEASURED_PEAKS.json"
    except Exception:
        return 6800.0, "of fallback: 6.8 TB/s, MEASURED_PEAKS.json absent"


# ----------------------------------------------------------------------------- bytes
def algorithmic_bytes(wl, n_fetch_blocks: float, valid_slots: float):
    """Bytes the method must move per layer-step (HBM) and over the host link."""
    U = wl.batch * wl.num_kv_heads
    blk = wl.block_size * wl.head_dim * 2 * 2          # K + V of one block: 8 KiB
    attn = valid_slots * blk + wl.batch * wl.num_q_heads * wl.head_dim * 2 * 2 + U * wl.slots * 4
    score = U * wl.num_blocks * wl.head_dim * 4 + wl.batch * wl.lookahead * wl.num_q_heads * wl.head_dim * 2 \
        + U * wl.num_blocks * 4
    topk = U * wl.num_blocks * 4 + U * wl.top_k * 4
    plan = U * (wl.top_k * 4 + wl.slots * 4 * 4)        # ids, maps, LRU (read + write)
    fetch_hbm = n_fetch_blocks * blk
    link = n_fetch_blocks * blk
    # joint attention: the same KV pass with the draft rows as queries and outputs too
    rows_io = wl.batch * wl.num_q_heads * wl.head_dim * 2 * (1 + wl.lookahead)
    joint = valid_slots * blk + 2 * rows_io + U * wl.slots * 4
    return dict(attn=attn, score=score, fused=attn + score, topk=topk, plan=plan, fetch=fetch_hbm,
                hbm=attn + score + topk + plan + fetch_hbm, link=link, joint=joint,
                score_mm=score,  # bf16 max + min rows: as many bytes as the fp32 mean
                chain=score + topk + plan, score_select=score + topk + plan)


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- reference arm
def oracle_layer_step_runner(wl, layer=0, units_per_call=None):
    """Oracle runner.  Each call runs one layer-step for `units_per_call`
    (request, KV head) units (all of them by default), cycling over units and
    steps; returns the fraction of a full layer-step that the call covered."""
    import oracle
    cfg = wl.config()
    qseq = W.query_sequence(wl, layer)
    k, v = W.gen_kv(wl, layer, qseq)
    sob, bos, lu = W.initial_resident(wl, layer)
    pk, pv = W.initial_pool(wl, k, v, bos)
    summ = oracle.build_summaries(cfg, k)
    U = wl.batch * wl.num_kv_heads
    G = wl.group
    n = U if units_per_call is None else max(1, min(U, units_per_call))
    if n == U:
        stepper = oracle.Stepper(cfg, k, v, summ, sob, bos, lu, pk, pv)
    else:
        ucfg = oracle.unit_cfg(cfg)
        units = []
        for u in range(U):
            b, h = divmod(u, wl.num_kv_heads)
            sl = lambda a: np.ascontiguousarray(a[b:b + 1, h:h + 1])
            units.append((b, h, oracle.Stepper(ucfg, sl(k), sl(v), sl(summ), sl(sob), sl(bos), sl(lu),
                                               sl(pk), sl(pv))))
    state = {"t": 0, "u": 0}

    def one():
        t = state["t"]
        q, qd = W.step_queries(wl, qseq, t % wl.steps)
        if n == U:
            stepper.step(t, q, qd)
            state["t"] += 1
            return 1.0
        for _ in range(n):
            if state["t"] != t:
                t = state["t"]
                q, qd = W.step_queries(wl, qseq, t % wl.steps)
            b, h, st = units[state["u"]]
            st.step(t, np.ascontiguousarray(q[b:b + 1, h * G:(h + 1) * G]),
                    np.ascontiguousarray(qd[b:b + 1, :, h * G:(h + 1) * G]))
            state["u"] += 1
            if state["u"] == U:
                state["u"] = 0
                state["t"] += 1
        return n / U
    return one


def reference_arm(args):
    """The CPU oracle, as it stands, on the same workload and metric.  Each
    step is a bounded sample of a layer-step: as many (request, KV head) units
    as fit a budget that keeps the whole run within a few minutes."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    wl = WORKLOAD
    probe = oracle_layer_step_runner(wl, units_per_call=1)
    probe()
    t0 = time.perf_counter()
    probe()
    t_unit = time.perf_counter() - t0
    budget = 150.0 / max(1, args.steps + args.warmup)
    units = max(1, min(wl.batch * wl.num_kv_heads, int(budget / max(t_unit, 1e-6))))
    one = oracle_layer_step_runner(wl, units_per_call=units)
    for _ in range(args.warmup):
        one()
    frac = 0.0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        frac += one()
    dt = time.perf_counter() - t0
    val = wl.batch * frac / dt
    line = {"metric": METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": wl.name, "global_batch": wl.batch, "seq_len": wl.ctx_tokens,
                       "kv_budget_tokens": wl.kv_budget_tokens, "layers": 1,
                       "parallelism": "replicas", "l2": "n/a (CPU)"},
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"each step: {units} of the 64 (request, KV head) units of one "
                                       "layer-step, single-threaded C oracle, double accumulation"},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cpu_baseline_all_cores(seconds: float):
    """The same oracle, its independent (request, KV head) units spread over
    all host cores: each unit keeps its own single-threaded oracle state and a
    thread pool runs the units of a layer-step side by side (the C calls
    release the interpreter lock)."""
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    wl = WORKLOAD
    cores = os.cpu_count() or 1
    cfg = wl.config()
    qseq = W.query_sequence(wl, 0)
    k, v = W.gen_kv(wl, 0, qseq)
    sob, bos, lu = W.initial_resident(wl, 0)
    pk, pv = W.initial_pool(wl, k, v, bos)
    summ = oracle.build_summaries(cfg, k)
    ucfg = oracle.unit_cfg(cfg)
    G = wl.group
    units = []
    for u in range(wl.batch * wl.num_kv_heads):
        b, h = divmod(u, wl.num_kv_heads)
        sl = lambda a: np.ascontiguousarray(a[b:b + 1, h:h + 1])
        units.append((b, h, oracle.Stepper(ucfg, sl(k), sl(v), sl(summ), sl(sob), sl(bos), sl(lu),
                                           sl(pk), sl(pv))))
    del k, v

    def one(pool, t):
        q, qd = W.step_queries(wl, qseq, t % wl.steps)
        jobs = [pool.submit(st.step, t, np.ascontiguousarray(q[b:b + 1, h * G:(h + 1) * G]),
                            np.ascontiguousarray(qd[b:b + 1, :, h * G:(h + 1) * G]))
                for b, h, st in units]
        for j in jobs:
            j.result()

    with ThreadPoolExecutor(max_workers=cores) as pool:
        one(pool, 0)
        n, t0 = 0, time.perf_counter()
        while True:
            one(pool, n + 1)
            n += 1
            dt = time.perf_counter() - t0
            if dt >= seconds or n >= 500:
                break
    return {"value": wl.batch * n / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n} full layer-steps of {wl.name}, its 64 units spread over {cores} threads "
                      "(one single-threaded C oracle per unit)"}


def cpu_baseline(seconds: float):
    wl = WORKLOAD
    one = oracle_layer_step_runner(wl)
    one()  # first step pays the one-off costs
    n, t0 = 0, time.perf_counter()
    while True:
        one()
        n += 1
        dt = time.perf_counter() - t0
        if dt >= seconds or n >= 50:
            break
    return {"value": wl.batch * n / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{n} full layer-steps of {wl.name} (all 64 units), single-threaded C oracle"}


# ----------------------------------------------------------------------------- GPU arm
def source_digest(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel's
    sources are unchanged since it was taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)[kernel]
        if d["source_digest"] != source_digest(d["sources"]):
            return None
        return float(d["dram_bytes_per_launch"])
    except Exception:
        return None


_uploaded = set()


def upload_graph(g, stream):
    """Uploads an instantiated CUDA graph to the device ahead of its first
    launch (the CUDA driver API's cuGraphUpload on the graph's executable),
    once per graph; a no-op where the executable is not exposed."""
    import ctypes
    get = getattr(g, "raw_cuda_graph_exec", None)
    if get is None or id(g) in _uploaded:
        return
    try:
        exe = get()
        drv = ctypes.CDLL("libcuda.so.1")
        drv.cuGraphUpload.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
        drv.cuGraphUpload.restype = ctypes.c_int
        rc = drv.cuGraphUpload(ctypes.c_void_p(exe), ctypes.c_void_p(stream.cuda_stream))
        if rc == 0:
            _uploaded.add(id(g))
    except Exception:
        pass


def gpu_arm(args):
    import torch
    import torch.distributed as dist

    from sparse_kv_cache_oasis_gb300 import binding as ob
    from sparse_kv_cache_oasis_gb300.layer import LayerState, bits_to_bf16

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    ob.lib()
    wl = WORKLOAD.with_(steps=QUERY_SETS)
    n_inst = args.instances
    dev = torch.device("cuda", local)

    # ---- layer copies (set-up, untimed)
    layers, qd_dev, q_dev, q_host, qd_host, qq_host = [], [], [], [], [], []
    for i in range(n_inst):
        qseq = W.query_sequence(wl, i)
        k, v = W.gen_kv(wl, i, qseq)
        sob, bos, lu = W.initial_resident(wl, i)
        layers.append(LayerState(wl, bits_to_bf16(k), bits_to_bf16(v), sob, bos, lu, device=str(dev)))
        del k, v
        qs, qds, hq, hqd, hqq = [], [], [], [], []
        for t in range(QUERY_SETS):
            q, qd = W.step_queries(wl, qseq, t)
            # a step's queries and draft queries sit in one pinned buffer: one copy per step
            both = torch.cat([bits_to_bf16(q).flatten(), bits_to_bf16(qd).flatten()]).pin_memory()
            hqq.append(both)
            hq.append(both[:q.size].view(q.shape))
            hqd.append(both[q.size:].view(qd.shape))
            qs.append(hq[-1].to(dev))
            qds.append(hqd[-1].to(dev))
        q_dev.append(qs)
        qd_dev.append(qds)
        q_host.append(hq)
        qd_host.append(hqd)
        qq_host.append(hqq)
    torch.cuda.synchronize()

    compute = torch.cuda.Stream(device=dev)
    score_st = torch.cuda.Stream(device=dev)
    select_st = torch.cuda.Stream(device=dev)
    copy = torch.cuda.Stream(device=dev, priority=-1)
    h2d = torch.cuda.Stream(device=dev)
    d2h = torch.cuda.Stream(device=dev)
    side = torch.cuda.Stream(device=dev)
    out_host = [torch.empty_like(L.out, device="cpu").pin_memory() for L in layers]
    # the decoded token's K and V rows per layer copy, for the growing-context run
    gen = torch.Generator(device=dev)
    gen.manual_seed(wl.seed + 7)
    kv_new = [tuple((torch.randn((wl.batch, wl.num_kv_heads, wl.head_dim), generator=gen,
                                 device=dev) * 0.5).to(torch.bfloat16) for _ in range(2))
              for _ in range(n_inst)]
    qq_in = [torch.empty_like(qq_host[i][0], device=dev) for i in range(n_inst)]
    nq = q_dev[0][0].numel()
    q_in = [qq_in[i][:nq].view(q_dev[i][0].shape) for i in range(n_inst)]
    qd_in = [qq_in[i][nq:].view(qd_dev[i][0].shape) for i in range(n_inst)]

    def qset(s):
        return s % n_inst, (s // n_inst) % QUERY_SETS

    def enqueue(s, active, host_io: bool, grow: bool = False, mm: bool = False):
        """Graph body of step s, a software pipeline over the layer copies as in
        Fig. 8 (each layer's prediction and transfer run in the background of
        the following layers): the attention of step s and the scoring of step
        s-1 in one launch on `compute`, and beside it top-K + plan of step s-2
        and the transfer of step s-3, each on its own stream.  `active` = which of the four run (the
        first and last graphs of a run fill and drain the pipeline).  The four
        steps use four different layer copies, and each one's inputs were
        produced by an earlier graph.  With host I/O, step s+2's queries are
        copied in from pinned host memory and step s-1's output is copied out
        beside step s's kernels (a run's first step copies its own queries in
        before its attention, and the second step's beside them): each copy has
        two steps to land, and its destination (the buffer of a layer copy
        last read two steps earlier) is free.  With `grow`, step s first appends its token to
        its layer copy (cache, working set, summaries, context length) and the
        selection uses the window at each context's end.  With `mm`, the
        scoring runs against the min/max compressed keys."""
        fork = torch.cuda.Event()
        fork.record(compute)
        joins = []

        def branch(stream, fn):
            stream.wait_event(fork)
            fn(stream)
            e = torch.cuda.Event()
            e.record(stream)
            joins.append(e)

        def copy_in(stream, step):
            i, qi = qset(step)
            with torch.cuda.stream(stream):
                qq_in[i].copy_(qq_host[i][qi], non_blocking=True)

        if "h2d_now" in active:
            branch(h2d, lambda st: copy_in(st, s))
            compute.wait_event(joins.pop())
        if "h2d_now1" in active:
            branch(h2d, lambda st: copy_in(st, s + 1))
        # the attention of step s and the scoring of step s-1 share one launch
        # (oasis_attend_and_score) when both run; it is enqueued first
        fused = "attn" in active and "score" in active
        if "attn" in active:
            i, qi = qset(s)
            L = layers[i]
            if grow:
                L.append(kv_new[i][0], kv_new[i][1], compute)
                # the newest block's summaries beside the attention; needed by
                # this copy's scoring in the next step
                appended = torch.cuda.Event()
                appended.record(compute)
                side.wait_event(appended)
                L.refresh_summaries(side)
                refreshed = torch.cuda.Event()
                refreshed.record(side)
                joins.append(refreshed)
            q = q_in[i] if host_io else q_dev[i][qi]
            if fused:
                i1, qi1 = qset(s - 1)
                qd1 = qd_in[i1] if host_io else qd_dev[i1][qi1]
                if mm:
                    L.attention_and_score_minmax(q, layers[i1], qd1, compute)
                else:
                    L.attention_and_score(q, layers[i1], qd1, compute)
            else:
                L.attention(q, compute)
        if "score" in active and not fused:
            i1, qi1 = qset(s - 1)
            qd = qd_in[i1] if host_io else qd_dev[i1][qi1]
            L1 = layers[i1]
            if mm:
                branch(score_st, lambda st: L1.score_minmax(qd, st))
            else:
                branch(score_st, lambda st: ob.oasis_score_blocks(L1.cfg, qd, L1.summ, L1.scores, st))
        if "select" in active and grow:
            L2 = layers[(s - 2) % n_inst]
            branch(select_st, lambda st: L2.select_ctx(st))
        elif "select" in active:
            L2 = layers[(s - 2) % n_inst]
            branch(select_st, lambda st: ob.oasis_predict_select(
                L2.cfg, L2.scores, 0, L2.clock, L2.topk, L2.slot_of_block, L2.block_of_slot,
                L2.last_used, L2.fetch_block, L2.fetch_slot, L2.evict_block, L2.n_fetch,
                L2.n_evict, st))
        if "fetch" in active:
            L3 = layers[(s - 3) % n_inst]
            branch(copy, lambda st: L3.fetch(st))
        if "h2d_next" in active:
            branch(h2d, lambda st: copy_in(st, s + 2))
        if "d2h_prev" in active:
            ip = (s - 1) % n_inst

            def copy_out(st):
                with torch.cuda.stream(st):
                    out_host[ip].copy_(layers[ip].out, non_blocking=True)
            branch(d2h, copy_out)
        for e in joins:
            compute.wait_event(e)

    def active_of(s, s0, n, host_io=False):
        parts = []
        for name, lag in (("attn", 0), ("score", 1), ("select", 2), ("fetch", 3)):
            if s0 <= s - lag < s0 + n:
                parts.append(name)
        if host_io:
            if s == s0:
                parts.append("h2d_now")
                if n > 1:
                    parts.append("h2d_now1")
            if s0 <= s + 2 < s0 + n:
                parts.append("h2d_next")
            if s0 <= s - 1 < s0 + n:
                parts.append("d2h_prev")
        return frozenset(parts)

    # ---- warm the library (first calls set up per-device state)
    with torch.cuda.stream(compute):
        for s_ in range(2 * n_inst + 3):
            enqueue(s_, active_of(s_, 0, 2 * n_inst), host_io=False)
    torch.cuda.synchronize()
    period = n_inst * QUERY_SETS
    graphs = {}

    def graph_for(s, active, host_io, grow=False, mm=False):
        key = (s % period, active, host_io, grow, mm)
        if key not in graphs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=compute):
                enqueue(s, active, host_io, grow, mm)
            graphs[key] = g
        return graphs[key]

    # Steady-state steps are replayed CHUNK at a time (one graph per four
    # cycles of the layer copies): fewer graph launches per step, both for the
    # host and for the GPU's front end (measured 29.3 / 28.2 / 27.6 us per step
    # at 4 / 8 / 16 steps per graph); the pipeline's fill and drain use one
    # graph per step.
    CHUNK = 4 * n_inst
    def full_mask(host_io):
        return frozenset(("attn", "score", "select", "fetch")
                         + (("h2d_next", "d2h_prev") if host_io else ()))

    def chunk_graph(s, host_io, grow=False, mm=False):
        key = ("chunk", s % period, host_io, grow, mm)
        if key not in graphs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=compute):
                for k in range(CHUNK):
                    enqueue(s + k, full_mask(host_io), host_io, grow, mm)
            graphs[key] = g
        return graphs[key]

    def run_steps(s0, n, host_io=False, grow=False, mm=False):
        """Exactly the work of layer-steps s0..s0+n-1 (the pipeline fills in
        the first three graph steps and drains in the last three)."""
        end = s0 + n + 3
        full = full_mask(host_io)
        torch.cuda.nvtx.range_push(f"layer-steps {s0}..{s0 + n - 1}"
                                   + (" host-io" if host_io else "") + (" grow" if grow else "")
                                   + (" minmax" if mm else ""))
        with torch.cuda.stream(compute):
            s = s0
            while s < end:
                if s + CHUNK <= end and all(active_of(s + k, s0, n, host_io) == full
                                            for k in range(CHUNK)):
                    chunk_graph(s, host_io, grow, mm).replay()
                    s += CHUNK
                else:
                    graph_for(s, active_of(s, s0, n, host_io), host_io, grow, mm).replay()
                    s += 1
        torch.cuda.nvtx.range_pop()

    # capture every graph the long runs below need, outside the timed regions,
    # and upload each to the device (a graph's first launch otherwise pays for
    # its upload, ~ms for a 16-step graph, inside whichever run launches it first)
    def capture_all(grow, mm=False):
        for io in ((False,) if (args.no_e2e or grow or mm) else (False, True)):
            masks = {active_of(s_, 100, 50, io) for s_ in range(100, 153)}
            for s_ in range(period):
                for m in masks:
                    graph_for(s_, m, io, grow, mm)
                chunk_graph(s_, io, grow, mm)
        for g_ in graphs.values():
            upload_graph(g_, compute)
        torch.cuda.synchronize()

    capture_all(False)

    if args.profile_steps:
        if args.profile_grow:  # the growing-context form of the step
            for L in layers:
                L.ctx_len = torch.full((wl.batch,), wl.ctx_tokens - GROW_ROOM, dtype=torch.int32,
                                       device=dev)
                L.cfg.local_blocks = max(L.cfg.local_blocks, 1)
        run_steps(0, args.profile_steps, grow=args.profile_grow)
        for r in range(args.profile_joint):  # joint attention launches after the steps
            layers[r % n_inst].attention_joint(q_dev[r % n_inst][0], qd_dev[r % n_inst][0], compute)
        if args.profile_minmax:
            for L in layers:
                L.build_minmax_summaries()
        for r in range(args.profile_minmax):  # then min/max scoring launches
            layers[r % n_inst].score_minmax(qd_dev[r % n_inst][0], compute)
        for r in range(args.profile_chain):  # then prediction-chain launches
            layers[r % n_inst].predict_chain(qd_dev[r % n_inst][0], compute)
        torch.cuda.synchronize()
        print(json.dumps({"profile_steps": args.profile_steps, "profile_joint": args.profile_joint,
                          "profile_minmax": args.profile_minmax, "profile_chain": args.profile_chain}),
              flush=True)
        return

    # ---- warm-up and timed region
    s = 0
    run_steps(s, args.warmup)
    s += args.warmup
    torch.cuda.synchronize()
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    gpu_index = int(vis.split(",")[local]) if vis and vis.split(",")[local].strip().isdigit() else local
    clocks = ClockSampler(gpu_index)
    clocks.start()
    # load soak: the sampler sees the GPU under this same work for ~0.6 s
    # before and through the timed region
    w0 = time.perf_counter()
    while time.perf_counter() - w0 < 0.6:
        run_steps(s, 2000)
        s += 2000
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(compute)
    run_steps(s, args.steps)
    t1.record(compute)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    s += args.steps
    ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    ms_per_step = ms / args.steps
    value = job_throughput(world, wl.batch, ms_per_step)

    # ---- per-kernel timing: a CUDA graph of 8 launches of one kernel over the
    # layer copies (cold L2), bracketed by events on the launching stream
    def kernel_graph(kind):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=compute):
            for r in range(8):
                i = r % n_inst
                L = layers[i]
                if kind == "attn":
                    L.attention(q_dev[i][0], compute)
                elif kind == "score":
                    ob.oasis_score_blocks(L.cfg, qd_dev[i][0], L.summ, L.scores, compute)
                elif kind == "topk":
                    ob.oasis_select_topk(L.cfg, L.scores, L.topk, compute)
                elif kind == "fused":
                    L.attention_and_score(q_dev[i][0], layers[(i + 1) % n_inst],
                                          qd_dev[(i + 1) % n_inst][0], compute)
                elif kind == "joint":
                    L.attention_joint(q_dev[i][0], qd_dev[i][0], compute)
                elif kind == "score_mm":
                    L.score_minmax(qd_dev[i][0], compute)
                elif kind == "chain":
                    L.predict_chain(qd_dev[i][0], compute)
                elif kind == "score_select":  # the same chain as two launches
                    ob.oasis_score_blocks(L.cfg, qd_dev[i][0], L.summ, L.scores, compute)
                    ob.oasis_predict_select(
                        L.cfg, L.scores, 0, L.clock, L.topk, L.slot_of_block, L.block_of_slot,
                        L.last_used, L.fetch_block, L.fetch_slot, L.evict_block, L.n_fetch,
                        L.n_evict, compute)
        return g

    for L in layers:  # min/max compressed keys for the scoring variant (set-up)
        L.build_minmax_summaries()
    torch.cuda.synchronize()
    kinds = ["attn", "score", "topk", "fused", "joint", "score_mm", "chain", "score_select"]
    mean_ms = {}
    for kind in kinds:
        g = kernel_graph(kind)
        with torch.cuda.stream(compute):
            g.replay()
        torch.cuda.synchronize()
        vals = []
        for _ in range(5):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(compute)
            with torch.cuda.stream(compute):
                g.replay()
            b.record(compute)
            torch.cuda.synchronize()
            vals.append(a.elapsed_time(b) / 8)
        mean_ms[kind] = statistics.mean(vals)
        del g
    # transfer volume and working-set occupancy over further (untimed) steps
    fetched, valid = [], []
    for r in range(n_inst * 10):
        run_steps(s, 1)
        s += 1
        torch.cuda.synchronize()
        L = layers[(s - 1) % n_inst]
        fetched.append(int(L.n_fetch.sum().item()))
        valid.append(int((L.block_of_slot >= 0).sum().item()))
    n_fetch_avg = statistics.mean(fetched)
    valid_avg = statistics.mean(valid)
    by = algorithmic_bytes(wl, n_fetch_avg, valid_avg)
    peak, peak_kind = measured_peaks()
    # the step's dominant kernel: the fused attention + scoring launch
    dominant = "fused"
    kname = "attn_score_kernel"
    achieved = by[dominant] / (mean_ms[dominant] * 1e-3) / 1e9
    traffic = committed_traffic(kname)

    # ---- host link peak (pinned cudaMemcpyAsync), for the step roofline
    hb = torch.empty(256 << 20, dtype=torch.uint8).pin_memory()
    db = torch.empty_like(hb, device=dev)
    best = 1e9
    for _ in range(4):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        db.copy_(hb, non_blocking=True)
        b.record()
        torch.cuda.synchronize()
        best = min(best, a.elapsed_time(b))
    link_gbs = hb.numel() / (best * 1e-3) / 1e9
    del hb, db
    t_roof = max(by["hbm"] / (peak * 1e9), by["link"] / (link_gbs * 1e9))
    step_frac = t_roof / (ms_per_step * 1e-3)
    # the narrower forms: resident KV read by the attention and the fetched
    # bytes only, as the slowest tier (max) and as the sum of the two tiers
    kv_read = valid_avg * wl.block_size * wl.head_dim * 2 * 2
    t_kv = kv_read / (peak * 1e9)
    t_link = by["link"] / (link_gbs * 1e9)

    # ---- end to end: inputs copied in from pinned host, output read back, every step
    e2e = None
    if not args.no_e2e:
        # its own untimed warm-up, one period of the query sets: the host-I/O
        # graphs' first launches and the device's first touch of every pinned
        # input buffer (measured: 512 timed steps after 16 warm-up steps ran
        # at 49 us per step, 10,000 at 33 us)
        n_warm = max(args.warmup, period + 4 * n_inst)
        run_steps(s, n_warm, host_io=True)
        s += n_warm
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_e2e = args.steps
        w0 = time.perf_counter()
        e0.record(compute)
        run_steps(s, n_e2e, host_io=True)
        e1.record(compute)
        torch.cuda.synchronize()
        wall = time.perf_counter() - w0
        s += n_e2e
        ems = max_over_ranks(e0.elapsed_time(e1), world, dev)
        q_bytes = q_host[0][0].numel() * 2 + qd_host[0][0].numel() * 2
        e2e = {"value": job_throughput(world, wl.batch, ems / n_e2e), "unit": UNIT,
               "h2d_bytes_per_step": q_bytes, "d2h_bytes_per_step": out_host[0].numel() * 2,
               "wall_s": wall}

    # ---- the same pipelined step with the min/max compressed keys (scoring
    # of the same bytes per block on bf16 tensor cores)
    mm_step = None
    if not args.no_minmax_step:
        capture_all(False, mm=True)
        n_warm = max(args.warmup, period + 4 * n_inst)
        run_steps(s, n_warm, mm=True)
        s += n_warm
        n_mm = min(args.steps, 4000)
        torch.cuda.synchronize()
        m0, m1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        m0.record(compute)
        run_steps(s, n_mm, mm=True)
        m1.record(compute)
        torch.cuda.synchronize()
        s += n_mm
        mms = max_over_ranks(m0.elapsed_time(m1), world, dev) / n_mm
        mm_step = {"ms_per_step": mms, "value": job_throughput(world, wl.batch, mms), "unit": UNIT,
                   "steps": n_mm, "step_roofline_frac": t_roof / (mms * 1e-3),
                   "vs_mean_keys_step": mms / ms_per_step,
                   "kernels": "attn_score_kernel (min/max keys) | topk_plan_kernel | fetch_kernel"}

    # ---- growing context: the same pipelined step with each step's token
    # appended first (cache, working set, summaries, context length) and the
    # selection's local window following the context (device-timed, like value)
    grow = None
    if not args.no_grow:
        ctx0 = wl.ctx_tokens - GROW_ROOM
        for L in layers:
            L.ctx_len = torch.full((wl.batch,), ctx0, dtype=torch.int32, device=dev)
            # a local window of at least the newest block, so that the planner
            # keeps the block the appends write into resident
            L.cfg.local_blocks = max(L.cfg.local_blocks, 1)
        capture_all(True)
        n_warm = max(args.warmup, period + 4 * n_inst)  # every chunk graph of the run once
        run_steps(s, n_warm, grow=True)
        s += n_warm
        n_grow = min(args.steps, GROW_ROOM * n_inst // 2 - n_warm)
        torch.cuda.synchronize()
        # timed in eight consecutive segments (one stream, no gap): the
        # per-segment times show how the working set settles to the moving window
        seg = [n_grow // 8] * 8
        seg[-1] += n_grow - sum(seg)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(9)]
        ev[0].record(compute)
        for k, n_k in enumerate(seg):
            run_steps(s, n_k, grow=True)
            s += n_k
            ev[k + 1].record(compute)
        torch.cuda.synchronize()
        gms = max_over_ranks(ev[0].elapsed_time(ev[8]), world, dev) / n_grow
        seg_us = [ev[k].elapsed_time(ev[k + 1]) / seg[k] * 1e3 for k in range(8)]
        # the append and refresh kernels alone: graphs of 8 launches over the copies
        def time_graph(fn):
            gx = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gx, stream=compute):
                for r in range(8):
                    fn(layers[r % n_inst], r % n_inst)
            vals = []
            for _ in range(5):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(compute)
                with torch.cuda.stream(compute):
                    gx.replay()
                b.record(compute)
                torch.cuda.synchronize()
                vals.append(a.elapsed_time(b) / 8)
            return statistics.mean(vals)
        append_ms = time_graph(lambda L, i: L.append(kv_new[i][0], kv_new[i][1], compute))
        refresh_ms = time_graph(lambda L, i: L.refresh_summaries(compute))
        ctx_end = [int(L.ctx_len.max().item()) for L in layers]
        gf = []
        for r in range(n_inst * 4):  # transfer volume over further (untimed) steps
            run_steps(s, 1, grow=True)
            s += 1
            torch.cuda.synchronize()
            gf.append(int(layers[(s - 1) % n_inst].n_fetch.sum().item()))
        grow = {"ms_per_step": gms, "value": job_throughput(world, wl.batch, gms), "unit": UNIT,
                "vs_fixed_context_step": gms / ms_per_step, "append_ms_per_launch": append_ms,
                "refresh_ms_per_launch": refresh_ms, "fetched_blocks_per_step": statistics.mean(gf),
                "us_per_step_by_eighth": seg_us,
                "ctx_start": ctx0, "ctx_end_per_copy": ctx_end, "steps": n_grow,
                "local_blocks": layers[0].cfg.local_blocks,
                "kernels": "append_kernel, then attn_score_kernel beside refresh_kernel; "
                           "topk_plan_kernel with the window at each context's end; fetch_kernel"}

    errs = ob.oasis_device_errors()
    cpu = cpu_all = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.cpu_seconds)
        cpu_all = cpu_baseline_all_cores(args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {
                "workload": wl.name, "global_batch": wl.batch * world, "seq_len": wl.ctx_tokens,
                "kv_budget_tokens": wl.kv_budget_tokens, "lookahead": wl.lookahead,
                "top_k": wl.top_k, "fetch_ratio": wl.fetch_ratio, "fetch_cap": ob.oasis_fetch_cap(wl),
                "layers": 1, "layer_copies_cycled": n_inst, "parallelism": f"replicas x{world}",
                "l2": f"inputs larger than L2: {n_inst} layer copies of {by['hbm'] / 1e6:.0f} MB cycled",
                "tok_s_if_32_layers": value / 32,
                "graphs": "step s: [attn(s) + score(s-1) fused] | select(s-2) | transfer(s-3); "
                          "16 steps per CUDA graph in the steady state; LRU step in device memory"},
            "roofline": {"bound": "hbm", "kernel": kname, "achieved": achieved, "peak": peak,
                         "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                         "peak_source": peak_kind,
                         "bytes_per_launch": by[dominant], "ms_per_launch": mean_ms[dominant]},
            "step_roofline": {"t_roof_us": t_roof * 1e6, "t_step_us": ms_per_step * 1e3,
                              "frac": step_frac, "hbm_bytes": by["hbm"], "link_bytes": by["link"],
                              "hbm_peak_gbs": peak, "link_peak_gbs": link_gbs,
                              "fetched_blocks_per_step": n_fetch_avg,
                              "kv_read_bytes": kv_read,
                              "frac_kv_read_and_link_max": max(t_kv, t_link) / (ms_per_step * 1e-3),
                              "frac_kv_read_plus_link_sum": (t_kv + t_link) / (ms_per_step * 1e-3)},
            "joint_attention": {
                "kernel": "attn_joint_kernel", "rows_per_unit": wl.group * (1 + wl.lookahead),
                "ms_per_launch": mean_ms["joint"], "bytes_per_launch": by["joint"],
                "achieved_gbs": by["joint"] / (mean_ms["joint"] * 1e-3) / 1e9,
                "frac_of_measured_hbm": by["joint"] / (mean_ms["joint"] * 1e-3) / 1e9 / peak,
                "vs_single_query_attention": mean_ms["joint"] / mean_ms["attn"]},
            "minmax_scoring": {
                "kernel": "score_kernel (min/max keys)", "ms_per_launch": mean_ms["score_mm"],
                "bytes_per_launch": by["score_mm"],
                "achieved_gbs": by["score_mm"] / (mean_ms["score_mm"] * 1e-3) / 1e9,
                "frac_of_measured_hbm": by["score_mm"] / (mean_ms["score_mm"] * 1e-3) / 1e9 / peak,
                "vs_mean_scoring": mean_ms["score_mm"] / mean_ms["score"]},
            "predict_chain": {
                "kernel": "chain_kernel", "ms_per_launch": mean_ms["chain"],
                "bytes_per_launch": by["chain"],
                "achieved_gbs": by["chain"] / (mean_ms["chain"] * 1e-3) / 1e9,
                "frac_of_measured_hbm": by["chain"] / (mean_ms["chain"] * 1e-3) / 1e9 / peak,
                "separate_launches_ms": mean_ms["score_select"],
                "vs_separate_launches": mean_ms["chain"] / mean_ms["score_select"]},
            "minmax_step": mm_step,
            "growing_context": grow,
            "kernels_ms": mean_ms,
            "kernel_gbs": {k: by[k] / (mean_ms[k] * 1e-3) / 1e9 for k in kinds},
            # in the timed run: n-1 fused attention + scoring launches, the
            # first step's attention and the last step's scoring alone, n top-K +
            # plan and n transfer launches
            "gpu_launches": 3 * args.steps + 1,
            "clocks": clk,
            "cpu_baseline": cpu,
            "cpu_baseline_all_cores": cpu_all,
            "e2e": e2e,
            "device_errors": errs,
        }
        print(json.dumps(line), flush=True)
    for L in layers:
        L.close()
    if world > 1:
        dist.destroy_process_group()


def sweep_arm(args):
    """Fetch-ratio x batch sweep on the Qwen3-8B layer shape (Tab. 2's columns:
    GB fetched per step, host-link GB/s, HBM GB/s, tok/s).  One layer copy per
    batch, its working set reset to the same random start for every ratio;
    each step is the whole hot path in stream order (attention, scoring, top-K
    + plan, transfer: no overlap between layers), timed with CUDA events after
    an L2 flush.  Prints one JSON line per point; not the benchmark line."""
    import torch
    from sparse_kv_cache_oasis_gb300 import binding as ob
    from sparse_kv_cache_oasis_gb300.layer import LayerState, bits_to_bf16
    ob.lib()
    dev = torch.device("cuda", 0)
    st = torch.cuda.Stream(device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # twice the L2
    peak, _ = measured_peaks()
    for B in [int(x) for x in args.sweep_batches.split(",")]:
        wl = W.sweep_point(-1.0, B)
        qseq = W.query_sequence(wl, 0)
        k, v = W.gen_kv(wl, 0, qseq)
        sob, bos, lu = W.initial_resident(wl, 0)
        L = LayerState(wl, bits_to_bf16(k), bits_to_bf16(v), sob, bos, lu, device=str(dev))
        del k, v
        start = [t.clone() for t in (L.slot_of_block, L.block_of_slot, L.last_used, L.pool_k, L.pool_v)]
        qs = [tuple(bits_to_bf16(a).to(dev) for a in W.step_queries(wl, qseq, t)) for t in range(wl.steps)]
        for ratio in W.SWEEP_RATIOS:
            L.cfg.fetch_ratio = ratio
            w = ob.cap_width(L.cfg)
            for name in ("fetch_block", "fetch_slot", "evict_block"):
                setattr(L, name, torch.full((B, wl.num_kv_heads, w), -1, dtype=torch.int32, device=dev))
            for dst, src in zip((L.slot_of_block, L.block_of_slot, L.last_used, L.pool_k, L.pool_v), start):
                dst.copy_(src)
            torch.cuda.synchronize()
            times, fetched = [], []
            for t in range(16 + wl.steps):
                q, qd = qs[t % wl.steps]
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(st):
                    st.wait_stream(torch.cuda.current_stream())
                    e0.record(st)
                    L.attention(q, st)
                    L.predict(qd, t, st)
                    L.fetch(st)
                    e1.record(st)
                torch.cuda.synchronize()
                if t >= 16:  # after sixteen warm-up steps
                    times.append(e0.elapsed_time(e1) * 1e-3)
                    fetched.append(int(L.n_fetch.sum().item()))
            t_step = statistics.mean(times)
            nf = statistics.mean(fetched)
            by = algorithmic_bytes(wl, nf, float((L.block_of_slot >= 0).sum().item()))
            print(json.dumps({
                "sweep": "qwen3-8b-layer ctx32k budget2k L4", "batch": B,
                "fetch_ratio": ratio if ratio >= 0 else "all", "fetch_cap": ob.oasis_fetch_cap(L.cfg),
                "us_per_step_serial": t_step * 1e6, "tok_s": B / t_step,
                "gb_per_step": by["link"] / 1e9, "link_gbs": by["link"] / t_step / 1e9,
                "hbm_gbs": by["hbm"] / t_step / 1e9, "hbm_frac_of_measured": by["hbm"] / t_step / 1e9 / peak,
                "fetched_blocks_per_step": nf, "steps": wl.steps, "data": "synthetic"}), flush=True)
        L.close()
        del L, start, qs
        torch.cuda.empty_cache()
    assert ob.oasis_device_errors() == 0


def main():
    args = parse()
    if args.impl == "reference":
        reference_arm(args)
        return
    if args.sweep:
        sweep_arm(args)
        return
    gpu_arm(args)


if __name__ == "__main__":
    main()
