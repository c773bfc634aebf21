"""The benchmark's byte counts against the per-unit figures of the method.

At the Llama-3.1-8B-shaped layer (64 (request, KV head) units, 2,048 blocks
of 16 tokens, 128 working-set slots, head_dim 128): the attention reads 128
slots x 8 KiB of K and V per unit (1 MiB), the scoring 2,048 summaries x
512 B per unit (1 MiB), and a transfer of n blocks moves n x 8 KiB over the
host link and writes as much to HBM.  The queries, outputs, scores, lists and
maps are the small remainder.  CPU only.
"""
import bench
from sparse_kv_cache_oasis_gb300 import workloads as W


def test_llama_layer_bytes_per_step():
    wl = W.LLAMA8B_LAYER
    by = bench.algorithmic_bytes(wl, n_fetch_blocks=430, valid_slots=64 * 128)
    MiB = 1 << 20
    assert by["attn"] == 64 * MiB + 8 * 32 * 128 * 2 * 2 + 64 * 128 * 4      # KV + q/out + slot map
    assert by["score"] == 64 * MiB + 8 * 4 * 32 * 128 * 2 + 64 * 2048 * 4    # summaries + drafts + scores
    assert by["fused"] == by["attn"] + by["score"] == 135_168_000
    assert by["link"] == by["fetch"] == 430 * 8192
    assert by["hbm"] == 135_168_000 + (64 * 2048 * 4 + 64 * 128 * 4) + 64 * (128 * 4 + 128 * 16) + 430 * 8192
    # the min/max keys move as many bytes per block as the fp32 mean
    assert by["score_mm"] == by["score"]
    # joint attention: one KV pass, 1 + L query and output rows per head
    assert by["joint"] == 64 * MiB + 2 * 8 * 32 * 128 * 2 * 5 + 64 * 128 * 4


def test_job_throughput_is_weak_scaling():
    assert bench.job_throughput(1, 8, 0.026) == 8 / 26e-6
    assert bench.job_throughput(4, 8, 0.026) == 4 * bench.job_throughput(1, 8, 0.026)
