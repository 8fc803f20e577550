"""Byte accounting behind bench.py's throughput and roofline (no GPU needed).

The roofline's `achieved` divides the algorithmic bytes of one attention launch by its time, so
those bytes are pinned here to their definition for the Llama-3-8B-layer decode workload
(batch 32, 32 query / 8 kv heads, context 32768, 64 selected pages plus the local page): every
selected page-head's K and V pages (2 x 64 tokens x 128 dims x bf16) read once.
"""
import numpy as np

import bench


def _workload():
    return {"B": 32, "Hk": 8, "Hq": 32, "np_max": 512, "seq_len": np.full(32, 32768, np.int32)}


def test_attention_bytes_are_every_selected_page_read_once():
    b = bench.step_bytes(_workload(), 64)
    assert b["attn_kv"] == 32 * 8 * 65 * (2 * 64 * 128 * 2) == 545_259_520


def test_score_bytes_are_the_pooled_sums_of_every_complete_page():
    b = bench.step_bytes(_workload(), 64)
    sums = 32 * 8 * 511 * (4 * 128 * 4)          # fp32 sums, 4 sub-blocks, pages before the local one
    tables = 32 * 512 * 4 + 32 * 32 * 128 * 2 + 32 * 8 * 512 * 4   # page table, q, scores out
    assert b["score"] == sums + tables


def test_replica_throughput_counts_all_ranks():
    assert bench.replica_throughput(1, 1e9, 1.0) == 1000.0
    assert bench.replica_throughput(4, 1e9, 2.0) == 2000.0


def test_committed_traffic_is_close_to_the_algorithmic_bytes():
    """When the ncu summary matches the attention source, its DRAM traffic per full launch lies
    within a few percent above the algorithmic bytes (outputs and split-K partials on top)."""
    t = bench.measured_traffic()
    if t is None:   # the source changed since the capture: the bench reports null
        return
    kv = bench.step_bytes(_workload(), 64)["attn_kv"]
    assert kv <= t <= 1.05 * kv
