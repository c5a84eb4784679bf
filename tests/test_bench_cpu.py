"""Host-side pieces of bench.py: the algorithmic byte counts (the FP8 pools
hold one byte per element, so the decode batch's K/V bytes halve), the kernel
launch count per step (the write inside the planner's launch), and the block manager's host timing on a small batch."""
import numpy as np

import bench
import workloads as wl


def test_fp8_halves_the_cached_bytes():
    w = wl.random_small(3, batch=4, max_ctx=200, max_q=1, num_q_heads=8, num_kv_heads=2)
    a, b = bench.algorithmic_bytes(w), bench.algorithmic_bytes(w, fp8=True)
    assert b["kv"] * 2 == a["kv"]
    assert b["attn_kernel"] - b["kv"] == a["attn_kernel"] - a["kv"]       # q and out stay bf16
    T, H, D = w.step.num_tokens, w.num_kv_heads, w.head_dim
    assert a["write"] - b["write"] == 2 * T * H * D                       # one byte less per written element


def test_launches_per_step():
    w = wl.random_small(4, batch=4, max_ctx=200, max_q=1, num_q_heads=8, num_kv_heads=2)
    # the step's write runs in the planner's launch (paged_kv_write_attention_forward)
    assert bench.launches_per_step(w, 1, False, fp8=True) == 2
    assert bench.launches_per_step(w, 1, False) == 2          # planner with the write, tensor-core decode
    assert bench.launches_per_step(w, 0, False) == 3          # + the multi-token kernel (no hint)
    assert bench.launches_per_step(w, 1, True) == 4           # + the prefix search and prefix items


def test_block_manager_timing_runs_on_the_host():
    w = wl.random_small(5, batch=6, max_ctx=300, max_q=4, num_q_heads=8, num_kv_heads=2)
    r = bench.block_manager_timing(w, reps=3, with_oracle=True)
    assert r["value"] > 0 and r["oracle_us_per_step"] > 0 and r["reps"] == 3

