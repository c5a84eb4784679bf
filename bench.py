#!/usr/bin/env python
"""Benchmark of the paged-KV hot path on GB300.

One step = one pass of the whole hot path over one batch: the write of the
batch's new K/V rows into the block pool, then attention over it, through
paged_kv_write_attention_forward (one call; the write runs in the planner's
launch).
Default workload: the decode batch (64 sequences, contexts U[512, 4096], one
query token each, 32 q / 8 kv heads, head_dim 128, block_size 16, bf16, a
20000-block pool, seeded random block permutation).  Also measured (extra
keys): the mixed continuous batch (8 prefill chunks of 512 tokens + 120
decodes) as query tokens/s.

Metric: algorithmic bytes of a step (unique K/V bytes read + q read + output
written + the write path's read and write of the new rows + block-table
entries used) / step time, in GB/s.  Inputs sit in HBM before the timed
region; L2 (129 MB) is flushed between steps by writing a 512 MB buffer
outside the timed events.

Prints one JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle
instead, on a bounded sample of the same workload, on the host cores.
Multi-GPU (torchrun): independent replicas, one per rank (the path needs no
exchange); value = all ranks' bytes / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged-attn decode KV GB/s (% HBM peak); mixed-batch query tokens/s"
BASE_SEED = {"decode": 1002, "mixed": 1003, "prefill": 1003, "specverify": 1004, "prefix": 1005, "prefix-long": 1006,
             "decode-fp8": 1002, "prefill-g7": 1003, "prefill-d64": 1003}
# The FP8 (E4M3) cache workload: the decode batch with both pools encoded with
# one scale each, chosen so that N(0, 1) values span the E4M3 range.
FP8_SCALE = 4.5 / 448
WORKLOAD_DESC = {
    "decode": "decode batch: 64 seqs, context U[512,4096], 1 query token, 32q/8kv heads, head_dim 128, "
              "block_size 16, 20000-block pool, random block permutation, bf16",
    "mixed": "mixed continuous batch: 8 prefill chunks of 512 tokens on U[0,2048] cached + 120 decodes with "
             "context U[256,8192], 32q/8kv heads, head_dim 128, block_size 16, 80000-block pool, bf16",
    "prefill": "the mixed batch's 8 prefill chunks alone (512 tokens on U[0,2048] cached), 32q/8kv, head_dim 128, "
               "block_size 16, bf16",
    "prefill-g7": "the prefill chunks (8 x 512 tokens on U[0,2048] cached) with 56q/8kv heads (GQA group 7), "
                  "head_dim 128, block_size 16, bf16",
    "prefill-d64": "the prefill chunks (8 x 512 tokens on U[0,2048] cached) with 32q/8kv heads and head_dim 64, "
                   "block_size 16, bf16",
    "specverify": "speculative verify: 32 seqs x 5 query tokens on 8192-token contexts, 64q/8kv heads, head_dim "
                  "128, block_size 32, 10240-block pool, bf16",
    "prefix": "prefix-shared decode: 256 seqs sharing a 2048-token prefix (128 blocks) + private U[128,1024] "
              "suffixes, 1 query token, 32q/8kv, head_dim 128, block_size 16, bf16; shared-prefix hint set",
    "prefix-long": "long-context prefix-shared decode: 4 seqs x 131072 tokens (2048 shared), 1 query token, "
                   "32q/8kv, head_dim 128, block_size 16, bf16; shared-prefix hint set",
    "decode-fp8": "decode batch with FP8 (E4M3) K/V pools: 64 seqs, context U[512,4096], 1 query token, 32q/8kv "
                  "heads, head_dim 128, block_size 16, 20000-block pool, q/out bf16, one scale per pool "
                  "(4.5/448)",
}


def workload_of(name: str, seed: int):
    import workloads as wl
    return wl.decode_batch(seed=seed) if name == "decode-fp8" else wl.CONFIGS[name](seed=seed)


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 1950.7)), "measured"
    return 6800.0, 1900.0, "fallback"


def algorithmic_bytes(w, fp8: bool = False) -> dict:
    """Bytes a perfect implementation must move for one step of workload w
    (fp8: the pools hold one-byte codes; q, out and the new rows stay bf16)."""
    st = w.step
    es = 2 if w.dtype == "bf16" else 4
    kv_es = 1 if fp8 else es
    Hkv, D, Hq = w.num_kv_heads, w.head_dim, w.num_q_heads
    L = st.context_lens.astype(np.int64)
    shared = int(w.meta.get("shared_prefix_tokens", 0))
    # unique KV tokens: a shared prefix is read from HBM once
    uniq_tokens = int(L.sum()) - (shared * (len(L) - 1) if shared else 0)
    kv = uniq_tokens * Hkv * D * kv_es * 2
    T = st.num_tokens
    qo = 2 * T * Hq * D * es
    write = 2 * T * Hkv * D * (es + kv_es) + 8 * T
    bt = int(((L + w.block_size - 1) // w.block_size).sum()) * 4 + 8 * len(L) + 4
    attn = kv + qo
    return {"step": attn + write + bt, "attn_kernel": kv + qo, "kv": kv, "write": write}


def mma_flops(w) -> float:
    """Unmasked QK^T and PV flops of the multi-token sequences."""
    st = w.step
    tot = 0.0
    for s in range(st.num_seqs):
        n, L = int(st.q_lens[s]), int(st.context_lens[s])
        if n * (w.num_q_heads // w.num_kv_heads) <= 4:
            continue
        pairs = sum(L - n + i + 1 for i in range(n)) if w.causal else n * L
        tot += 4.0 * w.head_dim * w.num_q_heads * pairs
    return tot


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest value of x over all ranks (x itself when world == 1)."""
    if world <= 1:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def launches_per_step(w, max_q_len: int, shared_prefix: bool, fp8: bool = False) -> int:
    """Our kernels per step, as paged_kv_write_attention_forward chooses them:
    [the shared-prefix search], the planner (whose extra CTAs write the new
    K/V rows), [the tensor-core kernel], the decode-shaped kernel (split
    merges run inside the attention kernels).  FP8 pools: the planner with
    the write, and one decode kernel."""
    if fp8:
        return 2
    g = w.num_q_heads // w.num_kv_heads
    tc = w.dtype == "bf16" and g <= 128                      # the multi-token tensor-core kernel
    dectc = tc and w.head_dim == 128 and g & (g - 1) == 0 and g <= 16
    dec_rows = 16 if dectc else 4
    cascade = shared_prefix and dectc
    mma = tc and (cascade or not (max_q_len > 0 and max_q_len * g <= dec_rows))
    return 2 + int(cascade) + int(mma)


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled in the background."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.proc = None
        self.lines = []
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "20"]
        if gpu_id:
            cmd += ["-i", gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        self.t0 = time.time()

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def _gpu_id(torch, dev):
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        return vis.split(",")[dev.index or 0] if vis else str(dev.index or 0)


def run_gpu(args, rank, world, local_rank):
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_236_gb300 as pkv
    import workloads as wl

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    hbm_peak, bf16_peak, peak_kind = _peaks()

    def to_dev(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(a).to(dev)

    def prepare(w, fp8=False):
        st = w.step
        kc, vc = to_dev(w.k_cache), to_dev(w.v_cache)
        if fp8:
            # the pools' bf16 rows encoded on the device by the library's FP8 write
            NB, bs = kc.shape[0], kc.shape[1]
            kc8 = torch.empty(kc.shape, dtype=torch.uint8, device=dev)
            vc8 = torch.empty_like(kc8)
            slots = torch.arange(NB * bs, dtype=torch.int64, device=dev)
            pkv.paged_kv_write_fp8(kc.view(NB * bs, kc.shape[2], kc.shape[3]), vc.view(NB * bs, kc.shape[2], kc.shape[3]),
                                   slots, kc8, vc8, FP8_SCALE, FP8_SCALE)
            torch.cuda.synchronize()
            del kc, vc, slots
            kc, vc = kc8, vc8
        return dict(kc=kc, vc=vc, fp8=fp8, q=to_dev(st.q), k=to_dev(st.k_new),
                    v=to_dev(st.v_new), slots=torch.from_numpy(st.slot_mapping).to(dev),
                    bt=torch.from_numpy(st.block_tables).to(dev), ctx=torch.from_numpy(st.context_lens).to(dev),
                    qsl=torch.from_numpy(st.query_start_loc).to(dev), mql=int(st.q_lens.max(initial=0)),
                    # a serving system knows when it shares cached prefix blocks between requests
                    sp=bool(w.meta.get("shared_prefix_tokens") or w.meta.get("share_groups")))

    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)

    def timed(w, t, steps, warmup, mma_alone=False):
        out = torch.empty_like(t["q"])
        ws = torch.empty(pkv.workspace_size(w.step.num_seqs, w.step.num_tokens, w.num_q_heads, w.num_kv_heads,
                                            w.head_dim), dtype=torch.uint8, device=dev)

        def one():
            # the step's write and attention in one call (the write in the planner's launch)
            if t["fp8"]:
                pkv.paged_kv_write_attention_forward_fp8kv(t["k"], t["v"], t["slots"], t["q"], t["kc"], t["vc"],
                                                           t["bt"], t["ctx"], t["qsl"], w.scale, FP8_SCALE, FP8_SCALE,
                                                           w.causal, out=out, workspace=ws, max_query_len=t["mql"])
                return
            pkv.paged_kv_write_attention_forward(t["k"], t["v"], t["slots"], t["q"], t["kc"], t["vc"], t["bt"],
                                                 t["ctx"], t["qsl"], w.scale, w.causal, out=out, workspace=ws,
                                                 max_query_len=t["mql"], shared_prefix=t["sp"])

        for _ in range(warmup):
            flush.fill_(1)
            one()
        torch.cuda.synchronize()
        ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(5)) for _ in range(steps)]
        for e in ev:  # torch creates CUDA events lazily: create them before the library records them
            e[2].record()
            e[3].record()
            e[4].record()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        # The step is timed without the library's instrumentation events: an
        # event recorded between the planner and the attention kernel would
        # serialise the two launches, which otherwise overlap (programmatic
        # dependent launch).  The attention kernels alone are then timed in a
        # second pass of the same steps, with those events.
        for e in ev:
            flush.fill_(1)
            e[0].record()
            one()
            e[1].record()
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        step_ms = [e[0].elapsed_time(e[1]) for e in ev]
        torch.cuda.synchronize()
        # mma_alone: the dominant kernel of a batch without decode-shaped work
        # is the tensor-core kernel; an event right after its launch times it
        # alone (the decode kernel's launch then waits for it, which changes
        # nothing when it has no items)
        for e in ev:
            flush.fill_(1)
            pkv.set_profile_events(e[2], e[3])
            pkv.set_profile_mid_event(e[4] if mma_alone else None)
            one()
        pkv.set_profile_events(None, None)
        pkv.set_profile_mid_event(None)
        torch.cuda.synchronize()
        kern_ms = [pkv.profile_elapsed_ms(e[2], e[4] if mma_alone else e[3]) for e in ev]
        return step_ms, kern_ms, out

    # ---------------- headline workload ----------------
    fp8 = args.workload == "decode-fp8"
    w = workload_of(args.workload, BASE_SEED[args.workload] + rank)
    t = prepare(w, fp8)
    sampler = ClockSampler(_gpu_id(torch, dev))
    time.sleep(0.3)
    # the tensor-core kernel alone is the dominant kernel of the prefill and
    # spec-verify batches (no decode-shaped rows)
    mma_alone = args.workload in ("prefill", "prefill-g7", "prefill-d64", "specverify")
    step_ms, kern_ms, out = timed(w, t, args.steps, args.warmup, mma_alone=mma_alone)
    clocks = sampler.stop()
    flags = pkv.device_errors()
    if flags:
        raise SystemExit(f"device error word set: {flags:#x}")
    ab = algorithmic_bytes(w, fp8)
    tot_ms = max_over_ranks(sum(step_ms), world, dev)
    value = ab["step"] * args.steps * world / (tot_ms * 1e-3) / 1e9
    kern_avg_ms = sum(kern_ms) / len(kern_ms)
    if args.workload in ("prefill", "prefill-g7", "prefill-d64"):
        fl = mma_flops(w)
        achieved = fl / (kern_avg_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "kernel": "mma_attn_kernel (tcgen05, per launch, timed alone)", "achieved": round(achieved, 1),
                "peak": bf16_peak, "unit": "TFLOP/s", "frac": round(achieved / bf16_peak, 4),
                "peak_kind": peak_kind + " bf16 dense (burst)", "traffic": ncu_traffic(args.workload),
                "kernel_ms": round(kern_avg_ms, 5), "algorithmic_flops_per_launch": fl}
    else:
        achieved = ab["attn_kernel"] / (kern_avg_ms * 1e-3) / 1e9
        # bf16 head_dim-128 batches run on the tensor-core kernels (the CUDA-core
        # decode_kernel serves the other shapes)
        kname = "mma_attn_kernel (tcgen05, timed alone)" if args.workload == "specverify" else (
            "mma_attn_kernel + dectc_kernel" if args.workload == "mixed" else
            "dectc_kernel (tcgen05 decode, fp16 MMAs on E4M3 tiles converted in shared memory)" if fp8 else
            "dectc_kernel (tcgen05 decode)")
        roof = {"bound": "hbm", "kernel": kname + ", attention kernels per launch", "achieved": round(achieved, 1),
                "peak": hbm_peak, "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                "peak_kind": peak_kind + " HBM copy", "traffic": ncu_traffic(args.workload),
                "kernel_ms": round(kern_avg_ms, 5),
                "algorithmic_bytes_per_launch": ab["attn_kernel"]}

    # ---------------- e2e through the public API, host buffers ----------------
    st = w.step
    pin = lambda a: (torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
                     if a.dtype == np.uint16 else torch.from_numpy(np.ascontiguousarray(a))).pin_memory()
    host_parts = dict(q=pin(st.q), k=pin(st.k_new), v=pin(st.v_new), slots=pin(st.slot_mapping),
                      bt=pin(st.block_tables), ctx=pin(st.context_lens), qsl=pin(st.query_start_loc))
    # As a serving loop would: the step's inputs staged in one pinned buffer
    # (each part 256-byte aligned), sent with one host-to-device copy into a
    # device buffer of the same layout, and read through views of it.
    offs, nbytes = {}, 0
    for k2, x in host_parts.items():
        offs[k2] = nbytes
        nbytes += (x.numel() * x.element_size() + 255) // 256 * 256
    host_buf = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dev_buf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d = {}
    for k2, x in host_parts.items():
        n = x.numel() * x.element_size()
        host_buf[offs[k2]:offs[k2] + n].copy_(x.reshape(-1).view(torch.uint8))
        d[k2] = dev_buf[offs[k2]:offs[k2] + n].view(x.dtype).view(x.shape)
    host_out = torch.empty(tuple(st.q.shape), dtype=t["q"].dtype).pin_memory()
    out_dev = torch.empty_like(t["q"])
    h2d = nbytes
    d2h = host_out.numel() * host_out.element_size()
    ws = torch.empty(pkv.workspace_size(st.num_seqs, st.num_tokens, w.num_q_heads, w.num_kv_heads, w.head_dim),
                     dtype=torch.uint8, device=dev)
    e2e_ms = []
    for it in range(args.warmup + args.steps):
        flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        dev_buf.copy_(host_buf, non_blocking=True)
        if fp8:
            o = pkv.paged_kv_write_attention_forward_fp8kv(d["k"], d["v"], d["slots"], d["q"], t["kc"], t["vc"],
                                                           d["bt"], d["ctx"], d["qsl"], w.scale, FP8_SCALE,
                                                           FP8_SCALE, w.causal, out=out_dev, workspace=ws,
                                                           max_query_len=t["mql"])
        else:
            o = pkv.paged_kv_write_attention_forward(d["k"], d["v"], d["slots"], d["q"], t["kc"], t["vc"], d["bt"],
                                                     d["ctx"], d["qsl"], w.scale, w.causal, out=out_dev,
                                                     workspace=ws, max_query_len=t["mql"], shared_prefix=t["sp"])
        host_out.copy_(o, non_blocking=True)
        b.record()
        b.synchronize()
        if it >= args.warmup:
            e2e_ms.append(a.elapsed_time(b))
    e2e_tot = max_over_ranks(sum(e2e_ms), world, dev)
    e2e_value = ab["step"] * args.steps * world / (e2e_tot * 1e-3) / 1e9

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(tot_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC[args.workload],
                   "step": "paged_kv_write_attention_forward: the write of the batch's new K/V rows and the "
                           "attention in one call (the write runs in the planner's launch)",
                   "l2": "flushed between steps (512 MB write outside the timed events)",
                   "bytes_per_step": ab["step"], "kv_bytes": ab["kv"], "query_tokens": w.step.num_tokens,
                   "parallelism": f"replicas x{world}"},
        "query_tokens_per_s": round(w.step.num_tokens * args.steps * world / (tot_ms * 1e-3), 1),
        "hbm_frac": round(value / hbm_peak, 4),
        "roofline": roof,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_tot / args.steps, 5)},
        "gpu_launches": launches_per_step(w, t["mql"], t["sp"], fp8) * args.steps,
        "clocks": clocks,
    }

    # ---------------- mixed continuous batch (query tokens/s) ----------------
    if args.mixed and args.workload != "mixed":
        wm = wl.mixed_batch(seed=1003 + rank)
        tm = prepare(wm)
        ms_m, kern_m, _ = timed(wm, tm, max(3, args.steps // 2), args.warmup)
        avg = sum(ms_m) / len(ms_m)
        fl = mma_flops(wm)
        result["mixed_batch"] = {
            "value": round(wm.step.num_tokens / (avg * 1e-3), 1), "unit": "query tokens/s",
            "ms_per_step": round(avg, 5), "attn_kernels_ms": round(sum(kern_m) / len(kern_m), 5),
            "bytes_per_step": algorithmic_bytes(wm)["step"],
            "hbm_frac": round(algorithmic_bytes(wm)["step"] / (avg * 1e-3) / 1e9 / hbm_peak, 4),
            "prefill_unmasked_tflop": round(fl / 1e12, 4)}
        result["gpu_launches"] += launches_per_step(wm, tm["mql"], tm["sp"]) * len(ms_m)
        del tm

    # ---------------- prefill chunks alone (tensor-bound multi-token q) ----------------
    if args.mixed and args.workload != "prefill":
        wp = wl.prefill_chunks(seed=1003 + rank)
        tp = prepare(wp)
        ms_p, kern_p, _ = timed(wp, tp, max(3, args.steps // 2), args.warmup, mma_alone=True)
        kavg = sum(kern_p) / len(kern_p)
        fl = mma_flops(wp)
        tfl = fl / (kavg * 1e-3) / 1e12
        result["prefill_chunks"] = {
            "kernel": "mma_attn_kernel (tcgen05, TMEM accumulators, timed alone)", "kernel_ms": round(kavg, 5),
            "achieved": round(tfl, 1), "unit": "TFLOP/s", "peak": bf16_peak, "frac": round(tfl / bf16_peak, 4),
            "peak_kind": peak_kind + " bf16 dense (burst)", "algorithmic_flops_per_launch": fl,
            "flops": "4 * head_dim per unmasked (query row, key) pair: QK^T and PV",
            "traffic": ncu_traffic("prefill"),
            "step_ms": round(sum(ms_p) / len(ms_p), 5),
            "query_tokens_per_s": round(wp.step.num_tokens / (sum(ms_p) / len(ms_p) * 1e-3), 1),
            "workload": WORKLOAD_DESC["prefill"]}
        result["gpu_launches"] += launches_per_step(wp, tp["mql"], tp["sp"]) * len(ms_p)
        del tp

    # ---------------- copy-on-write block copy (HBM-bound) ----------------
    if rank == 0:
        result["copy_blocks"] = copy_blocks_timing(pkv, torch, dev, flush, hbm_peak, args.warmup)
        result["gpu_launches"] += result["copy_blocks"]["launches"]
    if rank == 0:
        result["block_manager"] = block_manager_timing(w, with_oracle=not args.no_cpu_baseline)
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_seconds, fp8=fp8)
    return result


def copy_blocks_timing(pkv, torch, dev, flush, hbm_peak, warmup, reps: int = 10) -> dict:
    """paged_kv_copy_blocks on 2048 (src, dst) pairs of a 4096-block bf16 pool
    (block_size 16, 8 kv heads, head_dim 128: 32 KB per block and pool), one
    layer: 2048 x 2 pools x 32 KB read and as much written (268 MB, above L2),
    L2 flushed before each call; CUDA events on the current stream."""
    nb, pairs_n = 4096, 2048
    kc = torch.zeros((nb, 16, 8, 128), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    perm = np.random.default_rng(9).permutation(nb).astype(np.int32)
    pairs = np.stack([perm[:pairs_n], perm[pairs_n:]], axis=1)
    block_bytes = 16 * 8 * 128 * 2
    moved = pairs_n * 2 * block_bytes * 2
    ms = []
    for i in range(warmup + reps):
        flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        pkv.copy_blocks(kc, vc, pairs)
        b.record()
        b.synchronize()
        if i >= warmup:
            ms.append(a.elapsed_time(b))
    med = statistics.median(ms)
    gbs = moved / (med * 1e-3) / 1e9
    del kc, vc
    return {"value": round(gbs, 1), "unit": "GB/s", "frac": round(gbs / hbm_peak, 4), "ms": round(med, 5),
            "bytes": moved, "pairs": pairs_n, "launches": reps * -(-pairs_n // 4000),
            "what": "copy-on-write of 2048 blocks (K and V, 32 KB each), read + write bytes / median call time"}


def block_manager_timing(w, reps: int = 50, with_oracle: bool = True) -> dict:
    """Host cost of one step's metadata through the library's C++ block
    manager (slots, block tables, context lengths, query offsets,
    copy-on-write pairs) for the workload's batch: each repetition allocates
    the sequences to their cached lengths (untimed), then times the step that
    appends every sequence's query tokens.  The reference model of the same
    manager is timed beside it (the oracle side, fewer repetitions)."""
    import paged_kv_cache_236_gb300 as pkv
    st = w.step
    B = st.num_seqs
    n_new = np.diff(st.query_start_loc).astype(np.int32)
    cached = (st.context_lens - n_new).astype(np.int32)
    width = st.block_tables.shape[1]
    ids = np.arange(B, dtype=np.int64)

    # the manager gives every sequence its own blocks (the workload's shared
    # prefixes are not registered with it): a pool with room for all of them
    nb = int(sum(-(-int(L) // w.block_size) for L in st.context_lens)) + B

    def run(make, k):
        tot = 0.0
        for _ in range(k):
            m = make(nb, w.block_size, width)
            m.step(ids, cached)
            t0 = time.perf_counter()
            m.step(ids, n_new)
            tot += time.perf_counter() - t0
        return tot / k * 1e6

    out = {"value": round(run(pkv.BlockManager, reps), 2), "unit": "us per step (host)", "reps": reps,
           "what": f"BlockManager.step for the workload's {B} sequences ({int(n_new.sum())} new tokens, "
                   f"{width}-block tables), through the Python binding"}
    if with_oracle:
        from oracle.block_manager import BlockManagerModel
        out["oracle_us_per_step"] = round(run(BlockManagerModel, 3), 2)
        out["oracle_reps"] = 3
    return out


def cpu_baseline(w, budget_s: float = 15.0, fp8: bool = False) -> dict:
    """The fp64 oracle, as it stands, on sequences of the same workload until
    the time budget is spent; GB/s over the algorithmic bytes of the rows it
    produced.  fp8: the oracle's E4M3 encoding of each gathered row, decoded,
    then the same attention (bytes counted at one per cached element)."""
    import workloads as wl
    from oracle import fp8 as ofp8
    from oracle import paged_oracle as po
    st = w.step
    es = 2 if w.dtype == "bf16" else 4
    kv_es = 1 if fp8 else es
    kc, vc = w.k_cache, w.v_cache
    done, nbytes = 0, 0
    t0 = time.perf_counter()
    for s in range(st.num_seqs):
        a, b = int(st.query_start_loc[s]), int(st.query_start_loc[s + 1])
        L = int(st.context_lens[s])
        K = wl.to_f64(po.gather(kc, st.block_tables[s], L), w.dtype)
        V = wl.to_f64(po.gather(vc, st.block_tables[s], L), w.dtype)
        if fp8:
            K = ofp8.dequantize(ofp8.quantize(K.astype(np.float32), FP8_SCALE), FP8_SCALE)
            V = ofp8.dequantize(ofp8.quantize(V.astype(np.float32), FP8_SCALE), FP8_SCALE)
        po.attend(wl.to_f64(st.q[a:b], w.dtype), K, V, w.scale, w.causal)
        done += 1
        nbytes += L * w.num_kv_heads * w.head_dim * kv_es * 2 + 2 * (b - a) * w.num_q_heads * w.head_dim * es
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0))
    return {"value": round(nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"first {done} of {st.num_seqs} sequences of {w.name} (gather + fp64 attention, "
                      f"numpy BLAS threads default), {dt:.1f} s"}


def run_reference(args):
    """The oracle as the reference arm: each step one bounded sample of the
    same workload (the oracle on its sequences for about a budget's worth of
    seconds), timed on the host cores."""
    import workloads as wl
    w = workload_of(args.workload, BASE_SEED[args.workload])
    vals, secs = [], []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        r = cpu_baseline(w, budget_s=max(1.0, args.cpu_seconds / max(1, args.steps)),
                         fp8=args.workload == "decode-fp8")
        if i >= args.warmup:
            vals.append(r)
            secs.append(time.perf_counter() - t0)
    value = round(statistics.median(v["value"] for v in vals), 4)
    cb = dict(vals[-1], value=value)
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * statistics.median(secs), 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD_DESC[args.workload] + "; bf16 inputs widened to fp64 by the oracle",
                       "step": "the fp64 oracle (gather through block tables + masked softmax attention) on a "
                               "bounded sample of the batch's sequences"},
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# DRAM bytes per launch of each workload's dominant kernel (dram__bytes_read.sum +
# dram__bytes_write.sum) from one ncu capture, each valid only for the sources
# whose hash is recorded with it (the shared launch path plus the kernels that
# workload runs); reported as null once those sources change.  The captures
# and their commands are summarised under profiles/.
NCU_TRAFFIC = {
    "decode": ("2a08660119772f1a", 613132032 + 4455424),  # dectc_kernel<4>, decode batch
    "prefill": ("2db9b0567d6cce62", 81409024 + 9590784),  # mma_attn_kernel<128>, prefill chunks
    "specverify": ("2db9b0567d6cce62", 1078138624 + 13500928),  # mma_attn_kernel<128>, spec-verify
    "prefix": ("ebbebfeac78de688", 10575872 + 0 + 648673792 + 1372672),  # mma_attn_kernel + dectc_kernel<4>
    "prefix-long": ("2a08660119772f1a", 2116409088 + 4201728),  # dectc_kernel<4>, long-context prefix-shared
    "decode-fp8": ("2a08660119772f1a", 306789888 + 4071168),  # dectc_kernel<4, FP8>, decode batch with FP8 pools
}


def _code_only(text: str) -> str:
    """C/C++ source without comments and blank space (string and character
    literals kept), so that editing a comment leaves the hash unchanged."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


# The sources of the write and attention path: the launch path and plan shared
# by every workload, and the attention kernels each workload runs.  The block
# manager and the block copy are not on it.
FORWARD_SOURCES = ("api.cu", "kv_write.cu", "planner.cu", "static_ws.cu", "pkv_device.cuh", "pkv_tc.cuh",
                   "pkv_internal.h")
WORKLOAD_KERNELS = {"decode": ("decode.cu", "dectc.cu"), "prefix-long": ("decode.cu", "dectc.cu"),
                    "decode-fp8": ("decode.cu", "dectc.cu"),
                    "prefill": ("mma_attn.cu",), "specverify": ("mma_attn.cu",),
                    "prefix": ("decode.cu", "dectc.cu", "mma_attn.cu")}


def _kernel_sources_hash(workload: str) -> str:
    import hashlib
    csrc = os.path.join(os.path.dirname(os.path.abspath(__file__)), "paged_kv_cache_236_gb300", "csrc")
    files = sorted(os.path.join(csrc, f) for f in FORWARD_SOURCES + WORKLOAD_KERNELS[workload])
    h = hashlib.sha256()
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    if workload not in NCU_TRAFFIC or _kernel_sources_hash(workload) != NCU_TRAFFIC[workload][0]:
        return None
    return NCU_TRAFFIC[workload][1]


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(BASE_SEED), default="decode")
    ap.add_argument("--no-mixed", dest="mixed", action="store_false")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)))
        return
    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    res = run_gpu(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
