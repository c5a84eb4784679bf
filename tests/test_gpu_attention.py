"""paged_attention_forward on the GPU against the fp64 oracle: the pages'
worked example (tiny fp32 config), ragged random batches over the supported
shapes, edge cases and invalid metadata."""
import numpy as np
import pytest
import torch

import paged_kv_cache_236_gb300 as pkv
import workloads as wl
from gpu_util import DeviceWorkload, check_step, to_dev, to_f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("case", ["1", "1b"])
def test_tiny_worked_example(case):
    """Block tables [7, 3] and [7, 9, 12] sharing block 7; an 8-token causal
    chunk, then (case 1) a 1-token decode into freshly allocated blocks."""
    dw = DeviceWorkload(wl.tiny(case, poison=True))
    for i in range(len(dw.w.steps)):
        out = dw.run_step(i)
        check_step(dw, out, i, what=f"tiny-{case} step {i}")
    assert pkv.device_errors() == 0


CASES = []
for dtype in ("bf16", "f32"):
    for D in (64, 128):
        for bs in (8, 16, 32, 64):
            for (hq, hkv) in ((8, 2), (4, 4), (8, 1), (16, 2)):
                CASES.append((dtype, D, bs, hq, hkv))


@pytest.mark.parametrize("dtype,D,bs,hq,hkv", CASES)
def test_random_batches(dtype, D, bs, hq, hkv):
    seed = 500 + CASES.index((dtype, D, bs, hq, hkv))
    w = wl.random_small(seed, dtype=dtype, batch=5, max_ctx=300, max_q=12, num_q_heads=hq, num_kv_heads=hkv,
                        head_dim=D, block_size=bs, poison=True)
    dw = DeviceWorkload(w)
    out = dw.run_step(0)
    check_step(dw, out, what=f"{dtype} D{D} bs{bs} {hq}/{hkv}")
    assert pkv.device_errors() == 0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_non_causal(dtype):
    w = wl.random_small(77, dtype=dtype, batch=4, max_ctx=150, max_q=9, causal=False)
    dw = DeviceWorkload(w)
    check_step(dw, dw.run_step(0), what="non-causal")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_prefill_chunks_multi_tile(dtype):
    """Longer causal chunks spanning many 128-row and 128-key tiles with a
    ragged tail."""
    w = wl.build("chunks", context_lens=[700, 333, 129, 1000], q_lens=[300, 333, 17, 1], num_blocks=200,
                 block_size=16, num_q_heads=8, num_kv_heads=2, head_dim=128, dtype=dtype, seed=31, poison=True)
    dw = DeviceWorkload(w)
    check_step(dw, dw.run_step(0), what="chunks")


def test_edge_cases_empty_and_single():
    """Sequences with no queries, a single-token context, contexts ending
    exactly on a block boundary, and a batch that is entirely empty."""
    w = wl.build("edges", context_lens=[1, 16, 17, 32, 5, 64], q_lens=[1, 0, 3, 1, 0, 16], num_blocks=40,
                 block_size=16, num_q_heads=8, num_kv_heads=2, head_dim=128, dtype="bf16", seed=3, poison=True)
    dw = DeviceWorkload(w)
    check_step(dw, dw.run_step(0), what="edges")
    # T == 0: nothing to do, must not fail
    q = torch.empty(0, 8, 128, dtype=torch.bfloat16, device="cuda")
    out = pkv.paged_attention_forward(q, dw.kc, dw.vc, torch.zeros(2, 1, dtype=torch.int32, device="cuda"),
                                      torch.zeros(2, dtype=torch.int32, device="cuda"),
                                      torch.zeros(3, dtype=torch.int32, device="cuda"), 0.1, True)
    assert out.shape == (0, 8, 128)
    assert pkv.device_errors() == 0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_long_context_split_kv(dtype):
    """One decode token over 20000 keys and a few short ones: the long one is
    split across many CTAs and merged; a minimum workspace (no room for
    partial rows, so no splits) gives the same rows within tolerance."""
    w = wl.build("long", context_lens=[20000, 100, 3000], q_lens=[1, 1, 2], num_blocks=1600, block_size=16,
                 num_q_heads=8, num_kv_heads=2, head_dim=128, dtype=dtype, seed=8, poison=True)
    dw = DeviceWorkload(w)
    out = dw.run_step(0)
    check_step(dw, out, what="split")
    st = w.step
    t = dw.step_tensors(st)
    ws = torch.empty(pkv.workspace_min(3, st.num_tokens, 8, 2, 128), dtype=torch.uint8, device="cuda")
    out2 = pkv.paged_attention_forward(t["q"], dw.kc, dw.vc, t["bt"], t["ctx"], t["qsl"], w.scale, True,
                                       workspace=ws)
    check_step(dw, out2, what="no-split")


def test_block_permutation_is_bit_identical():
    """Relabelling physical blocks (moving pool rows accordingly) changes no
    output bit: the kernels reduce in logical order."""
    w = wl.random_small(12, dtype="bf16", batch=6, max_ctx=400, max_q=10, poison=True)
    dw = DeviceWorkload(w)
    out = dw.run_step(0)
    perm = np.random.Generator(np.random.PCG64(4)).permutation(w.num_blocks)
    kc = torch.empty_like(dw.kc)
    vc = torch.empty_like(dw.vc)
    pt = torch.from_numpy(perm).cuda()
    kc[pt] = dw.kc
    vc[pt] = dw.vc
    st = w.step
    bt = np.where(st.block_tables >= 0, perm[np.maximum(st.block_tables, 0)], -1).astype(np.int32)
    t = dw.step_tensors(st)
    out2 = pkv.paged_attention_forward(t["q"], kc, vc, torch.from_numpy(bt).cuda(), t["ctx"], t["qsl"], w.scale,
                                       True)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


def test_invalid_metadata_is_flagged_and_zeroed():
    """A sequence with more queries than tokens and one whose table names a
    block outside the pool: no fault, both raise device error bits; the
    first's rows are zero, the second reads that block as a block of zeros
    (its rows equal the oracle's over a pool where the entry names an all-zero
    block), and the valid sequence is still right."""
    w = wl.build("bad", context_lens=[40, 30, 50], q_lens=[2, 1, 1], num_blocks=12, block_size=16,
                 num_q_heads=4, num_kv_heads=2, head_dim=128, dtype="bf16", seed=2, poison=False)
    dw = DeviceWorkload(w)
    st = w.step
    t = dw.step_tensors(st)
    pkv.paged_kv_write(t["k"], t["v"], t["slots"], dw.kc, dw.vc)
    ctx = t["ctx"].clone()
    ctx[0] = 1                       # 2 queries but 1 token
    bt = t["bt"].clone()
    bt[1, 1] = 10_000                # outside the pool
    pkv.device_errors(clear=True)
    out = pkv.paged_attention_forward(t["q"], dw.kc, dw.vc, bt, ctx, t["qsl"], w.scale, True)
    flags = pkv.device_errors(clear=True)
    assert flags & pkv.DEVERR["bad_sequence"] and flags & pkv.DEVERR["block_out_of_range"]
    o = to_f64(out)
    assert np.all(o[0:2] == 0)
    assert np.all(np.isfinite(o))
    from oracle import paged_oracle as po
    po.kv_write(st.k_new, st.v_new, st.slot_mapping, dw.kc_host, dw.vc_host)
    rows = dw.oracle_rows(0, [2])
    a, b, ref = rows[2]
    from gpu_util import check_close
    check_close(o[a:b], ref, "bf16", "valid sequence next to bad ones")
    # sequence 1: its second block reads as zeros; the oracle sees a pool with
    # one extra all-zero block that the corrupted entry names
    zk = np.concatenate([dw.kc_host, np.zeros_like(dw.kc_host[:1])])
    zv = np.concatenate([dw.vc_host, np.zeros_like(dw.vc_host[:1])])
    bt1 = st.block_tables[1].copy()
    bt1[1] = w.num_blocks
    L1 = int(st.context_lens[1])
    a1, b1 = int(st.query_start_loc[1]), int(st.query_start_loc[2])
    K = wl.to_f64(po.gather(zk, bt1, L1), "bf16")
    V = wl.to_f64(po.gather(zv, bt1, L1), "bf16")
    ref1 = po.attend(wl.to_f64(st.q[a1:b1], "bf16"), K, V, w.scale, True)
    check_close(o[a1:b1], ref1, "bf16", "sequence with an out-of-pool block id")


def test_host_side_errors():
    q = torch.zeros(4, 6, 128, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(4, 16, 4, 128, dtype=torch.bfloat16, device="cuda")
    i32 = lambda *s: torch.zeros(*s, dtype=torch.int32, device="cuda")
    with pytest.raises(pkv.LibraryError) as e:
        pkv.paged_attention_forward(q, kc, kc, i32(1, 1), i32(1), i32(2), 0.1, True)
    assert "num_kv_heads" in str(e.value)
    q = torch.zeros(4, 8, 96, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(4, 16, 4, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pkv.LibraryError) as e:
        pkv.paged_attention_forward(q, kc, kc, i32(1, 1), i32(1), i32(2), 0.1, True)
    assert e.value.status == 2
    with pytest.raises(ValueError):
        pkv.paged_attention_forward(q.cpu(), kc, kc, i32(1, 1), i32(1), i32(2), 0.1, True)


@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 4), (8, 2), (16, 2), (32, 2)])
@pytest.mark.parametrize("max_q", [1, 2])
def test_decode_with_length_hint(hq, hkv, max_q):
    """Decode-shaped batches (1-2 query tokens) with the host's max_query_len
    hint, which selects the narrower per-key row counts (4, 8) of the
    decode kernel; also a long context to exercise its split merge."""
    g = np.random.Generator(np.random.PCG64(hq * 10 + hkv + max_q))
    B = 7
    L = np.concatenate([[5000], g.integers(1, 700, size=B - 1)])
    n = np.minimum(L, g.integers(1, max_q, size=B, endpoint=True))
    nb = int(np.sum((L + 15) // 16)) + 3
    w = wl.build("hint", context_lens=L, q_lens=n, num_blocks=nb, block_size=16, num_q_heads=hq,
                 num_kv_heads=hkv, head_dim=128, dtype="bf16", seed=hq + 3 * max_q, poison=True)
    dw = DeviceWorkload(w)
    out = dw.run_step(0, max_query_len=int(n.max()))
    check_step(dw, out, what=f"hint {hq}/{hkv} q<={max_q}")
    assert pkv.device_errors() == 0


# GQA groups that are not powers of two (3, 5, 6, 7) and large groups (32,
# 64): decode over a long split context, a speculative-verify window of 5
# tokens, a 300-token prefill chunk and short ragged sequences in one batch.
GQA_GROUPS = [(12, 4), (10, 2), (6, 1), (14, 2), (32, 1), (64, 1)]
GQA_CASES = [(dt, D, hq, hkv) for (hq, hkv) in GQA_GROUPS for (dt, D) in (("bf16", 128), ("bf16", 64), ("f32", 128))]


def _gqa_workload(dtype, D, hq, hkv, seed):
    L = [6000, 3000, 700, 40, 17, 1]
    n = [1, 5, 300, 1, 2, 1]
    nb = sum(-(-x // 16) for x in L) + 5
    return wl.build(f"gqa-{hq}-{hkv}", context_lens=L, q_lens=n, num_blocks=nb, block_size=16, num_q_heads=hq,
                    num_kv_heads=hkv, head_dim=D, dtype=dtype, seed=seed, poison=True)


@pytest.mark.parametrize("dtype,D,hq,hkv", GQA_CASES)
def test_gqa_groups(dtype, D, hq, hkv):
    w = _gqa_workload(dtype, D, hq, hkv, 900 + GQA_CASES.index((dtype, D, hq, hkv)))
    dw = DeviceWorkload(w)
    out = dw.run_step(0)
    check_step(dw, out, what=f"{dtype} D{D} G{hq // hkv}")
    # the same batch with the query-length hint (kernel choice by rows)
    st = w.step
    t = dw.step_tensors(st)
    out2 = pkv.paged_attention_forward(t["q"], dw.kc, dw.vc, t["bt"], t["ctx"], t["qsl"], w.scale, True,
                                       max_query_len=int(st.q_lens.max()))
    torch.cuda.synchronize()
    check_step(dw, out2, what=f"{dtype} D{D} G{hq // hkv}, length hint")
    assert pkv.device_errors() == 0


@pytest.mark.parametrize("hq,hkv", GQA_GROUPS)
def test_gqa_groups_fp8(hq, hkv):
    from test_gpu_fp8 import Fp8Run
    w = _gqa_workload("bf16", 128, hq, hkv, 950 + GQA_GROUPS.index((hq, hkv)))
    run = Fp8Run(w, 0.02, 0.015)
    run.check(run.step(), what=f"fp8 G{hq // hkv}")
    assert pkv.device_errors() == 0


def test_back_to_back_calls_share_the_cached_workspace():
    """Mixed batches forwarded back to back on one stream, with the default
    cached workspace and no host synchronisation between the calls: the
    tensor-core kernel of one call runs beside its decode kernel, and the next
    call's planner must not rewrite the shared plan while it still reads it.
    Every call's rows are checked against the oracle afterwards."""
    mk = lambda name, seed, L, n: wl.build(name, context_lens=L, q_lens=n, num_blocks=sum(-(-x // 16) for x in L) + 4,
                                           block_size=16, num_q_heads=16, num_kv_heads=4, head_dim=128,
                                           dtype="bf16", seed=seed, poison=True)
    # a: long prefill chunks (tensor-core work dominates) beside short decodes
    wa = mk("b2b-a", 61, [3000, 2600] + [150 + 37 * i for i in range(24)], [1024, 900] + [1] * 24)
    # b: long decodes beside a short chunk
    wb = mk("b2b-b", 62, [7000, 5000, 900] + [4000 - 101 * i for i in range(20)], [1, 1, 200] + [1] * 20)
    dws = [DeviceWorkload(wa), DeviceWorkload(wb)]
    ts = []
    for dw in dws:
        st = dw.w.step
        t = dw.step_tensors(st)
        pkv.paged_kv_write(t["k"], t["v"], t["slots"], dw.kc, dw.vc)
        po_write(dw, st)
        ts.append(t)
    torch.cuda.synchronize()
    outs = []
    for rep in range(3):
        for i, dw in enumerate(dws):
            t = ts[i]
            outs.append((i, pkv.paged_attention_forward(t["q"], dw.kc, dw.vc, t["bt"], t["ctx"], t["qsl"],
                                                        dw.w.scale, True)))
    torch.cuda.synchronize()
    for k, (i, out) in enumerate(outs):
        check_step(dws[i], out, what=f"call {k} (batch {'ab'[i]})")
    assert pkv.device_errors() == 0


def po_write(dw, st):
    from oracle import paged_oracle as po
    po.kv_write(st.k_new, st.v_new, st.slot_mapping, dw.kc_host, dw.vc_host)
