"""Pins for the fp64 oracle: the pages' worked example, closed forms, a
library routine (torch SDPA on contiguous K/V), invariants the pages imply and
pure-Python brute force.  CPU only.

Each pin is written so that a plausible slip in the oracle (wrong GQA head,
off-by-one causal mask, dropped scale, transposed operand, wrong block/slot
split) breaks at least one of them; ``test_planted_mistakes_are_caught``
plants such slips in the oracle and checks that.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import paged_oracle as po
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example.json")


def rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def unique_id_pool(nb, bs, hkv=1, d=1):
    """Pool whose every slot holds its own id (block * 1000 + slot)."""
    ids = (np.arange(nb)[:, None] * 1000 + np.arange(bs)[None, :]).astype(np.float64)
    return np.broadcast_to(ids[:, :, None, None], (nb, bs, hkv, d)).copy()


def paged_from_contiguous(K, V, bs, nb, perm_seed):
    """Scatter contiguous K/V [L, Hkv, D] into a pool through a random table."""
    L = K.shape[0]
    nblk = (L + bs - 1) // bs
    table = rng(perm_seed).permutation(nb)[:nblk].astype(np.int32)
    kc = np.full((nb, bs) + K.shape[1:], np.nan)
    vc = np.full((nb, bs) + V.shape[1:], np.nan)
    slots = wl.slots_of(table, np.arange(L), bs)
    po.kv_write(K, V, slots, kc, vc)
    return kc, vc, table


def sdpa_reference(q_rows, K, V, scale, causal):
    """torch SDPA (fp64, CPU) on contiguous K/V with an explicit
    bottom-right-aligned causal mask."""
    n, Hq, D = q_rows.shape
    L, Hkv, _ = K.shape
    G = Hq // Hkv
    qt = torch.from_numpy(q_rows).permute(1, 0, 2)[None]                 # [1, Hq, n, D]
    kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(G, 0)[None]
    vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(G, 0)[None]
    i = torch.arange(n)[:, None]
    j = torch.arange(L)[None, :]
    mask = (j <= (L - n + i)) if causal else torch.ones(n, L, dtype=torch.bool)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    return o[0].permute(1, 0, 2).numpy()


# ----------------------------------------------------------------------------
# the pages' worked example
# ----------------------------------------------------------------------------

def test_worked_example_block_translation():
    fx = json.load(open(GOLDEN))
    bs = fx["block_size"]
    pool = unique_id_pool(16, bs)
    for name in ("A", "B"):
        seq = fx[name]
        got = po.gather(pool, np.asarray(seq["block_table"]), seq["num_tokens"])[:, 0, 0]
        want = [b * 1000 + s for b, s in seq["token_block_slot"]]
        assert got.tolist() == want, name
    # B shares physical block 7 with A: its tokens 0..15 are the same pool rows
    a = po.gather(pool, np.asarray(fx["A"]["block_table"]), 16)
    b = po.gather(pool, np.asarray(fx["B"]["block_table"]), 16)
    assert np.array_equal(a, b)
    # block 3 holds A's tokens 16..23 in its first 8 slots only
    used3 = [s for blk, s in fx["A"]["token_block_slot"] if blk == 3]
    assert used3 == list(range(8))


def test_worked_example_write_then_query23():
    """Write A's 24 tokens through the slot mapping, then the query at position
    23 sees exactly tokens 0..23, read from blocks [7, 3]."""
    fx = json.load(open(GOLDEN))
    bs, D = fx["block_size"], 8
    g = rng(3)
    K = g.standard_normal((24, 1, D))
    V = g.standard_normal((24, 1, D))
    q = g.standard_normal((1, 1, D))
    kc = np.full((16, bs, 1, D), np.nan)
    vc = np.full((16, bs, 1, D), np.nan)
    slots = wl.slots_of(np.asarray(fx["A"]["block_table"]), np.arange(24), bs)
    po.kv_write(K, V, slots, kc, vc)
    for t, (blk, s) in enumerate(fx["A"]["token_block_slot"]):
        assert np.array_equal(kc[blk, s], K[t]) and np.array_equal(vc[blk, s], V[t])
    touched = sorted({int(x) // bs for x in slots})
    assert touched == sorted(fx["query"]["physical_blocks_visited"])
    out = po.paged_attention(q, kc, vc, np.asarray([fx["A"]["block_table"]]), [24], [0, 1], 0.3, True)
    want = sdpa_reference(q, K, V, 0.3, True)
    assert np.max(np.abs(out - want)) < 1e-12


def test_tiny_config_reading():
    """The tiny config's block-pressure reading: the chunk fills A's block 3
    slots 8..15 and B's block 12 slots 8..15; the decode tokens go to fresh
    blocks 0 (A) and 1 (B); shared block 7 is common to both tables."""
    w = wl.tiny("1")
    s1, s2 = w.steps
    assert s1.slot_mapping.tolist() == [3 * 16 + i for i in range(8, 16)] + [12 * 16 + i for i in range(8, 16)]
    assert s2.slot_mapping.tolist() == [0 * 16 + 0, 1 * 16 + 0]
    assert s1.block_tables[0, 0] == s1.block_tables[1, 0] == 7
    assert s2.context_lens.tolist() == [33, 49]
    wb = wl.tiny("1b")
    assert wb.step.slot_mapping.tolist() == [3 * 16 + i for i in range(8)] + [12 * 16 + i for i in range(8)]


# ----------------------------------------------------------------------------
# closed forms
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [True, False])
def test_equal_keys_give_mean_of_visible_values(causal):
    g = rng(11)
    n, L, Hq, Hkv, D = 4, 13, 4, 2, 6
    K = np.broadcast_to(g.standard_normal((1, Hkv, D)), (L, Hkv, D)).copy()
    V = g.standard_normal((L, Hkv, D))
    q = g.standard_normal((n, Hq, D))
    out = po.attend(q, K, V, 0.7, causal)
    for h in range(Hq):
        kv = h // (Hq // Hkv)
        for i in range(n):
            cnt = (L - n + i + 1) if causal else L
            np.testing.assert_allclose(out[i, h], V[:cnt, kv].mean(axis=0), rtol=0, atol=1e-13)


def test_constant_values_are_returned_exactly():
    g = rng(12)
    K = g.standard_normal((29, 2, 8))
    V = np.full((29, 2, 8), 0.375)
    out = po.attend(g.standard_normal((5, 6, 8)), K, V, 1.3, True)
    np.testing.assert_allclose(out, 0.375, rtol=0, atol=1e-15)


def test_single_key_returns_its_value():
    g = rng(13)
    K = g.standard_normal((1, 2, 8))
    V = g.standard_normal((1, 2, 8))
    out = po.attend(g.standard_normal((1, 4, 8)), K, V, 0.2, True)
    for h in range(4):
        assert np.array_equal(out[0, h], V[0, h // 2])


def test_zero_query_averages_visible_values():
    g = rng(14)
    K = g.standard_normal((20, 1, 4))
    V = g.standard_normal((20, 1, 4))
    out = po.attend(np.zeros((3, 1, 4)), K, V, 1.0, True)
    for i in range(3):
        np.testing.assert_allclose(out[i, 0], V[: 20 - 3 + i + 1, 0].mean(axis=0), atol=1e-14)


def test_two_keys_logistic_weight():
    """Two visible keys: the weight of key 1 is the logistic function of the
    scaled logit difference."""
    q = np.array([[[0.5, -1.0, 2.0]]])
    K = np.array([[[1.0, 0.0, 0.5]], [[-0.5, 1.0, 0.25]]])
    V = np.array([[[1.0, 0.0, 0.0]], [[0.0, 1.0, 0.0]]])
    scale = 0.9
    z0 = scale * (0.5 * 1.0 + 0.0 + 2.0 * 0.5)
    z1 = scale * (0.5 * -0.5 - 1.0 + 2.0 * 0.25)
    w1 = 1.0 / (1.0 + math.exp(z0 - z1))
    out = po.attend(q, K, V, scale, True)
    np.testing.assert_allclose(out[0, 0], [1 - w1, w1, 0.0], atol=1e-15)


# ----------------------------------------------------------------------------
# library routine: torch SDPA on contiguous K/V
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("causal", [True, False])
def test_paged_equals_contiguous_sdpa(seed, causal):
    g = rng(100 + seed)
    Hkv = int(g.choice([1, 2, 4]))
    G = int(g.choice([1, 2, 4]))
    Hq, D, bs = Hkv * G, int(g.choice([8, 16])), int(g.choice([4, 16]))
    B = 3
    Ls = g.integers(1, 70, size=B)
    ns = np.array([int(g.integers(1, L + 1)) for L in Ls])
    nb = int(sum((L + bs - 1) // bs for L in Ls)) + 5
    kc = np.full((nb, bs, Hkv, D), np.nan)
    vc = np.full((nb, bs, Hkv, D), np.nan)
    perm = g.permutation(nb)
    mb = int(max((L + bs - 1) // bs for L in Ls))
    bt = np.full((B, mb), -1, np.int32)
    cur = 0
    Ks, Vs = [], []
    for s, L in enumerate(Ls):
        k = (L + bs - 1) // bs
        bt[s, :k] = perm[cur:cur + k]
        cur += k
        K = g.standard_normal((L, Hkv, D))
        V = g.standard_normal((L, Hkv, D))
        po.kv_write(K, V, wl.slots_of(bt[s], np.arange(L), bs), kc, vc)
        Ks.append(K)
        Vs.append(V)
    qsl = np.concatenate([[0], np.cumsum(ns)])
    q = g.standard_normal((int(qsl[-1]), Hq, D))
    scale = float(g.uniform(0.05, 1.0))
    out = po.paged_attention(q, kc, vc, bt, Ls, qsl, scale, causal)
    for s in range(B):
        want = sdpa_reference(q[qsl[s]:qsl[s + 1]], Ks[s], Vs[s], scale, causal)
        assert np.max(np.abs(out[qsl[s]:qsl[s + 1]] - want)) < 1e-12


# ----------------------------------------------------------------------------
# invariants the pages imply
# ----------------------------------------------------------------------------

def _relabel(w: wl.Workload, seed: int):
    """The same workload with physical block ids permuted (pool rows moved)."""
    perm = rng(seed).permutation(w.num_blocks)          # old id -> new id
    kc = np.empty_like(w.k_cache)
    vc = np.empty_like(w.v_cache)
    kc[perm] = w.k_cache
    vc[perm] = w.v_cache
    st = w.step
    bt = np.where(st.block_tables >= 0, perm[np.maximum(st.block_tables, 0)], -1).astype(np.int32)
    bs = w.block_size
    sm = np.where(st.slot_mapping >= 0,
                  perm[st.slot_mapping // bs] * bs + st.slot_mapping % bs, -1)
    return kc, vc, bt, sm


def _run_oracle(w, kc, vc, bt, sm):
    st = w.step
    kc, vc = kc.copy(), vc.copy()
    po.kv_write(st.k_new, st.v_new, sm, kc, vc)
    f = lambda a: wl.to_f64(a, w.dtype)
    return po.paged_attention(f(st.q), f(kc), f(vc), bt, st.context_lens, st.query_start_loc,
                              w.scale, w.causal)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_block_id_permutation_invariance(seed):
    w = wl.random_small(seed, dtype="f32", head_dim=16, batch=4, max_ctx=90, max_q=9)
    base = _run_oracle(w, w.k_cache, w.v_cache, w.step.block_tables, w.step.slot_mapping)
    kc, vc, bt, sm = _relabel(w, seed + 50)
    again = _run_oracle(w, kc, vc, bt, sm)
    assert np.array_equal(base, again)


def test_private_copy_of_shared_blocks_is_identical():
    w = wl.build("shared", context_lens=[40, 37, 52], q_lens=[1, 3, 2], num_blocks=40,
                 block_size=8, num_q_heads=4, num_kv_heads=2, head_dim=8, dtype="f32",
                 seed=5, shared_prefix_tokens=16)
    st = w.step
    assert (st.block_tables[:, :2] == st.block_tables[0, :2]).all()
    base = _run_oracle(w, w.k_cache, w.v_cache, st.block_tables, st.slot_mapping)
    # give sequences 1 and 2 their own copies of the two shared blocks
    kc, vc, bt = w.k_cache.copy(), w.v_cache.copy(), st.block_tables.copy()
    used = set(bt[bt >= 0].tolist()) | set((st.slot_mapping // 8).tolist())
    free = [b for b in range(w.num_blocks) if b not in used]
    for s in (1, 2):
        for j in range(2):
            nbid = free.pop()
            kc[nbid], vc[nbid] = kc[bt[s, j]], vc[bt[s, j]]
            bt[s, j] = nbid
    again = _run_oracle(w, kc, vc, bt, st.slot_mapping)
    assert np.array_equal(base, again)


def test_chunk_then_decode_equals_one_call():
    """Prefill and decode share one call: a sequence's n queries attended at
    once equal the first n-1 attended with context L-1 followed by the last
    one attended with context L."""
    g = rng(21)
    L, n, Hq, Hkv, D = 45, 6, 4, 2, 8
    K = g.standard_normal((L, Hkv, D))
    V = g.standard_normal((L, Hkv, D))
    q = g.standard_normal((n, Hq, D))
    full = po.attend(q, K, V, 0.4, True)
    first = po.attend(q[:-1], K[:-1], V[:-1], 0.4, True)
    last = po.attend(q[-1:], K, V, 0.4, True)
    np.testing.assert_allclose(full, np.concatenate([first, last]), rtol=0, atol=1e-13)


@pytest.mark.parametrize("splits", [1, 2, 3, 5, 17])
@pytest.mark.parametrize("causal", [True, False])
def test_split_merge_equals_unsplit(splits, causal):
    g = rng(30 + splits)
    L, n, Hq, Hkv, D = 80, 7, 6, 3, 8
    K = g.standard_normal((L, Hkv, D))
    V = g.standard_normal((L, Hkv, D))
    q = g.standard_normal((n, Hq, D))
    edges = np.linspace(0, L, splits + 1).round().astype(int)
    parts = [po.partial_attend(q, K, V, 0.5, causal, a, b) for a, b in zip(edges[:-1], edges[1:])]
    got = po.merge_partials(parts)
    want = po.attend(q, K, V, 0.5, causal)
    assert np.max(np.abs(got - want)) < 1e-12


# ----------------------------------------------------------------------------
# pure-Python brute force on tiny inputs
# ----------------------------------------------------------------------------

def brute_force(q, kc, vc, bt, ctx, qsl, scale, causal):
    """Scalar loops, lists and math.exp only."""
    q, kc, vc = q.tolist(), kc.tolist(), vc.tolist()
    T, Hq, D = len(q), len(q[0]), len(q[0][0])
    Hkv, bs = len(kc[0][0]), len(kc[0])
    out = [[[0.0] * D for _ in range(Hq)] for _ in range(T)]
    for s in range(len(ctx)):
        L, a, b = int(ctx[s]), int(qsl[s]), int(qsl[s + 1])
        n = b - a
        for i in range(n):
            for h in range(Hq):
                kvh = h * Hkv // Hq
                last = (L - n + i) if causal else (L - 1)
                logits = []
                for j in range(last + 1):
                    blk, off = int(bt[s][j // bs]), j % bs
                    logits.append(scale * sum(q[a + i][h][d] * kc[blk][off][kvh][d] for d in range(D)))
                mx = max(logits)
                ws = [math.exp(z - mx) for z in logits]
                tot = sum(ws)
                for d in range(D):
                    acc = 0.0
                    for j, wgt in enumerate(ws):
                        blk, off = int(bt[s][j // bs]), j % bs
                        acc += wgt * vc[blk][off][kvh][d]
                    out[a + i][h][d] = acc / tot
    return np.asarray(out)


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("causal", [True, False])
def test_brute_force_tiny(seed, causal):
    w = wl.random_small(seed, dtype="f32", batch=3, max_ctx=40, max_q=6, num_q_heads=4,
                        num_kv_heads=2, head_dim=8, block_size=4, causal=causal)
    st = w.step
    kc, vc = w.k_cache.astype(np.float64), w.v_cache.astype(np.float64)
    po.kv_write(st.k_new, st.v_new, st.slot_mapping, kc, vc)
    got = po.paged_attention(st.q.astype(np.float64), kc, vc, st.block_tables, st.context_lens,
                             st.query_start_loc, w.scale, causal)
    want = brute_force(st.q.astype(np.float64), kc, vc, st.block_tables, st.context_lens,
                       st.query_start_loc, w.scale, causal)
    assert np.max(np.abs(got - want)) < 1e-12


def test_write_skips_negative_slots_and_is_a_copy():
    kc = np.zeros((3, 4, 1, 2), np.uint16)
    vc = np.zeros((3, 4, 1, 2), np.uint16)
    k = np.arange(8, dtype=np.uint16).reshape(4, 1, 2) + 100
    v = k + 50
    po.kv_write(k, v, np.array([5, -1, 0, 11]), kc, vc)
    assert kc[1, 1].tolist() == [[100, 101]] and kc[0, 0].tolist() == [[104, 105]]
    assert kc[2, 3].tolist() == [[106, 107]] and vc[2, 3].tolist() == [[156, 157]]
    assert int((kc != 0).sum()) == 6


# ----------------------------------------------------------------------------
# planted mistakes must be caught by the pins above
# ----------------------------------------------------------------------------

def _pins_pass():
    try:
        test_worked_example_write_then_query23()
        for s in range(2):
            for c in (True, False):
                test_paged_equals_contiguous_sdpa(s, c)
                test_brute_force_tiny(s, c)
        test_equal_keys_give_mean_of_visible_values(True)
        test_two_keys_logistic_weight()
    except AssertionError:
        return False
    return True


def test_planted_mistakes_are_caught(monkeypatch):
    assert _pins_pass()
    mutations = {
        "gqa head modulo": ("kv_head_of", lambda h, hq, hkv: h % hkv),
        "mask off by one": ("visible_keys", lambda i, n, L, c: (L - n + i) if c else L),
        "mask not bottom-right": ("visible_keys", lambda i, n, L, c: (i + 1) if c else L),
    }
    for name, (attr, fn) in mutations.items():
        with monkeypatch.context() as m:
            m.setattr(po, attr, fn)
            assert not _pins_pass(), name
    orig_attend = po.attend

    def no_scale(q, K, V, scale, causal):
        return orig_attend(q, K, V, 1.0, causal)

    def transposed_gather(cache, table, L):
        bs = cache.shape[1]
        pos = np.arange(int(L))
        return cache[np.asarray(table)[pos % bs % len(table)], pos // bs]

    for name, (attr, fn) in {"dropped scale": ("attend", no_scale),
                             "block/slot swapped": ("gather", transposed_gather)}.items():
        with monkeypatch.context() as m:
            m.setattr(po, attr, fn)
            assert not _pins_pass(), name
