"""The library's C++ block manager against the reference model
(oracle/block_manager.py), call by call on the same seeded operation
streams: slots, block tables, context lengths, query offsets, copy-on-write
pairs, prefix hits, refusals and block counts must be identical (bit-exact
integer work), and every live sequence's K/V read through its C++ block
table must be its logical rows.  Host code only: no GPU needed.

Also the host-side argument checks of paged_kv_copy_blocks (rejected before
any launch) and the edge cases of the manager's C ABI."""
import numpy as np
import pytest

from oracle.block_manager import BlockManagerModel, OutOfBlocks as ModelOOB
from tests.block_util import Driver
from workloads.block_ops import op_stream


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_236_gb300 import build
    build.build()
    import paged_kv_cache_236_gb300 as p
    return p


def run_pair(pkv, seed, nb, bs, max_tokens, n_ops, check=True, **kw):
    mb = -(-max_tokens // bs)
    dm = Driver(BlockManagerModel(nb, bs, mb), nb, bs, ModelOOB, pool=False)
    dc = Driver(pkv.BlockManager(nb, bs, mb), nb, bs, pkv.OutOfBlocks, pool=check)
    gm = op_stream(seed, n_ops, bs, max_tokens=max_tokens, **kw)
    gc = op_stream(seed, n_ops, bs, max_tokens=max_tokens, **kw)
    om, oc = next(gm), next(gc)
    i = 0
    while True:
        assert om == oc
        okm, okc = dm.apply(om), dc.apply(oc)
        assert okm == okc, (i, om[0])
        assert dm.log[-1] == dc.log[-1], (i, om[0], dm.log[-1], dc.log[-1])
        assert dm.mgr.stats() == dc.mgr.stats(), i
        if check:
            dc.check_content()
        i += 1
        try:
            om, oc = gm.send(okm), gc.send(okc)
        except StopIteration:
            break
    for s in dm.tokens:
        assert dm.mgr.block_table(s) == dc.mgr.block_table(s)
    return dm, dc


@pytest.mark.parametrize("seed,nb,bs,max_tokens", [
    (1, 400, 4, 60), (2, 40, 4, 48), (3, 24, 2, 30), (4, 64, 8, 96), (5, 18, 4, 40),
    (6, 30, 16, 128), (7, 12, 1, 11), (8, 200, 32, 512)])
def test_cpp_matches_model(pkv, seed, nb, bs, max_tokens):
    run_pair(pkv, seed, nb, bs, max_tokens, 400)


def test_cpp_matches_model_long_stream(pkv):
    """A longer stream under pressure (evictions, refusals, many forks)."""
    run_pair(pkv, 99, 60, 4, 64, 3000, check=False, max_live=20, p_fork=0.12)


def test_edge_cases(pkv):
    m, ref = pkv.BlockManager(8, 4, 3), BlockManagerModel(8, 4, 3)
    # a sequence exactly max_blocks_per_seq blocks long, then one token more
    for mm in (m, ref):
        slots, copies = mm.update(1, 12)
        assert list(slots) == list(range(12)) and len(copies) == 0
    with pytest.raises(pkv.LibraryError):
        m.update(1, 1)
    assert m.block_table(1) == ref.block_table(1) == [0, 1, 2]
    # zero-token update creates an empty sequence; an empty step is a no-op
    m.update(2, 0)
    assert m.block_table(2) == [] and m.num_tokens(2) == 0
    meta = m.step([], [])
    assert meta["query_start_loc"].tolist() == [0] and meta["slot_mapping"].size == 0
    # a step with a zero-token member and a fresh sequence
    meta = m.step([2, 3], [0, 5])
    assert meta["context_lens"].tolist() == [0, 5] and meta["query_start_loc"].tolist() == [0, 0, 5]
    assert meta["block_tables"][0].tolist() == [-1, -1, -1]
    # refusals leave everything as it was
    before = m.stats()
    for bad in (lambda: m.free(77), lambda: m.fork(77, 78), lambda: m.fork(1, 3), lambda: m.step([1, 1], [0, 0]),
                lambda: m.add_prefix(1, [0] * 11), lambda: m.try_get_prefix_blocks(1, [0] * 5),
                lambda: m.step([3, 1], [1, 1]), lambda: m.update(4, 13)):
        with pytest.raises(pkv.LibraryError):
            bad()
        assert m.stats() == before
    with pytest.raises(pkv.OutOfBlocks):
        m.step([4, 5], [8, 8])              # 4 blocks, 3 free
    assert m.stats() == before
    # pool exhaustion exactly: the last free blocks can be taken
    m.step([4], [12])
    assert m.stats()["free"] == 0
    with pytest.raises(pkv.OutOfBlocks):
        m.update(6, 1)


def test_copy_on_write_pairs(pkv):
    """Forked sequences sharing a partly filled block: the first to append
    copies it, the next finds it unshared (reading B5 / policy P4)."""
    m = pkv.BlockManager(16, 4, 8)
    m.update(1, 6)                           # blocks [0, 1], block 1 half full
    m.fork(1, 2)
    m.fork(1, 3)
    meta = m.step([2, 3, 1], [1, 1, 1])
    assert meta["copies"].tolist() == [[1, 2], [1, 3]]
    assert meta["block_tables"][:, :2].tolist() == [[0, 2], [0, 3], [0, 1]]
    assert meta["slot_mapping"].tolist() == [2 * 4 + 2, 3 * 4 + 2, 1 * 4 + 2]
    # full shared blocks are never copied
    m.update(4, 8)
    m.fork(4, 5)
    slots, copies = m.update(5, 1)
    assert len(copies) == 0 and m.block_table(5)[:2] == m.block_table(4)


def test_copy_blocks_host_checks(pkv):
    """paged_kv_copy_blocks rejects bad pairs on the host, before any launch."""
    L = pkv.lib()
    pairs = np.asarray([[0, 1], [2, 3]], dtype=np.int32)
    call = lambda p, n, nb=8, layers=1, stride=0: L.paged_kv_copy_blocks(8, 8, p.ctypes.data, n, layers, stride, nb,
                                                                         16, 4, 128, 1, None)
    assert call(pairs, 0) == 0                                           # nothing to do
    assert call(np.asarray([[0, 8]], dtype=np.int32), 1) == 1            # outside the pool
    assert call(np.asarray([[-1, 2]], dtype=np.int32), 1) == 1
    assert call(np.asarray([[0, 2], [1, 2]], dtype=np.int32), 2) == 1    # a destination twice
    assert call(np.asarray([[0, 2], [2, 3]], dtype=np.int32), 2) == 1    # a destination that is a source
    assert call(pairs, 2, layers=2, stride=100) == 1                     # layer stride below one pool
    assert L.paged_kv_copy_blocks(8, 8, pairs.ctypes.data, 2, 1, 0, 8, 16, 4, 128, 7, None) == 2  # dtype
    assert L.paged_kv_copy_blocks(None, None, pairs.ctypes.data, 2, 1, 0, 8, 16, 4, 128, 1, None) == 1


def test_large_pool_is_fast(pkv):
    """A 200 000-block pool and 512 sequences stepping one token: host cost
    per step stays small (O(batch), not O(pool))."""
    import time
    m = pkv.BlockManager(200000, 16, 512)
    ids = list(range(512))
    m.step(ids, [1000] * 512)
    t0 = time.perf_counter()
    for _ in range(50):
        m.step(ids, [1] * 512)
    dt = (time.perf_counter() - t0) / 50
    assert dt < 0.05, dt


def test_step_with_reused_buffers_matches(pkv):
    """step(..., reuse=True) returns the same metadata (views into buffers
    the manager keeps, grown as batches grow)."""
    a, b = pkv.BlockManager(3000, 16, 64), pkv.BlockManager(3000, 16, 64)
    rng = np.random.default_rng(3)
    live = []
    for it in range(60):
        new = [1000 + it] if rng.random() < 0.5 or not live else []
        live += new
        ids = np.asarray(sorted(rng.choice(live, size=min(len(live), int(rng.integers(1, 40))), replace=False)),
                         dtype=np.int64)
        n = rng.integers(0, 40, size=len(ids)).astype(np.int32)
        ra, rb = a.step(ids, n), b.step(ids, n, reuse=True)
        for k in ra:
            assert np.array_equal(ra[k], rb[k]), (it, k)
        if it % 7 == 3 and len(live) > 3:
            s = live.pop(int(rng.integers(0, len(live))))
            a.free(s)
            b.free(s)
