"""Pins of the block manager's reference model (oracle/block_manager.py) to
what the pages and plain counting fix, with no implementation to compare to:

* the worked example of "Paged Attention 基础", section 2 (24 tokens in
  blocks of 16: the second block holds 8 live slots; a second sequence with
  the same first 16 tokens names the same first block and its own second);
* K/V content: after every operation of long seeded streams (prompts with
  shared system prompts, chunked and single-token steps, forks, frees,
  prefix registration, eviction under pressure), gathering each live
  sequence through its block table gives exactly its logical rows;
* accounting: every block is free, idle-cached or in use, and a block's
  count equals the number of table entries naming it;
* brute force: with no eviction, the tokens a prompt finds cached equal the
  longest full-block prefix it shares with any registered token list, capped
  to leave one token;
* all or nothing: a refused update changes nothing;
* planted mistakes in a copy of the model (copy-on-write skipped, an
  evicted entry kept, a shared block released to the free list) are caught.
"""
import copy

import numpy as np
import pytest

from oracle.block_manager import BlockManagerModel, OutOfBlocks
from tests.block_util import WIDTH, Driver
from workloads.block_ops import kv_rows, op_stream


def check_accounting(m: BlockManagerModel) -> None:
    count = [0] * m.num_blocks
    for table in m.tables.values():
        for b in table:
            count[b] += 1
    assert count == m.ref
    in_use = {b for b in range(m.num_blocks) if m.ref[b] > 0}
    free, idle = set(m.free_list), set(m.idle)
    assert len(free) == len(m.free_list) and len(idle) == len(m.idle)
    assert not (free & idle) and not (free & in_use) and not (idle & in_use)
    assert free | idle | in_use == set(range(m.num_blocks))
    assert idle <= set(m.entry_of_block) and not (free & set(m.entry_of_block))
    for key, (eid, b) in m.entries.items():
        assert m.entry_of_block[b] == (key, eid)
    assert len(m.entries) == len(m.entry_of_block)
    for s, table in m.tables.items():
        assert len(table) == -(-m.lens[s] // m.block_size)


def run_checked(m, seed, n_ops, **kw):
    d = Driver(m, m.num_blocks, m.block_size, OutOfBlocks)
    g = op_stream(seed, n_ops, m.block_size, **kw)
    op = next(g)
    refused = 0
    while True:
        ok = d.apply(op)
        refused += not ok
        d.check_content()
        check_accounting(m)
        try:
            op = g.send(ok)
        except StopIteration:
            break
    return d, refused


def test_worked_example_structure():
    """Sequence A: 24 tokens in blocks of 16 -> two blocks, the second with
    8 live slots; B shares A's first 16 tokens and names the same block."""
    m = BlockManagerModel(num_blocks=10, block_size=16, max_blocks_per_seq=4)
    a = list(range(100, 124))
    slots, copies = m.update(1, 24)
    assert copies == []
    ta = m.block_table(1)
    assert len(ta) == 2 and ta[0] != ta[1]
    assert slots == [ta[p // 16] * 16 + p % 16 for p in range(24)]
    assert [s // 16 for s in slots].count(ta[1]) == 8            # block "3": first 8 slots
    assert [s % 16 for s in slots if s // 16 == ta[1]] == list(range(8))
    m.add_prefix(1, a)
    b = a[:16] + list(range(500, 508))
    assert m.try_get_prefix_blocks(2, b) == 16                   # block "7" found
    slots_b, copies_b = m.update(2, 8)
    tb = m.block_table(2)
    assert tb[0] == ta[0] and tb[1] not in ta and copies_b == []
    assert m.ref[ta[0]] == 2 and m.ref[ta[1]] == 1 and m.ref[tb[1]] == 1
    # the content both sequences see through their tables
    pool = np.full((10, 16, 1, WIDTH), np.nan)
    ra, rb = kv_rows(a, WIDTH), kv_rows(b, WIDTH)
    from oracle import paged_oracle as po
    scratch = np.empty_like(pool)
    po.kv_write(ra[:, None], ra[:, None], np.asarray(slots), pool, scratch)
    po.kv_write(rb[16:, None], rb[16:, None], np.asarray(slots_b), pool, scratch)
    assert np.array_equal(po.gather(pool, ta, 24)[:, 0], ra)
    assert np.array_equal(po.gather(pool, tb, 24)[:, 0], rb)
    # B's first 16 rows were never written for B: they are A's, read through block "7"
    m.free(1)
    assert m.ref[ta[0]] == 1 and m.stats()["in_use"] == 2
    m.free(2)
    # A's first block stays cached (idle); the two unregistered blocks are free
    assert m.stats() == {"free": 9, "idle": 1, "in_use": 0, "cached": 1}


@pytest.mark.parametrize("seed,nb,bs,max_tokens", [(1, 400, 4, 60), (2, 40, 4, 48), (3, 24, 2, 30),
                                                     (4, 64, 8, 96), (5, 18, 4, 40)])
def test_content_and_accounting_over_streams(seed, nb, bs, max_tokens):
    m = BlockManagerModel(nb, bs, max_blocks_per_seq=-(-max_tokens // bs))
    run_checked(m, seed, 400, max_tokens=max_tokens)


def test_streams_exercise_every_path():
    """The stream parameters above reach copy-on-write, prefix hits,
    eviction and refusal (so the content pin covers them)."""
    seen = {"cow": 0, "hit": 0, "evict": 0, "oob": 0}

    class Spy(BlockManagerModel):
        def _take(self):
            if not self.free_list and self.idle:
                seen["evict"] += 1
            return super()._take()

    for seed, nb in ((2, 40), (3, 24), (5, 18)):
        m = Spy(nb, 4 if seed != 3 else 2, 16)
        d = Driver(m, nb, m.block_size, OutOfBlocks)
        g = op_stream(seed, 400, m.block_size, max_tokens=m.block_size * 16 - 4)
        op = next(g)
        while True:
            ok = d.apply(op)
            if op[0] == "prompt" and d.log[-1][2] > 0:
                seen["hit"] += 1
            if not ok:
                seen["oob"] += 1
            if d.log[-1][0] == "step" and d.log[-1][1] != "oob" and len(d.log[-1][5]) > 0:
                seen["cow"] += 1
            if d.log[-1][0] == "prompt" and d.log[-1][3] != "oob" and len(d.log[-1][4]) > 0:
                seen["cow"] += 1
            try:
                op = g.send(ok)
            except StopIteration:
                break
    assert all(v > 0 for v in seen.values()), seen


def test_prefix_hits_match_brute_force():
    """No eviction (large pool): cached tokens = the longest common
    full-block prefix with any registered token list, leaving one token."""
    bs = 4
    m = BlockManagerModel(20000, bs, 32)
    registered: list[list[int]] = []
    rng = np.random.default_rng(11)
    live = {}
    for it in range(300):
        toks = [int(t) for t in rng.integers(0, 2, size=int(rng.integers(1, 40)))]
        seq = it + 1
        want = 0
        for r in registered:
            j = 0
            while (j + 1) * bs <= len(r) and (j + 1) * bs <= len(toks) - 1 and r[:(j + 1) * bs] == toks[:(j + 1) * bs]:
                j += 1
            want = max(want, j * bs)
        got = m.try_get_prefix_blocks(seq, toks)
        assert got == want, (it, got, want)
        m.update(seq, len(toks) - got)
        live[seq] = toks
        if rng.random() < 0.6:
            m.add_prefix(seq, toks)
            registered.append(toks)
        if rng.random() < 0.3:
            s = sorted(live)[int(rng.integers(0, len(live)))]
            m.free(s)
            del live[s]
    assert m.stats()["cached"] > 10


def test_refused_update_changes_nothing():
    m = BlockManagerModel(6, 4, 8)
    m.update(1, 10)            # 3 blocks
    m.fork(1, 2)               # shares all 3 (the last one partly filled)
    before = (copy.deepcopy(m.tables), list(m.ref), list(m.free_list), m.stats())
    with pytest.raises(OutOfBlocks):
        m.step([2, 1], [2, 16])   # 1 copy + 0 for seq 2, then 4 new blocks for seq 1: 5 > 3
    assert (m.tables, m.ref, m.free_list, m.stats()) == before
    with pytest.raises(ValueError):
        m.update(1, 30)        # beyond max_blocks_per_seq: refused, unchanged
    assert (m.tables, m.ref, m.free_list, m.stats()) == before
    slots, copies = m.update(2, 1)   # copy-on-write of the shared partial block
    assert len(copies) == 1 and copies[0][0] == before[0][1][2]
    assert m.block_table(2)[:2] == m.block_table(1)[:2] and m.block_table(2)[2] != m.block_table(1)[2]


def test_worked_allocation_policy():
    """Reading B1: block 0 first; the block released last is reused first;
    B6: a sequence's blocks are released last to first."""
    m = BlockManagerModel(8, 2, 8)
    m.update(1, 5)
    assert m.block_table(1) == [0, 1, 2]
    m.update(2, 2)
    assert m.block_table(2) == [3]
    m.free(1)                               # releases 2, 1, 0 -> free list ends ..., 2, 1, 0
    m.update(3, 3)
    assert m.block_table(3) == [0, 1]


# --- planted mistakes: each must be caught by the pins above ---------------

class SkipCopyOnWrite(BlockManagerModel):
    def _update(self, seq, n):
        table = self.tables.setdefault(seq, [])
        L = self.lens.setdefault(seq, 0)
        copies = []
        while len(table) < self._blocks_for(L + n):
            table.append(self._take())
        slots = [table[p // self.block_size] * self.block_size + p % self.block_size for p in range(L, L + n)]
        self.lens[seq] = L + n
        return slots, copies


class KeepEvictedEntry(BlockManagerModel):
    def _take(self):
        if self.free_list:
            b = self.free_list.pop()
        else:
            b = self.idle.pop(0)   # entry left in place: a later hit names a reused block
        self.ref[b] = 1
        return b


class ReleaseSharedToFree(BlockManagerModel):
    def _release(self, b):
        self.ref[b] -= 1
        if self.ref[b] <= 0 or b in self.entry_of_block:
            if b not in self.free_list:
                self.free_list.append(b)


@pytest.mark.parametrize("bad", [SkipCopyOnWrite, KeepEvictedEntry, ReleaseSharedToFree])
def test_planted_mistakes_are_caught(bad):
    caught = False
    for seed, nb in ((2, 40), (3, 24), (5, 18), (6, 30)):
        m = bad(nb, 4, 16)
        try:
            run_checked(m, seed, 400, max_tokens=60)
        except (AssertionError, ValueError, KeyError, IndexError):
            caught = True
            break
    assert caught
