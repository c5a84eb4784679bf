"""Reference model of the host block manager of a block-paged KV cache.

TEST INFRASTRUCTURE.  Only ``tests/`` and the CPU legs of ``bench.py`` may
import this module.  The C++ block manager of the library never calls it and
shares no code with it; the two are compared call by call on the same seeded
operation streams.

What a block manager does, from the pages:

* "Paged Attention 基础 - 原理与实现进度", section 3.1 C: a block manager
  that allocates and frees blocks from a Python list, and block-table
  management producing a ``[batch_size, max_blocks_per_seq]`` table.
  Section 1, problem 2: a growing sequence takes one new block and one more
  table entry; nothing already written moves.  Section 1, problem 3 and
  section 2: several block tables may name the same physical block (prefix
  caching: sequence B = [7, 9] shares block 7 of A = [7, 3]).
* "ADR 004: Paged Attention Serving Integration", Decision 5: block tables
  live in the block manager keyed by sequence id and are cleared when
  ``free(seq_id)`` ends a request.  Consequences: ``update`` both allocates a
  fresh sequence and extends an existing one, so prefill and decode steps use
  one call.  Limitations: ``add_prefix`` and ``try_get_prefix_blocks`` replay
  a cached prompt prefix.
* Dao-AILab/flash-attention issue #660: the caller's cache manager copies and
  updates the pages; the kernels only read and write them.

Readings of what the pages leave open (each also listed in the design notes):

B1  The free list is a list holding [num_blocks - 1, ..., 1, 0].  Allocation
    pops from its end (block 0 first); a released block is appended (the
    block released last is reused first).
B2  A block's reference count is the number of block-table entries that name
    it.  A block is in exactly one of: the free list, in use (count > 0), or
    cached idle (B3).
B3  Prefix cache: only full blocks are cached.  An entry's key is (the
    parent entry's id, the block's block_size token ids); the root id is 0
    and entry ids are never reused, so a key names the whole token prefix up
    to the block's end.  A cached block whose count drops to 0 stays cached
    ("idle", kept in release order).  Allocation takes the free list first,
    then evicts the idle block released longest ago and drops its entry.
B4  try_get_prefix_blocks(seq, tokens) starts a fresh sequence on the
    longest chain of cached entries that match its prompt's leading full
    blocks, counting at most len(tokens) - 1 tokens: the last prompt token is
    always left to compute, so no step writes into a block it shares.
B5  update(seq, n) creates the sequence when it is unknown, then appends n
    tokens.  When n > 0 and the last block is partly filled and shared
    (count > 1), copy-on-write first: a new block replaces it in this table,
    the caller gets the (src, dst) pair to copy, and src's count drops by
    one.  Then it takes the blocks the new tokens need.  If the free and idle
    blocks cannot cover that, nothing changes and OutOfBlocks is raised.
B6  free(seq) releases the sequence's blocks from its last to its first, so
    that a prompt's deepest blocks are the first evicted.
B7  fork(parent, child): the child's table is the parent's, every count + 1.
B8  step(seq_ids, n_new) applies update to each sequence in order, all or
    nothing, and returns the call metadata of paged attention: slot_mapping,
    block_tables (padded with -1), context_lens, query_start_loc, copies.
B9  add_prefix(seq, tokens), tokens = all of the sequence's tokens: walks its
    full blocks from the root.  A block whose key is already cached follows
    that entry (even on another physical block, which then stays
    unregistered); an unregistered block gets a new entry; a block cached
    under a key that no longer chains from the root is re-keyed.
"""
from __future__ import annotations

import copy

import numpy as np

__all__ = ["BlockManagerModel", "OutOfBlocks"]


class OutOfBlocks(Exception):
    """The free and idle blocks do not cover an update (reading B5)."""


class BlockManagerModel:
    def __init__(self, num_blocks: int, block_size: int, max_blocks_per_seq: int):
        if num_blocks <= 0 or block_size <= 0 or max_blocks_per_seq <= 0:
            raise ValueError("sizes must be positive")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.max_blocks = max_blocks_per_seq
        self.free_list = list(range(num_blocks - 1, -1, -1))  # B1
        self.ref = [0] * num_blocks                             # B2
        self.tables: dict[int, list[int]] = {}
        self.lens: dict[int, int] = {}
        self.entries: dict[tuple, tuple[int, int]] = {}         # key -> (entry id, block)  B3
        self.entry_of_block: dict[int, tuple[tuple, int]] = {}  # block -> (key, entry id)
        self.idle: list[int] = []                               # cached blocks with count 0, oldest first
        self.next_entry = 1

    # -- block pool ------------------------------------------------------
    def available(self) -> int:
        return len(self.free_list) + len(self.idle)

    def _take(self) -> int:
        if self.free_list:
            b = self.free_list.pop()
        else:
            b = self.idle.pop(0)
            key, _ = self.entry_of_block.pop(b)
            del self.entries[key]
        self.ref[b] = 1
        return b

    def _release(self, b: int) -> None:
        self.ref[b] -= 1
        if self.ref[b] == 0:
            if b in self.entry_of_block:
                self.idle.append(b)
            else:
                self.free_list.append(b)

    def _blocks_for(self, tokens: int) -> int:
        return -(-tokens // self.block_size)

    # -- sequences -------------------------------------------------------
    def _update(self, seq: int, n: int) -> tuple[list[int], list[tuple[int, int]]]:
        if n < 0:
            raise ValueError("negative token count")
        table = self.tables.setdefault(seq, [])
        L = self.lens.setdefault(seq, 0)
        if self._blocks_for(L + n) > self.max_blocks:
            raise ValueError("sequence longer than max_blocks_per_seq blocks")
        copies = []
        if n > 0 and L % self.block_size != 0 and self.ref[table[-1]] > 1:   # B5 copy-on-write
            src = table[-1]
            dst = self._take()
            self.ref[src] -= 1
            table[-1] = dst
            copies.append((src, dst))
        while len(table) < self._blocks_for(L + n):
            table.append(self._take())
        slots = [table[p // self.block_size] * self.block_size + p % self.block_size for p in range(L, L + n)]
        self.lens[seq] = L + n
        return slots, copies

    def _atomic(self, fn):
        saved = copy.deepcopy(self.__dict__)
        try:
            return fn()
        except (OutOfBlocks, ValueError, KeyError):
            self.__dict__.update(saved)
            raise
        except IndexError:  # a pool ran dry part way: nothing changes (B5)
            self.__dict__.update(saved)
            raise OutOfBlocks()

    def update(self, seq: int, n: int):
        """Slots of the n new tokens and the copy-on-write pairs (B5)."""
        return self._atomic(lambda: self._update(seq, n))

    def step(self, seq_ids, n_new):
        """B8: update every sequence in order, all or nothing; the metadata."""
        if len(set(seq_ids)) != len(seq_ids):
            raise ValueError("a sequence twice in one step")

        def run():
            slots, copies = [], []
            for s, n in zip(seq_ids, n_new):
                sl, cp = self._update(s, n)
                slots += sl
                copies += cp
            return slots, copies

        slots, copies = self._atomic(run)
        B = len(seq_ids)
        tables = np.full((B, self.max_blocks), -1, dtype=np.int32)
        for i, s in enumerate(seq_ids):
            tables[i, :len(self.tables[s])] = self.tables[s]
        qsl = np.zeros(B + 1, dtype=np.int32)
        qsl[1:] = np.cumsum(np.asarray(n_new, dtype=np.int64))
        return {
            "slot_mapping": np.asarray(slots, dtype=np.int64),
            "block_tables": tables,
            "context_lens": np.asarray([self.lens[s] for s in seq_ids], dtype=np.int32),
            "query_start_loc": qsl,
            "copies": np.asarray(copies, dtype=np.int32).reshape(-1, 2),
        }

    def free(self, seq: int) -> None:
        """B6: release from the last block to the first; forget the sequence."""
        table = self.tables.pop(seq)
        del self.lens[seq]
        for b in reversed(table):
            self._release(b)

    def fork(self, parent: int, child: int) -> None:
        """B7."""
        if child in self.tables:
            raise ValueError("child exists")
        table = self.tables[parent]
        self.tables[child] = list(table)
        self.lens[child] = self.lens[parent]
        for b in table:
            self.ref[b] += 1

    # -- prefix cache ----------------------------------------------------
    def add_prefix(self, seq: int, tokens) -> None:
        """B9: cache the sequence's full blocks under their token prefix."""
        tokens = [int(t) for t in tokens]
        if len(tokens) != self.lens[seq]:
            raise ValueError("tokens must be all of the sequence's tokens")
        table, bs, parent = self.tables[seq], self.block_size, 0
        for j in range(len(tokens) // bs):
            key = (parent, tuple(tokens[j * bs:(j + 1) * bs]))
            if key in self.entries:
                parent = self.entries[key][0]
                continue
            b = table[j]
            if b in self.entry_of_block:      # cached under a stale key: re-key
                old_key, eid = self.entry_of_block[b]
                del self.entries[old_key]
            else:
                eid = self.next_entry
                self.next_entry += 1
            self.entries[key] = (eid, b)
            self.entry_of_block[b] = (key, eid)
            parent = eid

    def try_get_prefix_blocks(self, seq: int, tokens) -> int:
        """B4: attach the cached chain; returns the tokens it covers."""
        tokens = [int(t) for t in tokens]
        if self.tables.get(seq):
            raise ValueError("sequence already has blocks")
        bs, parent, hits = self.block_size, 0, []
        for j in range(min(max(len(tokens) - 1, 0) // bs, self.max_blocks)):
            key = (parent, tuple(tokens[j * bs:(j + 1) * bs]))
            if key not in self.entries:
                break
            parent, b = self.entries[key]
            hits.append(b)
        for b in hits:
            if self.ref[b] == 0:
                self.idle.remove(b)
            self.ref[b] += 1
        self.tables[seq] = hits
        self.lens[seq] = len(hits) * bs
        return len(hits) * bs

    # -- views -----------------------------------------------------------
    def block_table(self, seq: int) -> list[int]:
        return list(self.tables[seq])

    def stats(self) -> dict:
        in_use = sum(1 for r in self.ref if r > 0)
        return {"free": len(self.free_list), "idle": len(self.idle), "in_use": in_use,
                "cached": len(self.entries)}
