"""Drives a block manager (the reference model or the library's) through an
operation stream, keeping a K/V pool in host memory so that what the block
tables name can be checked against each sequence's logical K/V rows."""
from __future__ import annotations

import numpy as np

from oracle import paged_oracle as po
from workloads.block_ops import kv_rows

WIDTH = 3  # values per K/V row in these checks


class Driver:
    """Applies ops to ``mgr`` and mirrors their writes into a host pool.

    ``mgr`` offers update / step / free / fork / add_prefix /
    try_get_prefix_blocks / block_table / stats, raising ``out_of_blocks``
    when the free and idle blocks do not cover an update.
    """

    def __init__(self, mgr, num_blocks: int, block_size: int, out_of_blocks, pool: bool = True):
        self.mgr = mgr
        self.bs = block_size
        self.oob = out_of_blocks
        self.tokens: dict[int, list[int]] = {}
        self.rows: dict[int, np.ndarray] = {}  # logical K/V rows of each live sequence
        self.pool = None
        if pool:
            self.pool = np.full((num_blocks, block_size, 1, WIDTH), np.nan)
            self._vpool = np.empty_like(self.pool)  # the V side of kv_write; unused here
        self.log: list = []  # what each op returned, for comparing two managers

    def _copy(self, copies) -> None:
        if self.pool is None:
            return
        for src, dst in np.asarray(copies).reshape(-1, 2):
            self.pool[dst] = self.pool[src]

    def _write(self, slots, rows) -> None:
        if self.pool is None or len(slots) == 0:
            return
        k = np.asarray(rows, dtype=np.float64).reshape(len(slots), 1, WIDTH)
        po.kv_write(k, k, np.asarray(slots, dtype=np.int64), self.pool, self._vpool)

    def apply(self, op) -> bool:
        kind = op[0]
        m = self.mgr
        if kind == "prompt":
            _, seq, tokens = op
            cached = m.try_get_prefix_blocks(seq, tokens)
            try:
                slots, copies = m.update(seq, len(tokens) - cached)
            except self.oob:
                self.log.append(("prompt", seq, cached, "oob"))
                m.free(seq)
                return False
            self.log.append(("prompt", seq, cached, list(slots), [tuple(c) for c in copies]))
            self._copy(copies)
            rows = kv_rows(tokens, WIDTH)
            self._write(slots, rows[cached:])
            self.tokens[seq] = list(tokens)
            self.rows[seq] = rows
            return True
        if kind == "step":
            _, seqs, n_new, new_tokens = op
            try:
                meta = m.step(seqs, n_new)
            except self.oob:
                self.log.append(("step", "oob"))
                return False
            self.log.append(("step",) + tuple(np.asarray(meta[k]).tolist() for k in
                                              ("slot_mapping", "block_tables", "context_lens",
                                               "query_start_loc", "copies")))
            self._copy(meta["copies"])
            rows = []
            for s, t in zip(seqs, new_tokens):
                L = len(self.tokens[s])
                self.tokens[s] = self.tokens[s] + list(t)
                self.rows[s] = kv_rows(self.tokens[s], WIDTH)
                rows.append(self.rows[s][L:])
            self._write(meta["slot_mapping"], np.concatenate(rows) if rows else [])
            return True
        if kind == "fork":
            _, parent, child = op
            m.fork(parent, child)
            self.tokens[child] = list(self.tokens[parent])
            self.rows[child] = self.rows[parent]
            self.log.append(("fork", parent, child))
            return True
        if kind == "free":
            m.free(op[1])
            del self.tokens[op[1]]
            del self.rows[op[1]]
            self.log.append(("free", op[1]))
            return True
        if kind == "add_prefix":
            m.add_prefix(op[1], op[2])
            self.log.append(("add_prefix", op[1]))
            return True
        raise ValueError(kind)

    def run(self, stream, check_every_op: bool = True) -> None:
        op = next(stream)
        while True:
            ok = self.apply(op)
            if check_every_op:
                self.check_content()
                self.log.append(("stats", tuple(sorted(self.mgr.stats().items()))))
            try:
                op = stream.send(ok)
            except StopIteration:
                break

    def check_content(self) -> None:
        """Gathering a sequence through its block table gives its logical rows."""
        if self.pool is None:
            return
        for s, toks in self.tokens.items():
            table = np.asarray(self.mgr.block_table(s), dtype=np.int64)
            assert len(table) == -(-len(toks) // self.bs), (s, len(table), len(toks))
            got = po.gather(self.pool, table, len(toks))[:, 0, :]
            assert np.array_equal(got, self.rows[s].reshape(-1, WIDTH)), \
                f"sequence {s}: content through its block table differs"
