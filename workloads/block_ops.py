"""Seeded operation streams for a block manager, and the K/V rows they write.

This module only *builds inputs*.  It tracks the logical token list of every
live sequence, and nothing of blocks or slots.  Both the reference model
(``oracle/block_manager.py``) and the library's C++ block manager consume the
same stream, which serves as the parity case for one against the other.

The stream follows the serving life cycle the pages describe:

* "ADR 004: Paged Attention Serving Integration", Decision 5 and
  Consequences: requests arrive, are extended step by step (one update call
  for prefill and decode) and are freed when they finish.  Limitations: a
  cached prompt prefix is replayed (add_prefix / try_get_prefix_blocks).
* "Paged Attention 基础", section 1, problem 3: many requests share a prefix
  (a system prompt).

The op kinds are:

* ``("prompt", seq, tokens)``: a new request.  The caller calls
  try_get_prefix_blocks, then update for the tokens that were not cached.
* ``("step", seqs, n_new, new_tokens)``: one batch step (prefill chunks,
  decode, several draft tokens).
* ``("fork", parent, child)``: a child starts from the parent's tokens.
* ``("free", seq)``: the request ends.
* ``("add_prefix", seq, tokens)``: the request's tokens so far become
  cacheable.

Use it as a generator: ``op = next(g)``, then ``op = g.send(ok)`` after
applying each op, with ``ok`` False when the manager refused it for want of
blocks (the stream then treats it as not having happened).

``kv_row(tokens)`` is the K (or V) row of the last of ``tokens``.  It depends
on the whole prefix, as a transformer's K/V do, so a block reused for a
different prefix shows up as wrong content.
"""
from __future__ import annotations

import numpy as np

__all__ = ["op_stream", "kv_row", "kv_rows", "kv_rows_normal"]

_P = (1 << 61) - 1


def _expand(h: int, width: int) -> np.ndarray:
    out = np.empty(width, dtype=np.float64)
    for i in range(width):
        h = (h * 6364136223846793005 + 1442695040888963407) % _P
        out[i] = (h % 2048) / 1024.0 - 1.0
    return out


def kv_row(tokens, width: int, salt: int = 0) -> np.ndarray:
    """A deterministic row of ``width`` values in [-1, 1) for a token prefix."""
    h = 1469598103934665603 + salt
    for t in tokens:
        h = (h * 1099511628211 + int(t) + 7) % _P
    return _expand(h, width)


def kv_rows(tokens, width: int, salt: int = 0) -> np.ndarray:
    """``kv_row(tokens[:p + 1])`` for every position p, as [len, width]."""
    h = 1469598103934665603 + salt
    out = np.empty((len(tokens), width), dtype=np.float64)
    for p, t in enumerate(tokens):
        h = (h * 1099511628211 + int(t) + 7) % _P
        out[p] = _expand(h, width)
    return out


def kv_rows_normal(tokens, width: int, salt: int = 0) -> np.ndarray:
    """Rows of N(0, 1) fp32 values, row p drawn from a generator seeded by the
    hash of ``tokens[:p + 1]`` (and ``salt``: K and V use different ones)."""
    h = 1469598103934665603
    out = np.empty((len(tokens), width), dtype=np.float32)
    for p, t in enumerate(tokens):
        h = (h * 1099511628211 + int(t) + 7) % _P
        out[p] = np.random.default_rng([h, salt]).standard_normal(width, dtype=np.float32)
    return out


def op_stream(seed: int, n_ops: int, block_size: int, *, max_tokens: int, vocab: int = 3,
              n_system: int = 3, p_fork: float = 0.08, p_free: float = 0.15, p_prefix: float = 0.12,
              max_live: int = 12, max_chunk: int = 0):
    """Yields ``n_ops`` operations (see the module docstring)."""
    rng = np.random.default_rng(seed)
    bs = block_size
    chunk_cap = max_chunk or 3 * bs
    # shared system prompts: whole blocks plus a ragged tail
    system = [list(rng.integers(0, vocab, size=int(rng.integers(1, 4)) * bs + int(rng.integers(0, bs))))
              for _ in range(n_system)]
    live: dict[int, list[int]] = {}
    next_seq = 1
    for _ in range(n_ops):
        r = rng.random()
        seqs = sorted(live)
        if (not seqs or (r < 0.25 and len(seqs) < max_live)):
            base = list(system[int(rng.integers(0, n_system))]) if rng.random() < 0.7 else []
            tail = list(rng.integers(0, vocab, size=int(rng.integers(1, 2 * bs + 2))))
            tokens = (base + tail)[:max_tokens]
            seq = next_seq
            next_seq += 1
            ok = yield ("prompt", seq, tokens)
            if ok:
                live[seq] = tokens
        elif r < 0.25 + p_fork and len(seqs) < max_live:
            parent = seqs[int(rng.integers(0, len(seqs)))]
            child = next_seq
            next_seq += 1
            ok = yield ("fork", parent, child)
            if ok:
                live[child] = list(live[parent])
        elif r < 0.25 + p_fork + p_free:
            seq = seqs[int(rng.integers(0, len(seqs)))]
            yield ("free", seq)
            del live[seq]
        elif r < 0.25 + p_fork + p_free + p_prefix:
            seq = seqs[int(rng.integers(0, len(seqs)))]
            yield ("add_prefix", seq, list(live[seq]))
        else:
            k = int(rng.integers(1, len(seqs) + 1))
            pick = sorted(rng.choice(seqs, size=k, replace=False).tolist())
            n_new, new_tokens = [], []
            for s in pick:
                room = max_tokens - len(live[s])
                n = int(rng.integers(0, chunk_cap + 1)) if rng.random() < 0.3 else 1
                n = max(0, min(n, room))
                n_new.append(n)
                new_tokens.append(list(rng.integers(0, vocab, size=n)))
            ok = yield ("step", pick, n_new, new_tokens)
            if ok:
                for s, t in zip(pick, new_tokens):
                    live[s] += t
