"""fp64 CPU oracle for attention over a block-paged KV cache.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this module.  The
product path (the CUDA library and its Python binding) never calls it and
shares no code with it.

Everything here is the plain definition, written out in NumPy float64 with no
blocking, fusion or reordering beyond what the definition states:

* ``kv_write``      - the slot-mapping scatter of new K/V rows into the block
                      pool ("ADR 004: Paged Attention Serving Integration",
                      Decision 4: the model writes K/V into the block
                      allocator; "Paged Attention 基础", section 2: token ->
                      (physical block, slot)).
* ``gather``        - block-table translation of a sequence's logical
                      positions into physical (block, slot) pairs and the
                      gather of their K/V ("Paged Attention 基础", section 2,
                      steps 1-3 of the simplified attention for q = 23).
* ``attend``        - causal-masked softmax(scale * q K^T) V over the gathered
                      keys ("Paged Attention 基础", section 2, steps 4-5;
                      flash-attention issue #660, the softmax(Q @ K^T *
                      softmax_scale) @ V formula).
* ``paged_attention`` - both of the above for every sequence of a varlen
                      batch: prefill chunks, decode and multi-token
                      speculative verification share one call ("ADR 004",
                      Consequences; flash-attention issue #660).
* ``partial_attend`` / ``merge_partials`` - the split-KV partial state
                      (running max, running sum, unnormalised accumulator)
                      and its merge; the merged result equals ``attend``.

Readings of points the pages leave open (each also listed in the design notes):

1. slot = physical_block * block_size + position % block_size; slot < 0 means
   "skip this token" (padding).
2. context_lens[s] counts the tokens of sequence s after this step's write,
   new ones included; query i of a sequence with n queries sits at position
   L - n + i and, when causal, sees keys 0..L-n+i.  Non-causal queries see
   all L keys.
3. GQA: query head h reads kv head h // (Hq / Hkv) (contiguous groups).
4. Softmax is exact (max-subtracted); the output has the query's dtype after
   the caller's cast, shape [T, Hq, D].
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "kv_write", "gather", "attend", "paged_attention", "partial_attend",
    "merge_partials", "kv_head_of", "visible_keys",
]


def kv_head_of(h: int, num_q_heads: int, num_kv_heads: int) -> int:
    """KV head read by query head ``h`` (contiguous GQA groups)."""
    group = num_q_heads // num_kv_heads
    return h // group


def visible_keys(i: int, n: int, L: int, causal: bool) -> int:
    """Number of keys (a prefix 0..count-1) visible to query ``i`` of ``n``
    queries of a sequence with ``L`` tokens (bottom-right aligned)."""
    if not causal:
        return L
    return L - n + i + 1


def kv_write(k, v, slot_mapping, k_cache, v_cache) -> None:
    """In place: for every new token t with slot s >= 0,
    ``k_cache[s // bs, s % bs] = k[t]`` and the same for V.

    Works on any element type (bf16 bit patterns included): it is a copy.
    """
    bs = k_cache.shape[1]
    for t, s in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if s < 0:
            continue
        blk, off = divmod(int(s), bs)
        k_cache[blk, off] = k[t]
        v_cache[blk, off] = v[t]


def gather(cache, block_table, L: int) -> np.ndarray:
    """Logical rows 0..L-1 of one sequence: position t lives in physical
    block ``block_table[t // bs]`` at slot ``t % bs``.  Returns [L, Hkv, D]."""
    bs = cache.shape[1]
    pos = np.arange(int(L))
    blocks = np.asarray(block_table)[pos // bs].astype(np.int64)
    return cache[blocks, pos % bs]


def attend(q_rows, K, V, scale: float, causal: bool) -> np.ndarray:
    """softmax(scale * q K^T) V for the ``n`` queries of one sequence.

    q_rows [n, Hq, D], K/V [L, Hkv, D] (fp64).  Returns [n, Hq, D] fp64.
    """
    q_rows = np.asarray(q_rows, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    n, Hq, D = q_rows.shape
    L, Hkv, _ = K.shape
    out = np.zeros((n, Hq, D), dtype=np.float64)
    for h in range(Hq):
        g = kv_head_of(h, Hq, Hkv)
        for i in range(n):
            cnt = visible_keys(i, n, L, causal)
            z = scale * (K[:cnt, g, :] @ q_rows[i, h, :])
            z = z - z.max()
            w = np.exp(z)
            w = w / w.sum()
            out[i, h, :] = w @ V[:cnt, g, :]
    return out


def paged_attention(q, k_cache, v_cache, block_tables, context_lens, query_start_loc,
                    scale: float, causal: bool) -> np.ndarray:
    """The varlen batch: for each sequence s, gather its L_s keys through its
    block table and attend its queries q[qsl[s]:qsl[s+1]].  Returns [T, Hq, D]
    fp64.  Inputs must already be fp64 (or exactly convertible)."""
    q = np.asarray(q, dtype=np.float64)
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    T = int(qsl[-1])
    out = np.zeros((T,) + q.shape[1:], dtype=np.float64)
    for s in range(len(context_lens)):
        a, b = int(qsl[s]), int(qsl[s + 1])
        L = int(context_lens[s])
        if b <= a:
            continue
        if b - a > L:
            raise ValueError("a sequence cannot have more queries than tokens")
        K = gather(k_cache, block_tables[s], L)
        V = gather(v_cache, block_tables[s], L)
        out[a:b] = attend(q[a:b], K, V, scale, causal)
    return out


def partial_attend(q_rows, K, V, scale: float, causal: bool, key_begin: int, key_end: int):
    """Split-KV partial state over keys [key_begin, key_end) of one sequence.

    Returns (m, l, acc): m [n, Hq] the maximum visible logit (-inf when no key
    of the range is visible), l [n, Hq] = sum exp(z - m), acc [n, Hq, D] =
    sum exp(z - m) v.  All fp64.
    """
    q_rows = np.asarray(q_rows, dtype=np.float64)
    n, Hq, D = q_rows.shape
    L, Hkv, _ = K.shape
    m = np.full((n, Hq), -np.inf)
    l = np.zeros((n, Hq))
    acc = np.zeros((n, Hq, D))
    for h in range(Hq):
        g = kv_head_of(h, Hq, Hkv)
        for i in range(n):
            hi = min(key_end, visible_keys(i, n, L, causal))
            if hi <= key_begin:
                continue
            z = scale * (K[key_begin:hi, g, :] @ q_rows[i, h, :])
            m[i, h] = z.max()
            w = np.exp(z - m[i, h])
            l[i, h] = w.sum()
            acc[i, h] = w @ V[key_begin:hi, g, :]
    return m, l, acc


def merge_partials(parts) -> np.ndarray:
    """Merge split-KV partial states: m = max_p m_p, l = sum_p l_p e^(m_p - m),
    O = sum_p acc_p e^(m_p - m) / l."""
    ms = np.stack([p[0] for p in parts])           # [P, n, Hq]
    m = ms.max(axis=0)
    wts = np.where(np.isneginf(ms), 0.0, np.exp(ms - m))
    l = sum(w * p[1] for w, p in zip(wts, parts))
    acc = sum(w[..., None] * p[2] for w, p in zip(wts, parts))
    return acc / l[..., None]
