"""Seeded synthetic inputs for attention over a block-paged KV cache.

This module only *builds inputs*: the contents of a physical block pool, the
per-sequence block tables, the slot mapping of the new tokens, the query rows
and the new K/V rows.  It computes no attention and performs no cache write;
both the fp64 oracle (``oracle/``) and the CUDA path consume what it returns.

Inputs follow the serving workloads the source pages describe:

* "Paged Attention 基础 - 原理与实现进度", section 2: a sequence's tokens are
  kept in fixed-size physical blocks named by a block table; several tables
  may name the same physical block (prefix sharing).
* "ADR 004: Paged Attention Serving Integration", Decision 4 and Consequences:
  new K/V rows are written into the block pool and prefill chunks and decode
  steps go through the same attention call.
* Dao-AILab/flash-attention issue #660: several query tokens per sequence
  (speculative decoding) next to single-token decode.

Conventions (readings of points the pages leave open):

* ``slot = physical_block * block_size + (position % block_size)``.
* ``context_lens[s]`` counts every token of sequence ``s`` after this step's
  write, the ``n_s`` new ones included; the new tokens sit at positions
  ``L_s - n_s .. L_s - 1`` (bottom-right aligned queries).
* Physical blocks come from a seeded permutation of the pool, consumed in
  sequence order and logical-block order, shared blocks first.
* Values are N(0, 1) drawn in fp32 from PCG64 streams and rounded to the
  workload dtype (round-to-nearest-even for bf16).  bf16 arrays are held as
  their uint16 bit patterns.

Unused pool slots hold zeros, or NaN when ``poison=True`` (to check that no
consumer reads a slot outside a sequence's context).
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

BF16_NAN_BITS = 0x7FC0
_CHUNK = 1 << 22  # values per independent PCG64 stream (fixed: results do not depend on threads)


# ----------------------------------------------------------------------------
# value representation helpers (data formats only)
# ----------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round-to-nearest-even), returned as uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    out = np.empty(u.shape, dtype=np.uint16)
    flat_u = u.reshape(-1)
    flat_o = out.reshape(-1)

    def work(lo: int, hi: int) -> None:
        s = flat_u[lo:hi]
        bias = ((s >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
        flat_o[lo:hi] = ((s + bias) >> np.uint32(16)).astype(np.uint16)

    _parallel_ranges(flat_u.size, work)
    return out


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp64."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact fp64 view of a workload array held in ``dtype`` ("bf16" bits or "f32")."""
    if dtype == "bf16":
        return bf16_bits_to_f64(a)
    return np.asarray(a, dtype=np.float64)


def _parallel_ranges(n: int, fn, chunk: int = _CHUNK) -> None:
    ranges = [(lo, min(n, lo + chunk)) for lo in range(0, n, chunk)]
    if len(ranges) <= 1:
        for lo, hi in ranges:
            fn(lo, hi)
        return
    with ThreadPoolExecutor(max_workers=16) as ex:
        list(ex.map(lambda r: fn(*r), ranges))


def normal_values(seed_seq: np.random.SeedSequence, count: int, dtype: str) -> np.ndarray:
    """``count`` N(0,1) values in the workload dtype, deterministic for ``seed_seq``.

    The draw is split into fixed 4 Mi-value chunks, each from its own spawned
    PCG64 stream, so the result does not depend on the number of threads.
    """
    nchunks = max(1, math.ceil(count / _CHUNK))
    children = seed_seq.spawn(nchunks)
    vals = np.empty(count, dtype=np.float32)

    def work(i: int) -> None:
        lo, hi = i * _CHUNK, min(count, (i + 1) * _CHUNK)
        if hi > lo:
            g = np.random.Generator(np.random.PCG64(children[i]))
            g.standard_normal(out=vals[lo:hi], dtype=np.float32)

    if nchunks == 1:
        work(0)
    else:
        with ThreadPoolExecutor(max_workers=16) as ex:
            list(ex.map(work, range(nchunks)))
    if dtype == "bf16":
        return f32_to_bf16_bits(vals)
    if dtype == "f32":
        return vals
    raise ValueError(f"unknown dtype {dtype!r}")


# ----------------------------------------------------------------------------
# workload containers
# ----------------------------------------------------------------------------

@dataclass
class Step:
    """One call of the hot path: write the new K/V rows, then attend."""
    q: np.ndarray               # [T, Hq, D]
    k_new: np.ndarray           # [T, Hkv, D]
    v_new: np.ndarray           # [T, Hkv, D]
    slot_mapping: np.ndarray    # [T] int64, <0 = skip
    block_tables: np.ndarray    # [B, max_blocks] int32, unused entries -1
    context_lens: np.ndarray    # [B] int32, includes the new tokens
    query_start_loc: np.ndarray  # [B+1] int32

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.query_start_loc[-1])

    @property
    def q_lens(self) -> np.ndarray:
        return np.diff(self.query_start_loc.astype(np.int64))


@dataclass
class Workload:
    name: str
    dtype: str                   # "bf16" or "f32"
    num_blocks: int
    block_size: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    k_cache: np.ndarray          # [NB, bs, Hkv, D] before the first step's write
    v_cache: np.ndarray
    steps: list[Step]
    scale: float
    causal: bool = True
    meta: dict = field(default_factory=dict)

    @property
    def step(self) -> Step:
        return self.steps[0]


# ----------------------------------------------------------------------------
# generic builder
# ----------------------------------------------------------------------------

def _empty_pool(nb: int, bs: int, hkv: int, d: int, dtype: str, poison: bool) -> np.ndarray:
    if dtype == "bf16":
        return np.full((nb, bs, hkv, d), BF16_NAN_BITS if poison else 0, dtype=np.uint16)
    return np.full((nb, bs, hkv, d), np.nan if poison else 0.0, dtype=np.float32)


def slots_of(block_table: np.ndarray, positions: np.ndarray, bs: int) -> np.ndarray:
    """Slot ids of logical positions under one block table (input recipe)."""
    positions = np.asarray(positions, dtype=np.int64)
    return block_table[positions // bs].astype(np.int64) * bs + positions % bs


def build(
    name: str,
    *,
    context_lens,
    q_lens,
    num_blocks: int,
    block_size: int,
    num_q_heads: int,
    num_kv_heads: int,
    head_dim: int,
    dtype: str,
    seed: int,
    shared_prefix_tokens: int = 0,
    share_groups=None,
    poison: bool = False,
    max_blocks_per_seq: int | None = None,
    causal: bool = True,
    scale: float | None = None,
    block_order: str = "permutation",
    meta: dict | None = None,
) -> Workload:
    """Build a one-step workload from per-sequence context and query lengths.

    ``shared_prefix_tokens`` (a multiple of ``block_size``) are held in the same
    physical blocks by every sequence.  ``share_groups``, a list of
    ``(first_seq, last_seq, tokens)``, instead gives each listed run of
    sequences its own shared prefix (disjoint runs; ``tokens`` a multiple of
    ``block_size``); other sequences keep all their blocks private.  ``block_order`` is ``"permutation"``
    (a seeded random permutation of the pool) or ``"sequential"``.
    """
    L = np.asarray(context_lens, dtype=np.int64)
    n = np.asarray(q_lens, dtype=np.int64)
    B = L.shape[0]
    bs = block_size
    if n.shape != L.shape or np.any(n < 0) or np.any(n > L):
        raise ValueError("need 0 <= q_len <= context_len per sequence")
    if share_groups is None:
        share_groups = [(0, B - 1, shared_prefix_tokens)] if B and shared_prefix_tokens else []
    elif shared_prefix_tokens:
        raise ValueError("give shared_prefix_tokens or share_groups, not both")
    share = np.zeros(B, dtype=np.int64)        # shared tokens of each sequence
    share_gid = np.full(B, -1, dtype=np.int64)
    for gi, (a, b, tok) in enumerate(share_groups):
        if tok % bs:
            raise ValueError("shared prefix must fill whole blocks")
        if not (0 <= a <= b < B) or np.any(share_gid[a:b + 1] >= 0):
            raise ValueError("share groups must be disjoint runs of sequences")
        if np.any(L[a:b + 1] - n[a:b + 1] < tok):
            raise ValueError("new tokens must lie after the shared prefix")
        share[a:b + 1] = tok
        share_gid[a:b + 1] = gi
    ss = np.random.SeedSequence(seed)
    s_layout, s_q, s_k, s_v, s_kc, s_vc = ss.spawn(6)
    g_layout = np.random.Generator(np.random.PCG64(s_layout))

    nblk = (L + bs - 1) // bs
    n_sh = share // bs  # shared blocks of each sequence
    mb = int(max_blocks_per_seq or max(1, int(nblk.max(initial=1))))
    if np.any(nblk > mb):
        raise ValueError("max_blocks_per_seq too small")
    need = sum(tok // bs for (_, _, tok) in share_groups) + int(np.sum(np.maximum(nblk - n_sh, 0)))
    if need > num_blocks:
        raise ValueError(f"pool too small: need {need} blocks, have {num_blocks}")
    order = g_layout.permutation(num_blocks) if block_order == "permutation" else np.arange(num_blocks)
    # the groups' shared blocks first (in group order), then private blocks in sequence order
    group_ids = []
    cursor = 0
    for (_, _, tok) in share_groups:
        group_ids.append(order[cursor:cursor + tok // bs])
        cursor += tok // bs
    bt = np.full((B, mb), -1, dtype=np.int32)
    for s in range(B):
        k = int(n_sh[s])
        if k:
            bt[s, :min(k, nblk[s])] = group_ids[share_gid[s]][:min(k, nblk[s])]
        priv = int(max(nblk[s] - k, 0))
        bt[s, k:k + priv] = order[cursor:cursor + priv]
        cursor += priv

    Hkv, D, Hq = num_kv_heads, head_dim, num_q_heads
    row = Hkv * D
    k_cache = _empty_pool(num_blocks, bs, Hkv, D, dtype, poison)
    v_cache = _empty_pool(num_blocks, bs, Hkv, D, dtype, poison)

    # cached (already written) tokens: the shared prefix once, then each
    # sequence's private cached positions
    cached_slots = [slots_of(bt[a], np.arange(tok), bs) for (a, _, tok) in share_groups if tok]
    for s in range(B):
        pos = np.arange(share[s], L[s] - n[s])
        cached_slots.append(slots_of(bt[s], pos, bs))
    cached_slots = np.concatenate(cached_slots) if cached_slots else np.zeros(0, np.int64)
    nc = cached_slots.shape[0]
    kflat = k_cache.reshape(num_blocks * bs, row)
    vflat = v_cache.reshape(num_blocks * bs, row)
    if nc:
        kflat[cached_slots] = normal_values(s_kc, nc * row, dtype).reshape(nc, row)
        vflat[cached_slots] = normal_values(s_vc, nc * row, dtype).reshape(nc, row)

    T = int(n.sum())
    qsl = np.zeros(B + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(n)
    slot_mapping = np.concatenate(
        [slots_of(bt[s], np.arange(L[s] - n[s], L[s]), bs) for s in range(B)]
    ) if B else np.zeros(0, np.int64)
    q = normal_values(s_q, T * Hq * D, dtype).reshape(T, Hq, D)
    k_new = normal_values(s_k, T * row, dtype).reshape(T, Hkv, D)
    v_new = normal_values(s_v, T * row, dtype).reshape(T, Hkv, D)
    step = Step(q=q, k_new=k_new, v_new=v_new, slot_mapping=slot_mapping.astype(np.int64),
                block_tables=bt, context_lens=L.astype(np.int32), query_start_loc=qsl)
    return Workload(
        name=name, dtype=dtype, num_blocks=num_blocks, block_size=bs, num_q_heads=Hq,
        num_kv_heads=Hkv, head_dim=D, k_cache=k_cache, v_cache=v_cache, steps=[step],
        scale=(1.0 / math.sqrt(D)) if scale is None else float(scale), causal=causal,
        meta=dict(meta or {}, shared_prefix_tokens=shared_prefix_tokens,
                  share_groups=[tuple(int(x) for x in g) for g in share_groups], seed=seed),
    )


# ----------------------------------------------------------------------------
# the serving workloads
# ----------------------------------------------------------------------------

def tiny(case: str = "1", poison: bool = False) -> Workload:
    """Tiny fp32 paged attention on the pages' worked example.

    Sequence A's first 24 tokens live in physical blocks [7, 3] (block 3 uses
    only its first 8 slots); sequence B shares physical block 7 and continues
    in blocks 9 and 12 ("Paged Attention 基础", section 2).  bs=16, 16 blocks,
    4 q heads / 2 kv heads, head_dim 64, scale 1/8.

    case "1": A has 24 cached tokens and B 40; each runs an 8-token causal
    prefill chunk (A: positions 24..31 in block 3 slots 8..15, B: 40..47 in
    block 12 slots 8..15) and then a 1-token decode whose position needs a
    fresh block: a lowest-free-id allocator hands block 0 to A and block 1 to
    B.  Two steps.

    case "1b": the page's literal state: A holds 24 tokens in total and its
    last 8 (positions 16..23, q=23 the last) are the chunk; B's chunk is its
    positions 32..39 in block 12.  One step.
    """
    nb, bs, hq, hkv, d = 16, 16, 4, 2, 64
    ss = np.random.SeedSequence(1001 if case == "1" else 1011)
    s_pref, s_a, s_b, s_q1, s_k1, s_v1, s_q2, s_k2, s_v2 = ss.spawn(9)
    row = hkv * d
    k_cache = _empty_pool(nb, bs, hkv, d, "f32", poison)
    v_cache = _empty_pool(nb, bs, hkv, d, "f32", poison)
    bt_a0, bt_b0 = [7, 3], [7, 9, 12]
    if case == "1":
        cached = {"A": 24, "B": 40}
    elif case == "1b":
        cached = {"A": 16, "B": 32}
    else:
        raise ValueError(case)
    # shared block 7 holds tokens 0..15 of both sequences: written once
    kp = normal_values(s_pref, 2 * 16 * row, "f32").reshape(2, 16, hkv, d)
    k_cache[7], v_cache[7] = kp[0], kp[1]
    for seqname, s_seq, bt in (("A", s_a, bt_a0), ("B", s_b, bt_b0)):
        cnt = cached[seqname] - 16
        if cnt > 0:
            vals = normal_values(s_seq, 2 * cnt * row, "f32").reshape(2, cnt, hkv, d)
            sl = slots_of(np.asarray(bt), np.arange(16, cached[seqname]), bs)
            k_cache.reshape(nb * bs, hkv, d)[sl] = vals[0]
            v_cache.reshape(nb * bs, hkv, d)[sl] = vals[1]

    def mk_step(bts, ctx, qlens, sq, sk, sv):
        mbps = 4
        bt = np.full((2, mbps), -1, dtype=np.int32)
        for i, b in enumerate(bts):
            bt[i, :len(b)] = b
        L = np.asarray(ctx, dtype=np.int64)
        n = np.asarray(qlens, dtype=np.int64)
        T = int(n.sum())
        qsl = np.zeros(3, dtype=np.int32)
        qsl[1:] = np.cumsum(n)
        sm = np.concatenate([slots_of(bt[s], np.arange(L[s] - n[s], L[s]), bs) for s in range(2)])
        return Step(
            q=normal_values(sq, T * hq * d, "f32").reshape(T, hq, d),
            k_new=normal_values(sk, T * row, "f32").reshape(T, hkv, d),
            v_new=normal_values(sv, T * row, "f32").reshape(T, hkv, d),
            slot_mapping=sm.astype(np.int64), block_tables=bt,
            context_lens=L.astype(np.int32), query_start_loc=qsl)

    if case == "1":
        steps = [
            mk_step([bt_a0, bt_b0], [32, 48], [8, 8], s_q1, s_k1, s_v1),
            # lowest free ids after {3, 7, 9, 12}: 0 for A, 1 for B
            mk_step([bt_a0 + [0], bt_b0 + [1]], [33, 49], [1, 1], s_q2, s_k2, s_v2),
        ]
    else:
        steps = [mk_step([bt_a0, bt_b0], [24, 40], [8, 8], s_q1, s_k1, s_v1)]
    return Workload(name=f"tiny-{case}", dtype="f32", num_blocks=nb, block_size=bs,
                    num_q_heads=hq, num_kv_heads=hkv, head_dim=d, k_cache=k_cache,
                    v_cache=v_cache, steps=steps, scale=1.0 / 8.0, causal=True,
                    meta={"seed": 1001, "shared_prefix_tokens": 16})


def decode_batch(poison: bool = False, batch: int = 64, seed: int = 1002) -> Workload:
    """Decode batch, bf16: 64 sequences, context U[512, 4096], one query token
    each, 32 q / 8 kv heads, head_dim 128, block_size 16, 20000-block pool."""
    g = np.random.Generator(np.random.PCG64(seed + 7_000_000))
    L = g.integers(512, 4096, size=batch, endpoint=True)
    return build("decode-b64", context_lens=L, q_lens=np.ones(batch, np.int64), num_blocks=20000,
                 block_size=16, num_q_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16",
                 seed=seed, poison=poison, max_blocks_per_seq=256)


def mixed_batch(poison: bool = False, seed: int = 1003) -> Workload:
    """Mixed continuous batch, bf16: 8 prefill chunks of 512 new tokens on
    U[0, 2048] cached tokens, then 120 one-token decodes with context
    U[256, 8192]; 32 q / 8 kv heads, head_dim 128, block_size 16, 80000 blocks."""
    g = np.random.Generator(np.random.PCG64(seed + 7_000_000))
    cached = g.integers(0, 2048, size=8, endpoint=True)
    dec = g.integers(256, 8192, size=120, endpoint=True)
    L = np.concatenate([cached + 512, dec])
    n = np.concatenate([np.full(8, 512), np.ones(120, np.int64)])
    return build("mixed-8x512+120", context_lens=L, q_lens=n, num_blocks=80000, block_size=16,
                 num_q_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16", seed=seed,
                 poison=poison, max_blocks_per_seq=512)


def prefill_chunks(poison: bool = False, seed: int = 1003) -> Workload:
    """The mixed batch's 8 prefill chunks alone (512 new tokens on U[0, 2048]
    cached tokens each, the same draw as the mixed batch): the compute-bound
    part of multi-token attention.  32 q / 8 kv heads, head_dim 128, bs 16."""
    g = np.random.Generator(np.random.PCG64(seed + 7_000_000))
    cached = g.integers(0, 2048, size=8, endpoint=True)
    return build("prefill-8x512", context_lens=cached + 512, q_lens=np.full(8, 512), num_blocks=2048,
                 block_size=16, num_q_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16", seed=seed,
                 poison=poison, max_blocks_per_seq=512)


def prefill_chunks_shape(num_q_heads: int, num_kv_heads: int, head_dim: int, poison: bool = False,
                         seed: int = 1003, name: str = "prefill-shape") -> Workload:
    """The prefill chunks' lengths (8 chunks of 512 new tokens on U[0, 2048]
    cached, the mixed batch's draw) with other head shapes: a GQA group that
    is not a power of two, or head_dim 64.  bf16, block_size 16."""
    g = np.random.Generator(np.random.PCG64(seed + 7_000_000))
    cached = g.integers(0, 2048, size=8, endpoint=True)
    return build(name, context_lens=cached + 512, q_lens=np.full(8, 512), num_blocks=2048, block_size=16,
                 num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim, dtype="bf16", seed=seed,
                 poison=poison, max_blocks_per_seq=512)


def spec_verify(poison: bool = False, seed: int = 1004) -> Workload:
    """Speculative verification, bf16: 32 sequences of 8192 tokens whose last
    5 are draft tokens (causal among themselves); 64 q / 8 kv heads, head_dim
    128, block_size 32, 10240-block pool."""
    B = 32
    return build("specverify-32x5", context_lens=np.full(B, 8192), q_lens=np.full(B, 5),
                 num_blocks=10240, block_size=32, num_q_heads=64, num_kv_heads=8, head_dim=128,
                 dtype="bf16", seed=seed, poison=poison, max_blocks_per_seq=256)


def prefix_shared(poison: bool = False, seed: int = 1005) -> Workload:
    """Prefix-shared decode, bf16: 256 sequences sharing the 128 physical blocks
    of a 2048-token prefix, then private suffixes of U[128, 1024] tokens; one
    decode token each; 32 q / 8 kv heads, head_dim 128, block_size 16."""
    g = np.random.Generator(np.random.PCG64(seed + 7_000_000))
    B = 256
    L = 2048 + g.integers(128, 1024, size=B, endpoint=True)
    return build("prefix-shared-256", context_lens=L, q_lens=np.ones(B, np.int64),
                 num_blocks=20000, block_size=16, num_q_heads=32, num_kv_heads=8, head_dim=128,
                 dtype="bf16", seed=seed, shared_prefix_tokens=2048, poison=poison,
                 max_blocks_per_seq=192)


def prefix_shared_long(poison: bool = False, seed: int = 1006) -> Workload:
    """Long-context variant: 4 sequences of 131072 tokens, the first 2048 in
    shared blocks, one decode token each; 40000-block pool."""
    B = 4
    return build("prefix-shared-long-4x128k", context_lens=np.full(B, 131072),
                 q_lens=np.ones(B, np.int64), num_blocks=40000, block_size=16, num_q_heads=32,
                 num_kv_heads=8, head_dim=128, dtype="bf16", seed=seed,
                 shared_prefix_tokens=2048, poison=poison, max_blocks_per_seq=8192)


def random_small(seed: int, *, dtype: str = "bf16", batch: int = 5, max_ctx: int = 300,
                 max_q: int = 12, num_q_heads: int = 8, num_kv_heads: int = 2,
                 head_dim: int = 128, block_size: int = 16, poison: bool = True,
                 num_blocks: int | None = None, causal: bool = True,
                 allow_empty: bool = True) -> Workload:
    """Random small case: ragged contexts and query lengths (0 allowed)."""
    g = np.random.Generator(np.random.PCG64(seed + 9_000_000))
    L = g.integers(1, max_ctx, size=batch, endpoint=True)
    n = np.minimum(L, g.integers(0 if allow_empty else 1, max_q, size=batch, endpoint=True))
    if not allow_empty:
        n = np.maximum(n, 1)
    nblk = int(np.sum((L + block_size - 1) // block_size))
    return build(f"random-{seed}", context_lens=L, q_lens=n,
                 num_blocks=num_blocks or max(nblk + 7, 2 * nblk), block_size=block_size,
                 num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                 dtype=dtype, seed=seed, poison=poison, causal=causal)


CONFIGS = {
    "tiny": tiny,
    "decode": decode_batch,
    "mixed": mixed_batch,
    "specverify": spec_verify,
    "prefill": prefill_chunks,
    # the same chunks with 56 q / 8 kv heads (G = 7) and with head_dim 64
    "prefill-g7": lambda poison=False, seed=1003: prefill_chunks_shape(56, 8, 128, poison, seed, "prefill-8x512-g7"),
    "prefill-d64": lambda poison=False, seed=1003: prefill_chunks_shape(32, 8, 64, poison, seed, "prefill-8x512-d64"),
    "prefix": prefix_shared,
    "prefix-long": prefix_shared_long,
}
