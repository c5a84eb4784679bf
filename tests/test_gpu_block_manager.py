"""GPU parity of the cache-manager path: the block copy (copy-on-write) is a
bit-exact block copy, and a serving loop run through the library's C++ block
manager gives, at every step, the attention the fp64 oracle computes on each
sequence's logical (unpaged) K/V rows.

The loop follows "ADR 004: Paged Attention Serving Integration"
(Consequences: one update call for prefill and decode; Limitations: a cached
prompt prefix replayed with add_prefix / try_get_prefix_blocks) and
"Paged Attention 基础", section 1, problem 3 (requests sharing a system
prompt share its blocks): prompts whose system prompt was cached start on
its blocks, a forked sequence copies the shared partly filled block before
appending, and the steps mix prefill, decode and 3-token verification."""
import numpy as np
import pytest
import torch

import paged_kv_cache_236_gb300 as pkv
import workloads as wl
from oracle import paged_oracle as po
from tests.gpu_util import TOL
from workloads.block_ops import kv_rows_normal

pytestmark = pytest.mark.gpu


def _bits(x: np.ndarray) -> np.ndarray:
    return wl.f32_to_bf16_bits(x)


def _dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _host_bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("dtype,layered,n_pairs", [("bf16", False, 7), ("f32", False, 5), ("bf16", True, 9),
                                                   ("bf16", False, 600), ("bf16", False, 4100)])
def test_copy_blocks_bit_exact(dtype, layered, n_pairs):
    rng = np.random.default_rng(40 + n_pairs)
    NB, bs, H, D, layers = max(1400, 2 * n_pairs + 8), 16, 4, 64 if dtype == "f32" else 128, 3
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    shape = (layers, NB + 5, bs, H, D) if layered else (NB, bs, H, D)
    k = torch.randn(shape, dtype=torch.float32).to(tdt).cuda()
    v = torch.randn(shape, dtype=torch.float32).to(tdt).cuda()
    if layered:                                  # each layer's pool contiguous, layer stride > one pool
        k, v = k[:, :NB], v[:, :NB]
    perm = rng.permutation(NB)
    pairs = np.stack([perm[:n_pairs], perm[n_pairs:2 * n_pairs]], axis=1).astype(np.int32)
    pairs[0] = [0, NB - 1] if 0 not in pairs[1:] and NB - 1 not in pairs[1:] else pairs[0]
    k_ref, v_ref = k.cpu().clone(), v.cpu().clone()
    for s, d in pairs:
        k_ref[..., d, :, :, :] = k_ref[..., s, :, :, :]
        v_ref[..., d, :, :, :] = v_ref[..., s, :, :, :]
    pkv.copy_blocks(k, v, pairs)
    torch.cuda.synchronize()
    for got, ref in ((k, k_ref), (v, v_ref)):
        g = got.cpu()
        if tdt == torch.bfloat16:
            assert torch.equal(g.view(torch.int16), ref.view(torch.int16))
        else:
            assert torch.equal(g.view(torch.int32), ref.view(torch.int32))
    assert pkv.device_errors() == 0


class Loop:
    """A pool on the device, the C++ manager, and each sequence's logical
    tokens, K/V rows (bf16 bits) for the oracle."""

    def __init__(self, NB=600, bs=16, Hq=16, Hkv=4, D=128, max_blocks=64, seed=7):
        self.NB, self.bs, self.Hq, self.Hkv, self.D = NB, bs, Hq, Hkv, D
        self.m = pkv.BlockManager(NB, bs, max_blocks)
        self.kc = torch.full((NB, bs, Hkv, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        self.vc = torch.full((NB, bs, Hkv, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        self.tokens: dict[int, list[int]] = {}
        self.k_rows: dict[int, np.ndarray] = {}
        self.v_rows: dict[int, np.ndarray] = {}
        self.rng = np.random.default_rng(seed)
        self.scale = 1.0 / np.sqrt(D)

    def _rows(self, s):
        w = self.Hkv * self.D
        self.k_rows[s] = _bits(kv_rows_normal(self.tokens[s], w, 1)).reshape(-1, self.Hkv, self.D)
        self.v_rows[s] = _bits(kv_rows_normal(self.tokens[s], w, 2)).reshape(-1, self.Hkv, self.D)

    def prompt(self, s, toks) -> int:
        """Starts s on the cached blocks of its prompt; returns the tokens left."""
        cached = self.m.try_get_prefix_blocks(s, toks)
        self.tokens[s] = list(toks)
        self._rows(s)
        self.pending = getattr(self, "pending", {})
        self.pending[s] = cached
        return len(toks) - cached

    def step(self, ids, new_tokens, shared_prefix) -> dict:
        """new_tokens[i]: tokens appended to ids[i] (for prompts started with
        `prompt`, None: the rest of the prompt)."""
        n_new, starts = [], []
        for s, t in zip(ids, new_tokens):
            if t is None:
                start = self.pending.pop(s)
                n = len(self.tokens[s]) - start
            else:
                start = len(self.tokens[s])
                self.tokens[s] = self.tokens[s] + list(t)
                self._rows(s)
                n = len(t)
            n_new.append(n)
            starts.append(start)
        meta = self.m.step(ids, n_new)
        pkv.copy_blocks(self.kc, self.vc, meta["copies"])
        knew = np.concatenate([self.k_rows[s][a:a + n] for s, a, n in zip(ids, starts, n_new)])
        vnew = np.concatenate([self.v_rows[s][a:a + n] for s, a, n in zip(ids, starts, n_new)])
        T = knew.shape[0]
        q = _bits(self.rng.standard_normal((T, self.Hq, self.D), dtype=np.float32))
        pkv.paged_kv_write(_dev_bf16(knew), _dev_bf16(vnew), torch.from_numpy(meta["slot_mapping"]).cuda(),
                           self.kc, self.vc)
        out = pkv.paged_attention_forward(
            _dev_bf16(q), self.kc, self.vc, torch.from_numpy(meta["block_tables"]).cuda(),
            torch.from_numpy(meta["context_lens"]).cuda(), torch.from_numpy(meta["query_start_loc"]).cuda(),
            float(self.scale), True, max_query_len=max(n_new), shared_prefix=shared_prefix)
        got = wl.bf16_bits_to_f64(_host_bits(out))
        qf = wl.bf16_bits_to_f64(q)
        qsl = meta["query_start_loc"]
        for i, s in enumerate(ids):
            a, b = qsl[i], qsl[i + 1]
            if a == b:
                continue
            ref = po.attend(qf[a:b], wl.bf16_bits_to_f64(self.k_rows[s]), wl.bf16_bits_to_f64(self.v_rows[s]),
                            self.scale, True)
            err = np.abs(got[a:b] - ref)
            assert err.max() <= TOL["bf16"][0] and err.mean() <= TOL["bf16"][1], (s, err.max(), err.mean())
        return meta

    def check_pool(self):
        """Every live sequence's rows, read through its table on the device
        pool, are its logical rows, bit for bit."""
        kc, vc = _host_bits(self.kc), _host_bits(self.vc)
        for s, toks in self.tokens.items():
            table = np.asarray(self.m.block_table(s))
            assert np.array_equal(po.gather(kc, table, len(toks)), self.k_rows[s]), s
            assert np.array_equal(po.gather(vc, table, len(toks)), self.v_rows[s]), s


@pytest.mark.parametrize("shared_prefix", [False, True])
def test_serving_loop_through_the_block_manager(shared_prefix):
    L = Loop()
    rng = np.random.default_rng(3)
    tok = lambda n: [int(t) for t in rng.integers(0, 50, size=n)]
    sys0, sys1 = tok(300), tok(70)                 # 18 (4) full blocks of 16
    # 1: the two system prompts' first requests, prefilled whole
    for s, p in ((1, sys0 + tok(20)), (2, sys1 + tok(9))):
        assert L.prompt(s, p) == len(p)
    L.step([1, 2], [None, None], shared_prefix)
    L.m.add_prefix(1, L.tokens[1])
    L.m.add_prefix(2, L.tokens[2])
    # 2: later requests start on the cached system-prompt blocks; 1 and 2 decode
    left = {}
    for s, base in ((3, sys0), (4, sys0), (5, sys0), (6, sys0), (8, sys0), (9, sys1)):
        p = base + tok(int(rng.integers(5, 60)))
        left[s] = L.prompt(s, p)
        assert len(p) - left[s] == (len(base) // 16) * 16      # the system prompt's full blocks
    blocks = lambda n: -(-n // 16)
    # shared blocks are named again, not taken: only the tails and growth take blocks
    want = L.m.stats()["in_use"] + sum(blocks(len(L.tokens[s])) - (len(L.tokens[s]) - n) // 16
                                       for s, n in left.items())
    want += sum(blocks(len(L.tokens[s]) + 1) - blocks(len(L.tokens[s])) for s in (1, 2))
    L.step([1, 3, 4, 5, 6, 8, 2, 9], [tok(1), None, None, None, None, None, tok(1), None], shared_prefix)
    assert L.m.stats()["in_use"] == want
    L.check_pool()
    # 3: a fork shares seq 3's partly filled last block; both append: one copy
    L.m.fork(3, 7)
    L.tokens[7], L.k_rows[7], L.v_rows[7] = list(L.tokens[3]), L.k_rows[3], L.v_rows[3]
    order = [1, 3, 7, 4, 5, 6, 8, 2, 9]
    partial = len(L.tokens[3]) % 16 != 0
    meta = L.step(order, [tok(1) for _ in order], shared_prefix)
    assert len(meta["copies"]) == (1 if partial else 0)
    L.check_pool()
    # 4-6: decode, 3-token verification windows, decode
    for n in (1, 3, 1):
        L.step(order, [tok(n) for _ in order], shared_prefix)
    L.check_pool()
    # a finished request frees its blocks; the cached prefix survives it
    L.m.free(4)
    del L.tokens[4]
    L.step([1, 3, 7], [tok(2), tok(1), tok(1)], shared_prefix)
    L.check_pool()
    torch.cuda.synchronize()
    assert pkv.device_errors() == 0
