"""Shared prefixes read once per run of sequences (PKV_HINT_SHARED_PREFIX)
against the fp64 oracle.  The hint changes how keys are read, never the
result: runs that qualify (at least four consecutive decode-shaped sequences
on the same leading blocks), runs too short to qualify, prefixes that end
inside a 128-key tile, suffixes long enough to be split, prefill chunks in
the same batch, and paths that ignore the hint."""
import numpy as np
import pytest
import torch

import paged_kv_cache_236_gb300 as pkv
import workloads as wl
from gpu_util import DeviceWorkload, check_close, check_step, to_f64

pytestmark = pytest.mark.gpu


def _runs_case(seed, *, bs=16, hq=32, hkv=8, qmax=1, suffix=(1, 900), extra=(), dtype="bf16"):
    """40 sequences: a run of 10 on a 608-token prefix (4 whole tiles + 96
    keys), 3 on 512 tokens (too few to qualify), 17 on 1024 tokens, 5 on 256
    tokens, the rest private; then `extra` (context, q_len) sequences."""
    g = np.random.Generator(np.random.PCG64(seed + 31_000_000))
    B0 = 40
    groups = [(a, b, tok // bs * bs) for a, b, tok in [(0, 9, 608), (10, 12, 512), (13, 29, 1024), (33, 37, 256)]]
    share = np.zeros(B0, np.int64)
    for a, b, tok in groups:
        share[a:b + 1] = tok
    n = g.integers(1, qmax, size=B0, endpoint=True)
    L = share + n + g.integers(suffix[0], suffix[1], size=B0, endpoint=True)
    L = np.concatenate([L, [c for c, _ in extra]]).astype(np.int64)
    n = np.concatenate([n, [q for _, q in extra]]).astype(np.int64)
    nblk = int(np.sum((L + bs - 1) // bs))
    return wl.build(f"runs-{seed}", context_lens=L, q_lens=n, num_blocks=nblk + 64, block_size=bs,
                    num_q_heads=hq, num_kv_heads=hkv, head_dim=128, dtype=dtype, seed=seed,
                    share_groups=groups, poison=True)


def _check_both(w, **kw):
    dw = DeviceWorkload(w)
    out = dw.run_step(0, shared_prefix=True, **kw)
    check_step(dw, out, what=f"{w.name} with the hint")
    assert pkv.device_errors() == 0
    # the same call without the hint: same attention (both against the oracle,
    # and close to each other)
    dw2 = DeviceWorkload(w)
    out2 = dw2.run_step(0, shared_prefix=False, **kw)
    check_step(dw2, out2, what=f"{w.name} without the hint")
    check_close(to_f64(out), to_f64(out2), w.dtype, "with vs without the hint")


@pytest.mark.parametrize("bs,hq,hkv,qmax", [(16, 32, 8, 1), (32, 32, 8, 4), (16, 32, 4, 2), (64, 16, 8, 1)])
def test_runs_match_oracle(bs, hq, hkv, qmax):
    _check_both(_runs_case(101 + bs + qmax, bs=bs, hq=hq, hkv=hkv, qmax=qmax))


def test_runs_with_max_query_len_hint():
    # a decode-only length hint does not turn the shared-prefix path off
    w = _runs_case(211)
    _check_both(w, max_query_len=1)


def test_runs_with_long_suffixes_split():
    # suffixes of ~20k keys are split over several items; the merge folds in
    # the prefix partials as well
    _check_both(_runs_case(223, suffix=(15000, 22000)))


def test_runs_beside_prefill_chunks():
    # multi-token sequences (tensor-core items) in the same call as the
    # prefix items; they never join a run
    _check_both(_runs_case(227, qmax=2, extra=[(900, 300), (2500, 512), (700, 1)]))


def test_hint_ignored_off_the_tensor_core_decode_path():
    # fp32 takes the CUDA-core kernels, which read every key per sequence
    _check_both(_runs_case(229, dtype="f32", hq=8, hkv=2))


def test_prefix_config_with_hint_sampled():
    w = wl.CONFIGS["prefix"]()
    dw = DeviceWorkload(w)
    out = dw.run_step(0, max_query_len=1, shared_prefix=True)
    g = np.random.Generator(np.random.PCG64(17))
    B = w.step.num_seqs
    seqs = sorted({0, 1, 2, 3, B - 1} | set(g.choice(B, size=8, replace=False).tolist()))
    check_step(dw, out, seqs=seqs, what="prefix config, shared-prefix hint")
    assert pkv.device_errors() == 0


def test_many_short_runs():
    # 600 sequences in runs of 5 on their own 256-token prefixes: more groups
    # than the planner shares out cooperatively, one item list per group
    g = np.random.Generator(np.random.PCG64(41))
    B, run, tok = 600, 5, 256
    groups = [(a, a + run - 1, tok) for a in range(0, B, run)]
    n = np.ones(B, np.int64)
    L = tok + n + g.integers(1, 300, size=B, endpoint=True)
    nblk = int(np.sum((L + 15) // 16))
    w = wl.build("many-runs", context_lens=L, q_lens=n, num_blocks=nblk + 64, block_size=16, num_q_heads=32,
                 num_kv_heads=8, head_dim=128, dtype="bf16", seed=43, share_groups=groups, poison=True)
    _check_both(w)


def test_prefix_rows_beyond_a_small_workspace():
    # with the smallest workspace the prefix partial rows may not fit: the call
    # then reads every key per sequence (or fewer prefix chunks), same result
    w = _runs_case(233)
    st = w.step
    ws = torch.empty(pkv.workspace_min(st.num_seqs, st.num_tokens, w.num_q_heads, w.num_kv_heads, w.head_dim),
                     dtype=torch.uint8, device="cuda")
    dw = DeviceWorkload(w)
    out = dw.run_step(0, shared_prefix=True, workspace=ws)
    check_step(dw, out, what="shared-prefix hint, minimum workspace")
    assert pkv.device_errors() == 0
