"""GPU parity of the FP8 (E4M3) cache path.

* paged_kv_write_fp8 is bit-exact against the oracle's encoding (x / scale in
  fp32, nearest E4M3 code with ties to even, saturation at 448), for bf16 and
  fp32 rows over the whole range: saturating, normal and subnormal codes.
* paged_attention_forward_fp8kv equals the fp64 oracle's attention over the
  decoded pools (code * scale), within the bf16 tolerance, on both of its
  kernels (the tensor-core decode kernel when a query-length hint bounds the
  rows by 8, the CUDA-core kernel otherwise): decode, several
  query tokens, prefill chunks, GQA groups 1 to 16, block sizes 8 to 64,
  non-causal, a long split context, and the decode batch at full size on
  sampled sequences.  Unused pool slots hold the NaN code, so a read outside
  a sequence's context shows up.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_236_gb300 as pkv
import workloads as wl
from oracle import fp8
from oracle import paged_oracle as po
from tests.gpu_util import TOL, check_close, to_dev

pytestmark = pytest.mark.gpu


def _u8(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("src", ["bf16", "f32"])
@pytest.mark.parametrize("ks,vs", [(0.01, 0.37), (1.0, 1.0), (3.0, 0.002)])
def test_write_fp8_bit_exact(src, ks, vs):
    rng = np.random.default_rng(int(ks * 1000) + (src == "f32"))
    NB, bs, H, D, T = 24, 16, 4, 128, 70
    mag = rng.choice([1.0, 100.0, 1e-3, 1e-6], size=(T, 1, 1))
    x = (rng.standard_normal((2, T, H, D)) * mag).astype(np.float32)
    if src == "bf16":
        bits = wl.f32_to_bf16_bits(x)
        xf = wl.bf16_bits_to_f64(bits).astype(np.float32)   # exact
        k, v = to_dev(bits[0], "bf16"), to_dev(bits[1], "bf16")
    else:
        xf = x
        k, v = torch.from_numpy(x[0]).cuda(), torch.from_numpy(x[1]).cuda()
    slots = rng.permutation(NB * bs)[:T].astype(np.int64)
    slots[::9] = -1
    kc_h = np.full((NB, bs, H, D), 0xAA, dtype=np.uint8)
    vc_h = kc_h.copy()
    kc, vc = _u8(kc_h), _u8(vc_h)
    pkv.paged_kv_write_fp8(k, v, torch.from_numpy(slots).cuda(), kc, vc, ks, vs)
    fp8.kv_write_fp8(xf[0], xf[1], slots, kc_h, vc_h, ks, vs)
    torch.cuda.synchronize()
    assert np.array_equal(kc.cpu().numpy(), kc_h) and np.array_equal(vc.cpu().numpy(), vc_h)
    assert pkv.device_errors() == 0


class Fp8Run:
    """A bf16 workload's pools encoded to E4M3 by the oracle, on the device
    and on the host; one step written on both sides, then attention."""

    def __init__(self, w: wl.Workload, ks: float, vs: float, blocks=None):
        """blocks: the pool blocks to encode (the rest hold code 0); all by default."""
        self.w, self.ks, self.vs = w, ks, vs
        if blocks is None:
            blocks = np.arange(w.k_cache.shape[0])
        self.kc_h = np.zeros(w.k_cache.shape, dtype=np.uint8)
        self.vc_h = np.zeros(w.v_cache.shape, dtype=np.uint8)
        for a in range(0, len(blocks), 4096):
            b = blocks[a:a + 4096]   # NaN slots -> the NaN code
            self.kc_h[b] = fp8.quantize(wl.bf16_bits_to_f64(w.k_cache[b]).astype(np.float32), ks)
            self.vc_h[b] = fp8.quantize(wl.bf16_bits_to_f64(w.v_cache[b]).astype(np.float32), vs)
        self.kc, self.vc = _u8(self.kc_h), _u8(self.vc_h)

    def step(self, i=0, workspace=None, max_query_len=0):
        st = self.w.steps[i]
        pkv.paged_kv_write_fp8(to_dev(st.k_new, "bf16"), to_dev(st.v_new, "bf16"),
                               torch.from_numpy(st.slot_mapping).cuda(), self.kc, self.vc, self.ks, self.vs)
        fp8.kv_write_fp8(wl.bf16_bits_to_f64(st.k_new).astype(np.float32),
                         wl.bf16_bits_to_f64(st.v_new).astype(np.float32), st.slot_mapping, self.kc_h, self.vc_h,
                         self.ks, self.vs)
        out = pkv.paged_attention_forward_fp8kv(
            to_dev(st.q, "bf16"), self.kc, self.vc, torch.from_numpy(st.block_tables).cuda(),
            torch.from_numpy(st.context_lens).cuda(), torch.from_numpy(st.query_start_loc).cuda(), self.w.scale,
            self.ks, self.vs, self.w.causal, workspace=workspace, max_query_len=max_query_len)
        torch.cuda.synchronize()
        return out

    def check(self, out, i=0, seqs=None, what=""):
        st = self.w.steps[i]
        got = wl.bf16_bits_to_f64(out.view(torch.int16).cpu().numpy().view(np.uint16))
        g, r = [], []
        for s in (range(st.num_seqs) if seqs is None else seqs):
            a, b = int(st.query_start_loc[s]), int(st.query_start_loc[s + 1])
            if b <= a:
                continue
            L = int(st.context_lens[s])
            K = fp8.dequantize(po.gather(self.kc_h, st.block_tables[s], L), self.ks)
            V = fp8.dequantize(po.gather(self.vc_h, st.block_tables[s], L), self.vs)
            g.append(got[a:b])
            r.append(po.attend(wl.to_f64(st.q[a:b], "bf16"), K, V, self.w.scale, self.w.causal))
        return check_close(np.concatenate(g), np.concatenate(r), "bf16", what)


# With a query-length hint that bounds every sequence's rows (tokens x G) by 8
# the tensor-core decode kernel runs (fp16 MMAs over converted tiles): seeds
# 1, 3, 7, 8, 9; the others take the CUDA-core kernel.
@pytest.mark.parametrize("seed,hq,hkv,bs,max_q", [(1, 8, 2, 16, 1), (2, 8, 2, 16, 5), (3, 16, 16, 8, 3),
                                                  (4, 32, 2, 32, 1), (5, 16, 1, 64, 7), (6, 32, 8, 16, 40),
                                                  (7, 16, 8, 64, 4), (8, 32, 8, 32, 2), (9, 8, 8, 16, 1)])
def test_attention_fp8_parity(seed, hq, hkv, bs, max_q):
    w = wl.random_small(seed, batch=6, max_ctx=700, max_q=max_q, num_q_heads=hq, num_kv_heads=hkv,
                        block_size=bs, poison=True)
    run = Fp8Run(w, 0.02, 0.015)
    out = run.step(max_query_len=max_q)
    run.check(out, what=f"fp8 seed {seed}")
    # the written pools are the oracle's, byte for byte
    assert np.array_equal(run.kc.cpu().numpy(), run.kc_h) and np.array_equal(run.vc.cpu().numpy(), run.vc_h)
    assert pkv.device_errors() == 0


def test_attention_fp8_noncausal_and_prefill_chunk():
    w = wl.build("fp8-chunk", context_lens=[300, 97, 1], q_lens=[120, 97, 1], num_blocks=40, block_size=16,
                 num_q_heads=8, num_kv_heads=2, head_dim=128, dtype="bf16", seed=31, poison=True, causal=False)
    run = Fp8Run(w, 1.0, 1.0)
    run.check(run.step(), what="non-causal, prefill chunk")


def test_attention_fp8_long_split_context():
    w = wl.build("fp8-long", context_lens=[20000, 3000], q_lens=[1, 2], num_blocks=1500, block_size=16,
                 num_q_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16", seed=32, poison=True)
    run = Fp8Run(w, 0.01, 0.01)
    run.check(run.step(max_query_len=2), what="long split context")
    # the smallest workspace (no splits) gives the same rows within tolerance
    ws = torch.empty(pkv.workspace_min(2, 3, 32, 8, 128), dtype=torch.uint8, device="cuda")
    run2 = Fp8Run(w, 0.01, 0.01)
    run2.check(run2.step(workspace=ws), what="minimum workspace")


def test_decode_batch_fp8_sampled():
    w = wl.decode_batch(poison=False)
    st = w.step
    seqs = [0, 7, 21, 40, 63]
    blocks = np.unique(np.concatenate([st.block_tables[s][:-(-int(st.context_lens[s]) // w.block_size)]
                                       for s in seqs]))
    run = Fp8Run(w, 4.5 / 448, 4.5 / 448, blocks=blocks)
    out = run.step(max_query_len=1)
    run.check(out, seqs=seqs, what="decode batch (sampled)")
