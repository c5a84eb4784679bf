"""The write of a step's new K/V rows and the attention in one call
(paged_kv_write_attention_forward and its FP8 form): the pools it leaves are
the oracle's write, byte for byte; its output equals the two separate calls'
output bit for bit (every item computes the same rows whichever launch
writes the new rows) and the oracle's within the parity tolerances."""
import numpy as np
import pytest
import torch

import paged_kv_cache_236_gb300 as pkv
import workloads as wl
from gpu_util import DeviceWorkload, check_step, to_dev
from oracle import paged_oracle as po

pytestmark = pytest.mark.gpu


def _bits_dev(t: torch.Tensor) -> np.ndarray:
    """A device pool's bit patterns (NaN poison compares equal to itself)."""
    return t.view(torch.int16 if t.element_size() == 2 else torch.int32).cpu().numpy()


def _bits_host(a: np.ndarray) -> np.ndarray:
    return a.view(np.int16 if a.dtype.itemsize == 2 else np.int32)


def _fused_and_separate(w, max_query_len=0, shared_prefix=False, strided=False):
    """Runs step 0 of w both ways on two copies of the pool; returns the
    fused run's DeviceWorkload (host pool advanced by the oracle's write) and
    both outputs."""
    a, b = DeviceWorkload(w), DeviceWorkload(w)
    st = w.step
    t = a.step_tensors(st)
    k, v = t["k"], t["v"]
    if strided:
        # rows as views into a wider projection output (token stride > Hkv * D)
        T, H, D = k.shape
        wide = torch.zeros(T, 3 * H, D, dtype=k.dtype, device=k.device)
        wide[:, H:2 * H] = k
        wide[:, 2 * H:] = v
        k, v = wide[:, H:2 * H], wide[:, 2 * H:]
    out_f = pkv.paged_kv_write_attention_forward(k, v, t["slots"], t["q"], a.kc, a.vc, t["bt"], t["ctx"], t["qsl"],
                                                 w.scale, w.causal, max_query_len=max_query_len,
                                                 shared_prefix=shared_prefix)
    pkv.paged_kv_write(k, v, t["slots"], b.kc, b.vc)
    out_s = pkv.paged_attention_forward(t["q"], b.kc, b.vc, t["bt"], t["ctx"], t["qsl"], w.scale, w.causal,
                                        max_query_len=max_query_len, shared_prefix=shared_prefix)
    torch.cuda.synchronize()
    po.kv_write(st.k_new, st.v_new, st.slot_mapping, a.kc_host, a.vc_host)
    return a, b, out_f, out_s


CASES = {
    "tiny-fp32": lambda: wl.tiny("1b", poison=True),
    "decode-hint": lambda: wl.build("fused-dec", context_lens=[300, 2100, 17, 950, 4000, 64], q_lens=[1] * 6,
                                    num_blocks=500, block_size=16, num_q_heads=32, num_kv_heads=8, head_dim=128,
                                    dtype="bf16", seed=41, poison=True),
    "mixed": lambda: wl.build("fused-mix", context_lens=[700, 300, 2100, 950, 64], q_lens=[300, 1, 5, 1, 1],
                              num_blocks=320, block_size=16, num_q_heads=16, num_kv_heads=4, head_dim=128,
                              dtype="bf16", seed=42, poison=True),
    "d64-f32": lambda: wl.random_small(43, dtype="f32", batch=5, max_ctx=300, max_q=9, num_q_heads=8,
                                       num_kv_heads=2, head_dim=64, poison=True),
    "prefix-hint": lambda: wl.build("fused-pre", context_lens=[400, 520, 390, 450, 610, 300], q_lens=[1] * 6,
                                    num_blocks=200, block_size=16, num_q_heads=16, num_kv_heads=4, head_dim=128,
                                    dtype="bf16", seed=44, share_groups=[(0, 4, 256)], poison=True),
}


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("strided", [False, True])
def test_fused_write_matches_two_calls(name, strided):
    w = CASES[name]()
    st = w.step
    mql = int(st.q_lens.max()) if name != "mixed" else 0
    a, b, out_f, out_s = _fused_and_separate(w, max_query_len=mql, shared_prefix=name == "prefix-hint",
                                             strided=strided)
    # the pools: the oracle's write, and the same as the separate write's
    assert np.array_equal(_bits_dev(a.kc), _bits_host(a.kc_host))
    assert np.array_equal(_bits_dev(a.vc), _bits_host(a.vc_host))
    assert np.array_equal(_bits_dev(a.kc), _bits_dev(b.kc)) and np.array_equal(_bits_dev(a.vc), _bits_dev(b.vc))
    # the output: bit for bit the two calls', and the oracle's within tolerance
    bits = (lambda x: x.view(torch.int16)) if out_f.dtype == torch.bfloat16 else (lambda x: x.view(torch.int32))
    assert torch.equal(bits(out_f), bits(out_s))
    check_step(a, out_f, what=f"fused {name}")
    assert pkv.device_errors() == 0


def test_fused_write_misaligned_rows_fall_back():
    """Rows whose starts are not 16-byte aligned (an odd token stride) are
    written by the separate write kernel first; the result is the same."""
    w = wl.build("fused-odd", context_lens=[90, 40, 33], q_lens=[3, 1, 2], num_blocks=20, block_size=16,
                 num_q_heads=8, num_kv_heads=2, head_dim=64, dtype="bf16", seed=45, poison=True)
    a = DeviceWorkload(w)
    st = w.step
    t = a.step_tensors(st)
    T, H, D = t["k"].shape
    wide = torch.zeros(T, H * D * 2 + 3, dtype=t["k"].dtype, device="cuda")   # token stride 259 elements
    k = torch.as_strided(wide, (T, H, D), (H * D * 2 + 3, D, 1))
    k.copy_(t["k"])
    v = torch.as_strided(wide, (T, H, D), (H * D * 2 + 3, D, 1), storage_offset=H * D)
    v.copy_(t["v"])
    out = pkv.paged_kv_write_attention_forward(k, v, t["slots"], t["q"], a.kc, a.vc, t["bt"], t["ctx"], t["qsl"],
                                               w.scale, True)
    torch.cuda.synchronize()
    po.kv_write(st.k_new, st.v_new, st.slot_mapping, a.kc_host, a.vc_host)
    assert np.array_equal(_bits_dev(a.kc), _bits_host(a.kc_host))
    assert np.array_equal(_bits_dev(a.vc), _bits_host(a.vc_host))
    check_step(a, out, what="fused, misaligned rows")
    assert pkv.device_errors() == 0


@pytest.mark.parametrize("max_q", [0, 1])
def test_fused_write_fp8(max_q):
    """FP8 pools: the fused call's codes are the oracle's encoding, byte for
    byte, and its output equals the two separate calls'."""
    from test_gpu_fp8 import Fp8Run
    w = wl.build("fused-fp8", context_lens=[300, 45, 700, 1200], q_lens=[1, 1, 1, 1], num_blocks=160, block_size=16,
                 num_q_heads=16, num_kv_heads=4, head_dim=128, dtype="bf16", seed=46, poison=True)
    a = Fp8Run(w, 0.02, 0.015)
    b = Fp8Run(w, 0.02, 0.015)
    st = w.step
    q = to_dev(st.q, "bf16")
    k, v = to_dev(st.k_new, "bf16"), to_dev(st.v_new, "bf16")
    slots = torch.from_numpy(st.slot_mapping).cuda()
    meta = (torch.from_numpy(st.block_tables).cuda(), torch.from_numpy(st.context_lens).cuda(),
            torch.from_numpy(st.query_start_loc).cuda())
    out_f = pkv.paged_kv_write_attention_forward_fp8kv(k, v, slots, q, a.kc, a.vc, *meta, w.scale, a.ks, a.vs,
                                                       True, max_query_len=max_q)
    pkv.paged_kv_write_fp8(k, v, slots, b.kc, b.vc, b.ks, b.vs)
    out_s = pkv.paged_attention_forward_fp8kv(q, b.kc, b.vc, *meta, w.scale, b.ks, b.vs, True, max_query_len=max_q)
    torch.cuda.synchronize()
    from oracle import fp8
    fp8.kv_write_fp8(wl.bf16_bits_to_f64(st.k_new).astype(np.float32), wl.bf16_bits_to_f64(st.v_new).astype(np.float32),
                     st.slot_mapping, a.kc_h, a.vc_h, a.ks, a.vs)
    assert np.array_equal(a.kc.cpu().numpy(), a.kc_h) and np.array_equal(a.vc.cpu().numpy(), a.vc_h)
    assert torch.equal(out_f.view(torch.int16), out_s.view(torch.int16))
    a.check(out_f, what="fused fp8")
    assert pkv.device_errors() == 0
