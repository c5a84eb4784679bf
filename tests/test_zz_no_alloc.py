"""The forward entry point that allocates nothing.

Some callers cannot give the library a workspace: they run under an
allocator that refuses new device allocations once started, or can only
pass through buffers that another component registered.  For them,
paged_attention_forward_static_ws uses a scratch array built into the
library.  This test calls it through the C ABI twice in a row, with no host
synchronisation between the two calls, and checks each result against the
regular entry point (which gets a caller-allocated workspace) and against
the fp64 oracle, within the parity tolerances used everywhere else; it also
checks that a batch too large for the built-in scratch is refused before any
launch.

Named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_236_gb300 as pkv
import workloads as wl
from gpu_util import DeviceWorkload, check_close, check_step, to_f64
from oracle import paged_oracle as po

pytestmark = pytest.mark.gpu

c_vp, c_i32, c_i64, c_f = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float


def _entry():
    f = pkv.lib().paged_attention_forward_static_ws
    f.restype = c_i32
    f.argtypes = [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i32, c_i64, c_i32, c_i32, c_i32, c_i64, c_i32, c_i32,
                  c_i32, c_f, c_i32, c_i32, c_i32, c_vp]
    return f


def _call(f, t, kc, vc, out, w, T, max_q):
    NB, bs, Hkv, D = kc.shape
    return f(t["q"].data_ptr(), kc.data_ptr(), vc.data_ptr(), t["bt"].data_ptr(), t["ctx"].data_ptr(),
             t["qsl"].data_ptr(), out.data_ptr(), t["ctx"].shape[0], T, w.num_q_heads, Hkv, D, NB, bs,
             t["bt"].shape[1], max_q, w.scale, 1 if w.causal else 0, 0, 1 if w.dtype == "bf16" else 0,
             torch.cuda.current_stream().cuda_stream)


def test_static_scratch_matches_workspace_entry_point():
    # a long context (split-KV partial rows live in the scratch), decode rows,
    # and a multi-token chunk (tensor-core path)
    w = wl.build("no-alloc", context_lens=[9000, 300, 1200, 64, 2500], q_lens=[1, 1, 40, 3, 1], num_blocks=900,
                 block_size=16, num_q_heads=16, num_kv_heads=4, head_dim=128, dtype="bf16", seed=77, poison=True)
    dw = DeviceWorkload(w)
    st = w.step
    t = dw.step_tensors(st)
    pkv.paged_kv_write(t["k"], t["v"], t["slots"], dw.kc, dw.vc)
    po.kv_write(st.k_new, st.v_new, st.slot_mapping, dw.kc_host, dw.vc_host)
    ref = pkv.paged_attention_forward(t["q"], dw.kc, dw.vc, t["bt"], t["ctx"], t["qsl"], w.scale, w.causal)
    torch.cuda.synchronize()
    ref64 = to_f64(ref)
    f = _entry()
    # two calls in a row on one stream, the second issued while the first may
    # still run (both share the one static scratch)
    outs = [torch.full_like(t["q"], float("nan")) for _ in range(2)]
    for call in range(2):
        status = _call(f, t, dw.kc, dw.vc, outs[call], w, st.num_tokens, 0)
        assert status == 0, pkv.lib().pkv_last_error()
    torch.cuda.synchronize()
    for call in range(2):
        check_close(to_f64(outs[call]), ref64, "bf16", f"static scratch, call {call}")
        check_step(dw, outs[call], what=f"static scratch against the oracle, call {call}")
    assert pkv.device_errors() == 0


def test_static_scratch_rejects_oversized_batch():
    f = _entry()
    cap = pkv.lib().paged_attention_static_workspace_bytes
    cap.restype = ctypes.c_size_t
    assert cap() == 8 << 20
    T = 400_000   # the work lists alone would exceed the built-in scratch
    assert pkv.workspace_min(4, T, 32, 8, 128) > cap()
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    p = dummy.data_ptr()
    status = f(p, p, p, p, p, p, p, 4, T, 32, 8, 128, 16, 16, 1, 0, 0.1, 1, 0, 1,
               torch.cuda.current_stream().cuda_stream)
    assert status == pkv.PKV_ERR_WORKSPACE
    assert b"static scratch" in pkv.lib().pkv_last_error()
