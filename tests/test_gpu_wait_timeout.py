"""Failure detection on the device without a GPU fault: a bounded in-kernel
wait is made to run out, through the testing hook ``pkv_debug_fault``, which
makes one CTA's K/V producer skip the loads of one key tile (nothing else is
wrong: no bad address, no trap).  The call must come back with
PKV_DEVERR_TIMEOUT set, after about the short limit given rather than the
default 2 s, and the next ordinary call on the same device must match the
fp64 oracle."""
import time

import numpy as np
import pytest
import torch

import paged_kv_cache_236_gb300 as pkv
import workloads as wl
from gpu_util import DeviceWorkload, check_step

pytestmark = pytest.mark.gpu

LIMIT_NS = 50_000_000  # 50 ms


def _run_with_fault(dw, fault_tile, **kw):
    st = dw.w.step
    t = dw.step_tensors(st)
    pkv.device_errors(clear=True)
    pkv.debug_fault(fault_tile, LIMIT_NS)
    t0 = time.perf_counter()
    pkv.paged_attention_forward(t["q"], dw.kc, dw.vc, t["bt"], t["ctx"], t["qsl"], dw.w.scale, True, **kw)
    flags = pkv.device_errors(clear=True)  # synchronises
    return flags, time.perf_counter() - t0


@pytest.mark.parametrize("fault_tile", [1, 2, 5])
def test_cuda_core_decode_wait_runs_out(fault_tile):
    """bf16, head_dim 64: the CUDA-core decode kernel (one producer warp,
    four consumer warps that agree on every tile before going on)."""
    w = wl.build("timeout-decode", context_lens=[3000 - 17 * i for i in range(48)], q_lens=[1] * 48,
                 num_blocks=48 * 188 + 8, block_size=16, num_q_heads=8, num_kv_heads=2, head_dim=64, dtype="bf16",
                 seed=71, poison=True)
    dw = DeviceWorkload(w)
    out = dw.run_step(0)  # writes the step's rows (host copy too) and checks nothing yet
    check_step(dw, out, what="before the fault")
    flags, secs = _run_with_fault(dw, fault_tile)
    assert flags & pkv.DEVERR["timeout"], f"no timeout recorded (flags {flags:#x})"
    assert secs < 1.5, f"the call took {secs:.2f} s: the short limit was not used"
    # the device is still usable: an ordinary call gives the oracle's rows
    st = w.step
    t = dw.step_tensors(st)
    out = pkv.paged_attention_forward(t["q"], dw.kc, dw.vc, t["bt"], t["ctx"], t["qsl"], w.scale, True)
    torch.cuda.synchronize()
    check_step(dw, out, what="after the fault")
    assert pkv.device_errors() == 0


def _decode_batch(seed):
    return wl.build("timeout-tc", context_lens=[2600 - 13 * i for i in range(64)], q_lens=[1] * 64,
                    num_blocks=64 * 163 + 8, block_size=16, num_q_heads=32, num_kv_heads=8, head_dim=128,
                    dtype="bf16", seed=seed, poison=True)


@pytest.mark.parametrize("fault_tile", [1, 2, 4])
def test_tensor_core_decode_wait_runs_out(fault_tile):
    """bf16, head_dim 128 with the query-length hint: the tensor-core decode
    kernel (K and V producers, item fetch, the MMA thread, four softmax and
    four epilogue warps that settle every wait across the group)."""
    dw = DeviceWorkload(_decode_batch(72))
    out = dw.run_step(0, max_query_len=1)
    check_step(dw, out, what="before the fault")
    flags, secs = _run_with_fault(dw, fault_tile, max_query_len=1)
    assert flags & pkv.DEVERR["timeout"], f"no timeout recorded (flags {flags:#x})"
    assert secs < 1.5, f"the call took {secs:.2f} s: the short limit was not used"
    st = dw.w.step
    t = dw.step_tensors(st)
    out = pkv.paged_attention_forward(t["q"], dw.kc, dw.vc, t["bt"], t["ctx"], t["qsl"], dw.w.scale, True,
                                      max_query_len=1)
    torch.cuda.synchronize()
    check_step(dw, out, what="after the fault")
    assert pkv.device_errors() == 0


@pytest.mark.parametrize("fault_tile", [1, 3])
def test_tensor_core_decode_fp8_wait_runs_out(fault_tile):
    """FP8 pools with the query-length hint: the same kernel with its K and V
    converter warps between the staged codes and the MMAs."""
    from test_gpu_fp8 import Fp8Run
    run = Fp8Run(_decode_batch(73), 0.02, 0.015)
    run.check(run.step(max_query_len=1), what="before the fault")
    st = run.w.step
    q = torch.from_numpy(st.q.view(np.int16)).cuda().view(torch.bfloat16)
    args = (q, run.kc, run.vc, torch.from_numpy(st.block_tables).cuda(), torch.from_numpy(st.context_lens).cuda(),
            torch.from_numpy(st.query_start_loc).cuda(), run.w.scale, run.ks, run.vs, True)
    pkv.device_errors(clear=True)
    pkv.debug_fault(fault_tile, LIMIT_NS)
    t0 = time.perf_counter()
    pkv.paged_attention_forward_fp8kv(*args, max_query_len=1)
    flags = pkv.device_errors(clear=True)
    secs = time.perf_counter() - t0
    assert flags & pkv.DEVERR["timeout"], f"no timeout recorded (flags {flags:#x})"
    assert secs < 1.5, f"the call took {secs:.2f} s"
    out = pkv.paged_attention_forward_fp8kv(*args, max_query_len=1)
    torch.cuda.synchronize()
    run.check(out, what="after the fault")
    assert pkv.device_errors() == 0


def _prefill_batch(seed, head_dim):
    # eight chunks of 384 new tokens after 1,500-1,800 cached ones: every CTA
    # of the multi-token kernel works on items of 13 to 17 key tiles
    ctx = [1900 + 40 * i for i in range(8)]
    return wl.build("timeout-mma", context_lens=ctx, q_lens=[384] * 8, num_blocks=sum((c + 15) // 16 for c in ctx) + 8,
                    block_size=16, num_q_heads=8, num_kv_heads=2, head_dim=head_dim, dtype="bf16", seed=seed,
                    poison=True)


@pytest.mark.parametrize("head_dim", [128, 64])
@pytest.mark.parametrize("fault_tile", [1, 2, 5])
def test_tensor_core_prefill_wait_runs_out(head_dim, fault_tile):
    """bf16 prefill chunks: the multi-token tensor-core kernel (item fetch
    and output stores, K and V producers, the Q K^T and P.V issuers, eight
    softmax / epilogue warps that settle failed waits pairwise and then all
    together before the stores)."""
    dw = DeviceWorkload(_prefill_batch(74 + head_dim, head_dim))
    out = dw.run_step(0)
    check_step(dw, out, what="before the fault")
    flags, secs = _run_with_fault(dw, fault_tile)
    assert flags & pkv.DEVERR["timeout"], f"no timeout recorded (flags {flags:#x})"
    assert secs < 1.5, f"the call took {secs:.2f} s: the short limit was not used"
    st = dw.w.step
    t = dw.step_tensors(st)
    out = pkv.paged_attention_forward(t["q"], dw.kc, dw.vc, t["bt"], t["ctx"], t["qsl"], dw.w.scale, True)
    torch.cuda.synchronize()
    check_step(dw, out, what="after the fault")
    assert pkv.device_errors() == 0
