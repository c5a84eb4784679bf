"""Failure detection on the device without a GPU fault: a bounded in-kernel
wait is made to run out, through the testing hook ``pkv_debug_fault``, which
makes one CTA's K/V producer skip the loads of one key tile (nothing else is
wrong: no bad address, no trap).  The call must come back with
PKV_DEVERR_TIMEOUT set, after about the short limit given rather than the
default 2 s, and the next ordinary call on the same device must match the
fp64 oracle."""
import time

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
