"""A max_query_len hint smaller than the batch's longest query only costs
speed: the planner routes rows by the kernels that actually launch, so longer
sequences are split into more decode-kernel items (bf16 and FP8 pools)."""
import numpy as np
import pytest
import torch

import paged_kv_cache_236_gb300 as pkv
import workloads as wl
from oracle import fp8
from oracle import paged_oracle as po
from tests.gpu_util import DeviceWorkload, check_close, check_step, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seed", [11, 12])
def test_too_small_hint_bf16(seed):
    w = wl.random_small(seed, batch=6, max_ctx=600, max_q=5, num_q_heads=16, num_kv_heads=4, poison=True,
                        allow_empty=False)
    assert int(w.step.q_lens.max()) > 1
    dw = DeviceWorkload(w)
    out = dw.run_step(0, max_query_len=1)
    check_step(dw, out, 0, what="bf16, hint below the longest query")


def test_too_small_hint_fp8():
    w = wl.random_small(13, batch=6, max_ctx=600, max_q=5, num_q_heads=16, num_kv_heads=4, poison=True,
                        allow_empty=False)
    st, ks, vs = w.step, 0.02, 0.015
    f32 = lambda bits: wl.bf16_bits_to_f64(bits).astype(np.float32)
    kh, vh = fp8.quantize(f32(w.k_cache), ks), fp8.quantize(f32(w.v_cache), vs)
    kc = torch.from_numpy(kh).cuda()
    vc = torch.from_numpy(vh).cuda()
    pkv.paged_kv_write_fp8(to_dev(st.k_new, "bf16"), to_dev(st.v_new, "bf16"), torch.from_numpy(st.slot_mapping).cuda(),
                           kc, vc, ks, vs)
    fp8.kv_write_fp8(f32(st.k_new), f32(st.v_new), st.slot_mapping, kh, vh, ks, vs)
    out = pkv.paged_attention_forward_fp8kv(to_dev(st.q, "bf16"), kc, vc, torch.from_numpy(st.block_tables).cuda(),
                                            torch.from_numpy(st.context_lens).cuda(),
                                            torch.from_numpy(st.query_start_loc).cuda(), w.scale, ks, vs, True,
                                            max_query_len=1)
    ref = po.paged_attention(wl.to_f64(st.q, "bf16"), fp8.dequantize(kh, ks), fp8.dequantize(vh, vs), st.block_tables,
                             st.context_lens, st.query_start_loc, w.scale, True)
    got = wl.bf16_bits_to_f64(out.view(torch.int16).cpu().numpy().view(np.uint16))
    check_close(got, ref, "bf16", "fp8, hint below the longest query")
    assert pkv.device_errors() == 0
