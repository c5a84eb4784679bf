"""The serving workloads at full size, in the launch configuration the
benchmark times: every row of sampled sequences against the fp64 oracle
(first, last and seeded random picks)."""
import numpy as np
import pytest

import paged_kv_cache_236_gb300 as pkv
import workloads as wl
from gpu_util import DeviceWorkload, check_step

pytestmark = pytest.mark.gpu


def _sample(B, k, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    picks = {0, B - 1} | set(g.choice(B, size=min(B, k), replace=False).tolist())
    return sorted(picks)


@pytest.mark.parametrize("name", ["decode", "mixed", "specverify", "prefix", "prefix-long"])
def test_config_sampled(name):
    w = wl.CONFIGS[name]()
    dw = DeviceWorkload(w)
    st = w.step
    out = dw.run_step(0, max_query_len=int(st.q_lens.max()))
    seqs = _sample(st.num_seqs, 6, 11)
    if name == "mixed":
        seqs = sorted(set(seqs) | {0, 3, 7, 8})   # prefill chunks and decodes
    check_step(dw, out, seqs=seqs, what=name)
    assert pkv.device_errors() == 0
