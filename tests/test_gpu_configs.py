"""The serving workloads at full size, in the launch configuration the
benchmark times (the same query-length hint and shared-prefix hint): every
output row of every sequence against the fp64 oracle.

Covered: the decode batch, the mixed continuous batch, speculative
verification, the prefix-shared decode batch and its long-context variant
(each prefix case with and without the shared-prefix hint), and the decode
batch over FP8 (E4M3) pools.
"""
import numpy as np
import pytest

import paged_kv_cache_236_gb300 as pkv
import workloads as wl
from gpu_util import DeviceWorkload, check_step

pytestmark = pytest.mark.gpu

RUNS = [("decode", False), ("mixed", False), ("specverify", False), ("prefix", True), ("prefix", False),
        ("prefix-long", True), ("prefix-long", False)]


@pytest.mark.parametrize("name,shared_prefix", RUNS)
def test_config_all_rows(name, shared_prefix):
    w = wl.CONFIGS[name]()
    dw = DeviceWorkload(w)
    st = w.step
    out = dw.run_step(0, max_query_len=int(st.q_lens.max()), shared_prefix=shared_prefix)
    check_step(dw, out, what=f"{name} (shared-prefix hint {shared_prefix})")
    assert pkv.device_errors() == 0


def test_decode_batch_fp8_all_rows():
    """The decode batch with both pools as E4M3 codes (one scale per pool,
    4.5/448, as the benchmark uses), through the tensor-core decode kernel
    (query-length hint 1): every row against the oracle over the decoded
    pools."""
    from test_gpu_fp8 import Fp8Run
    w = wl.decode_batch(poison=False)
    st = w.step
    used = np.unique(np.concatenate([st.block_tables[s][:-(-int(st.context_lens[s]) // w.block_size)]
                                     for s in range(st.num_seqs)]))
    run = Fp8Run(w, 4.5 / 448, 4.5 / 448, blocks=used)
    out = run.step(max_query_len=1)
    run.check(out, what="decode batch, FP8 pools")
    assert pkv.device_errors() == 0
