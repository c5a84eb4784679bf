"""paged_kv_write on the GPU against the oracle's write: bit-exact."""
import numpy as np
import pytest
import torch

import paged_kv_cache_236_gb300 as pkv
import workloads as wl
from oracle import paged_oracle as po
from gpu_util import to_dev, to_host_bits

pytestmark = pytest.mark.gpu


def _pool_equal(a, b):
    return np.array_equal(a.view(np.uint8) if a.dtype != np.uint8 else a, b.view(np.uint8) if b.dtype != np.uint8 else b)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("seed", range(4))
def test_write_bit_exact(dtype, seed):
    w = wl.random_small(seed, dtype=dtype, batch=6, max_ctx=200, max_q=40, head_dim=128 if seed % 2 else 64,
                        block_size=[8, 16, 32, 64][seed], poison=True)
    st = w.step
    kc, vc = to_dev(w.k_cache, dtype), to_dev(w.v_cache, dtype)
    pkv.paged_kv_write(to_dev(st.k_new, dtype), to_dev(st.v_new, dtype), torch.from_numpy(st.slot_mapping).cuda(),
                       kc, vc)
    kr, vr = w.k_cache.copy(), w.v_cache.copy()
    po.kv_write(st.k_new, st.v_new, st.slot_mapping, kr, vr)
    assert _pool_equal(to_host_bits(kc), kr) and _pool_equal(to_host_bits(vc), vr)
    assert pkv.device_errors() == 0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_write_strided_views_and_skips(dtype):
    """k and v as views into a fused [T, 3, Hkv, D] projection output; some
    slots are -1 (padding) and must be skipped."""
    g = np.random.Generator(np.random.PCG64(5))
    T, Hkv, D, NB, bs = 37, 4, 64, 20, 16
    fused = wl.normal_values(np.random.SeedSequence(9), T * 3 * Hkv * D, dtype).reshape(T, 3, Hkv, D)
    slots = g.permutation(NB * bs)[:T].astype(np.int64)
    slots[[3, 10, 11]] = -1
    pool = wl._empty_pool(NB, bs, Hkv, D, dtype, poison=True)
    fd = to_dev(fused, dtype)
    kc, vc = to_dev(pool, dtype), to_dev(pool, dtype)
    pkv.paged_kv_write(fd[:, 1], fd[:, 2], torch.from_numpy(slots).cuda(), kc, vc)
    kr, vr = pool.copy(), pool.copy()
    po.kv_write(fused[:, 1], fused[:, 2], slots, kr, vr)
    assert _pool_equal(to_host_bits(kc), kr) and _pool_equal(to_host_bits(vc), vr)


def test_write_out_of_range_slot_is_flagged_not_written():
    dtype = "bf16"
    T, Hkv, D, NB, bs = 4, 2, 64, 3, 16
    k = wl.normal_values(np.random.SeedSequence(1), T * Hkv * D, dtype).reshape(T, Hkv, D)
    slots = np.array([0, NB * bs, 5, NB * bs + 100], np.int64)   # two past the pool's end
    pool = np.zeros((NB, bs, Hkv, D), np.uint16)
    kc, vc = to_dev(pool, dtype), to_dev(pool, dtype)
    pkv.device_errors(clear=True)
    pkv.paged_kv_write(to_dev(k, dtype), to_dev(k, dtype), torch.from_numpy(slots).cuda(), kc, vc)
    flags = pkv.device_errors(clear=True)
    assert flags & pkv.DEVERR["slot_out_of_range"]
    kr = pool.copy()
    po.kv_write(k[[0, 2]], k[[0, 2]], slots[[0, 2]], kr, kr.copy())
    assert np.array_equal(to_host_bits(kc), kr)


def test_write_mixed_batch_rows():
    """The mixed serving batch's 4216 new tokens: every written pool row equals
    its token's row."""
    w = wl.mixed_batch()
    st = w.step
    dtype = w.dtype
    kc, vc = to_dev(w.k_cache, dtype), to_dev(w.v_cache, dtype)
    pkv.paged_kv_write(to_dev(st.k_new, dtype), to_dev(st.v_new, dtype), torch.from_numpy(st.slot_mapping).cuda(),
                       kc, vc)
    bs = w.block_size
    sl = torch.from_numpy(st.slot_mapping).cuda()
    krows = kc.view(-1, w.num_kv_heads, w.head_dim)[sl]
    vrows = vc.view(-1, w.num_kv_heads, w.head_dim)[sl]
    assert np.array_equal(to_host_bits(krows), st.k_new)
    assert np.array_equal(to_host_bits(vrows), st.v_new)
    # a sample of untouched rows kept their old contents
    g = np.random.Generator(np.random.PCG64(3))
    other = np.setdiff1d(g.integers(0, w.num_blocks * bs, 4096), st.slot_mapping)
    ot = torch.from_numpy(other).cuda()
    assert np.array_equal(to_host_bits(kc.view(-1, w.num_kv_heads, w.head_dim)[ot]),
                          w.k_cache.reshape(-1, w.num_kv_heads, w.head_dim)[other])
