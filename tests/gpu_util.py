"""Helpers for the GPU parity tests: move seeded workloads to the device, run
the library (write then attention), and compute expected rows with the fp64
oracle on the CPU from the same inputs."""
from __future__ import annotations

import numpy as np
import torch

import paged_kv_cache_236_gb300 as pkv
import workloads as wl
from oracle import paged_oracle as po

# max-abs, mean-abs error bounds against the fp64 oracle
TOL = {"bf16": (2e-2, 2e-3), "f32": (1e-4, 1e-4)}


def to_dev(a: np.ndarray, dtype: str, dev="cuda") -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(a).to(dev)


def to_host_bits(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def to_f64(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return wl.bf16_bits_to_f64(to_host_bits(t))
    return t.double().cpu().numpy()


class DeviceWorkload:
    """A workload's pool on the device plus a host copy kept in step with the
    oracle's own write."""

    def __init__(self, w: wl.Workload, dev="cuda"):
        self.w = w
        self.dev = dev
        self.kc = to_dev(w.k_cache, w.dtype, dev)
        self.vc = to_dev(w.v_cache, w.dtype, dev)
        self.kc_host = w.k_cache.copy()
        self.vc_host = w.v_cache.copy()

    def step_tensors(self, st: wl.Step) -> dict:
        d = self.dev
        return dict(q=to_dev(st.q, self.w.dtype, d), k=to_dev(st.k_new, self.w.dtype, d),
                    v=to_dev(st.v_new, self.w.dtype, d), slots=torch.from_numpy(st.slot_mapping).to(d),
                    bt=torch.from_numpy(st.block_tables).to(d), ctx=torch.from_numpy(st.context_lens).to(d),
                    qsl=torch.from_numpy(st.query_start_loc).to(d))

    def run_step(self, i: int = 0, *, workspace=None, max_query_len: int = 0,
                 shared_prefix: bool = False) -> torch.Tensor:
        st = self.w.steps[i]
        t = self.step_tensors(st)
        pkv.paged_kv_write(t["k"], t["v"], t["slots"], self.kc, self.vc)
        po.kv_write(st.k_new, st.v_new, st.slot_mapping, self.kc_host, self.vc_host)
        out = pkv.paged_attention_forward(t["q"], self.kc, self.vc, t["bt"], t["ctx"], t["qsl"], self.w.scale,
                                          self.w.causal, workspace=workspace, max_query_len=max_query_len,
                                          shared_prefix=shared_prefix)
        torch.cuda.synchronize()
        return out

    def oracle_rows(self, i: int, seqs) -> dict:
        """Expected output rows (fp64) of the given sequences of step i."""
        st = self.w.steps[i]
        res = {}
        for s in seqs:
            a, b = int(st.query_start_loc[s]), int(st.query_start_loc[s + 1])
            L = int(st.context_lens[s])
            if b <= a:
                continue
            K = wl.to_f64(po.gather(self.kc_host, st.block_tables[s], L), self.w.dtype)
            V = wl.to_f64(po.gather(self.vc_host, st.block_tables[s], L), self.w.dtype)
            q = wl.to_f64(st.q[a:b], self.w.dtype)
            res[s] = (a, b, po.attend(q, K, V, self.w.scale, self.w.causal))
        return res


def check_close(got: np.ndarray, want: np.ndarray, dtype: str, what: str = "") -> tuple[float, float]:
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - want)
    mx, mean = float(err.max(initial=0.0)), float(err.mean()) if err.size else 0.0
    tmax, tmean = TOL[dtype]
    assert mx <= tmax and mean <= tmean, f"{what}: max abs {mx:.3g} (<= {tmax}), mean abs {mean:.3g} (<= {tmean})"
    return mx, mean


def check_step(dw: DeviceWorkload, out: torch.Tensor, i: int = 0, seqs=None, what: str = ""):
    st = dw.w.steps[i]
    if seqs is None:
        seqs = range(st.num_seqs)
    got = to_f64(out)
    rows = dw.oracle_rows(i, seqs)
    g, r = [], []
    for s, (a, b, ref) in rows.items():
        g.append(got[a:b])
        r.append(ref)
    if not g:
        return 0.0, 0.0
    return check_close(np.concatenate(g), np.concatenate(r), dw.w.dtype, what)
