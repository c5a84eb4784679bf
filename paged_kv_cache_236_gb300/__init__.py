"""Attention over a block-paged KV cache on GB300 (sm_103a).

A thin ctypes binding over the C ABI of ``libpaged_kv.so`` (declared in
``include/paged_kv.h``): argument marshalling only - every step of the path
runs in the library's CUDA kernels.  PyTorch supplies device memory and the
current stream.  There is no CPU fallback: if the library is missing or the
tensors are not on a CUDA device, the calls raise.

    paged_kv_write(k, v, slot_mapping, k_cache, v_cache)
    paged_attention_forward(q, k_cache, v_cache, block_tables, context_lens,
                            query_start_loc, scale, causal)
    paged_kv_write_fp8(k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale)
    paged_attention_forward_fp8kv(q, k_cache, v_cache, ..., scale, k_scale, v_scale)
    BlockManager(num_blocks, block_size, max_blocks_per_seq)   (host, C++)
    copy_blocks(k_cache, v_cache, copies)                      (copy-on-write)

Block pool per layer: ``[num_blocks, block_size, num_kv_heads, head_dim]``
("ADR 004: Paged Attention Serving Integration", Decision 4 - a per-layer
cache tensor; "Paged Attention 基础", section 2 - fixed-size physical
blocks named by block tables).
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

__all__ = [
    "paged_kv_write", "paged_attention_forward", "workspace_size", "workspace_min",
    "device_errors", "debug_fault", "set_profile_events", "set_profile_mid_event", "profile_elapsed_ms", "lib", "LibraryError", "DEVERR",
    "BlockManager", "OutOfBlocks", "copy_blocks", "paged_kv_write_fp8", "paged_attention_forward_fp8kv",
    "paged_kv_write_attention_forward", "paged_kv_write_attention_forward_fp8kv",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpaged_kv.so")

PKV_OK, PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_CUDA, PKV_ERR_WORKSPACE, PKV_ERR_OUT_OF_BLOCKS = range(6)
DTYPE = {torch.float32: 0, torch.bfloat16: 1}
HINT_SHARED_PREFIX = 0x1  # PKV_HINT_SHARED_PREFIX
DEVERR = {
    "slot_out_of_range": 0x1,
    "block_out_of_range": 0x2,
    "bad_sequence": 0x4,
    "timeout": 0x8,
    "plan_overflow": 0x10,
    "internal": 0x20,
}


class LibraryError(RuntimeError):
    """A non-OK status from the C ABI."""

    def __init__(self, status: int, message: str):
        super().__init__(f"paged_kv status {status}: {message}")
        self.status = status


class OutOfBlocks(LibraryError):
    """The block manager's free and evictable blocks do not cover a request
    (``PKV_ERR_OUT_OF_BLOCKS``); the manager is unchanged."""


_lib = None
_lock = threading.Lock()

c_vp, c_i32, c_i64, c_sz, c_f = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with `python -m paged_kv_cache_236_gb300.build` "
                    "(there is no CPU fallback)")
            L = ctypes.CDLL(LIB_PATH)
            L.paged_kv_write.restype = c_i32
            L.paged_kv_write.argtypes = [c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_i32, c_i32, c_i32,
                                         c_i64, c_i64, c_i32, c_vp]
            L.paged_attention_workspace_size.restype = c_sz
            L.paged_attention_workspace_size.argtypes = [c_i32, c_i64, c_i32, c_i32, c_i32]
            L.paged_attention_workspace_min.restype = c_sz
            L.paged_attention_workspace_min.argtypes = [c_i32, c_i64, c_i32, c_i32, c_i32]
            L.paged_attention_forward.restype = c_i32
            L.paged_attention_forward.argtypes = [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i32, c_i64, c_i32,
                                                  c_i32, c_i32, c_i64, c_i32, c_i32, c_i32, c_f, c_i32, c_i32,
                                                  c_vp, c_sz, c_i32, c_vp]
            L.pkv_last_error.restype = ctypes.c_char_p
            L.pkv_last_error.argtypes = []
            L.pkv_device_errors.restype = c_i32
            L.pkv_device_errors.argtypes = [ctypes.POINTER(c_i32), c_i32]
            L.pkv_set_profile_events.restype = None
            L.pkv_set_profile_events.argtypes = [c_vp, c_vp]
            L.pkv_set_profile_mid_event.restype = None
            L.pkv_set_profile_mid_event.argtypes = [c_vp]
            L.pkv_event_elapsed_ms.restype = c_i32
            L.pkv_event_elapsed_ms.argtypes = [c_vp, c_vp, ctypes.POINTER(c_f)]
            L.pkv_version.restype = ctypes.c_char_p
            L.pkv_version.argtypes = []
            L.pkv_debug_fault.restype = c_i32
            L.pkv_debug_fault.argtypes = [c_i32, c_i64]
            L.paged_kv_write_attention_forward.restype = c_i32
            L.paged_kv_write_attention_forward.argtypes = [c_vp, c_vp, c_vp, c_i64, c_i64, c_i64] + \
                L.paged_attention_forward.argtypes
            L.paged_kv_write_attention_forward_fp8kv.restype = c_i32
            L.paged_kv_write_attention_forward_fp8kv.argtypes = [
                c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i32, c_i64,
                c_i32, c_i32, c_i32, c_i64, c_i32, c_i32, c_i32, c_f, c_i32, c_f, c_f, c_i32, c_vp, c_sz, c_vp]
            c_p32 = ctypes.POINTER(c_i32)
            for name, args in (
                    ("pkv_bm_create", [c_i32, c_i32, c_i32, ctypes.POINTER(c_vp)]),
                    ("pkv_bm_update", [c_vp, c_i64, c_i32, c_vp, c_p32, c_p32]),
                    ("pkv_bm_step", [c_vp, c_vp, c_vp, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_p32]),
                    ("pkv_bm_free", [c_vp, c_i64]),
                    ("pkv_bm_fork", [c_vp, c_i64, c_i64]),
                    ("pkv_bm_add_prefix", [c_vp, c_i64, c_vp, c_i32]),
                    ("pkv_bm_try_get_prefix_blocks", [c_vp, c_i64, c_vp, c_i32, c_p32]),
                    ("pkv_bm_block_table", [c_vp, c_i64, c_vp, c_p32, c_p32]),
                    ("pkv_bm_stats", [c_vp, c_p32, c_p32, c_p32, c_p32]),
                    ("paged_kv_copy_blocks", [c_vp, c_vp, c_vp, c_i32, c_i32, c_i64, c_i64, c_i32, c_i32, c_i32,
                                              c_i32, c_vp]),
                    ("paged_kv_write_fp8", [c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_i32, c_i32, c_i32, c_i64,
                                            c_i64, c_i32, c_f, c_f, c_vp]),
                    ("paged_attention_forward_fp8kv", [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i32, c_i64, c_i32,
                                                       c_i32, c_i32, c_i64, c_i32, c_i32, c_i32, c_f, c_i32, c_f,
                                                       c_f, c_i32, c_vp, c_sz, c_vp])):
                getattr(L, name).restype = c_i32
                getattr(L, name).argtypes = args
            L.pkv_bm_destroy.restype = None
            L.pkv_bm_destroy.argtypes = [c_vp]
            _lib = L
    return _lib


def _check(status: int) -> None:
    if status != PKV_OK:
        msg = lib().pkv_last_error().decode(errors="replace")
        raise (OutOfBlocks if status == PKV_ERR_OUT_OF_BLOCKS else LibraryError)(status, msg)


def _stream(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _need_cuda(*tensors: torch.Tensor) -> torch.device:
    dev = tensors[0].device
    for t in tensors:
        if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
            raise ValueError("all tensors must be CUDA tensors (no CPU path)")
        if t.device != dev:
            raise ValueError("all tensors must be on the same device")
    return dev


def paged_kv_write(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, k_cache: torch.Tensor,
                   v_cache: torch.Tensor) -> None:
    """Scatter ``k, v [T, Hkv, D]`` into ``k_cache, v_cache [NB, bs, Hkv, D]``
    at ``slot_mapping [T]`` (int64; slot = block * bs + offset; < 0 skips)."""
    dev = _need_cuda(k, v, slot_mapping, k_cache, v_cache)
    if k_cache.dtype not in DTYPE or k.dtype != k_cache.dtype or v.dtype != k_cache.dtype or \
            v_cache.dtype != k_cache.dtype:
        raise ValueError("k, v, k_cache, v_cache must share dtype bfloat16 or float32")
    if k_cache.dim() != 4 or v_cache.shape != k_cache.shape or not k_cache.is_contiguous() or \
            not v_cache.is_contiguous():
        raise ValueError("caches must be contiguous [num_blocks, block_size, num_kv_heads, head_dim]")
    NB, bs, Hkv, D = k_cache.shape
    T = k.shape[0]
    for name, t in (("k", k), ("v", v)):
        if t.dim() != 3 or tuple(t.shape[1:]) != (Hkv, D) or t.stride(2) != 1 or t.stride(1) != D:
            raise ValueError(f"{name} must be [T, {Hkv}, {D}] with contiguous heads")
    if v.shape[0] != T or slot_mapping.shape != (T,) or slot_mapping.dtype != torch.int64 or \
            not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be contiguous int64 [T]")
    with torch.cuda.device(dev):
        _check(lib().paged_kv_write(k.data_ptr(), v.data_ptr(), slot_mapping.data_ptr(), k_cache.data_ptr(),
                                    v_cache.data_ptr(), T, NB, bs, Hkv, D, k.stride(0) if T else 0,
                                    v.stride(0) if T else 0, DTYPE[k_cache.dtype], _stream(dev)))


def workspace_size(num_seqs: int, num_tokens: int, num_q_heads: int, num_kv_heads: int, head_dim: int) -> int:
    return int(lib().paged_attention_workspace_size(num_seqs, num_tokens, num_q_heads, num_kv_heads, head_dim))


def workspace_min(num_seqs: int, num_tokens: int, num_q_heads: int, num_kv_heads: int, head_dim: int) -> int:
    return int(lib().paged_attention_workspace_min(num_seqs, num_tokens, num_q_heads, num_kv_heads, head_dim))


_ws_cache: dict = {}


def _workspace(dev: torch.device, nbytes: int) -> torch.Tensor:
    key = (dev.index, torch.cuda.current_stream(dev).cuda_stream)
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
        _ws_cache[key] = ws
    return ws


def paged_attention_forward(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                            block_tables: torch.Tensor, context_lens: torch.Tensor,
                            query_start_loc: torch.Tensor, scale: float, causal: bool = True, *,
                            out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                            max_query_len: int = 0, shared_prefix: bool = False) -> torch.Tensor:
    """Varlen attention of ``q [T, Hq, D]`` through per-sequence block tables.

    ``context_lens[s]`` counts sequence s's tokens after this step's write
    (its query tokens included); query i of n sits at position L - n + i.
    ``workspace`` (uint8, >= ``workspace_min``) defaults to a cached buffer
    per (device, stream).  ``max_query_len`` is an optional host hint.
    ``shared_prefix`` tells the call that consecutive sequences may start
    with the same physical blocks (prefix caching): runs of them then read
    their common prefix once (``PKV_HINT_SHARED_PREFIX``).
    """
    dev = _need_cuda(q, k_cache, v_cache, block_tables, context_lens, query_start_loc)
    args, out = _forward_args(q, k_cache, v_cache, block_tables, context_lens, query_start_loc, scale, causal, out,
                              workspace, max_query_len, shared_prefix, dev)
    with torch.cuda.device(dev):
        _check(lib().paged_attention_forward(*args))
    return out


def _forward_args(q, k_cache, v_cache, block_tables, context_lens, query_start_loc, scale, causal, out, workspace,
                  max_query_len, shared_prefix, dev) -> tuple:
    """Checks paged_attention_forward's tensors; returns (its C arguments, out)."""
    if q.dtype not in DTYPE or k_cache.dtype != q.dtype or v_cache.dtype != q.dtype:
        raise ValueError("q, k_cache, v_cache must share dtype bfloat16 or float32")
    if q.dim() != 3 or not q.is_contiguous():
        raise ValueError("q must be contiguous [T, Hq, D]")
    if k_cache.dim() != 4 or v_cache.shape != k_cache.shape or not k_cache.is_contiguous() or \
            not v_cache.is_contiguous():
        raise ValueError("caches must be contiguous [num_blocks, block_size, num_kv_heads, head_dim]")
    T, Hq, D = q.shape
    NB, bs, Hkv, Dk = k_cache.shape
    if Dk != D:
        raise ValueError("head_dim of q and the caches differ")
    B = context_lens.shape[0]
    for name, t, shape in (("block_tables", block_tables, None), ("context_lens", context_lens, (B,)),
                           ("query_start_loc", query_start_loc, (B + 1,))):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous int32")
        if shape is not None and tuple(t.shape) != shape:
            raise ValueError(f"{name} must have shape {shape}")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or (B > 0 and block_tables.shape[1] == 0):
        raise ValueError("block_tables must be [num_seqs, max_blocks_per_seq] with max_blocks_per_seq > 0")
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous() or out.device != dev:
        raise ValueError("out must match q")
    with torch.cuda.device(dev):
        need = workspace_min(B, T, Hq, Hkv, D)
        if workspace is None:
            workspace = _workspace(dev, workspace_size(B, T, Hq, Hkv, D))
        if workspace.dtype != torch.uint8 or workspace.device != dev or workspace.numel() < need:
            raise ValueError(f"workspace must be a uint8 CUDA tensor of at least {need} bytes")
    args = (q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(), context_lens.data_ptr(),
            query_start_loc.data_ptr(), out.data_ptr(), B, T, Hq, Hkv, D, NB, bs, max(1, block_tables.shape[1]),
            int(max_query_len), float(scale), 1 if causal else 0, HINT_SHARED_PREFIX if shared_prefix else 0,
            workspace.data_ptr(), workspace.numel(), DTYPE[q.dtype], _stream(dev))
    return args, out


def _new_rows(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, Hkv: int, D: int, dtypes) -> tuple:
    """Checks a step's new K/V rows [T, Hkv, D] (contiguous heads) and returns
    (T, k token stride, v token stride)."""
    if k.dtype not in dtypes or v.dtype != k.dtype:
        raise ValueError("k and v must share a dtype the pools accept")
    T = k.shape[0]
    for name, t in (("k", k), ("v", v)):
        if t.dim() != 3 or tuple(t.shape[1:]) != (Hkv, D) or t.stride(2) != 1 or t.stride(1) != D:
            raise ValueError(f"{name} must be [T, {Hkv}, {D}] with contiguous heads")
    if v.shape[0] != T or slot_mapping.shape != (T,) or slot_mapping.dtype != torch.int64 or \
            not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be contiguous int64 [T]")
    return T, (k.stride(0) if T else 0), (v.stride(0) if T else 0)


def paged_kv_write_attention_forward(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                                     q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                     block_tables: torch.Tensor, context_lens: torch.Tensor,
                                     query_start_loc: torch.Tensor, scale: float, causal: bool = True, *,
                                     out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                                     max_query_len: int = 0, shared_prefix: bool = False) -> torch.Tensor:
    """``paged_kv_write(k, v, slot_mapping, k_cache, v_cache)`` then
    ``paged_attention_forward(q, k_cache, v_cache, ...)`` in one call: the
    new rows are written by extra CTAs of the planner's launch (one launch
    fewer per step).  Same arguments and result as the two calls."""
    dev = _need_cuda(k, v, slot_mapping, q, k_cache, v_cache, block_tables, context_lens, query_start_loc)
    Tn, ks, vs = _new_rows(k, v, slot_mapping, k_cache.shape[2], k_cache.shape[3], {k_cache.dtype})
    args, out = _forward_args(q, k_cache, v_cache, block_tables, context_lens, query_start_loc, scale, causal, out,
                              workspace, max_query_len, shared_prefix, dev)
    with torch.cuda.device(dev):
        _check(lib().paged_kv_write_attention_forward(k.data_ptr(), v.data_ptr(), slot_mapping.data_ptr(), Tn, ks, vs,
                                                      *args))
    return out


def set_profile_events(start, stop) -> None:
    """Record ``start``/``stop`` (torch.cuda.Event) around the attention
    kernels of later forward calls on this thread; ``None, None`` stops."""
    if start is None or stop is None:
        lib().pkv_set_profile_events(None, None)
    else:
        lib().pkv_set_profile_events(start.cuda_event, stop.cuda_event)


def set_profile_mid_event(mid) -> None:
    """Also record ``mid`` (torch.cuda.Event) right after the multi-token
    tensor-core kernel of later forward calls on this thread; ``None`` stops."""
    lib().pkv_set_profile_mid_event(None if mid is None else mid.cuda_event)


def profile_elapsed_ms(start, stop) -> float:
    """Milliseconds between two events recorded through ``set_profile_events``."""
    ms = c_f(0.0)
    _check(lib().pkv_event_elapsed_ms(start.cuda_event, stop.cuda_event, ctypes.byref(ms)))
    return float(ms.value)


def debug_fault(fault_tile: int, wait_ns: int) -> None:
    """Testing hook (``pkv_debug_fault``): arm the next forward call of this
    thread to give up its waits after ``wait_ns`` ns and, with
    ``fault_tile`` >= 1, to skip the loads of one key tile in one CTA, so
    that the bounded waits run out."""
    _check(lib().pkv_debug_fault(int(fault_tile), int(wait_ns)))


def device_errors(clear: bool = True) -> int:
    """Sticky device error bits (``DEVERR``) of the current device; synchronises."""
    flags = c_i32(0)
    _check(lib().pkv_device_errors(ctypes.byref(flags), 1 if clear else 0))
    return int(flags.value)


# ----------------------------------------------------------------------------
# host block manager (include/paged_kv_blocks.h)
# ----------------------------------------------------------------------------

def _host(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=dtype))


class BlockManager:
    """The library's host block manager: block ids, slots and tables for a
    pool of ``num_blocks`` blocks of ``block_size`` tokens ("Paged Attention
    基础", section 3.1 C; "ADR 004", Decision 5 and Consequences).

    ``update(seq, n)`` -> (slots int64 [n], copies int32 [c, 2]);
    ``step(seq_ids, n_new)`` -> dict of the call metadata (host numpy
    arrays: slot_mapping, block_tables, context_lens, query_start_loc,
    copies); ``free``, ``fork``, ``add_prefix``, ``try_get_prefix_blocks``,
    ``block_table``, ``stats``.  Refused requests raise ``OutOfBlocks`` or
    ``LibraryError`` and change nothing.
    """

    def __init__(self, num_blocks: int, block_size: int, max_blocks_per_seq: int):
        h = c_vp()
        _check(lib().pkv_bm_create(num_blocks, block_size, max_blocks_per_seq, ctypes.byref(h)))
        self._h = h
        self.num_blocks, self.block_size, self.max_blocks = num_blocks, block_size, max_blocks_per_seq

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value and _lib is not None:
            try:
                _lib.pkv_bm_destroy(h)
            except Exception:  # interpreter shutdown: the library may be gone already
                pass
            self._h = None

    def update(self, seq: int, n: int):
        slots = np.empty(max(n, 0), dtype=np.int64)
        pair = (c_i32 * 2)()
        nc = c_i32(0)
        _check(lib().pkv_bm_update(self._h, int(seq), int(n), slots.ctypes.data if n > 0 else None, pair,
                                   ctypes.byref(nc)))
        return slots, np.asarray(list(pair)[:2 * nc.value], dtype=np.int32).reshape(-1, 2)

    def step(self, seq_ids, n_new, reuse: bool = False) -> dict:
        """One batch step (``pkv_bm_step``): the call metadata as host numpy
        arrays.  With ``reuse=True`` they are views into buffers the manager
        keeps, valid until its next ``step(..., reuse=True)``; this saves the
        per-call allocations of a serving loop."""
        ids = _host(seq_ids, np.int64)
        n = _host(n_new, np.int32)
        B = len(ids)
        if len(n) != B:
            raise ValueError("seq_ids and n_new differ in length")
        total = int(n.sum(dtype=np.int64)) if B else 0
        if reuse:
            bufs = self._buffers(B, total)
            out = {k: v for k, v in bufs["arrays"].items()}
            ptr = bufs["ptr"]
            nc = bufs["nc"]
            _check(lib().pkv_bm_step(self._h, ids.ctypes.data if B else None, n.ctypes.data if B else None, B,
                                     ptr["slot_mapping"], ptr["block_tables"], ptr["context_lens"],
                                     ptr["query_start_loc"], ptr["copies"], ctypes.byref(nc)))
            return {"slot_mapping": out["slot_mapping"][:total], "block_tables": out["block_tables"][:B],
                    "context_lens": out["context_lens"][:B], "query_start_loc": out["query_start_loc"][:B + 1],
                    "copies": out["copies"][:nc.value]}
        out = {
            "slot_mapping": np.empty(max(total, 0), dtype=np.int64),
            "block_tables": np.empty((B, self.max_blocks), dtype=np.int32),
            "context_lens": np.empty(B, dtype=np.int32),
            "query_start_loc": np.empty(B + 1, dtype=np.int32),
            "copies": np.empty((max(B, 1), 2), dtype=np.int32),
        }
        nc = c_i32(0)
        ptr = lambda a: a.ctypes.data if a.size else None
        _check(lib().pkv_bm_step(self._h, ptr(ids), ptr(n), B, ptr(out["slot_mapping"]), ptr(out["block_tables"]),
                                 ptr(out["context_lens"]), out["query_start_loc"].ctypes.data,
                                 out["copies"].ctypes.data, ctypes.byref(nc)))
        out["copies"] = out["copies"][:nc.value]
        return out

    def _buffers(self, B: int, total: int) -> dict:
        """Output buffers of at least B sequences and `total` new tokens,
        grown geometrically, with their addresses computed once."""
        b = getattr(self, "_bufs", None)
        if b is None or b["B"] < B or b["T"] < total:
            cb = max(B, 2 * b["B"] if b else 64, 1)
            ct = max(total, 2 * b["T"] if b else 256, 1)
            arrays = {
                "slot_mapping": np.empty(ct, dtype=np.int64),
                "block_tables": np.empty((cb, self.max_blocks), dtype=np.int32),
                "context_lens": np.empty(cb, dtype=np.int32),
                "query_start_loc": np.empty(cb + 1, dtype=np.int32),
                "copies": np.empty((cb, 2), dtype=np.int32),
            }
            b = {"B": cb, "T": ct, "arrays": arrays, "nc": c_i32(0),
                 "ptr": {k: a.ctypes.data for k, a in arrays.items()}}
            self._bufs = b
        return b

    def free(self, seq: int) -> None:
        _check(lib().pkv_bm_free(self._h, int(seq)))

    def fork(self, parent: int, child: int) -> None:
        _check(lib().pkv_bm_fork(self._h, int(parent), int(child)))

    def add_prefix(self, seq: int, tokens) -> None:
        t = _host(tokens, np.int64)
        _check(lib().pkv_bm_add_prefix(self._h, int(seq), t.ctypes.data if t.size else None, len(t)))

    def try_get_prefix_blocks(self, seq: int, tokens) -> int:
        t = _host(tokens, np.int64)
        got = c_i32(0)
        _check(lib().pkv_bm_try_get_prefix_blocks(self._h, int(seq), t.ctypes.data if t.size else None, len(t),
                                                  ctypes.byref(got)))
        return int(got.value)

    def block_table(self, seq: int) -> list:
        table = np.empty(self.max_blocks, dtype=np.int32)
        nb, nt = c_i32(0), c_i32(0)
        _check(lib().pkv_bm_block_table(self._h, int(seq), table.ctypes.data, ctypes.byref(nb), ctypes.byref(nt)))
        return table[:nb.value].tolist()

    def num_tokens(self, seq: int) -> int:
        nt = c_i32(0)
        _check(lib().pkv_bm_block_table(self._h, int(seq), None, None, ctypes.byref(nt)))
        return int(nt.value)

    def stats(self) -> dict:
        f, i, u, c = c_i32(0), c_i32(0), c_i32(0), c_i32(0)
        _check(lib().pkv_bm_stats(self._h, ctypes.byref(f), ctypes.byref(i), ctypes.byref(u), ctypes.byref(c)))
        return {"free": f.value, "idle": i.value, "in_use": u.value, "cached": c.value}


def copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, copies) -> None:
    """Copy-on-write on the device pool: block ``dst`` of every layer's K and
    V pool becomes a copy of block ``src`` for each host pair (src, dst) of
    ``copies`` (int32 [n, 2], as ``BlockManager.update`` / ``step`` return).
    Caches are ``[NB, bs, Hkv, D]`` or ``[layers, NB, bs, Hkv, D]`` (each
    layer's pool contiguous).  Runs on the current stream."""
    dev = _need_cuda(k_cache, v_cache)
    pairs = _host(copies, np.int32).reshape(-1, 2)
    if k_cache.dtype not in DTYPE or v_cache.dtype != k_cache.dtype or v_cache.shape != k_cache.shape or \
            v_cache.stride() != k_cache.stride():
        raise ValueError("k_cache and v_cache must share dtype (bfloat16 or float32), shape and strides")
    if k_cache.dim() == 4:
        layers, stride = 1, 0
        pool = k_cache
    elif k_cache.dim() == 5:
        layers, stride = k_cache.shape[0], k_cache.stride(0)
        pool = k_cache[0]
    else:
        raise ValueError("caches must be [NB, bs, Hkv, D] or [layers, NB, bs, Hkv, D]")
    if not pool.is_contiguous():
        raise ValueError("each layer's pool must be contiguous")
    NB, bs, Hkv, D = pool.shape
    with torch.cuda.device(dev):
        _check(lib().paged_kv_copy_blocks(k_cache.data_ptr(), v_cache.data_ptr(),
                                          pairs.ctypes.data if len(pairs) else None, len(pairs), layers, stride,
                                          NB, bs, Hkv, D, DTYPE[k_cache.dtype], _stream(dev)))


# ----------------------------------------------------------------------------
# FP8 (E4M3) pools (include/paged_kv.h: paged_kv_write_fp8,
# paged_attention_forward_fp8kv)
# ----------------------------------------------------------------------------

_FP8_TYPES = {torch.uint8} | ({torch.float8_e4m3fn} if hasattr(torch, "float8_e4m3fn") else set())


def _check_fp8_pools(k_cache: torch.Tensor, v_cache: torch.Tensor) -> None:
    if k_cache.dtype not in _FP8_TYPES or v_cache.dtype != k_cache.dtype:
        raise ValueError("FP8 pools must be uint8 (E4M3 codes) or float8_e4m3fn tensors")
    if k_cache.dim() != 4 or v_cache.shape != k_cache.shape or not k_cache.is_contiguous() or \
            not v_cache.is_contiguous():
        raise ValueError("caches must be contiguous [num_blocks, block_size, num_kv_heads, head_dim]")


def paged_kv_write_fp8(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, k_cache: torch.Tensor,
                       v_cache: torch.Tensor, k_scale: float, v_scale: float) -> None:
    """Encode ``k, v [T, Hkv, D]`` (bf16 or f32) as E4M3 codes of x / scale
    and scatter them into the FP8 pools at ``slot_mapping`` (< 0 skips)."""
    dev = _need_cuda(k, v, slot_mapping, k_cache, v_cache)
    _check_fp8_pools(k_cache, v_cache)
    if k.dtype not in DTYPE or v.dtype != k.dtype:
        raise ValueError("k and v must share dtype bfloat16 or float32")
    NB, bs, Hkv, D = k_cache.shape
    T = k.shape[0]
    for name, t in (("k", k), ("v", v)):
        if t.dim() != 3 or tuple(t.shape[1:]) != (Hkv, D) or t.stride(2) != 1 or t.stride(1) != D:
            raise ValueError(f"{name} must be [T, {Hkv}, {D}] with contiguous heads")
    if v.shape[0] != T or slot_mapping.shape != (T,) or slot_mapping.dtype != torch.int64 or \
            not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be contiguous int64 [T]")
    with torch.cuda.device(dev):
        _check(lib().paged_kv_write_fp8(k.data_ptr(), v.data_ptr(), slot_mapping.data_ptr(), k_cache.data_ptr(),
                                        v_cache.data_ptr(), T, NB, bs, Hkv, D, k.stride(0) if T else 0,
                                        v.stride(0) if T else 0, DTYPE[k.dtype], float(k_scale), float(v_scale),
                                        _stream(dev)))


def paged_attention_forward_fp8kv(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                  block_tables: torch.Tensor, context_lens: torch.Tensor,
                                  query_start_loc: torch.Tensor, scale: float, k_scale: float, v_scale: float,
                                  causal: bool = True, *, out: torch.Tensor | None = None,
                                  workspace: torch.Tensor | None = None, max_query_len: int = 0) -> torch.Tensor:
    """``paged_attention_forward`` over FP8 pools read as code * k_scale and
    code * v_scale; q and the result are bf16, head_dim 128."""
    dev = _need_cuda(q, k_cache, v_cache, block_tables, context_lens, query_start_loc)
    args, out = _fp8_forward_args(q, k_cache, v_cache, block_tables, context_lens, query_start_loc, scale, k_scale,
                                  v_scale, causal, out, workspace, max_query_len, dev)
    with torch.cuda.device(dev):
        _check(lib().paged_attention_forward_fp8kv(*args))
    return out


def paged_kv_write_attention_forward_fp8kv(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                                           q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                           block_tables: torch.Tensor, context_lens: torch.Tensor,
                                           query_start_loc: torch.Tensor, scale: float, k_scale: float,
                                           v_scale: float, causal: bool = True, *, out: torch.Tensor | None = None,
                                           workspace: torch.Tensor | None = None,
                                           max_query_len: int = 0) -> torch.Tensor:
    """``paged_kv_write_fp8`` of a step's new rows (bf16 or f32) then
    ``paged_attention_forward_fp8kv``, in one call (the rows are encoded by
    extra CTAs of the planner's launch)."""
    dev = _need_cuda(k, v, slot_mapping, q, k_cache, v_cache, block_tables, context_lens, query_start_loc)
    _check_fp8_pools(k_cache, v_cache)
    Tn, ks, vs = _new_rows(k, v, slot_mapping, k_cache.shape[2], k_cache.shape[3], set(DTYPE))
    args, out = _fp8_forward_args(q, k_cache, v_cache, block_tables, context_lens, query_start_loc, scale, k_scale,
                                  v_scale, causal, out, workspace, max_query_len, dev)
    with torch.cuda.device(dev):
        _check(lib().paged_kv_write_attention_forward_fp8kv(k.data_ptr(), v.data_ptr(), slot_mapping.data_ptr(), Tn,
                                                            ks, vs, DTYPE[k.dtype], *args))
    return out


def _fp8_forward_args(q, k_cache, v_cache, block_tables, context_lens, query_start_loc, scale, k_scale, v_scale,
                      causal, out, workspace, max_query_len, dev) -> tuple:
    """Checks paged_attention_forward_fp8kv's tensors; returns (its C arguments, out)."""
    _check_fp8_pools(k_cache, v_cache)
    if q.dtype != torch.bfloat16 or q.dim() != 3 or not q.is_contiguous():
        raise ValueError("q must be contiguous bfloat16 [T, Hq, D]")
    T, Hq, D = q.shape
    NB, bs, Hkv, Dk = k_cache.shape
    if Dk != D:
        raise ValueError("head_dim of q and the caches differ")
    B = context_lens.shape[0]
    for name, t, shape in (("block_tables", block_tables, None), ("context_lens", context_lens, (B,)),
                           ("query_start_loc", query_start_loc, (B + 1,))):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous int32")
        if shape is not None and tuple(t.shape) != shape:
            raise ValueError(f"{name} must have shape {shape}")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or (B > 0 and block_tables.shape[1] == 0):
        raise ValueError("block_tables must be [num_seqs, max_blocks_per_seq] with max_blocks_per_seq > 0")
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous() or out.device != dev:
        raise ValueError("out must match q")
    with torch.cuda.device(dev):
        need = workspace_min(B, T, Hq, Hkv, D)
        if workspace is None:
            workspace = _workspace(dev, workspace_size(B, T, Hq, Hkv, D))
        if workspace.dtype != torch.uint8 or workspace.device != dev or workspace.numel() < need:
            raise ValueError(f"workspace must be a uint8 CUDA tensor of at least {need} bytes")
    args = (q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(), context_lens.data_ptr(),
            query_start_loc.data_ptr(), out.data_ptr(), B, T, Hq, Hkv, D, NB, bs, max(1, block_tables.shape[1]),
            int(max_query_len), float(scale), 1 if causal else 0, float(k_scale), float(v_scale), 0,
            workspace.data_ptr(), workspace.numel(), _stream(dev))
    return args, out
