"""FP8 (E4M3) KV-cache encoding: the reference definition.

TEST INFRASTRUCTURE.  Only ``tests/`` and the CPU legs of ``bench.py`` may
import this module; the CUDA library never calls it and shares no code with
it.

The pages give no quantised cache format (they name block pools of K/V rows
and nothing about their precision), so this is the library's own format,
stated here from its definition:

* Element: the OCP 8-bit floating point format E4M3 ("e4m3fn"): 1 sign bit, 4
  exponent bits with bias 7, 3 mantissa bits.  Exponent field 0 holds
  subnormals m/8 * 2^-6; fields 1..15 hold (1 + m/8) * 2^(e-7), except
  S.1111.111, which is NaN (no infinities).  Largest finite value 448.
* Encoding of a real x given a scale: q = x / scale in IEEE fp32 (as the
  kernel divides), then rounded to the nearest E4M3 value, ties to the even
  mantissa; magnitudes beyond 448 saturate to +-448 ("satfinite"); NaN stays
  NaN.
* Decoding: the code's value times the scale, exact in fp64.

Functions: ``e4m3_value`` (code -> value), ``e4m3_encode`` (fp32 -> code),
``quantize`` (rows and a scale -> codes), ``dequantize`` (codes and a scale ->
fp64), ``kv_write_fp8`` (the quantising slot-mapping scatter).
"""
from __future__ import annotations

import numpy as np

__all__ = ["E4M3_MAX", "e4m3_value", "e4m3_encode", "quantize", "dequantize", "kv_write_fp8"]

E4M3_MAX = 448.0


def e4m3_value(code: int) -> float:
    """The real value of an 8-bit E4M3 code (NaN for S.1111.111)."""
    code = int(code) & 0xFF
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)
# finite non-negative codes in increasing value order (0x00 .. 0x7E)
_POS = np.arange(0x7F)
_POS_VAL = _TABLE[_POS]


def e4m3_encode(x) -> np.ndarray:
    """Nearest E4M3 code of each fp32 value (ties to the even mantissa,
    i.e. the even code), saturating at +-448; NaN -> 0x7F."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    nan = np.isnan(x)
    sign = np.where(np.signbit(x), 0x80, 0)
    a = np.minimum(np.abs(np.where(nan, 0.0, x)), E4M3_MAX)
    # the neighbouring codes: hi = the first with value >= a, lo = the one below
    hi = np.minimum(np.searchsorted(_POS_VAL, a, side="left"), len(_POS_VAL) - 1)
    lo = np.maximum(hi - 1, 0)
    dlo, dhi = a - _POS_VAL[lo], _POS_VAL[hi] - a
    tie_even = np.where(lo % 2 == 0, lo, hi)   # codes alternate mantissa parity
    c = np.where(dhi == 0, hi, np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, tie_even)))
    return np.where(nan, 0x7F, sign | c).astype(np.uint8)


def quantize(x, scale: float) -> np.ndarray:
    """Codes of x / scale (the division in fp32, as the kernel does).
    Large arrays are encoded in slices (memory only; every element is
    independent)."""
    x = np.asarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    flat, res = x.reshape(-1), out.reshape(-1)
    step = 1 << 22
    for a in range(0, flat.size, step):
        res[a:a + step] = e4m3_encode((flat[a:a + step] / np.float32(scale)).astype(np.float32))
    return out


def dequantize(codes, scale: float) -> np.ndarray:
    """Values of the codes times the scale, fp64."""
    return _TABLE[np.asarray(codes, dtype=np.uint8)] * float(np.float32(scale))


def kv_write_fp8(k, v, slot_mapping, k_cache, v_cache, k_scale: float, v_scale: float) -> None:
    """In place: for every new token t with slot s >= 0, the codes of
    k[t] / k_scale go to ``k_cache[s // bs, s % bs]`` (and V likewise).
    k, v are fp32 values (bf16 inputs widened exactly); caches are uint8."""
    bs = k_cache.shape[1]
    for t, s in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if s < 0:
            continue
        blk, off = divmod(int(s), bs)
        k_cache[blk, off] = quantize(k[t], k_scale)
        v_cache[blk, off] = quantize(v[t], v_scale)
