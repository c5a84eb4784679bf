"""Pins of the E4M3 cache encoding (oracle/fp8.py) to the format's
definition and to an independent conversion:

* the code table: fixed codes with values that follow from the bit layout
  (zero, the smallest subnormal, the largest subnormal, the smallest normal,
  one, the largest finite value, NaN, negative zero);
* round trip: every finite code encodes back to itself;
* nearest value by exhaustive search over all codes, ties to the even code;
* ties and saturation at chosen points;
* torch's float8_e4m3fn conversion (a library routine, run as a black box)
  on random values inside the finite range;
* the relative error bound of 3 mantissa bits (half an ulp, 2^-4) in the
  normal range, and the absolute bound 2^-10 in the subnormal range;
* the quantising scatter skips negative slots and writes whole rows.
"""
import numpy as np
import pytest

from oracle import fp8


def test_code_table_closed_forms():
    v = fp8.e4m3_value
    assert v(0x00) == 0.0 and v(0x80) == 0.0 and np.signbit(v(0x80))
    assert v(0x01) == 2.0 ** -9                 # smallest subnormal: 1/8 * 2^-6
    assert v(0x07) == 7 * 2.0 ** -9             # largest subnormal
    assert v(0x08) == 2.0 ** -6                 # smallest normal
    assert v(0x38) == 1.0                       # exponent field 7 = bias
    assert v(0x3C) == 1.5
    assert v(0x7E) == 448.0 and v(0xFE) == -448.0
    assert np.isnan(v(0x7F)) and np.isnan(v(0xFF))
    finite = [c for c in range(256) if not np.isnan(v(c))]
    assert len(finite) == 254
    pos = sorted(v(c) for c in range(0x7F))
    assert pos == [v(c) for c in range(0x7F)]   # codes 0..0x7E increase with their value


def test_round_trip_every_finite_code():
    codes = np.array([c for c in range(256) if not np.isnan(fp8.e4m3_value(c))], dtype=np.uint8)
    vals = np.array([fp8.e4m3_value(c) for c in codes], dtype=np.float32)
    assert np.array_equal(fp8.e4m3_encode(vals), codes)


def brute_nearest(x: float) -> int:
    """Exhaustive search: the finite code nearest to x, ties to the even code,
    saturating beyond the largest value."""
    a = min(abs(x), 448.0)
    best, bd = None, None
    for c in range(0x7F):
        d = abs(fp8.e4m3_value(c) - a)
        if bd is None or d < bd or (d == bd and c % 2 == 0):
            best, bd = c, d
    return (0x80 if (x < 0 or (x == 0 and np.signbit(x))) else 0) | best


def test_nearest_by_exhaustive_search():
    rng = np.random.default_rng(5)
    xs = np.concatenate([rng.standard_normal(600) * 10, rng.standard_normal(200) * 0.01,
                         rng.uniform(-500, 500, 200)]).astype(np.float32)
    got = fp8.e4m3_encode(xs)
    for x, c in zip(xs, got):
        assert c == brute_nearest(float(x)), (x, c)


def test_ties_and_saturation():
    enc = lambda x: int(fp8.e4m3_encode(np.float32(x)))
    assert enc(1.0625) == 0x38      # midway 1 and 1.125: even mantissa (1.0)
    assert enc(1.1875) == 0x3A      # midway 1.125 (0x39) and 1.25 (0x3A): 0x3A
    assert enc(1.0626) == 0x39 and enc(1.0624) == 0x38
    assert enc(2.0 ** -10) == 0x00  # midway 0 and the smallest subnormal: 0
    assert enc(3 * 2.0 ** -10) == 0x02   # midway 1/8 and 2/8 of 2^-6: even (2)
    assert enc(464.0) == 0x7E and enc(1e6) == 0x7E and enc(-1e30) == 0xFE
    assert enc(-0.0) == 0x80 and enc(-1e-12) == 0x80
    assert enc(float("nan")) == 0x7F


def test_agrees_with_torch_e4m3fn():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8_e4m3fn")
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(50000) * 40, rng.standard_normal(20000) * 0.003]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.e4m3_encode(x), ref)


def test_error_bounds():
    rng = np.random.default_rng(9)
    scale = 0.37
    x = (rng.standard_normal(20000) * 20).astype(np.float32)
    dq = fp8.dequantize(fp8.quantize(x, scale), scale)
    q = x.astype(np.float64) / np.float64(np.float32(scale))
    normal = np.abs(q) >= 2.0 ** -6
    inside = np.abs(q) <= 448
    rel = np.abs(dq / np.float32(scale) - q)
    assert np.all(rel[normal & inside] <= 2.0 ** -4 * np.abs(q[normal & inside]) * (1 + 1e-6))
    assert np.all(rel[~normal] <= 2.0 ** -10 * (1 + 1e-6))
    assert np.all(np.abs(dq[~inside]) == 448 * np.float32(scale))


def test_quantising_scatter():
    kc = np.zeros((3, 4, 2, 8), dtype=np.uint8)
    vc = np.zeros_like(kc)
    rng = np.random.default_rng(1)
    k = rng.standard_normal((3, 2, 8)).astype(np.float32)
    v = rng.standard_normal((3, 2, 8)).astype(np.float32)
    fp8.kv_write_fp8(k, v, np.array([5, -1, 11]), kc, vc, 0.5, 0.25)
    assert np.array_equal(kc[1, 1], fp8.quantize(k[0], 0.5)) and np.array_equal(vc[2, 3], fp8.quantize(v[2], 0.25))
    assert kc[0].sum() == 0 and int((kc != 0).any(axis=(2, 3)).sum()) == 2
