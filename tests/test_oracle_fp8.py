"""Pins for the oracle's FP8 E4M3 codec and per-(token, head) quantiser.

Anchored to the format's definition (bias 7, 3 mantissa bits, no inf, max
448, smallest subnormal 2^-9), round-to-nearest-even, and cross-checked
against torch's float8_e4m3fn cast (a library routine) on in-range values.
"""
import math

import numpy as np
import pytest

from oracle import fp8
from oracle.cache import quantize_rows


def test_defined_values():
    assert fp8.decode_value(0x38) == 1.0
    assert fp8.decode_value(0x7E) == 448.0
    assert fp8.decode_value(0x01) == 2.0 ** -9
    assert fp8.decode_value(0x07) == 7 * 2.0 ** -9
    assert fp8.decode_value(0x08) == 2.0 ** -6           # smallest normal
    assert fp8.decode_value(0x40) == 2.0
    assert fp8.decode_value(0xB8) == -1.0
    assert math.copysign(1.0, fp8.decode_value(0x80)) == -1.0 and fp8.decode_value(0x80) == 0.0
    assert math.isnan(fp8.decode_value(0x7F)) and math.isnan(fp8.decode_value(0xFF))


def test_monotone_and_spacing():
    v = fp8.decode_table()[:0x7F]
    assert np.all(np.diff(v) > 0)
    # within one binade the step is 2^(e-10); subnormal step 2^-9
    for code in range(1, 0x7E):
        e = max((code >> 3) & 0xF, 1)
        assert v[code + 1] - v[code] == pytest.approx(2.0 ** (e - 10), rel=0, abs=0) or \
            (code & 7) == 7  # crossing into the next binade


def test_round_trip_all_finite_codes():
    codes = np.array([c for c in range(256) if c not in fp8.NAN_CODES], dtype=np.uint8)
    assert len(codes) == 254
    vals = fp8.decode(codes).astype(np.float32)
    back = fp8.encode(vals)
    assert np.array_equal(back, codes)


def test_ties_to_even_and_saturation():
    cases = [
        (1.0625, 0x38),           # midway 1.0 (0x38) / 1.125 (0x39) -> even 0x38
        (1.1875, 0x3A),           # midway 1.125 / 1.25 -> even 0x3A
        (2.0 ** -10, 0x00),       # midway 0 / 2^-9 -> 0
        (3 * 2.0 ** -10, 0x02),   # midway 2^-9 / 2^-8 -> even 0x02
        (2.0 ** -11, 0x00),
        (449.0, 0x7E), (1e30, 0x7E), (463.9, 0x7E), (480.0, 0x7E),
        (-1e30, 0xFE), (-449.0, 0xFE),
        (0.0, 0x00), (-0.0, 0x80),  # the sign of zero is kept
    ]
    got = fp8.encode(np.array([c[0] for c in cases], dtype=np.float32))
    assert [int(g) for g in got] == [c[1] for c in cases]


def test_nearest_on_random_values():
    rng = np.random.default_rng(0)
    y = (rng.standard_normal(20000) * 100).astype(np.float32)
    codes = fp8.encode(y)
    vals = fp8.decode(codes)
    grid = fp8.decode_table()[:0x7F]
    a = np.minimum(np.abs(y.astype(np.float64)), 448.0)
    best = np.min(np.abs(grid[None, :] - a[:, None]), axis=1)
    assert np.all(np.abs(np.abs(vals) - a) == best)
    assert np.all(np.signbit(vals) == np.signbit(y))


def test_agrees_with_torch_cast_in_range():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(1)
    y = np.concatenate([
        (rng.standard_normal(50000) * 40).astype(np.float32),
        (rng.standard_normal(5000) * 1e-2).astype(np.float32),
        (rng.uniform(-448, 448, 5000)).astype(np.float32),
    ])
    y = y[np.abs(y) <= 448]
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.encode(y), ref)


def test_quantize_rows_scale_and_extreme_code():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((64, 8, 128)) * rng.uniform(0.01, 50, (64, 8, 1))).astype(np.float32)
    codes, s = quantize_rows(x)
    amax = np.abs(x).max(axis=-1)
    # fp32 round-to-nearest division, checked through fp64 (exact for fp32 operands)
    assert np.array_equal(s, (amax.astype(np.float64) / 448.0).astype(np.float32))
    # the element of largest magnitude lands on +-448
    idx = np.abs(x).argmax(axis=-1)
    top = np.take_along_axis(codes, idx[..., None], axis=-1)[..., 0]
    assert np.all((top & 0x7F) == 0x7E)
    # error bound: half an E4M3 step at the value's binade, or half a subnormal step
    deq = fp8.decode(codes) * s[..., None].astype(np.float64)
    y = x.astype(np.float64) / s[..., None]
    bound = np.maximum(np.abs(y) * 2.0 ** -4, 2.0 ** -10) * s[..., None] * (1 + 1e-6)
    assert np.all(np.abs(deq - x) <= bound + np.abs(x) * 2.0 ** -23)


def test_quantize_zero_row():
    codes, s = quantize_rows(np.zeros((3, 16), dtype=np.float32))
    assert np.all(s == 1.0) and np.all(codes == 0)


def test_quantize_single_outlier_row():
    x = np.zeros(128, dtype=np.float32)
    x[5] = -20.0
    x[6] = 1.0
    codes, s = quantize_rows(x[None])
    assert s[0] == np.float32(20.0) / np.float32(448.0)
    assert codes[0, 5] == 0xFE
    assert fp8.decode(codes[0, 6]) == pytest.approx(22.4, rel=2 ** -4)
