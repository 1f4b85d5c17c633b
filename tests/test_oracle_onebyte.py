"""Pins for the oracle's E5M2 and INT8 codecs and their per-(token, head) quantisers.

E5M2 is anchored to the format's definition (bias 15, 2 mantissa bits,
IEEE-style inf/NaN, max finite 57344, smallest subnormal 2^-16), to the
fact that every E5M2 code is the high byte of the binary16 number with the
same value, and to torch's float8_e5m2 cast (a library routine) on
in-range values.  INT8 is anchored to round-half-even integer rounding and
to the absmax scale's defining properties.
"""
import math

import numpy as np
import pytest

from oracle import fp8, int8
from oracle.cache import CODE_TYPES, PagedCacheModel, dequantize_rows, quantize_rows


# ---- E5M2 -------------------------------------------------------------------
def test_e5m2_defined_values():
    assert fp8.e5m2_decode_value(0x3C) == 1.0
    assert fp8.e5m2_decode_value(0x7B) == 57344.0
    assert fp8.e5m2_decode_value(0x01) == 2.0 ** -16
    assert fp8.e5m2_decode_value(0x04) == 2.0 ** -14          # smallest normal
    assert fp8.e5m2_decode_value(0x40) == 2.0
    assert fp8.e5m2_decode_value(0xBC) == -1.0
    assert fp8.e5m2_decode_value(0x7C) == math.inf and fp8.e5m2_decode_value(0xFC) == -math.inf
    for c in (0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF):
        assert math.isnan(fp8.e5m2_decode_value(c))
    assert math.copysign(1.0, fp8.e5m2_decode_value(0x80)) == -1.0


def test_e5m2_is_the_high_byte_of_binary16():
    codes = np.arange(256, dtype=np.uint16)
    as_f16 = (codes << 8).astype(np.uint16).view(np.float16).astype(np.float64)
    table = fp8.e5m2_decode_table()
    finite = np.isfinite(as_f16)
    assert np.array_equal(table[finite], as_f16[finite])
    assert np.array_equal(np.isnan(table), np.isnan(as_f16))
    assert np.array_equal(np.isinf(table), np.isinf(as_f16))


def test_e5m2_monotone_and_round_trip():
    v = fp8.e5m2_decode_table()[:0x7C]
    assert np.all(np.diff(v) > 0)
    codes = np.array([c for c in range(256) if np.isfinite(fp8.e5m2_decode_value(c))], dtype=np.uint8)
    assert len(codes) == 248
    back = fp8.e5m2_encode(fp8.e5m2_decode(codes).astype(np.float32))
    assert np.array_equal(back, codes)


def test_e5m2_ties_to_even_and_saturation():
    cases = [
        (1.125, 0x3C),            # midway 1.0 (0x3C) / 1.25 (0x3D) -> even 0x3C
        (1.375, 0x3E),            # midway 1.25 / 1.5 -> even 0x3E
        (2.0 ** -17, 0x00),       # midway 0 / 2^-16 -> 0
        (3 * 2.0 ** -17, 0x02),   # midway 2^-16 / 2^-15 -> even 0x02
        (57345.0, 0x7B), (61440.0, 0x7B), (1e30, 0x7B), (-1e30, 0xFB),
        (0.0, 0x00), (-0.0, 0x80),
    ]
    got = fp8.e5m2_encode(np.array([c[0] for c in cases], dtype=np.float32))
    assert [int(g) for g in got] == [c[1] for c in cases]


def test_e5m2_agrees_with_torch_in_range():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e5m2"):
        pytest.skip("torch has no float8_e5m2")
    rng = np.random.default_rng(5)
    y = np.concatenate([rng.standard_normal(20000) * s for s in (1e-4, 1e-1, 1, 100, 3e4)]).astype(np.float32)
    y = y[np.abs(y) <= fp8.E5M2_MAX_FINITE]
    ref = torch.from_numpy(y).to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(fp8.e5m2_encode(y), ref)


# ---- INT8 -------------------------------------------------------------------
def test_int8_rounding_and_clamp():
    y = np.array([0.0, 0.49, 0.5, 1.5, 2.5, -2.5, -3.5, 126.5, 127.4, 128.0, -200.0, 7.0], dtype=np.float32)
    assert int8.encode(y).tolist() == [0, 0, 0, 2, 2, -2, -4, 126, 127, 127, -127, 7]
    assert int8.decode(np.array([-127, 0, 127], dtype=np.int8)).tolist() == [-127.0, 0.0, 127.0]


def test_int8_storage_bytes():
    # stored byte = code + 128: codes -127..127 take bytes 1..255, zero is 0x80
    codes = np.arange(-127, 128, dtype=np.int8)
    b = int8.to_bytes(codes)
    assert b.dtype == np.uint8 and b.tolist() == list(range(1, 256))
    assert int8.to_bytes(np.array([-127, -1, 0, 1, 127], dtype=np.int8)).tolist() == [0x01, 0x7F, 0x80, 0x81, 0xFF]
    assert np.array_equal(int8.from_bytes(b), codes)
    # the cache's decoder reads stored bytes
    assert CODE_TYPES["int8"][2](np.array([0x01, 0x80, 0xFF], dtype=np.uint8)).tolist() == [-127.0, 0.0, 127.0]
    with pytest.raises(TypeError):
        int8.decode(np.array([0x81], dtype=np.uint8))


@pytest.mark.parametrize("dtype", ["int8", "fp8_e5m2", "fp8_e4m3"])
def test_absmax_element_takes_the_largest_code(dtype):
    r = CODE_TYPES[dtype][0]
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((500, 128)) * rng.uniform(1e-3, 1e3, (500, 1))).astype(np.float32)
    codes, s = quantize_rows(x, dtype)
    vals = CODE_TYPES[dtype][2](codes)
    arg = np.argmax(np.abs(x), axis=1)
    top = vals[np.arange(500), arg]
    assert np.array_equal(np.abs(top), np.full(500, r))
    assert np.array_equal(np.sign(top), np.sign(x[np.arange(500), arg]))
    assert np.all(np.abs(vals) <= r)


def test_int8_error_bound_and_zero_rows():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((300, 64)).astype(np.float32)
    x[7] = 0.0
    codes, s = quantize_rows(x, "int8")
    assert s[7] == 1.0 and not int8.from_bytes(codes[7]).any()
    err = np.abs(dequantize_rows(x, "int8") - x.astype(np.float64))
    # half a step of the scale, plus the fp32 rounding of the quotient
    assert np.all(err <= s.astype(np.float64)[:, None] * (0.5 + 1e-5))


@pytest.mark.parametrize("dtype", ["fp8_e5m2", "int8"])
def test_paged_gather_matches_contiguous_dequantisation(dtype):
    rng = np.random.default_rng(9)
    nb, hkv, d, L = 8, 2, 16, 37
    cache = PagedCacheModel(nb, hkv, d, dtype)
    table = rng.permutation(nb)[: -(-L // 16)]
    k = rng.standard_normal((L, hkv, d)).astype(np.float32)
    v = rng.standard_normal((L, hkv, d)).astype(np.float32)
    slots = [int(table[n // 16]) * 16 + n % 16 for n in range(L)]
    cache.write(slots, k, v)
    gk, gv = cache.gather(table, L)
    assert np.array_equal(gk, dequantize_rows(k, dtype))
    assert np.array_equal(gv, dequantize_rows(v, dtype))
