"""OCP FP8 E4M3 ("e4m3fn") codec, written out from the format's definition.

The FP8 KV cache the pages enable with ``--kv-cache-dtype fp8_e4m3``
("KV Cache优化实战" §3.3) stores each element in one byte:

* bit 7: sign; bits 6..3: exponent with bias 7; bits 2..0: mantissa;
* exponent field 0 encodes subnormals m/8 * 2^-6 (smallest 2^-9);
* there is no infinity; S.1111.111 is NaN, so the largest finite
  magnitude is 1.75 * 2^8 = 448.

Encoding is round-to-nearest, ties to the even code, saturating to +-448
("satfinite"), keeping the sign of zero.  The pages do not spell out the
rounding; this is the plain reading of "fp8_e4m3" and the one that lets the
cache bytes be compared bit for bit.
"""
from __future__ import annotations

import numpy as np

MAX_FINITE = 448.0
NAN_CODES = (0x7F, 0xFF)


def decode_value(code: int) -> float:
    """Value of one E4M3 code as a Python float (NaN for the two NaN codes)."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    exp = (code >> 3) & 0xF
    man = code & 0x7
    if exp == 0xF and man == 0x7:
        return float("nan")
    if exp == 0:
        return sign * (man / 8.0) * 2.0 ** (1 - 7)
    return sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)


def decode_table() -> np.ndarray:
    """float64[256]: value of every code."""
    return np.array([decode_value(c) for c in range(256)], dtype=np.float64)


_TABLE = decode_table()
# Non-negative finite codes 0x00..0x7E in increasing order of value.
_POS_CODES = np.arange(0x7F, dtype=np.int64)
_POS_VALUES = _TABLE[:0x7F]


def decode(codes: np.ndarray) -> np.ndarray:
    """float64 values of an array of uint8 codes."""
    return _TABLE[np.asarray(codes, dtype=np.uint8)]


def encode(y: np.ndarray) -> np.ndarray:
    """Encode float32 values: nearest code, ties to the even code, saturate at 448.

    ``y`` must be free of NaN (the cache never feeds one: the scale keeps
    every value within +-448, up to one rounding).
    """
    y = np.asarray(y, dtype=np.float32)
    if np.isnan(y).any():
        raise ValueError("NaN has no place in the FP8 cache")
    a = np.minimum(np.abs(y.astype(np.float64)), MAX_FINITE)
    hi = np.searchsorted(_POS_VALUES, a, side="left")  # first value >= a
    hi = np.clip(hi, 0, 0x7E)
    lo = np.clip(hi - 1, 0, 0x7E)
    d_lo = a - _POS_VALUES[lo]
    d_hi = _POS_VALUES[hi] - a
    exact = d_hi == 0.0
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (_POS_CODES[hi] % 2 == 0))
    mag = np.where(exact | pick_hi, _POS_CODES[hi], _POS_CODES[lo])
    sign = np.signbit(y).astype(np.int64) << 7
    return (mag | sign).astype(np.uint8)


# ---------------------------------------------------------------------------
# OCP FP8 E5M2, the other FP8 cache type the pages name
# (``--kv-cache-dtype fp8_e5m2``, "KV Cache优化实战" §3.3):
#
# * bit 7: sign; bits 6..2: exponent with bias 15; bits 1..0: mantissa;
# * exponent field 0 encodes subnormals m/4 * 2^-14 (smallest 2^-16);
# * exponent field 31 is infinity (mantissa 0) or NaN, as in IEEE binary16,
#   so the largest finite magnitude is 1.75 * 2^15 = 57344.
#
# Encoding mirrors E4M3: nearest finite code, ties to the even code,
# saturating to +-57344, keeping the sign of zero.
# ---------------------------------------------------------------------------
E5M2_MAX_FINITE = 57344.0


def e5m2_decode_value(code: int) -> float:
    """Value of one E5M2 code as a Python float (inf / NaN for the special codes)."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    exp = (code >> 2) & 0x1F
    man = code & 0x3
    if exp == 0x1F:
        return sign * float("inf") if man == 0 else float("nan")
    if exp == 0:
        return sign * (man / 4.0) * 2.0 ** (1 - 15)
    return sign * (1.0 + man / 4.0) * 2.0 ** (exp - 15)


def e5m2_decode_table() -> np.ndarray:
    return np.array([e5m2_decode_value(c) for c in range(256)], dtype=np.float64)


_E5M2_TABLE = e5m2_decode_table()
# Non-negative finite codes 0x00..0x7B in increasing order of value.
_E5M2_POS_CODES = np.arange(0x7C, dtype=np.int64)
_E5M2_POS_VALUES = _E5M2_TABLE[:0x7C]


def e5m2_decode(codes: np.ndarray) -> np.ndarray:
    return _E5M2_TABLE[np.asarray(codes, dtype=np.uint8)]


def e5m2_encode(y: np.ndarray) -> np.ndarray:
    """Encode float32 values: nearest finite code, ties to the even code, saturate at 57344."""
    y = np.asarray(y, dtype=np.float32)
    if np.isnan(y).any():
        raise ValueError("NaN has no place in the FP8 cache")
    a = np.minimum(np.abs(y.astype(np.float64)), E5M2_MAX_FINITE)
    hi = np.searchsorted(_E5M2_POS_VALUES, a, side="left")
    hi = np.clip(hi, 0, 0x7B)
    lo = np.clip(hi - 1, 0, 0x7B)
    d_lo = a - _E5M2_POS_VALUES[lo]
    d_hi = _E5M2_POS_VALUES[hi] - a
    exact = d_hi == 0.0
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (_E5M2_POS_CODES[hi] % 2 == 0))
    mag = np.where(exact | pick_hi, _E5M2_POS_CODES[hi], _E5M2_POS_CODES[lo])
    sign = np.signbit(y).astype(np.int64) << 7
    return (mag | sign).astype(np.uint8)
