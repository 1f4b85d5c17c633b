"""Symmetric 4-bit integer codes for the V half of a mixed K-FP8 / V-INT4 cache.

Test infrastructure only: plain NumPy, shares nothing with the CUDA path.

The pages name the mixed scheme -- 8-bit (INT8 or FP8) keys with 4-bit
values, because attention is more sensitive to errors in K than in V
("KV Cache优化实战" §3.2) -- and 4-bit storage at half a byte per element
("企业官网建设流程全解析" §9.1; llama.cpp's q4_0 in "KV Cache优化实战"
§3.3).  They fix no formula.  Readings adopted here, the INT8 ones carried
over to four bits so that codes compare bit for bit:

* per (token, KV head) ``scale = amax / 7`` (IEEE fp32; 1 when
  ``amax == 0``), ``code = round(x / scale)`` with the fp32 quotient
  rounded to the nearest integer, ties to even, clamped to [-7, 7]
  (symmetric, like INT8's [-127, 127]); the value is ``code * scale``;
* storage: two codes a byte, element 2i in the low nibble and element
  2i + 1 in the high nibble of byte i, each nibble holding ``code + 8``
  (offset binary, 1..15; nibble 0, the value -8, is never written).
"""
from __future__ import annotations

import numpy as np

MAX_CODE = 7.0


def encode(y: np.ndarray) -> np.ndarray:
    """float32 quotients -> int8 codes in [-7, 7] (nearest, ties to even)."""
    y = np.asarray(y, dtype=np.float32)
    if np.isnan(y).any():
        raise ValueError("NaN has no place in the INT4 cache")
    r = np.rint(y.astype(np.float64))          # rint rounds halves to even
    return np.clip(r, -MAX_CODE, MAX_CODE).astype(np.int8)


def pack(codes: np.ndarray) -> np.ndarray:
    """int8 codes ``[..., n]`` (n even) -> bytes ``[..., n / 2]``, element 2i in the low nibble."""
    c = np.asarray(codes).astype(np.int16)
    if c.shape[-1] % 2:
        raise ValueError("an odd number of elements cannot be packed two a byte")
    if c.min(initial=0) < -8 or c.max(initial=0) > 7:
        raise ValueError("code outside [-8, 7]")
    nib = (c + 8).astype(np.uint8)
    return (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)


def unpack(data: np.ndarray) -> np.ndarray:
    """bytes ``[..., m]`` -> int8 codes ``[..., 2 m]``."""
    b = np.asarray(data, dtype=np.uint8)
    lo = (b & 0x0F).astype(np.int8) - 8
    hi = (b >> 4).astype(np.int8) - 8
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.int8)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def decode(data: np.ndarray) -> np.ndarray:
    """fp64 values of packed INT4 bytes ``[..., m]`` -> ``[..., 2 m]``."""
    return unpack(data).astype(np.float64)
