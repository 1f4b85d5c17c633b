"""Symmetric 8-bit integer codes for the INT8 KV cache.

The pages name 8-bit integer KV caches ("KV Cache优化实战" §3.2: INT8 for
keys in mixed schemes; §3.3: llama.cpp's q8_0 cache type; "企业官网建设流程
全解析" §9.1: 8-bit storage at one byte per element) and prefer a scale per
token or per head to one per tensor (§3.2).  They fix no formula.  Reading
adopted here, the plain symmetric absmax one, chosen so codes compare bit
for bit: per (token, KV head) ``scale = amax / 127`` (IEEE fp32, 1 when
``amax == 0``), ``code = round(x / scale)`` with the fp32 quotient rounded
to the nearest integer, ties to even, clamped to [-127, 127]; the value is
``code * scale``.  (llama.cpp's q8_0 uses 32-element groups and an fp16
scale; the per-(token, head) granularity matches the other one-byte
caches here.)

The pages fix no byte encoding either.  A code is stored as the byte
``code + 128`` (an unsigned byte with zero point 128, as asymmetric uint8
schemes store theirs), so bytes 1..255 hold codes -127..127; byte 0 is
never written.
"""
from __future__ import annotations

import numpy as np

MAX_CODE = 127.0


def encode(y: np.ndarray) -> np.ndarray:
    """float32 quotients -> int8 codes (nearest, ties to even, clamped to +-127)."""
    y = np.asarray(y, dtype=np.float32)
    if np.isnan(y).any():
        raise ValueError("NaN has no place in the INT8 cache")
    r = np.rint(y.astype(np.float64))          # rint rounds halves to even
    return np.clip(r, -MAX_CODE, MAX_CODE).astype(np.int8)


def decode(codes: np.ndarray) -> np.ndarray:
    """fp64 values of signed int8 codes."""
    c = np.asarray(codes)
    if c.dtype == np.uint8:
        raise TypeError("decode takes signed codes; stored bytes go through from_bytes first")
    return c.astype(np.float64)


def to_bytes(codes: np.ndarray) -> np.ndarray:
    """Signed codes in [-127, 127] -> stored bytes (code + 128)."""
    return (np.asarray(codes).astype(np.int16) + 128).astype(np.uint8)


def from_bytes(data: np.ndarray) -> np.ndarray:
    """Stored bytes -> signed codes (byte - 128)."""
    return (np.asarray(data, dtype=np.uint8).astype(np.int16) - 128).astype(np.int8)
