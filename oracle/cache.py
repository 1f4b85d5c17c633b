"""Paged KV cache model: reshape-and-cache writes, block copies, gather.

The pages give only logical shapes for one layer's cache
("KV Cache优化实战" §1.2: [layers, kv_heads, seq, head_dim];
"企业官网建设流程全解析" §1.3: [batch, seq, kv_heads, head_dim]).  Paging
("KV Cache 与 vLLM" (zwxr.cn) §3.1-§3.2) only changes where each token's
K/V lives: token ``n`` of a sequence sits at slot ``table[n // 16] * 16 +
n % 16``.  Reading adopted for the physical pool of one layer:
``[num_blocks, num_kv_heads, block_size, head_dim]``.

Storage types:

* ``f16`` / ``bf16``: the value is stored as is (the inputs are already in
  that type, so the write is an exact copy);
* one-byte codes, per (token, KV head) -- the finer granularity the pages
  recommend over one scale per tensor ("KV Cache优化实战" §3.2, §7.3) --
  ``amax = max |x|`` over head_dim, ``s = amax / R`` (``1`` when
  ``amax == 0``), code = Q(x / s); ``s`` and ``x / s`` are IEEE fp32
  round-to-nearest divisions (reading: the pages give no formula; this is
  the plain absmax one, fixed so that codes compare bit for bit):

  - ``fp8_e4m3``: R = 448, Q = nearest E4M3 code (``fp8.encode``);
  - ``fp8_e5m2``: R = 57344, Q = nearest E5M2 code (``fp8.e5m2_encode``);
  - ``int8``: R = 127, Q = nearest integer in [-127, 127] (``int8.encode``),
    stored as the byte Q + 128 (``int8.to_bytes``).

  The dequantised value is ``value(code) * s`` in fp64.
* ``fp8_e4m3_int4``: the mixed scheme of "KV Cache优化实战" §3.2 (8-bit
  keys, 4-bit values): K as ``fp8_e4m3`` above, V as ``int4`` -- R = 7,
  Q = nearest integer in [-7, 7], two codes a byte (``int4``), so one
  token's V row is head_dim / 2 bytes and the V pool is
  ``[num_blocks, num_kv_heads, block_size, head_dim / 2]``.

Slots never written hold NaN in this model (fp32 storage, and an fp32 NaN
scale for one-byte codes), so that a gather that strays onto one shows up
at once.
"""
from __future__ import annotations

import numpy as np

from . import fp8, int4, int8

DTYPES = ("f16", "bf16", "fp8_e4m3", "fp8_e5m2", "int8", "fp8_e4m3_int4")
# coded storage types: (R, encode float32 quotients -> stored bytes, decode stored bytes -> fp64)
CODE_TYPES = {
    "fp8_e4m3": (fp8.MAX_FINITE, fp8.encode, fp8.decode),
    "fp8_e5m2": (fp8.E5M2_MAX_FINITE, fp8.e5m2_encode, fp8.e5m2_decode),
    "int8": (int8.MAX_CODE, lambda y: int8.to_bytes(int8.encode(y)), lambda b: int8.decode(int8.from_bytes(b))),
    "int4": (int4.MAX_CODE, lambda y: int4.pack(int4.encode(y)), int4.decode),
}
# cache types whose K and V halves are stored differently: (K type, V type)
MIXED = {"fp8_e4m3_int4": ("fp8_e4m3", "int4")}


def part_types(dtype: str):
    """(K storage type, V storage type) of a cache type."""
    return MIXED.get(dtype, (dtype, dtype))


def row_bytes(part: str, head_dim: int) -> int:
    """Stored bytes of one token's row of one K or V storage type."""
    return {"f16": 2, "bf16": 2, "int4": 0.5}.get(part, 1) * head_dim


def quantize_rows(x: np.ndarray, dtype: str = "fp8_e4m3"):
    """Per-row quantisation of float32 rows ``[..., head_dim]`` to codes.

    Returns (stored bytes uint8 [..., head_dim] -- an int8 code as the byte code + 128;
    [..., head_dim / 2] for int4 --, scale float32 [...]).
    """
    r, enc, _ = CODE_TYPES[dtype]
    x = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x), axis=-1)
    scale = np.where(amax == 0, np.float32(1.0),
                     amax.astype(np.float32) / np.float32(r)).astype(np.float32)
    y = (x / scale[..., None]).astype(np.float32)
    return enc(y), scale


def code_values(codes: np.ndarray, dtype: str) -> np.ndarray:
    """fp64 values of stored codes (before the scale)."""
    return CODE_TYPES[dtype][2](codes)


class PagedCacheModel:
    """One layer's K and V pools."""

    def __init__(self, num_blocks: int, num_kv_heads: int, head_dim: int,
                 dtype: str, block_size: int = 16):
        if dtype not in DTYPES:
            raise ValueError(f"unknown cache dtype {dtype}")
        self.num_blocks, self.num_kv_heads, self.head_dim = num_blocks, num_kv_heads, head_dim
        self.block_size, self.dtype = block_size, dtype
        self.k_type, self.v_type = part_types(dtype)
        self.k, self.k_scale = self._pool(self.k_type)
        self.v, self.v_scale = self._pool(self.v_type)
        # which slots have been written (parity compares filled slots only)
        self.filled = np.zeros((num_blocks, block_size), dtype=bool)

    def _pool(self, part):
        shape = (self.num_blocks, self.num_kv_heads, self.block_size)
        if part in CODE_TYPES:
            data = np.full(shape + (int(row_bytes(part, self.head_dim)),), 0x7F if part != "int4" else 0,
                           dtype=np.uint8)
            return data, np.full(shape, np.nan, dtype=np.float32)
        return np.full(shape + (self.head_dim,), np.nan, dtype=np.float32), None

    def write(self, slot_mapping, k: np.ndarray, v: np.ndarray) -> None:
        """Reshape-and-cache: token t's K/V ``[num_kv_heads, head_dim]`` to slot_mapping[t].

        A slot of -1 skips the token.
        """
        bs = self.block_size
        for t, slot in enumerate(slot_mapping):
            slot = int(slot)
            if slot < 0:
                continue
            blk, off = divmod(slot, bs)
            if blk >= self.num_blocks:
                raise IndexError(f"slot {slot} outside the pool")
            for part, pool, scales, x in ((self.k_type, self.k, self.k_scale, k[t]),
                                          (self.v_type, self.v, self.v_scale, v[t])):
                if part in CODE_TYPES:
                    codes, sc = quantize_rows(x, part)
                    pool[blk, :, off, :] = codes
                    scales[blk, :, off] = sc
                else:
                    pool[blk, :, off, :] = x
            self.filled[blk, off] = True

    def copy_block(self, src: int, dst: int) -> None:
        """Copy all slots of a physical block (K, V and scales) for copy-on-write."""
        self.k[dst] = self.k[src]
        self.v[dst] = self.v[src]
        if self.k_scale is not None:
            self.k_scale[dst] = self.k_scale[src]
        if self.v_scale is not None:
            self.v_scale[dst] = self.v_scale[src]
        self.filled[dst] = self.filled[src]

    @staticmethod
    def _dequant(part, stored, scales):
        if part in CODE_TYPES:
            return code_values(stored, part) * scales.astype(np.float64)[..., None]
        return stored.astype(np.float64)

    def gather(self, table, length: int):
        """Contiguous fp64 K, V ``[length, num_kv_heads, head_dim]`` of one sequence.

        Logical token n lives in physical block table[n // bs] at offset n % bs.
        """
        bs = self.block_size
        pos = np.arange(length)
        blocks = np.asarray(table, dtype=np.int64)[pos // bs]
        offs = pos % bs
        out = []
        for part, pool, scales in ((self.k_type, self.k, self.k_scale), (self.v_type, self.v, self.v_scale)):
            stored = pool[blocks, :, offs, :]          # [L, Hkv, row]
            sc = scales[blocks, :, offs] if scales is not None else None
            out.append(self._dequant(part, stored, sc))
        return out[0], out[1]


def dequantize_rows(x: np.ndarray, dtype: str, part: str = "k"):
    """fp64 values a cache of ``dtype`` holds for float32 input rows ``[..., head_dim]``.

    The contiguous counterpart of write + gather: what token rows read back
    as, without the paging.  ``part`` ("k" or "v") picks the half of a
    mixed cache type.
    """
    x = np.asarray(x, dtype=np.float32)
    t = part_types(dtype)[0 if part == "k" else 1]
    if t in CODE_TYPES:
        codes, s = quantize_rows(x, t)
        return code_values(codes, t) * s.astype(np.float64)[..., None]
    return x.astype(np.float64)
