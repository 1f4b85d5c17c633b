"""Pins for the oracle's INT4 codec and the mixed K-FP8 / V-INT4 cache.

INT4 is anchored to round-half-even integer rounding, the symmetric clamp,
a hand-packed byte example (the nibble order), an exhaustive pack/unpack
round trip, and the absmax scale's defining properties.  The mixed cache
is anchored to its two halves: K must read back exactly as an E4M3 cache
would, V exactly as the INT4 quantiser gives, and the pool sizes to the
byte counts of each half.
"""
import numpy as np
import pytest

from oracle import fp8, int4, sizing
from oracle.attention import decode_attention
from oracle.cache import CODE_TYPES, PagedCacheModel, dequantize_rows, part_types, quantize_rows


def test_int4_rounds_half_to_even_and_clamps():
    y = np.array([0.5, 1.5, 2.5, -0.5, -3.5, 6.5, 6.49, 7.5, 8.0, -9.0, 1e9, -0.0, 0.49], dtype=np.float32)
    want = [0, 2, 2, 0, -4, 6, 6, 7, 7, -7, 7, 0, 0]
    assert int4.encode(y).tolist() == want
    with pytest.raises(ValueError):
        int4.encode(np.array([np.nan], dtype=np.float32))


def test_int4_packing_by_hand():
    # codes -7, 7, 0, -1 -> nibbles 1, 15, 8, 7 -> bytes 0xF1, 0x78 (even element low)
    assert int4.pack(np.array([-7, 7, 0, -1])).tolist() == [0xF1, 0x78]
    assert int4.pack(np.zeros(6, dtype=np.int8)).tolist() == [0x88] * 3
    assert int4.unpack(np.array([0x0F], dtype=np.uint8)).tolist() == [7, -8]
    with pytest.raises(ValueError):
        int4.pack(np.array([1, 2, 3]))
    with pytest.raises(ValueError):
        int4.pack(np.array([8, 0]))


def test_int4_pack_unpack_exhaustive():
    a, b = np.meshgrid(np.arange(-8, 8), np.arange(-8, 8), indexing="ij")
    codes = np.stack([a.ravel(), b.ravel()], axis=-1).astype(np.int8)   # every pair
    packed = int4.pack(codes)
    assert packed.shape == (256, 1) and len(set(packed.ravel().tolist())) == 256
    assert np.array_equal(int4.unpack(packed), codes)
    assert np.array_equal(int4.decode(packed), codes.astype(np.float64))


def test_int4_quantiser_scale_and_error_bound():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((200, 64)) * rng.uniform(0.01, 50, (200, 1))).astype(np.float32)
    packed, s = quantize_rows(x, "int4")
    assert packed.shape == (200, 32) and s.dtype == np.float32
    amax = np.abs(x).max(axis=1)
    assert np.array_equal(s, (amax / np.float32(7)).astype(np.float32))
    codes = int4.unpack(packed)
    # the absmax element takes the code +-7 with the element's sign
    i = np.argmax(np.abs(x), axis=1)
    top = codes[np.arange(200), i]
    assert np.array_equal(top, np.where(x[np.arange(200), i] > 0, 7, -7))
    # each value is within half a scale step (plus the fp32 quotient's rounding)
    err = np.abs(codes * s[:, None].astype(np.float64) - x.astype(np.float64))
    assert np.all(err <= 0.5 * s[:, None] * (1 + 1e-6))
    zero, sz = quantize_rows(np.zeros((2, 8), dtype=np.float32), "int4")
    assert sz.tolist() == [1.0, 1.0] and zero.tolist() == [[0x88] * 4] * 2


def test_mixed_type_halves():
    assert part_types("fp8_e4m3_int4") == ("fp8_e4m3", "int4")
    assert part_types("bf16") == ("bf16", "bf16")
    assert CODE_TYPES["int4"][0] == 7.0
    rng = np.random.default_rng(4)
    x = rng.standard_normal((5, 3, 32)).astype(np.float32)
    assert np.array_equal(dequantize_rows(x, "fp8_e4m3_int4", "k"), dequantize_rows(x, "fp8_e4m3"))
    c, s = quantize_rows(x, "int4")
    assert np.array_equal(dequantize_rows(x, "fp8_e4m3_int4", "v"), int4.decode(c) * s.astype(np.float64)[..., None])


def test_mixed_paged_cache_layout_and_gather():
    rng = np.random.default_rng(5)
    nb, hkv, d = 6, 2, 16
    m = PagedCacheModel(nb, hkv, d, "fp8_e4m3_int4")
    assert m.k.shape == (nb, hkv, 16, d) and m.v.shape == (nb, hkv, 16, d // 2)
    k = rng.standard_normal((20, hkv, d)).astype(np.float32)
    v = rng.standard_normal((20, hkv, d)).astype(np.float32)
    table = [4, 1]
    m.write([4 * 16 + t for t in range(16)] + [16 + t for t in range(4)], k, v)
    K, V = m.gather(table, 20)
    assert np.array_equal(K, dequantize_rows(k, "fp8_e4m3"))
    assert np.array_equal(V, dequantize_rows(v, "fp8_e4m3_int4", "v"))
    # the stored bytes of token 17 (block 1, offset 1) are the packed INT4 codes
    c, s = quantize_rows(v[17], "int4")
    assert np.array_equal(m.v[1, :, 1, :], c) and np.array_equal(m.v_scale[1, :, 1], s)
    ks = (np.abs(k[17]).max(-1, keepdims=True) / np.float32(448)).astype(np.float32)
    assert np.array_equal(m.k[1, :, 1, :], fp8.encode((k[17] / ks).astype(np.float32)))
    # one cached token: attention returns that token's dequantised V
    out = decode_attention(rng.standard_normal((4, d)).astype(np.float32), K[:1], V[:1], 0.25)
    assert np.array_equal(out, np.repeat(V[:1], 2, axis=1)[0])


def test_mixed_sizing():
    # K: d bytes + 4-byte scale; V: d / 2 bytes + 4-byte scale; per (token, KV head)
    assert sizing.token_head_bytes(128, "fp8_e4m3_int4") == 128 + 64 + 8
    assert sizing.token_head_bytes(128, "fp8_e4m3") == 2 * (128 + 4)
    assert sizing.token_head_bytes(128, "bf16") == 512
    per_block = 32 * 8 * 16 * 200
    assert sizing.pool_blocks(7 * per_block + per_block - 1, 32, 8, 128, "fp8_e4m3_int4") == 7
