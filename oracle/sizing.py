"""KV-cache size, utilisation and capacity arithmetic as the pages state it.

* General form ("KV Cache优化实战" §2.1):
  bytes = 2 x layers x kv_heads x head_dim x seq_len x batch x bytes_per_element
  (the 2 is one copy for K and one for V).
* Hidden-size form for multi-head attention ("KV Cache 与 vLLM" (zwxr.cn)
  §1.3): layers x seq_len x hidden x 2 x 2 x batch (K/V and two FP16 bytes);
  equal to the general form when kv_heads x head_dim = hidden.
* Per-layer elements ("企业官网建设流程全解析" §2.1):
  2 x batch x seq_len x kv_heads x head_dim.
* Per-request bound ("企业官网建设流程全解析" §7.1):
  2 x max_seq_len x layers x kv_heads x head_dim x bytes.
* Capacity planning ("KV Cache 与 vLLM" §4.3, "企业官网建设流程全解析" §4.1):
  budget = memory x utilisation - weights; concurrency = budget / per-request KV.

Paging allocates whole blocks, so a sequence of L tokens holds
ceil(L / bs) x bs token slots ("KV Cache 与 vLLM" §3.1); max-length
preallocation holds max_len slots per request (§2.2).
"""
from __future__ import annotations

BYTES_PER_ELEMENT = {"f16": 2, "bf16": 2, "fp8_e4m3": 1, "fp8_e5m2": 1, "int8": 1, "int4": 0.5}
# cache types stored as one-byte codes plus one fp32 scale per (token, KV head)
SCALED_ONE_BYTE = ("fp8_e4m3", "fp8_e5m2", "int8")
# mixed cache types ("KV Cache优化实战" §3.2: 8-bit keys, 4-bit values), each
# half with one fp32 scale per (token, KV head): (K bytes, V bytes) per element
SCALED_MIXED = {"fp8_e4m3_int4": (1, 0.5)}


def kv_bytes(layers, kv_heads, head_dim, seq_len, batch, bytes_per_element):
    return 2 * layers * kv_heads * head_dim * seq_len * batch * bytes_per_element


def kv_bytes_from_hidden(layers, seq_len, hidden, batch, bytes_per_element=2):
    return layers * seq_len * hidden * 2 * bytes_per_element * batch


def layer_kv_elements(batch, seq_len, kv_heads, head_dim):
    return 2 * batch * seq_len * kv_heads * head_dim


def request_kv_bound(max_seq_len, layers, kv_heads, head_dim, bytes_per_element):
    return 2 * max_seq_len * layers * kv_heads * head_dim * bytes_per_element


def paged_token_slots(lengths, block_size=16):
    """Token slots held under paging: sum of ceil(L / bs) x bs."""
    return sum(-(-int(L) // block_size) * block_size for L in lengths)


def paged_utilisation(lengths, block_size=16):
    """Share of allocated slots that hold a token."""
    held = paged_token_slots(lengths, block_size)
    return sum(int(L) for L in lengths) / held if held else 1.0


def prealloc_utilisation(lengths, max_len):
    """Share of max-length reservations that hold a token."""
    return sum(int(L) for L in lengths) / (len(lengths) * max_len)


def fp8_bytes_per_token(layers, kv_heads, head_dim, scale_bytes=4):
    """FP8 cache bytes per token: one byte per element plus one fp32 scale per (token, KV head), for K and V."""
    return 2 * layers * kv_heads * (head_dim + scale_bytes)


def kv_budget(memory_bytes, utilisation, weight_bytes):
    return memory_bytes * utilisation - weight_bytes


def max_concurrency(budget_bytes, per_request_bytes):
    return int(budget_bytes // per_request_bytes)


def token_head_bytes(head_dim, dtype, scale_bytes=4):
    """K plus V bytes one token holds for one KV head (scales included)."""
    if dtype in SCALED_ONE_BYTE:
        return 2 * (head_dim + scale_bytes)
    if dtype in SCALED_MIXED:
        kb, vb = SCALED_MIXED[dtype]
        return int(head_dim * kb + head_dim * vb) + 2 * scale_bytes
    return 2 * head_dim * BYTES_PER_ELEMENT[dtype]


def pool_blocks(budget_bytes, layers, kv_heads, head_dim, dtype, block_size=16):
    """Whole blocks a byte budget buys for every layer's K and V (plus coded caches' scales)."""
    per_block = layers * kv_heads * block_size * token_head_bytes(head_dim, dtype)
    return int(budget_bytes // per_block)
