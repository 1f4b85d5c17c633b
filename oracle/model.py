"""Plays a paged-cache operation script on the oracle: allocator + per-layer caches.

One decode step, as the pages lay it out ("KV Cache 与 vLLM" (zwxr.cn)
§3.1-§3.4, "企业官网建设流程全解析" §3.2): each running sequence appends the
new token's K and V (taking a block or copying a shared one as needed),
then its new query attends over all of its cached tokens through its block
table.
"""
from __future__ import annotations

import numpy as np

from .allocator import AllocatorModel
from .attention import decode_attention
from .cache import PagedCacheModel


class PagedKVOracle:
    def __init__(self, num_layers, num_blocks, num_kv_heads, head_dim, dtype,
                 block_size=16, alloc_order=None):
        self.alloc = AllocatorModel(num_blocks, block_size, alloc_order)
        self.layers = [PagedCacheModel(num_blocks, num_kv_heads, head_dim, dtype, block_size)
                       for _ in range(num_layers)]
        self.cow_log = []     # every (src, dst) pair, in order

    def create(self, seq):
        self.alloc.create(seq)

    def fork(self, parent, child):
        self.alloc.fork(parent, child)

    def free(self, seq):
        self.alloc.free_seq(seq)

    def append(self, seq_ids, k_rows, v_rows):
        """Append one token per entry of seq_ids.

        k_rows / v_rows: per layer, float32 [len(seq_ids), Hkv, D] (or a
        callable layer -> array).  Returns (slot_mapping, cow_pairs).
        """
        slots, cows = self.alloc.append_slots(list(seq_ids))
        for li, cache in enumerate(self.layers):
            for src, dst in cows:
                cache.copy_block(src, dst)
            k = k_rows(li) if callable(k_rows) else k_rows[li]
            v = v_rows(li) if callable(v_rows) else v_rows[li]
            cache.write(slots, k, v)
        self.cow_log.extend(cows)
        return slots, cows

    def decode(self, seq_ids, q, scale, layer=0):
        """fp64 attention output [n, Hq, D] for one layer; q: [n, Hq, D]."""
        cache = self.layers[layer]
        out = []
        for i, s in enumerate(seq_ids):
            K, V = cache.gather(self.alloc.tables[s], self.alloc.lens[s])
            out.append(decode_attention(q[i], K, V, scale))
        return np.stack(out) if out else np.zeros((0,) + np.shape(q)[1:])
