"""Runs a seeded workload's operation script on the GPU through the engine.

Input values come from ``workloads`` (host, numpy); everything the method
computes happens in libpkv.so.
"""
from __future__ import annotations

import numpy as np

from .engine import PagedKVCache, torch_dtype
from .workloads import Workload

PREFILL_CHUNK = 8192  # tokens per append call while pre-filling


def to_device(x: np.ndarray, dtype: str, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).to(device=device).to(torch_dtype(dtype))


def new_cache(w: Workload, device="cuda", poison=False, alloc_order=None) -> PagedKVCache:
    return PagedKVCache(num_layers=w.num_layers, num_blocks=w.num_blocks, num_kv_heads=w.num_kv_heads,
                        head_dim=w.head_dim, cache_dtype=w.cache_dtype,
                        alloc_order=w.alloc_order if alloc_order is None else alloc_order,
                        device=device, poison=poison, block_size=w.block_size)


def prefill(w: Workload, cache: PagedKVCache, device="cuda") -> None:
    """Create / fork sequences and write every token before the decode step."""
    for op in w.prefill_ops():
        if op[0] == "create":
            cache.create(op[1])
        elif op[0] == "fork":
            cache.fork(op[1], op[2])
        else:
            seqs = op[1]
            s = seqs[0]
            start = cache.seq_len(s)
            for lo in range(0, len(seqs), PREFILL_CHUNK):
                n = min(PREFILL_CHUNK, len(seqs) - lo)
                k = to_device(w.kv_rows(0, s, start + lo, start + lo + n), w.q_dtype, device)
                v = to_device(w.kv_rows(1, s, start + lo, start + lo + n), w.q_dtype, device)
                cache.append([s] * n, k, v)


def step_inputs(w: Workload, step: int = 0, device="cuda"):
    """Device tensors for decode step ``step``: k, v [B, Hkv, D]; q [layers, B, Hq, D]."""
    k = to_device(w.step_rows(0, step), w.q_dtype, device)
    v = to_device(w.step_rows(1, step), w.q_dtype, device)
    q = to_device(np.stack([w.q_rows(layer, step) for layer in range(w.num_layers)]), w.q_dtype, device)
    return k, v, q


def run(w: Workload, device="cuda", poison=False, alloc_order=None, out_dtype=None, cascade=True):
    """Pre-fill, then one decode step; returns (cache, out [layers, B, Hq, D]).

    ``out_dtype``: None for the query's dtype, "f32" for the fp32 result.
    ``cascade``: let the step attend shared prefixes with the prefix kernel.
    """
    import torch
    cache = new_cache(w, device, poison, alloc_order)
    cache.use_cascade(cascade)
    prefill(w, cache, device)
    k, v, q = step_inputs(w, 0, device)
    out = torch.empty(q.shape, dtype=torch.float32, device=q.device) if out_dtype == "f32" else None
    out = cache.step(w.seq_ids, k, v, q, scale=w.scale, out=out)
    return cache, out
