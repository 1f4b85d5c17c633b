"""Prefix-cache hits attended by the cascade, through the step executor, against the oracle.

Requests that share a system prompt are admitted through the prefix cache
("KV Cache优化实战" §5.2, "企业官网建设流程全解析" §6.2): their tables start
with the same physical blocks, so the step executor's cascade attends those
blocks once for the whole group with the prefix kernel ("KV Cache 与 vLLM"
(zwxr.cn) §3.3) and the decode merges the partials with each member's own
tiles.  The same admissions, writes, commits and steps drive the oracle's
``PrefixCachingAllocator`` and one ``PagedCacheModel`` per layer.  After every
step: block tables, lengths and copy-on-write pairs bit-exact, every layer's
fp32 output within max |err| <= 1e-2 and relative L2 <= 2e-3 of the fp64
attention; the cascade must have run.
"""
import zlib

import numpy as np
import pytest

from oracle.attention import decode_attention
from oracle.cache import PagedCacheModel
from oracle.prefix_cache import PrefixCachingAllocator
from paged_kv_cache_163_gb300 import workloads as wl

from helpers import assert_close, to_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

LAYERS, HKV, HQ, D = 2, 4, 16, 128
SCALE = float(np.float32(1) / np.sqrt(np.float32(D)))


def prompt_rows(tokens, start, stop, seed=11):
    """K/V rows [2, n, HKV, D] of prompt positions start..stop: a function of the token ids up to each."""
    out = np.empty((2, stop - start, HKV, D), dtype=np.float32)
    for i, pos in enumerate(range(start, stop)):
        key = zlib.crc32(np.asarray(tokens[:pos + 1], dtype=np.int64).tobytes())
        g = np.random.default_rng([seed, pos, key])
        out[:, i] = wl.round_to(g.standard_normal((2, HKV, D)).astype(np.float32), "bf16")
    return out


@pytest.mark.parametrize("cache_dtype,prefix_kernel", [("bf16", "tcgen05"), ("bf16", "mma_sync"),
                                                       ("fp8_e4m3", "auto")])
def test_prefix_cache_hits_through_the_cascade(cache_dtype, prefix_kernel):
    from paged_kv_cache_163_gb300 import capi
    from paged_kv_cache_163_gb300.engine import PagedKVCache
    from paged_kv_cache_163_gb300.play import to_device
    capi.load()
    capi.pkv_set_prefix_kernel(prefix_kernel, 0)
    try:
        rng = np.random.default_rng(52)
        nb = 600
        order = rng.permutation(nb).astype(np.int32)
        cache = PagedKVCache(num_layers=LAYERS, num_blocks=nb, num_kv_heads=HKV, head_dim=D, cache_dtype=cache_dtype,
                             alloc_order=order, poison=True)
        cache.enable_prefix_cache(config_key=3)
        alloc = PrefixCachingAllocator(nb, 16, order, 3)
        models = [PagedCacheModel(nb, HKV, D, cache_dtype) for _ in range(LAYERS)]

        def write(seq, rows):
            n = rows.shape[1]
            slots, cs, cd = cache.append([seq] * n, to_device(rows[0], "bf16", "cuda"),
                                         to_device(rows[1], "bf16", "cuda"))
            o_slots, cows = alloc.append_slots([seq] * n)
            assert list(slots) == list(o_slots)
            for m in models:
                for src, dst in cows:
                    m.copy_block(src, dst)
                m.write(o_slots, rows[0], rows[1])

        system = rng.integers(0, 32000, 400).tolist()   # 25 full blocks: more than the cascade's 16 tiles
        seqs, tokens = [], {}
        for i in range(6):
            prompt = system + rng.integers(0, 32000, int(rng.integers(20, 150))).tolist()
            seq = 10 + i
            got, want = cache.admit(seq, prompt), alloc.admit(seq, prompt)
            assert got == want == (0 if i == 0 else 400)
            write(seq, prompt_rows(prompt, got, len(prompt)))
            assert cache.commit(seq, prompt) == alloc.commit(seq, prompt)
            seqs.append(seq)
            tokens[seq] = prompt
        c0 = cache.cascade_count()
        for step in range(4):
            n = len(seqs)
            k = np.stack([prompt_rows(tokens[s] + [step], len(tokens[s]), len(tokens[s]) + 1)[0, 0] for s in seqs])
            v = np.stack([prompt_rows(tokens[s] + [step], len(tokens[s]), len(tokens[s]) + 1)[1, 0] for s in seqs])
            for s in seqs:
                tokens[s] = tokens[s] + [step]
            q = wl.round_to(rng.standard_normal((LAYERS, n, HQ, D)).astype(np.float32), "bf16")
            out = torch.full((LAYERS, n, HQ, D), float("nan"), dtype=torch.float32, device="cuda")
            cache.step(seqs, to_device(k, "bf16", "cuda"), to_device(v, "bf16", "cuda"), to_device(q, "bf16", "cuda"),
                       scale=SCALE, out=out)
            o_slots, cows = alloc.append_slots(seqs)
            for m in models:
                for src, dst in cows:
                    m.copy_block(src, dst)
                m.write(o_slots, k, v)
            assert cache.check() == 0, f"step {step}"
            t, lens = cache.tables(seqs)
            mt, ml = alloc.block_tables(seqs, t.shape[1])
            assert t.tolist() == mt and lens.tolist() == ml, f"step {step}: tables"
            got = to_f64(out)
            for li, m in enumerate(models):
                for i, s in enumerate(seqs):
                    K, V = m.gather(alloc.tables[s], alloc.lens[s])
                    ref = decode_attention(q[li, i].astype(np.float64), K, V, SCALE)
                    assert_close(got[li, i], ref, f"step {step} layer {li} sequence {s}")
        assert cache.cascade_count() - c0 == 4, "every step should attend the shared prefix by the cascade"
        st = cache.prefix_stats()
        assert st["hits"] == 5 * 25 and st == {k2: v2 for k2, v2 in alloc.stats().items() if k2 in st}
        cache.close()
    finally:
        capi.pkv_set_prefix_kernel("auto", 0)
