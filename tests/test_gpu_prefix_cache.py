"""Prefix caching on the GPU, checked against the fp64 oracle.

The pages' second sharing mechanism ("KV Cache优化实战" §5.2;
"企业官网建设流程全解析" §6.2-§6.3): a request whose prompt starts with
blocks already in the cache maps them at admission, writes only the rest
of its prompt, and attends over the cached blocks and its own.

Two checks:

* a trace of requests sharing a system prompt, in a pool small enough that
  released chains are evicted, played on the native block manager + GPU
  cache and on the oracle's ``PrefixCachingAllocator`` + ``PagedCacheModel``:
  admitted token counts, commits, block tables and lengths bit-exact after
  every call; every filled cache slot (codes and scales for coded caches)
  bit-exact; every decode output (fp32) within max |err| <= 1e-2 and
  relative L2 <= 2e-3 of ``decode_attention``; the counters equal at the end;
* a request served from the cache attends bit-identically to the same
  request written whole into a cache without reuse (the result does not
  depend on which physical blocks hold the rows).
"""
import zlib

import numpy as np
import pytest

from oracle.attention import decode_attention
from oracle.cache import PagedCacheModel
from oracle.prefix_cache import PrefixCachingAllocator
from paged_kv_cache_163_gb300 import workloads as wl

from helpers import assert_close, compare_cache_bytes, to_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

HKV, HQ, D = 4, 16, 128
SCALE = float(np.float32(1) / np.sqrt(np.float32(D)))


class RowSource:
    """K/V rows of a prompt position, a function of the token ids up to it.

    Identical prefixes give identical rows, as they would in a model, so a
    cached block holds exactly what recomputing it would write.  Values are
    N(0, 1) rounded to bf16, times 20 on a Bernoulli(outlier_p) mask.
    """

    def __init__(self, seed, outlier_p):
        self.seed, self.p = seed, outlier_p

    def rows(self, tokens, start, stop):
        out = np.empty((2, stop - start, HKV, D), dtype=np.float32)
        for i, pos in enumerate(range(start, stop)):
            key = zlib.crc32(np.asarray(tokens[:pos + 1], dtype=np.int64).tobytes())
            g = np.random.default_rng([self.seed, pos, key])
            x = g.standard_normal((2, HKV, D)).astype(np.float32)
            if self.p:
                x = np.where(g.random((2, HKV, D)) < self.p, x * np.float32(20), x)
            out[:, i] = wl.round_to(x, "bf16")
        return out


class Pair:
    """The native cache and the oracle, driven by the same calls."""

    def __init__(self, num_blocks, cache_dtype, alloc_order, config_key=11):
        from paged_kv_cache_163_gb300.engine import PagedKVCache
        self.gpu = PagedKVCache(num_layers=1, num_blocks=num_blocks, num_kv_heads=HKV, head_dim=D,
                                cache_dtype=cache_dtype, alloc_order=alloc_order)
        self.gpu.enable_prefix_cache(config_key=config_key)
        self.alloc = PrefixCachingAllocator(num_blocks, 16, alloc_order, config_key)
        self.model = PagedCacheModel(num_blocks, HKV, D, cache_dtype)
        self.dtype = cache_dtype

    def admit(self, seq, tokens):
        got = self.gpu.admit(seq, tokens)
        want = self.alloc.admit(seq, tokens)
        assert got == want, f"admit {seq}: {got} cached tokens, oracle {want}"
        self.check_table(seq)
        return got

    def append(self, seq, rows):
        from paged_kv_cache_163_gb300.play import to_device
        n = rows.shape[1]
        slots, _, _ = self.gpu.append([seq] * n, to_device(rows[0], "bf16", "cuda"),
                                      to_device(rows[1], "bf16", "cuda"))
        o_slots, cows = self.alloc.append_slots([seq] * n)
        assert list(slots) == list(o_slots)
        for src, dst in cows:
            self.model.copy_block(src, dst)
        self.model.write(o_slots, rows[0], rows[1])
        self.check_table(seq)

    def commit(self, seq, tokens):
        got = self.gpu.commit(seq, tokens)
        want = self.alloc.commit(seq, tokens)
        assert got == want, f"commit {seq}: {got} blocks, oracle {want}"

    def free(self, seq):
        self.gpu.free(seq)
        self.alloc.free_seq(seq)
        assert self.gpu.prefix_stats()["evictable"] == self.alloc.stats()["evictable"]

    def check_table(self, seq):
        t, lens = self.gpu.tables([seq])
        mt, ml = self.alloc.block_tables([seq], t.shape[1])
        assert t.tolist() == mt and lens.tolist() == ml, f"table of {seq}"

    def decode(self, seq, q):
        """fp32 GPU output [Hq, D] of one sequence, checked against the oracle."""
        from paged_kv_cache_163_gb300.play import to_device
        qd = to_device(q[None], "bf16", "cuda")
        out = torch.empty(qd.shape, dtype=torch.float32, device="cuda")
        self.gpu.decode([seq], qd, scale=SCALE, out=out)
        assert self.gpu.check() == 0
        K, V = self.model.gather(self.alloc.tables[seq], self.alloc.lens[seq])
        ref = decode_attention(q.astype(np.float64), K, V, SCALE)
        assert_close(to_f64(out[0]), ref, f"{self.dtype} sequence {seq}")
        return out

    def check_bytes(self):
        torch.cuda.synchronize()
        compare_cache_bytes(self.gpu, self.model, self.dtype)

    def check_stats(self):
        got, want = self.gpu.prefix_stats(), self.alloc.stats()
        for k in ("lookups", "hits", "evictions", "registered", "evictable"):
            assert got[k] == want[k], f"{k}: {got[k]} vs oracle {want[k]}"


@pytest.mark.parametrize("cache_dtype,outlier_p", [("bf16", 0.0), ("fp8_e4m3", 0.001), ("int8", 0.001),
                                                   ("fp8_e4m3_int4", 0.001)])
def test_prefix_cache_trace_matches_oracle(cache_dtype, outlier_p):
    from paged_kv_cache_163_gb300 import capi
    capi.load()
    rng = np.random.default_rng(163)
    num_blocks = 32
    order = rng.permutation(num_blocks)
    pair = Pair(num_blocks, cache_dtype, order)
    src = RowSource(5, outlier_p)
    system = rng.integers(0, 32000, 70).tolist()           # 4 full blocks + 6 tokens
    live = []
    hits_seen = 0
    for i in range(14):
        if i % 4 == 3:
            # another system prompt now and then: a chain the earlier ones must make room for
            prompt = rng.integers(0, 32000, int(rng.integers(40, 120))).tolist()
        else:
            prompt = system + rng.integers(0, 32000, int(rng.integers(1, 90))).tolist()
        seq = 100 + i
        cached = pair.admit(seq, prompt)
        hits_seen += cached > 0
        rows = src.rows(prompt, 0, len(prompt))
        if len(prompt) > cached:
            pair.append(seq, rows[:, cached:])
        pair.commit(seq, prompt)
        # one decode step: append the new token, attend
        step_tokens = prompt + [int(rng.integers(0, 32000))]
        pair.append(seq, src.rows(step_tokens, len(prompt), len(prompt) + 1))
        q = wl.round_to(rng.standard_normal((HQ, D)).astype(np.float32), "bf16")
        pair.decode(seq, q)
        live.append(seq)
        # release the oldest requests so the pool keeps cycling through cached chains
        while len(live) > 2:
            pair.free(live.pop(0))
        pair.check_bytes()
    assert hits_seen >= 8
    pair.check_stats()
    assert pair.alloc.stats()["evictions"] > 0, "the trace should evict"
    for seq in live:
        pair.free(seq)
    pair.check_stats()
    pair.gpu.close()


@pytest.mark.parametrize("cache_dtype", ["bf16", "fp8_e4m3"])
def test_prefix_hit_equals_recompute(cache_dtype):
    from paged_kv_cache_163_gb300 import capi
    from paged_kv_cache_163_gb300.engine import PagedKVCache
    from paged_kv_cache_163_gb300.play import to_device
    capi.load()
    rng = np.random.default_rng(3)
    hkv, hq, d = 4, 16, 128
    p1 = rng.integers(0, 32000, 100).tolist()
    p2 = p1[:96] + rng.integers(0, 32000, 24).tolist()
    rows1 = wl.round_to(rng.standard_normal((2, 100, hkv, d)).astype(np.float32), "bf16")
    rows2 = np.concatenate([rows1[:, :96], wl.round_to(rng.standard_normal((2, 24, hkv, d)).astype(np.float32),
                                                       "bf16")], axis=1)
    q = to_device(wl.round_to(rng.standard_normal((1, hq, d)).astype(np.float32), "bf16"), "bf16", "cuda")

    def write(cache, seq, rows, start, stop):
        k = to_device(rows[0, start:stop], "bf16", "cuda")
        v = to_device(rows[1, start:stop], "bf16", "cuda")
        cache.append([seq] * (stop - start), k, v)

    a = PagedKVCache(num_layers=1, num_blocks=32, num_kv_heads=hkv, head_dim=d, cache_dtype=cache_dtype)
    a.enable_prefix_cache(config_key=7)
    assert a.admit(1, p1) == 0
    write(a, 1, rows1, 0, 100)
    assert a.commit(1, p1) == 6
    a.free(1)
    assert a.admit(2, p2) == 96
    write(a, 2, rows2, 96, 120)
    out_a = a.decode([2], q, scale=SCALE)

    b = PagedKVCache(num_layers=1, num_blocks=32, num_kv_heads=hkv, head_dim=d, cache_dtype=cache_dtype)
    b.create(2)
    write(b, 2, rows2, 0, 120)
    out_b = b.decode([2], q, scale=SCALE)
    assert a.check() == 0 and b.check() == 0
    assert torch.equal(out_a, out_b)
    st = a.prefix_stats()
    assert st["hits"] == 6 and st["registered"] == 6
    a.close()
    b.close()
