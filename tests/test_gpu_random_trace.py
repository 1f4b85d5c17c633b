"""Random traces through the step executor against the oracle, step by step.

Sequences are created with prompts of random length, forked (sharing their
blocks), freed, and stepped over two layers, with the cascade on (forks
make shared prefixes) and, in one case, graph replay.  After every step the
block tables, context lengths and copy-on-write pairs must equal the oracle
allocator's bit for bit, and every layer's output must match the oracle's
fp64 attention within the tolerance.
"""
import numpy as np
import pytest

from oracle.model import PagedKVOracle
from paged_kv_cache_163_gb300 import workloads as wl

from helpers import assert_close, to_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def play():
    from paged_kv_cache_163_gb300 import capi, play as p
    capi.load()
    return p


def _rows(rng, n, hkv, d, dtype):
    x = rng.standard_normal((n, hkv, d)).astype(np.float32)
    return wl.round_to(x, dtype)


class _Buffers:
    """One set of step buffers per batch size, so a graph sees the same pointers step after step."""

    def __init__(self, play, layers, hq, hkv, d, dtype):
        self.play, self.shape, self.dtype, self.sets = play, (layers, hq, hkv, d), dtype, {}

    def fill(self, k, v, q):
        n = k.shape[0]
        layers, hq, hkv, d = self.shape
        if n not in self.sets:
            td = torch.bfloat16 if self.dtype == "bf16" else torch.float16
            self.sets[n] = (torch.empty((n, hkv, d), dtype=td, device="cuda"),
                            torch.empty((n, hkv, d), dtype=td, device="cuda"),
                            torch.empty((layers, n, hq, d), dtype=td, device="cuda"),
                            torch.empty((layers, n, hq, d), dtype=torch.float32, device="cuda"))
        kb, vb, qb, ob = self.sets[n]
        for dst, src in ((kb, k), (vb, v), (qb, q)):
            dst.copy_(self.play.to_device(src, self.dtype, "cuda"))
        ob.fill_(float("nan"))
        return kb, vb, qb, ob


@pytest.mark.parametrize("cache_dtype,bs,graphs,seed", [("bf16", 16, False, 1), ("fp8_e4m3", 16, False, 2),
                                                        ("int8", 32, False, 3), ("fp8_e4m3_int4", 16, False, 5),
                                                        ("bf16", 16, True, 4)])
def test_random_trace_matches_oracle(play, cache_dtype, bs, graphs, seed):
    from paged_kv_cache_163_gb300.engine import PagedKVCache
    rng = np.random.default_rng(seed)
    layers, hq, hkv, d, q_dtype = 2, 16, 4, 128, "bf16"
    nb = 4000
    order = rng.permutation(nb).astype(np.int32)
    cache = PagedKVCache(num_layers=layers, num_blocks=nb, num_kv_heads=hkv, head_dim=d, cache_dtype=cache_dtype,
                         alloc_order=order, block_size=bs, poison=True)
    cache.use_graphs(graphs)
    oracle = PagedKVOracle(layers, nb, hkv, d, cache_dtype, block_size=bs, alloc_order=order)
    bufs = _Buffers(play, layers, hq, hkv, d, q_dtype)
    scale = float(np.float32(1.0) / np.sqrt(np.float32(d)))
    live, nxt, cascades, replays = [], 0, 0, 0
    for step in range(24):
        # lifecycle: new prompts, forks, frees (every fourth step only with graphs,
        # so that the batch stays the same for the steps between)
        if not graphs or step % 4 == 0:
            for _ in range(int(rng.integers(0, 3)) if len(live) > 1 else 4):
                if len(live) >= 16:
                    break
                s, nxt = nxt, nxt + 1
                n = int(rng.integers(1, 700))
                k, v = _rows(rng, n, hkv, d, q_dtype), _rows(rng, n, hkv, d, q_dtype)
                cache.create(s)
                oracle.create(s)
                cache.append([s] * n, play.to_device(k, q_dtype, "cuda"), play.to_device(v, q_dtype, "cuda"))
                oracle.append([s] * n, [k] * layers, [v] * layers)
                live.append(s)
            if rng.random() < 0.6:
                for _ in range(int(rng.integers(1, 4))):
                    p, c = live[int(rng.integers(len(live)))], nxt
                    nxt += 1
                    cache.fork(p, c)
                    oracle.fork(p, c)
                    live.append(c)
            while len(live) > 12 or (len(live) > 4 and rng.random() < 0.3):
                s = live.pop(int(rng.integers(len(live))))
                cache.free(s)
                oracle.free(s)
        # a step over a random subset (all live sequences with graphs)
        if graphs:
            ids = list(live)
        else:
            ids = sorted(rng.choice(live, size=int(rng.integers(1, len(live) + 1)), replace=False).tolist())
        n = len(ids)
        k, v = _rows(rng, n, hkv, d, q_dtype), _rows(rng, n, hkv, d, q_dtype)
        q = np.stack([_rows(rng, n, hq, d, q_dtype) for _ in range(layers)])
        kb, vb, qb, ob = bufs.fill(k, v, q)
        st = cache._stepper
        c0, r0 = cache.cascade_count(), cache.graph_stats()[1]
        cache.step(ids, kb, vb, qb, scale=scale, out=ob)
        same = cache._stepper is st
        cascades += cache.cascade_count() - (c0 if same else 0)
        replays += cache.graph_stats()[1] - (r0 if same else 0)
        oracle.append(ids, [k] * layers, [v] * layers)
        assert cache.check() == 0, f"step {step}"
        t, lens = cache.tables(ids)
        mt, ml = oracle.alloc.block_tables(ids, t.shape[1])
        assert t.tolist() == mt and lens.tolist() == ml, f"step {step}: tables"
        assert cache.cow_pairs == oracle.cow_log, f"step {step}: copy-on-write pairs"
        got = to_f64(ob)
        for li in range(layers):
            ref = oracle.decode(ids, q[li], scale, layer=li)
            for i, s in enumerate(ids):
                assert_close(got[li, i], ref[i], f"step {step} layer {li} sequence {s}")
    if graphs:
        assert replays > 0
    else:
        assert cascades > 0
    cache.close()
