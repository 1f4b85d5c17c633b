"""A request served from the prefix cache attends exactly as one computed from scratch.

Request 1 writes a 100-token prompt and commits it, then finishes.
Request 2 shares its first 96 tokens: admission maps the six cached blocks,
the request writes only the rest, and its decode output must equal, bit for
bit, that of the same request written whole into a cache without reuse (the
result does not depend on which physical blocks hold the rows).
"""
import numpy as np
import pytest

from paged_kv_cache_163_gb300 import workloads as wl

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


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
    out_a = a.decode([2], q, scale=float(np.float32(1) / np.sqrt(np.float32(d))))

    b = PagedKVCache(num_layers=1, num_blocks=32, num_kv_heads=hkv, head_dim=d, cache_dtype=cache_dtype)
    b.create(2)
    write(b, 2, rows2, 0, 120)
    out_b = b.decode([2], q, scale=float(np.float32(1) / np.sqrt(np.float32(d))))
    assert a.check() == 0 and b.check() == 0
    assert torch.equal(out_a, out_b)
    st = a.prefix_stats()
    assert st["hits"] == 6 and st["registered"] == 6
    a.close()
    b.close()
