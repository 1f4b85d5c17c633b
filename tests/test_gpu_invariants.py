"""GPU invariants the pages' semantics imply ("KV Cache 与 vLLM" (zwxr.cn) §3.2-§3.3).

* Block permutation: where the blocks live must not change the result; the
  kernel's reduction order follows logical positions, so outputs are
  bit-identical.
* Shared prefix == duplicated prefix: forked sequences reading the same
  physical blocks give bit-identical outputs to sequences holding private
  copies.
* A context of one token returns that token's V.
* Bad block ids and context lengths are reported through the device error
  word; the kernels skip the access instead of faulting.
"""
import numpy as np
import pytest

from paged_kv_cache_163_gb300 import workloads as wl

from helpers import to_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def play():
    from paged_kv_cache_163_gb300 import capi, play as p
    capi.load()
    return p


@pytest.mark.parametrize("wid", [1, 2])
def test_block_permutation_bit_identical(play, wid):
    w = wl.make(wid)
    c1, o1 = play.run(w)
    c2, o2 = play.run(w, alloc_order=np.arange(w.num_blocks, dtype=np.int32)[::-1].copy())
    t1, _ = c1.tables(w.seq_ids)
    t2, _ = c2.tables(w.seq_ids)
    assert not np.array_equal(t1, t2)
    assert torch.equal(o1, o2)
    c1.close(); c2.close()


@pytest.mark.parametrize("cache_dtype", ["bf16", "fp8_e4m3", "fp8_e5m2", "int8", "fp8_e4m3_int4"])
def test_shared_prefix_equals_private_copies(play, cache_dtype):
    prefix = 1500
    lens = [prefix + s for s in (64, 100, 512, 77, 1, 300, 250, 129)]
    w = wl.custom("share", lens=lens, num_q_heads=32, num_kv_heads=8, head_dim=128, q_dtype="bf16",
                  cache_dtype=cache_dtype, prefix_len=prefix, seed=21)
    shared, out_shared = play.run(w, cascade=False)   # same summation order as the private copies
    assert len(shared.cow_pairs) == len(lens) - 1
    # private copies: every sequence appends the whole prefix itself
    from paged_kv_cache_163_gb300.engine import PagedKVCache
    dup = PagedKVCache(num_layers=1, num_blocks=sum(-(-L // 16) for L in lens) + 8, num_kv_heads=8,
                       head_dim=128, cache_dtype=cache_dtype)
    for s, L in enumerate(lens):
        dup.create(s)
        k = play.to_device(w.kv_rows(0, s, 0, L - 1), "bf16", "cuda")
        v = play.to_device(w.kv_rows(1, s, 0, L - 1), "bf16", "cuda")
        dup.append([s] * (L - 1), k, v)
    k, v, q = play.step_inputs(w)
    out_dup = dup.step(w.seq_ids, k, v, q, scale=w.scale)
    assert dup.check() == 0 and shared.check() == 0
    assert torch.equal(out_shared, out_dup)
    shared.close(); dup.close()


@pytest.mark.parametrize("q_dtype,cache_dtype", [("f16", "f16"), ("bf16", "bf16"), ("bf16", "fp8_e4m3"),
                                                 ("bf16", "fp8_e5m2"), ("f16", "int8"), ("bf16", "fp8_e4m3_int4")])
def test_length_one_returns_v(play, q_dtype, cache_dtype):
    w = wl.custom("one", lens=[1, 1, 1], num_q_heads=16, num_kv_heads=4, head_dim=128, q_dtype=q_dtype,
                  cache_dtype=cache_dtype, outlier_p=0.01, seed=2)
    cache, out = play.run(w)
    v = w.step_rows(1)                                  # [B, Hkv, D]
    got = to_f64(out[0])
    if cache_dtype in ("fp8_e4m3", "fp8_e5m2", "int8", "fp8_e4m3_int4"):
        from oracle.cache import dequantize_rows
        want = np.repeat(dequantize_rows(v, cache_dtype, "v"), 4, axis=1)
        assert np.allclose(got, want, rtol=2 ** -8, atol=0)
    else:
        want = np.repeat(v.astype(np.float64), 4, axis=1)
        assert np.array_equal(got, want)
    cache.close()


def test_bad_block_id_and_context_len_are_flagged(play):
    from paged_kv_cache_163_gb300 import capi
    w = wl.custom("bad", lens=[40, 40], num_q_heads=8, num_kv_heads=2, head_dim=64, q_dtype="f16",
                  cache_dtype="f16", seed=3)
    cache, out = play.run(w)
    assert cache.check() == 0
    tables, lens = cache.tables(w.seq_ids)
    dev = torch.device("cuda")
    q = play.to_device(w.q_rows(0), "f16", dev)
    ws = cache.workspace(2, 8, "f16")
    bad_t = tables.copy()
    bad_t[1, 1] = w.num_blocks + 5                      # outside the pool
    capi.paged_attention_decode(torch.empty_like(q), q, cache.k[0], cache.v[0], None, None,
                                torch.from_numpy(bad_t).to(dev), torch.from_numpy(lens).to(dev),
                                int(lens.max()), w.scale, ws, d_error=cache.err)
    assert cache.check() & capi.DEVERR_BAD_BLOCK
    bad_l = lens.copy()
    bad_l[0] = tables.shape[1] * 16 + 1                 # longer than its table
    capi.paged_attention_decode(torch.empty_like(q), q, cache.k[0], cache.v[0], None, None,
                                torch.from_numpy(tables).to(dev), torch.from_numpy(bad_l).to(dev),
                                int(bad_l.max()), w.scale, ws, d_error=cache.err)
    assert cache.check() & capi.DEVERR_BAD_CONTEXT_LEN
    # the context stays usable
    out2 = cache.decode(w.seq_ids, q, scale=w.scale)
    assert cache.check() == 0 and torch.equal(out2, out[0])
    cache.close()


def test_workspace_too_small_is_rejected(play):
    from paged_kv_cache_163_gb300 import capi
    w = wl.make(1)
    cache, out = play.run(w)
    tables, lens = cache.tables(w.seq_ids)
    dev = torch.device("cuda")
    q = play.to_device(w.q_rows(0), "f16", dev)
    small = torch.empty(64, dtype=torch.uint8, device=dev)
    with pytest.raises(capi.PkvError) as e:
        capi.paged_attention_decode(torch.empty_like(q), q, cache.k[0], cache.v[0], None, None,
                                    torch.from_numpy(tables).to(dev), torch.from_numpy(lens).to(dev),
                                    int(lens.max()), w.scale, small)
    assert e.value.status == -6
    cache.close()
