"""Pins for the oracle's paged cache: paged == contiguous, permutation invariance,
shared prefix == duplicated prefix, and the concatenation cache of the pages.

"KV Cache 与 vLLM" (zwxr.cn) §3.2: the block table only changes where
tokens live, so attention through any table must equal attention over the
logically contiguous cache (§1.3's ``torch.cat`` cache); §3.3: sharing a
prefix's blocks must give the same result as private copies.
"""
import numpy as np
import pytest

from oracle.attention import decode_attention
from oracle.cache import PagedCacheModel, dequantize_rows
from oracle.model import PagedKVOracle
from paged_kv_cache_163_gb300 import workloads as wl


def play(w, alloc_order=None, layers=1):  # same as helpers.oracle_play
    o = PagedKVOracle(layers, w.num_blocks, w.num_kv_heads, w.head_dim, w.cache_dtype,
                      alloc_order=w.alloc_order if alloc_order is None else alloc_order)
    for op in w.prefill_ops():
        if op[0] == "create":
            o.create(op[1])
        elif op[0] == "fork":
            o.fork(op[1], op[2])
        else:
            seqs = op[1]              # prefill appends name one sequence
            start = o.alloc.lens[seqs[0]]
            k = w.kv_rows(0, seqs[0], start, start + len(seqs))
            v = w.kv_rows(1, seqs[0], start, start + len(seqs))
            o.append(seqs, [k] * layers, [v] * layers)
    o.append(w.seq_ids, [w.step_rows(0)] * layers, [w.step_rows(1)] * layers)
    return o


@pytest.mark.parametrize("dtype", ["f16", "bf16", "fp8_e4m3", "fp8_e4m3_int4"])
def test_paged_equals_contiguous(dtype):
    w = wl.custom("t", lens=[1, 16, 17, 45, 100], num_q_heads=8, num_kv_heads=2, head_dim=32,
                  q_dtype="bf16" if dtype.startswith("fp8") else dtype, cache_dtype=dtype, outlier_p=0.01)
    o = play(w)
    q = w.q_rows()
    out = o.decode(w.seq_ids, q, w.scale)
    for s, L in enumerate(w.context_lens):
        k = w.kv_rows(0, s, 0, int(L)); v = w.kv_rows(1, s, 0, int(L))
        K, V = o.layers[0].gather(o.alloc.tables[s], int(L))
        assert np.array_equal(K, dequantize_rows(k, dtype))
        assert np.array_equal(V, dequantize_rows(v, dtype, "v"))
        # the concatenation cache: tokens appended one by one with np.concatenate
        kc = np.zeros((0, w.num_kv_heads, w.head_dim)); vc = np.zeros_like(kc)
        for t in range(int(L)):
            kc = np.concatenate([kc, dequantize_rows(k[t:t + 1], dtype)])
            vc = np.concatenate([vc, dequantize_rows(v[t:t + 1], dtype, "v")])
        assert np.array_equal(out[s], decode_attention(q[s], kc, vc, w.scale))
    # cache length == tokens processed, and blocks held == ceil(L / 16)
    for s, L in enumerate(w.context_lens):
        assert o.alloc.lens[s] == L and len(o.alloc.tables[s]) == -(-int(L) // 16)


def test_block_permutation_invariance():
    w = wl.make(1)
    a = play(w)
    b = play(w, alloc_order=np.arange(w.num_blocks)[::-1].copy())
    assert a.alloc.tables != b.alloc.tables
    q = w.q_rows()
    assert np.array_equal(a.decode(w.seq_ids, q, w.scale), b.decode(w.seq_ids, q, w.scale))


@pytest.mark.parametrize("dtype", ["bf16", "fp8_e4m3"])
def test_shared_prefix_equals_duplicated_prefix(dtype):
    prefix, n = 45, 6
    lens = [prefix + s for s in (1, 3, 20, 5, 33, 2)]
    w = wl.custom("p", lens=lens, num_q_heads=8, num_kv_heads=2, head_dim=32, q_dtype="bf16",
                  cache_dtype=dtype, prefix_len=prefix)
    shared = play(w)
    # 45 = 2 full blocks + 13 tokens: every sharer but the last copies the partial block
    assert len(shared.cow_log) == n - 1
    assert all(src == shared.cow_log[0][0] for src, _ in shared.cow_log)
    # private copies: every sequence appends the prefix itself
    dup = PagedKVOracle(1, 200, 2, 32, dtype)
    for s, L in enumerate(lens):
        dup.create(s)
        k = w.kv_rows(0, s, 0, L); v = w.kv_rows(1, s, 0, L)
        dup.append([s] * L, [k], [v])
    q = w.q_rows()
    assert np.array_equal(shared.decode(w.seq_ids, q, w.scale), dup.decode(w.seq_ids, q, w.scale))
    # the shared blocks are held once
    full_prefix_blocks = prefix // 16
    assert all(shared.alloc.refcount[b] == n for b in shared.alloc.tables[0][:full_prefix_blocks])


def test_cow_copy_moves_whole_block():
    c = PagedCacheModel(4, 2, 8, "fp8_e4m3")
    rng = np.random.default_rng(0)
    c.write([16 + 3, 16 + 4], rng.standard_normal((2, 2, 8)).astype(np.float32),
            rng.standard_normal((2, 2, 8)).astype(np.float32))
    c.copy_block(1, 3)
    assert np.array_equal(c.k[3], c.k[1]) and np.array_equal(c.v_scale[3], c.v_scale[1], equal_nan=True)
    assert c.filled[3].sum() == 2


def test_length_one_paged_returns_v_exactly():
    w = wl.make(1)
    o = play(w)
    out = o.decode(w.seq_ids, w.q_rows(), w.scale)
    v0 = w.kv_rows(1, 0, 0, 1)[0]                   # seq 0 has L = 1
    assert np.array_equal(out[0], np.repeat(v0, w.group, axis=0))
