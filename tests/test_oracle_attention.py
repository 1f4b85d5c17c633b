"""Pins for the oracle's decode attention, split/merge model and causal recompute.

Each test anchors the oracle to something other than itself: printed
closed forms, special cases whose answer is known in closed form, an
independent loop form, and the no-cache full recompute that a cached
decode must reproduce ("KV Cache 与 vLLM" (zwxr.cn) §1.2-§1.3).
"""
import math

import numpy as np
import pytest

from oracle.attention import (causal_attention_all_positions, decode_attention,
                              decode_attention_loops, lse_merge, split_partials)


def test_two_token_closed_form():
    # q . k1 = 2, q . k2 = 0, scale 1/2 -> scores (1, 0) -> weights (e, 1) / (e + 1)
    d = 4
    q = np.zeros((1, d)); q[0, 0] = 1.0
    K = np.zeros((2, 1, d)); K[0, 0, 0] = 2.0
    V = np.zeros((2, 1, d)); V[0, 0] = [1, 2, 3, 4]; V[1, 0] = [-1, 0, 5, 0]
    out = decode_attention(q, K, V, 0.5)
    w1 = math.e / (math.e + 1)
    w2 = 1 / (math.e + 1)
    assert np.allclose(out[0], w1 * V[0, 0] + w2 * V[1, 0], rtol=0, atol=1e-15)


def test_scale_is_applied_not_inverted():
    # same keys, scale 2 vs scale 1/2 give different, predictable weights
    q = np.array([[1.0, 0.0]])
    K = np.array([[[1.0, 0.0]], [[0.0, 0.0]]])
    V = np.array([[[1.0, 0.0]], [[0.0, 1.0]]])
    for scale in (2.0, 0.5, 1 / math.sqrt(2)):
        out = decode_attention(q, K, V, scale)
        w = 1 / (1 + math.exp(-scale))
        assert np.allclose(out[0], [w, 1 - w], atol=1e-15)


def test_length_one_returns_v():
    rng = np.random.default_rng(0)
    q = rng.standard_normal((8, 64))
    K = rng.standard_normal((1, 2, 64))
    V = rng.standard_normal((1, 2, 64))
    out = decode_attention(q, K, V, 0.125)
    assert np.array_equal(out[:4], np.repeat(V[0, 0][None], 4, 0))
    assert np.array_equal(out[4:], np.repeat(V[0, 1][None], 4, 0))


def test_empty_context_is_zero():
    out = decode_attention(np.ones((4, 8)), np.zeros((0, 2, 8)), np.zeros((0, 2, 8)), 1.0)
    assert np.array_equal(out, np.zeros((4, 8)))


def test_zero_scale_or_equal_keys_give_mean():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((4, 16))
    V = rng.standard_normal((37, 1, 16))
    K = rng.standard_normal((37, 1, 16))
    assert np.allclose(decode_attention(q, K, V, 0.0), V[:, 0].mean(0)[None].repeat(4, 0), atol=1e-14)
    Ksame = np.repeat(K[:1], 37, 0)
    assert np.allclose(decode_attention(q, Ksame, V, 0.3), V[:, 0].mean(0)[None].repeat(4, 0), atol=1e-14)


def test_gqa_head_mapping_is_contiguous():
    # 8 q heads, 2 kv heads: heads 0-3 read kv head 0, heads 4-7 kv head 1
    rng = np.random.default_rng(2)
    K = rng.standard_normal((5, 2, 8))
    V = np.zeros((5, 2, 8)); V[:, 0] = 1.0; V[:, 1] = -3.0
    out = decode_attention(rng.standard_normal((8, 8)), K, V, 0.2)
    assert np.allclose(out[:4], 1.0) and np.allclose(out[4:], -3.0)


def test_dominant_key_and_no_overflow():
    d = 32
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, d))
    K = rng.standard_normal((50, 1, d))
    K[17, 0] = q[0] * 50.0              # score ~ 50 |q|^2 * scale, far above the rest
    V = rng.standard_normal((50, 1, d))
    out = decode_attention(q, K, V, 10.0)
    assert np.all(np.isfinite(out))
    assert np.allclose(out[0], V[17, 0], atol=1e-12)


@pytest.mark.parametrize("hq,hkv,d,L", [(8, 2, 8, 1), (8, 2, 8, 17), (4, 4, 6, 9), (6, 1, 5, 23)])
def test_matches_loop_form(hq, hkv, d, L):
    rng = np.random.default_rng(hq * 100 + L)
    q = rng.standard_normal((hq, d))
    K = rng.standard_normal((L, hkv, d))
    V = rng.standard_normal((L, hkv, d))
    a = decode_attention(q, K, V, 1 / math.sqrt(d))
    b = decode_attention_loops(q.tolist(), K.tolist(), V.tolist(), 1 / math.sqrt(d))
    assert np.allclose(a, b, rtol=1e-13, atol=1e-13)


def test_cached_decode_equals_full_causal_recompute():
    # generate T tokens; at step t the cache holds tokens 0..t and the new query attends over it
    rng = np.random.default_rng(4)
    T, hq, hkv, d = 40, 4, 2, 16
    Q = rng.standard_normal((T, hq, d))
    K = rng.standard_normal((T, hkv, d))
    V = rng.standard_normal((T, hkv, d))
    full = causal_attention_all_positions(Q, K, V, 0.25)
    k_cache = np.zeros((0, hkv, d)); v_cache = np.zeros((0, hkv, d))
    for t in range(T):
        k_cache = np.concatenate([k_cache, K[t:t + 1]])     # append, then attend
        v_cache = np.concatenate([v_cache, V[t:t + 1]])
        assert len(k_cache) == t + 1                        # cache length == tokens processed
        step = decode_attention(Q[t], k_cache, v_cache, 0.25)
        assert np.allclose(step, full[t], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("bounds", [
    [(0, 100)],
    [(0, 16), (16, 32), (32, 100)],
    [(0, 1), (1, 99), (99, 100)],
    [(0, 50), (50, 50), (50, 100)],         # an empty split
    [(0, 0), (0, 100), (100, 100)],
])
def test_split_merge_equals_unsplit(bounds):
    rng = np.random.default_rng(5)
    q = rng.standard_normal((8, 32))
    K = rng.standard_normal((100, 2, 32)) * 3
    V = rng.standard_normal((100, 2, 32))
    whole = decode_attention(q, K, V, 0.3)
    merged = lse_merge(split_partials(q, K, V, 0.3, bounds))
    assert np.allclose(merged, whole, rtol=1e-12, atol=1e-12)


def test_merge_of_all_empty_is_zero():
    q = np.ones((2, 4)); K = np.zeros((0, 1, 4)); V = np.zeros((0, 1, 4))
    assert np.array_equal(lse_merge(split_partials(q, K, V, 1.0, [(0, 0), (0, 0)])), np.zeros((2, 4)))
