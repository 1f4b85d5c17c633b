"""Pins for the oracle's prefix cache (hash chain, reuse, chain-aware eviction).

The hash is pinned to the published FNV-1a-64 test vectors.  Reuse is
pinned to the pages' worked figures (tests/golden/prefix_cache_examples.json)
and to what "identical prefix, block by block" implies.  Eviction is pinned
to the pages' rule that a middle block must not go before the blocks that
depend on it, plus least-recently-used order between chains.
"""
import json
import os
import random

import pytest

from oracle.allocator import NoBlocks
from oracle.prefix_cache import PrefixCachingAllocator, block_hash, fnv1a64

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "prefix_cache_examples.json")


def test_fnv1a64_published_vectors():
    assert fnv1a64(b"") == 0xCBF29CE484222325
    assert fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert fnv1a64(b"foobar") == 0x85944171F73967E8


def test_block_hash_depends_on_every_input():
    toks = list(range(16))
    h = block_hash(0, toks, 7)
    assert block_hash(0, toks, 7) == h
    for j in range(16):
        t2 = list(toks)
        t2[j] += 1
        assert block_hash(0, t2, 7) != h
    assert block_hash(1, toks, 7) != h
    assert block_hash(0, toks, 8) != h
    # negative ids are hashed as their 32-bit two's complement
    assert block_hash(0, [-1] * 16, 0) == block_hash(0, [0xFFFFFFFF] * 16, 0)


def _prompt(n, seed):
    r = random.Random(seed)
    return [r.randrange(0, 128000) for _ in range(n)]


def _prefill(a, seq, tokens):
    """Admit, write the rest of the prompt, commit; return the cached token count."""
    cached = a.admit(seq, tokens)
    for _ in range(len(tokens) - cached):
        a.append_slots([seq])
    a.commit(seq, tokens)
    return cached


@pytest.mark.parametrize("ex", json.load(open(GOLDEN))["examples"], ids=lambda e: e["id"])
def test_pages_worked_examples(ex):
    n, seen = ex["inputs"]["request_tokens"], ex["inputs"]["seen_tokens"]
    a = PrefixCachingAllocator(1024)
    prompt = _prompt(n, 1)
    assert _prefill(a, 0, prompt[:seen]) == 0
    a.free_seq(0)
    cached = a.admit(1, prompt)
    assert cached == ex["reused_tokens"]
    assert cached / n >= ex["printed_share_min"]


def test_one_changed_token_stops_reuse_at_its_block():
    base = _prompt(160, 2)
    for k in range(10):
        a = PrefixCachingAllocator(64)
        _prefill(a, 0, base)
        probe = list(base)
        probe[16 * k + 5] += 1
        assert a.admit(1, probe + [9]) == 16 * k


def test_config_key_is_part_of_the_key():
    base = _prompt(64, 3)
    a = PrefixCachingAllocator(64, config_key=1)
    _prefill(a, 0, base)
    b = PrefixCachingAllocator(64, config_key=2)
    _prefill(b, 0, base)
    assert a.admit(1, base + [1]) == 64
    assert block_hash(0, base[:16], 1) != block_hash(0, base[:16], 2)


def test_at_least_one_prompt_token_is_computed():
    base = _prompt(32, 4)
    a = PrefixCachingAllocator(16)
    _prefill(a, 0, base)
    assert a.admit(1, base) == 16          # two cached blocks, but the last token must run
    assert a.admit(2, base[:17]) == 16
    assert a.admit(3, base[:16]) == 0
    assert a.admit(4, []) == 0


def test_shared_blocks_are_referenced_and_survive_release():
    base = _prompt(48, 5)
    a = PrefixCachingAllocator(16)
    _prefill(a, 0, base)
    t0 = list(a.tables[0])
    assert a.admit(1, base + [3]) == 48
    assert a.tables[1] == t0 and all(a.refcount[b] == 2 for b in t0)
    a.free_seq(0)
    a.free_seq(1)
    assert all(a.refcount[b] == 0 for b in t0)
    assert a.num_free() == 16 and len(a.free) == 13   # three cached blocks stay out of the FIFO
    assert a.admit(2, base + [4]) == 48 and a.tables[2] == t0


def test_eviction_takes_leaves_deepest_first_and_never_orphans():
    base = _prompt(64, 6)
    a = PrefixCachingAllocator(4)
    _prefill(a, 0, base)
    chain = list(a.tables[0])
    a.free_seq(0)
    assert a.num_free() == 4 and not a.free
    a.create(9)
    got = []
    for _ in range(4):
        a.append_slots([9] * 16)
        got.append(a.tables[9][-1])
    assert got == chain[::-1]                 # same release tick: the deepest block goes first
    assert a.evictions == 4 and not a.by_hash


def test_least_recently_released_chain_goes_first():
    p, q = _prompt(32, 7), _prompt(32, 8)
    a = PrefixCachingAllocator(6)
    _prefill(a, 0, p)
    _prefill(a, 1, q)
    tp, tq = list(a.tables[0]), list(a.tables[1])
    a.free_seq(1)                            # q released first
    a.free_seq(0)
    a.create(9)
    a.append_slots([9] * (16 * 2 + 16 * 2 + 1))   # needs 5 blocks: 2 free + 3 evicted
    assert a.tables[9][2:5] == [tq[1], tq[0], tp[1]]
    assert a.admit(10, p + [1]) == 16 and a.admit(11, q + [1]) == 0


def test_all_or_nothing_counts_evictable_blocks():
    base = _prompt(32, 9)
    a = PrefixCachingAllocator(3)
    _prefill(a, 0, base)
    a.free_seq(0)
    a.create(5)
    with pytest.raises(NoBlocks):
        a.append_slots([5] * (16 * 3 + 1))
    assert a.tables[5] == [] and len(a.by_hash) == 2 and a.evictions == 0
    a.append_slots([5] * 48)
    assert a.evictions == 2


def test_duplicate_content_stays_private():
    base = _prompt(32, 10)
    a = PrefixCachingAllocator(8)
    a.create(0)
    a.append_slots([0] * 32)
    a.create(1)
    a.append_slots([1] * 32)
    assert a.commit(0, base) == 2
    assert a.commit(1, base) == 0            # same hashes already registered to seq 0's blocks
    t1 = list(a.tables[1])
    a.free_seq(1)
    assert list(a.free)[-2:] == t1           # never registered: back to the FIFO


def test_commit_stops_at_a_duplicate_block():
    base = _prompt(48, 12)
    a = PrefixCachingAllocator(10)
    for s in (0, 1):
        a.create(s)
        a.append_slots([s] * 48)
    assert a.commit(0, base[:16]) == 1       # seq 0 registers only its first block
    assert a.commit(1, base) == 0            # seq 1's first block duplicates it: nothing registered
    first = a.tables[0][0]
    a.free_seq(0)                            # seq 0's blocks: the registered one stays cached, a leaf
    assert a.reg.keys() == {first} and a._victim() == first


def test_random_trace_invariants():
    rng = random.Random(11)
    prompts = [_prompt(rng.randrange(1, 120), 100 + i) for i in range(6)]
    a = PrefixCachingAllocator(40)
    live = {}
    for step in range(400):
        op = rng.random()
        if op < 0.4 and len(live) < 6:
            sid = step
            base = prompts[rng.randrange(6)]
            cut = rng.randrange(1, len(base) + 1)
            toks = base[:cut] + _prompt(rng.randrange(0, 20), step)
            try:
                cached = a.admit(sid, toks)
                for _ in range(len(toks) - cached):
                    a.append_slots([sid])
                a.commit(sid, toks)
                live[sid] = toks
            except NoBlocks:
                a.free_seq(sid)
        elif live:
            sid = rng.choice(sorted(live))
            a.free_seq(sid)
            del live[sid]
        # conservation: every block is free, cached-unreferenced, or referenced
        held = sum(a.refcount)
        assert held == sum(len(t) for t in a.tables.values())
        assert len(a.free) + len(a._evictable()) + sum(1 for r in a.refcount if r > 0) == a.num_blocks
        # a registered block's parent is registered too (no orphaned chain), and
        # whoever holds a block holds its parent
        for b, (h, parent, depth, _) in a.reg.items():
            assert a.by_hash[h] == b
            assert (parent == -1) == (depth == 0)
            if parent >= 0:
                assert parent in a.reg
                assert a.refcount[parent] >= a.refcount[b]
                assert all(t[depth - 1] == parent for t in a.tables.values() if len(t) > depth and t[depth] == b)
        if a._evictable():
            assert any(a.children[b] == 0 for b in a._evictable())
        for b in range(a.num_blocks):
            assert a.children[b] == sum(1 for r in a.reg.values() if r[1] == b)
