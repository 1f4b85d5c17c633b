"""The native prefix cache against the oracle, bit for bit (host code only).

Same calls on the C++ block manager and on the oracle model: admissions,
appends, commits, releases, single-block frees.  After every call the
tables, lengths, reference counts, FIFO free list, free capacity, hit and
eviction counters must agree, and so must every return value and every
out-of-blocks refusal.
"""
import os

import numpy as np
import pytest

from oracle.allocator import NoBlocks
from oracle.prefix_cache import PrefixCachingAllocator, block_hash
from paged_kv_cache_163_gb300 import build, capi


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not os.path.exists(capi.LIB_PATH):
        build.build()
    return capi.load()


def test_block_hash_matches_oracle():
    rng = np.random.default_rng(1)
    for _ in range(300):
        parent = int(rng.integers(0, 2 ** 63)) * 2 + int(rng.integers(0, 2))
        key = int(rng.integers(0, 2 ** 63)) * 2 + int(rng.integers(0, 2))
        toks = rng.integers(-2 ** 31, 2 ** 31, 16).tolist()
        assert capi.pkv_block_hash(parent, toks, key) == block_hash(parent, toks, key)


class Mirror:
    def __init__(self, n, key, order=None):
        self.bm = capi.pkv_bm_create(n, 16, order)
        capi.pkv_bm_enable_prefix_cache(self.bm, key)
        self.m = PrefixCachingAllocator(n, 16, order, config_key=key)

    def same(self):
        m = self.m
        assert list(capi.pkv_bm_free_list(self.bm)) == list(m.free)
        assert capi.pkv_bm_num_free(self.bm) == m.num_free()
        for b in range(m.num_blocks):
            assert capi.pkv_bm_refcount(self.bm, b) == m.refcount[b]
        st = capi.pkv_prefix_cache_stats(self.bm)
        assert st == m.stats()
        seqs = sorted(m.tables)
        if seqs:
            mb = max(1, max(len(t) for t in m.tables.values()))
            t, lens = capi.pkv_build_block_tables(self.bm, seqs, mb)
            mt, ml = m.block_tables(seqs, mb)
            assert t.tolist() == mt and lens.tolist() == ml

    def append(self, batch):
        try:
            ms, mc = self.m.append_slots(batch)
        except NoBlocks:
            with pytest.raises(capi.NoBlocksError):
                capi.pkv_seq_append_slots(self.bm, batch)
            return False
        s, a, b = capi.pkv_seq_append_slots(self.bm, batch)
        assert s.tolist() == ms and list(zip(a.tolist(), b.tolist())) == mc
        return True


def _prompts(rng, k):
    """k base prompts, and variants that share their prefixes."""
    bases = [rng.integers(0, 50000, int(rng.integers(1, 150))).tolist() for _ in range(k)]
    return bases


@pytest.mark.parametrize("trial", range(12))
def test_random_traces_match_oracle(trial):
    rng = np.random.default_rng(100 + trial)
    n = int(rng.integers(6, 60))
    key = int(rng.integers(0, 2 ** 62))
    mir = Mirror(n, key, rng.permutation(n))
    bases = _prompts(rng, 4)
    live, nid = {}, 0
    for _ in range(120):
        op = int(rng.integers(0, 10))
        if op < 4 or not live:
            base = bases[int(rng.integers(len(bases)))]
            cut = int(rng.integers(0, len(base) + 1))
            toks = base[:cut] + rng.integers(0, 50000, int(rng.integers(0, 40))).tolist()
            sid = nid
            nid += 1
            got = capi.pkv_seq_admit(mir.bm, sid, toks)
            assert got == mir.m.admit(sid, toks)
            ok = mir.append([sid] * (len(toks) - got)) if len(toks) > got else True
            if ok:
                assert capi.pkv_seq_commit_prefix(mir.bm, sid, toks) == mir.m.commit(sid, toks)
                live[sid] = toks
            else:
                capi.pkv_seq_free(mir.bm, sid)
                mir.m.free_seq(sid)
        elif op < 6:
            sid = list(live)[int(rng.integers(len(live)))]
            capi.pkv_seq_free(mir.bm, sid)
            mir.m.free_seq(sid)
            del live[sid]
        elif op < 8:
            batch = [list(live)[int(i)] for i in rng.integers(0, len(live), int(rng.integers(1, 20)))]
            if mir.append(batch):
                for s in batch:
                    live[s] = live[s] + [7]
        elif op == 8:
            sid = list(live)[int(rng.integers(len(live)))]
            cut = int(rng.integers(0, len(live[sid]) + 1))
            got = capi.pkv_seq_commit_prefix(mir.bm, sid, live[sid][:cut])
            assert got == mir.m.commit(sid, live[sid][:cut])
        else:
            try:
                b = mir.m.alloc_block()
                ok = True
            except NoBlocks:
                ok = False
            if ok:
                assert capi.kv_block_alloc(mir.bm) == b
                capi.kv_block_free(mir.bm, b)
                mir.m.release_block(b)
            else:
                with pytest.raises(capi.NoBlocksError):
                    capi.kv_block_alloc(mir.bm)
        mir.same()
    for sid in list(live):
        capi.pkv_seq_free(mir.bm, sid)
        mir.m.free_seq(sid)
    mir.same()
    assert capi.pkv_bm_num_free(mir.bm) == n
    capi.pkv_bm_destroy(mir.bm)


def test_admit_and_commit_need_the_cache_enabled():
    bm = capi.pkv_bm_create(8, 16)
    with pytest.raises(capi.PkvError):
        capi.pkv_seq_admit(bm, 0, list(range(40)))
    capi.pkv_bm_enable_prefix_cache(bm, 3)
    with pytest.raises(capi.PkvError):
        capi.pkv_bm_enable_prefix_cache(bm, 3)
    assert capi.pkv_seq_admit(bm, 0, list(range(40))) == 0
    with pytest.raises(capi.PkvError):      # more tokens than the sequence holds
        capi.pkv_seq_commit_prefix(bm, 0, list(range(40)))
    capi.pkv_bm_destroy(bm)


def test_pages_agent_history_example():
    """6000-token request, 5500 tokens seen last round ("KV Cache优化实战" §5.1): 5488 reused."""
    rng = np.random.default_rng(5)
    prompt = rng.integers(0, 100000, 6000).tolist()
    bm = capi.pkv_bm_create(512, 16)
    capi.pkv_bm_enable_prefix_cache(bm, 1)
    assert capi.pkv_seq_admit(bm, 0, prompt[:5500]) == 0
    capi.pkv_seq_append_slots(bm, [0] * 5500)
    assert capi.pkv_seq_commit_prefix(bm, 0, prompt[:5500]) == 343
    capi.pkv_seq_free(bm, 0)
    assert capi.pkv_seq_admit(bm, 1, prompt) == 5488
    st = capi.pkv_prefix_cache_stats(bm)
    assert st["hits"] == 343 and st["lookups"] == 1 + 344 and st["evictable"] == 0  # each admit stops at its first miss
    capi.pkv_bm_destroy(bm)
