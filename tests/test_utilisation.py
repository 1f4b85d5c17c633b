"""The utilisation simulator: static utilisation against the oracle's sizing
closed forms, the pages' claims for ragged lengths, the block-size trade-off,
and closed-form cases of the continuous-batching simulation (host only).
"""
import os

import numpy as np
import pytest

from oracle import sizing
from paged_kv_cache_163_gb300 import build, capi, utilisation as ut


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not os.path.exists(capi.LIB_PATH):
        build.build()
    return capi.load()


def test_static_utilisation_matches_oracle():
    rng = np.random.default_rng(4)
    for _ in range(50):
        lens = rng.integers(1, 5000, int(rng.integers(1, 64))).tolist()
        for bs in (16, 32):
            assert ut.paged_slots(lens, bs) == sizing.paged_token_slots(lens, bs)
            assert ut.paged(lens, bs) == sizing.paged_utilisation(lens, bs)
        assert ut.prealloc(lens, 8192) == sizing.prealloc_utilisation(lens, 8192)


def test_pages_claims_for_ragged_lengths():
    """Above 90% paged against well under 60% reserved ("KV Cache 与 vLLM" §3.1; "KV Cache优化实战" §4.2)."""
    rng = np.random.default_rng(5)
    for lo, hi in ((512, 4096), (64, 4096), (16, 2048)):
        lens = rng.integers(lo, hi + 1, 256).tolist()
        assert ut.paged(lens, 16) > 0.9
        assert ut.prealloc(lens, hi) < 0.6


def test_block_size_trade_off():
    """Larger blocks: more tail waste, half the table entries ("KV Cache优化实战" §7.5)."""
    rng = np.random.default_rng(6)
    lens = rng.integers(1, 300, 500).tolist()
    assert ut.paged(lens, 32) < ut.paged(lens, 16)
    assert ut.table_entries(lens, 32) <= (ut.table_entries(lens, 16) + len(lens)) // 2
    short = [3] * 100                                    # short requests favour small blocks
    assert ut.paged(short, 16) == 3 / 16 and ut.paged(short, 32) == 3 / 32


def test_simulation_closed_forms():
    reqs = [(100, 28)] * 12
    # room for everything: every request runs from the first step, each step adds one token
    r = ut.simulate(reqs, 12 * 128 + 64, block_size=16)
    assert (r.steps, r.peak_batch, r.preemptions) == (28, 12, 0)
    # preallocation of 512 tokens a request in 2048 tokens: 4 at a time, three waves of 28 steps
    r = ut.simulate(reqs, 2048, block_size=None, max_len=512)
    assert (r.steps, r.peak_batch) == (84, 4)
    assert r.mean_utilisation == pytest.approx(np.mean([(100 + k) / 512 for k in range(1, 29)]))


def test_paged_serves_more_requests_at_once():
    rng = np.random.default_rng(7)
    reqs = [(int(p), int(o)) for p, o in zip(rng.integers(50, 1500, 64), rng.integers(10, 300, 64))]
    budget = 16 * 2048
    paged = ut.simulate(reqs, budget, block_size=16)
    paged32 = ut.simulate(reqs, budget, block_size=32)
    pre = ut.simulate(reqs, budget, block_size=None, max_len=2048)
    assert paged.peak_batch > 2 * pre.peak_batch
    assert paged.steps < pre.steps
    assert paged.mean_utilisation > 0.9 > pre.mean_utilisation
    assert paged32.mean_utilisation <= paged.mean_utilisation + 1e-12
