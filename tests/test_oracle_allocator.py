"""Pins for the oracle's block manager: on-demand blocks, tables, CoW, freeing.

Checked against what "KV Cache 与 vLLM" (zwxr.cn) §3.1-§3.4 and
"KV Cache优化实战" §4.2 state (new block only when the last one is full;
prefix blocks shared; copy on write where a shared block changes; finished
requests' blocks reused) and against conservation invariants that any
correct allocator keeps.
"""
import numpy as np
import pytest

from oracle.allocator import AllocatorModel, InvalidRequest, NoBlocks


def check_invariants(a: AllocatorModel):
    held = [b for t in a.tables.values() for b in t]
    assert sum(a.refcount) == len(held)
    for b in range(a.num_blocks):
        assert a.refcount[b] == held.count(b)
    assert len(set(a.free)) == len(a.free)
    assert set(a.free).isdisjoint(held)
    assert len(a.free) + len(set(held)) == a.num_blocks
    for s, t in a.tables.items():
        assert len(t) == -(-a.lens[s] // a.block_size)     # ceil(len / 16) blocks, no more


def test_on_demand_blocks_and_slots():
    a = AllocatorModel(8, 16, alloc_order=[5, 2, 7, 0, 1, 3, 4, 6])
    a.create(0)
    slots, cows = a.append_slots([0] * 17)
    assert cows == []
    assert a.tables[0] == [5, 2]
    assert slots == [5 * 16 + i for i in range(16)] + [2 * 16]
    assert a.num_free() == 6
    check_invariants(a)


def test_fifo_reuse_after_free():
    a = AllocatorModel(4, 16)
    a.create(0); a.create(1)
    a.append_slots([0] * 20)            # blocks 0, 1
    a.append_slots([1])                 # block 2
    a.free_seq(0)                       # 0 then 1 join the tail: free = [3, 0, 1]
    assert list(a.free) == [3, 0, 1]
    a.create(2)
    a.append_slots([2] * 33)
    assert a.tables[2] == [3, 0, 1]
    check_invariants(a)


def test_fork_shares_and_cow_copies_partial_block():
    a = AllocatorModel(64, 16)
    a.create(0)
    a.append_slots([0] * 40)            # blocks 0,1 full; 2 holds 8 tokens
    for c in (1, 2, 3):
        a.fork(0, c)
    assert a.refcount[:3] == [4, 4, 4]
    slots, cows = a.append_slots([0, 1, 2, 3])
    # the first three sharers copy block 2; the last holder writes in place
    assert cows == [(2, 3), (2, 4), (2, 5)]
    assert [s // 16 for s in slots] == [3, 4, 5, 2]
    assert [s % 16 for s in slots] == [8, 8, 8, 8]
    assert a.tables[3] == [0, 1, 2] and a.tables[0] == [0, 1, 3]
    assert a.refcount[0] == 4 and a.refcount[2] == 1
    check_invariants(a)


def test_fork_at_block_boundary_needs_no_copy():
    a = AllocatorModel(16, 16)
    a.create(0)
    a.append_slots([0] * 32)
    a.fork(0, 1)
    slots, cows = a.append_slots([1, 0])
    assert cows == [] and [s // 16 for s in slots] == [2, 3]
    check_invariants(a)


def test_no_blocks_is_all_or_nothing():
    a = AllocatorModel(3, 16)
    a.create(0); a.create(1)
    a.append_slots([0] * 16)
    before = (list(a.free), list(a.refcount), {k: list(v) for k, v in a.tables.items()}, dict(a.lens))
    with pytest.raises(NoBlocks):
        a.append_slots([1] * 16 + [0] * 17 + [1] * 16)     # needs 3 blocks, 2 free
    assert (list(a.free), list(a.refcount), a.tables, a.lens) == before
    a.append_slots([1] * 16 + [0])                          # exactly 2
    assert a.num_free() == 0
    check_invariants(a)


def test_invalid_requests():
    a = AllocatorModel(4)
    with pytest.raises(InvalidRequest):
        a.append_slots([9])
    a.create(0)
    with pytest.raises(InvalidRequest):
        a.create(0)
    with pytest.raises(InvalidRequest):
        a.fork(5, 6)
    with pytest.raises(InvalidRequest):
        a.free_block(2)
    with pytest.raises(InvalidRequest):
        AllocatorModel(4, alloc_order=[0, 1, 1, 2])


def test_random_traces_keep_invariants_and_drain():
    rng = np.random.default_rng(7)
    for trial in range(20):
        n = int(rng.integers(8, 64))
        a = AllocatorModel(n, 16, alloc_order=rng.permutation(n))
        live, next_id = [], 0
        for _ in range(200):
            op = rng.integers(0, 10)
            if op == 0 or not live:
                a.create(next_id); live.append(next_id); next_id += 1
            elif op == 1:
                p = live[int(rng.integers(len(live)))]
                a.fork(p, next_id); live.append(next_id); next_id += 1
            elif op == 2 and len(live) > 1:
                s = live.pop(int(rng.integers(len(live))))
                a.free_seq(s)
            else:
                batch = [live[int(i)] for i in rng.integers(0, len(live), int(rng.integers(1, 6)))]
                try:
                    a.append_slots(batch)
                except NoBlocks:
                    pass
            check_invariants(a)
        for s in live:
            a.free_seq(s)
        assert a.num_free() == n and sum(a.refcount) == 0


def test_block_tables_export():
    a = AllocatorModel(8, 16, alloc_order=[3, 1, 4, 0, 5, 2, 6, 7])
    a.create(10); a.create(11)
    a.append_slots([10] * 33 + [11])
    tables, lens = a.block_tables([11, 10], 4)
    assert tables == [[0, -1, -1, -1], [3, 1, 4, -1]] and lens == [1, 33]
    with pytest.raises(InvalidRequest):
        a.block_tables([10], 2)
