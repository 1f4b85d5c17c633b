"""Block-manager model: paged KV blocks, block tables, prefix sharing, copy-on-write.

What the pages fix ("KV Cache 与 vLLM" (zwxr.cn) §3.1-§3.4,
"KV Cache优化实战" §4.2):

* the cache is cut into fixed physical blocks of 16 tokens by default;
* blocks are taken on demand: when a sequence's last block is full, a new
  physical block is taken and added to the end of its block table;
* the block table maps the sequence's logical blocks (tokens 0-15 are
  logical block 0, 16-31 logical block 1, ...) to physical blocks;
* sequences with the same prefix point at the same physical blocks; where a
  shared block has to be modified it is copied on write;
* a finished request's blocks are freed at once and reused.

Readings of what the pages leave open (each one fixed so that tables, slot
mappings and copy pairs are unique and can be compared bit for bit):

* free list: FIFO, initialised to ``alloc_order`` (default 0..n-1); a block
  is taken from the head and returned to the tail;
* a block is shared when its reference count exceeds 1; fork copies the
  parent's table and adds one reference to each block;
* copy-on-write happens when a sequence appends into a partially filled
  last block that is still shared: it takes a new block, records the pair
  (old -> new) and drops its reference to the old block; the last holder,
  left with a count of 1, writes in place;
* a batch of appends is applied in the order given (a sequence may appear
  several times) and is all-or-nothing: if the free list cannot cover every
  block the batch needs, nothing changes and ``NoBlocks`` is raised (the
  pages ask that running out of memory must not crash a request:
  "企业官网建设流程全解析" §6.4);
* freeing a sequence drops its references in logical order; blocks whose
  count reaches 0 join the tail of the free list in that order.
"""
from __future__ import annotations

import copy
from collections import deque


class NoBlocks(Exception):
    """The free list cannot cover a request; nothing was changed."""


class InvalidRequest(Exception):
    """An argument is out of range or names an unknown sequence or block."""


class AllocatorModel:
    def __init__(self, num_blocks: int, block_size: int = 16, alloc_order=None):
        if num_blocks <= 0 or block_size <= 0:
            raise InvalidRequest("pool must hold at least one block")
        order = list(range(num_blocks)) if alloc_order is None else [int(b) for b in alloc_order]
        if sorted(order) != list(range(num_blocks)):
            raise InvalidRequest("alloc_order must be a permutation of 0..num_blocks-1")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free = deque(order)
        self.refcount = [0] * num_blocks
        self.tables: dict[int, list[int]] = {}
        self.lens: dict[int, int] = {}

    # -- single blocks -------------------------------------------------
    def alloc_block(self) -> int:
        if not self.free:
            raise NoBlocks("free list is empty")
        b = self.free.popleft()
        self.refcount[b] = 1
        return b

    def free_block(self, b: int) -> None:
        if not (0 <= b < self.num_blocks) or self.refcount[b] <= 0:
            raise InvalidRequest(f"block {b} is not held")
        self.refcount[b] -= 1
        if self.refcount[b] == 0:
            self.free.append(b)

    # -- sequences -----------------------------------------------------
    def create(self, seq: int) -> None:
        if seq in self.tables:
            raise InvalidRequest(f"sequence {seq} exists")
        self.tables[seq] = []
        self.lens[seq] = 0

    def fork(self, parent: int, child: int) -> None:
        if parent not in self.tables or child in self.tables:
            raise InvalidRequest("fork needs an existing parent and a new child")
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        for b in self.tables[child]:
            self.refcount[b] += 1

    def free_seq(self, seq: int) -> None:
        if seq not in self.tables:
            raise InvalidRequest(f"unknown sequence {seq}")
        for b in self.tables.pop(seq):
            self.free_block(b)
        del self.lens[seq]

    def _append_one(self, seq: int):
        """Apply one append; return (slot, cow pair or None)."""
        table = self.tables[seq]
        n = self.lens[seq]
        bs = self.block_size
        cow = None
        if n % bs == 0:
            table.append(self.alloc_block())
        else:
            last = table[-1]
            if self.refcount[last] > 1:
                new = self.alloc_block()
                self.refcount[last] -= 1
                table[-1] = new
                cow = (last, new)
        slot = table[n // bs] * bs + n % bs
        self.lens[seq] = n + 1
        return slot, cow

    def append_slots(self, seq_ids):
        """Append one token to each listed sequence, in order.

        Returns (slot_mapping, cow_pairs) where slot = block * block_size +
        offset and cow_pairs lists (src, dst) blocks in the order they arose.
        All-or-nothing: on NoBlocks the state is exactly as before.
        """
        for s in seq_ids:
            if s not in self.tables:
                raise InvalidRequest(f"unknown sequence {s}")
        saved = (copy.copy(self.free), list(self.refcount),
                 {k: list(v) for k, v in self.tables.items()}, dict(self.lens))
        slots, cows = [], []
        try:
            for s in seq_ids:
                slot, cow = self._append_one(s)
                slots.append(slot)
                if cow is not None:
                    cows.append(cow)
        except NoBlocks:
            self.free, self.refcount, self.tables, self.lens = saved
            raise
        return slots, cows

    # -- export ----------------------------------------------------------
    def block_tables(self, seq_ids, max_blocks: int):
        """(tables [n][max_blocks] padded with -1, context_lens [n])."""
        rows, lens = [], []
        for s in seq_ids:
            if s not in self.tables:
                raise InvalidRequest(f"unknown sequence {s}")
            t = self.tables[s]
            if len(t) > max_blocks:
                raise InvalidRequest("table longer than max_blocks")
            rows.append(t + [-1] * (max_blocks - len(t)))
            lens.append(self.lens[s])
        return rows, lens

    def num_free(self) -> int:
        return len(self.free)
