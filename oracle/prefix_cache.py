"""Automatic prefix caching on top of the block-manager model.

What the pages fix:

* cached KV blocks are identified by a hash of their content; a new request
  compares its prefix block by block against the cache and reuses the
  blocks that hit instead of recomputing them ("KV Cache优化实战" §5.2);
* a hit needs the prefix to be identical token for token
  ("KV Cache优化实战" §5.2);
* the key covers the model, the token id sequence and the configuration
  that affects the computation ("企业官网建设流程全解析" §6.2);
* eviction cannot be plain LRU: a block's later tokens depend on the
  earlier ones, so evicting a middle block breaks every block after it;
  production systems evict along a prefix tree or hash chain
  ("企业官网建设流程全解析" §6.3).

Readings of what the pages leave open, each fixed so that tables, hit
counts and eviction order are unique and can be compared bit for bit:

* only full blocks (16 tokens) are cached;
* the key of logical block j of a prompt is the hash chain
  h_j = FNV-1a-64(h_{j-1} as 8 little-endian bytes, the block's 16 token
  ids as 4-byte little-endian two's complement each, the config key as 8
  little-endian bytes), with h_{-1} = 0.  FNV-1a-64 is the published
  Fowler-Noll-Vo hash (offset basis 0xcbf29ce484222325, prime
  0x100000001b3); the stored token ids are compared on a hit as well, so a
  hash collision cannot hand out a wrong block;
* admitting a request walks its prompt's full blocks from the start and
  stops at the first miss; at most (n - 1) // 16 blocks are reused for an n
  token prompt, so at least one prompt token is always computed;
* a sequence's blocks are registered by an explicit commit once their K/V
  are written (the block manager never sees token ids otherwise), in chain
  order; at the first block whose hash is already registered to another
  block the sequence's chain stops, and that block and the ones after it
  stay private.  So whoever holds a registered block also holds its parent,
  and an unreferenced registered block has only unreferenced descendants:
  there is always a leaf to evict;
* a registered block whose reference count drops to 0 stays cached and
  counts as free capacity; plain free blocks (never registered) are taken
  first, in FIFO order;
* when no plain free block is left, the victim is the registered
  unreferenced block with no registered child, least recently used first
  (use = the call that last admitted, committed or released it), then the
  deepest, then the lowest id.  Evicting it unregisters it and may turn its
  parent into a leaf;
* every admit, commit and release is one tick of the use clock.
"""
from __future__ import annotations

import copy

from .allocator import AllocatorModel, InvalidRequest, NoBlocks

FNV_OFFSET = 0xCBF29CE484222325
FNV_PRIME = 0x100000001B3
MASK64 = (1 << 64) - 1


def fnv1a64(data: bytes) -> int:
    h = FNV_OFFSET
    for byte in data:
        h ^= byte
        h = (h * FNV_PRIME) & MASK64
    return h


def block_hash(parent_hash: int, tokens, config_key: int) -> int:
    """Chain hash of one full block of token ids."""
    data = bytearray(int(parent_hash & MASK64).to_bytes(8, "little"))
    for t in tokens:
        data += (int(t) & 0xFFFFFFFF).to_bytes(4, "little")
    data += int(config_key & MASK64).to_bytes(8, "little")
    return fnv1a64(bytes(data))


class PrefixCachingAllocator(AllocatorModel):
    def __init__(self, num_blocks: int, block_size: int = 16, alloc_order=None, config_key: int = 0):
        super().__init__(num_blocks, block_size, alloc_order)
        self.config_key = int(config_key) & MASK64
        self.by_hash: dict[int, int] = {}
        # registered block -> (hash, parent block or -1, depth, token ids)
        self.reg: dict[int, tuple] = {}
        self.children = [0] * num_blocks
        self.last_use = [0] * num_blocks
        self.tick = 0
        self.lookups = self.hits = self.evictions = 0

    # -- capacity ----------------------------------------------------------
    def _evictable(self):
        return [b for b in self.reg if self.refcount[b] == 0]

    def num_free(self) -> int:
        return len(self.free) + len(self._evictable())

    def _victim(self) -> int:
        leaves = [b for b in self._evictable() if self.children[b] == 0]
        return min(leaves, key=lambda b: (self.last_use[b], -self.reg[b][2], b))

    def _unregister(self, b: int) -> None:
        h, parent, _, _ = self.reg.pop(b)
        del self.by_hash[h]
        if parent >= 0:
            self.children[parent] -= 1
        self.evictions += 1

    def alloc_block(self) -> int:
        if self.free:
            return super().alloc_block()
        if not self._evictable():
            raise NoBlocks("no free or evictable block")
        b = self._victim()
        self._unregister(b)
        self.refcount[b] = 1
        return b

    def free_block(self, b: int) -> None:
        if not (0 <= b < self.num_blocks) or self.refcount[b] <= 0:
            raise InvalidRequest(f"block {b} is not held")
        self.refcount[b] -= 1
        if self.refcount[b] == 0:
            if b in self.reg:
                self.last_use[b] = self.tick
            else:
                self.free.append(b)

    # -- calls ---------------------------------------------------------------
    def free_seq(self, seq: int) -> None:
        if seq not in self.tables:
            raise InvalidRequest(f"unknown sequence {seq}")
        self.tick += 1
        super().free_seq(seq)

    def release_block(self, b: int) -> None:
        """The single-block release call (kv_block_free)."""
        if not (0 <= b < self.num_blocks) or self.refcount[b] <= 0:
            raise InvalidRequest(f"block {b} is not held")
        self.tick += 1
        self.free_block(b)

    def append_slots(self, seq_ids):
        saved = copy.deepcopy(self.__dict__)
        try:
            return super().append_slots(seq_ids)
        except NoBlocks:
            self.__dict__.clear()
            self.__dict__.update(saved)
            raise

    def admit(self, seq: int, tokens) -> int:
        """Create `seq` for a prompt; map its longest cached prefix; return the cached token count."""
        if seq in self.tables:
            raise InvalidRequest(f"sequence {seq} exists")
        tokens = [int(t) for t in tokens]
        self.tick += 1
        self.create(seq)
        bs = self.block_size
        usable = (len(tokens) - 1) // bs if tokens else 0
        h, parent = 0, -1
        table = self.tables[seq]
        for j in range(usable):
            blk_tokens = tuple(tokens[j * bs:(j + 1) * bs])
            h = block_hash(h, blk_tokens, self.config_key)
            self.lookups += 1
            b = self.by_hash.get(h)
            if b is None or self.reg[b][3] != blk_tokens or self.reg[b][1] != parent:
                break
            self.hits += 1
            self.refcount[b] += 1
            self.last_use[b] = self.tick
            table.append(b)
            parent = b
        self.lens[seq] = len(table) * bs
        return self.lens[seq]

    def commit(self, seq: int, tokens) -> int:
        """Register the full blocks among the first len(tokens) tokens of `seq`; return how many."""
        if seq not in self.tables:
            raise InvalidRequest(f"unknown sequence {seq}")
        tokens = [int(t) for t in tokens]
        if len(tokens) > self.lens[seq]:
            raise InvalidRequest("more tokens than the sequence holds")
        self.tick += 1
        bs = self.block_size
        h, parent, added = 0, -1, 0
        for j in range(len(tokens) // bs):
            blk_tokens = tuple(tokens[j * bs:(j + 1) * bs])
            h = block_hash(h, blk_tokens, self.config_key)
            b = self.tables[seq][j]
            holder = self.by_hash.get(h)
            if holder is not None:
                if holder != b:      # a duplicate of another block: the chain stops here
                    break
            elif b in self.reg:      # registered under another chain: the chain stops here
                break
            else:
                self.by_hash[h] = b
                self.reg[b] = (h, parent, j, blk_tokens)
                if parent >= 0:
                    self.children[parent] += 1
                self.last_use[b] = self.tick
                added += 1
            parent = b
        return added

    def stats(self):
        return {"lookups": self.lookups, "hits": self.hits, "evictions": self.evictions,
                "registered": len(self.reg), "evictable": len(self._evictable())}
