"""Seeded synthetic workloads for paged decode attention.

This module only draws random inputs and lays out operation scripts; it
holds none of the method's arithmetic (no allocation, no quantisation, no
attention), so the CUDA path and the CPU oracle can both consume it.

Recipe (every value is reproducible from the workload's seed):

* RNG: ``numpy.random.Generator(PCG64(SeedSequence([seed, ...])))``;
  seed = 1630 + workload id.
* Token K/V rows are drawn per 64-token chunk of one sequence stream
  ``SeedSequence([seed, 1, kind, owner, chunk])`` so any row range can be
  regenerated on its own (kind 0 = K, 1 = V; ``owner`` is the sequence, or
  the shared-prefix stream).  Values: N(0, 1) in fp32, optionally times 20
  on a Bernoulli(p) mask (outliers), then rounded to nearest-even in the
  token dtype (fp16 or bf16).  Every layer reads the same K/V streams; the
  per-layer caches are still separate buffers.
* Queries: ``SeedSequence([seed, 2, layer, step])``, N(0, 1) rounded to the
  query dtype.
* Lengths: uniform integers (inclusive) from ``SeedSequence([seed, 0])``.
* Pools: the blocks the workload needs plus 10% free, ids handed out in a
  shuffled order (except where a workload fixes the order).

Lengths are post-append: a sequence of length L is pre-filled with L - 1
tokens, then the decode step appends one token and attends over all L.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np

BLOCK_SIZE = 16
CHUNK = 64
SEED_BASE = 1630
PREFIX_OWNER = -1


def _rng(*keys) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(k) & 0xFFFFFFFF for k in keys])))


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to fp16 / bf16 (nearest-even); returns float32 holding exact values."""
    x = np.asarray(x, dtype=np.float32)
    if dtype == "f16":
        return x.astype(np.float16).astype(np.float32)
    if dtype == "bf16":
        u = x.view(np.uint32)
        r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) & np.uint32(0xFFFF0000)
        return r.view(np.float32)
    raise ValueError(f"no rounding for {dtype}")


# cache types stored as one-byte codes plus an fp32 scale per (token, KV head)
ONE_BYTE_CACHES = ("fp8_e4m3", "fp8_e5m2", "int8")
# ... and every cache type with scales: K FP8 E4M3 codes + V 4-bit codes as well
SCALED_CACHES = ONE_BYTE_CACHES + ("fp8_e4m3_int4",)


def token_head_bytes(cache_dtype: str, head_dim: int) -> int:
    """K plus V bytes one token holds for one KV head, scales included."""
    if cache_dtype in ONE_BYTE_CACHES:
        return 2 * (head_dim + 4)
    if cache_dtype == "fp8_e4m3_int4":
        return head_dim + head_dim // 2 + 8
    return 4 * head_dim


@dataclass
class Workload:
    name: str
    wid: int
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    q_dtype: str              # 'f16' | 'bf16'  (also the dtype of appended K/V rows)
    cache_dtype: str          # 'f16' | 'bf16' | 'fp8_e4m3' | 'fp8_e5m2' | 'int8' | 'fp8_e4m3_int4'
    num_layers: int
    context_lens: np.ndarray  # int64 [B], post-append
    num_blocks: int
    alloc_order: np.ndarray   # int32 [num_blocks]
    scale: float              # fp32 value of 1/sqrt(head_dim)
    prefix_len: int = 0       # shared prefix (sequence 0's first tokens, forked to all)
    outlier_p: float = 0.0
    outlier_mult: float = 20.0
    seed: int = 0
    description: str = ""
    extra: dict = field(default_factory=dict)
    block_size: int = BLOCK_SIZE  # tokens per physical block: 16 or 32

    @property
    def seq_ids(self):
        return list(range(self.num_seqs))

    @property
    def group(self):
        return self.num_q_heads // self.num_kv_heads

    @property
    def max_context_len(self):
        return int(self.context_lens.max()) if len(self.context_lens) else 0

    # -- operation script ---------------------------------------------
    def prefill_ops(self):
        """Operations that build the cache before the decode step.

        ``("create", s)``, ``("fork", parent, child)``, ``("append", seq_ids)``.
        Every appended token of sequence s at position p carries the rows
        ``kv_rows(kind, s, p, p + 1)``.
        """
        ops = []
        lens = [int(x) for x in self.context_lens]
        if self.prefix_len:
            ops.append(("create", 0))
            ops.append(("append", [0] * self.prefix_len))
            for s in range(1, self.num_seqs):
                ops.append(("fork", 0, s))
            for s in range(self.num_seqs):
                n = lens[s] - 1 - self.prefix_len
                if n > 0:
                    ops.append(("append", [s] * n))
        else:
            for s in range(self.num_seqs):
                ops.append(("create", s))
            for s in range(self.num_seqs):
                if lens[s] > 1:
                    ops.append(("append", [s] * (lens[s] - 1)))
        return ops

    def owner(self, seq: int, pos: int) -> int:
        return PREFIX_OWNER if pos < self.prefix_len else seq

    # -- values ---------------------------------------------------------
    def _chunk(self, kind: int, owner: int, chunk: int) -> np.ndarray:
        g = _rng(self.seed, 1, kind, owner, chunk)
        x = g.standard_normal((CHUNK, self.num_kv_heads, self.head_dim), dtype=np.float32)
        if self.outlier_p > 0:
            mask = g.random((CHUNK, self.num_kv_heads, self.head_dim)) < self.outlier_p
            x = np.where(mask, x * np.float32(self.outlier_mult), x)
        return round_to(x, self.q_dtype)

    def kv_rows(self, kind: int, seq: int, start: int, stop: int) -> np.ndarray:
        """float32 [stop - start, Hkv, D] rows of K (kind 0) or V (kind 1) for positions start..stop-1."""
        out = np.empty((max(stop - start, 0), self.num_kv_heads, self.head_dim), dtype=np.float32)
        pos = start
        while pos < stop:
            owner = self.owner(seq, pos)
            end = stop if owner == seq else min(stop, self.prefix_len)
            c0 = pos // CHUNK
            c_last = (end - 1) // CHUNK
            for c in range(c0, c_last + 1):
                lo = max(pos, c * CHUNK)
                hi = min(end, (c + 1) * CHUNK)
                out[lo - start:hi - start] = self._chunk(kind, owner, c)[lo - c * CHUNK:hi - c * CHUNK]
            pos = end
        return out

    def step_rows(self, kind: int, step: int = 0) -> np.ndarray:
        """Rows appended by decode step ``step`` (one per sequence): [B, Hkv, D]."""
        return np.stack([self.kv_rows(kind, s, int(L) - 1 + step, int(L) + step)[0]
                         for s, L in enumerate(self.context_lens)])

    def q_rows(self, layer: int = 0, step: int = 0) -> np.ndarray:
        g = _rng(self.seed, 2, layer, step)
        x = g.standard_normal((self.num_seqs, self.num_q_heads, self.head_dim), dtype=np.float32)
        return round_to(x, self.q_dtype)

    def kv_bytes(self, step: int = 0) -> int:
        """Bytes of K and V (codes + fp32 scales for coded caches) the decode step reads per layer."""
        tokens = int(self.context_lens.sum()) + step * self.num_seqs
        return tokens * self.num_kv_heads * token_head_bytes(self.cache_dtype, self.head_dim)


def _pool(need_blocks: int, slack=0.10) -> int:
    return int(math.ceil((1.0 + slack) * need_blocks))


def _blocks(lengths) -> int:
    return int(sum(-(-int(L) // BLOCK_SIZE) for L in lengths))


def make(wid: int, *, extra_steps: int = 0, num_seqs: int | None = None,
         cache_dtype: str | None = None, block_size: int = BLOCK_SIZE) -> Workload:
    """Workload 1..5.  ``extra_steps`` reserves pool room for that many more decode steps.

    ``cache_dtype`` swaps the cache for a one-byte type (same shapes, seeds
    and values; the rows are quantised on append).  ``block_size`` 32 sizes
    the pool in 32-token blocks (same lengths and values).
    """
    w = _make(wid, extra_steps=extra_steps, num_seqs=num_seqs)
    if block_size != BLOCK_SIZE:
        w = _resize_blocks(w, block_size, extra_steps)
    if cache_dtype is None or cache_dtype == w.cache_dtype:
        return w
    if cache_dtype not in SCALED_CACHES:
        raise ValueError(f"a workload's cache can only be swapped for a coded type, not {cache_dtype}")
    if w.cache_dtype in SCALED_CACHES:
        name = w.name.rsplit("-", 1)[0]
        desc = w.description.replace(w.cache_dtype.replace("_", " "), cache_dtype.replace("_", " "))
    else:
        name = w.name
        desc = f"{w.description}; cache swapped to {cache_dtype} + fp32 scales"
    return replace(w, name=f"{name}-{cache_dtype}", cache_dtype=cache_dtype, description=desc)


def _resize_blocks(w: Workload, bs: int, extra_steps: int) -> Workload:
    """The same workload on a pool of `bs`-token blocks (shuffled ids, or the interleave of workload 3)."""
    g = _rng(w.seed, 3)
    if w.prefix_len:
        p = w.prefix_len
        need = -(-p // bs) + int(sum(-(-(p % bs + int(L) - p + extra_steps) // bs) for L in w.context_lens))
    else:
        need = int(sum(-(-(int(L) + extra_steps) // bs) for L in w.context_lens))
    if w.wid == 3:
        per = -(-(int(w.context_lens.max()) + extra_steps) // bs)
        order = np.array([j * w.num_seqs + s for s in range(w.num_seqs) for j in range(per)], dtype=np.int32)
        nb = w.num_seqs * per
    else:
        nb = _pool(need)
        order = g.permutation(nb).astype(np.int32)
    return replace(w, block_size=bs, num_blocks=nb, alloc_order=order,
                   name=f"{w.name}-bs{bs}", description=f"{w.description}; {bs}-token blocks")


def _make(wid: int, *, extra_steps: int = 0, num_seqs: int | None = None) -> Workload:
    seed = SEED_BASE + wid
    rlen = _rng(seed, 0)
    scale = lambda d: float(np.float32(1.0) / np.sqrt(np.float32(d)))
    if wid == 1:
        lens = np.array([1, 17, 33, 100], dtype=np.int64)
        order = rlen.permutation(32).astype(np.int32)
        nb = 32
        if extra_steps:  # room for more steps: further blocks after the 32, in order
            nb = max(32, _blocks(lens + extra_steps))
            order = np.concatenate([order, np.arange(32, nb, dtype=np.int32)])
        return Workload("tiny-gqa-fp16", 1, 4, 8, 2, 64, "f16", "f16", 1, lens, nb, order,
                        scale(64), seed=seed,
                        description="4 seqs L={1,17,33,100}, Hq8/Hkv2/d64 fp16, 32-block pool")
    if wid == 2:
        b = num_seqs or 16
        lens = rlen.integers(512, 4096, size=b, endpoint=True).astype(np.int64)
        nb = _pool(_blocks(lens + extra_steps))
        order = rlen.permutation(nb).astype(np.int32)
        return Workload("llama3-8b-bf16", 2, b, 32, 8, 128, "bf16", "bf16", 1, lens, nb, order,
                        scale(128), seed=seed,
                        description=f"B{b} L~U[512,4096], Hq32/Hkv8/d128 bf16, pool +10% shuffled")
    if wid == 3:
        b = num_seqs or 8
        lens = np.full(b, 2048, dtype=np.int64)
        per = -(-(2048 + extra_steps) // BLOCK_SIZE)
        order = np.array([j * b + s for s in range(b) for j in range(per)], dtype=np.int32)
        return Workload("mha-7b-40layer-fp16", 3, b, 32, 32, 128, "f16", "f16", 40, lens,
                        b * per, order, scale(128), seed=seed,
                        description=f"40 layers, B{b} L=2048, MHA 32/32/d128 fp16, interleaved blocks")
    if wid == 4:
        b = num_seqs or 32
        prefix = 1500
        suffix = rlen.integers(64, 512, size=b, endpoint=True).astype(np.int64)
        lens = prefix + suffix
        need = -(-prefix // BLOCK_SIZE) + int(sum(-(-(prefix % BLOCK_SIZE + int(s) + extra_steps) // BLOCK_SIZE)
                                                for s in suffix))
        nb = _pool(need)
        order = rlen.permutation(nb).astype(np.int32)
        return Workload("prefix-share-bf16", 4, b, 32, 8, 128, "bf16", "bf16", 1, lens, nb, order,
                        scale(128), prefix_len=prefix, seed=seed,
                        description=f"{b} seqs share a 1500-token prefix, suffix U[64,512], 32/8/d128 bf16")
    if wid == 5:
        b = num_seqs or 16
        lens = rlen.integers(16384, 32768, size=b, endpoint=True).astype(np.int64)
        nb = _pool(_blocks(lens + extra_steps))
        order = rlen.permutation(nb).astype(np.int32)
        return Workload("long-fp8-e4m3", 5, b, 32, 8, 128, "bf16", "fp8_e4m3", 1, lens, nb, order,
                        scale(128), outlier_p=0.001, outlier_mult=20.0, seed=seed,
                        description=f"B{b} L~U[16384,32768], 32/8/d128, fp8 e4m3 KV + fp32 scales, "
                                    "bf16 q, 0.1% outliers x20")
    raise ValueError(f"no workload {wid}")


def custom(name, *, lens, num_q_heads, num_kv_heads, head_dim, q_dtype, cache_dtype,
           num_blocks=None, seed=7, prefix_len=0, outlier_p=0.0, num_layers=1,
           shuffle=True, slack=0.10, block_size=BLOCK_SIZE) -> Workload:
    """A small ad-hoc workload (edge cases in tests)."""
    lens = np.asarray(lens, dtype=np.int64)
    g = _rng(seed, 0)
    bs = block_size
    if num_blocks is None:
        need = int(sum(-(-int(L) // bs) for L in lens)) if not prefix_len else (
            -(-prefix_len // bs) + int(sum(-(-(prefix_len % bs + int(L) - prefix_len) // bs) for L in lens)))
        num_blocks = max(1, _pool(need, slack))
    order = (g.permutation(num_blocks) if shuffle else np.arange(num_blocks)).astype(np.int32)
    return Workload(name, 0, len(lens), num_q_heads, num_kv_heads, head_dim, q_dtype, cache_dtype,
                    num_layers, lens, num_blocks, order,
                    float(np.float32(1.0) / np.sqrt(np.float32(head_dim))),
                    prefix_len=prefix_len, outlier_p=outlier_p, seed=seed, block_size=block_size)
