"""KV-memory utilisation of paged allocation against max-length preallocation.

The pages' headline claims about PagedAttention are about memory, not
speed: blocks taken on demand keep KV-cache utilisation above 90% where
reserving each request's maximum length wastes 50-70% ("KV Cache 与 vLLM"
§3.1: above 90% against 30-50%; "KV Cache优化实战" §4.2: from under 60% to
close to 100%, and many more concurrent requests on the same GPU).  The
block size is the tuning knob: smaller blocks waste less of each
sequence's last block, larger ones need fewer table entries
("KV Cache优化实战" §7.5).

Two tools:

* static utilisation of a set of sequence lengths (``paged`` for a block
  size, ``prealloc`` for a reserved maximum length);
* ``simulate``: continuous batching of a request trace in a fixed KV
  budget.  The paged side runs the library's native block manager
  (blocks on demand, all-or-nothing appends; when a step's appends do not
  fit, the most recently admitted request is preempted and requeued, its
  blocks freed).  The preallocation side reserves ``max_len`` tokens per
  admitted request.  Both admit in arrival order while they can, and report
  steps to drain the trace, mean and peak running batch and mean
  utilisation (tokens held / token slots held).
"""
from __future__ import annotations

from collections import deque
from dataclasses import dataclass

from . import capi


def paged_slots(lengths, block_size: int = capi.BLOCK_SIZE) -> int:
    """Token slots a paged cache holds for these lengths: sum of ceil(L / bs) * bs."""
    return sum(-(-int(n) // block_size) * block_size for n in lengths)


def paged(lengths, block_size: int = capi.BLOCK_SIZE) -> float:
    """Share of the paged cache's slots that hold a token."""
    held = paged_slots(lengths, block_size)
    return sum(int(n) for n in lengths) / held if held else 1.0


def prealloc(lengths, max_len: int) -> float:
    """Share of max-length reservations that hold a token."""
    lengths = [int(n) for n in lengths]
    return sum(lengths) / (len(lengths) * max_len) if lengths else 1.0


def table_entries(lengths, block_size: int = capi.BLOCK_SIZE) -> int:
    """Block-table entries the lengths need (the per-step metadata a decode reads)."""
    return sum(-(-int(n) // block_size) for n in lengths)


@dataclass
class SimResult:
    steps: int              # decode steps until every request finished
    mean_batch: float       # running requests per step
    peak_batch: int
    mean_utilisation: float  # tokens held / token slots held, averaged over steps
    preemptions: int = 0


def simulate(requests, budget_tokens: int, *, block_size: int | None = capi.BLOCK_SIZE,
             max_len: int | None = None) -> SimResult:
    """Continuous batching of `requests` = [(prompt_len, output_len), ...] in `budget_tokens` of KV.

    ``block_size`` set: paged allocation on the native block manager with
    budget_tokens // block_size blocks.  ``block_size`` None: reserve
    ``max_len`` tokens per admitted request.  Each step every running
    request holds its prompt plus the tokens generated so far and adds one.
    """
    reqs = [(int(p), int(o)) for p, o in requests]
    if block_size is None:
        return _simulate_prealloc(reqs, budget_tokens, max_len)
    return _simulate_paged(reqs, budget_tokens, block_size)


def _simulate_prealloc(reqs, budget_tokens, max_len):
    if max_len is None:
        raise ValueError("preallocation needs max_len")
    if any(p + o > max_len for p, o in reqs):
        raise ValueError("a request is longer than max_len")
    slots = budget_tokens // max_len
    waiting = deque(range(len(reqs)))
    running = {}     # request -> tokens held
    steps = batch_sum = peak = 0
    util_sum = 0.0
    while waiting or running:
        while waiting and len(running) < slots:
            r = waiting.popleft()
            running[r] = reqs[r][0]
        if not running:
            raise ValueError("budget cannot hold one request")
        for r in list(running):
            running[r] += 1
        steps += 1
        batch_sum += len(running)
        peak = max(peak, len(running))
        util_sum += sum(running.values()) / (len(running) * max_len)
        for r in list(running):
            if running[r] >= sum(reqs[r]):
                del running[r]
    return SimResult(steps, batch_sum / steps, peak, util_sum / steps)


def _simulate_paged(reqs, budget_tokens, bs):
    nblocks = budget_tokens // bs
    bm = capi.pkv_bm_create(nblocks, bs)
    try:
        waiting = deque(range(len(reqs)))
        running = []     # admission order
        steps = batch_sum = peak = preempt = 0
        util_sum = 0.0
        while waiting or running:
            # admit in order while the prompt (and this step's token) fits
            while waiting:
                r = waiting[0]
                need = -(-(reqs[r][0] + 1) // bs)
                if need > capi.pkv_bm_num_free(bm):
                    break
                waiting.popleft()
                capi.pkv_seq_create(bm, r)
                if reqs[r][0]:
                    capi.pkv_seq_append_slots(bm, [r] * reqs[r][0])
                running.append(r)
            if not running:
                raise ValueError("budget cannot hold one request")
            # this step's tokens, all or nothing; preempt the newest request until they fit
            while True:
                try:
                    capi.pkv_seq_append_slots(bm, running)
                    break
                except capi.NoBlocksError:
                    victim = running.pop()
                    capi.pkv_seq_free(bm, victim)
                    waiting.appendleft(victim)
                    preempt += 1
                    if not running:
                        raise ValueError("budget cannot hold one request") from None
            steps += 1
            batch_sum += len(running)
            peak = max(peak, len(running))
            lens = [capi.pkv_seq_len(bm, r) for r in running]
            util_sum += sum(lens) / paged_slots(lens, bs)
            for r in list(running):
                if capi.pkv_seq_len(bm, r) >= sum(reqs[r]):
                    capi.pkv_seq_free(bm, r)
                    running.remove(r)
        return SimResult(steps, batch_sum / steps, peak, util_sum / steps, preempt)
    finally:
        capi.pkv_bm_destroy(bm)
