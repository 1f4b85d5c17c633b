#!/usr/bin/env python
"""Benchmark: paged decode attention on one GB300 (per GPU; weak scaling under torchrun).

One step = the whole decode hot path for one batch: host block manager
(append slots + block tables into page-locked staging), copy-on-write block
copies (when a shared block is appended to), then for every layer one
decode kernel that appends the step's K/V rows (reshape-and-cache) and
attends through the block tables, merging split-KV partials by log-sum-exp
inside the same launch.  Inputs (new K/V rows and queries for every step)
are resident in HBM before the timed region; between timed steps the L2 is
flushed (a 256 MiB write, then a 256 MiB read of another buffer) so the KV
cache is read from HBM, and only the steps themselves are timed (CUDA
events on the launching stream).

The default workload is long-fp8: 16 sequences of 16K-32K tokens, 32 query
/ 8 KV heads of 128, an FP8 E4M3 cache with fp32 per-(token, head) scales
and bf16 queries.  ``--workload`` selects the others.

Prints one JSON line.  ``--impl reference`` times the CPU fp64 oracle on the
same workload instead (bounded samples per step).
"""
from __future__ import annotations

import argparse
import contextlib
import gc
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
os.environ.setdefault("OMP_NUM_THREADS", "1")
os.environ.setdefault("MKL_NUM_THREADS", "1")

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_163_gb300 import workloads as wl  # noqa: E402

METRIC = "decode attn KV-read GB/s (% of GB300 HBM peak); seq-tokens/s per layer"
WORKLOADS = {"tiny": 1, "llama3-8b": 2, "mha7b-40layer": 3, "prefix-share": 4, "long-fp8": 5}
DEFAULT_WORKLOAD = "long-fp8"
SCRUB_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6800.0

# DRAM traffic per decode call (dram__bytes_read.sum + dram__bytes_write.sum, one
# ncu capture), keyed by workload and by the hash of the decode kernel source it
# was taken on; reported only while the source is unchanged.
NCU_TRAFFIC = {
    # decode kernel source 35280b6bc0d3afb8: tensor-core kernel with the step's append fused in, 16-warp
    # CTAs for one-byte caches, biased INT8 (stored code + 128) / 4-bit MMA operands, K and V scales of a tile in one
    # 128-byte unit, first cache copies before the programmatic wait behind kernels that write no cache,
    # cascade with the mma.sync prefix kernel, approximate softmax exponentials for 4-bit V; default "auto" variants.
    # dram__bytes_read.sum + dram__bytes_write.sum of one call (the fifth decode call of a --steps 4
    # --warmup 3 run; prefix-share: its prefix kernel plus its decode, whose DRAM reads include the
    # prefix partials ncu's replay flushed from L2)
    ("llama3-8b", "35280b6bc0d3afb8"): 145_818_368,
    ("llama3-8b:bs32", "35280b6bc0d3afb8"): 145_939_968,
    ("mha7b-40layer", "35280b6bc0d3afb8"): 271_543_808,
    ("prefix-share", "35280b6bc0d3afb8"): 52_880_128,
    ("long-fp8", "35280b6bc0d3afb8"): 796_624_384,
    ("long-fp8:fp8_e5m2", "35280b6bc0d3afb8"): 796_783_104,
    ("long-fp8:int8", "35280b6bc0d3afb8"): 796_804_864,
    ("long-fp8:fp8_e4m3_int4", "35280b6bc0d3afb8"): 604_555_008,
    ("long-fp8:bs32", "35280b6bc0d3afb8"): 797_113_344,
}


@contextlib.contextmanager
def no_gc():
    """Python's cyclic garbage collector off inside a timed region (as timeit does), so a
    collection pass of the host interpreter does not land in a step's time.  (No collection
    on entry: a full pass right before the first timed step left that step's host work slow.)"""
    was = gc.isenabled()
    gc.disable()
    try:
        yield
    finally:
        if was:
            gc.enable()


def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in ("decode.cuh", "decode_mma.cuh", "decode_prefix.cuh", "decode_prefix_umma.cuh", "common.cuh", "dtypes.h"):
        with open(os.path.join(ROOT, "paged_kv_cache_163_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--cache-dtype", choices=["fp8_e4m3", "fp8_e5m2", "int8", "fp8_e4m3_int4"], default=None,
                    help="swap the workload's cache for this coded type (same shapes and values)")
    ap.add_argument("--block-size", type=int, choices=[16, 32], default=16,
                    help="tokens per physical block (the pool is sized for it)")
    ap.add_argument("--graph", action="store_true",
                    help="replay each step's launches from a CUDA graph (inputs refilled into fixed buffers)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the CPU-baseline sample")
    ap.add_argument("--kernel", choices=["auto", "simt", "mma"], default="auto",
                    help="decode kernel variant (auto: tensor-core tiles for head_dim 128)")
    ap.add_argument("--prefix-kernel", choices=["auto", "mma_sync", "tcgen05"], default="auto",
                    help="cascade prefix kernel (auto: mma.sync; tcgen05 for 16-bit caches when asked)")
    ap.add_argument("--prefix-chunk-tiles", type=int, default=0,
                    help="16-token tiles per tcgen05 prefix CTA (0: the library default)")
    return ap.parse_args(argv)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(values, device=None):
    """Element-wise maximum of per-rank values (identity on one rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_rate(world: int, units_per_rank: float, seconds_max: float) -> float:
    """Units all ranks processed over the slowest rank's time (weak scaling: equal shards)."""
    return world * units_per_rank / seconds_max


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# Workload accounting
# ---------------------------------------------------------------------------
def step_accounting(w: wl.Workload, step: int):
    """Algorithmic bytes of one attention call and the step's KV bytes / tokens."""
    lens = w.context_lens + step
    tokens = int(lens.sum())
    kv = w.kv_bytes(step)                                      # K + V (+ scales) of all sequences
    q_bytes = w.num_seqs * w.num_q_heads * w.head_dim * 2
    table_bytes = int(sum(-(-int(L) // w.block_size) for L in lens)) * 4
    lens_bytes = w.num_seqs * 4
    out_bytes = q_bytes
    # Bytes in HBM: a shared prefix's full blocks are held (and need reading) once;
    # every sequence holds its own copy of the partial block and its suffix.
    shared = (w.prefix_len // w.block_size) * w.block_size
    unique_tokens = shared + int((lens - shared).sum()) if shared else tokens
    kv_unique = kv * unique_tokens // tokens
    return {"tokens": tokens, "kv_bytes": kv, "kv_unique_bytes": kv_unique,
            "algo_bytes": kv_unique + q_bytes + table_bytes + lens_bytes + out_bytes,
            "roofline_bytes": kv_unique + q_bytes + table_bytes + lens_bytes}


def kv_utilisation(w: wl.Workload) -> dict:
    """Token slots held that hold a token, for the workload's lengths (paged blocks vs max-length reservation)."""
    from paged_kv_cache_163_gb300 import utilisation as ut
    lens = [int(x) for x in w.context_lens]
    return {"paged_bs16": round(ut.paged(lens, 16), 4), "paged_bs32": round(ut.paged(lens, 32), 4),
            "prealloc_max_len": round(ut.prealloc(lens, w.max_context_len), 4), "max_len": w.max_context_len}


def decode_kernel_name(w: wl.Workload, kind: str) -> str:
    """The decode kernel a call runs: tensor cores for head_dim 128 unless 'simt' is forced."""
    return "paged_decode_mma_kernel" if w.head_dim == 128 and kind != "simt" else "paged_decode_kernel"


class L2Flush:
    """Cold, clean L2 before a timed step (outside the timed region).

    A write of SCRUB_BYTES (twice the 129 MB L2) evicts everything the last
    step left; a read of a second buffer of that size then evicts the
    write's dirty lines, so the timed step neither finds its data in L2 nor
    pays to write back the flush's own data.
    """

    def __init__(self, dev):
        import torch
        self.w = torch.empty(SCRUB_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(SCRUB_BYTES // 4, dtype=torch.int32, device=dev)

    def __call__(self, i: int) -> None:
        self.w.fill_(i & 0xFF)
        self.r.amax()


def workload_config(w: wl.Workload, name: str, extra=None):
    cfg = {"workload": name, "description": w.description, "num_seqs": w.num_seqs,
           "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
           "layers": w.num_layers, "q_dtype": w.q_dtype, "cache_dtype": w.cache_dtype,
           "context_tokens": int(w.context_lens.sum()), "max_context_len": w.max_context_len,
           "seed": w.seed, "block_size": w.block_size,
           "l2": "flushed between timed steps: 256 MiB write, then 256 MiB read of another buffer"}
    if extra:
        cfg.update(extra)
    return cfg


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def mark(self, which):
        setattr(self, which, time.time())

    @staticmethod
    def _summary(inside, window):
        sm = [float(s[1]) for s in inside if s[1].replace(".", "").isdigit()]
        mx = [float(s[2]) for s in inside if s[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for s in inside for n, v in zip(names, s[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside), "window": window,
                "power_w_max": max((float(s[3]) for s in inside if s[3].replace(".", "").isdigit()), default=None)}

    def stop(self):
        """Clock summary of the timed region [t0, t1]; with a sustained pass [s0, s1], its summary too."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.count(",") >= 9]
        os.unlink(self.file.name)
        import datetime as dt
        samples = []
        for r in rows:
            try:
                ts = dt.datetime.strptime(r[0].strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            samples.append((ts, [x.strip() for x in r[1:]]))
        inside = [s for ts, s in samples if self.t0 is not None and self.t0 - 0.06 <= ts <= self.t1 + 0.06]
        window = "timed"
        if not inside:
            inside = [s for _, s in samples]
            window = "whole run (timed region shorter than the sampling interval)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        out = self._summary(inside, window)
        s0, s1 = getattr(self, "s0", None), getattr(self, "s1", None)
        if s0 is not None and s1 is not None:
            sus = [s for ts, s in samples if s0 <= ts <= s1]
            if sus:
                out["sustained"] = self._summary(sus, "back-to-back attention calls after the timed steps")
                out["sustained"]["seconds"] = round(s1 - s0, 3)
                out["reasons"] = sorted(set(out["reasons"]) | set(out["sustained"]["reasons"]))
        return out


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------
def run_ours(args, world, rank, local):
    import torch
    from paged_kv_cache_163_gb300 import capi, play

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    capi.load()
    capi.pkv_set_decode_kernel(args.kernel)
    capi.pkv_set_prefix_kernel(args.prefix_kernel, args.prefix_chunk_tiles)
    wid = WORKLOADS[args.workload]
    e2e_steps = 0 if args.no_e2e else max(3, min(args.steps, 20))
    e2e_warmup = 0 if args.no_e2e else max(3, args.warmup)
    attn_steps = max(3, min(args.steps, 30))
    host_steps = max(3, min(args.steps, 10))
    total_steps = args.warmup + args.steps + attn_steps + host_steps + e2e_warmup + e2e_steps
    w = wl.make(wid, extra_steps=max(total_steps, CPU_MAX_STEPS) + 1, cache_dtype=args.cache_dtype,
                block_size=args.block_size)
    cache = play.new_cache(w, device=dev)
    play.prefill(w, cache, device=dev)
    torch.cuda.synchronize()
    assert cache.check() == 0

    # every step's inputs resident in HBM before timing
    ins = [play.step_inputs(w, s, device=dev) for s in range(args.warmup + args.steps + attn_steps + host_steps)]
    out = torch.empty_like(ins[0][2])
    scrub = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    if args.graph:
        # graph replay: the step reads fixed buffers, refilled before each step (before the L2 flush)
        cache.use_graphs(True)
        static = [torch.empty_like(t) for t in ins[0]]

    def feed(s):
        if not args.graph:
            return ins[s]
        for dst, src in zip(static, ins[s]):
            dst.copy_(src)
        return static

    # the clock sampler starts before the warm-up steps: its start-up (a subprocess and a pause
    # for its first samples) left the host slow for the first timed step when it came just before
    clocks = ClockSampler(local)
    clocks.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for s in range(args.warmup):
        k, v, q = feed(s)
        scrub(s)
        cache.step(w.seq_ids, k, v, q, scale=w.scale, out=out)
    torch.cuda.synchronize()
    assert cache.check() == 0

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launches0 = capi.pkv_launch_count()
    clocks.mark("t0")
    with no_gc():
        for i in range(args.steps):
            k, v, q = feed(args.warmup + i)
            scrub(i + 7)
            ev[i][0].record(stream)
            cache.step(w.seq_ids, k, v, q, scale=w.scale, out=out)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    clocks.mark("t1")
    if world > 1:
        torch.distributed.barrier()
    launches = capi.pkv_launch_count() - launches0
    # clock evidence: the timed steps last milliseconds, nvidia-smi samples every
    # 50 ms, so keep sampling through >= 0.6 s of attention calls on the same
    # cache (layer 0, L2 flushed before each call as in the timed loop)
    sustained_calls = sustain_load(cache, w, ins[0][2], scrub, clocks, seconds=0.6)
    clk = clocks.stop()
    if "sustained" in clk:
        clk["sustained"]["calls"] = sustained_calls
    step_ms = [a.elapsed_time(b) for a, b in ev]
    assert cache.check() == 0

    # the attention launches alone: further steps with events around them (the
    # two extra events per step stay out of the step timing above)
    marks = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(attn_steps)]
    first_attn = args.warmup + args.steps
    with no_gc():
        for i in range(attn_steps):
            k, v, q = feed(first_attn + i)
            scrub(i + 3)
            cache.step(w.seq_ids, k, v, q, scale=w.scale, out=out, marks=marks[i])
        torch.cuda.synchronize()
    attn_ms = [a.elapsed_time(b) for a, b in marks]
    assert cache.check() == 0

    # host cost of one step call (block manager, staging, launches): the
    # device is idle before each call, so the call never waits for it
    first_host = first_attn + attn_steps
    host_us = []
    for i in range(host_steps):
        k, v, q = feed(first_host + i)
        torch.cuda.synchronize()
        h0 = time.perf_counter()
        cache.step(w.seq_ids, k, v, q, scale=w.scale, out=out)
        host_us.append((time.perf_counter() - h0) * 1e6)
    torch.cuda.synchronize()
    assert cache.check() == 0

    steps_acc = [step_accounting(w, args.warmup + i) for i in range(args.steps)]
    attn_acc = [step_accounting(w, first_attn + i) for i in range(attn_steps)]
    kv_total = sum(a["kv_bytes"] for a in steps_acc) * w.num_layers
    kv_attn = sum(a["kv_bytes"] for a in attn_acc) * w.num_layers
    tok_total = sum(a["tokens"] for a in steps_acc)
    t_total = sum(step_ms) / 1e3
    t_attn = sum(attn_ms) / 1e3
    t_total, t_attn = max_over_ranks([t_total, t_attn], device=dev)

    # end to end: inputs from pinned host memory, result read back, every step
    e2e = None
    if e2e_steps:
        e2e = run_e2e(w, cache, e2e_steps, first_host + host_steps, dev, scrub, warmup=e2e_warmup)

    peak, peak_kind = measured_peak()
    per_launch_bytes = statistics.mean(a["roofline_bytes"] for a in attn_acc)
    per_launch_s = t_attn / (attn_steps * w.num_layers)
    achieved = per_launch_bytes / per_launch_s / 1e9
    traffic_key = args.workload if args.cache_dtype is None else f"{args.workload}:{args.cache_dtype}"
    if args.block_size != 16:
        traffic_key += f":bs{args.block_size}"
    traffic = (NCU_TRAFFIC.get((traffic_key, kernel_hash()))
               if args.kernel == "auto" and args.prefix_kernel == "auto" else None)
    value = whole_job_rate(world, kv_total, t_total) / 1e9
    result = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_total * 1e3 / args.steps, 4),
        # spread of the timed steps on this rank (CUDA events around each step)
        "step_ms_percentiles": {f"p{q}": round(float(np.percentile(step_ms, q)), 4) for q in (10, 50, 90)},
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.cache_dtype if w.cache_dtype not in wl.SCALED_CACHES else
        f"{w.cache_dtype} ({w.q_dtype} q, fp32 accumulate)",
        "data": "synthetic (seeded N(0,1); no dataset or weights)",
        "config": workload_config(w, args.workload, {"parallelism": f"replicas x{world} (sequences sharded)",
                                                     "decode_kernel": args.kernel,
                                                     "prefix_kernel": args.prefix_kernel,
                                                     "step_launch": "cuda graph replay" if args.graph else "eager"}),
        "hbm_frac_step": round(value / world / peak, 4),
        "seq_tokens_per_s_per_layer": round(world * tok_total / (t_total / w.num_layers), 1),
        "attn_only": {"kv_read_gbs": round(kv_attn / t_attn / 1e9, 2),
                      "kv_unique_gbs": round(sum(a["kv_unique_bytes"] for a in attn_acc) * w.num_layers
                                             / t_attn / 1e9, 2),
                      "ms_per_step": round(t_attn * 1e3 / attn_steps, 4), "steps": attn_steps},
        "roofline": {"bound": "hbm", "kernel": decode_kernel_name(w, args.kernel) + " (one decode call)",
                     "achieved": round(achieved, 1), "peak": peak, "peak_kind": f"{peak_kind} copy GB/s",
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic, "algorithmic_bytes_per_launch": int(per_launch_bytes),
                     "launch_us": round(per_launch_s * 1e6, 3)},
        "gpu_launches": int(launches),
        "host_us_per_step": round(statistics.median(host_us), 1),
        "clocks": clk,
        "kv_utilisation": kv_utilisation(w),
    }
    if e2e is not None:
        result["e2e"] = e2e
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    cache.close()
    if world > 1:
        torch.distributed.destroy_process_group()
    return result if rank == 0 else None


def sustain_load(cache, w, q, scrub, clocks, seconds):
    """Back-to-back attention calls (no append) for about `seconds` of device time; returns the call count."""
    import torch
    q0 = q if q.dim() == 3 else q[0]
    out = torch.empty_like(q0)
    calls = 0
    torch.cuda.synchronize()
    clocks.mark("s0")
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        for i in range(32):
            scrub(i)
            cache.decode(w.seq_ids, q0, scale=w.scale, out=out)
        calls += 32
        torch.cuda.synchronize()
    clocks.mark("s1")
    assert cache.check() == 0
    return calls


def run_e2e(w, cache, steps, first_step, dev, scrub, warmup=3):
    """Same metric through the public API with host buffers: H2D inputs and D2H output every step.

    The first `warmup` steps run untimed (as for the device-input steps): the
    first host-buffer step sets up the step's device-side input buffers.
    """
    import torch
    from paged_kv_cache_163_gb300 import play
    hosts = []
    for s in range(first_step, first_step + warmup + steps):
        k = torch.from_numpy(w.step_rows(0, s)).to(play.torch_dtype(w.q_dtype)).pin_memory()
        v = torch.from_numpy(w.step_rows(1, s)).to(play.torch_dtype(w.q_dtype)).pin_memory()
        q = torch.from_numpy(np.stack([w.q_rows(layer, s) for layer in range(w.num_layers)])) \
            .to(play.torch_dtype(w.q_dtype)).pin_memory()
        hosts.append((k, v, q))
    out_h = torch.empty(hosts[0][2].shape, dtype=hosts[0][2].dtype).pin_memory()
    stream = torch.cuda.current_stream(dev)
    for i, (k, v, q) in enumerate(hosts[:warmup]):
        scrub(i)
        cache.step(w.seq_ids, k, v, q, scale=w.scale, out=out_h)
    hosts = hosts[warmup:]
    first_step += warmup
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    with no_gc():
        _e2e_steps(w, cache, hosts, ev, stream, scrub, out_h)
    torch.cuda.synchronize()
    assert cache.check() == 0
    t = sum(a.elapsed_time(b) for a, b in ev) / 1e3
    kv = sum(step_accounting(w, first_step + i)["kv_bytes"] for i in range(steps)) * w.num_layers
    lens = w.context_lens + first_step
    max_blocks = int(max(-(-int(L) // w.block_size) for L in lens))
    meta_bytes = 4 * (w.num_seqs + w.num_seqs * max_blocks + w.num_seqs)
    h2d = sum(x.numel() * x.element_size() for x in hosts[0]) + meta_bytes
    step_ms = [a.elapsed_time(b) for a, b in ev]
    return {"value": round(kv / t / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(out_h.numel() * out_h.element_size()), "steps": steps,
            "ms_per_step": round(t * 1e3 / steps, 4),
            "step_ms_percentiles": {f"p{q}": round(float(np.percentile(step_ms, q)), 4) for q in (10, 50, 90)},
            "step_ms_max": round(max(step_ms), 4)}


def _e2e_steps(w, cache, hosts, ev, stream, scrub, out_h):
    """The timed host-buffer steps of run_e2e (CUDA events around each step)."""
    for i, (k, v, q) in enumerate(hosts):
        scrub(i)
        ev[i][0].record(stream)
        # host tensors in, host tensor out: the step copies the inputs in with one kernel, and the
        # decode stores the output straight into the page-locked host tensor
        cache.step(w.seq_ids, k, v, q, scale=w.scale, out=out_h)
        ev[i][1].record(stream)


# ---------------------------------------------------------------------------
# CPU oracle arm
# ---------------------------------------------------------------------------
CPU_MAX_STEPS = 400


def oracle_sample_state(w: wl.Workload, seqs, max_steps=CPU_MAX_STEPS):
    """Oracle allocator + paged cache pre-filled for the sampled sequences (setup, untimed)."""
    from oracle.model import PagedKVOracle
    need = sum(-(-int(w.context_lens[s] + max_steps + 1) // 16) for s in seqs) + 8
    o = PagedKVOracle(1, need, w.num_kv_heads, w.head_dim, w.cache_dtype)
    for s in seqs:
        o.create(s)
        L = int(w.context_lens[s]) - 1
        if L > 0:
            o.append([s] * L, [w.kv_rows(0, s, 0, L)], [w.kv_rows(1, s, 0, L)])
    return o


def oracle_steps(w, o, seqs, step0, budget_s, max_steps=None):
    """Timed oracle decode steps (append + attention) over the sampled sequences."""
    t_total, n, kv, toks = 0.0, 0, 0, 0
    step = step0
    while (t_total < budget_s and (max_steps is None or n < max_steps)) or n == 0:
        k = np.stack([w.kv_rows(0, s, int(w.context_lens[s]) - 1 + step, int(w.context_lens[s]) + step)[0]
                      for s in seqs])
        v = np.stack([w.kv_rows(1, s, int(w.context_lens[s]) - 1 + step, int(w.context_lens[s]) + step)[0]
                      for s in seqs])
        q = w.q_rows(0, step)[list(seqs)]
        t0 = time.perf_counter()
        o.append(list(seqs), [k], [v])
        o.decode(list(seqs), q, w.scale)
        t_total += time.perf_counter() - t0
        lens = [int(w.context_lens[s]) + step for s in seqs]
        kv += sum(lens) * w.num_kv_heads * wl.token_head_bytes(w.cache_dtype, w.head_dim)
        toks += sum(lens)
        n += 1
        step += 1
    return t_total, n, kv, toks


def sample_seqs(w, budget_tokens):
    order = np.argsort(w.context_lens)[::-1]
    seqs, tot = [], 0
    for s in order[len(order) // 2:].tolist() + order[:len(order) // 2].tolist():
        if tot > 0 and tot + w.context_lens[s] > budget_tokens:
            continue
        seqs.append(int(s))
        tot += int(w.context_lens[s])
        if tot >= budget_tokens:
            break
    return sorted(seqs)


def cores_available() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_worker(spec, barrier, results):
    """One process of the all-cores oracle baseline (spawned; BLAS threads 1).

    Builds the oracle state of its own sequences (untimed), waits for every
    worker at the barrier, then runs timed oracle decode steps for the
    budget and reports (seqs, seconds, steps, KV bytes, context tokens).
    """
    wid, extra, cache_dtype, block_size, seqs, budget_s = spec
    try:
        w = wl.make(wid, extra_steps=extra, cache_dtype=cache_dtype, block_size=block_size)
        o = oracle_sample_state(w, seqs)
        barrier.wait(timeout=900)
        t, n, kv, toks = oracle_steps(w, o, seqs, 0, budget_s, max_steps=CPU_MAX_STEPS)
        results.put((seqs, t, n, kv, toks, None))
    except BaseException as e:  # report, so the parent never waits for a dead worker
        barrier.abort()
        results.put((seqs, 0.0, 0, 0, 0, repr(e)))


def cpu_baseline_all_cores(w, budget_s, workers):
    """The oracle on every host core: a process pool over the workload's sequences.

    Each spawned worker takes every workers-th sequence of the batch, so the
    pool runs whole decode steps of the workload; the rate is the KV bytes
    all workers processed over the slowest worker's time.
    """
    import multiprocessing as mp
    ctx = mp.get_context("spawn")  # never fork a process that has touched the GPU
    n = max(1, min(workers, w.num_seqs))
    shards = [list(range(i, w.num_seqs, n)) for i in range(n)]
    barrier = ctx.Barrier(n)
    results = ctx.Queue()
    extra = CPU_MAX_STEPS + 1
    procs = [ctx.Process(target=_oracle_worker, daemon=True,
                         args=((w.wid, extra, w.cache_dtype if w.cache_dtype in wl.SCALED_CACHES else None,
                                w.block_size, sh, budget_s), barrier, results)) for sh in shards]
    for p in procs:
        p.start()
    got = []
    try:
        for _ in procs:
            got.append(results.get(timeout=1800))
    finally:
        for p in procs:
            p.join(timeout=30)
            if p.is_alive():
                p.terminate()
    errors = [g[5] for g in got if g[5]]
    if errors:
        raise RuntimeError(f"all-cores oracle baseline failed: {errors[0]}")
    t = max(g[1] for g in got)
    kv = sum(g[3] for g in got)
    toks = sum(g[4] for g in got)
    steps = min(g[2] for g in got)
    return {"value": round(kv / t / 1e9, 4), "unit": "GB/s", "cores": n, "kind": "oracle",
            "seq_tokens_per_s_per_layer": round(toks / t, 1),
            "sample": f"{n} spawned processes (BLAS threads = 1 each), each with every {n}th sequence of all "
                      f"{w.num_seqs}; {steps}-{max(g[2] for g in got)} oracle decode steps per process "
                      f"(append + fp64 attention, layer 0), {t:.1f} s for the slowest"}


def cpu_baseline(w, budget_s):
    """The oracle timed on the host: one core, then every core (a process pool over sequences)."""
    seqs = sample_seqs(w, 20000 if w.cache_dtype in wl.SCALED_CACHES else 6000)
    o = oracle_sample_state(w, seqs)
    t, n, kv, toks = oracle_steps(w, o, seqs, 0, budget_s, max_steps=CPU_MAX_STEPS)
    del o
    one = {"value": round(kv / t / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
           "seq_tokens_per_s_per_layer": round(toks / t, 1),
           "sample": f"{n} oracle decode steps (append + fp64 attention, layer 0) over sequences {seqs} "
                     f"of {len(w.context_lens)} ({toks // max(n, 1)} context tokens per step), "
                     f"{t:.1f} s on 1 host core (BLAS threads = 1)"}
    avail = cores_available()
    try:
        allc = cpu_baseline_all_cores(w, budget_s, avail)
    except Exception as e:  # the single-core figure still stands
        allc = {"error": str(e)[:300]}
    top = dict(allc) if "value" in allc else dict(one)
    top["cores_available"] = avail
    top["modes"] = {"one_core": one, "all_cores": allc}
    return top


def run_reference(args, world, rank):
    if rank != 0:
        return None
    wid = WORKLOADS[args.workload]
    w = wl.make(wid, extra_steps=max(args.warmup + args.steps + 1, CPU_MAX_STEPS + 1), cache_dtype=args.cache_dtype,
                block_size=args.block_size)
    seqs = sample_seqs(w, 17000 if w.cache_dtype in wl.SCALED_CACHES else 3000)
    o = oracle_sample_state(w, seqs, max_steps=args.warmup + args.steps + 1)
    oracle_steps(w, o, seqs, 0, 0.0, max_steps=args.warmup)
    t, n, kv, toks = oracle_steps(w, o, seqs, args.warmup, float("inf"), max_steps=args.steps)
    value = kv / t / 1e9
    peak, peak_kind = measured_peak()
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t * 1e3 / n, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded N(0,1); no dataset or weights)",
        "config": workload_config(w, args.workload, {"parallelism": "single host process"}),
        "seq_tokens_per_s_per_layer": round(toks / t, 1),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "cores_available": cores_available(),
                         "sample": f"each step: oracle append + fp64 attention over sequences {seqs} "
                                   f"of {len(w.context_lens)}, layer 0, on 1 host core (BLAS threads = 1)"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main(argv=None):
    args = parse_args(argv)
    world, rank, local = dist_env()
    if args.impl == "reference":
        res = run_reference(args, world, rank)
    else:
        res = run_ours(args, world, rank, local)
    if res is not None and rank == 0:
        print(json.dumps(res), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
