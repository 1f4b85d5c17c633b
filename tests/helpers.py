"""Shared test helpers: play a workload on the oracle, compare GPU and oracle results."""
import numpy as np

from oracle.attention import decode_attention
from oracle.cache import dequantize_rows
from oracle.model import PagedKVOracle

# Attention tolerance (stated for bf16 / fp16 and FP8-dequantised caches):
# max |gpu - oracle| <= 1e-2 and ||gpu - oracle||_2 / ||oracle||_2 <= 2e-3,
# applied to the kernel's fp32 result.  A 16-bit output is that result rounded
# once (checked bit for bit by check_rounding): rounding alone moves a bf16
# value by up to 2^-8 of itself, more than 1e-2 once |x| >= 2.56, which the
# x20 outliers of the FP8 workload produce.
MAX_ABS = 1e-2
REL_L2 = 2e-3


def oracle_play(w, alloc_order=None, layers=1, with_step=True):
    """Pre-fill (and the decode step's append) on the oracle; returns the oracle state."""
    o = PagedKVOracle(layers, w.num_blocks, w.num_kv_heads, w.head_dim, w.cache_dtype,
                      block_size=w.block_size,
                      alloc_order=w.alloc_order if alloc_order is None else alloc_order)
    for op in w.prefill_ops():
        if op[0] == "create":
            o.create(op[1])
        elif op[0] == "fork":
            o.fork(op[1], op[2])
        else:
            seqs = op[1]
            start = o.alloc.lens[seqs[0]]
            k = w.kv_rows(0, seqs[0], start, start + len(seqs))
            v = w.kv_rows(1, seqs[0], start, start + len(seqs))
            o.append(seqs, [k] * layers, [v] * layers)
    if with_step:
        o.append(w.seq_ids, [w.step_rows(0)] * layers, [w.step_rows(1)] * layers)
    return o


def oracle_seq_output(w, seq, q_seq, step=0):
    """fp64 [Hq, D] attention of one sequence from its token rows (paged == contiguous)."""
    L = int(w.context_lens[seq]) + step
    K = dequantize_rows(w.kv_rows(0, seq, 0, L), w.cache_dtype)
    V = dequantize_rows(w.kv_rows(1, seq, 0, L), w.cache_dtype, "v")
    return decode_attention(q_seq, K, V, w.scale)


def to_f64(t):
    import torch
    return t.detach().to(torch.float64).cpu().numpy()


def errors(gpu, ref):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    max_abs = float(np.max(np.abs(gpu - ref))) if gpu.size else 0.0
    den = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(gpu - ref) / den) if den > 0 else float(np.linalg.norm(gpu - ref))
    return max_abs, rel


def assert_close(gpu, ref, what=""):
    max_abs, rel = errors(gpu, ref)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite output"
    assert max_abs <= MAX_ABS and rel <= REL_L2, f"{what}: max_abs={max_abs:.3g} rel_l2={rel:.3g}"
    return max_abs, rel


def cache_bits(t):
    """Raw bits of a device cache tensor as a numpy array (uint16 for 16-bit, uint8 for FP8)."""
    import torch
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.detach().cpu().numpy()


def oracle_bits(values, dtype):
    """Bits of exact float32 values in a 16-bit cache dtype."""
    v = np.asarray(values, dtype=np.float32)
    if dtype == "bf16":
        return (v.view(np.uint32) >> 16).astype(np.uint16)
    return v.astype(np.float16).view(np.uint16)


def check_rounding(cache, w, out32, layers=None):
    """The query-dtype output equals the fp32 output rounded once to nearest even; returns it."""
    import torch
    from paged_kv_cache_163_gb300.play import to_device
    q = to_device(np.stack([w.q_rows(li) for li in range(w.num_layers)]), w.q_dtype, out32.device)
    out16 = cache.decode(w.seq_ids, q, scale=w.scale, layers=layers)
    sel = out32 if layers is None else out32[list(layers)]
    got = out16 if layers is None else out16[list(layers)]
    assert torch.equal(got, sel.to(got.dtype)), "16-bit output is not the fp32 result rounded once"
    return out16


def coded_seq_reference(args):
    """Oracle results of one sequence of a coded-cache workload, for a process pool.

    args = (workload id, cache dtype, sequence).  Returns (sequence, K codes
    [L, Hkv, row], K scales [L, Hkv], V codes, V scales, fp64 attention
    output [Hq, D] of the step's query over the dequantised codes).
    """
    from oracle.cache import code_values, part_types, quantize_rows
    from paged_kv_cache_163_gb300 import workloads as wl
    wid, cache_dtype, seq = args
    w = wl.make(wid, cache_dtype=cache_dtype)
    L = int(w.context_lens[seq])
    kt, vt = part_types(w.cache_dtype)
    kc, ks = quantize_rows(w.kv_rows(0, seq, 0, L), kt)
    vc, vs = quantize_rows(w.kv_rows(1, seq, 0, L), vt)
    K = code_values(kc, kt) * ks.astype(np.float64)[..., None]
    V = code_values(vc, vt) * vs.astype(np.float64)[..., None]
    ref = decode_attention(w.q_rows(0)[seq], K, V, w.scale)
    return seq, kc, ks, vc, vs, ref


def parallel_map(fn, items, max_workers=16):
    """fn over items in spawned processes (BLAS threads 1 each); results in item order."""
    import multiprocessing as mp
    import os
    from concurrent.futures import ProcessPoolExecutor
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        cores = os.cpu_count() or 1
    n = max(1, min(max_workers, cores, len(items)))
    keys = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {k: os.environ.get(k) for k in keys}
    for k in keys:
        os.environ[k] = "1"
    try:
        with ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn")) as ex:
            return list(ex.map(fn, items))
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def compare_cache_bytes(cache, model, cache_dtype, layer=0):
    """Every slot the oracle's PagedCacheModel marks filled holds the same bytes (and scales) on the GPU."""
    filled = model.filled
    scaled = model.k_scale is not None or model.v_scale is not None
    for got, want, part in ((cache.k[layer], model.k, model.k_type), (cache.v[layer], model.v, model.v_type)):
        g = cache_bits(got).transpose(0, 2, 1, 3)[filled]
        w = want.transpose(0, 2, 1, 3)[filled]
        if part in ("f16", "bf16"):
            w = oracle_bits(w, part)
        assert np.array_equal(g, w), f"{part} cache bytes differ"
    if scaled:
        for got, want in ((cache.k_scale[layer], model.k_scale), (cache.v_scale[layer], model.v_scale)):
            if want is None:
                continue
            g = got.cpu().numpy().transpose(0, 2, 1)[filled]
            assert np.array_equal(g, want.transpose(0, 2, 1)[filled]), f"{cache_dtype} scales differ"
