"""The decode entry point that allocates nothing, checked against the workspace one.

Some callers of this library cannot allocate device memory: a plugin whose
host framework owns every device allocation, or a latency-critical loop
where an allocation could synchronise the device.
paged_attention_decode_static serves them with scratch that lives inside
the library.  Here it must give the same attention output as
paged_attention_decode with a caller workspace, within the tolerance the
other parity tests use, on two calls in a row (the second call reuses the
scratch the first one left behind), on back-to-back calls whose batch
sizes differ, and when a fresh process makes its first call on a
non-blocking stream (checked against the oracle).  It must also reject
shapes whose scratch would not fit.  This file is collected last so that a
failure here stops a `-x` run only after every other test has run.
"""
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest

from paged_kv_cache_163_gb300 import workloads as wl

from helpers import assert_close, to_f64

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mods():
    from paged_kv_cache_163_gb300 import capi, play
    capi.load()
    return capi, play


@pytest.mark.parametrize("wid", [2, 0])
def test_static_scratch_matches_workspace_entry(mods, wid):
    capi, play = mods
    if wid == 0:
        w = wl.custom("fp8-small", lens=[1, 40, 300, 2500, 17], num_q_heads=32, num_kv_heads=8,
                      head_dim=128, q_dtype="bf16", cache_dtype="fp8_e4m3", outlier_p=0.001, seed=8)
    else:
        w = wl.make(wid)
    cache, _ = play.run(w)
    assert cache.check() == 0
    dev = torch.device("cuda")
    tables, lens = cache.tables(w.seq_ids)
    d_tables = torch.from_numpy(tables).to(dev)
    d_lens = torch.from_numpy(lens).to(dev)
    q = play.to_device(w.q_rows(0), w.q_dtype, dev)
    ks = cache.k_scale[0] if cache.k_scale is not None else None
    vs = cache.v_scale[0] if cache.v_scale is not None else None
    ws = cache.workspace(w.num_seqs, w.num_q_heads, w.q_dtype)
    ref = torch.empty(q.shape, dtype=torch.float32, device=dev)
    capi.paged_attention_decode(ref, q, cache.k[0], cache.v[0], ks, vs, d_tables, d_lens, int(lens.max()),
                                w.scale, ws, d_error=cache.err)
    assert cache.check() == 0
    for call in range(2):
        out = torch.full(q.shape, float("nan"), dtype=torch.float32, device=dev)
        capi.paged_attention_decode_static(out, q, cache.k[0], cache.v[0], ks, vs, d_tables, d_lens,
                                           int(lens.max()), w.scale, d_error=cache.err)
        assert cache.check() == 0
        assert_close(to_f64(out), to_f64(ref), f"static scratch call {call}")
    # the 16-bit output through the same entry point
    out16 = torch.empty_like(q)
    capi.paged_attention_decode_static(out16, q, cache.k[0], cache.v[0], ks, vs, d_tables, d_lens,
                                       int(lens.max()), w.scale, d_error=cache.err)
    assert cache.check() == 0
    assert torch.equal(out16, ref.to(q.dtype))
    cache.close()


def test_static_scratch_rejects_oversized_shapes(mods):
    capi, _ = mods
    dev = torch.device("cuda")
    b, hq, hkv, d = 1024, 64, 8, 128
    need = capi.paged_attention_workspace_bytes(b, hq, hkv, d, "bf16", "bf16")
    assert need > (16 << 20)
    q = torch.zeros((b, hq, d), dtype=torch.bfloat16, device=dev)
    kc = torch.zeros((4, hkv, 16, d), dtype=torch.bfloat16, device=dev)
    tables = torch.zeros((b, 1), dtype=torch.int32, device=dev)
    lens = torch.ones(b, dtype=torch.int32, device=dev)
    with pytest.raises(capi.PkvError) as e:
        capi.paged_attention_decode_static(torch.empty_like(q), q, kc, kc, None, None, tables, lens, 1, 0.1)
    assert e.value.status == -6
    assert "static buffer" in str(e.value)


def test_static_scratch_batch_size_changes(mods):
    """Back-to-back calls with different num_seqs (the split counters are cleared again for each shape)."""
    capi, play = mods
    w = wl.custom("fp8-batches", lens=[5000, 40, 3000, 1, 700, 17], num_q_heads=32, num_kv_heads=8,
                  head_dim=128, q_dtype="bf16", cache_dtype="fp8_e4m3", outlier_p=0.001, seed=21)
    cache, _ = play.run(w)
    assert cache.check() == 0
    dev = torch.device("cuda")
    tables, lens = cache.tables(w.seq_ids)
    d_tables = torch.from_numpy(tables).to(dev)
    d_lens = torch.from_numpy(lens).to(dev)
    q = play.to_device(w.q_rows(0), w.q_dtype, dev)
    ks, vs = cache.k_scale[0], cache.v_scale[0]
    for b in (6, 2, 5, 6, 1, 6):
        ws = cache.workspace(b, w.num_q_heads, w.q_dtype)
        ref = torch.empty((b,) + tuple(q.shape[1:]), dtype=torch.float32, device=dev)
        capi.paged_attention_decode(ref, q[:b], cache.k[0], cache.v[0], ks, vs, d_tables[:b], d_lens[:b],
                                    int(lens[:b].max()), w.scale, ws, d_error=cache.err)
        out = torch.full(ref.shape, float("nan"), dtype=torch.float32, device=dev)
        capi.paged_attention_decode_static(out, q[:b], cache.k[0], cache.v[0], ks, vs, d_tables[:b], d_lens[:b],
                                           int(lens[:b].max()), w.scale, d_error=cache.err)
        assert cache.check() == 0
        assert_close(to_f64(out), to_f64(ref), f"static scratch, {b} sequences")
    cache.close()


FIRST_CALL_ON_SIDE_STREAM = textwrap.dedent("""
    import sys
    import numpy as np
    import torch
    sys.path[:0] = [{root!r}, {tests!r}]
    from paged_kv_cache_163_gb300 import capi, play, workloads as wl
    from helpers import assert_close, oracle_play, to_f64
    capi.load()
    w = wl.custom("fp8-side", lens=[3000, 17, 1, 900], num_q_heads=32, num_kv_heads=8, head_dim=128,
                  q_dtype="bf16", cache_dtype="fp8_e4m3", outlier_p=0.001, seed=23)
    cache, _ = play.run(w)
    tables, lens = cache.tables(w.seq_ids)
    dev = torch.device("cuda")
    d_tables = torch.from_numpy(tables).to(dev)
    d_lens = torch.from_numpy(lens).to(dev)
    q = play.to_device(w.q_rows(0), w.q_dtype, dev)
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()            # torch creates its streams non-blocking
    with torch.cuda.stream(side):
        # the process's first static call: its set-up and the counter clear go on `side`
        capi.paged_attention_decode_static(out, q, cache.k[0], cache.v[0], cache.k_scale[0], cache.v_scale[0],
                                           d_tables, d_lens, int(lens.max()), w.scale, d_error=cache.err,
                                           stream=side)
    side.synchronize()
    assert cache.check() == 0
    o = oracle_play(w)
    ref = o.decode(w.seq_ids, w.q_rows(0), w.scale)
    m, r = assert_close(to_f64(out), ref, "first static call on a side stream")
    print("ok", m, r)
""")


def test_static_scratch_first_call_on_side_stream():
    """A fresh process whose first static call runs on a non-blocking stream matches the oracle."""
    script = FIRST_CALL_ON_SIDE_STREAM.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    r = subprocess.run([sys.executable, "-c", script], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert r.stdout.strip().startswith("ok")
