"""The decode entry point that allocates nothing, checked against the workspace one.

Some callers of this library cannot allocate device memory: a plugin whose
host framework owns every device allocation, or a latency-critical loop
where an allocation could synchronise the device.
paged_attention_decode_static serves them with scratch that lives inside
the library.  Here it must give the same attention output as
paged_attention_decode with a caller workspace, within the tolerance the
other parity tests use, on two calls in a row (the second call reuses the
scratch the first one left behind).  It must also reject shapes whose
scratch would not fit.  This file is collected last so that a failure here
stops a `-x` run only after every other test has run.
"""
import numpy as np
import pytest

from paged_kv_cache_163_gb300 import workloads as wl

from helpers import assert_close, to_f64

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
