"""The fused append + decode call against the separate append and decode.

``paged_attention_decode_append`` writes each sequence's new K/V row from
inside the decode kernel (by the warp that owns the sequence's last tile)
and then attends.  It must leave the cache byte for byte as
``paged_kv_append`` does and produce bit for bit the output of
``paged_attention_decode`` run after that append.  The step executor uses
the fused call for every layer; its parity with the oracle is covered by
the decode tests.
"""
import numpy as np
import pytest

from paged_kv_cache_163_gb300 import workloads as wl

from helpers import cache_bits

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def play():
    from paged_kv_cache_163_gb300 import capi, play as p
    capi.load()
    return p


@pytest.fixture
def kernel_kind(request):
    from paged_kv_cache_163_gb300 import capi
    capi.pkv_set_decode_kernel(request.param)
    yield request.param
    capi.pkv_set_decode_kernel("auto")


def _two_caches(play, w):
    a, b = play.new_cache(w, poison=True), play.new_cache(w, poison=True)
    play.prefill(w, a)
    play.prefill(w, b)
    return a, b


@pytest.mark.parametrize("kernel_kind", ["simt", "mma"], indirect=True)
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("q_dtype,cache_dtype", [("bf16", "bf16"), ("f16", "f16"), ("bf16", "fp8_e4m3"),
                                                 ("f16", "int8"), ("bf16", "fp8_e5m2"),
                                                 ("bf16", "fp8_e4m3_int4"), ("f16", "fp8_e4m3_int4")])
def test_fused_equals_separate(play, kernel_kind, d, q_dtype, cache_dtype):
    from paged_kv_cache_163_gb300 import capi
    # lengths before the step's token: block starts, block ends, mid-block, an empty cache
    lens = [16, 17, 31, 32, 1, 48, 700, 5, 2, 129]
    w = wl.custom(f"fused-{d}-{cache_dtype}", lens=lens, num_q_heads=8, num_kv_heads=2, head_dim=d,
                  q_dtype=q_dtype, cache_dtype=cache_dtype, outlier_p=0.01, seed=40 + d)
    a, b = _two_caches(play, w)
    k, v, q = play.step_inputs(w, 0)
    q0 = q[0]
    # separate: append kernel, then decode
    a.append(w.seq_ids, k, v)
    out_a = a.decode(w.seq_ids, q0, scale=w.scale, out=torch.empty(q0.shape, dtype=torch.float32, device="cuda"))
    # fused: the block manager grows the tables, then one launch appends and attends
    slots, cs, cd = capi.pkv_seq_append_slots(b.bm, w.seq_ids)
    assert len(cs) == 0
    tables, ctx = b.tables(w.seq_ids)
    dev = torch.device("cuda")
    d_tables = torch.from_numpy(tables).to(dev)
    d_ctx = torch.from_numpy(ctx).to(dev)
    ws = b.workspace(len(lens), w.num_q_heads, q_dtype)
    out_b = torch.empty(q0.shape, dtype=torch.float32, device=dev)
    ks = b.k_scale[0] if b.k_scale is not None else None
    vs = b.v_scale[0] if b.v_scale is not None else None
    capi.paged_attention_decode_append(out_b, q0, k, v, b.k[0], b.v[0], ks, vs, d_tables, d_ctx, int(ctx.max()),
                                       w.scale, ws, d_error=b.err, cache_dtype=cache_dtype)
    assert a.check() == 0 and b.check() == 0
    assert np.array_equal(cache_bits(a.k[0]), cache_bits(b.k[0]))
    assert np.array_equal(cache_bits(a.v[0]), cache_bits(b.v[0]))
    if ks is not None:
        assert np.array_equal(a.k_scale[0].cpu().numpy().view(np.uint32), ks.cpu().numpy().view(np.uint32))
        assert np.array_equal(a.v_scale[0].cpu().numpy().view(np.uint32), vs.cpu().numpy().view(np.uint32))
    assert torch.equal(out_a, out_b)
    a.close()
    b.close()


def test_fused_step_over_many_layers_equals_separate(play):
    """The step executor (fused, 6 layers, shared prefix blocks) against per-layer append + decode."""
    prefix = 40
    lens = [prefix + s for s in (3, 30, 1, 70)]
    w = wl.custom("fused-layers", lens=lens, num_q_heads=16, num_kv_heads=4, head_dim=128, q_dtype="bf16",
                  cache_dtype="fp8_e4m3", prefix_len=prefix, num_layers=6, seed=77)
    a, b = _two_caches(play, w)
    k, v, q = play.step_inputs(w, 0)
    out_a = a.step(w.seq_ids, k, v, q, scale=w.scale)
    b.append(w.seq_ids, k, v)
    assert a.cow_pairs == b.cow_pairs
    out_b = b.decode(w.seq_ids, q, scale=w.scale)
    assert a.check() == 0 and b.check() == 0
    for li in range(6):
        assert np.array_equal(cache_bits(a.k[li]), cache_bits(b.k[li]))
        assert np.array_equal(cache_bits(a.v[li]), cache_bits(b.v[li]))
    assert torch.equal(out_a, out_b)
    a.close()
    b.close()
