"""Cascade decode for shared prefixes, against the oracle and the plain decode.

Sequences forked from one parent share their prefix's blocks.  With the
cascade, a prefix kernel attends the shared tiles once for every member's
queries and the decode merges its partials with each member's own tiles.
The attention is unchanged: results must match the oracle (fp64 over each
member's whole context) within the tolerance, match the step without the
cascade within it too (the fp32 additions come in another order), and
leave the cache byte for byte as the plain step does.

16-bit caches run both prefix kernels: the tcgen05 one (tensor-memory
accumulators, 64-token sub-chunks; also with chunks that are not a
multiple of a sub-chunk, and with one chunk of many sub-chunks) and the
warp-level mma.sync one, for GQA groups of 1, 2, 4 and 8; asking for the
tcgen05 kernel with a one-byte cache keeps the mma.sync one.
"""
import numpy as np
import pytest

from oracle.attention import decode_attention
from oracle.cache import dequantize_rows
from paged_kv_cache_163_gb300 import workloads as wl

from helpers import assert_close, cache_bits, to_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def play():
    from paged_kv_cache_163_gb300 import capi, play as p
    capi.load()
    return p


@pytest.fixture
def prefix_kernel(request):
    """Run a test under one prefix kernel (and chunk size), then restore the default."""
    from paged_kv_cache_163_gb300 import capi
    kind, chunk = request.param
    capi.pkv_set_prefix_kernel(kind, chunk)
    yield kind
    capi.pkv_set_prefix_kernel("auto", 0)


def _rows(rng, n, hkv, d, dtype):
    x = rng.standard_normal((n, hkv, d)).astype(np.float32)
    x[rng.random((n, hkv, d)) < 0.002] *= 20
    return wl.round_to(x, dtype)


def _build(play, groups, loners, *, hq, hkv, d, q_dtype, cache_dtype, bs, seed, cascade):
    """Groups of (prefix length, [member lengths after the step]); loners: lengths of unshared sequences.

    Returns (cache, members in step order, their rows [(K, V)] including the step's token, q, out).
    """
    from paged_kv_cache_163_gb300.engine import PagedKVCache
    rng = np.random.default_rng(seed)
    need = sum(-(-P // bs) + sum(-(-(P % bs + L) // bs) + 1 for L in ls) for P, ls in groups)
    need += sum(-(-L // bs) + 1 for L in loners)
    cache = PagedKVCache(num_layers=1, num_blocks=need + 16, num_kv_heads=hkv, head_dim=d,
                         cache_dtype=cache_dtype, block_size=bs, poison=True)
    cache.use_cascade(cascade)
    dev = "cuda"
    seq, members, rows = 0, [], []
    for P, lens in groups:
        parent = seq
        seq += 1
        kp, vp = _rows(rng, P, hkv, d, q_dtype), _rows(rng, P, hkv, d, q_dtype)
        cache.create(parent)
        cache.append([parent] * P, play.to_device(kp, q_dtype, dev), play.to_device(vp, q_dtype, dev))
        for L in lens:
            m = seq
            seq += 1
            cache.fork(parent, m)
            ks, vs = _rows(rng, L - P, hkv, d, q_dtype), _rows(rng, L - P, hkv, d, q_dtype)
            if L - P > 1:
                cache.append([m] * (L - P - 1), play.to_device(ks[:-1], q_dtype, dev),
                             play.to_device(vs[:-1], q_dtype, dev))
            members.append(m)
            rows.append((np.concatenate([kp, ks]), np.concatenate([vp, vs])))
        cache.free(parent)
    for L in loners:
        m = seq
        seq += 1
        ks, vs = _rows(rng, L, hkv, d, q_dtype), _rows(rng, L, hkv, d, q_dtype)
        cache.create(m)
        if L > 1:
            cache.append([m] * (L - 1), play.to_device(ks[:-1], q_dtype, dev), play.to_device(vs[:-1], q_dtype, dev))
        members.append(m)
        rows.append((ks, vs))
    # interleave the batch order so groups are not contiguous
    order = np.random.default_rng(seed + 1).permutation(len(members))
    members = [members[i] for i in order]
    rows = [rows[i] for i in order]
    q = _rows(rng, len(members), hq, d, q_dtype)[None]
    kn = np.stack([r[0][-1] for r in rows])
    vn = np.stack([r[1][-1] for r in rows])
    out = torch.empty(q.shape, dtype=torch.float32, device=dev)
    scale = float(np.float32(1.0) / np.sqrt(np.float32(d)))
    cache.step(members, play.to_device(kn, q_dtype, dev), play.to_device(vn, q_dtype, dev),
               play.to_device(q, q_dtype, dev), scale=scale, out=out)
    return cache, members, rows, q, out, scale


CASES = [("bf16", "bf16", 32, 8, 16), ("f16", "f16", 32, 4, 16), ("bf16", "fp8_e4m3", 32, 8, 16),
         ("bf16", "fp8_e4m3_int4", 32, 8, 16), ("f16", "int8", 8, 8, 16), ("bf16", "bf16", 32, 8, 32),
         ("bf16", "fp8_e5m2", 16, 8, 16), ("bf16", "bf16", 8, 8, 16), ("f16", "f16", 16, 8, 16)]


SIXTEEN_BIT = [c for c in CASES if c[1] in ("bf16", "f16")]
PREFIX_KERNELS = [("tcgen05", 0), ("tcgen05", 5), ("tcgen05", 200), ("mma_sync", 0)]


@pytest.mark.parametrize("prefix_kernel", PREFIX_KERNELS, indirect=True, ids=lambda k: f"{k[0]}-{k[1]}")
@pytest.mark.parametrize("q_dtype,cache_dtype,hq,hkv,bs", SIXTEEN_BIT)
def test_cascade_16bit_both_prefix_kernels(play, prefix_kernel, q_dtype, cache_dtype, hq, hkv, bs):
    test_cascade_matches_oracle_and_plain_step(play, q_dtype, cache_dtype, hq, hkv, bs)


@pytest.mark.parametrize("prefix_kernel", [("tcgen05", 0)], indirect=True, ids=lambda k: k[0])
@pytest.mark.parametrize("q_dtype,cache_dtype,hq,hkv,bs", [("bf16", "fp8_e4m3", 32, 8, 16), ("f16", "int8", 8, 8, 16)])
def test_tcgen05_request_on_one_byte_cache_falls_back(play, prefix_kernel, q_dtype, cache_dtype, hq, hkv, bs):
    """The tcgen05 prefix kernel takes 16-bit caches; a one-byte cache keeps the mma.sync one, correctly."""
    test_cascade_matches_oracle_and_plain_step(play, q_dtype, cache_dtype, hq, hkv, bs)


@pytest.mark.parametrize("q_dtype,cache_dtype,hq,hkv,bs", CASES)
def test_cascade_matches_oracle_and_plain_step(play, q_dtype, cache_dtype, hq, hkv, bs):
    groups = [(1500, [1564, 1600, 1501, 1800, 1517]), (700, [705, 1600]), (300, [340, 341, 342])]
    loners = [900, 33]
    kw = dict(hq=hq, hkv=hkv, d=128, q_dtype=q_dtype, cache_dtype=cache_dtype, bs=bs, seed=hq + hkv + bs)
    on, members, rows, q, out_on, scale = _build(play, groups, loners, cascade=True, **kw)
    off, _, _, _, out_off, _ = _build(play, groups, loners, cascade=False, **kw)
    assert on.check() == 0 and off.check() == 0
    assert on.cascade_count() == 1 and off.cascade_count() == 0
    got, plain = to_f64(out_on[0]), to_f64(out_off[0])
    for i, (k, v) in enumerate(rows):
        K = dequantize_rows(k, cache_dtype, "k")
        V = dequantize_rows(v, cache_dtype, "v")
        ref = decode_attention(q[0, i].astype(np.float32), K, V, scale)
        assert_close(got[i], ref, f"member {members[i]}")
        assert_close(got[i], plain[i], f"member {members[i]} against the plain step")
    assert np.array_equal(cache_bits(on.k[0]), cache_bits(off.k[0]))
    assert np.array_equal(cache_bits(on.v[0]), cache_bits(off.v[0]))
    on.close()
    off.close()


@pytest.mark.parametrize("prefix_kernel", [("tcgen05", 0), ("mma_sync", 0)], indirect=True, ids=lambda k: k[0])
def test_cascade_with_more_rows_than_one_cta(play, prefix_kernel):
    """40 members x 4 query heads = 160 rows: two row blocks of the prefix kernel."""
    groups = [(1024, [1024 + 1 + 7 * i for i in range(40)])]
    kw = dict(hq=32, hkv=8, d=128, q_dtype="bf16", cache_dtype="bf16", bs=16, seed=3)
    on, members, rows, q, out_on, scale = _build(play, groups, [], cascade=True, **kw)
    assert on.check() == 0 and on.cascade_count() == 1
    got = to_f64(out_on[0])
    for i in range(0, len(members), 3):
        k, v = rows[i]
        ref = decode_attention(q[0, i].astype(np.float32), k.astype(np.float64), v.astype(np.float64), scale)
        assert_close(got[i], ref, f"member {members[i]}")
    on.close()


def test_short_shared_prefix_stays_plain(play):
    """Fewer than 16 shared tiles: the decode attends everything itself."""
    groups = [(200, [230, 260, 300])]
    kw = dict(hq=32, hkv=8, d=128, q_dtype="bf16", cache_dtype="bf16", bs=16, seed=4)
    on, members, rows, q, out_on, scale = _build(play, groups, [500], cascade=True, **kw)
    assert on.check() == 0 and on.cascade_count() == 0
    on.close()


@pytest.mark.parametrize("prefix_kernel", [("tcgen05", 0), ("mma_sync", 0)], indirect=True, ids=lambda k: k[0])
def test_prefix_share_workload_through_the_step(play, prefix_kernel):
    """The prefix-share workload (32 forks of a 1500-token prefix) steps with the cascade, several steps."""
    w = wl.make(4, extra_steps=4)
    cache, out = play.run(w, out_dtype="f32")
    assert cache.check() == 0 and cache.cascade_count() == 1
    from helpers import oracle_seq_output
    q = w.q_rows(0)
    got = to_f64(out[0])
    for s in (0, 7, 31):
        assert_close(got[s], oracle_seq_output(w, s, q[s]), f"sequence {s}")
    for step in range(1, 3):
        k, v, qs = play.step_inputs(w, step)
        out = cache.step(w.seq_ids, k, v, qs, scale=w.scale, out=torch.empty(qs.shape, device="cuda"))
        qh = w.q_rows(0, step)
        got = to_f64(out[0])
        for s in (3, 30):
            assert_close(got[s], oracle_seq_output(w, s, qh[s], step=step), f"step {step} sequence {s}")
    assert cache.check() == 0 and cache.cascade_count() == 3
    cache.close()
