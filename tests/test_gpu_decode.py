"""GPU parity of paged decode attention against the fp64 oracle.

Every workload runs through the C ABI exactly as the benchmark does (host
block manager -> append -> decode).  Integer results (block tables, slot
mappings, copy-on-write pairs, cache bytes) must be bit-exact; attention
outputs must satisfy max |err| <= 1e-2 and relative L2 <= 2e-3.

Every workload compares every output and every filled cache slot: the
16 x 16K-32K FP8 one too, with the oracle's quantisation and attention of
its sequences computed once, in a pool of spawned processes.  Workloads
without outliers also compare the 16-bit output with the oracle directly.
"""
import numpy as np
import pytest

from oracle.allocator import AllocatorModel
from paged_kv_cache_163_gb300.capi import SCALED_CACHES
from paged_kv_cache_163_gb300 import workloads as wl

from helpers import (assert_close, cache_bits, check_rounding, coded_seq_reference, oracle_bits, oracle_play,
                     oracle_seq_output, parallel_map, to_f64)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def play():
    from paged_kv_cache_163_gb300 import capi, play as p
    capi.load()
    return p


@pytest.fixture
def kernel_kind(request):
    """Run a test under one decode kernel variant, then restore the default."""
    from paged_kv_cache_163_gb300 import capi
    capi.pkv_set_decode_kernel(request.param)
    yield request.param
    capi.pkv_set_decode_kernel("auto")


def check_tables(cache, o, seqs):
    t, lens = cache.tables(seqs)
    mt, ml = o.alloc.block_tables(seqs, t.shape[1])
    assert t.tolist() == mt and lens.tolist() == ml


def check_cache_bytes(cache, o, w, layer=0):
    model = o.layers[0]
    filled = model.filled
    if w.cache_dtype in SCALED_CACHES:
        for got, want in ((cache.k[layer], model.k), (cache.v[layer], model.v)):
            g = cache_bits(got).transpose(0, 2, 1, 3)[filled]
            assert np.array_equal(g, want.transpose(0, 2, 1, 3)[filled])
        for got, want in ((cache.k_scale[layer], model.k_scale), (cache.v_scale[layer], model.v_scale)):
            g = got.cpu().numpy().transpose(0, 2, 1)[filled]
            assert np.array_equal(g, want.transpose(0, 2, 1)[filled])
    else:
        for got, want in ((cache.k[layer], model.k), (cache.v[layer], model.v)):
            g = cache_bits(got).transpose(0, 2, 1, 3)[filled]
            assert np.array_equal(g, oracle_bits(want.transpose(0, 2, 1, 3)[filled], w.cache_dtype))


def full_oracle_check(play, w, layers=1):
    # without the cascade: the 16-bit check below decodes again by the public call, which must
    # sum in the same order (the cascade has its own tests)
    cache, out = play.run(w, poison=True, out_dtype="f32", cascade=False)
    assert cache.check() == 0
    o = oracle_play(w, layers=1)
    check_tables(cache, o, w.seq_ids)
    assert cache.cow_pairs == o.cow_log
    check_cache_bytes(cache, o, w)
    res, refs = [], []
    for li in range(layers):
        ref = o.decode(w.seq_ids, w.q_rows(li), w.scale)
        refs.append(ref)
        res.append(assert_close(to_f64(out[li]), ref, f"{w.name} layer {li}"))
    out16 = check_rounding(cache, w, out)
    if w.outlier_p == 0:
        # no x20 outliers: the rounded 16-bit output itself stays inside the tolerance
        for li in range(layers):
            assert_close(to_f64(out16[li]), refs[li], f"{w.name} layer {li}, {w.q_dtype} output")
    assert cache.check() == 0
    cache.close()
    return res


def test_tiny_gqa_fp16(play):
    full_oracle_check(play, wl.make(1))


@pytest.mark.parametrize("kernel_kind", ["simt", "mma"], indirect=True)
def test_llama3_8b_shape_bf16(play, kernel_kind):
    full_oracle_check(play, wl.make(2))


@pytest.mark.parametrize("kernel_kind", ["simt", "mma"], indirect=True)
def test_prefix_sharing_bf16(play, kernel_kind):
    w = wl.make(4)
    full_oracle_check(play, w)


@pytest.mark.parametrize("kernel_kind", ["simt", "mma"], indirect=True)
def test_mha_40_layers_fp16(play, kernel_kind):
    w = wl.make(3)
    cache, out = play.run(w, poison=False, out_dtype="f32")
    assert cache.check() == 0
    # tables: logical block j of sequence b is physical j * 8 + b
    t, lens = cache.tables(w.seq_ids)
    assert np.array_equal(t, np.arange(128)[None, :] * 8 + np.arange(8)[:, None])
    assert np.all(lens == 2048)
    # all 40 layers hold the same K/V rows; queries differ per layer
    K = [wl.round_to(w.kv_rows(0, s, 0, 2048), "f16").astype(np.float64) for s in range(8)]
    V = [wl.round_to(w.kv_rows(1, s, 0, 2048), "f16").astype(np.float64) for s in range(8)]
    from oracle.attention import decode_attention
    refs = {}
    for li in range(0, 40, 3):
        q = w.q_rows(li)
        refs[li] = np.stack([decode_attention(q[s], K[s], V[s], w.scale) for s in range(8)])
        assert_close(to_f64(out[li]), refs[li], f"layer {li}")
    # cache bytes of sampled layers equal the input rows
    for li in (0, 39):
        got = cache_bits(cache.k[li])[t[3]]                     # [128, 32, 16, 128] of sequence 3
        want = oracle_bits(K[3].reshape(128, 16, 32, 128).transpose(0, 2, 1, 3), "f16")
        assert np.array_equal(got, want)
    out16 = check_rounding(cache, w, out, layers=[0, 18, 39])
    for li in (0, 18, 39):
        assert_close(to_f64(out16[li]), refs[li], f"layer {li}, fp16 output")
    cache.close()


@pytest.fixture(scope="module")
def long_fp8_reference():
    """Oracle codes, scales and fp64 outputs of every sequence of the 16 x 16K-32K FP8 workload."""
    w = wl.make(5)
    return {r[0]: r[1:] for r in parallel_map(coded_seq_reference, [(5, None, s) for s in range(w.num_seqs)])}


def gathered(t, table_row, n_blocks, length):
    """A sequence's rows of a paged pool [blocks, Hkv, bs, ...] -> [length, Hkv, ...] (host)."""
    idx = torch.as_tensor(np.asarray(table_row[:n_blocks], dtype=np.int64), device=t.device)
    g = t.index_select(0, idx).cpu().numpy()                  # [nb, Hkv, bs, ...]
    g = np.swapaxes(g, 1, 2)                                  # [nb, bs, Hkv, ...]
    return g.reshape((-1,) + g.shape[2:])[:length]


@pytest.mark.parametrize("kernel_kind", ["simt", "mma"], indirect=True)
def test_long_context_fp8_every_sequence(play, kernel_kind, long_fp8_reference):
    w = wl.make(5)
    cache, out = play.run(w, poison=False, out_dtype="f32")
    assert cache.check() == 0
    # tables bit-exact against the oracle allocator
    model = AllocatorModel(w.num_blocks, 16, w.alloc_order)
    for op in w.prefill_ops() + [("append", w.seq_ids)]:
        if op[0] == "create":
            model.create(op[1])
        else:
            model.append_slots(op[1])
    t, lens = cache.tables(w.seq_ids)
    mt, ml = model.block_tables(w.seq_ids, t.shape[1])
    assert t.tolist() == mt and lens.tolist() == ml
    got = to_f64(out[0])
    for s in range(w.num_seqs):
        kc, ks, vc, vs, ref = long_fp8_reference[s]
        assert_close(got[s], ref, f"sequence {s}")
        # every filled slot: codes and scales equal the oracle's quantisation of the rows
        L = int(lens[s])
        nb = -(-L // 16)
        assert np.array_equal(gathered(cache.k[0], t[s], nb, L), kc), f"K codes of sequence {s}"
        assert np.array_equal(gathered(cache.v[0], t[s], nb, L), vc), f"V codes of sequence {s}"
        assert np.array_equal(gathered(cache.k_scale[0], t[s], nb, L), ks), f"K scales of sequence {s}"
        assert np.array_equal(gathered(cache.v_scale[0], t[s], nb, L), vs), f"V scales of sequence {s}"
    check_rounding(cache, w, out)
    cache.close()


@pytest.mark.parametrize("kernel_kind", ["simt", "mma"], indirect=True)
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("group", [1, 2, 4, 8])
@pytest.mark.parametrize("q_dtype,cache_dtype", [("f16", "f16"), ("bf16", "bf16"),
                                                 ("bf16", "fp8_e4m3"), ("f16", "fp8_e4m3"),
                                                 ("bf16", "fp8_e5m2"), ("f16", "fp8_e5m2"),
                                                 ("bf16", "int8"), ("f16", "int8"),
                                                 ("bf16", "fp8_e4m3_int4"), ("f16", "fp8_e4m3_int4")])
def test_every_instance_ragged(play, kernel_kind, d, group, q_dtype, cache_dtype):
    hkv = 2
    lens = [1, 15, 16, 17, 31, 33, 200, 777, 2]
    w = wl.custom(f"inst-{d}-{group}-{cache_dtype}", lens=lens, num_q_heads=hkv * group, num_kv_heads=hkv,
                  head_dim=d, q_dtype=q_dtype, cache_dtype=cache_dtype, outlier_p=0.002,
                  seed=d * 10 + group)
    full_oracle_check(play, w)


@pytest.mark.parametrize("kernel_kind", ["simt", "mma"], indirect=True)
def test_one_long_sequence_among_short(play, kernel_kind):
    # one sequence holds most tiles: its (sequence, head) pairs are split across many warps
    lens = [40000, 3, 16, 1, 100]
    w = wl.custom("split-heavy", lens=lens, num_q_heads=32, num_kv_heads=8, head_dim=128,
                  q_dtype="bf16", cache_dtype="bf16", seed=9)
    cache, out = play.run(w, out_dtype="f32")
    assert cache.check() == 0
    q = w.q_rows(0)
    got = to_f64(out[0])
    for s in range(len(lens)):
        assert_close(got[s], oracle_seq_output(w, s, q[s]), f"sequence {s}")
    cache.close()


def test_max_batch_short_contexts(play):
    lens = (np.arange(1024) % 70) + 1
    w = wl.custom("max-batch", lens=lens, num_q_heads=8, num_kv_heads=2, head_dim=64, q_dtype="f16",
                  cache_dtype="f16", seed=12)
    cache, out = play.run(w, out_dtype="f32")
    assert cache.check() == 0
    q = w.q_rows(0)
    got = to_f64(out[0])
    for s in range(0, 1024, 37):
        assert_close(got[s], oracle_seq_output(w, s, q[s]), f"sequence {s}")
    cache.close()


def test_empty_context_and_empty_batch(play):
    from paged_kv_cache_163_gb300 import capi
    w = wl.custom("with-empty", lens=[5, 40], num_q_heads=8, num_kv_heads=2, head_dim=128,
                  q_dtype="bf16", cache_dtype="bf16", seed=4)
    cache = play.new_cache(w, poison=True)
    play.prefill(w, cache)
    cache.create(99)                                  # a sequence with no tokens
    q = play.to_device(np.stack([w.q_rows(0)[0], w.q_rows(0)[1], w.q_rows(0)[0]]), "bf16", "cuda")
    out = cache.decode([0, 1, 99], q, scale=w.scale, out=torch.empty(q.shape, device="cuda"))
    assert cache.check() == 0
    got = to_f64(out)
    assert np.all(got[2] == 0.0)
    for i, s in enumerate([0, 1]):
        L = w.context_lens[s] - 1                     # pre-fill only: no decode-step append here
        from oracle.attention import decode_attention
        from oracle.cache import dequantize_rows
        K = dequantize_rows(w.kv_rows(0, s, 0, L), "bf16")
        V = dequantize_rows(w.kv_rows(1, s, 0, L), "bf16")
        assert_close(got[i], decode_attention(q[i].float().cpu().numpy(), K, V, w.scale))
    # an empty batch is a no-op
    capi.paged_attention_decode(out[:0], q[:0], cache.k[0], cache.v[0], None, None,
                                torch.zeros((0, 1), dtype=torch.int32, device="cuda"),
                                torch.zeros(0, dtype=torch.int32, device="cuda"), 0, w.scale,
                                cache.workspace(3, 8, "bf16"), num_seqs=0)
    cache.close()


def test_multi_step_decode_matches_oracle(play):
    w = wl.make(2, extra_steps=4, num_seqs=6)
    cache, out = play.run(w)
    for step in range(1, 4):
        k, v, q = play.step_inputs(w, step)
        out = cache.step(w.seq_ids, k, v, q, scale=w.scale, out=torch.empty(q.shape, device="cuda"))
        qh = w.q_rows(0, step)
        got = to_f64(out[0])
        for s in range(w.num_seqs):
            assert_close(got[s], oracle_seq_output(w, s, qh[s], step=step), f"step {step} seq {s}")
    assert cache.check() == 0
    cache.close()


def test_copy_on_write_inside_the_step(play):
    # every sequence's first own token lands in the shared 12-token partial block during the step
    w = wl.custom("cow-step", lens=[1501] * 6, num_q_heads=32, num_kv_heads=8, head_dim=128, q_dtype="bf16",
                  cache_dtype="bf16", prefix_len=1500, seed=31)
    full_oracle_check(play, w)


def test_stepper_rejects_bad_batches_without_changes(play):
    from paged_kv_cache_163_gb300 import capi
    w = wl.custom("tight", lens=[16, 16], num_q_heads=8, num_kv_heads=2, head_dim=64, q_dtype="f16",
                  cache_dtype="f16", seed=5, slack=0.0)
    cache, _ = play.run(w)                    # 2 sequences of 16 tokens fill the 2-block pool
    assert capi.pkv_bm_num_free(cache.bm) == 0
    k, v, q = play.step_inputs(w, 1)
    before = [cache.seq_len(s) for s in w.seq_ids]
    with pytest.raises(capi.NoBlocksError):   # the 17th tokens need new blocks
        cache.step(w.seq_ids, k, v, q, scale=w.scale)
    assert [cache.seq_len(s) for s in w.seq_ids] == before
    with pytest.raises(capi.PkvError):
        cache.step([0, 0], k, v, q, scale=w.scale)
    assert [cache.seq_len(s) for s in w.seq_ids] == before
    assert cache.check() == 0
    cache.close()


@pytest.mark.parametrize("kernel_kind", ["simt", "mma"], indirect=True)
def test_more_warps_than_tiles(play, kernel_kind):
    # the grid is sized from the longest context, so one long sequence among many
    # one-token ones leaves some warps without a tile (and items split across few)
    lens = [3000] + [1] * 40 + [17] * 23
    w = wl.custom("sparse", lens=lens, num_q_heads=4, num_kv_heads=2, head_dim=128, q_dtype="bf16",
                  cache_dtype="bf16", seed=41)
    cache, out = play.run(w, out_dtype="f32")
    assert cache.check() == 0
    q = w.q_rows(0)
    got = to_f64(out[0])
    for s in (0, 1, 20, 41, 63):
        assert_close(got[s], oracle_seq_output(w, s, q[s]), f"sequence {s}")
    cache.close()


@pytest.mark.parametrize("kernel_kind", ["simt", "mma"], indirect=True)
def test_repeated_calls_reuse_the_workspace(play, kernel_kind):
    # split items are merged through per-item counters kept in the workspace across calls
    w = wl.make(2, num_seqs=8)
    cache, out = play.run(w, out_dtype="f32")
    q = play.to_device(w.q_rows(0), w.q_dtype, "cuda")
    first = cache.decode(w.seq_ids, q, scale=w.scale, out=torch.empty(q.shape, device="cuda"))
    for _ in range(5):
        again = cache.decode(w.seq_ids, q, scale=w.scale, out=torch.empty(q.shape, device="cuda"))
        assert torch.equal(first, again)
    assert torch.equal(first, out[0])
    assert cache.check() == 0
    cache.close()


@pytest.mark.parametrize("kernel_kind", ["simt", "mma"], indirect=True)
@pytest.mark.parametrize("q_dtype,cache_dtype,d", [("bf16", "bf16", 128), ("f16", "f16", 64),
                                                   ("bf16", "fp8_e4m3", 128), ("f16", "int8", 128),
                                                   ("bf16", "fp8_e4m3_int4", 128), ("f16", "fp8_e4m3_int4", 64)])
def test_block_size_32(play, kernel_kind, q_dtype, cache_dtype, d):
    """32-token blocks: two 16-token tiles per block; a shared prefix with copy-on-write in the step."""
    prefix = 70                              # two full 32-token blocks + 6 tokens: the partial block is shared
    lens = [prefix + s for s in (1, 2, 31, 32, 33, 100, 500)]
    w = wl.custom(f"bs32-{cache_dtype}-{d}", lens=lens, num_q_heads=4 * 2, num_kv_heads=2, head_dim=d,
                  q_dtype=q_dtype, cache_dtype=cache_dtype, prefix_len=prefix, outlier_p=0.003, seed=55,
                  block_size=32)
    full_oracle_check(play, w)


@pytest.mark.parametrize("kernel_kind", ["simt", "mma"], indirect=True)
def test_block_size_32_ragged_no_sharing(play, kernel_kind):
    lens = [1, 15, 16, 17, 31, 32, 33, 63, 64, 65, 1000, 2]
    w = wl.custom("bs32-ragged", lens=lens, num_q_heads=32, num_kv_heads=8, head_dim=128, q_dtype="bf16",
                  cache_dtype="bf16", seed=56, block_size=32)
    full_oracle_check(play, w)
