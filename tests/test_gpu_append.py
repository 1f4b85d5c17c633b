"""GPU parity of reshape-and-cache (append) and copy-on-write block copies.

Bit-exact against the oracle: 16-bit caches hold the input bits; coded
caches (FP8 E4M3, FP8 E5M2, INT8, and K FP8 E4M3 with 4-bit V) hold the
oracle's codes and fp32 scales, including exhaustive sweeps over every
code value and every midpoint between two neighbours (round-to-nearest-even
ties), subnormals, +-0 and saturation.
"""
import numpy as np
import pytest

from oracle import fp8
from oracle.cache import CODE_TYPES, PagedCacheModel
from paged_kv_cache_163_gb300 import workloads as wl
from paged_kv_cache_163_gb300.capi import SCALED_CACHES, v_row_elems

from helpers import cache_bits, oracle_bits

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def capi():
    from paged_kv_cache_163_gb300 import capi as c
    c.load()
    return c


def run_append(capi, rows_k, rows_v, slots, num_blocks, hkv, d, in_dtype, cache_dtype):
    from paged_kv_cache_163_gb300.engine import torch_dtype
    dev = torch.device("cuda")
    kc = torch.empty((num_blocks, hkv, 16, d), dtype=torch_dtype(cache_dtype), device=dev)
    vc = torch.empty((num_blocks, hkv, 16, v_row_elems(cache_dtype, d)), dtype=kc.dtype, device=dev)
    kc.view(torch.uint8).fill_(0xFF)
    vc.view(torch.uint8).fill_(0xFF)
    ks = vs = None
    if cache_dtype in SCALED_CACHES:  # one array: a (block, head)'s K scales, then its V scales
        both = torch.full((num_blocks, hkv, 2, 16), float("nan"), device=dev)
        ks, vs = both[:, :, 0], both[:, :, 1]
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    k = torch.from_numpy(rows_k).to(dev).to(torch_dtype(in_dtype))
    v = torch.from_numpy(rows_v).to(dev).to(torch_dtype(in_dtype))
    s = torch.from_numpy(np.asarray(slots, dtype=np.int32)).to(dev)
    capi.paged_kv_append(k, v, s, kc, vc, ks, vs, d_error=err, cache_dtype=cache_dtype)
    flag = capi.pkv_read_device_error(err)
    return kc, vc, ks, vs, flag


def compare_with_oracle(kc, vc, ks, vs, model: PagedCacheModel, cache_dtype):
    filled = model.filled            # [blocks, 16]
    if cache_dtype in SCALED_CACHES:
        for got, want in ((cache_bits(kc), model.k), (cache_bits(vc), model.v)):
            g = got.transpose(0, 2, 1, 3)[filled]      # [n, hkv, d]
            w = want.transpose(0, 2, 1, 3)[filled]
            assert np.array_equal(g, w), f"{np.sum(g != w)} codes differ"
        for got, want in ((ks, model.k_scale), (vs, model.v_scale)):
            g = got.cpu().numpy().transpose(0, 2, 1)[filled]
            w = want.transpose(0, 2, 1)[filled]
            assert np.array_equal(g.view(np.uint32), w.view(np.uint32))
    else:
        for got, want in ((cache_bits(kc), model.k), (cache_bits(vc), model.v)):
            g = got.transpose(0, 2, 1, 3)[filled]
            w = oracle_bits(want.transpose(0, 2, 1, 3)[filled], cache_dtype)
            assert np.array_equal(g, w)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("in_dtype,cache_dtype", [("f16", "f16"), ("bf16", "bf16"),
                                                  ("bf16", "fp8_e4m3"), ("f16", "fp8_e4m3"),
                                                  ("bf16", "fp8_e5m2"), ("f16", "fp8_e5m2"),
                                                  ("bf16", "int8"), ("f16", "int8"),
                                                  ("bf16", "fp8_e4m3_int4"), ("f16", "fp8_e4m3_int4")])
def test_append_random_rows_bit_exact(capi, d, in_dtype, cache_dtype):
    rng = np.random.default_rng(d + len(cache_dtype))
    nb, hkv, t = 37, 4, 300
    x = rng.standard_normal((2, t, hkv, d)).astype(np.float32)
    x *= rng.uniform(1e-3, 30, (2, t, hkv, 1)).astype(np.float32)
    x[:, ::17] *= 20                      # outlier tokens
    x[:, 5, 1] = 0.0                      # an all-zero row
    x[:, 6, 2] = -0.0
    x = wl.round_to(x, in_dtype)
    slots = rng.permutation(nb * 16)[:t].astype(np.int32)
    slots[::23] = -1                      # skipped tokens
    kc, vc, ks, vs, flag = run_append(capi, x[0], x[1], slots, nb, hkv, d, in_dtype, cache_dtype)
    assert flag == 0
    model = PagedCacheModel(nb, hkv, d, cache_dtype)
    model.write(slots, x[0], x[1])
    compare_with_oracle(kc, vc, ks, vs, model, cache_dtype)
    # slots never written keep their poison bytes
    untouched = ~model.filled
    raw = kc.view(torch.uint8).cpu().numpy().reshape(nb, hkv, 16, -1).transpose(0, 2, 1, 3)[untouched]
    assert np.all(raw == 0xFF)


@pytest.mark.parametrize("in_dtype", ["bf16", "f16"])
def test_fp8_grid_and_midpoint_sweep(capi, in_dtype):
    """Rows whose amax is 448 (scale exactly 1): every E4M3 value and every tie."""
    grid = fp8.decode_table()[:0x7F]                      # 0 .. 448
    mids = (grid[:-1] + grid[1:]) / 2
    vals = np.concatenate([grid, mids, -grid, -mids, [2.0 ** -11, 3 * 2.0 ** -11, -0.0]])
    vals = vals[np.abs(vals) <= 448]
    if in_dtype == "f16":                                 # keep values f16 can hold exactly
        vals = vals[(vals == 0) | (np.abs(vals) >= 2.0 ** -24)]
    d = 128
    per = d - 1
    n = -(-len(vals) // per)
    rows = np.zeros((n, per), dtype=np.float64)
    rows.flat[:len(vals)] = vals
    rows = np.concatenate([np.full((n, 1), 448.0), rows], axis=1).astype(np.float32)
    assert np.array_equal(wl.round_to(rows, in_dtype), rows)
    x = rows[:, None, :]                                  # [n, 1 head, d]
    slots = np.arange(n, dtype=np.int32)
    nb = -(-n // 16)
    kc, vc, ks, vs, flag = run_append(capi, x, -x, slots, nb, 1, d, in_dtype, "fp8_e4m3")
    assert flag == 0
    model = PagedCacheModel(nb, 1, d, "fp8_e4m3")
    model.write(slots, x, -x)
    assert np.all(model.k_scale.reshape(-1)[:n] == 1.0)
    compare_with_oracle(kc, vc, ks, vs, model, "fp8_e4m3")


def _grid_rows(vals, top, d=128):
    """Rows of d values whose first element is `top` (so amax = top and the scale is exactly 1)."""
    per = d - 1
    n = -(-len(vals) // per)
    rows = np.zeros((n, per), dtype=np.float64)
    rows.flat[:len(vals)] = vals
    return np.concatenate([np.full((n, 1), top), rows], axis=1).astype(np.float32)


@pytest.mark.parametrize("in_dtype", ["bf16", "f16"])
@pytest.mark.parametrize("cache_dtype", ["fp8_e5m2", "int8"])
def test_onebyte_grid_and_midpoint_sweep(capi, in_dtype, cache_dtype):
    """Rows whose amax is the format's largest value R (scale exactly 1): every value and every tie."""
    if cache_dtype == "fp8_e5m2":
        grid = fp8.e5m2_decode_table()[:0x7C]             # 0 .. 57344
        extra = [2.0 ** -17, 3 * 2.0 ** -17]
    else:
        grid = np.arange(128, dtype=np.float64)            # 0 .. 127
        extra = [0.49, 0.51]
    top = CODE_TYPES[cache_dtype][0]
    mids = (grid[:-1] + grid[1:]) / 2
    vals = np.concatenate([grid, mids, -grid, -mids, extra, [-0.0]])
    vals = vals[np.abs(vals) <= top]
    rows = _grid_rows(vals, top)
    keep = np.array_equal(wl.round_to(rows, in_dtype), rows)
    if not keep:                                          # drop what the input type cannot hold
        ok = wl.round_to(vals.astype(np.float32), in_dtype) == vals
        rows = _grid_rows(vals[ok], top)
    assert np.array_equal(wl.round_to(rows, in_dtype), rows)
    x = rows[:, None, :]
    n = x.shape[0]
    slots = np.arange(n, dtype=np.int32)
    nb = -(-n // 16)
    kc, vc, ks, vs, flag = run_append(capi, x, -x, slots, nb, 1, 128, in_dtype, cache_dtype)
    assert flag == 0
    model = PagedCacheModel(nb, 1, 128, cache_dtype)
    model.write(slots, x, -x)
    assert np.all(model.k_scale.reshape(-1)[:n] == 1.0)
    compare_with_oracle(kc, vc, ks, vs, model, cache_dtype)


@pytest.mark.parametrize("cache_dtype", ["fp8_e5m2", "int8"])
def test_onebyte_scale_ties(capi, cache_dtype):
    """Rows of code values times amax / R: quotients land on or next to code values after a real division."""
    rng = np.random.default_rng(7)
    d, hkv, t = 128, 2, 512
    r, _, dec = CODE_TYPES[cache_dtype]
    amax = wl.round_to(rng.uniform(1e-6, 1e4, (t, hkv)).astype(np.float32), "bf16")
    if cache_dtype == "fp8_e5m2":
        codes = rng.integers(0, 0x7C, (t, hkv, d))
        base = fp8.e5m2_decode_table()[codes] / r
    else:
        base = (rng.integers(-127, 128, (t, hkv, d)) + rng.choice([0.0, 0.5], (t, hkv, d))) / r
    x = wl.round_to((base * amax[..., None]).astype(np.float32), "bf16")
    x[..., 0] = amax
    slots = rng.permutation(64 * 16)[:t].astype(np.int32)
    kc, vc, ks, vs, flag = run_append(capi, x, x[::-1].copy(), slots, 64, hkv, d, "bf16", cache_dtype)
    assert flag == 0
    model = PagedCacheModel(64, hkv, d, cache_dtype)
    model.write(slots, x, x[::-1].copy())
    compare_with_oracle(kc, vc, ks, vs, model, cache_dtype)


@pytest.mark.parametrize("in_dtype", ["bf16", "f16"])
def test_int4_grid_and_midpoint_sweep(capi, in_dtype):
    """4-bit V rows whose amax is 7 (scale exactly 1): every code, every tie, values near ties."""
    grid = np.arange(8, dtype=np.float64)                 # 0 .. 7
    mids = grid[:-1] + 0.5
    near = np.concatenate([mids - 2.0 ** -4, mids + 2.0 ** -4])
    vals = np.concatenate([grid, mids, near, -grid, -mids, -near, [-0.0]])
    rows = np.tile(_grid_rows(vals, 7.0), (3, 1))         # several rows: both nibbles see every value
    rows[1] = np.roll(rows[1], 1)
    rows[2] = rows[2][::-1]
    assert np.array_equal(wl.round_to(rows, in_dtype), rows)
    x = rows[:, None, :]
    n = x.shape[0]
    slots = np.arange(n, dtype=np.int32)
    kc, vc, ks, vs, flag = run_append(capi, x, x, slots, 1, 1, 128, in_dtype, "fp8_e4m3_int4")
    assert flag == 0
    model = PagedCacheModel(1, 1, 128, "fp8_e4m3_int4")
    model.write(slots, x, x)
    assert np.all(model.v_scale.reshape(-1)[:n] == 1.0)
    compare_with_oracle(kc, vc, ks, vs, model, "fp8_e4m3_int4")


def test_int4_scale_ties(capi):
    """4-bit V rows of half-integers times amax / 7: quotients land on or next to ties after a real division."""
    rng = np.random.default_rng(8)
    d, hkv, t = 128, 2, 512
    amax = wl.round_to(rng.uniform(1e-6, 1e4, (t, hkv)).astype(np.float32), "bf16")
    base = (rng.integers(-7, 8, (t, hkv, d)) + rng.choice([0.0, 0.5], (t, hkv, d))) / 7.0
    x = wl.round_to((np.clip(base, -1, 1) * amax[..., None]).astype(np.float32), "bf16")
    x[..., 0] = amax
    slots = rng.permutation(64 * 16)[:t].astype(np.int32)
    kc, vc, ks, vs, flag = run_append(capi, x[::-1].copy(), x, slots, 64, hkv, d, "bf16", "fp8_e4m3_int4")
    assert flag == 0
    model = PagedCacheModel(64, hkv, d, "fp8_e4m3_int4")
    model.write(slots, x[::-1].copy(), x)
    compare_with_oracle(kc, vc, ks, vs, model, "fp8_e4m3_int4")


def test_fp8_scale_ties_and_tiny_rows(capi):
    """Rows whose amax makes x / s land on ties and subnormals after a real division."""
    rng = np.random.default_rng(5)
    d, hkv, t = 128, 2, 512
    amax = wl.round_to(rng.uniform(1e-6, 1e4, (t, hkv)).astype(np.float32), "bf16")
    codes = rng.integers(0, 0x7F, (t, hkv, d))
    base = fp8.decode_table()[codes] / 448.0              # grid points scaled by amax / 448
    x = wl.round_to((base * amax[..., None]).astype(np.float32), "bf16")
    x[..., 0] = amax
    x[..., 1::2] *= -1
    slots = rng.permutation(64 * 16)[:t].astype(np.int32)
    kc, vc, ks, vs, flag = run_append(capi, x, x[::-1].copy(), slots, 64, hkv, d, "bf16", "fp8_e4m3")
    assert flag == 0
    model = PagedCacheModel(64, hkv, d, "fp8_e4m3")
    model.write(slots, x, x[::-1].copy())
    compare_with_oracle(kc, vc, ks, vs, model, "fp8_e4m3")


def test_bad_slot_sets_flag_and_skips(capi):
    x = np.ones((3, 2, 64), dtype=np.float32)
    kc, vc, ks, vs, flag = run_append(capi, x, x, [0, 5 * 16, 17], 4, 2, 64, "bf16", "bf16")
    assert flag & capi.DEVERR_BAD_SLOT
    raw = cache_bits(kc)
    assert np.all(raw[0, :, 0] == 0x3F80) and np.all(raw[1, :, 1] == 0x3F80)


@pytest.mark.parametrize("cache_dtype,d", [("bf16", 128), ("f16", 64), ("fp8_e4m3", 128),
                                           ("fp8_e4m3_int4", 128), ("fp8_e4m3_int4", 64)])
def test_copy_blocks(capi, cache_dtype, d):
    from paged_kv_cache_163_gb300.engine import torch_dtype
    dev = torch.device("cuda")
    nb, hkv = 20, 8
    g = torch.Generator(device="cpu").manual_seed(3)
    kbytes = d * (1 if cache_dtype in SCALED_CACHES else 2)
    vbytes = d // 2 if cache_dtype == "fp8_e4m3_int4" else kbytes
    kc = torch.randint(0, 255, (nb, hkv, 16, kbytes), generator=g, dtype=torch.uint8).to(dev)
    vc = torch.randint(0, 255, (nb, hkv, 16, vbytes), generator=g, dtype=torch.uint8).to(dev)
    kc_t, vc_t = kc.view(torch_dtype(cache_dtype)), vc.view(torch_dtype(cache_dtype))
    ks = vs = None
    if cache_dtype in SCALED_CACHES:
        both = torch.rand((nb, hkv, 2, 16), generator=g).to(dev)
        ks, vs = both[:, :, 0], both[:, :, 1]
    before = [t.clone() if t is not None else None for t in (kc, vc, ks, vs)]
    src = torch.tensor([3, 7, 11], dtype=torch.int32, device=dev)
    dst = torch.tensor([15, 0, 19], dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    capi.paged_kv_copy_blocks(kc_t, vc_t, ks, vs, src, dst, d_error=err, cache_dtype=cache_dtype)
    assert capi.pkv_read_device_error(err) == 0
    for now, old in zip((kc, vc, ks, vs), before):
        if now is None:
            continue
        exp = old.clone()
        exp[dst.long()] = old[src.long()]
        assert torch.equal(now, exp)
    bad = torch.tensor([25], dtype=torch.int32, device=dev)
    capi.paged_kv_copy_blocks(kc_t, vc_t, ks, vs, bad, src[:1], d_error=err, cache_dtype=cache_dtype)
    assert capi.pkv_read_device_error(err) & capi.DEVERR_BAD_BLOCK
