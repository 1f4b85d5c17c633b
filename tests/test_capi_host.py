"""CPU tests of the C-ABI library: it loads, exports every declared call, and its
host block manager matches the oracle allocator bit for bit.

No compute call is made here (no GPU on this machine); the device calls are
covered by the gpu-marked tests.
"""
import os
import re

import numpy as np
import pytest

from oracle import sizing
from oracle.allocator import AllocatorModel, NoBlocks
from paged_kv_cache_163_gb300 import build, capi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not os.path.exists(capi.LIB_PATH):
        build.build()
    return capi.load()


def header_functions():
    text = open(os.path.join(ROOT, "include", "pkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)) - {"defined"})


def test_exports_every_declared_symbol(lib):
    names = header_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(capi.declared_symbols())


def test_status_strings(lib):
    assert capi.pkv_status_string(0) == "ok"
    assert capi.pkv_status_string(-2) == "out of KV blocks"


class Mirror:
    """Drive the C++ block manager and the oracle allocator with the same calls."""

    def __init__(self, n, order=None, bs=16):
        self.bm = capi.pkv_bm_create(n, bs, order)
        self.model = AllocatorModel(n, bs, order)

    def same_state(self):
        assert list(capi.pkv_bm_free_list(self.bm)) == list(self.model.free)
        assert capi.pkv_bm_num_free(self.bm) == self.model.num_free()
        for b in range(self.model.num_blocks):
            assert capi.pkv_bm_refcount(self.bm, b) == self.model.refcount[b]
        seqs = sorted(self.model.tables)
        if seqs:
            mb = max(1, max(len(t) for t in self.model.tables.values()))
            t, lens = capi.pkv_build_block_tables(self.bm, seqs, mb)
            mt, ml = self.model.block_tables(seqs, mb)
            assert t.tolist() == mt and lens.tolist() == ml


def test_fork_cow_example_matches_oracle():
    m = Mirror(64)
    capi.pkv_seq_create(m.bm, 0); m.model.create(0)
    s1, *_ = capi.pkv_seq_append_slots(m.bm, [0] * 40)
    s2, _ = m.model.append_slots([0] * 40)
    assert s1.tolist() == s2
    for c in (1, 2, 3):
        capi.pkv_seq_fork(m.bm, 0, c); m.model.fork(0, c)
    slots, src, dst = capi.pkv_seq_append_slots(m.bm, [0, 1, 2, 3])
    mslots, mcows = m.model.append_slots([0, 1, 2, 3])
    assert slots.tolist() == mslots
    assert list(zip(src.tolist(), dst.tolist())) == mcows == [(2, 3), (2, 4), (2, 5)]
    m.same_state()


@pytest.mark.parametrize("bs", [16, 32])
def test_random_traces_match_oracle_bit_exact(bs):
    rng = np.random.default_rng(11 + bs)
    for trial in range(25):
        n = int(rng.integers(4, 80))
        order = rng.permutation(n)
        m = Mirror(n, order, bs)
        assert capi.pkv_bm_block_size(m.bm) == bs
        live, nid = [], 0
        for _ in range(150):
            op = int(rng.integers(0, 10))
            if op == 0 or not live:
                capi.pkv_seq_create(m.bm, nid); m.model.create(nid); live.append(nid); nid += 1
            elif op == 1:
                p = live[int(rng.integers(len(live)))]
                capi.pkv_seq_fork(m.bm, p, nid); m.model.fork(p, nid); live.append(nid); nid += 1
            elif op == 2 and len(live) > 1:
                s = live.pop(int(rng.integers(len(live))))
                capi.pkv_seq_free(m.bm, s); m.model.free_seq(s)
            else:
                batch = [live[int(i)] for i in rng.integers(0, len(live), int(rng.integers(1, 40)))]
                try:
                    ms, mc = m.model.append_slots(batch)
                    ok = True
                except NoBlocks:
                    ok = False
                if ok:
                    s, a, b = capi.pkv_seq_append_slots(m.bm, batch)
                    assert s.tolist() == ms and list(zip(a.tolist(), b.tolist())) == mc
                else:
                    with pytest.raises(capi.NoBlocksError):
                        capi.pkv_seq_append_slots(m.bm, batch)
            m.same_state()
        for s in live:
            capi.pkv_seq_free(m.bm, s); m.model.free_seq(s)
        m.same_state()
        assert capi.pkv_bm_num_free(m.bm) == n
        capi.pkv_bm_destroy(m.bm)


def test_no_blocks_changes_nothing():
    m = Mirror(3)
    for s in (0, 1):
        capi.pkv_seq_create(m.bm, s); m.model.create(s)
    capi.pkv_seq_append_slots(m.bm, [0] * 16); m.model.append_slots([0] * 16)
    before = (capi.pkv_bm_free_list(m.bm).tolist(), capi.pkv_seq_len(m.bm, 0), capi.pkv_seq_len(m.bm, 1))
    with pytest.raises(capi.NoBlocksError):
        capi.pkv_seq_append_slots(m.bm, [1] * 16 + [0] * 17 + [1] * 16)
    assert (capi.pkv_bm_free_list(m.bm).tolist(), capi.pkv_seq_len(m.bm, 0), capi.pkv_seq_len(m.bm, 1)) == before
    m.same_state()


def test_invalid_arguments_raise():
    bm = capi.pkv_bm_create(4)
    with pytest.raises(capi.PkvError):
        capi.pkv_seq_append_slots(bm, [7])
    capi.pkv_seq_create(bm, 1)
    with pytest.raises(capi.PkvError):
        capi.pkv_seq_create(bm, 1)
    with pytest.raises(capi.PkvError):
        capi.kv_block_free(bm, 3)
    with pytest.raises(capi.PkvError):
        capi.pkv_bm_create(4, 16, [0, 1, 1, 2])
    with pytest.raises(capi.PkvError):
        capi.pkv_bm_create(4, 24)
    capi.pkv_seq_append_slots(bm, [1] * 40)
    with pytest.raises(capi.PkvError):
        capi.pkv_build_block_tables(bm, [1], 2)
    b = capi.kv_block_alloc(bm)
    assert capi.pkv_bm_refcount(bm, b) == 1
    capi.kv_block_free(bm, b)
    assert capi.pkv_bm_free_list(bm).tolist()[-1] == b
    capi.pkv_bm_destroy(bm)


@pytest.mark.parametrize("bs", [16, 32])
def test_coded_caches_take_one_scale_array(bs):
    """Scales are one array [blocks][heads][2][block_size] (K, then V): v_scale must be k_scale + block_size.

    Stand-in addresses (16-byte aligned, never dereferenced): the call
    rejects the pointers before it touches the device.
    """
    lib = capi.load()
    base = 1 << 24
    k, v, slots, kc, vc, err = base, base + 4096, base + 8192, base + 12288, base + 16384, base + 20480
    ks = base + 65536
    for vs in (ks + 4 * bs * 2, ks + 4 * (bs - 16), ks + 4 * bs * 64, ks):
        st = lib.paged_kv_append(k, v, capi.PKV_BF16, 1, 2, 128, slots, kc, vc, capi.PKV_FP8_E4M3, ks, vs, 4, bs,
                                 err, None)
        assert capi.STATUS[st] == "PKV_ERR_INVALID"
        st = lib.paged_kv_copy_blocks(kc, vc, ks, vs, slots, slots, 1, 2, 128, capi.PKV_INT8, 4, bs, err, None)
        assert capi.STATUS[st] == "PKV_ERR_INVALID"
    st = lib.paged_kv_append(k, v, capi.PKV_BF16, 1, 2, 128, slots, kc, vc, capi.PKV_FP8_E4M3, None, ks + 4 * bs, 4,
                             bs, err, None)
    assert capi.STATUS[st] == "PKV_ERR_INVALID"


def test_workload_allocations_match_oracle():
    from paged_kv_cache_163_gb300 import workloads as wl
    for wid in (1, 2, 4):
        w = wl.make(wid)
        m = Mirror(w.num_blocks, w.alloc_order)
        for op in w.prefill_ops() + [("append", w.seq_ids)]:
            if op[0] == "create":
                capi.pkv_seq_create(m.bm, op[1]); m.model.create(op[1])
            elif op[0] == "fork":
                capi.pkv_seq_fork(m.bm, op[1], op[2]); m.model.fork(op[1], op[2])
            else:
                s, a, b = capi.pkv_seq_append_slots(m.bm, op[1])
                ms, mc = m.model.append_slots(op[1])
                assert s.tolist() == ms and list(zip(a.tolist(), b.tolist())) == mc
        m.same_state()
        if wid == 4:   # 32 sharers of a 12-token partial block: 31 copies, the last writes in place
            cows = []
            # replay to count copies
            mm = AllocatorModel(w.num_blocks, 16, w.alloc_order)
            for op in w.prefill_ops():
                if op[0] == "create":
                    mm.create(op[1])
                elif op[0] == "fork":
                    mm.fork(op[1], op[2])
                else:
                    cows += mm.append_slots(op[1])[1]
            assert len(cows) == 31 and len({c[0] for c in cows}) == 1


def test_sizing_calls_match_oracle():
    for layers, hkv, d, tokens in [(40, 32, 128, 2048), (32, 8, 128, 32768), (1, 2, 64, 100)]:
        assert capi.pkv_kv_bytes(layers, hkv, d, tokens, "f16") == sizing.kv_bytes(layers, hkv, d, tokens, 1, 2)
        assert capi.pkv_kv_bytes(layers, hkv, d, tokens, "fp8_e4m3") == \
            sizing.fp8_bytes_per_token(layers, hkv, d) * tokens
        budget = 80 * 10 ** 9
        assert capi.pkv_kv_bytes(layers, hkv, d, tokens, "fp8_e4m3_int4") == \
            layers * hkv * tokens * sizing.token_head_bytes(d, "fp8_e4m3_int4")
        for dt in ("bf16", "fp8_e4m3", "int8", "fp8_e4m3_int4"):
            assert capi.pkv_pool_blocks(budget, layers, hkv, d, dt) == sizing.pool_blocks(budget, layers, hkv, d, dt)
    assert capi.pkv_kv_bytes(-1, 1, 64, 1, "f16") == -1


def test_kernel_selectors_validate_and_round_trip():
    """The decode- and prefix-kernel selectors refuse unknown values and keep the last valid one."""
    capi.pkv_set_prefix_kernel("tcgen05", 24)
    assert capi.pkv_get_prefix_kernel() == "tcgen05"
    with pytest.raises(capi.PkvError):
        capi.pkv_set_prefix_kernel(7, 0)
    with pytest.raises(capi.PkvError):
        capi.pkv_set_prefix_kernel("mma_sync", -1)
    with pytest.raises(capi.PkvError):
        capi.pkv_set_prefix_kernel("mma_sync", 4097)
    assert capi.pkv_get_prefix_kernel() == "tcgen05"
    capi.pkv_set_prefix_kernel("auto", 0)
    assert capi.pkv_get_prefix_kernel() == "auto"
    with pytest.raises(capi.PkvError):
        capi.pkv_set_decode_kernel(9)
    assert capi.pkv_get_decode_kernel() == "auto"
