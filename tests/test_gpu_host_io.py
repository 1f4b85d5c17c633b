"""Steps whose inputs and output live in page-locked host memory.

``pkv_copy_segments`` copies several tensors in one kernel launch, reading
and writing page-locked host memory in place.  A step given host tensors
moves them with it (one launch each way) and must produce exactly what the
same step on device tensors produces.
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


def test_copy_segments_both_ways(play):
    from paged_kv_cache_163_gb300 import capi
    dev = torch.device("cuda")
    g = torch.Generator().manual_seed(5)
    sizes = [16, 4096, 0, 48, 1 << 20, 32]
    hosts = [torch.randint(0, 255, (n,), generator=g, dtype=torch.uint8).pin_memory() for n in sizes]
    devs = [torch.empty(n, dtype=torch.uint8, device=dev) for n in sizes]
    n0 = capi.pkv_launch_count()
    capi.pkv_copy_segments(list(zip(devs, hosts)), torch.cuda.current_stream().cuda_stream)
    assert capi.pkv_launch_count() - n0 == 1
    back = [torch.zeros(n, dtype=torch.uint8).pin_memory() for n in sizes]
    capi.pkv_copy_segments(list(zip(back, devs)), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    for h, d, b in zip(hosts, devs, back):
        assert torch.equal(d.cpu(), h) and torch.equal(b, h)
    with pytest.raises(capi.PkvError):            # not a multiple of 16 bytes
        capi.pkv_copy_segments([(devs[1][:24], hosts[1][:24])], torch.cuda.current_stream().cuda_stream)
    with pytest.raises(capi.PkvError):            # misaligned
        capi.pkv_copy_segments([(devs[1][8:24], hosts[1][8:24])], torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("cache_dtype,layers", [("bf16", 1), ("fp8_e4m3", 2)])
def test_host_tensors_step_like_device_tensors(play, cache_dtype, layers):
    rng = np.random.default_rng(9)
    lens = rng.integers(100, 900, 6).tolist()
    w = wl.custom(f"hostio-{cache_dtype}", lens=lens, num_q_heads=16, num_kv_heads=4, head_dim=128,
                  q_dtype="bf16", cache_dtype=cache_dtype, num_layers=layers, seed=31, slack=0.5)
    a, b = play.new_cache(w, poison=True), play.new_cache(w, poison=True)
    play.prefill(w, a)
    play.prefill(w, b)
    for step in range(3):
        k, v, q = play.step_inputs(w, step)
        out_d = a.step(w.seq_ids, k, v, q, scale=w.scale)
        out_h = torch.empty(q.shape, dtype=q.dtype).pin_memory()
        b.step(w.seq_ids, k.cpu().pin_memory(), v.cpu().pin_memory(), q.cpu().pin_memory(), scale=w.scale,
               out=out_h)
        torch.cuda.synchronize()
        assert torch.equal(out_d.cpu(), out_h), f"step {step}"
    assert a.check() == 0 and b.check() == 0
    for li in range(layers):
        assert np.array_equal(cache_bits(a.k[li]), cache_bits(b.k[li]))
        assert np.array_equal(cache_bits(a.v[li]), cache_bits(b.v[li]))
    a.close()
    b.close()
