"""Steps whose inputs and output live in page-locked host memory.

``pkv_copy_segments`` copies several tensors in one kernel launch, reading
and writing page-locked host memory in place.  A step given host tensors
registers its input copies with the step executor
(``pkv_stepper_copy_inputs``), which launches them after its host work and
right before the attention; the step must produce exactly what the same
step on device tensors produces, also when copy-on-write copies come first.
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


@pytest.mark.parametrize("cache_dtype,layers,prefix", [("bf16", 1, 0), ("fp8_e4m3", 2, 0), ("bf16", 1, 300),
                                                        ("fp8_e4m3", 1, 300)])
def test_host_tensors_step_like_device_tensors(play, cache_dtype, layers, prefix):
    rng = np.random.default_rng(9)
    lens = rng.integers(100, 900, 6).tolist()
    if prefix:  # forks of a 300-token prefix: the first step copies the shared partial block first
        lens = [prefix + 1 + int(x) % 200 for x in lens]
    w = wl.custom(f"hostio-{cache_dtype}", lens=lens, num_q_heads=16, num_kv_heads=4, head_dim=128,
                  q_dtype="bf16", cache_dtype=cache_dtype, num_layers=layers, seed=31, slack=0.5,
                  prefix_len=prefix)
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
    if prefix:
        assert len(a.cow_pairs) > 0 and a.cow_pairs == b.cow_pairs
    assert a.check() == 0 and b.check() == 0
    for li in range(layers):
        assert np.array_equal(cache_bits(a.k[li]), cache_bits(b.k[li]))
        assert np.array_equal(cache_bits(a.v[li]), cache_bits(b.v[li]))
    a.close()
    b.close()


def test_registered_input_copies_rules(play):
    """pkv_stepper_copy_inputs validates like pkv_copy_segments; a step that fails drops its registration."""
    from paged_kv_cache_163_gb300 import capi
    w = wl.custom("hostio-rules", lens=[40, 70], num_q_heads=8, num_kv_heads=2, head_dim=128, q_dtype="bf16",
                  cache_dtype="bf16", seed=33, slack=0.0)
    cache = play.new_cache(w)
    play.prefill(w, cache)
    k, v, q = play.step_inputs(w, 0)
    cache.step(w.seq_ids, k, v, q, scale=w.scale)          # creates the step executor
    st = cache._stepper
    dev = torch.empty(64, dtype=torch.uint8, device="cuda")
    host = torch.zeros(64, dtype=torch.uint8).pin_memory()
    with pytest.raises(capi.PkvError):                     # not a multiple of 16 bytes
        capi.pkv_stepper_copy_inputs(st, [(dev[:24], host[:24])])
    with pytest.raises(capi.PkvError):                     # misaligned
        capi.pkv_stepper_copy_inputs(st, [(dev[8:24], host[8:24])])
    with pytest.raises(capi.PkvError):                     # too many segments
        capi.pkv_stepper_copy_inputs(st, [(dev[:16], host[:16])] * 9)
    # a registration the next step consumes: one more launch than a plain step
    k, v, q = play.step_inputs(w, 1)
    n0 = capi.pkv_launch_count()
    cache.step(w.seq_ids, k, v, q, scale=w.scale)
    plain = capi.pkv_launch_count() - n0
    capi.pkv_stepper_copy_inputs(st, [(dev[:16], host[:16])])
    k, v, q = play.step_inputs(w, 2)
    n0 = capi.pkv_launch_count()
    cache.step(w.seq_ids, k, v, q, scale=w.scale)
    assert capi.pkv_launch_count() - n0 == plain + 1
    # a step that fails before launching (a sequence twice) drops it: the next step launches as usual
    capi.pkv_stepper_copy_inputs(st, [(dev[:16], host[:16])])
    with pytest.raises(capi.PkvError):
        cache.step([w.seq_ids[0], w.seq_ids[0]], k[:2], v[:2], q[:, :2], scale=w.scale)
    k, v, q = play.step_inputs(w, 3)
    n0 = capi.pkv_launch_count()
    cache.step(w.seq_ids, k, v, q, scale=w.scale)
    assert capi.pkv_launch_count() - n0 == plain
    torch.cuda.synchronize()
    assert cache.check() == 0
    cache.close()


def test_host_tensors_with_graph_replay(play):
    """Host-buffer steps replayed from CUDA graphs (the input copy launched before the graph) equal device steps.

    Graph steps widen the tables to a power of two, which sets the grid from a
    larger context bound; the lengths here are large enough that both kinds
    of step run a full wave, so the work split (and the sum order) is the same.
    """
    rng = np.random.default_rng(12)
    lens = rng.integers(2500, 3000, 8).tolist()
    w = wl.custom("hostio-graph", lens=lens, num_q_heads=32, num_kv_heads=8, head_dim=128, q_dtype="bf16",
                  cache_dtype="fp8_e4m3", num_layers=2, seed=35, slack=0.5)
    a, b = play.new_cache(w), play.new_cache(w)
    play.prefill(w, a)
    play.prefill(w, b)
    b.use_graphs(True)
    out_h = None
    for step in range(4):
        k, v, q = play.step_inputs(w, step)
        out_d = a.step(w.seq_ids, k, v, q, scale=w.scale)
        if out_h is None:
            out_h = torch.empty(q.shape, dtype=q.dtype).pin_memory()
        b.step(w.seq_ids, k.cpu().pin_memory(), v.cpu().pin_memory(), q.cpu().pin_memory(), scale=w.scale,
               out=out_h)
        torch.cuda.synchronize()
        assert torch.equal(out_d.cpu(), out_h), f"step {step}"
    assert b.graph_stats()[1] > 0, "the host-buffer steps should replay graphs"
    assert a.check() == 0 and b.check() == 0
    a.close()
    b.close()
