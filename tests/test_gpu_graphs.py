"""CUDA-graph replay of the decode step against eager steps.

A step executor with graphs enabled captures the step's launches (the
metadata copy and every layer's fused append + attention) once per
metadata half and replays them.  Over several steps it must leave the
cache byte for byte as eager steps do and produce bit for bit the same
outputs (the workloads are large enough that both run a full wave, so the
work split is the same), with odd and even layer counts (the split-counter
bank alternates across replays), through a copy-on-write step that runs
eagerly, and after a change of buffers, which captures again.
"""
import numpy as np
import pytest

from paged_kv_cache_163_gb300 import workloads as wl

from helpers import assert_close, cache_bits, oracle_seq_output, to_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def play():
    from paged_kv_cache_163_gb300 import capi, play as p
    capi.load()
    return p


def _workload(cache_dtype, layers, seed, n=8):
    rng = np.random.default_rng(seed)
    lens = rng.integers(2500, 3000, n).tolist()
    return wl.custom(f"graph-{cache_dtype}-{layers}", lens=lens, num_q_heads=32, num_kv_heads=8, head_dim=128,
                     q_dtype="bf16", cache_dtype=cache_dtype, num_layers=layers, outlier_p=0.002, seed=seed,
                     slack=0.5)


def _static_step(cache, w, step, bufs, play, seqs=None):
    """Copy step `step`'s inputs into the fixed buffers, then step."""
    k, v, q = play.step_inputs(w, step)
    kb, vb, qb, ob = bufs
    seqs = w.seq_ids if seqs is None else seqs
    n = len(seqs)
    kb[:n].copy_(k[:n])
    vb[:n].copy_(v[:n])
    qb[:, :n].copy_(q[:, :n])
    cache.step(seqs, kb[:n], vb[:n], qb[:, :n], scale=w.scale, out=ob[:, :n])
    return ob[:, :n]


def _bufs(w):
    dev = torch.device("cuda")
    dt = torch.bfloat16
    kb = torch.empty((w.num_seqs, w.num_kv_heads, w.head_dim), dtype=dt, device=dev)
    vb = torch.empty_like(kb)
    qb = torch.empty((w.num_layers, w.num_seqs, w.num_q_heads, w.head_dim), dtype=dt, device=dev)
    ob = torch.empty(qb.shape, dtype=torch.float32, device=dev)
    return kb, vb, qb, ob


@pytest.mark.parametrize("cache_dtype,layers", [("bf16", 1), ("bf16", 2), ("bf16", 3), ("fp8_e4m3", 3),
                                                ("fp8_e4m3_int4", 2)])
def test_replayed_steps_equal_eager_steps(play, cache_dtype, layers):
    from paged_kv_cache_163_gb300 import capi
    w = _workload(cache_dtype, layers, seed=60 + layers)
    eager, graph = play.new_cache(w, poison=True), play.new_cache(w, poison=True)
    for c in (eager, graph):                 # graph replays attend without the cascade: compare like with like
        c.use_cascade(False)
    play.prefill(w, eager)
    play.prefill(w, graph)
    graph.use_graphs(True)
    be, bg = _bufs(w), _bufs(w)
    steps = 6
    for step in range(steps):
        oe = _static_step(eager, w, step, be, play)
        n0 = capi.pkv_launch_count()
        og = _static_step(graph, w, step, bg, play)
        assert capi.pkv_launch_count() - n0 == layers + (1 if layers > 1 else 0)
        assert torch.equal(oe, og), f"step {step}"
    assert eager.check() == 0 and graph.check() == 0
    assert graph.graph_stats() == (2, steps)            # one capture per metadata half
    for li in range(layers):
        assert np.array_equal(cache_bits(eager.k[li]), cache_bits(graph.k[li]))
        assert np.array_equal(cache_bits(eager.v[li]), cache_bits(graph.v[li]))
    # and both are right
    q = w.q_rows(layers - 1, steps - 1)
    got = to_f64(og[layers - 1])
    for s in (0, w.num_seqs - 1):
        assert_close(got[s], oracle_seq_output(w, s, q[s], step=steps - 1), f"sequence {s}")
    eager.close()
    graph.close()


def test_copy_on_write_step_runs_eagerly_and_replays_resume(play):
    w = _workload("bf16", 2, seed=70, n=6)
    eager, graph = play.new_cache(w, poison=True), play.new_cache(w, poison=True)
    for c in (eager, graph):                 # graph replays attend without the cascade: compare like with like
        c.use_cascade(False)
    play.prefill(w, eager)
    play.prefill(w, graph)
    graph.use_graphs(True)
    be, bg = _bufs(w), _bufs(w)
    for step in range(2):
        assert torch.equal(_static_step(eager, w, step, be, play), _static_step(graph, w, step, bg, play))
    # sequence 5 is replaced by a fork of sequence 0: its next append copies the shared partial block
    for c in (eager, graph):
        c.free(5)
        c.fork(0, 5)
    seqs = list(range(6))
    cows = len(graph.cow_pairs)
    for step in range(2, 5):
        oe = _static_step(eager, w, step, be, play, seqs)
        og = _static_step(graph, w, step, bg, play, seqs)
        assert torch.equal(oe, og), f"step {step}"
    assert len(graph.cow_pairs) == cows + 1 and eager.cow_pairs == graph.cow_pairs
    captures, replays = graph.graph_stats()
    assert captures == 2 and replays == 4               # the copy-on-write step did not replay
    assert eager.check() == 0 and graph.check() == 0
    eager.close()
    graph.close()


def test_new_buffers_capture_again(play):
    w = _workload("bf16", 1, seed=71)
    eager, graph = play.new_cache(w, poison=True), play.new_cache(w, poison=True)
    for c in (eager, graph):                 # graph replays attend without the cascade: compare like with like
        c.use_cascade(False)
    play.prefill(w, eager)
    play.prefill(w, graph)
    graph.use_graphs(True)
    be, bg = _bufs(w), _bufs(w)
    for step in range(2):
        assert torch.equal(_static_step(eager, w, step, be, play), _static_step(graph, w, step, bg, play))
    assert graph.graph_stats() == (2, 2)
    bg2 = _bufs(w)                                       # other buffers: captured again
    for step in range(2, 4):
        assert torch.equal(_static_step(eager, w, step, be, play), _static_step(graph, w, step, bg2, play))
    assert graph.graph_stats() == (4, 4)
    # graphs off: eager steps with the usual layout, still right
    graph.use_graphs(False)
    k, v, q = play.step_inputs(w, 4)
    out = graph.step(w.seq_ids, k, v, q, scale=w.scale, out=torch.empty(q.shape, device="cuda"))
    got = to_f64(out[0])
    for s in range(w.num_seqs):
        assert_close(got[s], oracle_seq_output(w, s, w.q_rows(0, 4)[s], step=4), f"sequence {s}")
    assert graph.check() == 0
    eager.close()
    graph.close()


def test_other_calls_on_the_workspace_between_replays(play):
    """A public decode call on the stepper's workspace shifts the counter-bank parity: steps stay right."""
    w = _workload("bf16", 1, seed=72)
    eager, graph = play.new_cache(w, poison=True), play.new_cache(w, poison=True)
    for c in (eager, graph):                 # graph replays attend without the cascade: compare like with like
        c.use_cascade(False)
    play.prefill(w, eager)
    play.prefill(w, graph)
    graph.use_graphs(True)
    be, bg = _bufs(w), _bufs(w)
    for step in range(6):
        oe = _static_step(eager, w, step, be, play)
        og = _static_step(graph, w, step, bg, play)
        assert torch.equal(oe, og), f"step {step}"
        if step in (1, 3):                   # one extra decode call on each cache's workspace
            q = play.to_device(w.q_rows(0, step), "bf16", "cuda")
            a = eager.decode(w.seq_ids, q, scale=w.scale, out=torch.empty(q.shape, device="cuda"))
            b = graph.decode(w.seq_ids, q, scale=w.scale, out=torch.empty(q.shape, device="cuda"))
            assert torch.equal(a, b) and torch.equal(a, oe[0])
    captures, replays = graph.graph_stats()
    assert captures == 2 and replays < 6                # steps after an odd shift ran eagerly
    assert eager.check() == 0 and graph.check() == 0
    eager.close()
    graph.close()
