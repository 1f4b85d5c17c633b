"""A multi-layer paged KV cache on one GPU, driven through the C ABI.

Orchestration only: the block manager, the cache writes, block copies and
attention all run in libpkv.so; torch supplies device memory, pinned
staging buffers and the stream.

One decode step, as the pages describe it ("KV Cache 与 vLLM" (zwxr.cn)
§3.1-§3.4): the block manager hands every sequence a slot for its new token
(taking a block when the last one is full, copying a shared block on
write); the block tables go to the device; per layer, shared blocks are
copied, the new K/V rows are written, and the new queries attend over each
sequence's cache through its table.
"""
from __future__ import annotations

import math

import numpy as np

from . import capi

_TORCH_DTYPES = None


def torch_dtype(name: str):
    global _TORCH_DTYPES
    import torch
    if _TORCH_DTYPES is None:
        # one-byte caches hold their codes as bytes; the type is passed by name
        _TORCH_DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16, "fp8_e4m3": torch.uint8,
                         "fp8_e5m2": torch.uint8, "int8": torch.uint8, "fp8_e4m3_int4": torch.uint8}
    return _TORCH_DTYPES[name]


class _PinnedRing:
    """Pinned int32 staging buffers reused round-robin, each guarded by an event."""

    def __init__(self, slots: int = 4):
        self.bufs = [None] * slots
        self.events = [None] * slots
        self.i = 0

    def take(self, n: int):
        import torch
        k = self.i
        self.i = (self.i + 1) % len(self.bufs)
        if self.events[k] is not None:
            self.events[k].synchronize()
        if self.bufs[k] is None or self.bufs[k].numel() < n:
            self.bufs[k] = torch.empty(max(n, 1024), dtype=torch.int32, pin_memory=True)
        return k, self.bufs[k]

    def done(self, k: int, stream):
        import torch
        ev = torch.cuda.Event()
        ev.record(stream)
        self.events[k] = ev


class PagedKVCache:
    def __init__(self, *, num_layers: int, num_blocks: int, num_kv_heads: int, head_dim: int,
                 cache_dtype: str, alloc_order=None, device="cuda", poison: bool = False,
                 block_size: int = capi.BLOCK_SIZE):
        import torch
        self.num_layers, self.num_blocks, self.block_size = num_layers, num_blocks, block_size
        self.num_kv_heads, self.head_dim, self.cache_dtype = num_kv_heads, head_dim, cache_dtype
        self.device = torch.device(device)
        self.bm = capi.pkv_bm_create(num_blocks, block_size, alloc_order)
        shape = (num_layers, num_blocks, num_kv_heads, block_size, head_dim)
        tdt = torch_dtype(cache_dtype)
        self.k = torch.empty(shape, dtype=tdt, device=self.device)
        self.v = torch.empty(shape[:4] + (capi.v_row_elems(cache_dtype, head_dim),), dtype=tdt, device=self.device)
        if cache_dtype in capi.SCALED_CACHES:
            # [layers][blocks][heads][2][block_size]: a (block, head)'s K scales, then its V scales
            self._scales = torch.empty(shape[:3] + (2, block_size), dtype=torch.float32, device=self.device)
            self.k_scale, self.v_scale = self._scales[:, :, :, 0, :], self._scales[:, :, :, 1, :]
        else:
            self._scales = self.k_scale = self.v_scale = None
        if poison:  # unwritten slots read as NaN: a kernel that strays onto one shows it
            for t in (self.k, self.v, self._scales):
                if t is not None:
                    t.view(torch.uint8).fill_(0xFF)
        self.err = torch.zeros(1, dtype=torch.int32, device=self.device)
        self._ring = _PinnedRing()
        self._meta = torch.empty(1024, dtype=torch.int32, device=self.device)
        self._ws = {}
        self._stepper = None
        self._stepper_key = None
        self._stepper_bufs = None
        self._scratch = None
        self._graphs = False
        self._cascade = True
        self._io = None
        self._io_key = None
        self._device_index = self.device.index if self.device.index is not None else torch.cuda.current_device()
        self._default_scale = float(np.float32(1.0) / np.sqrt(np.float32(head_dim)))
        self.cow_pairs = []          # every (src, dst) copy, in order

    def close(self):
        if self._stepper is not None:
            capi.pkv_stepper_destroy(self._stepper)
            self._stepper = None
        if self.bm is not None:
            capi.pkv_bm_destroy(self.bm)
            self.bm = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- sequences ---------------------------------------------------------------
    def create(self, seq: int):
        capi.pkv_seq_create(self.bm, seq)

    def fork(self, parent: int, child: int):
        capi.pkv_seq_fork(self.bm, parent, child)

    def free(self, seq: int):
        capi.pkv_seq_free(self.bm, seq)

    def seq_len(self, seq: int) -> int:
        return capi.pkv_seq_len(self.bm, seq)

    # -- prefix cache --------------------------------------------------------------
    def enable_prefix_cache(self, config_key: int = 0):
        """Key full blocks by their token ids so later requests can reuse them."""
        capi.pkv_bm_enable_prefix_cache(self.bm, config_key)

    def admit(self, seq: int, tokens) -> int:
        """Create `seq` for a prompt and map its longest cached prefix; returns the tokens mapped.

        The caller appends the K/V rows of the remaining prompt tokens, then commits.
        """
        return capi.pkv_seq_admit(self.bm, seq, tokens)

    def commit(self, seq: int, tokens) -> int:
        """Register the full blocks of `seq`'s first len(tokens) tokens; returns how many."""
        return capi.pkv_seq_commit_prefix(self.bm, seq, tokens)

    def prefix_stats(self) -> dict:
        return capi.pkv_prefix_cache_stats(self.bm)

    # -- metadata upload ---------------------------------------------------------
    def _upload(self, parts, stream):
        """Copy int32 host arrays to the device in one transfer; returns device views."""
        import torch
        sizes = [int(np.asarray(p).size) for p in parts]
        total = sum(sizes)
        k, pin = self._ring.take(total)
        host = pin.numpy()
        off = 0
        for p, n in zip(parts, sizes):
            host[off:off + n] = np.asarray(p, dtype=np.int32).reshape(-1)
            off += n
        if self._meta.numel() < total:
            self._meta = torch.empty(max(total, 2 * self._meta.numel()), dtype=torch.int32, device=self.device)
        with torch.cuda.stream(stream):
            self._meta[:total].copy_(pin[:total], non_blocking=True)
        self._ring.done(k, stream)
        views, off = [], 0
        for n in sizes:
            views.append(self._meta[off:off + n])
            off += n
        return views

    def _stream(self, stream):
        import torch
        return torch.cuda.current_stream(self.device) if stream is None else stream

    # -- append --------------------------------------------------------------------
    def append(self, seq_ids, k_rows, v_rows, layers=None, stream=None):
        """Append one token per entry of seq_ids.

        k_rows / v_rows: device tensors [num_layers, n, Hkv, D] (or [n, Hkv, D]
        applied to every layer) in f16 / bf16.  Returns (slots, cow_src, cow_dst).
        """
        stream = self._stream(stream)
        slots, cs, cd = capi.pkv_seq_append_slots(self.bm, seq_ids)
        d_slots, d_src, d_dst = self._upload([slots, cs, cd], stream)
        self._apply_append(slots, cs, d_slots, d_src, d_dst, k_rows, v_rows, layers, stream)
        self.cow_pairs.extend(zip(cs.tolist(), cd.tolist()))
        return slots, cs, cd

    def _apply_append(self, slots, cs, d_slots, d_src, d_dst, k_rows, v_rows, layers, stream):
        layers = range(self.num_layers) if layers is None else layers
        for li in layers:
            ks = self.k_scale[li] if self.k_scale is not None else None
            vs = self.v_scale[li] if self.v_scale is not None else None
            if len(cs):
                capi.paged_kv_copy_blocks(self.k[li], self.v[li], ks, vs, d_src, d_dst, len(cs),
                                          d_error=self.err, stream=stream, cache_dtype=self.cache_dtype)
            kr = k_rows[li] if k_rows.dim() == 4 else k_rows
            vr = v_rows[li] if v_rows.dim() == 4 else v_rows
            if len(slots):
                capi.paged_kv_append(kr, vr, d_slots, self.k[li], self.v[li], ks, vs,
                                     d_error=self.err, stream=stream, cache_dtype=self.cache_dtype)

    # -- decode ------------------------------------------------------------------
    def tables(self, seq_ids):
        lens = [self.seq_len(s) for s in seq_ids]
        max_blocks = max(1, max((-(-L // self.block_size) for L in lens), default=1))
        tables, ctx = capi.pkv_build_block_tables(self.bm, seq_ids, max_blocks)
        return tables, ctx

    def workspace(self, num_seqs, num_q_heads, q_dtype):
        import torch
        key = (num_seqs, num_q_heads, q_dtype)
        if key not in self._ws:
            n = capi.paged_attention_workspace_bytes(num_seqs, num_q_heads, self.num_kv_heads, self.head_dim,
                                                     q_dtype, self.cache_dtype)
            self._ws[key] = torch.zeros(max(n, 256), dtype=torch.uint8, device=self.device)  # zero once
        return self._ws[key]

    def decode(self, seq_ids, q, scale=None, out=None, layers=None, stream=None):
        """q: device [num_layers, B, Hq, D] (or [B, Hq, D] for layer 0); returns out like q."""
        import torch
        stream = self._stream(stream)
        tables, ctx = self.tables(seq_ids)
        d_tables, d_ctx = self._upload([tables, ctx], stream)
        d_tables = d_tables.view(tables.shape)
        return self._decode_layers(seq_ids, q, scale, out, layers, d_tables, d_ctx, int(ctx.max(initial=0)),
                                   stream)

    def _decode_layers(self, seq_ids, q, scale, out, layers, d_tables, d_ctx, max_len, stream, marks=None):
        import torch
        one = q.dim() == 3
        if scale is None:
            scale = float(np.float32(1.0) / np.sqrt(np.float32(self.head_dim)))
        if out is None:
            out = torch.empty_like(q)
        b, hq = q.shape[-3], q.shape[-2]
        ws = self.workspace(b, hq, {torch.float16: "f16", torch.bfloat16: "bf16"}[q.dtype])
        layers = ([0] if one else range(self.num_layers)) if layers is None else layers
        if marks is not None:          # events bracketing the attention launches only
            marks[0].record(stream)
        for li in layers:
            ks = self.k_scale[li] if self.k_scale is not None else None
            vs = self.v_scale[li] if self.v_scale is not None else None
            capi.paged_attention_decode(out if one else out[li], q if one else q[li], self.k[li], self.v[li],
                                        ks, vs, d_tables, d_ctx, max_len, scale, ws, d_error=self.err,
                                        stream=stream, cache_dtype=self.cache_dtype)
        if marks is not None:
            marks[1].record(stream)
        return out

    def _stepper_for(self, n: int, num_q_heads: int, q_torch_dtype):
        """The native step executor for batches of n sequences (created on first use)."""
        import torch
        key = (n, num_q_heads, q_torch_dtype)
        q_dtype = {torch.float16: "f16", torch.bfloat16: "bf16"}[q_torch_dtype]
        if self._stepper is not None and self._stepper_key == key:
            return self._stepper
        if self._stepper is not None:
            torch.cuda.synchronize(self.device)
            capi.pkv_stepper_destroy(self._stepper)
            self._stepper = None
        max_blocks = self.num_blocks
        host = torch.empty(capi.pkv_stepper_host_bytes(n, max_blocks) // 4, dtype=torch.int32, pin_memory=True)
        dev = torch.empty(capi.pkv_stepper_device_bytes(n, max_blocks) // 4, dtype=torch.int32, device=self.device)
        ws = self.workspace(n, num_q_heads, q_dtype)
        kb = self.k.element_size()
        pool = capi.PoolDesc(
            num_layers=self.num_layers, num_blocks=self.num_blocks, num_kv_heads=self.num_kv_heads,
            num_q_heads=num_q_heads, head_dim=self.head_dim, q_dtype=capi.DTYPE_NAMES[q_dtype],
            cache_dtype=capi.DTYPE_NAMES[self.cache_dtype], k_cache=self.k.data_ptr(), v_cache=self.v.data_ptr(),
            cache_layer_stride=self.k.stride(0) * kb,
            k_scale=self.k_scale.data_ptr() if self.k_scale is not None else None,
            v_scale=self.v_scale.data_ptr() if self.v_scale is not None else None,
            scale_layer_stride=self.k_scale.stride(0) * 4 if self.k_scale is not None else 0,
            block_size=self.block_size, v_cache_layer_stride=self.v.stride(0) * self.v.element_size())
        self._stepper = capi.pkv_stepper_create(pool, n, max_blocks, host, dev, ws)
        if self._graphs:
            capi.pkv_stepper_use_graphs(self._stepper, True)
        if not self._cascade:
            capi.pkv_stepper_use_cascade(self._stepper, False)
        self._stepper_bufs = (host, dev, ws)
        self._stepper_key = key
        self._scratch = capi.StepScratch(n)
        return self._stepper

    def step(self, seq_ids, k_rows, v_rows, q, scale=None, out=None, stream=None, marks=None):
        """One decode step for all layers through the native executor: append then attend.

        k_rows / v_rows: [num_layers, B, Hkv, D] (or [B, Hkv, D] for every layer);
        q, out: [num_layers, B, Hq, D] (or [B, Hq, D] with one layer); out may be
        float32 or q's dtype.  ``marks``: optional pair of CUDA events recorded
        around the attention launches.
        """
        if scale is None:
            scale = self._default_scale
        if out is None:
            import torch
            out = torch.empty_like(q)
        if not (q.is_cuda and k_rows.is_cuda and v_rows.is_cuda and out.is_cuda):
            return self._step_host_io(seq_ids, k_rows, v_rows, q, scale, out, stream, marks)
        return self._step_native(seq_ids, k_rows, v_rows, q, scale, out, stream, marks)

    def _step_native(self, seq_ids, k_rows, v_rows, q, scale, out, stream, marks):
        key = (len(seq_ids), q.shape[-2], q.dtype)
        st = self._stepper if key == self._stepper_key else self._stepper_for(*key)
        if marks is not None:
            for ev in marks:
                if ev.cuda_event == 0:     # torch creates the event on its first record
                    ev.record(self._stream(stream))
        sh = capi.current_stream_handle(self._device_index) if stream is None else stream
        cs, cd = capi.pkv_stepper_step(st, self.bm, seq_ids, k_rows, v_rows, q, out, scale, self.num_layers,
                                       d_error=self.err, events=marks, stream=sh, scratch=self._scratch)
        if len(cs):
            self.cow_pairs.extend(zip(cs.tolist(), cd.tolist()))
        return out

    def _step_host_io(self, seq_ids, k_rows, v_rows, q, scale, out, stream, marks):
        """A step whose inputs and output are page-locked host tensors.

        One copy kernel moves the step's K/V rows and queries from host to
        device buffers (read in place over the host link), launched by the
        step executor after its host work and right before the attention (the
        step's first decode starts meanwhile), and the decode kernels store
        the output straight into the host tensor.  Synchronise the stream
        before reading ``out`` on the host.
        """
        import torch
        for t in (k_rows, v_rows, q, out):
            if not t.is_cuda and not t.is_pinned():
                raise ValueError("host tensors of a step must be page-locked (pin_memory())")
            if not t.is_contiguous():
                raise ValueError("tensors of a step must be contiguous")
        key = tuple((tuple(t.shape), t.dtype) for t in (k_rows, v_rows, q))
        if self._io_key != key:
            self._io = [torch.empty(t.shape, dtype=t.dtype, device=self.device) for t in (k_rows, v_rows, q)]
            self._io_key = key
        kd, vd, qd = self._io
        ins = [(d, h) for d, h in ((kd, k_rows), (vd, v_rows), (qd, q)) if not h.is_cuda]
        if ins:
            key = (len(seq_ids), q.shape[-2], q.dtype)
            st = self._stepper if key == self._stepper_key else self._stepper_for(*key)
            capi.pkv_stepper_copy_inputs(st, ins)
        return self._step_native(seq_ids, k_rows if k_rows.is_cuda else kd, v_rows if v_rows.is_cuda else vd,
                                 q if q.is_cuda else qd, scale, out, stream, marks)

    def use_graphs(self, enable: bool = True) -> None:
        """Replay each step's attention launches from a CUDA graph (steps without copy-on-write copies).

        Pays off when the step's k/v/q/out buffers stay the same from step to
        step; a change of buffers or batch size captures the graph again.
        """
        self._graphs = bool(enable)
        if self._stepper is not None:
            capi.pkv_stepper_use_graphs(self._stepper, self._graphs)

    def use_cascade(self, enable: bool = True) -> None:
        """Attend shared prefixes once for all sharing sequences (prefix kernel + merge); on by default."""
        self._cascade = bool(enable)
        if self._stepper is not None:
            capi.pkv_stepper_use_cascade(self._stepper, self._cascade)

    def cascade_count(self) -> int:
        """Steps of the current step executor that used the cascade."""
        return capi.pkv_stepper_cascade_count(self._stepper) if self._stepper is not None else 0

    def graph_stats(self):
        """(graphs captured, graphs replayed) by the current step executor."""
        return capi.pkv_stepper_graph_stats(self._stepper) if self._stepper is not None else (0, 0)

    def check(self, stream=None) -> int:
        """Synchronise and return (and clear) the device error bits."""
        return capi.pkv_read_device_error(self.err, clear=True, stream=self._stream(stream))


def blocks_for(length: int, block_size: int = capi.BLOCK_SIZE) -> int:
    return int(math.ceil(length / block_size))
