"""ctypes binding of libpkv.so: the C ABI's calls under the same names.

Argument marshalling only: host arrays become pointers, torch tensors give
their device pointers, shapes and dtypes are read off the tensors.  Every
non-OK status raises ``PkvError`` (``NoBlocksError`` for PKV_ERR_NO_BLOCKS)
with the library's one-line reason.  The library is loaded on first use; if
it has not been built the first call raises -- there is no fallback path.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")

PKV_F16, PKV_BF16, PKV_FP8_E4M3, PKV_F32, PKV_FP8_E5M2, PKV_INT8 = 0, 1, 2, 3, 4, 5
PKV_FP8_E4M3_INT4 = 6
DTYPE_NAMES = {"f16": PKV_F16, "bf16": PKV_BF16, "fp8_e4m3": PKV_FP8_E4M3, "f32": PKV_F32,
               "fp8_e5m2": PKV_FP8_E5M2, "int8": PKV_INT8, "fp8_e4m3_int4": PKV_FP8_E4M3_INT4}
# cache types stored as one-byte codes (uint8 tensors) plus fp32 scales
ONE_BYTE_CACHES = ("fp8_e4m3", "fp8_e5m2", "int8")
# cache types with k_scale / v_scale: the one-byte ones, and K FP8 E4M3 + V INT4
# (uint8 tensors; the V rows hold head_dim / 2 bytes)
SCALED_CACHES = ONE_BYTE_CACHES + ("fp8_e4m3_int4",)


def v_row_elems(cache_dtype: str, head_dim: int) -> int:
    """Last dimension of a V cache tensor: head_dim, or head_dim / 2 bytes for 4-bit V."""
    return head_dim // 2 if cache_dtype == "fp8_e4m3_int4" else head_dim
BLOCK_SIZE = 16
MAX_SEQS_PER_CALL = 1024
DEVERR_BAD_SLOT, DEVERR_BAD_BLOCK, DEVERR_BAD_CONTEXT_LEN, DEVERR_WAIT_TIMEOUT = 1, 2, 4, 8

STATUS = {0: "PKV_OK", -1: "PKV_ERR_INVALID", -2: "PKV_ERR_NO_BLOCKS", -3: "PKV_ERR_CUDA",
          -4: "PKV_ERR_UNSUPPORTED", -5: "PKV_ERR_DEVICE_CHECK", -6: "PKV_ERR_WORKSPACE"}


class PkvError(RuntimeError):
    def __init__(self, status: int, where: str, reason: str):
        super().__init__(f"{where}: {STATUS.get(status, status)}: {reason}")
        self.status = status


class NoBlocksError(PkvError):
    pass


_lib = None


class CopySegment(C.Structure):
    """pkv_copy_segment."""
    _fields_ = [("dst", C.c_void_p), ("src", C.c_void_p), ("bytes", C.c_int64)]


MAX_COPY_SEGMENTS = 8


class PoolDesc(C.Structure):
    """pkv_pool_desc: per-layer pools as base pointers plus byte strides."""
    _fields_ = [("num_layers", C.c_int32), ("num_blocks", C.c_int32), ("num_kv_heads", C.c_int32),
                ("num_q_heads", C.c_int32), ("head_dim", C.c_int32), ("q_dtype", C.c_int),
                ("cache_dtype", C.c_int), ("k_cache", C.c_void_p), ("v_cache", C.c_void_p),
                ("cache_layer_stride", C.c_int64), ("k_scale", C.c_void_p), ("v_scale", C.c_void_p),
                ("scale_layer_stride", C.c_int64), ("block_size", C.c_int32),
                ("v_cache_layer_stride", C.c_int64)]


_i32p = C.POINTER(C.c_int32)
_i64p = C.POINTER(C.c_int64)
_vp = C.c_void_p

# name: (restype, argtypes)
_PROTOS = {
    "pkv_bm_create": (C.c_int, [C.c_int32, C.c_int32, _i32p, C.POINTER(_vp)]),
    "pkv_bm_destroy": (None, [_vp]),
    "kv_block_alloc": (C.c_int, [_vp, _i32p]),
    "kv_block_free": (C.c_int, [_vp, C.c_int32]),
    "pkv_seq_create": (C.c_int, [_vp, C.c_int64]),
    "pkv_seq_fork": (C.c_int, [_vp, C.c_int64, C.c_int64]),
    "pkv_seq_free": (C.c_int, [_vp, C.c_int64]),
    "pkv_seq_append_slots": (C.c_int, [_vp, _i64p, C.c_int32, _i32p, _i32p, _i32p, _i32p]),
    "pkv_build_block_tables": (C.c_int, [_vp, _i64p, C.c_int32, C.c_int32, _i32p, _i32p]),
    "pkv_bm_num_free": (C.c_int32, [_vp]),
    "pkv_bm_num_blocks": (C.c_int32, [_vp]),
    "pkv_bm_block_size": (C.c_int32, [_vp]),
    "pkv_bm_free_list": (C.c_int, [_vp, _i32p, C.c_int32, _i32p]),
    "pkv_bm_refcount": (C.c_int, [_vp, C.c_int32, _i32p]),
    "pkv_seq_len": (C.c_int, [_vp, C.c_int64, _i32p]),
    "pkv_kv_bytes": (C.c_int64, [C.c_int32, C.c_int32, C.c_int32, C.c_int64, C.c_int]),
    "pkv_pool_blocks": (C.c_int64, [C.c_int64, C.c_int32, C.c_int32, C.c_int32, C.c_int, C.c_int32]),
    "paged_kv_copy_blocks": (C.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, C.c_int32, C.c_int32, C.c_int32,
                                       C.c_int, C.c_int32, C.c_int32, _vp, _vp]),
    "paged_kv_append": (C.c_int, [_vp, _vp, C.c_int, C.c_int32, C.c_int32, C.c_int32, _vp, _vp, _vp,
                                  C.c_int, _vp, _vp, C.c_int32, C.c_int32, _vp, _vp]),
    "paged_attention_workspace_bytes": (C.c_int, [C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int,
                                                  C.c_int, C.POINTER(C.c_size_t)]),
    "paged_attention_decode": (C.c_int, [_vp, C.c_int, _vp, C.c_int, _vp, _vp, C.c_int, _vp, _vp, _vp, C.c_int32,
                                         _vp, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32,
                                         C.c_int32, C.c_int32, C.c_float, _vp, C.c_size_t, _vp, _vp]),
    # out, out_dtype, q, q_dtype, k_new, v_new, k_cache, v_cache, cache_dtype, k_scale, v_scale, tables,
    # max_blocks, lens, max_len, num_seqs, hq, hkv, d, num_blocks, block_size, scale, workspace, bytes,
    # d_error, stream
    "paged_attention_decode_append": (C.c_int, [_vp, C.c_int, _vp, C.c_int, _vp, _vp, _vp, _vp, C.c_int, _vp, _vp,
                                                _vp, C.c_int32, _vp, C.c_int32, C.c_int32, C.c_int32, C.c_int32,
                                                C.c_int32, C.c_int32, C.c_int32, C.c_float, _vp, C.c_size_t, _vp,
                                                _vp]),
    "paged_attention_decode_static": (C.c_int, [_vp, C.c_int, _vp, C.c_int, _vp, _vp, C.c_int, _vp, _vp, _vp,
                                                C.c_int32, _vp, C.c_int32, C.c_int32, C.c_int32, C.c_int32,
                                                C.c_int32, C.c_int32, C.c_int32, C.c_float, _vp, _vp]),
    "pkv_block_hash": (C.c_uint64, [C.c_uint64, _i32p, C.c_uint64]),
    "pkv_bm_enable_prefix_cache": (C.c_int, [_vp, C.c_uint64]),
    "pkv_seq_admit": (C.c_int, [_vp, C.c_int64, _i32p, C.c_int32, _i32p]),
    "pkv_seq_commit_prefix": (C.c_int, [_vp, C.c_int64, _i32p, C.c_int32, _i32p]),
    "pkv_prefix_cache_stats": (C.c_int, [_vp, C.c_void_p]),
    "pkv_stepper_host_bytes": (C.c_size_t, [C.c_int32, C.c_int32]),
    "pkv_stepper_device_bytes": (C.c_size_t, [C.c_int32, C.c_int32]),
    "pkv_stepper_create": (C.c_int, [C.POINTER(PoolDesc), C.c_int32, C.c_int32, _vp, C.c_size_t, _vp, C.c_size_t,
                                     _vp, C.c_size_t, C.POINTER(_vp)]),
    "pkv_stepper_destroy": (None, [_vp]),
    "pkv_stepper_use_graphs": (C.c_int, [_vp, C.c_int32]),
    "pkv_stepper_use_cascade": (C.c_int, [_vp, C.c_int32]),
    "pkv_stepper_cascade_count": (C.c_int64, [_vp]),
    "pkv_stepper_graph_stats": (C.c_int, [_vp, _i64p, _i64p]),
    # pointer arguments as addresses (ints): the per-step call marshals no ctypes pointer objects
    "pkv_stepper_step": (C.c_int, [_vp, _vp, _vp, C.c_int32, _vp, _vp, C.c_int64, _vp, C.c_int64, _vp, C.c_int,
                                   C.c_int64, C.c_float, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "pkv_read_device_error": (C.c_int, [_vp, _i32p, C.c_int32, _vp]),
    "pkv_launch_count": (C.c_int64, []),
    "pkv_copy_segments": (C.c_int, [C.c_void_p, C.c_int32, _vp]),
    "pkv_stepper_copy_inputs": (C.c_int, [_vp, C.c_void_p, C.c_int32]),
    "pkv_set_decode_kernel": (C.c_int, [C.c_int]),
    "pkv_set_prefix_kernel": (C.c_int, [C.c_int, C.c_int32]),
    "pkv_get_prefix_kernel": (C.c_int, []),
    "pkv_get_decode_kernel": (C.c_int, []),
    "pkv_status_string": (C.c_char_p, [C.c_int]),
    "pkv_last_error": (C.c_char_p, []),
}


def load(path: str = LIB_PATH):
    """Load libpkv.so once; raises if it is missing (build it first)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -m paged_kv_cache_163_gb300.build` (no fallback path exists)")
        lib = C.CDLL(path)
        for name, (res, args) in _PROTOS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def declared_symbols():
    return list(_PROTOS)


def _check(status: int, where: str):
    if status != 0:
        reason = load().pkv_last_error().decode(errors="replace")
        cls = NoBlocksError if status == -2 else PkvError
        raise cls(status, where, reason)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def _i64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int64)


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(C.POINTER(ctype))


# ---- host block manager -------------------------------------------------------
def pkv_bm_create(num_blocks: int, block_size: int = BLOCK_SIZE, alloc_order=None):
    h = _vp()
    order = None if alloc_order is None else _i32(alloc_order)
    if order is not None and len(order) != num_blocks:
        raise PkvError(-1, "pkv_bm_create", "alloc_order must have num_blocks entries")
    _check(load().pkv_bm_create(num_blocks, block_size, None if order is None else _ptr(order, C.c_int32),
                                C.byref(h)), "pkv_bm_create")
    return h


def pkv_bm_destroy(bm) -> None:
    load().pkv_bm_destroy(bm)


def kv_block_alloc(bm) -> int:
    out = C.c_int32()
    _check(load().kv_block_alloc(bm, C.byref(out)), "kv_block_alloc")
    return out.value


def kv_block_free(bm, block_id: int) -> None:
    _check(load().kv_block_free(bm, block_id), "kv_block_free")


def pkv_seq_create(bm, seq_id: int) -> None:
    _check(load().pkv_seq_create(bm, seq_id), "pkv_seq_create")


def pkv_seq_fork(bm, parent: int, child: int) -> None:
    _check(load().pkv_seq_fork(bm, parent, child), "pkv_seq_fork")


def pkv_seq_free(bm, seq_id: int) -> None:
    _check(load().pkv_seq_free(bm, seq_id), "pkv_seq_free")


def pkv_seq_append_slots(bm, seq_ids):
    """Returns (slot_mapping int32[n], cow_src int32[k], cow_dst int32[k])."""
    ids = _i64(seq_ids)
    n = len(ids)
    slots = np.empty(n, np.int32)
    src = np.empty(max(n, 1), np.int32)
    dst = np.empty(max(n, 1), np.int32)
    ncow = C.c_int32()
    _check(load().pkv_seq_append_slots(bm, _ptr(ids, C.c_int64), n, _ptr(slots, C.c_int32),
                                       _ptr(src, C.c_int32), _ptr(dst, C.c_int32), C.byref(ncow)),
           "pkv_seq_append_slots")
    return slots, src[:ncow.value].copy(), dst[:ncow.value].copy()


def pkv_build_block_tables(bm, seq_ids, max_blocks: int, tables=None, context_lens=None):
    """Returns (tables int32[n, max_blocks] padded with -1, context_lens int32[n]).

    ``tables`` / ``context_lens`` may be preallocated C-contiguous int32 arrays.
    """
    ids = _i64(seq_ids)
    n = len(ids)
    if tables is None:
        tables = np.empty((n, max_blocks), np.int32)
    if context_lens is None:
        context_lens = np.empty(n, np.int32)
    assert tables.dtype == np.int32 and tables.flags.c_contiguous and tables.size >= n * max_blocks
    assert context_lens.dtype == np.int32 and context_lens.flags.c_contiguous and context_lens.size >= n
    _check(load().pkv_build_block_tables(bm, _ptr(ids, C.c_int64), n, max_blocks, _ptr(tables, C.c_int32),
                                         _ptr(context_lens, C.c_int32)), "pkv_build_block_tables")
    return tables, context_lens


def pkv_bm_num_free(bm) -> int:
    return int(load().pkv_bm_num_free(bm))


def pkv_bm_num_blocks(bm) -> int:
    return int(load().pkv_bm_num_blocks(bm))


def pkv_bm_free_list(bm) -> np.ndarray:
    n = C.c_int32()
    _check(load().pkv_bm_free_list(bm, None, 0, C.byref(n)), "pkv_bm_free_list")
    out = np.empty(max(n.value, 1), np.int32)
    _check(load().pkv_bm_free_list(bm, _ptr(out, C.c_int32), n.value, C.byref(n)), "pkv_bm_free_list")
    return out[:n.value].copy()


def pkv_bm_refcount(bm, block_id: int) -> int:
    out = C.c_int32()
    _check(load().pkv_bm_refcount(bm, block_id, C.byref(out)), "pkv_bm_refcount")
    return out.value


def pkv_seq_len(bm, seq_id: int) -> int:
    out = C.c_int32()
    _check(load().pkv_seq_len(bm, seq_id, C.byref(out)), "pkv_seq_len")
    return out.value


def pkv_kv_bytes(layers, kv_heads, head_dim, tokens, cache_dtype) -> int:
    return int(load().pkv_kv_bytes(layers, kv_heads, head_dim, tokens, _dt(cache_dtype)))


def pkv_pool_blocks(budget_bytes, layers, kv_heads, head_dim, cache_dtype, block_size=BLOCK_SIZE) -> int:
    return int(load().pkv_pool_blocks(budget_bytes, layers, kv_heads, head_dim, _dt(cache_dtype), block_size))


def pkv_bm_block_size(bm) -> int:
    return int(load().pkv_bm_block_size(bm))


# ---- prefix cache --------------------------------------------------------------
class PrefixStats(C.Structure):
    _fields_ = [("lookups", C.c_int64), ("hits", C.c_int64), ("evictions", C.c_int64),
                ("registered", C.c_int64), ("evictable", C.c_int64)]


def pkv_block_hash(parent_hash: int, tokens, config_key: int) -> int:
    t = _i32(tokens)
    if t.size != BLOCK_SIZE:
        raise ValueError("a block hash takes exactly 16 token ids")
    return int(load().pkv_block_hash(parent_hash & 0xFFFFFFFFFFFFFFFF, _ptr(t, C.c_int32),
                                     config_key & 0xFFFFFFFFFFFFFFFF))


def pkv_bm_enable_prefix_cache(bm, config_key: int = 0) -> None:
    _check(load().pkv_bm_enable_prefix_cache(bm, config_key & 0xFFFFFFFFFFFFFFFF), "pkv_bm_enable_prefix_cache")


def pkv_seq_admit(bm, seq_id, tokens) -> int:
    t = _i32(tokens)
    out = C.c_int32()
    _check(load().pkv_seq_admit(bm, int(seq_id), _ptr(t, C.c_int32), t.size, C.byref(out)), "pkv_seq_admit")
    return out.value


def pkv_seq_commit_prefix(bm, seq_id, tokens) -> int:
    t = _i32(tokens)
    out = C.c_int32()
    _check(load().pkv_seq_commit_prefix(bm, int(seq_id), _ptr(t, C.c_int32), t.size, C.byref(out)),
           "pkv_seq_commit_prefix")
    return out.value


def pkv_prefix_cache_stats(bm) -> dict:
    st = PrefixStats()
    _check(load().pkv_prefix_cache_stats(bm, C.byref(st)), "pkv_prefix_cache_stats")
    return {k: int(getattr(st, k)) for k, _ in PrefixStats._fields_}


# ---- device calls --------------------------------------------------------------
def _dt(x) -> int:
    """pkv_dtype of a name ('bf16'), an int, or a torch dtype."""
    if isinstance(x, int):
        return x
    if isinstance(x, str):
        return DTYPE_NAMES[x]
    import torch
    # INT8 caches hold uint8 bytes (code + 128): name them ("int8"), a uint8 tensor reads as FP8 E4M3
    m = {torch.float16: PKV_F16, torch.bfloat16: PKV_BF16, torch.uint8: PKV_FP8_E4M3, torch.float32: PKV_F32}
    if hasattr(torch, "float8_e4m3fn"):
        m[torch.float8_e4m3fn] = PKV_FP8_E4M3
    if hasattr(torch, "float8_e5m2"):
        m[torch.float8_e5m2] = PKV_FP8_E5M2
    return m[x]


def _cdt(k_cache, cache_dtype) -> int:
    """Cache pkv_dtype: given by name, else read off the tensor (uint8 reads as FP8 E4M3)."""
    return _dt(cache_dtype) if cache_dtype is not None else _dt(k_cache.dtype)


def _dp(t):
    """Device pointer of a tensor (or None / an int address)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def paged_kv_copy_blocks(k_cache, v_cache, k_scale, v_scale, src, dst, num_pairs=None,
                         d_error=None, stream=None, cache_dtype=None) -> None:
    nb, hkv, bs, d = k_cache.shape
    n = src.numel() if num_pairs is None else num_pairs
    _check(load().paged_kv_copy_blocks(_dp(k_cache), _dp(v_cache), _dp(k_scale), _dp(v_scale), _dp(src),
                                       _dp(dst), n, hkv, d, _cdt(k_cache, cache_dtype), nb, bs, _dp(d_error),
                                       _stream(stream)), "paged_kv_copy_blocks")


def paged_kv_append(k, v, slot_mapping, k_cache, v_cache, k_scale=None, v_scale=None,
                    d_error=None, stream=None, cache_dtype=None) -> None:
    t, hkv, d = k.shape
    nb, bs = k_cache.shape[0], k_cache.shape[2]
    _check(load().paged_kv_append(_dp(k), _dp(v), _dt(k.dtype), t, hkv, d, _dp(slot_mapping), _dp(k_cache),
                                  _dp(v_cache), _cdt(k_cache, cache_dtype), _dp(k_scale), _dp(v_scale), nb, bs,
                                  _dp(d_error), _stream(stream)), "paged_kv_append")


def paged_attention_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, q_dtype,
                                    cache_dtype) -> int:
    out = C.c_size_t()
    _check(load().paged_attention_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, _dt(q_dtype),
                                                  _dt(cache_dtype), C.byref(out)),
           "paged_attention_workspace_bytes")
    return out.value


def paged_attention_decode(out, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                           max_context_len, scale, workspace, d_error=None, stream=None,
                           num_seqs=None, cache_dtype=None) -> None:
    b, hq, d = q.shape
    if num_seqs is not None:
        b = num_seqs
    nb, hkv, bs = k_cache.shape[0], k_cache.shape[1], k_cache.shape[2]
    _check(load().paged_attention_decode(
        _dp(out), _dt(out.dtype), _dp(q), _dt(q.dtype), _dp(k_cache), _dp(v_cache), _cdt(k_cache, cache_dtype),
        _dp(k_scale),
        _dp(v_scale), _dp(block_tables), block_tables.shape[-1], _dp(context_lens), int(max_context_len), b, hq,
        hkv, d, nb, bs, float(scale), _dp(workspace), workspace.numel() * workspace.element_size(),
        _dp(d_error), _stream(stream)), "paged_attention_decode")


def paged_attention_decode_append(out, q, k_new, v_new, k_cache, v_cache, k_scale, v_scale, block_tables,
                                  context_lens, max_context_len, scale, workspace, d_error=None, stream=None,
                                  num_seqs=None, cache_dtype=None) -> None:
    """Append row b of k_new / v_new at position context_lens[b] - 1, then decode (one launch)."""
    b, hq, d = q.shape
    if num_seqs is not None:
        b = num_seqs
    nb, hkv, bs = k_cache.shape[0], k_cache.shape[1], k_cache.shape[2]
    _check(load().paged_attention_decode_append(
        _dp(out), _dt(out.dtype), _dp(q), _dt(q.dtype), _dp(k_new), _dp(v_new), _dp(k_cache), _dp(v_cache),
        _cdt(k_cache, cache_dtype), _dp(k_scale), _dp(v_scale), _dp(block_tables), block_tables.shape[-1],
        _dp(context_lens), int(max_context_len), b, hq, hkv, d, nb, bs, float(scale), _dp(workspace),
        workspace.numel() * workspace.element_size(), _dp(d_error), _stream(stream)), "paged_attention_decode_append")


def paged_attention_decode_static(out, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                                  max_context_len, scale, d_error=None, stream=None, num_seqs=None,
                                  cache_dtype=None) -> None:
    """paged_attention_decode with the library's static scratch (no workspace, no allocation)."""
    b, hq, d = q.shape
    if num_seqs is not None:
        b = num_seqs
    nb, hkv, bs = k_cache.shape[0], k_cache.shape[1], k_cache.shape[2]
    _check(load().paged_attention_decode_static(
        _dp(out), _dt(out.dtype), _dp(q), _dt(q.dtype), _dp(k_cache), _dp(v_cache), _cdt(k_cache, cache_dtype),
        _dp(k_scale), _dp(v_scale), _dp(block_tables), block_tables.shape[-1], _dp(context_lens),
        int(max_context_len), b, hq, hkv, d, nb, bs, float(scale), _dp(d_error), _stream(stream)),
        "paged_attention_decode_static")


def pkv_stepper_host_bytes(max_seqs, max_blocks_per_seq) -> int:
    return int(load().pkv_stepper_host_bytes(max_seqs, max_blocks_per_seq))


def pkv_stepper_device_bytes(max_seqs, max_blocks_per_seq) -> int:
    return int(load().pkv_stepper_device_bytes(max_seqs, max_blocks_per_seq))


def pkv_stepper_create(pool: PoolDesc, max_seqs, max_blocks_per_seq, host_staging, dev_meta, workspace):
    h = _vp()
    _check(load().pkv_stepper_create(C.byref(pool), max_seqs, max_blocks_per_seq, host_staging.data_ptr(),
                                     host_staging.numel() * host_staging.element_size(), _dp(dev_meta),
                                     dev_meta.numel() * dev_meta.element_size(), _dp(workspace),
                                     workspace.numel() * workspace.element_size(), C.byref(h)),
           "pkv_stepper_create")
    return h


def pkv_stepper_destroy(st) -> None:
    load().pkv_stepper_destroy(st)


def pkv_stepper_use_graphs(st, enable: bool) -> None:
    _check(load().pkv_stepper_use_graphs(st, 1 if enable else 0), "pkv_stepper_use_graphs")


def pkv_stepper_use_cascade(st, enable: bool) -> None:
    _check(load().pkv_stepper_use_cascade(st, 1 if enable else 0), "pkv_stepper_use_cascade")


def pkv_stepper_cascade_count(st) -> int:
    return int(load().pkv_stepper_cascade_count(st))


def pkv_stepper_graph_stats(st):
    """(graphs captured, graphs replayed) by this stepper."""
    c, r = C.c_int64(0), C.c_int64(0)
    _check(load().pkv_stepper_graph_stats(st, C.byref(c), C.byref(r)), "pkv_stepper_graph_stats")
    return int(c.value), int(r.value)


def _layer_stride(t, layers):
    """Byte stride between layers of a per-layer tensor ([layers, ...] or one tensor for all: 0)."""
    return t.stride(0) * t.element_size() if t.dim() == 4 and layers > 1 else 0


class StepScratch:
    """Host arrays a step writes its copy pairs into, allocated once per stepper."""

    def __init__(self, max_seqs: int):
        self.src = np.empty(max(max_seqs, 1), np.int32)
        self.dst = np.empty(max(max_seqs, 1), np.int32)
        self.ncow = np.zeros(1, np.int32)
        self.addr = (self.src.ctypes.data, self.dst.ctypes.data, self.ncow.ctypes.data)


def _segments(pairs, where):
    segs = (CopySegment * max(1, len(pairs)))()
    for i, (dst, src) in enumerate(pairs):
        nb = src.numel() * src.element_size()
        if dst.numel() * dst.element_size() != nb:
            raise ValueError(f"{where}: sizes differ")
        segs[i].dst, segs[i].src, segs[i].bytes = dst.data_ptr(), src.data_ptr(), nb
    return segs


def pkv_copy_segments(pairs, stream) -> None:
    """One-launch copy of [(dst tensor, src tensor), ...] (same byte sizes; device or pinned host memory)."""
    _check(load().pkv_copy_segments(_segments(pairs, "pkv_copy_segments"), len(pairs), stream), "pkv_copy_segments")


def pkv_stepper_copy_inputs(st, pairs) -> None:
    """Register [(device tensor, pinned host tensor), ...] copies for the stepper's next step."""
    _check(load().pkv_stepper_copy_inputs(st, _segments(pairs, "pkv_stepper_copy_inputs"), len(pairs)),
           "pkv_stepper_copy_inputs")


def current_stream_handle(device_index: int) -> int:
    """cudaStream_t of torch's current stream on a device."""
    import torch
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:
        return raw(device_index)
    return torch.cuda.current_stream(device_index).cuda_stream


_TORCH_DT = None


def _dt_torch(dtype) -> int:
    global _TORCH_DT
    if _TORCH_DT is None:
        import torch
        _TORCH_DT = {torch.float16: PKV_F16, torch.bfloat16: PKV_BF16, torch.float32: PKV_F32,
                     torch.uint8: PKV_FP8_E4M3}
    return _TORCH_DT[dtype]


def pkv_stepper_step(st, bm, seq_ids, k_new, v_new, q, out, scale, layers, d_error=None, events=None,
                     stream=None, scratch: StepScratch | None = None):
    """One decode step; returns (cow_src, cow_dst) of the step.

    ``stream``: a torch stream, a cudaStream_t address, or None for the current
    stream of q's device.  ``scratch``: reusable host arrays (else allocated).
    """
    ids = seq_ids if isinstance(seq_ids, np.ndarray) and seq_ids.dtype == np.int64 else \
        np.asarray(seq_ids, dtype=np.int64)
    if not ids.flags.c_contiguous:
        ids = np.ascontiguousarray(ids)
    n = ids.shape[0]
    if scratch is None or scratch.src.shape[0] < n:
        scratch = StepScratch(n)
    ev0 = ev1 = None
    if events is not None:
        ev0, ev1 = events[0].cuda_event, events[1].cuda_event
    if stream is None:
        sh = current_stream_handle(q.device.index)
    elif isinstance(stream, int):
        sh = stream
    else:
        sh = stream.cuda_stream
    a_src, a_dst, a_n = scratch.addr
    status = load().pkv_stepper_step(
        st, bm, ids.ctypes.data, n, k_new.data_ptr(), v_new.data_ptr(), _layer_stride(k_new, layers),
        q.data_ptr(), _layer_stride(q, layers), out.data_ptr(), _dt_torch(out.dtype), _layer_stride(out, layers),
        float(scale), a_src, a_dst, a_n, _dp(d_error), ev0, ev1, sh)
    if status != 0:
        _check(status, "pkv_stepper_step")
    ncow = int(scratch.ncow[0])
    if ncow == 0:
        return _EMPTY_I32, _EMPTY_I32
    return scratch.src[:ncow].copy(), scratch.dst[:ncow].copy()


_EMPTY_I32 = np.empty(0, np.int32)


def pkv_read_device_error(d_error, clear: bool = True, stream=None, raise_on_error: bool = False) -> int:
    h = C.c_int32()
    st = load().pkv_read_device_error(_dp(d_error), C.byref(h), 1 if clear else 0, _stream(stream))
    if st != -5 or raise_on_error:
        _check(st, "pkv_read_device_error")
    return h.value


DECODE_KERNELS = {"auto": 0, "simt": 1, "mma": 2}


def pkv_set_decode_kernel(kind) -> None:
    """Select the decode kernel process-wide: 'auto', 'simt' or 'mma'."""
    _check(load().pkv_set_decode_kernel(DECODE_KERNELS.get(kind, kind)), "pkv_set_decode_kernel")


def pkv_get_decode_kernel() -> str:
    v = int(load().pkv_get_decode_kernel())
    return {k: n for n, k in DECODE_KERNELS.items()}[v]


PREFIX_KERNELS = {"auto": 0, "mma_sync": 1, "tcgen05": 2}


def pkv_set_prefix_kernel(kind, chunk_tiles: int = 0) -> None:
    """Select the cascade's prefix kernel process-wide: 'auto', 'mma_sync' or 'tcgen05'."""
    _check(load().pkv_set_prefix_kernel(PREFIX_KERNELS.get(kind, kind), int(chunk_tiles)), "pkv_set_prefix_kernel")


def pkv_get_prefix_kernel() -> str:
    v = int(load().pkv_get_prefix_kernel())
    return {k: n for n, k in PREFIX_KERNELS.items()}[v]


def pkv_launch_count() -> int:
    return int(load().pkv_launch_count())


def pkv_status_string(status: int) -> str:
    return load().pkv_status_string(status).decode()
