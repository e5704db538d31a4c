"""ctypes binding of libkvpaged.so — argument marshalling only.

Every function here has the name of the C entry point it calls (include/kvpaged.h)
and does nothing but convert arguments and raise ``KvError`` on a negative status.
There is no Python or CPU fallback: if the library is missing, loading fails.
"""

from __future__ import annotations

import ctypes as C
import os

from . import build as _build

KV_OK, KV_ERR_INVALID_ARG, KV_ERR_NO_BLOCKS, KV_ERR_STATE = 0, -1, -2, -3
KV_ERR_CUDA, KV_ERR_DEVICE, KV_ERR_UNSUPPORTED = -4, -5, -6
KV_F32, KV_F16, KV_FP8_E4M3 = 0, 1, 2
KV_DEVERR_SLOT, KV_DEVERR_BLOCK_ID, KV_DEVERR_CONTEXT, KV_DEVERR_TIMEOUT = 1, 2, 4, 8
KV_DEVERR_PREFIX = 16
KV_FEATURE_TENSOR_MAPS = 1
KV_DECODE_WORKSPACE_ZEROED, KV_DECODE_PDL, KV_DECODE_EARLY_TABLES, KV_DECODE_OUT_F16 = 1, 2, 4, 8
KV_DECODE_EARLY_POOL = 16
KV_MAX_DECODE_BATCH = 65536


class KvError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status} ({kv_status_str(status)})")


class kv_pool_desc(C.Structure):
    _fields_ = [("num_layers", C.c_int), ("num_blocks", C.c_int), ("block_size", C.c_int),
                ("num_heads", C.c_int), ("head_dim", C.c_int), ("dtype", C.c_int)]


class kv_decode_args(C.Structure):
    _fields_ = [("layer", C.c_int), ("q", C.c_void_p), ("num_q_heads", C.c_int),
                ("k_new", C.c_void_p), ("v_new", C.c_void_p), ("in_dtype", C.c_int),
                ("out", C.c_void_p), ("block_tables", C.c_void_p), ("max_blocks_per_seq", C.c_int),
                ("context_lens", C.c_void_p), ("batch", C.c_int), ("max_context", C.c_int),
                ("window", C.c_int), ("scale", C.c_float), ("partition_tokens", C.c_int),
                ("workspace", C.c_void_p), ("workspace_bytes", C.c_size_t), ("stream", C.c_void_p),
                ("flags", C.c_uint), ("prefix_groups", C.c_void_p), ("num_prefix_groups", C.c_int)]


class kv_alloc_stats_t(C.Structure):
    _fields_ = [("num_blocks", C.c_int), ("free_blocks", C.c_int), ("shared_blocks", C.c_int),
                ("num_seqs", C.c_int), ("used_slots", C.c_int64), ("wasted_slots", C.c_int64)]


_VP, _I32P, _I64P = C.c_void_p, C.POINTER(C.c_int32), C.POINTER(C.c_int64)
_SIGS = {
    "kv_status_str": (C.c_char_p, [C.c_int]),
    "kv_version": (C.c_int, []),
    "kv_pool_create": (C.c_int, [C.POINTER(kv_pool_desc), C.POINTER(_VP), C.POINTER(_VP),
                                 C.POINTER(_VP), C.POINTER(_VP), C.POINTER(_VP)]),
    "kv_pool_destroy": (C.c_int, [_VP]),
    "kv_pool_get_desc": (C.c_int, [_VP, C.POINTER(kv_pool_desc)]),
    "kv_pool_features": (C.c_int, [_VP, C.POINTER(C.c_uint)]),
    "kv_get_device_error": (C.c_int, [_VP, _VP, C.c_int, C.POINTER(C.c_int)]),
    "kv_selftest_wait_timeout": (C.c_int, [_VP, C.c_uint64, _VP]),
    "kv_append": (C.c_int, [_VP, C.c_int, _VP, _VP, C.c_int, _VP, C.c_int, _VP]),
    "kv_copy_blocks": (C.c_int, [_VP, _VP, C.c_int, C.c_int, C.c_int, _VP]),
    "kv_swap_bytes": (C.c_size_t, [_VP, C.c_int, C.c_int, C.c_int]),
    "kv_swap_out": (C.c_int, [_VP, _VP, C.c_int, C.c_int, C.c_int, _VP, _VP]),
    "kv_swap_in": (C.c_int, [_VP, _VP, _VP, C.c_int, C.c_int, C.c_int, _VP]),
    "paged_decode_workspace_size": (C.c_size_t, [_VP, C.c_int, C.c_int, C.c_int]),
    "paged_decode_attention": (C.c_int, [_VP, C.c_int, _VP, _VP, _VP, C.c_int, _VP, C.c_int,
                                         C.c_int, C.c_float, C.c_int, _VP, C.c_size_t, _VP]),
    "paged_decode_attention_append": (C.c_int, [_VP, C.c_int, _VP, _VP, _VP, C.c_int, _VP, _VP, C.c_int,
                                                _VP, C.c_int, C.c_int, C.c_float, C.c_int, _VP,
                                                C.c_size_t, _VP]),
    "paged_decode_workspace_size_gqa": (C.c_size_t, [_VP, C.c_int, C.c_int, C.c_int, C.c_int]),
    "paged_decode_attention_gqa": (C.c_int, [_VP, C.c_int, _VP, C.c_int, _VP, _VP, C.c_int, _VP, _VP,
                                             C.c_int, _VP, C.c_int, C.c_int, C.c_float, C.c_int, _VP,
                                             C.c_size_t, _VP]),
    "paged_decode_attention_static": (C.c_int, [_VP, C.c_int, _VP, _VP, _VP, C.c_int, _VP, C.c_int,
                                                C.c_int, C.c_float, C.c_int, _VP]),
    "kv_alloc_create": (C.c_int, [C.c_int, C.c_int, _I32P, C.POINTER(_VP)]),
    "kv_alloc_destroy": (C.c_int, [_VP]),
    "kv_alloc_seq_new": (C.c_int, [_VP, C.POINTER(C.c_int)]),
    "kv_alloc_seq_fork": (C.c_int, [_VP, C.c_int, C.POINTER(C.c_int)]),
    "kv_alloc_append_slots": (C.c_int, [_VP, C.c_int, C.c_int, _I64P, _I32P]),
    "kv_alloc_decode_step": (C.c_int, [_VP, _I32P, C.c_int, _I64P, _I32P, C.POINTER(C.c_int)]),
    "kv_alloc_seq_free": (C.c_int, [_VP, C.c_int]),
    "kv_alloc_seq_trim": (C.c_int, [_VP, C.c_int, C.c_int64, C.POINTER(C.c_int)]),
    "paged_decode_workspace_size_ex": (C.c_size_t, [_VP, _VP]),
    "paged_decode_attention_ex": (C.c_int, [_VP, _VP]),
    "kv_decode_step": (C.c_int, [_VP, _VP, _I32P, C.c_int, C.c_int, _VP, _VP, _VP, _VP, C.c_size_t, _VP,
                                 C.c_size_t, _VP]),
    "kv_alloc_seq_info": (C.c_int, [_VP, C.c_int, C.POINTER(C.c_int), C.POINTER(C.c_int)]),
    "kv_alloc_block_table": (C.c_int, [_VP, C.c_int, _I32P, C.c_int, C.POINTER(C.c_int)]),
    "kv_alloc_build_tables": (C.c_int, [_VP, _I32P, C.c_int, _I32P, C.c_int, _I32P]),
    "kv_alloc_ref_count": (C.c_int, [_VP, C.c_int, C.POINTER(C.c_int)]),
    "kv_alloc_free_list": (C.c_int, [_VP, _I32P, C.c_int, C.POINTER(C.c_int)]),
    "kv_alloc_stats": (C.c_int, [_VP, C.POINTER(kv_alloc_stats_t)]),
}

_lib = None


def library_path() -> str:
    return _build.LIB


def load() -> C.CDLL:
    """Load libkvpaged.so (must have been built: ``paged_kv_cache_169_gb300.build.build()``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"{_build.LIB} is not built; run paged_kv_cache_169_gb300.build.build()")
        lib = C.CDLL(_build.LIB)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _check(fn: str, rc: int) -> None:
    if rc != KV_OK:
        raise KvError(fn, rc)


def _ptr_array(ptrs):
    arr = (_VP * len(ptrs))(*[int(p) for p in ptrs])
    return arr


def _i32(buf):
    return C.cast(buf, _I32P)


def _i64(buf):
    return C.cast(buf, _I64P)


# ---------------------------------------------------------------- misc
def kv_status_str(status: int) -> str:
    return load().kv_status_str(status).decode()


def kv_version() -> int:
    return load().kv_version()


# ---------------------------------------------------------------- pool
def kv_pool_create(num_layers, num_blocks, block_size, num_heads, head_dim, dtype,
                   k_layers, v_layers, k_scales=None, v_scales=None) -> int:
    """k_layers/v_layers (and scales for FP8): sequences of device addresses (ints)."""
    desc = kv_pool_desc(num_layers, num_blocks, block_size, num_heads, head_dim, dtype)
    out = _VP()
    ks = _ptr_array(k_scales) if k_scales is not None else None
    vs = _ptr_array(v_scales) if v_scales is not None else None
    _check("kv_pool_create", load().kv_pool_create(C.byref(desc), _ptr_array(k_layers),
                                                   _ptr_array(v_layers), ks, vs, C.byref(out)))
    return out.value


def kv_pool_destroy(pool: int) -> None:
    _check("kv_pool_destroy", load().kv_pool_destroy(pool))


def kv_pool_get_desc(pool: int) -> kv_pool_desc:
    d = kv_pool_desc()
    _check("kv_pool_get_desc", load().kv_pool_get_desc(pool, C.byref(d)))
    return d


def kv_pool_features(pool: int) -> int:
    """Bit flags of the pool's fast paths (KV_FEATURE_*)."""
    f = C.c_uint(0)
    _check("kv_pool_features", load().kv_pool_features(pool, C.byref(f)))
    return f.value


def kv_selftest_wait_timeout(pool: int, limit_ns: int, stream: int = 0) -> None:
    """Launch the bounded-wait self-test (a wait that must time out after limit_ns)."""
    _check("kv_selftest_wait_timeout", load().kv_selftest_wait_timeout(pool, limit_ns, stream))


def kv_get_device_error(pool: int, stream: int = 0, clear: bool = True) -> int:
    """Device error bits (0 = none).  Synchronises ``stream``."""
    code = C.c_int(0)
    rc = load().kv_get_device_error(pool, stream, int(clear), C.byref(code))
    if rc not in (KV_OK, KV_ERR_DEVICE):
        _check("kv_get_device_error", rc)
    return code.value


def kv_append(pool: int, layer: int, k: int, v: int, in_dtype: int, slot_mapping: int,
              num_tokens: int, stream: int = 0) -> None:
    _check("kv_append", load().kv_append(pool, layer, k, v, in_dtype, slot_mapping, num_tokens, stream))


def kv_copy_blocks(pool: int, pairs: int, num_pairs: int, layer_begin: int, layer_end: int,
                   stream: int = 0) -> None:
    _check("kv_copy_blocks", load().kv_copy_blocks(pool, pairs, num_pairs, layer_begin, layer_end, stream))


def kv_swap_bytes(pool: int, num_blocks: int, layer_begin: int, layer_end: int) -> int:
    return load().kv_swap_bytes(pool, num_blocks, layer_begin, layer_end)


def kv_swap_out(pool: int, blocks: int, num_blocks: int, layer_begin: int, layer_end: int, host_dst: int,
                stream: int = 0) -> None:
    _check("kv_swap_out", load().kv_swap_out(pool, blocks, num_blocks, layer_begin, layer_end, host_dst, stream))


def kv_swap_in(pool: int, host_src: int, blocks: int, num_blocks: int, layer_begin: int, layer_end: int,
               stream: int = 0) -> None:
    _check("kv_swap_in", load().kv_swap_in(pool, host_src, blocks, num_blocks, layer_begin, layer_end, stream))


def paged_decode_workspace_size(pool: int, batch: int, max_context: int, partition_tokens: int = 0) -> int:
    n = load().paged_decode_workspace_size(pool, batch, max_context, partition_tokens)
    if n == 0:
        raise KvError("paged_decode_workspace_size", KV_ERR_INVALID_ARG)
    return n


def paged_decode_attention(pool: int, layer: int, q: int, out: int, block_tables: int,
                           max_blocks_per_seq: int, context_lens: int, batch: int, max_context: int,
                           scale: float, partition_tokens: int, workspace: int, workspace_bytes: int,
                           stream: int = 0) -> None:
    _check("paged_decode_attention", load().paged_decode_attention(
        pool, layer, q, out, block_tables, max_blocks_per_seq, context_lens, batch, max_context,
        scale, partition_tokens, workspace, workspace_bytes, stream))


def paged_decode_attention_append(pool: int, layer: int, q: int, k_new: int, v_new: int,
                                  in_dtype: int, out: int, block_tables: int, max_blocks_per_seq: int,
                                  context_lens: int, batch: int, max_context: int, scale: float,
                                  partition_tokens: int, workspace: int, workspace_bytes: int,
                                  stream: int = 0) -> None:
    _check("paged_decode_attention_append", load().paged_decode_attention_append(
        pool, layer, q, k_new, v_new, in_dtype, out, block_tables, max_blocks_per_seq, context_lens,
        batch, max_context, scale, partition_tokens, workspace, workspace_bytes, stream))


def paged_decode_workspace_size_gqa(pool: int, batch: int, num_q_heads: int, max_context: int,
                                    partition_tokens: int = 0) -> int:
    n = load().paged_decode_workspace_size_gqa(pool, batch, num_q_heads, max_context, partition_tokens)
    if n == 0:
        raise KvError("paged_decode_workspace_size_gqa", KV_ERR_INVALID_ARG)
    return n


def paged_decode_attention_gqa(pool: int, layer: int, q: int, num_q_heads: int, k_new: int, v_new: int,
                               in_dtype: int, out: int, block_tables: int, max_blocks_per_seq: int,
                               context_lens: int, batch: int, max_context: int, scale: float,
                               partition_tokens: int, workspace: int, workspace_bytes: int,
                               stream: int = 0) -> None:
    _check("paged_decode_attention_gqa", load().paged_decode_attention_gqa(
        pool, layer, q, num_q_heads, k_new, v_new, in_dtype, out, block_tables, max_blocks_per_seq,
        context_lens, batch, max_context, scale, partition_tokens, workspace, workspace_bytes, stream))


def paged_decode_workspace_size_ex(pool: int, args: "kv_decode_args") -> int:
    n = load().paged_decode_workspace_size_ex(pool, C.byref(args))
    if n == 0:
        raise KvError("paged_decode_workspace_size_ex", KV_ERR_INVALID_ARG)
    return n


def paged_decode_attention_ex(pool: int, args: "kv_decode_args") -> None:
    _check("paged_decode_attention_ex", load().paged_decode_attention_ex(pool, C.byref(args)))


def kv_decode_step(alloc: int, pool: int, seqs, n: int, max_blocks: int, staging: int, dev_meta: int,
                   inputs_h: int, inputs_d: int, inputs_bytes: int, out_h: int, out_bytes: int,
                   args: "kv_decode_args") -> int:
    """One decode step of a batch through the host allocator and one fused call (see the C
    header): seqs is a ctypes int32 array of n ids; staging / inputs_h / out_h are host
    addresses (pinned), dev_meta / inputs_d device addresses.  Returns the number of
    planned block copies."""
    rc = load().kv_decode_step(alloc, pool, C.cast(seqs, _I32P), n, max_blocks, staging, dev_meta, inputs_h,
                               inputs_d, inputs_bytes, out_h, out_bytes, C.byref(args))
    if rc < 0:
        _check("kv_decode_step", rc)
    return rc


KV_STATIC_SCRATCH_BYTES = 16 << 20


def paged_decode_attention_static(pool: int, layer: int, q: int, out: int, block_tables: int,
                                  max_blocks_per_seq: int, context_lens: int, batch: int,
                                  max_context: int, scale: float, partition_tokens: int,
                                  stream: int = 0) -> None:
    """paged_decode_attention with the library's fixed device scratch instead of a caller
    workspace: for callers that cannot allocate device memory.  The first call on a device
    looks up the scratch address (make it before any stream capture); calls that overlap
    on the GPU race on the shared scratch."""
    _check("paged_decode_attention_static", load().paged_decode_attention_static(
        pool, layer, q, out, block_tables, max_blocks_per_seq, context_lens, batch, max_context,
        scale, partition_tokens, stream))


# ---------------------------------------------------------------- allocator
def kv_alloc_create(num_blocks: int, block_size: int, free_order=None) -> int:
    out = _VP()
    buf = None
    if free_order is not None:
        buf = (C.c_int32 * num_blocks)(*[int(x) for x in free_order])
    _check("kv_alloc_create", load().kv_alloc_create(num_blocks, block_size,
                                                     _i32(buf) if buf is not None else None, C.byref(out)))
    return out.value


def kv_alloc_destroy(a: int) -> None:
    _check("kv_alloc_destroy", load().kv_alloc_destroy(a))


def kv_alloc_seq_new(a: int) -> int:
    sid = C.c_int()
    _check("kv_alloc_seq_new", load().kv_alloc_seq_new(a, C.byref(sid)))
    return sid.value


def kv_alloc_seq_fork(a: int, parent: int) -> int:
    sid = C.c_int()
    _check("kv_alloc_seq_fork", load().kv_alloc_seq_fork(a, parent, C.byref(sid)))
    return sid.value


def kv_alloc_append_slots(a: int, seq: int, count: int):
    """Returns (slots: list[int], cow: (src, dst) or None)."""
    slots = (C.c_int64 * count)()
    pair = (C.c_int32 * 2)()
    _check("kv_alloc_append_slots", load().kv_alloc_append_slots(a, seq, count, _i64(slots), _i32(pair)))
    cow = (pair[0], pair[1]) if pair[0] >= 0 else None
    return list(slots), cow


def kv_alloc_decode_step(a: int, seqs, n: int, slots_out, pairs_out) -> int:
    """seqs: ctypes int32 array of n ids; slots_out: ctypes int64 [n]; pairs_out: ctypes int32
    [2n] (or host addresses).  Returns the number of planned block copies."""
    ncow = C.c_int(0)
    _check("kv_alloc_decode_step", load().kv_alloc_decode_step(a, C.cast(seqs, _I32P), n, C.cast(slots_out, _I64P),
                                                               C.cast(pairs_out, _I32P), C.byref(ncow)))
    return ncow.value


def kv_alloc_seq_trim(a: int, seq: int, keep_from: int) -> int:
    """Release the blocks wholly before token keep_from; returns how many entries were cleared."""
    n = C.c_int(0)
    _check("kv_alloc_seq_trim", load().kv_alloc_seq_trim(a, seq, keep_from, C.byref(n)))
    return n.value


def kv_alloc_seq_free(a: int, seq: int) -> None:
    _check("kv_alloc_seq_free", load().kv_alloc_seq_free(a, seq))


def kv_alloc_seq_info(a: int, seq: int):
    n, nb = C.c_int(), C.c_int()
    _check("kv_alloc_seq_info", load().kv_alloc_seq_info(a, seq, C.byref(n), C.byref(nb)))
    return n.value, nb.value


def kv_alloc_block_table(a: int, seq: int):
    _, nb = kv_alloc_seq_info(a, seq)
    buf = (C.c_int32 * max(nb, 1))()
    n = C.c_int()
    _check("kv_alloc_block_table", load().kv_alloc_block_table(a, seq, _i32(buf), nb, C.byref(n)))
    return list(buf)[: n.value]


def kv_alloc_build_tables(a: int, seqs, max_blocks: int):
    """Returns (tables: list of rows, context_lens: list)."""
    n = len(seqs)
    sbuf = (C.c_int32 * max(n, 1))(*seqs)
    tab = (C.c_int32 * max(n * max_blocks, 1))()
    lens = (C.c_int32 * max(n, 1))()
    _check("kv_alloc_build_tables", load().kv_alloc_build_tables(a, _i32(sbuf), n, _i32(tab), max_blocks,
                                                                 _i32(lens)))
    flat = list(tab)
    return [flat[i * max_blocks:(i + 1) * max_blocks] for i in range(n)], list(lens)[:n]


def kv_alloc_build_tables_into(a: int, seqs, n: int, tables: int, max_blocks: int, context_lens: int) -> None:
    """kv_alloc_build_tables writing into caller memory: seqs a ctypes int32 array of n ids,
    tables / context_lens host addresses of int32 [n][max_blocks] / [n] (e.g. pinned)."""
    _check("kv_alloc_build_tables", load().kv_alloc_build_tables(a, _i32(seqs), n, C.cast(tables, _I32P), max_blocks,
                                                                 C.cast(context_lens, _I32P)))


def kv_alloc_ref_count(a: int, block: int) -> int:
    r = C.c_int()
    _check("kv_alloc_ref_count", load().kv_alloc_ref_count(a, block, C.byref(r)))
    return r.value


def kv_alloc_free_list(a: int, cap: int):
    buf = (C.c_int32 * max(cap, 1))()
    n = C.c_int()
    _check("kv_alloc_free_list", load().kv_alloc_free_list(a, _i32(buf), cap, C.byref(n)))
    return list(buf)[: n.value]


def kv_alloc_stats(a: int) -> kv_alloc_stats_t:
    st = kv_alloc_stats_t()
    _check("kv_alloc_stats", load().kv_alloc_stats(a, C.byref(st)))
    return st
