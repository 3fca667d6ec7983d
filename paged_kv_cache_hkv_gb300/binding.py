"""Thin ctypes binding of libpagedkv.so (C ABI: include/pagedkv.h).

The functions carry the ABI's names and only marshal arguments: torch
tensors become device pointers and the current CUDA stream becomes the
stream handle. Every computation runs in the library's kernels. There is no
CPU path: if the library is missing or the device is not an sm_103 GPU, the
call raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

c_i32, c_i64, c_u32, c_void_p, c_size_t, c_float = (
    ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_void_p, ctypes.c_size_t,
    ctypes.c_float)

PKV_OK = 0
PKV_ERR_SCRATCH_LIMIT = -8
DEVERR_SLOT_RANGE = 0x1
DEVERR_BLOCK_RANGE = 0x2
DEVERR_LENGTHS = 0x4
DEVERR_TIMEOUT = 0x8
DEVERR_SHARED = 0x10


class pkv_cache_layout(ctypes.Structure):
    _fields_ = [("num_blocks", c_i32), ("block_size", c_i32), ("num_kv_heads", c_i32),
                ("head_dim", c_i32)]


PKV_TRACE_EVENTS = 5


class pkv_attention_options(ctypes.Structure):
    _fields_ = [("decode_splits", c_i32), ("shared_prefix_len", c_i32),
                ("shared_first_req", c_i32), ("shared_num_reqs", c_i32),
                ("reserved", c_i32 * 4), ("trace_events", ctypes.POINTER(c_void_p))]


_SIGNATURES = {
    "pkv_abi_version": (c_i32, []),
    "pkv_status_string": (ctypes.c_char_p, [c_i32]),
    "pkv_last_cuda_error": (ctypes.c_char_p, []),
    "pkv_slot_mapping": (c_i32, [c_void_p, c_void_p, c_i32, c_void_p, c_void_p, c_i32, c_i32,
                                 c_i32, c_i32, c_void_p]),
    "pkv_paged_kv_write": (c_i32, [c_void_p, c_void_p, c_void_p, c_i64, c_i64, c_void_p, c_i32,
                                   pkv_cache_layout, c_void_p]),
    "pkv_attention_workspace_size": (c_i64, [c_i32, c_i32, pkv_cache_layout,
                                             ctypes.POINTER(pkv_attention_options)]),
    "pkv_paged_attention": (c_i32, [c_void_p, c_void_p, c_i64, c_void_p, c_void_p, c_i32,
                                    c_void_p, c_void_p, c_void_p, c_i32, c_i32, c_i32, c_i32,
                                    c_i32, c_float, pkv_cache_layout, c_void_p, c_size_t,
                                    ctypes.POINTER(pkv_attention_options), c_void_p]),
    "pkv_get_device_errors": (c_i32, [ctypes.POINTER(c_u32), c_i32, c_void_p]),
    "pkv_copy_blocks": (c_i32, [c_void_p, c_i32, c_void_p, c_i32, c_void_p, c_i32,
                                pkv_cache_layout, c_void_p]),
    "pkv_slot_mapping_and_write": (c_i32, [c_void_p, c_void_p, c_void_p, c_i64, c_i64, c_void_p,
                                           c_void_p, c_i32, c_void_p, c_void_p, c_i32, c_i32,
                                           pkv_cache_layout, c_void_p]),
    "pkv_paged_attention_with_write": (
        c_i32, [c_void_p, c_void_p, c_i64, c_void_p, c_void_p, c_void_p, c_i64, c_i64, c_void_p,
                c_void_p, c_i32, c_void_p, c_void_p, c_void_p, c_i32, c_i32, c_i32, c_i32, c_i32,
                c_float, pkv_cache_layout, c_void_p, c_size_t,
                ctypes.POINTER(pkv_attention_options), c_void_p]),
    "pkv_paged_attention_static_workspace": (
        c_i32, [c_void_p, c_void_p, c_i64, c_void_p, c_void_p, c_i32, c_void_p, c_void_p,
                c_void_p, c_i32, c_i32, c_i32, c_i32, c_i32, c_float, pkv_cache_layout,
                ctypes.POINTER(pkv_attention_options), c_void_p]),
}

_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libpagedkv.so (building it first when it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing and not _build.up_to_date():
        _build.build_library()
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built; run paged_kv_cache_hkv_gb300.build")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class PagedKVError(RuntimeError):
    def __init__(self, name, status):
        lib = load()
        msg = lib.pkv_status_string(status).decode()
        extra = lib.pkv_last_cuda_error().decode()
        super().__init__(f"{name} failed: {msg} ({status})" + (f": {extra}" if extra else ""))
        self.status = status


def _check(name, status):
    if status != PKV_OK:
        raise PagedKVError(name, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _require(t, dtype, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def layout_of(kv_cache: torch.Tensor) -> pkv_cache_layout:
    """Layout struct of a pool tensor [num_blocks, 2, block_size, Hkv, D]."""
    if kv_cache.dim() != 5 or kv_cache.shape[1] != 2 or not kv_cache.is_contiguous():
        raise ValueError("kv_cache must be a contiguous [num_blocks, 2, block_size, Hkv, D] tensor")
    nb, _, bs, hkv, d = kv_cache.shape
    return pkv_cache_layout(nb, bs, hkv, d)


def abi_version() -> int:
    return load().pkv_abi_version()


def pkv_slot_mapping(slot_mapping, block_table, query_start_loc, num_computed_tokens,
                     num_blocks: int, block_size: int = 16, stream=None):
    """slot_mapping (int64 [T]) <- slot of each new token (see pagedkv.h)."""
    _require(slot_mapping, torch.int64, "slot_mapping")
    for t, n in ((block_table, "block_table"), (query_start_loc, "query_start_loc"),
                 (num_computed_tokens, "num_computed_tokens")):
        _require(t, torch.int32, n)
    if not block_table.is_contiguous():
        raise ValueError("block_table must be contiguous")
    _check("pkv_slot_mapping", load().pkv_slot_mapping(
        _ptr(slot_mapping), _ptr(block_table), block_table.shape[1], _ptr(query_start_loc),
        _ptr(num_computed_tokens), num_computed_tokens.shape[0], slot_mapping.shape[0],
        num_blocks, block_size, _stream(stream)))
    return slot_mapping


def pkv_paged_kv_write(kv_cache, key, value, slot_mapping, stream=None):
    """Scatter key/value rows ([T, Hkv, D] bf16, row-strided allowed) into the pool."""
    for t, n in ((kv_cache, "kv_cache"), (key, "key"), (value, "value")):
        _require(t, torch.bfloat16, n)
    _require(slot_mapping, torch.int64, "slot_mapping")
    for t, n in ((key, "key"), (value, "value")):
        if t.dim() != 3 or t.stride(2) != 1 or t.stride(1) != t.shape[2]:
            raise ValueError(f"{n} must be [T, Hkv, D] with contiguous rows")
    lay = layout_of(kv_cache)
    _check("pkv_paged_kv_write", load().pkv_paged_kv_write(
        _ptr(kv_cache), _ptr(key), _ptr(value), key.stride(0), value.stride(0),
        _ptr(slot_mapping), key.shape[0], lay, _stream(stream)))


def pkv_slot_mapping_and_write(kv_cache, key, value, block_table, query_start_loc,
                               num_computed_tokens, slot_mapping=None, stream=None):
    """Slot mapping and cache write in one launch (see pagedkv.h). slot_mapping
    (int64 [T]) receives the slots when given."""
    for t, n in ((kv_cache, "kv_cache"), (key, "key"), (value, "value")):
        _require(t, torch.bfloat16, n)
    for t, n in ((block_table, "block_table"), (query_start_loc, "query_start_loc"),
                 (num_computed_tokens, "num_computed_tokens")):
        _require(t, torch.int32, n)
    if slot_mapping is not None:
        _require(slot_mapping, torch.int64, "slot_mapping")
    for t, n in ((key, "key"), (value, "value")):
        if t.dim() != 3 or t.stride(2) != 1 or t.stride(1) != t.shape[2]:
            raise ValueError(f"{n} must be [T, Hkv, D] with contiguous rows")
    if not block_table.is_contiguous():
        raise ValueError("block_table must be contiguous")
    lay = layout_of(kv_cache)
    _check("pkv_slot_mapping_and_write", load().pkv_slot_mapping_and_write(
        _ptr(kv_cache), _ptr(key), _ptr(value), key.stride(0), value.stride(0),
        _ptr(slot_mapping), _ptr(block_table), block_table.shape[1], _ptr(query_start_loc),
        _ptr(num_computed_tokens), num_computed_tokens.shape[0], key.shape[0], lay,
        _stream(stream)))
    return slot_mapping


def pkv_copy_blocks(dst_pool, src_pool, block_pairs, stream=None):
    """dst_pool[d] = src_pool[s] for each (s, d) row of block_pairs (int32
    [n, 2] on the device). Pools are CUDA tensors or pinned host tensors."""
    for t, n in ((dst_pool, "dst_pool"), (src_pool, "src_pool")):
        if t.dtype != torch.bfloat16:
            raise ValueError(f"{n} must be bfloat16")
        if not (t.is_cuda or t.is_pinned()):
            raise ValueError(f"{n} must be a CUDA tensor or pinned host memory")
    _require(block_pairs, torch.int32, "block_pairs")
    if block_pairs.dim() != 2 or block_pairs.shape[1] != 2 or not block_pairs.is_contiguous():
        raise ValueError("block_pairs must be a contiguous [n, 2] int32 tensor")
    lay = layout_of(src_pool)
    if tuple(dst_pool.shape[1:]) != tuple(src_pool.shape[1:]) or not dst_pool.is_contiguous():
        raise ValueError("pools must share the block shape")
    _check("pkv_copy_blocks", load().pkv_copy_blocks(
        _ptr(dst_pool), dst_pool.shape[0], _ptr(src_pool), src_pool.shape[0],
        _ptr(block_pairs), block_pairs.shape[0], lay, _stream(stream)))


def _options(decode_splits, trace_events=None, shared_prefix=None):
    """Options struct (or None for the defaults). shared_prefix: None, or
    (shared_prefix_len, shared_first_req, shared_num_reqs) -- see pagedkv.h."""
    if decode_splits is None and trace_events is None and shared_prefix is None:
        return None
    o = pkv_attention_options()
    o.decode_splits = int(decode_splits or 0)
    if shared_prefix is not None:
        o.shared_prefix_len, o.shared_first_req, o.shared_num_reqs = (int(x) for x in shared_prefix)
    if trace_events is not None:
        if len(trace_events) != PKV_TRACE_EVENTS:
            raise ValueError(f"trace_events needs {PKV_TRACE_EVENTS} torch.cuda.Event")
        handles = [e.cuda_event for e in trace_events]
        if not all(handles):
            raise ValueError("trace events must be created (recorded once) before use")
        arr = (c_void_p * PKV_TRACE_EVENTS)(*[c_void_p(h) for h in handles])
        o.trace_events = ctypes.cast(arr, ctypes.POINTER(c_void_p))
        o._keep = arr
    return ctypes.pointer(o)


def pkv_attention_workspace_size(num_reqs: int, num_q_heads: int, kv_cache,
                                 decode_splits=None, shared_prefix=None) -> int:
    """Workspace bytes for pkv_paged_attention; kv_cache is the pool tensor
    or a pkv_cache_layout."""
    lay = kv_cache if isinstance(kv_cache, pkv_cache_layout) else layout_of(kv_cache)
    n = load().pkv_attention_workspace_size(num_reqs, num_q_heads, lay,
                                            _options(decode_splits, None, shared_prefix))
    if n < 0:
        raise PagedKVError("pkv_attention_workspace_size", int(n))
    return int(n)


def pkv_paged_attention(out, q, kv_cache, block_table, seq_lens, query_start_loc,
                        num_computed_tokens, *, max_query_len: int, max_seq_len: int,
                        scale: float, workspace, decode_splits=None, trace_events=None,
                        shared_prefix=None, stream=None):
    """out [T, Hq, D] bf16 <- attention of one mixed step (see pagedkv.h).

    trace_events: optional list of PKV_TRACE_EVENTS torch.cuda.Event (created
    with enable_timing=True) recorded around the call's kernels."""
    for t, n in ((out, "out"), (q, "q"), (kv_cache, "kv_cache")):
        _require(t, torch.bfloat16, n)
    for t, n in ((block_table, "block_table"), (seq_lens, "seq_lens"),
                 (query_start_loc, "query_start_loc"),
                 (num_computed_tokens, "num_computed_tokens")):
        _require(t, torch.int32, n)
    if not out.is_contiguous() or not block_table.is_contiguous():
        raise ValueError("out and block_table must be contiguous")
    if q.dim() != 3 or q.stride(2) != 1 or q.stride(1) != q.shape[2]:
        raise ValueError("q must be [T, Hq, D] with contiguous rows")
    lay = layout_of(kv_cache)
    _check("pkv_paged_attention", load().pkv_paged_attention(
        _ptr(out), _ptr(q), q.stride(0), _ptr(kv_cache), _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), _ptr(query_start_loc), _ptr(num_computed_tokens),
        seq_lens.shape[0], q.shape[0], int(max_query_len), int(max_seq_len), q.shape[1],
        float(scale), lay, _ptr(workspace), workspace.numel() * workspace.element_size(),
        _options(decode_splits, trace_events, shared_prefix), _stream(stream)))
    return out


def pkv_paged_attention_with_write(out, q, kv_cache, key, value, block_table, seq_lens,
                                   query_start_loc, num_computed_tokens, *, max_query_len: int,
                                   max_seq_len: int, scale: float, workspace, slot_mapping=None,
                                   decode_splits=None, trace_events=None, shared_prefix=None,
                                   stream=None):
    """The step of one layer in one call: slot mapping and cache write of the
    new tokens, then attention (see pagedkv.h). slot_mapping (int64 [T])
    receives the slots when given."""
    for t, n in ((out, "out"), (q, "q"), (kv_cache, "kv_cache"), (key, "key"),
                 (value, "value")):
        _require(t, torch.bfloat16, n)
    for t, n in ((block_table, "block_table"), (seq_lens, "seq_lens"),
                 (query_start_loc, "query_start_loc"),
                 (num_computed_tokens, "num_computed_tokens")):
        _require(t, torch.int32, n)
    if slot_mapping is not None:
        _require(slot_mapping, torch.int64, "slot_mapping")
    if not out.is_contiguous() or not block_table.is_contiguous():
        raise ValueError("out and block_table must be contiguous")
    for t, n in ((q, "q"), (key, "key"), (value, "value")):
        if t.dim() != 3 or t.stride(2) != 1 or t.stride(1) != t.shape[2]:
            raise ValueError(f"{n} must be [T, H, D] with contiguous rows")
    if key.shape[0] != q.shape[0]:
        raise ValueError("key and q must have the same number of rows")
    lay = layout_of(kv_cache)
    _check("pkv_paged_attention_with_write", load().pkv_paged_attention_with_write(
        _ptr(out), _ptr(q), q.stride(0), _ptr(kv_cache), _ptr(key), _ptr(value), key.stride(0),
        value.stride(0), _ptr(slot_mapping), _ptr(block_table), block_table.shape[1],
        _ptr(seq_lens), _ptr(query_start_loc), _ptr(num_computed_tokens), seq_lens.shape[0],
        q.shape[0], int(max_query_len), int(max_seq_len), q.shape[1], float(scale), lay,
        _ptr(workspace), workspace.numel() * workspace.element_size(),
        _options(decode_splits, trace_events, shared_prefix), _stream(stream)))
    return out


def pkv_get_device_errors(clear: bool = True, stream=None) -> int:
    """Synchronise and read (optionally clear) the sticky device error bits."""
    v = c_u32(0)
    _check("pkv_get_device_errors",
           load().pkv_get_device_errors(ctypes.byref(v), int(clear), _stream(stream)))
    return int(v.value)


def pkv_paged_attention_static_workspace(out, q, kv_cache, block_table, seq_lens,
                                         query_start_loc, num_computed_tokens, *,
                                         max_query_len: int, max_seq_len: int, scale: float,
                                         decode_splits=None, shared_prefix=None, stream=None):
    """pkv_paged_attention without a caller workspace: for callers that cannot
    allocate device memory, the library uses its built-in scratch array (see
    pagedkv.h for the size limit and the one-stream rule)."""
    for t, n in ((out, "out"), (q, "q"), (kv_cache, "kv_cache")):
        _require(t, torch.bfloat16, n)
    for t, n in ((block_table, "block_table"), (seq_lens, "seq_lens"),
                 (query_start_loc, "query_start_loc"),
                 (num_computed_tokens, "num_computed_tokens")):
        _require(t, torch.int32, n)
    if not out.is_contiguous() or not block_table.is_contiguous():
        raise ValueError("out and block_table must be contiguous")
    if q.dim() != 3 or q.stride(2) != 1 or q.stride(1) != q.shape[2]:
        raise ValueError("q must be [T, Hq, D] with contiguous rows")
    _check("pkv_paged_attention_static_workspace", load().pkv_paged_attention_static_workspace(
        _ptr(out), _ptr(q), q.stride(0), _ptr(kv_cache), _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), _ptr(query_start_loc), _ptr(num_computed_tokens),
        seq_lens.shape[0], q.shape[0], int(max_query_len), int(max_seq_len), q.shape[1],
        float(scale), layout_of(kv_cache), _options(decode_splits, None, shared_prefix),
        _stream(stream)))
    return out


class StepCalls:
    """The calls of one step -- pkv_slot_mapping, pkv_paged_kv_write,
    pkv_paged_attention; with fused_write pkv_slot_mapping_and_write then
    pkv_paged_attention; with write_in_attention the one call
    pkv_paged_attention_with_write -- with their arguments checked and
    marshalled once.

    A serving loop that keeps its step buffers (as DeviceStep does) pays the
    argument checks and the tensor-to-pointer conversion once, not on every
    step; ``run`` then makes the three C calls in a row on the given stream.
    The buffers must stay allocated and keep their shapes while the object is
    used."""

    def __init__(self, *, slot_mapping, block_table, query_start_loc, num_computed_tokens,
                 kv_cache, key, value, out, q, seq_lens, max_query_len: int,
                 max_seq_len: int, scale: float, workspace, decode_splits=None,
                 shared_prefix=None, fused_write=False, write_in_attention=False):
        _require(slot_mapping, torch.int64, "slot_mapping")
        for t, n in ((block_table, "block_table"), (query_start_loc, "query_start_loc"),
                     (num_computed_tokens, "num_computed_tokens"), (seq_lens, "seq_lens")):
            _require(t, torch.int32, n)
        for t, n in ((kv_cache, "kv_cache"), (key, "key"), (value, "value"), (out, "out"),
                     (q, "q")):
            _require(t, torch.bfloat16, n)
        for t, n in ((key, "key"), (value, "value"), (q, "q")):
            if t.dim() != 3 or t.stride(2) != 1 or t.stride(1) != t.shape[2]:
                raise ValueError(f"{n} must be [T, H, D] with contiguous rows")
        if not out.is_contiguous() or not block_table.is_contiguous():
            raise ValueError("out and block_table must be contiguous")
        lay = layout_of(kv_cache)
        self.lib = load()
        self._opts = _options(decode_splits, None, shared_prefix)
        self.slot_args = (
            _ptr(slot_mapping), _ptr(block_table), block_table.shape[1], _ptr(query_start_loc),
            _ptr(num_computed_tokens), num_computed_tokens.shape[0], slot_mapping.shape[0],
            lay.num_blocks, lay.block_size)
        self.write_args = (
            _ptr(kv_cache), _ptr(key), _ptr(value), key.stride(0), value.stride(0),
            _ptr(slot_mapping), key.shape[0], lay)
        self.fused_write = bool(fused_write)
        self.write_in_attention = bool(write_in_attention)
        if self.write_in_attention and key.shape[0] != q.shape[0]:
            raise ValueError("key and q must have the same number of rows")
        self.mapped_write_args = (
            _ptr(kv_cache), _ptr(key), _ptr(value), key.stride(0), value.stride(0),
            _ptr(slot_mapping), _ptr(block_table), block_table.shape[1], _ptr(query_start_loc),
            _ptr(num_computed_tokens), num_computed_tokens.shape[0], key.shape[0], lay)
        self.attn_args = (
            _ptr(out), _ptr(q), q.stride(0), _ptr(kv_cache), _ptr(block_table),
            block_table.shape[1], _ptr(seq_lens), _ptr(query_start_loc),
            _ptr(num_computed_tokens), seq_lens.shape[0], q.shape[0], int(max_query_len),
            int(max_seq_len), q.shape[1], float(scale), lay, _ptr(workspace),
            workspace.numel() * workspace.element_size(), self._opts)
        self.attn_write_args = (
            _ptr(out), _ptr(q), q.stride(0), _ptr(kv_cache), _ptr(key), _ptr(value),
            key.stride(0), value.stride(0), _ptr(slot_mapping), _ptr(block_table),
            block_table.shape[1], _ptr(seq_lens), _ptr(query_start_loc),
            _ptr(num_computed_tokens), seq_lens.shape[0], q.shape[0], int(max_query_len),
            int(max_seq_len), q.shape[1], float(scale), lay, _ptr(workspace),
            workspace.numel() * workspace.element_size(), self._opts)
        # the tensors stay referenced, so their memory stays valid
        self._keep = (slot_mapping, block_table, query_start_loc, num_computed_tokens,
                      kv_cache, key, value, out, q, seq_lens, workspace)

    def slot_map(self, stream=None):
        status = self.lib.pkv_slot_mapping(*self.slot_args, _stream(stream))
        if status:
            raise PagedKVError("pkv_slot_mapping", status)

    def write(self, stream=None):
        status = self.lib.pkv_paged_kv_write(*self.write_args, _stream(stream))
        if status:
            raise PagedKVError("pkv_paged_kv_write", status)

    def slot_map_and_write(self, stream=None):
        status = self.lib.pkv_slot_mapping_and_write(*self.mapped_write_args, _stream(stream))
        if status:
            raise PagedKVError("pkv_slot_mapping_and_write", status)

    def attend(self, stream=None):
        status = self.lib.pkv_paged_attention(*self.attn_args, _stream(stream))
        if status:
            raise PagedKVError("pkv_paged_attention", status)

    def run(self, stream=None):
        st = _stream(stream)
        lib = self.lib
        if self.write_in_attention:
            status = lib.pkv_paged_attention_with_write(*self.attn_write_args, st)
            if status:
                raise PagedKVError("pkv_paged_attention_with_write", status)
            return
        if self.fused_write:
            status = lib.pkv_slot_mapping_and_write(*self.mapped_write_args, st)
            if status:
                raise PagedKVError("pkv_slot_mapping_and_write", status)
        else:
            status = lib.pkv_slot_mapping(*self.slot_args, st)
            if status:
                raise PagedKVError("pkv_slot_mapping", status)
            status = lib.pkv_paged_kv_write(*self.write_args, st)
            if status:
                raise PagedKVError("pkv_paged_kv_write", status)
        status = lib.pkv_paged_attention(*self.attn_args, st)
        if status:
            raise PagedKVError("pkv_paged_attention", status)
