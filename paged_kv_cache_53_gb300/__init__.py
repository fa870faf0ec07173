"""Python binding of libpagedattn, the sm_103a paged KV-cache attention library.

Argument marshalling only: each function reads shapes, dtypes and data pointers off torch
tensors and calls the C entry point of the same name declared in include/pa.h.  Every
step of the path runs in the library's CUDA kernels; there is no CPU or PyTorch
fallback, and a missing or unloadable library raises.

Tensors must be contiguous CUDA tensors on the current device.  Calls are asynchronous on
the current torch stream unless `stream` (a torch.cuda.Stream) is given.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence

import torch

from .build import LIB as LIB_PATH

__all__ = [
    "PA_F32", "PA_F16", "PA_BF16", "PaError", "lib", "dtype_code",
    "slot_mapping", "reshape_and_cache", "cache_append", "copy_blocks", "swap_blocks",
    "decode_workspace_bytes",
    "decode", "decode_shared_prefix_workspace_bytes", "decode_shared_prefix",
    "prefill_workspace_bytes", "prefill_chunk", "get_status", "version",
    "set_stream_status", "release_thread_resources",
    "testing_decode_workspace_bytes", "testing_decode_partitions",
    "STATUS_BAD_BLOCK", "STATUS_BAD_SLOT", "STATUS_BAD_CONTEXT", "STATUS_TIMEOUT", "STATUS_RANGE",
]

PA_F32, PA_F16, PA_BF16 = 0, 1, 2
STATUS_BAD_BLOCK, STATUS_BAD_SLOT, STATUS_BAD_CONTEXT, STATUS_TIMEOUT = 0x1, 0x2, 0x4, 0x8
STATUS_RANGE = 0x10  # reserved: no longer set
_ERRORS = {1: "PA_ERR_INVALID_ARG", 2: "PA_ERR_UNSUPPORTED", 3: "PA_ERR_WORKSPACE",
           4: "PA_ERR_CUDA"}

_DT = {torch.float32: PA_F32, torch.float16: PA_F16, torch.bfloat16: PA_BF16}


class PaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{_ERRORS.get(code, code)}: {msg}")
        self.code = code


_lib = None
_lock = threading.Lock()

_i, _u64, _f, _p, _sz = ctypes.c_int, ctypes.c_uint64, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t

_SIGNATURES = {
    "pa_version": ([], _i),
    "pa_last_error_string": ([], ctypes.c_char_p),
    "pa_get_status": ([_p], _i),
    "pa_set_stream_status": ([_p, _p], _i),
    "pa_release_thread_resources": ([], _i),
    "pa_testing_decode_workspace_bytes": ([_i, _i, _i, _i, _i, _i, _i], _sz),
    "pa_testing_decode_partitions": ([_p, _i, _p, _p, _p, _p, _i, _p, _i, _i, _i, _i, _i, _i,
                                      _i, _f, _i, _i, _p, _sz, _p], _i),
    "pa_selftest_wait_timeout": ([_i, _p], _i),
    "pa_mixed_step": ([_p, _p, _p, _p, _i, _i, _i, _i, _i, _f, _i, _p], _i),
    "pa_slot_mapping": ([_p, _p, _i, _p, _p, _i, _i, _i, _i, _p], _i),
    "pa_reshape_and_cache": ([_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _p], _i),
    "pa_copy_blocks": ([_p, _p, _i, _p, _i, _i, _i, _i, _i, _i, _p], _i),
    "pa_swap_blocks": ([_p, _p, _p, _p, _i, _p, _i, _i, _i, _i, _i, _i, _i, _p], _i),
    "pa_cache_append": ([_p, _p, _p, _p, _p, _p, _i, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i,
                         _p], _i),
    "pa_decode_workspace_bytes": ([_i, _i, _i, _i, _i, _i], _sz),
    "pa_decode_shared_prefix_workspace_bytes": ([_i, _i, _i, _i, _i, _i, _i, _i], _sz),
    "pa_decode_shared_prefix": ([_p, _i, _p, _p, _p, _p, _i, _p, _i, _i, _i, _i, _i, _i, _i,
                                 _p, _i, _p, _i, _f, _i, _p, _sz, _p], _i),
    "pa_decode": ([_p, _i, _p, _p, _p, _p, _i, _p, _i, _i, _i, _i, _i, _i, _i, _f, _i, _p, _sz,
                   _p], _i),
    "pa_decode_append": ([_p, _i, _p, _p, _p, _p, _p, _p, _p, _i, _p, _i, _i, _i, _i, _i, _i,
                          _i, _f, _i, _p, _sz, _p], _i),
    "pa_prefill_workspace_bytes": ([_i, _i, _i, _i, _i, _i, _i, _i], _sz),
    "pa_prefill_chunk": ([_p, _i, _p, _p, _p, _p, _i, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i,
                          _i, _f, _i, _p, _sz, _p], _i),
}


def lib(path: Optional[str] = None):
    """Loads libpagedattn.so once (raising if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise ImportError(
                    f"libpagedattn.so is not built ({p}); build it with "
                    "`python -m paged_kv_cache_53_gb300.build`")
            handle = ctypes.CDLL(p)
            for name, (args, res) in _SIGNATURES.items():
                fn = getattr(handle, name)
                fn.argtypes = args
                fn.restype = res
            _lib = handle
    return _lib


def version() -> int:
    return lib().pa_version()


def _check(rc: int):
    if rc != 0:
        raise PaError(rc, lib().pa_last_error_string().decode())


def dtype_code(t: torch.dtype) -> int:
    try:
        return _DT[t]
    except KeyError:
        raise TypeError(f"unsupported dtype {t}") from None


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to libpagedattn must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _i32(t: torch.Tensor, name: str):
    if t.dtype != torch.int32:
        raise TypeError(f"{name} must be int32")


def slot_mapping(slots: torch.Tensor, block_tables: torch.Tensor, cu_q_lens: torch.Tensor,
                 context_lens: torch.Tensor, block_size: int, num_blocks: int, stream=None):
    """slots[t] (int64) = physical slot of new token t (see pa_slot_mapping)."""
    _i32(block_tables, "block_tables")
    if slots.dtype != torch.int64:
        raise TypeError("slots must be int64")
    _check(lib().pa_slot_mapping(_ptr(slots), _ptr(block_tables), block_tables.shape[1],
                                 _ptr(cu_q_lens), _ptr(context_lens), context_lens.shape[0],
                                 slots.shape[0], block_size, num_blocks, _stream(stream)))


def reshape_and_cache(k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                      v_cache: torch.Tensor, slots: torch.Tensor, stream=None):
    """Writes k_new/v_new [T, H_kv, D] into the caches [NB, H_kv, BS, D] at `slots`."""
    nb, h_kv, bs, d = k_cache.shape
    _check(lib().pa_reshape_and_cache(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                      _ptr(slots), k_new.shape[0], h_kv, d, bs, nb,
                                      dtype_code(k_cache.dtype), _stream(stream)))


def cache_append(k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                 v_cache: torch.Tensor, block_tables: torch.Tensor, cu_q_lens: torch.Tensor,
                 context_lens: torch.Tensor, max_q: int, slots: Optional[torch.Tensor] = None,
                 stream=None):
    """Slot mapping and cache write of the step's new tokens in one launch."""
    nb, h_kv, bs, d = k_cache.shape
    _i32(block_tables, "block_tables")
    if slots is not None and slots.dtype != torch.int64:
        raise TypeError("slots must be int64")
    _check(lib().pa_cache_append(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                 _ptr(slots), _ptr(block_tables), block_tables.shape[1],
                                 _ptr(cu_q_lens), _ptr(context_lens), context_lens.shape[0],
                                 k_new.shape[0], max_q, h_kv, d, bs, nb,
                                 dtype_code(k_cache.dtype), _stream(stream)))


def copy_blocks(k_caches: Sequence[torch.Tensor], v_caches: Sequence[torch.Tensor],
                pairs: torch.Tensor, stream=None):
    """Block dst <- block src for every (src, dst) row of `pairs`, in every layer."""
    n = len(k_caches)
    if n != len(v_caches) or n == 0:
        raise ValueError("need the same non-zero number of K and V caches")
    nb, h_kv, bs, d = k_caches[0].shape
    karr = (ctypes.c_void_p * n)(*[_ptr(t) for t in k_caches])
    varr = (ctypes.c_void_p * n)(*[_ptr(t) for t in v_caches])
    _check(lib().pa_copy_blocks(karr, varr, n, _ptr(pairs), pairs.shape[0], h_kv, d, bs, nb,
                                dtype_code(k_caches[0].dtype), _stream(stream)))


def swap_blocks(src_k: Sequence[torch.Tensor], src_v: Sequence[torch.Tensor],
                dst_k: Sequence[torch.Tensor], dst_v: Sequence[torch.Tensor],
                pairs: torch.Tensor, stream=None):
    """Block dst of every destination pool <- block src of the matching source pool, for
    every (src, dst) row of `pairs` (see pa_swap_blocks).  Pools are CUDA tensors or
    pinned CPU tensors of one geometry [blocks, H_kv, block_size, D]."""
    n = len(src_k)
    if not (n == len(src_v) == len(dst_k) == len(dst_v)) or n == 0:
        raise ValueError("need the same non-zero number of pools on every side")
    _i32(pairs, "pairs")
    if pairs.device.type == "cpu" and not pairs.is_pinned():
        raise ValueError("pairs must be a CUDA tensor or a pinned CPU tensor")
    nbs, h_kv, bs, d = src_k[0].shape
    nbd = dst_k[0].shape[0]
    arr = lambda ts: (ctypes.c_void_p * n)(*[_ptr(t) for t in ts])
    _check(lib().pa_swap_blocks(arr(src_k), arr(src_v), arr(dst_k), arr(dst_v), n, _ptr(pairs),
                                pairs.shape[0], h_kv, d, bs, nbs, nbd,
                                dtype_code(src_k[0].dtype), _stream(stream)))


def decode_workspace_bytes(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                           max_ctx: int, block_size: int) -> int:
    return int(lib().pa_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                               max_ctx, block_size))


def decode(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
           block_tables: torch.Tensor, context_lens: torch.Tensor, max_ctx: int, scale: float,
           workspace: torch.Tensor, stream=None):
    """Paged decode attention (see pa_decode); `workspace` is a uint8 device tensor of at
    least decode_workspace_bytes(...) bytes."""
    nb, h_kv, bs, d = k_cache.shape
    b, h_q, _ = q.shape
    _check(lib().pa_decode(_ptr(out), dtype_code(out.dtype), _ptr(q), _ptr(k_cache),
                           _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
                           _ptr(context_lens), max_ctx, b, h_q, h_kv, d, bs, nb, float(scale),
                           dtype_code(k_cache.dtype), _ptr(workspace),
                           workspace.numel() * workspace.element_size(), _stream(stream)))


def decode_append(out: torch.Tensor, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                  k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                  context_lens: torch.Tensor, max_ctx: int, scale: float,
                  workspace: torch.Tensor, slots: Optional[torch.Tensor] = None, stream=None):
    """One decode step (see pa_decode_append): row b of k_new / v_new is written at
    position context_lens[b] - 1 of sequence b (its slot into `slots` if given), then the
    decode attends over every context."""
    nb, h_kv, bs, d = k_cache.shape
    b, h_q, _ = q.shape
    if slots is not None and slots.dtype != torch.int64:
        raise TypeError("slots must be int64")
    _check(lib().pa_decode_append(_ptr(out), dtype_code(out.dtype), _ptr(q), _ptr(k_new),
                                  _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(slots),
                                  _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
                                  max_ctx, b, h_q, h_kv, d, bs, nb, float(scale),
                                  dtype_code(k_cache.dtype), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream)))


class _DecodeBatch(ctypes.Structure):
    """pa_decode_batch of include/pa.h."""
    _fields_ = [("out", ctypes.c_void_p), ("out_dtype", ctypes.c_int), ("q", ctypes.c_void_p),
                ("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p),
                ("slots", ctypes.c_void_p), ("block_tables", ctypes.c_void_p),
                ("max_blocks_per_seq", ctypes.c_int), ("context_lens", ctypes.c_void_p),
                ("max_ctx", ctypes.c_int), ("num_seqs", ctypes.c_int),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t)]


class _PrefillBatch(ctypes.Structure):
    """pa_prefill_batch of include/pa.h."""
    _fields_ = [("out", ctypes.c_void_p), ("out_dtype", ctypes.c_int), ("q", ctypes.c_void_p),
                ("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p),
                ("slots", ctypes.c_void_p), ("block_tables", ctypes.c_void_p),
                ("max_blocks_per_seq", ctypes.c_int), ("cu_q_lens", ctypes.c_void_p),
                ("context_lens", ctypes.c_void_p), ("max_q", ctypes.c_int),
                ("max_ctx", ctypes.c_int), ("num_seqs", ctypes.c_int),
                ("num_tokens", ctypes.c_int), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t)]


def mixed_step(k_cache: torch.Tensor, v_cache: torch.Tensor, scale: float,
               decode: Optional[dict] = None, prefill: Optional[dict] = None, stream=None):
    """One step of a batch of decodes and prefill chunks run side by side (see
    pa_mixed_step).  `decode`: out, q, k_new, v_new, block_tables, context_lens, max_ctx,
    workspace[, slots]; `prefill`: the same plus cu_q_lens and max_q (k_new / v_new hold the
    chunks' new tokens)."""
    nb, h_kv, bs, d = k_cache.shape
    h_q = None
    dp = pp = None
    if decode is not None:
        m = decode
        h_q = m["q"].shape[1]
        ws = m["workspace"]
        dp = _DecodeBatch(_ptr(m["out"]), dtype_code(m["out"].dtype), _ptr(m["q"]),
                          _ptr(m["k_new"]), _ptr(m["v_new"]), _ptr(m.get("slots")),
                          _ptr(m["block_tables"]), m["block_tables"].shape[1],
                          _ptr(m["context_lens"]), int(m["max_ctx"]), m["q"].shape[0],
                          _ptr(ws), ws.numel() * ws.element_size())
    if prefill is not None:
        m = prefill
        h_q = m["q"].shape[1]
        ws = m["workspace"]
        pp = _PrefillBatch(_ptr(m["out"]), dtype_code(m["out"].dtype), _ptr(m["q"]),
                           _ptr(m["k_new"]), _ptr(m["v_new"]), _ptr(m.get("slots")),
                           _ptr(m["block_tables"]), m["block_tables"].shape[1],
                           _ptr(m["cu_q_lens"]), _ptr(m["context_lens"]), int(m["max_q"]),
                           int(m["max_ctx"]), m["cu_q_lens"].shape[0] - 1, m["q"].shape[0],
                           _ptr(ws), ws.numel() * ws.element_size())
    if h_q is None:
        return
    _check(lib().pa_mixed_step(ctypes.byref(dp) if dp is not None else None,
                               ctypes.byref(pp) if pp is not None else None, _ptr(k_cache),
                               _ptr(v_cache), h_q, h_kv, d, bs, nb, float(scale),
                               dtype_code(k_cache.dtype), _stream(stream)))


def decode_shared_prefix_workspace_bytes(num_seqs: int, num_q_heads: int, num_kv_heads: int,
                                         head_dim: int, max_ctx: int, block_size: int,
                                         num_sharers: int, prefix_len: int) -> int:
    return int(lib().pa_decode_shared_prefix_workspace_bytes(
        num_seqs, num_q_heads, num_kv_heads, head_dim, max_ctx, block_size, num_sharers,
        prefix_len))


def decode_shared_prefix(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                         v_cache: torch.Tensor, block_tables: torch.Tensor,
                         context_lens: torch.Tensor, max_ctx: int, prefix_blocks: torch.Tensor,
                         prefix_len: int, sharers: torch.Tensor, scale: float,
                         workspace: torch.Tensor, stream=None):
    """pa_decode with the prefix shared by the rows in `sharers` attended once per KV head
    (see pa_decode_shared_prefix)."""
    nb, h_kv, bs, d = k_cache.shape
    b, h_q, _ = q.shape
    _i32(prefix_blocks, "prefix_blocks")
    _i32(sharers, "sharers")
    _check(lib().pa_decode_shared_prefix(
        _ptr(out), dtype_code(out.dtype), _ptr(q), _ptr(k_cache), _ptr(v_cache),
        _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), max_ctx, b, h_q, h_kv, d,
        bs, nb, _ptr(prefix_blocks), prefix_len, _ptr(sharers), sharers.shape[0], float(scale),
        dtype_code(k_cache.dtype), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def prefill_workspace_bytes(num_seqs: int, num_tokens: int, max_q: int, num_q_heads: int,
                            num_kv_heads: int, head_dim: int, max_ctx: int,
                            block_size: int) -> int:
    return int(lib().pa_prefill_workspace_bytes(num_seqs, num_tokens, max_q, num_q_heads,
                                                num_kv_heads, head_dim, max_ctx, block_size))


def prefill_chunk(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                  v_cache: torch.Tensor, block_tables: torch.Tensor, cu_q_lens: torch.Tensor,
                  context_lens: torch.Tensor, max_q: int, max_ctx: int, scale: float,
                  workspace: Optional[torch.Tensor] = None, stream=None):
    """Causal chunked-prefill attention over paged context (see pa_prefill_chunk)."""
    nb, h_kv, bs, d = k_cache.shape
    t, h_q, _ = q.shape
    ws_ptr = _ptr(workspace) if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().pa_prefill_chunk(_ptr(out), dtype_code(out.dtype), _ptr(q), _ptr(k_cache),
                                  _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
                                  _ptr(cu_q_lens), _ptr(context_lens), context_lens.shape[0], t,
                                  max_q, max_ctx, h_q, h_kv, d, bs, nb, float(scale),
                                  dtype_code(k_cache.dtype), ws_ptr, ws_bytes, _stream(stream)))


def testing_decode_workspace_bytes(num_seqs: int, num_q_heads: int, num_kv_heads: int,
                                   head_dim: int, max_ctx: int, block_size: int,
                                   part_blocks: int) -> int:
    return int(lib().pa_testing_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads,
                                                       head_dim, max_ctx, block_size,
                                                       part_blocks))


def testing_decode_partitions(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                              v_cache: torch.Tensor, block_tables: torch.Tensor,
                              context_lens: torch.Tensor, max_ctx: int, scale: float,
                              part_blocks: int, workspace: torch.Tensor, stream=None):
    """pa_decode with every context cut into partitions of `part_blocks` blocks (see
    pa_testing_decode_partitions in include/pa_testing.h)."""
    nb, h_kv, bs, d = k_cache.shape
    b, h_q, _ = q.shape
    _check(lib().pa_testing_decode_partitions(
        _ptr(out), dtype_code(out.dtype), _ptr(q), _ptr(k_cache), _ptr(v_cache),
        _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), max_ctx, b, h_q, h_kv, d,
        bs, nb, float(scale), dtype_code(k_cache.dtype), int(part_blocks), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def set_stream_status(stream, status: Optional[torch.Tensor]):
    """Routes the status bits of calls on `stream` (a torch.cuda.Stream) into `status`, a
    one-element int32 CUDA tensor the caller reads and clears; None removes the route
    (see pa_set_stream_status)."""
    if status is not None:
        if status.dtype != torch.int32 or status.device.type != "cuda" or status.numel() < 1:
            raise TypeError("status must be an int32 CUDA tensor")
    _check(lib().pa_set_stream_status(_stream(stream), _ptr(status)))


def release_thread_resources():
    """Destroys the side stream and events pa_mixed_step created for this thread."""
    _check(lib().pa_release_thread_resources())


def get_status() -> int:
    """Reads and clears the device status word (synchronises the device)."""
    v = ctypes.c_int32(0)
    _check(lib().pa_get_status(ctypes.byref(v)))
    return int(v.value)


def selftest_wait_timeout(timeout_us: int, stream=None):
    """Runs the bounded-wait self-test: one kernel waits on an mbarrier nothing arrives
    on, gives up after `timeout_us` microseconds and sets STATUS_TIMEOUT."""
    _check(lib().pa_selftest_wait_timeout(int(timeout_us), _stream(stream)))
