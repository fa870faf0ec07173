"""Python binding of the host block manager (include/pa_block_manager.h).

Argument marshalling only: every decision (which block, when to copy, what is cached,
what is evicted) is taken by the C++ manager in libpagedattn.  Arrays come back as
numpy arrays ready to be copied to the device for pa_copy_blocks, pa_cache_append,
pa_decode and pa_prefill_chunk.
"""
from __future__ import annotations

import ctypes
from typing import Sequence, Tuple

import numpy as np

from . import PaError, lib

__all__ = ["BlockManager", "NoBlocks", "sha256"]

PA_ERR_INVALID_ARG, PA_ERR_NO_BLOCKS = 1, 5

_i, _p, _i64, _sz = ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
_SIGNATURES = {
    "pa_bm_create": ([_i, _i, _i, _i, ctypes.POINTER(_p)], _i),
    "pa_bm_destroy": ([_p], None),
    "pa_bm_num_free_blocks": ([_p], _i),
    "pa_bm_num_free_host_blocks": ([_p], _i),
    "pa_bm_can_allocate": ([_p, _i, _i], _i),
    "pa_bm_add_sequence": ([_p, _i64, _p, _i, _p, _i, _p], _i),
    "pa_bm_append_tokens": ([_p, _i64, _p, _i], _i),
    "pa_bm_append_tokens_batch": ([_p, _p, _i, _p, _p], _i),
    "pa_bm_fork": ([_p, _i64, _i64], _i),
    "pa_bm_free_sequence": ([_p, _i64], _i),
    "pa_bm_take_copies": ([_p, _p, _i, _p], _i),
    "pa_bm_swap_out": ([_p, _p, _i, _p, _i, _p], _i),
    "pa_bm_swap_in": ([_p, _p, _i, _p, _i, _p], _i),
    "pa_bm_num_tokens": ([_p, _i64], _i),
    "pa_bm_block_tables": ([_p, _p, _i, _i, _p, _p], _i),
    "pa_bm_slot_mapping": ([_p, _p, _i, _p, _p, _i, _p], _i),
    "pa_bm_refcount": ([_p, _i], _i),
    "pa_bm_is_cached": ([_p, _i], _i),
    "pa_bm_free_queue": ([_p, _p, _i, _p], _i),
    "pa_sha256": ([_p, _sz, _p], None),
}
_bound = False


def _lib():
    global _bound
    L = lib()
    if not _bound:
        for name, (args, res) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _bound = True
    return L


class NoBlocks(PaError):
    """The pool (or the host pool) has too few free blocks; nothing was changed."""


def _check(rc: int):
    if rc != 0:
        msg = _lib().pa_last_error_string().decode()
        raise (NoBlocks if rc == PA_ERR_NO_BLOCKS else PaError)(rc, msg)


def _arr(a, dtype):
    a = np.ascontiguousarray(np.asarray(a, dtype=dtype))
    return a, a.ctypes.data if a.size else None


def sha256(data: bytes) -> bytes:
    out = ctypes.create_string_buffer(32)
    _lib().pa_sha256(data if data else None, len(data), out)
    return out.raw


class BlockManager:
    """Block tables, reference counts, copy-on-write, prefix cache and swap bookkeeping
    for one pool of `num_blocks` blocks of `block_size` tokens."""

    def __init__(self, num_blocks: int, block_size: int, prefix_caching: bool = False,
                 num_host_blocks: int = 0):
        h = _p()
        _check(_lib().pa_bm_create(num_blocks, block_size, int(prefix_caching), num_host_blocks,
                                   ctypes.byref(h)))
        self._h = h
        self.block_size = int(block_size)
        self.num_blocks = int(num_blocks)

    def close(self):
        if getattr(self, "_h", None):
            _lib().pa_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------------ counters
    def num_free_blocks(self) -> int:
        return _lib().pa_bm_num_free_blocks(self._h)

    def num_free_host_blocks(self) -> int:
        return _lib().pa_bm_num_free_host_blocks(self._h)

    def can_allocate(self, num_tokens: int, watermark: int = 0) -> bool:
        return bool(_lib().pa_bm_can_allocate(self._h, num_tokens, watermark))

    # ------------------------------------------------------------------ sequences
    def add_sequence(self, seq_id: int, tokens: Sequence[int], extra: bytes = b"") -> int:
        t, tp = _arr(tokens, np.int32)
        cached = ctypes.c_int(0)
        _check(_lib().pa_bm_add_sequence(self._h, seq_id, tp, t.size, extra or None, len(extra),
                                         ctypes.byref(cached)))
        return cached.value

    def append_tokens(self, seq_id: int, tokens: Sequence[int]):
        t, tp = _arr(tokens, np.int32)
        _check(_lib().pa_bm_append_tokens(self._h, seq_id, tp, t.size))

    def append_tokens_batch(self, seq_ids: Sequence[int], tokens: Sequence[int],
                            counts: Sequence[int] = None):
        """Sequence seq_ids[i] appends counts[i] tokens (default one each), taken in turn
        from `tokens`; all or nothing."""
        s, sp = _arr(seq_ids, np.int64)
        t, tp = _arr(tokens, np.int32)
        if counts is None:
            cp = None
            total = s.size
        else:
            c, cp = _arr(counts, np.int32)
            self._keep_c = c
            total = int(c.sum())
        if t.size != total:
            raise ValueError(f"{t.size} tokens for {total} appends")
        _check(_lib().pa_bm_append_tokens_batch(self._h, sp, s.size, tp, cp))

    def fork(self, parent_id: int, child_id: int):
        _check(_lib().pa_bm_fork(self._h, parent_id, child_id))

    def free_sequence(self, seq_id: int):
        _check(_lib().pa_bm_free_sequence(self._h, seq_id))

    def _pairs(self, fn, *args) -> np.ndarray:
        """Calls a pair-emitting entry point, sizing the output from a first call."""
        n = ctypes.c_int(0)
        rc = fn(self._h, *args, None, 0, ctypes.byref(n))
        if rc == 0:
            return np.zeros((0, 2), dtype=np.int32)
        if rc != PA_ERR_INVALID_ARG or n.value == 0:
            _check(rc)
        out = np.empty((n.value, 2), dtype=np.int32)
        _check(fn(self._h, *args, out.ctypes.data, n.value, ctypes.byref(n)))
        return out

    def take_copies(self) -> np.ndarray:
        """int32 [N, 2] (source, destination) copy-on-write pairs since the last call."""
        return self._pairs(_lib().pa_bm_take_copies)

    def swap_out(self, seq_ids: Sequence[int]) -> np.ndarray:
        """int32 [N, 2] (device block, host block) pairs to copy device -> host."""
        s, sp = _arr(seq_ids, np.int64)
        self._keep = s
        return self._pairs(_lib().pa_bm_swap_out, sp, s.size)

    def swap_in(self, seq_ids: Sequence[int]) -> np.ndarray:
        """int32 [N, 2] (host block, device block) pairs to copy host -> device."""
        s, sp = _arr(seq_ids, np.int64)
        self._keep = s
        return self._pairs(_lib().pa_bm_swap_in, sp, s.size)

    # ------------------------------------------------------------------ emission
    def num_tokens(self, seq_id: int) -> int:
        return _lib().pa_bm_num_tokens(self._h, seq_id)

    def block_tables(self, seq_ids: Sequence[int], width: int) -> Tuple[np.ndarray, np.ndarray]:
        """(int32 [n, width] tables padded with -1, int32 [n] context lengths)."""
        s, sp = _arr(seq_ids, np.int64)
        tables = np.empty((s.size, max(width, 0)), dtype=np.int32)
        ctx = np.empty(s.size, dtype=np.int32)
        _check(_lib().pa_bm_block_tables(self._h, sp, s.size, width,
                                         tables.ctypes.data if tables.size else None,
                                         ctx.ctypes.data if ctx.size else None))
        return tables, ctx

    def block_table(self, seq_id: int) -> list:
        n = self.num_tokens(seq_id)
        width = -(-n // self.block_size)
        return self.block_tables([seq_id], width)[0][0].tolist()

    def slot_mapping(self, seq_ids: Sequence[int], query_lens: Sequence[int]) -> np.ndarray:
        s, sp = _arr(seq_ids, np.int64)
        q, qp = _arr(query_lens, np.int32)
        total = int(q.sum()) if q.size else 0
        out = np.empty(total, dtype=np.int64)
        n = ctypes.c_int(0)
        _check(_lib().pa_bm_slot_mapping(self._h, sp, s.size, qp,
                                         out.ctypes.data if total else None, total,
                                         ctypes.byref(n)))
        return out

    # ------------------------------------------------------------------ introspection
    def refcount(self, block: int) -> int:
        return _lib().pa_bm_refcount(self._h, block)

    def is_cached(self, block: int) -> bool:
        return _lib().pa_bm_is_cached(self._h, block) == 1

    def free_queue(self) -> list:
        n = self.num_free_blocks()
        out = np.empty(max(n, 1), dtype=np.int32)
        m = ctypes.c_int(0)
        _check(_lib().pa_bm_free_queue(self._h, out.ctypes.data, n, ctypes.byref(m)))
        return out[:m.value].tolist()
