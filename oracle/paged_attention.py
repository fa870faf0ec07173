"""float64 reference of the paged KV-cache path.  Test infrastructure only; see the
package docstring for who may use it and which passages it follows.

Cache layout (a reading: the pages give none): each of K and V is one array
[num_blocks, num_kv_heads, block_size, head_dim]; token `off` of physical block `blk`
for KV head `h` sits at [blk, h, off, :].
"""
from __future__ import annotations

import numpy as np


# ----------------------------------------------------------------------------------
# Sizes
# ----------------------------------------------------------------------------------

def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, bytes_per_value: int) -> int:
    """Cache bytes one token costs: one key and one value vector per layer and KV head.

    "PagedAttention and Continuous Batching Explained (2026)", section "Why the KV cache
    is the problem": 2 (K and V) x layers x KV heads x head dimension x bytes per value.
    """
    return 2 * layers * kv_heads * head_dim * bytes_per_value


def blocks_for_tokens(tokens: int, block_size: int) -> int:
    """Blocks a sequence of `tokens` tokens occupies when blocks are allocated one at a
    time as it grows ("PagedAttention: a block table for the KV cache" on the same page;
    "Blocks and Block Tables" in "KV Cache in Serving Engines")."""
    return -(-int(tokens) // int(block_size))


def full_blocks(tokens: int, block_size: int) -> int:
    """Blocks that are completely filled; only these can be keyed for prefix reuse
    ("PagedAttention and Continuous Batching Explained (2026)", section "Prefix
    caching")."""
    return int(tokens) // int(block_size)


def tail_waste(tokens: int, block_size: int) -> int:
    """Unused slots in the last block: the only waste paging leaves per sequence
    ("KV Cache in Serving Engines", section "Blocks and Block Tables")."""
    return blocks_for_tokens(tokens, block_size) * int(block_size) - int(tokens)


# ----------------------------------------------------------------------------------
# Storage types
# ----------------------------------------------------------------------------------

def widen(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of stored values to float64.  bf16 arrives as uint16 bits: the
    bits are the top half of the float32 with the same value."""
    if dtype == "bf16":
        a = np.asarray(a)
        assert a.dtype == np.uint16, "bf16 is carried as uint16 bit patterns"
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if dtype in ("f16", "f32"):
        return np.asarray(a).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype}")


# ----------------------------------------------------------------------------------
# Block-table walks and cache updates (bit-exact operations)
# ----------------------------------------------------------------------------------

def slot_mapping(block_tables: np.ndarray, cu_q_lens: np.ndarray, context_lens: np.ndarray,
                 block_size: int) -> np.ndarray:
    """Physical slot of every new token of a step, as block_id * block_size + offset.

    Sequence b appends the tokens cu_q_lens[b] .. cu_q_lens[b+1]-1 of the step; they are
    the last positions of its context, whose length context_lens[b] counts them (a
    reading: decode appends position context_lens[b]-1).  Position `pos` lives in
    logical block pos // block_size at offset pos % block_size, and the block table gives
    the physical block ("PagedAttention: a block table for the KV cache").
    """
    n_tok = int(cu_q_lens[-1])
    slots = np.empty(n_tok, dtype=np.int64)
    for b in range(len(context_lens)):
        first_new = int(context_lens[b]) - (int(cu_q_lens[b + 1]) - int(cu_q_lens[b]))
        for t in range(int(cu_q_lens[b]), int(cu_q_lens[b + 1])):
            pos = first_new + (t - int(cu_q_lens[b]))
            logical_block, offset = divmod(pos, block_size)
            slots[t] = int(block_tables[b, logical_block]) * block_size + offset
    return slots


def reshape_and_cache(k_new: np.ndarray, v_new: np.ndarray, k_cache: np.ndarray,
                      v_cache: np.ndarray, slots: np.ndarray) -> None:
    """Writes each new token's K and V [num_kv_heads, head_dim] into its slot, in place.

    A negative slot marks a padding token and is skipped (a reading).  The write is a
    copy of stored values, so the result is bit-exact.
    """
    block_size = k_cache.shape[2]
    for t, slot in enumerate(np.asarray(slots).tolist()):
        if slot < 0:
            continue
        blk, off = divmod(slot, block_size)
        k_cache[blk, :, off, :] = k_new[t]
        v_cache[blk, :, off, :] = v_new[t]


def copy_blocks(caches, pairs: np.ndarray) -> None:
    """Copy-on-write: for each (src, dst) pair, physical block dst of every cache array
    becomes a copy of block src ("KV Cache in Serving Engines", section "Sharing
    Blocks": a shared block is copied when a sequence needs to append to it).  Pairs are
    applied in order."""
    for src, dst in np.asarray(pairs).reshape(-1, 2).tolist():
        for cache in caches:
            cache[dst] = cache[src]


def swap_blocks(src_pools, dst_pools, pairs: np.ndarray) -> None:
    """Pre-emption by swap ("Continuous batching and paged attention", section "Why they
    depend on each other": swap to host memory instead of recomputing): for each (src,
    dst) pair, block dst of every destination pool becomes a copy of block src of the
    matching source pool.  Pairs are applied in order."""
    for src, dst in np.asarray(pairs).reshape(-1, 2).tolist():
        for s_pool, d_pool in zip(src_pools, dst_pools):
            d_pool[dst] = s_pool[src]


def gather_context(cache: np.ndarray, table_row: np.ndarray, ctx: int) -> np.ndarray:
    """Walks one block table row and returns the sequence's logical cache
    [ctx, num_kv_heads, head_dim]: token t comes from physical block
    table_row[t // block_size] at offset t % block_size."""
    block_size = cache.shape[2]
    out = np.empty((ctx,) + (cache.shape[1], cache.shape[3]), dtype=cache.dtype)
    for t in range(0, ctx, block_size):
        blk = int(table_row[t // block_size])
        n = min(block_size, ctx - t)
        out[t:t + n] = cache[blk, :, :n, :].transpose(1, 0, 2)
    return out


# ----------------------------------------------------------------------------------
# Attention
# ----------------------------------------------------------------------------------

def _softmax_attend(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                    visible: np.ndarray | None = None) -> np.ndarray:
    """softmax(scale * q k^T) v for q [R, D], k/v [N, D]; `visible` [R, N] masks keys
    a row may not see.  The max-subtracted form is used; rows with no visible key
    return zeros."""
    s = scale * (q @ k.T)
    if visible is not None:
        s = np.where(visible, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    out = np.zeros((q.shape[0], v.shape[1]))
    ok = np.isfinite(m[:, 0])
    if not ok.any():
        return out
    p = np.exp(s[ok] - m[ok])
    p /= p.sum(axis=1, keepdims=True)
    out[ok] = p @ v
    return out


def _kv_head_of(q_head: int, num_q_heads: int, num_kv_heads: int) -> int:
    """Grouped-query mapping (a reading: the pages name grouped-query attention but not
    its grouping): consecutive runs of num_q_heads / num_kv_heads query heads share one
    KV head."""
    return q_head // (num_q_heads // num_kv_heads)


def decode_attention_rows(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                          block_tables: np.ndarray, context_lens: np.ndarray, scale: float,
                          dtype: str, seqs) -> np.ndarray:
    """decode_attention for the listed sequences only; returns [len(seqs), H_q, D]."""
    h_q, d = q.shape[1], q.shape[2]
    h_kv = k_cache.shape[1]
    out = np.zeros((len(seqs), h_q, d))
    for i, b in enumerate(seqs):
        ctx = int(context_lens[b])
        if ctx <= 0:
            continue
        k = widen(gather_context(k_cache, block_tables[b], ctx), dtype)
        v = widen(gather_context(v_cache, block_tables[b], ctx), dtype)
        qb = widen(q[b], dtype)
        for hq in range(h_q):
            h = _kv_head_of(hq, h_q, h_kv)
            out[i, hq] = _softmax_attend(qb[hq:hq + 1], k[:, h, :], v[:, h, :], scale)[0]
    return out


def decode_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                     block_tables: np.ndarray, context_lens: np.ndarray, scale: float,
                     dtype: str) -> np.ndarray:
    """One query token per sequence attends over its whole paged context.

    q [B, H_q, D]; caches [num_blocks, H_kv, block_size, D]; block_tables [B, max_blocks];
    context_lens [B] (the appended token included).  Returns float64 [B, H_q, D]; a
    sequence with an empty context returns zeros (a reading).
    """
    return decode_attention_rows(q, k_cache, v_cache, block_tables, context_lens, scale,
                                 dtype, range(q.shape[0]))


def prefill_chunk_attention_rows(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                                 block_tables: np.ndarray, cu_q_lens: np.ndarray,
                                 context_lens: np.ndarray, scale: float, dtype: str,
                                 tokens) -> np.ndarray:
    """prefill_chunk_attention for the listed query tokens only; returns
    [len(tokens), H_q, D]."""
    h_q, d = q.shape[1], q.shape[2]
    h_kv = k_cache.shape[1]
    cu = np.asarray(cu_q_lens)
    tokens = np.asarray(list(tokens), dtype=np.int64)
    out = np.zeros((len(tokens), h_q, d))
    seq_of = np.searchsorted(cu, tokens, side="right") - 1
    for b in np.unique(seq_of):
        rows = np.nonzero(seq_of == b)[0]
        ctx = int(context_lens[b])
        chunk = int(cu[b + 1] - cu[b])
        first_pos = ctx - chunk
        k = widen(gather_context(k_cache, block_tables[b], ctx), dtype)
        v = widen(gather_context(v_cache, block_tables[b], ctx), dtype)
        pos = first_pos + (tokens[rows] - int(cu[b]))  # absolute position of each query
        visible = np.arange(ctx)[None, :] <= pos[:, None]
        qb = widen(q[tokens[rows]], dtype)
        for hq in range(h_q):
            h = _kv_head_of(hq, h_q, h_kv)
            out[rows, hq] = _softmax_attend(qb[:, hq, :], k[:, h, :], v[:, h, :], scale,
                                            visible)
    return out


def prefill_chunk_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                            block_tables: np.ndarray, cu_q_lens: np.ndarray,
                            context_lens: np.ndarray, scale: float, dtype: str) -> np.ndarray:
    """Causal attention of a chunk of query tokens over a paged context.

    Sequence b owns query rows cu_q_lens[b] .. cu_q_lens[b+1]-1 of q [T, H_q, D].  Its
    context holds context_lens[b] tokens, the chunk's own K/V included (the chunk is
    written to the cache before attention), so query i of the chunk sits at absolute
    position context_lens[b] - chunk_len + i and sees positions 0 .. that position.
    Returns float64 [T, H_q, D].
    """
    return prefill_chunk_attention_rows(q, k_cache, v_cache, block_tables, cu_q_lens,
                                        context_lens, scale, dtype, range(q.shape[0]))
