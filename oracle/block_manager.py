"""Reference block manager: paged allocation, sharing with copy-on-write, prefix-cache keys
with least-recently-used eviction, and swap to host blocks.  Test infrastructure only.

Plain Python over lists and dicts, written from the pages' description, so that a
reader can check each step by eye.  The library's C++ block manager is compared with it
operation by operation on random traces; the two share no code.

What the pages fix:

* The cache is a pool of fixed-size physical blocks; each sequence has a block table
  from logical to physical blocks; a block is allocated only when the sequence's last
  block is full (or it has none), and freed when the sequence finishes.
  ("PagedAttention and Continuous Batching Explained (2026)", section "PagedAttention: a
  block table for the KV cache"; "Continuous batching and paged attention", section
  "Paged attention"; "KV Cache in Serving Engines", section "Blocks and Block Tables".)
* Sequences may point at the same physical blocks; blocks carry reference counts, and a
  shared block is copied only when someone needs to append to it (copy-on-write).
  ("KV Cache in Serving Engines", section "Sharing Blocks"; "Continuous batching, paged
  attention, prefix caching", section "Prefix caching".)
* Admission asks whether enough free blocks exist for the prompt plus a margin
  ("Continuous batching and paged attention", section "Paged attention").
* Prefix caching keys each full block by a hash of the previous block's key, the
  block's own token ids and extra keys; only full blocks are keyed; a new sequence
  reuses its leading blocks while their keys are found and stops at the first miss.
  Blocks whose last reader finished keep their contents in a queue, oldest evicted
  first, and a finished sequence's blocks enter that queue tail first so that its tail
  blocks go before its head blocks.  The hash is sha256.
  ("KV Cache in Serving Engines", section "4. Prefix Caching: Computing the Same Prefix
  Only Once"; "PagedAttention and Continuous Batching Explained (2026)", section
  "Prefix caching".)
* Pre-emption can swap a sequence's blocks to host memory instead of recomputing them
  ("Continuous batching and paged attention", section "Why they depend on each other").

Readings where the pages are silent (each one a choice the C++ manager makes the same
way, because the tests compare the block ids both hand out):

1. One queue holds every device block with no reader, in least-recently-used order:
   initially blocks 0, 1, ..., N-1; allocation takes the front; a freed block joins the
   back; a cached block found by a lookup leaves the queue wherever it is.  Taking a
   block that still carries a key evicts it: the key is forgotten.
2. Key of a block = sha256(parent key || token ids || extra), with parent key = 32 zero
   bytes for a sequence's first block, token ids as little-endian int32, and `extra`
   the sequence's extra-key bytes (adapter id, cache salt, ...).
3. A block is keyed the moment it becomes full, from the token ids the manager was
   given, whether it filled at admission or by an append.  If the key is already held
   by another block, the new block stays unkeyed (no duplicate entries).
4. Copy-on-write: appending into a last block that another sequence also reads takes a
   new block, records (source, destination) for the cache copy, and moves this sequence
   to the copy.  The last reader appends in place.
5. Swap-out copies every block the listed sequences read to a host block (one host
   block per distinct device block, shared blocks once) and drops those sequences'
   device references; swap-in does the reverse onto freshly allocated device blocks.
   Host blocks come from a first-in first-out free list (initially 0 .. H-1).  Blocks
   brought back are not keyed.
6. An operation that lacks blocks changes nothing and fails.
"""
from __future__ import annotations

import hashlib
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

ROOT_KEY = bytes(32)


class NoBlocks(RuntimeError):
    """Not enough free blocks (device or host) for the operation."""


def block_key(parent: bytes, tokens: Sequence[int], extra: bytes = b"") -> bytes:
    """sha256(parent key || token ids as little-endian int32 || extra keys)."""
    body = np.asarray(list(tokens), dtype="<i4").tobytes()
    return hashlib.sha256(parent + body + extra).digest()


def key_chain(tokens: Sequence[int], block_size: int, extra: bytes = b"") -> List[bytes]:
    """Keys of every full block of a token sequence, each chained on the one before."""
    keys, parent = [], ROOT_KEY
    for i in range(len(tokens) // block_size):
        parent = block_key(parent, tokens[i * block_size:(i + 1) * block_size], extra)
        keys.append(parent)
    return keys


class _Seq:
    def __init__(self, tokens, extra):
        self.tokens: List[int] = list(tokens)
        self.blocks: List[int] = []
        self.keys: List[bytes] = []  # keys of the sequence's full blocks, in order
        self.extra: bytes = extra
        self.swapped = False


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int, prefix_caching: bool = False,
                 num_host_blocks: int = 0):
        self.bs = int(block_size)
        self.num_blocks = int(num_blocks)
        self.prefix_caching = bool(prefix_caching)
        self.queue: List[int] = list(range(self.num_blocks))  # front = least recently used
        self.ref = [0] * self.num_blocks
        self.key: List[Optional[bytes]] = [None] * self.num_blocks
        self.cached: Dict[bytes, int] = {}
        self.host_free: List[int] = list(range(int(num_host_blocks)))
        self.host_ref = [0] * int(num_host_blocks)
        self.seqs: Dict[int, _Seq] = {}
        self.copies: List[Tuple[int, int]] = []

    # -------------------------------------------------------------- counters
    def num_free_blocks(self) -> int:
        return len(self.queue)

    def num_free_host_blocks(self) -> int:
        return len(self.host_free)

    def can_allocate(self, num_tokens: int, watermark: int = 0) -> bool:
        return -(-num_tokens // self.bs) + watermark <= len(self.queue)

    # -------------------------------------------------------------- blocks
    def _take(self) -> int:
        b = self.queue.pop(0)
        if self.key[b] is not None:  # evict: the cached contents are given up
            del self.cached[self.key[b]]
            self.key[b] = None
        self.ref[b] = 1
        return b

    def _release(self, b: int):
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self.queue.append(b)

    def _on_full(self, seq: _Seq, i: int):
        """Block i of `seq` just became full: its key joins the chain, and the block
        is registered for reuse unless another block holds that key."""
        parent = seq.keys[i - 1] if i > 0 else ROOT_KEY
        k = block_key(parent, seq.tokens[i * self.bs:(i + 1) * self.bs], seq.extra)
        seq.keys.append(k)
        b = seq.blocks[i]
        if self.prefix_caching and k not in self.cached and self.key[b] is None:
            self.cached[k] = b
            self.key[b] = k

    # -------------------------------------------------------------- sequences
    def add_sequence(self, seq_id: int, tokens: Sequence[int], extra: bytes = b"") -> int:
        """Admits a sequence with its prompt; returns the prompt tokens whose blocks
        were found in the prefix cache."""
        if seq_id in self.seqs:
            raise KeyError(f"sequence {seq_id} exists")
        n = len(tokens)
        nblocks = -(-n // self.bs)
        hits: List[int] = []
        if self.prefix_caching:
            for k in key_chain(tokens, self.bs, extra):
                b = self.cached.get(k)
                if b is None:
                    break
                hits.append(b)
        idle_hits = sum(1 for b in hits if self.ref[b] == 0)
        if nblocks - len(hits) > len(self.queue) - idle_hits:
            raise NoBlocks("not enough free blocks for the prompt")
        seq = _Seq(tokens, extra)
        for b in hits:
            if self.ref[b] == 0:
                self.queue.remove(b)
            self.ref[b] += 1
            seq.blocks.append(b)
        for _ in range(nblocks - len(hits)):
            seq.blocks.append(self._take())
        for i in range(n // self.bs):
            self._on_full(seq, i)
        self.seqs[seq_id] = seq
        return len(hits) * self.bs

    def append_tokens(self, seq_id: int, tokens: Sequence[int]):
        """Appends tokens (one per decode step, or a chunk), allocating at block
        boundaries and copying a shared last block before writing into it."""
        seq = self.seqs[seq_id]
        if seq.swapped:
            raise RuntimeError(f"sequence {seq_id} is swapped out")
        n0, k = len(seq.tokens), len(tokens)
        if k == 0:
            return
        need = -(-(n0 + k) // self.bs) - -(-n0 // self.bs)
        if n0 % self.bs != 0 and self.ref[seq.blocks[-1]] > 1:
            need += 1  # the shared last block is copied first
        if need > len(self.queue):
            raise NoBlocks("not enough free blocks to append")
        for t in tokens:
            pos = len(seq.tokens)
            if pos % self.bs == 0:
                seq.blocks.append(self._take())
            elif self.ref[seq.blocks[-1]] > 1:
                src = seq.blocks[-1]
                dst = self._take()
                self.copies.append((src, dst))
                self.ref[src] -= 1
                seq.blocks[-1] = dst
            seq.tokens.append(int(t))
            if (pos + 1) % self.bs == 0:
                self._on_full(seq, pos // self.bs)

    def append_tokens_batch(self, seq_ids: Sequence[int], tokens: Sequence[int],
                            counts: Optional[Sequence[int]] = None):
        """append_tokens for each listed sequence in turn (one token each unless
        `counts` says otherwise), all or nothing: the blocks the whole batch takes are
        counted first, copies included (a copy leaves its source with one reader fewer,
        so a later sequence of the batch on the same block may append in place)."""
        counts = [1] * len(seq_ids) if counts is None else list(counts)
        if len(set(seq_ids)) != len(seq_ids):
            raise ValueError("a sequence is listed twice")
        need, copied = 0, {}
        for s, k in zip(seq_ids, counts):
            seq = self.seqs[s]
            if seq.swapped:
                raise RuntimeError(f"sequence {s} is swapped out")
            if k == 0:
                continue
            n0 = len(seq.tokens)
            need += -(-(n0 + k) // self.bs) - -(-n0 // self.bs)
            if n0 % self.bs != 0:
                last = seq.blocks[-1]
                if self.ref[last] - copied.get(last, 0) > 1:
                    need += 1
                    copied[last] = copied.get(last, 0) + 1
        if need > len(self.queue):
            raise NoBlocks("not enough free blocks to append")
        pos = 0
        for s, k in zip(seq_ids, counts):
            self.append_tokens(s, tokens[pos:pos + k])
            pos += k

    def fork(self, parent_id: int, child_id: int):
        """The child reads every block of the parent (parallel sampling, beam search)."""
        if child_id in self.seqs:
            raise KeyError(f"sequence {child_id} exists")
        p = self.seqs[parent_id]
        if p.swapped:
            raise RuntimeError(f"sequence {parent_id} is swapped out")
        c = _Seq(p.tokens, p.extra)
        c.blocks = list(p.blocks)
        c.keys = list(p.keys)
        for b in c.blocks:
            self.ref[b] += 1
        self.seqs[child_id] = c

    def free_sequence(self, seq_id: int):
        """Drops a finished sequence; its blocks with no other reader join the queue,
        tail first."""
        seq = self.seqs.pop(seq_id)
        if seq.swapped:
            for h in reversed(seq.blocks):
                self.host_ref[h] -= 1
                if self.host_ref[h] == 0:
                    self.host_free.append(h)
            return
        for b in reversed(seq.blocks):
            self._release(b)

    def take_copies(self) -> List[Tuple[int, int]]:
        out, self.copies = self.copies, []
        return out

    # -------------------------------------------------------------- swap
    def _distinct_blocks(self, seq_ids):
        order: List[int] = []
        seen = set()
        for s in seq_ids:
            for b in self.seqs[s].blocks:
                if b not in seen:
                    seen.add(b)
                    order.append(b)
        return order

    def swap_out(self, seq_ids: Sequence[int]) -> List[Tuple[int, int]]:
        """Moves the sequences to host blocks; returns (device block, host block) pairs
        to copy before the device blocks are reused."""
        for s in seq_ids:
            if self.seqs[s].swapped:
                raise RuntimeError(f"sequence {s} is already swapped out")
        blocks = self._distinct_blocks(seq_ids)
        if len(blocks) > len(self.host_free):
            raise NoBlocks("not enough host blocks")
        to_host = {}
        for b in blocks:
            to_host[b] = self.host_free.pop(0)
        for s in seq_ids:
            seq = self.seqs[s]
            for b in reversed(seq.blocks):
                self.host_ref[to_host[b]] += 1
                self._release(b)
            seq.blocks = [to_host[b] for b in seq.blocks]
            seq.swapped = True
        return [(b, to_host[b]) for b in blocks]

    def swap_in(self, seq_ids: Sequence[int]) -> List[Tuple[int, int]]:
        """Brings swapped sequences back onto new device blocks; returns (host block,
        device block) pairs to copy before they are read."""
        for s in seq_ids:
            if not self.seqs[s].swapped:
                raise RuntimeError(f"sequence {s} is not swapped out")
        blocks = self._distinct_blocks(seq_ids)
        if len(blocks) > len(self.queue):
            raise NoBlocks("not enough free blocks to swap in")
        to_dev = {}
        for h in blocks:
            to_dev[h] = self._take()
            self.ref[to_dev[h]] = 0
        for s in seq_ids:
            seq = self.seqs[s]
            for h in reversed(seq.blocks):
                self.ref[to_dev[h]] += 1
                self.host_ref[h] -= 1
                if self.host_ref[h] == 0:
                    self.host_free.append(h)
            seq.blocks = [to_dev[h] for h in seq.blocks]
            seq.swapped = False
        return [(h, to_dev[h]) for h in blocks]

    # -------------------------------------------------------------- emission
    def num_tokens(self, seq_id: int) -> int:
        return len(self.seqs[seq_id].tokens)

    def block_table(self, seq_id: int) -> List[int]:
        return list(self.seqs[seq_id].blocks)

    def block_tables(self, seq_ids: Sequence[int], width: int) -> np.ndarray:
        """int32 [len(seq_ids), width]; unused entries -1."""
        t = np.full((len(seq_ids), width), -1, dtype=np.int32)
        for i, s in enumerate(seq_ids):
            b = self.seqs[s].blocks
            if len(b) > width:
                raise ValueError("table wider than `width`")
            t[i, :len(b)] = b
        return t

    def context_lens(self, seq_ids: Sequence[int]) -> np.ndarray:
        return np.array([len(self.seqs[s].tokens) for s in seq_ids], dtype=np.int32)

    def slot_mapping(self, seq_ids: Sequence[int], query_lens: Sequence[int]) -> np.ndarray:
        """Physical slot of each sequence's last query_lens[i] tokens, sequence by
        sequence: block_table[pos // bs] * bs + pos % bs."""
        out = []
        for s, q in zip(seq_ids, query_lens):
            seq = self.seqs[s]
            n = len(seq.tokens)
            for pos in range(n - int(q), n):
                out.append(seq.blocks[pos // self.bs] * self.bs + pos % self.bs)
        return np.asarray(out, dtype=np.int64)

    def refcount(self, block: int) -> int:
        return self.ref[block]

    def is_cached(self, block: int) -> bool:
        return self.key[block] is not None
