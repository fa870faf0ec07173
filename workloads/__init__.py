"""Seeded synthetic inputs for the paged KV-cache attention path.

This module only lays inputs out: how long each sequence is, which physical block
holds each logical block, how many new tokens each sequence appends in a step, which
shared blocks are copied before an append, and the random q/K/V values.  It performs
none of the attention arithmetic and derives no slot numbers: the CUDA library and the
CPU oracle each compute everything else from these inputs on their own, and this is the
only code the two share.

Every workload is reproducible from its seed.  Structure (lengths, block ids) is drawn
with numpy's PCG64; values are drawn with torch's generator on the device that will hold
them (the CPU for oracle-only tests, the GPU for the full-size pools), as float32
N(0, 1) rounded to the storage dtype.

The five named workloads follow the shapes the pages use as examples:

* the Llama 3.1 8B and OPT-13B head shapes from "PagedAttention and Continuous
  Batching Explained (2026)", section "Why the KV cache is the problem";
* the default block size of 16 tokens from the same page, section "PagedAttention: a
  block table for the KV cache";
* block sharing with copy-on-write for parallel sampling, from "KV Cache in Serving
  Engines: PagedAttention, Continuous Batching, and Prefix Caching", section "Sharing
  Blocks";
* chunked prefill mixed with decodes in one step, from "PagedAttention and Continuous
  Batching Explained (2026)", section "Chunked prefill".
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass
from typing import Dict, Optional, Tuple

import numpy as np

DTYPES = ("f32", "f16", "bf16")
DTYPE_BYTES = {"f32": 4, "f16": 2, "bf16": 2}
UNUSED_BLOCK = -1  # block-table entries past a sequence's last block


@dataclass(frozen=True)
class Shape:
    """Per-layer head shape and cache geometry."""

    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: str

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def elem_bytes(self) -> int:
        return DTYPE_BYTES[self.dtype]


@dataclass
class Batch:
    """Metadata of one attention call.

    context_lens[b] counts every token of sequence b once this step's new tokens are in
    the cache; query_lens[b] of them are new this step (1 for a decode).  Row b of
    block_tables lists the physical block of each logical block; entries past the last
    block hold UNUSED_BLOCK.
    """

    context_lens: np.ndarray  # int32 [B]
    query_lens: np.ndarray  # int32 [B]
    block_tables: np.ndarray  # int32 [B, max_blocks]

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def cu_q_lens(self) -> np.ndarray:
        out = np.zeros(self.num_seqs + 1, dtype=np.int32)
        np.cumsum(self.query_lens, out=out[1:])
        return out

    @property
    def num_new_tokens(self) -> int:
        return int(self.query_lens.sum())

    @property
    def max_ctx(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    @property
    def max_q(self) -> int:
        return int(self.query_lens.max()) if self.num_seqs else 0


@dataclass
class Step:
    """One step of the hot path over one batch of synthetic input.

    Order of a step: copy the `cow_pairs` blocks (when present), write each batch's new
    K/V through its slot mapping, then run decode attention over `decode` and chunked
    prefill attention over `prefill`.
    """

    name: str
    shape: Shape
    num_blocks: int
    seed: int
    scale: float
    decode: Optional[Batch] = None
    prefill: Optional[Batch] = None
    cow_pairs: Optional[np.ndarray] = None  # int32 [N, 2] (src, dst)
    decode_tables_before_cow: Optional[np.ndarray] = None
    # one physical prefix read by several decode sequences: (prefix blocks int32,
    # prefix length in tokens, indices of the decode rows that start with it)
    shared_prefix: Optional[Tuple[np.ndarray, int, np.ndarray]] = None
    notes: str = ""

    def batches(self):
        return [b for b in (self.decode, self.prefill) if b is not None]


def _pool_with_headroom(used_blocks: int, headroom: float = 0.10) -> int:
    return used_blocks + int(np.ceil(used_blocks * headroom))


def _tables(block_counts, width: int, ids: np.ndarray) -> np.ndarray:
    """Hands out `ids` in order, block_counts[b] of them to row b."""
    tables = np.full((len(block_counts), max(width, 1)), UNUSED_BLOCK, dtype=np.int32)
    pos = 0
    for b, n in enumerate(block_counts):
        tables[b, :n] = ids[pos:pos + n]
        pos += n
    return tables


def _nblocks(tokens, block_size: int) -> np.ndarray:
    tokens = np.asarray(tokens, dtype=np.int64)
    return (tokens + block_size - 1) // block_size


def decode_step(name: str, shape: Shape, context_lens, seed: int, *,
                headroom: float = 0.10, scale: Optional[float] = None,
                rng: Optional[np.random.Generator] = None,
                num_blocks: Optional[int] = None) -> Step:
    """A decode step: every sequence appends one token and attends over its context."""
    rng = rng if rng is not None else np.random.default_rng(seed)
    ctx = np.asarray(context_lens, dtype=np.int32)
    counts = _nblocks(ctx, shape.block_size)
    used = int(counts.sum())
    nb = num_blocks if num_blocks is not None else max(_pool_with_headroom(used, headroom), 1)
    ids = rng.permutation(nb).astype(np.int32)
    width = int(counts.max()) if len(counts) else 1
    batch = Batch(context_lens=ctx, query_lens=np.ones_like(ctx),
                  block_tables=_tables(counts, width, ids))
    return Step(name=name, shape=shape, num_blocks=nb, seed=seed,
                scale=scale if scale is not None else 1.0 / np.sqrt(shape.head_dim),
                decode=batch)


def shared_prefix_step(name: str, shape: Shape, prefix_len: int, suffix_lens, other_ctx,
                       seed: int, *, headroom: float = 0.10) -> Step:
    """A decode step in which rows 0 .. len(suffix_lens)-1 start with one shared
    `prefix_len`-token prefix (a whole number of blocks held once in the pool) followed by
    suffix_lens[i] private tokens (the appended token included when > 0; a row with suffix
    0 appends the prefix's last token itself, so at most one such row is allowed), and
    rows after them have private contexts `other_ctx`."""
    bs = shape.block_size
    if prefix_len % bs:
        raise ValueError("prefix_len must be a whole number of blocks")
    suf = np.asarray(suffix_lens, dtype=np.int64)
    if int((suf == 0).sum()) > 1:
        raise ValueError("at most one sharer may end at the prefix")
    oth = np.asarray(other_ctx, dtype=np.int64)
    rng = np.random.default_rng(seed)
    pb = prefix_len // bs
    counts_suf, counts_oth = _nblocks(suf, bs), _nblocks(oth, bs)
    used = pb + int(counts_suf.sum()) + int(counts_oth.sum())
    nb = max(_pool_with_headroom(used, headroom), 1)
    ids = iter(rng.permutation(nb).astype(np.int32).tolist())
    take = lambda n: [next(ids) for _ in range(int(n))]
    prefix = take(pb)
    rows = [prefix + take(n) for n in counts_suf] + [take(n) for n in counts_oth]
    ctx = np.concatenate([prefix_len + suf, oth]).astype(np.int32)
    width = max(1, max(len(r) for r in rows))
    t = np.full((len(rows), width), UNUSED_BLOCK, dtype=np.int32)
    for b, r in enumerate(rows):
        t[b, :len(r)] = r
    batch = Batch(context_lens=ctx, query_lens=np.ones_like(ctx), block_tables=t)
    return Step(name=name, shape=shape, num_blocks=nb, seed=seed,
                scale=1.0 / np.sqrt(shape.head_dim), decode=batch,
                shared_prefix=(np.asarray(prefix, dtype=np.int32), int(prefix_len),
                               np.arange(len(suf), dtype=np.int32)))


def prefill_step(name: str, shape: Shape, context_lens, query_lens, seed: int, *,
                 headroom: float = 0.10, scale: Optional[float] = None) -> Step:
    """A chunked-prefill step: sequence b appends query_lens[b] tokens (its chunk) at the
    end of a context that then holds context_lens[b] tokens."""
    rng = np.random.default_rng(seed)
    ctx = np.asarray(context_lens, dtype=np.int32)
    ql = np.asarray(query_lens, dtype=np.int32)
    counts = _nblocks(ctx, shape.block_size)
    nb = max(_pool_with_headroom(int(counts.sum()), headroom), 1)
    ids = rng.permutation(nb).astype(np.int32)
    batch = Batch(context_lens=ctx, query_lens=ql,
                  block_tables=_tables(counts, int(counts.max()), ids))
    return Step(name=name, shape=shape, num_blocks=nb, seed=seed,
                scale=scale if scale is not None else 1.0 / np.sqrt(shape.head_dim),
                prefill=batch)


# ----------------------------------------------------------------------------------
# The five named workloads
# ----------------------------------------------------------------------------------

def tiny_decode() -> Step:
    """4 sequences with contexts {1, 17, 33, 100}, 4 query heads = 4 KV heads, head
    dim 64, block size 16, fp32, scale 1/8; block ids drawn as a random permutation of a
    64-block pool."""
    shape = Shape(4, 4, 64, 16, "f32")
    return decode_step("tiny_decode_b4_mha_d64_f32", shape, [1, 17, 33, 100], 53_000,
                       num_blocks=64, scale=1.0 / 8.0)


def opt13b_decode() -> Step:
    """OPT-13B-shaped decode layer: 40 heads MHA, head dim 128, fp16, block size 16,
    64 sequences with contexts uniform in [128, 2048]; pool = used blocks + 10% free."""
    rng = np.random.default_rng(53_001)
    ctx = rng.integers(128, 2048, size=64, endpoint=True)
    shape = Shape(40, 40, 128, 16, "f16")
    return decode_step("opt13b_decode_b64_mha40_d128_f16", shape, ctx, 53_001, rng=rng)


def llama8b_gqa_lengths(num_seqs: int = 256, seed: int = 53_002):
    rng = np.random.default_rng(seed)
    ctx = np.clip(np.rint(rng.lognormal(mean=6.5, sigma=0.9, size=num_seqs)), 16, 8192)
    return ctx.astype(np.int32), rng


def llama8b_gqa_decode() -> Step:
    """Llama-3.1-8B-shaped GQA decode layer: 32 query heads, 8 KV heads, head dim 128,
    bf16, block size 16, 256 sequences with contexts round(lognormal(6.5, 0.9)) clipped
    to [16, 8192]; block ids shuffled over a pool of used blocks + 10% free."""
    ctx, rng = llama8b_gqa_lengths()
    shape = Shape(32, 8, 128, 16, "bf16")
    return decode_step("llama8b_gqa_decode_b256_h32kv8_d128_bf16", shape, ctx, 53_002,
                       rng=rng)


def prefix_sharing_cow() -> Step:
    """Prefix sharing plus parallel sampling, Llama-3.1-8B GQA shape, bf16, block 16.

    * 128 sequences share one 2048-token prefix (128 physical blocks referenced 128
      times); each has a private suffix of uniform [1, 512] tokens, the appended token
      included.
    * 8 groups of 4 samples share a private prompt of uniform [1, 512] tokens, redrawn
      while it is a whole number of blocks so that its last block is partly filled.
      Every sample appends one token into that shared last block.  The block is copied
      for three of the four samples, which are remapped to their copies; the fourth is
      then the block's only reader and appends in place.  That gives 24 copies.
    """
    shape = Shape(32, 8, 128, 16, "bf16")
    bs = shape.block_size
    rng = np.random.default_rng(53_003)
    n_prefix_seqs, prefix_tokens = 128, 2048
    suffix = rng.integers(1, 512, size=n_prefix_seqs, endpoint=True)
    n_groups, n_samples = 8, 4
    prompts = []
    for _ in range(n_groups):
        n = int(rng.integers(1, 512, endpoint=True))
        while n % bs == 0:
            n = int(rng.integers(1, 512, endpoint=True))
        prompts.append(n)
    prompts = np.asarray(prompts)

    prefix_blocks = prefix_tokens // bs
    suffix_blocks = _nblocks(suffix, bs)
    prompt_blocks = _nblocks(prompts, bs)
    n_copies = n_groups * (n_samples - 1)
    used = prefix_blocks + int(suffix_blocks.sum()) + int(prompt_blocks.sum()) + n_copies
    nb = _pool_with_headroom(used)
    ids = iter(rng.permutation(nb).astype(np.int32).tolist())

    take = lambda n: [next(ids) for _ in range(int(n))]
    shared_prefix = take(prefix_blocks)
    rows_before, rows_after, ctx, pairs = [], [], [], []
    for i in range(n_prefix_seqs):
        row = shared_prefix + take(suffix_blocks[i])
        rows_before.append(row)
        rows_after.append(row)
        ctx.append(prefix_tokens + int(suffix[i]))
    for g in range(n_groups):
        prompt = take(prompt_blocks[g])
        for s in range(n_samples):
            rows_before.append(list(prompt))
            after = list(prompt)
            if s < n_samples - 1:
                dst = next(ids)
                pairs.append((prompt[-1], dst))
                after[-1] = dst
            rows_after.append(after)
            ctx.append(int(prompts[g]) + 1)

    width = max(len(r) for r in rows_after)

    def pack(rows):
        t = np.full((len(rows), width), UNUSED_BLOCK, dtype=np.int32)
        for b, r in enumerate(rows):
            t[b, :len(r)] = r
        return t

    ctx = np.asarray(ctx, dtype=np.int32)
    batch = Batch(context_lens=ctx, query_lens=np.ones_like(ctx), block_tables=pack(rows_after))
    return Step(name="prefix_cow_decode_b160_h32kv8_d128_bf16", shape=shape, num_blocks=nb,
                seed=53_003, scale=1.0 / np.sqrt(shape.head_dim), decode=batch,
                cow_pairs=np.asarray(pairs, dtype=np.int32).reshape(-1, 2),
                decode_tables_before_cow=pack(rows_before),
                shared_prefix=(np.asarray(shared_prefix, dtype=np.int32), prefix_tokens,
                               np.arange(n_prefix_seqs, dtype=np.int32)),
                notes="rows 0-127 share a 2048-token prefix; rows 128-159 are 8 groups of "
                      "4 samples")


def mixed_prefill_decode(decode_scale: float = 1.0) -> Step:
    """Chunked prefill mixed with long-context decodes, Llama-3.1-8B GQA shape, bf16,
    block size 32.

    * prefill: 8 sequences, each a 512-token causal chunk over an existing context drawn
      uniformly from the integers in [0, 16384]; the first is pinned to 0 and the last to
      16384 so both ends are covered.
    * decode: 240 sequences with contexts uniform in [1024, 32768] and 8 with 131072.

    `decode_scale` < 1 shrinks every decode context by that factor (for reduced-size
    tests); 1 gives the full workload.
    """
    shape = Shape(32, 8, 128, 32, "bf16")
    bs = shape.block_size
    rng = np.random.default_rng(53_004)
    chunk = 512
    ctx0 = rng.integers(0, 16384, size=8, endpoint=True)
    ctx0[0], ctx0[-1] = 0, 16384
    pre_ctx = (ctx0 + chunk).astype(np.int32)
    dec_ctx = np.concatenate([rng.integers(1024, 32768, size=240, endpoint=True),
                              np.full(8, 131072)])
    dec_ctx = np.maximum(1, np.rint(dec_ctx * decode_scale)).astype(np.int32)

    dec_counts = _nblocks(dec_ctx, bs)
    pre_counts = _nblocks(pre_ctx, bs)
    nb = _pool_with_headroom(int(dec_counts.sum() + pre_counts.sum()))
    ids = rng.permutation(nb).astype(np.int32)
    dec_tables = _tables(dec_counts, int(dec_counts.max()), ids)
    pre_tables = _tables(pre_counts, int(pre_counts.max()), ids[int(dec_counts.sum()):])
    return Step(
        name="mixed_prefill8x512_decode248_h32kv8_d128_bf16_bs32", shape=shape, num_blocks=nb,
        seed=53_004, scale=1.0 / np.sqrt(shape.head_dim),
        decode=Batch(dec_ctx, np.ones_like(dec_ctx), dec_tables),
        prefill=Batch(pre_ctx, np.full(8, chunk, dtype=np.int32), pre_tables))


def mixed_prefill_only() -> Step:
    """The mixed workload's prefill batch alone (8 chunks of 512 over the same contexts),
    on a pool that holds just its blocks: the chunked-prefill case for timing and
    profiling."""
    pre = mixed_prefill_decode().prefill
    return prefill_step("mixed_prefill8x512_h32kv8_d128_bf16_bs32", Shape(32, 8, 128, 32, "bf16"),
                        pre.context_lens, pre.query_lens, 53_004)


NAMED = {
    "tiny_decode": tiny_decode,
    "opt13b_decode": opt13b_decode,
    "llama8b_gqa_decode": llama8b_gqa_decode,
    "prefix_sharing_cow": prefix_sharing_cow,
    "mixed_prefill_decode": mixed_prefill_decode,
    "mixed_prefill_only": mixed_prefill_only,
}


# ----------------------------------------------------------------------------------
# Values
# ----------------------------------------------------------------------------------

def _torch_dtype(dtype: str):
    import torch
    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]


def randn(shape, dtype: str, device, generator, chunk_elems: int = 1 << 27):
    """N(0, 1) drawn as float32 and rounded to `dtype`, filled in chunks so that a
    multi-GB pool never needs a float32 copy of itself."""
    import torch
    out = torch.empty(tuple(shape), dtype=_torch_dtype(dtype), device=device)
    flat = out.view(-1)
    for start in range(0, flat.numel(), chunk_elems):
        n = min(chunk_elems, flat.numel() - start)
        flat[start:start + n] = torch.randn(n, dtype=torch.float32, device=device,
                                            generator=generator).to(flat.dtype)
    return out


def make_values(step: Step, device="cpu") -> Dict[str, "object"]:
    """Random q/K/V for `step`, as torch tensors on `device`.

    Returns k_cache/v_cache [num_blocks, H_kv, block_size, D] (the pool before the step;
    slots not yet written hold noise too), and per batch kind ('decode', 'prefill'):
    q_<kind> [new tokens, H_q, D], k_new_<kind>/v_new_<kind> [new tokens, H_kv, D].
    """
    import torch
    sh = step.shape
    gen = torch.Generator(device=device)
    gen.manual_seed(step.seed)
    vals = {
        "k_cache": randn((step.num_blocks, sh.num_kv_heads, sh.block_size, sh.head_dim),
                         sh.dtype, device, gen),
        "v_cache": randn((step.num_blocks, sh.num_kv_heads, sh.block_size, sh.head_dim),
                         sh.dtype, device, gen),
    }
    for kind in ("decode", "prefill"):
        batch = getattr(step, kind)
        if batch is None:
            continue
        t = batch.num_new_tokens
        vals[f"q_{kind}"] = randn((t, sh.num_q_heads, sh.head_dim), sh.dtype, device, gen)
        vals[f"k_new_{kind}"] = randn((t, sh.num_kv_heads, sh.head_dim), sh.dtype, device, gen)
        vals[f"v_new_{kind}"] = randn((t, sh.num_kv_heads, sh.head_dim), sh.dtype, device, gen)
    return vals


def to_numpy(t) -> np.ndarray:
    """A CPU copy of a torch tensor as numpy; bfloat16 comes back as its uint16 bits."""
    import torch
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def replace(step: Step, **kw) -> Step:
    return dataclasses.replace(step, **kw)
