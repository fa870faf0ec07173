"""CPU oracle for paged KV-cache attention: plain, slow and obviously correct.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check and the
benchmark's CPU-baseline leg may import this package.  The library under
paged_kv_cache_53_gb300/ never does, and shares no code with it: the two meet only at
the seeded inputs of the `workloads` module.

Everything here is numpy in float64.  Stored inputs (fp32, fp16, or bf16 carried as its
uint16 bit pattern) are first widened to float64, which is exact for all three.

What it computes follows the pages:

* The KV cache is split into fixed-size blocks, and a per-sequence block table maps each
  logical block to the physical block that holds it; blocks need not be contiguous.
  ("PagedAttention and Continuous Batching Explained (2026)", section "PagedAttention:
  a block table for the KV cache"; "KV Cache in Serving Engines: PagedAttention,
  Continuous Batching, and Prefix Caching", section "Blocks and Block Tables".)
* The attention reached through the table is the same attention as over a contiguous
  cache ("PagedAttention and Continuous Batching Explained (2026)", FAQ "Is
  PagedAttention a different attention algorithm?"; "KV Cache in Serving Engines",
  section "Blocks and Block Tables").  So the oracle first walks the table to
  materialise each sequence's logical K and V, then applies textbook
  softmax(scale * q K^T) V.
* Shared blocks are copied only when a sequence must append to one (copy-on-write;
  "KV Cache in Serving Engines", section "Sharing Blocks").
* A chunk of a long prompt is processed in one step alongside decodes ("PagedAttention
  and Continuous Batching Explained (2026)", section "Chunked prefill"); each query
  token of the chunk attends to every context token up to and including its own
  position.

Readings taken where the pages are silent (the block layout, whether a context length
counts the appended token, the grouped-query head mapping, negative slots) are stated on
the functions that depend on them.

Pins: every function here is checked in tests/test_oracle.py against numbers the pages
print, closed forms and invariants, and against torch's CPU scaled-dot-product attention
in float64 on contiguous tensors.

`oracle.block_manager` is the reference for the host-side block manager (allocation,
sharing with copy-on-write, prefix-cache keys with least-recently-used eviction, swap to
host blocks), pinned in tests/test_block_manager_oracle.py.
"""
from .paged_attention import (  # noqa: F401
    blocks_for_tokens,
    copy_blocks,
    decode_attention,
    decode_attention_rows,
    full_blocks,
    gather_context,
    kv_bytes_per_token,
    prefill_chunk_attention,
    prefill_chunk_attention_rows,
    reshape_and_cache,
    slot_mapping,
    swap_blocks,
    tail_waste,
    widen,
)
