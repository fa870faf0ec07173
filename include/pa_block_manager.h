/*
 * pa_block_manager.h -- the host-side block manager of libpagedattn (C ABI).
 *
 * It decides where each sequence's keys and values live in a pool of fixed-size
 * physical blocks, and emits what the device operations of pa.h take: block tables,
 * context lengths, slot mappings, copy-on-write pairs for pa_copy_blocks, and
 * device/host pairs for pa_swap_blocks.
 *
 * What it follows:
 *  - A pool of fixed-size physical blocks; each sequence has a block table from logical
 *    to physical blocks; a block is allocated only when the sequence's last block is
 *    full, and the blocks of a finished sequence are freed at once.
 *    ("PagedAttention and Continuous Batching Explained (2026)", section "PagedAttention:
 *    a block table for the KV cache"; "Continuous batching and paged attention", section
 *    "Paged attention"; "KV Cache in Serving Engines", section "Blocks and Block Tables".)
 *  - Blocks are reference counted and may be read by several sequences; a shared block
 *    is copied only when a sequence needs to append to it (copy-on-write).
 *    ("KV Cache in Serving Engines", section "Sharing Blocks".)
 *  - Admission asks whether enough free blocks exist for a prompt plus a margin
 *    ("Continuous batching and paged attention", section "Paged attention").
 *  - Prefix caching: each full block is keyed by sha256 of its parent block's key, its
 *    token ids and extra keys; a new sequence reuses its leading blocks while their
 *    keys are found; blocks no sequence reads keep their contents in a queue, oldest
 *    evicted first, entered tail first when a sequence finishes.
 *    ("KV Cache in Serving Engines", section "4. Prefix Caching: Computing the Same
 *    Prefix Only Once"; "PagedAttention and Continuous Batching Explained (2026)",
 *    section "Prefix caching".)
 *  - Pre-emption by swapping a sequence's blocks to host memory ("Continuous batching
 *    and paged attention", section "Why they depend on each other").
 *
 * Policies the pages leave open, fixed here:
 *  1. One queue holds every device block no sequence reads, least recently used at the
 *     front: initially blocks 0 .. num_blocks-1 in order.  Allocation takes the front; a
 *     block whose last reader is gone joins the back; a cached block found by a lookup
 *     leaves the queue.  Taking a block that still has a key evicts it (forgets the key).
 *  2. key = sha256(parent key || token ids as little-endian int32 || extra bytes); the
 *     parent key of a sequence's first block is 32 zero bytes.
 *  3. A block is keyed when it becomes full (at admission or by an append), unless
 *     another block already holds the key.  Keys are computed only with prefix caching
 *     on.
 *  4. Copy-on-write: appending into a last block that other sequences also read takes a
 *     new block and records (source, destination); the last reader appends in place.
 *  5. Swap-out gives every distinct device block the listed sequences read one host
 *     block (shared blocks once), from a first-in first-out host free list (initially
 *     0 .. num_host_blocks-1), and drops their device references.  Swap-in maps each
 *     host block to a newly taken device block.  Blocks brought back are not keyed.
 *  6. A call that lacks blocks (or output room) returns PA_ERR_NO_BLOCKS (or
 *     PA_ERR_INVALID_ARG) and changes nothing.
 *
 * Ownership and threads: the manager owns its state; callers own every array they pass.
 * One manager must not be used from two threads at once.  Nothing here touches a GPU.
 * Errors: PA_OK or a PA_ERR_* code of pa.h (reason in pa_last_error_string()).
 */
#ifndef PA_BLOCK_MANAGER_H
#define PA_BLOCK_MANAGER_H

#include <stddef.h>
#include <stdint.h>

#include "pa.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pa_block_manager pa_block_manager;

/* A pool of num_blocks device blocks of block_size tokens (and num_host_blocks host
 * blocks for swapping; 0 disables swapping).  prefix_caching != 0 keys full blocks. */
int pa_bm_create(int num_blocks, int block_size, int prefix_caching, int num_host_blocks,
                 pa_block_manager** out);
void pa_bm_destroy(pa_block_manager* bm);

/* Device blocks no sequence reads (free or cached-but-idle), and free host blocks. */
int pa_bm_num_free_blocks(const pa_block_manager* bm);
int pa_bm_num_free_host_blocks(const pa_block_manager* bm);

/* 1 if ceil(num_tokens / block_size) + watermark_blocks <= free device blocks. */
int pa_bm_can_allocate(const pa_block_manager* bm, int num_tokens, int watermark_blocks);

/* Admits sequence seq_id with its prompt tokens[num_tokens] (num_tokens >= 1) and extra
 * key bytes extra[extra_bytes] (may be null when 0).  With prefix caching, leading full
 * blocks whose keys are cached are reused; *cached_tokens (may be null) receives the
 * number of prompt tokens they hold.  PA_ERR_NO_BLOCKS if the pool cannot hold the
 * prompt; PA_ERR_INVALID_ARG if seq_id exists. */
int pa_bm_add_sequence(pa_block_manager* bm, int64_t seq_id, const int32_t* tokens,
                       int num_tokens, const void* extra, int extra_bytes,
                       int* cached_tokens);

/* Appends tokens[n] to a resident sequence, allocating at block boundaries and copying
 * a shared last block first (the pair is queued for pa_bm_take_copies). */
int pa_bm_append_tokens(pa_block_manager* bm, int64_t seq_id, const int32_t* tokens, int n);

/* pa_bm_append_tokens for n distinct sequences in one call, in the order given: sequence
 * seq_ids[i] appends counts[i] tokens (counts may be null: one each) taken in turn from
 * tokens.  All or nothing: PA_ERR_NO_BLOCKS (or PA_ERR_INVALID_ARG for an unknown,
 * swapped-out or repeated sequence) leaves every sequence as it was. */
int pa_bm_append_tokens_batch(pa_block_manager* bm, const int64_t* seq_ids, int n,
                              const int32_t* tokens, const int32_t* counts);

/* child_id reads every block of parent_id (parallel sampling, beam search). */
int pa_bm_fork(pa_block_manager* bm, int64_t parent_id, int64_t child_id);

/* Drops a finished sequence (resident or swapped out). */
int pa_bm_free_sequence(pa_block_manager* bm, int64_t seq_id);

/* Hands over the queued copy-on-write pairs as pairs[2*i] = source, pairs[2*i+1] =
 * destination, and clears the queue.  *num_pairs receives the count; if it exceeds
 * max_pairs, PA_ERR_INVALID_ARG is returned and nothing is taken. */
int pa_bm_take_copies(pa_block_manager* bm, int32_t* pairs, int max_pairs, int* num_pairs);

/* Moves the listed resident sequences to host blocks.  pairs[2*i] = device block,
 * pairs[2*i+1] = host block, one pair per distinct block, to copy device->host before
 * the device blocks are reused.  PA_ERR_NO_BLOCKS without enough host blocks. */
int pa_bm_swap_out(pa_block_manager* bm, const int64_t* seq_ids, int n, int32_t* pairs,
                   int max_pairs, int* num_pairs);

/* Brings the listed swapped-out sequences back onto new device blocks.  pairs[2*i] =
 * host block, pairs[2*i+1] = device block, to copy host->device before they are read. */
int pa_bm_swap_in(pa_block_manager* bm, const int64_t* seq_ids, int n, int32_t* pairs,
                  int max_pairs, int* num_pairs);

/* Tokens of a sequence, or -1 if unknown. */
int pa_bm_num_tokens(const pa_block_manager* bm, int64_t seq_id);

/* Block tables [n, width] (row-major, unused entries -1) and context lengths [n] of the
 * listed resident sequences; PA_ERR_INVALID_ARG if a table is wider than width. */
int pa_bm_block_tables(const pa_block_manager* bm, const int64_t* seq_ids, int n, int width,
                       int32_t* tables, int32_t* context_lens);

/* Slots (block * block_size + offset) of each listed sequence's last query_lens[i]
 * tokens, sequence after sequence.  *num_slots receives the total; PA_ERR_INVALID_ARG if
 * it exceeds max_slots. */
int pa_bm_slot_mapping(const pa_block_manager* bm, const int64_t* seq_ids, int n,
                       const int32_t* query_lens, int64_t* slots, int max_slots,
                       int* num_slots);

/* Introspection: reference count of a device block, whether it holds a key, and the
 * idle-block queue from least to most recently used (*n receives its length). */
int pa_bm_refcount(const pa_block_manager* bm, int block);
int pa_bm_is_cached(const pa_block_manager* bm, int block);
int pa_bm_free_queue(const pa_block_manager* bm, int32_t* out, int max, int* n);

/* sha256 of data[n] into digest[32] (the block-key hash; exposed for tests). */
void pa_sha256(const void* data, size_t n, uint8_t digest[32]);

#ifdef __cplusplus
}
#endif

#endif /* PA_BLOCK_MANAGER_H */
