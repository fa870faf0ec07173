/*
 * pa.h -- C ABI of the paged KV-cache attention library (libpagedattn.so, sm_103a).
 *
 * The KV cache of one layer is a pool of fixed-size physical blocks.  A per-sequence
 * block table maps each logical block of a sequence to the physical block holding it,
 * so blocks need not be contiguous, and attention reads K/V through that table
 * ("PagedAttention and Continuous Batching Explained (2026)", section "PagedAttention:
 * a block table for the KV cache"; "KV Cache in Serving Engines: PagedAttention,
 * Continuous Batching, and Prefix Caching", section "Blocks and Block Tables").
 *
 * Conventions shared by every call
 * --------------------------------
 * Layout.  K and V caches are separate arrays [num_blocks, num_kv_heads, block_size,
 *   head_dim], row-major: token `off` of physical block `blk` for KV head `h` starts at
 *   element ((blk * num_kv_heads + h) * block_size + off) * head_dim.  Block tables are
 *   int32 [num_seqs, max_blocks_per_seq] row-major; entries past a sequence's last
 *   block are never read.  Query/output rows are [tokens, num_q_heads, head_dim].
 * Grouped-query attention.  Query head i reads KV head i / (num_q_heads / num_kv_heads).
 * Context length.  context_lens[b] counts every token of sequence b once this step's
 *   new tokens are in the cache (a decode's appended token included).
 * Memory.  Every pointer argument named *_cache, q, out, k_new, v_new, block_tables,
 *   context_lens, cu_q_lens, slot_mapping, pairs and workspace is a DEVICE pointer
 *   owned by the caller and must be 16-byte aligned.  The library allocates no device
 *   memory.  What it keeps between calls: a status word per device, the table of
 *   caller-owned status words (pa_set_stream_status), the fixed scratch array of
 *   pa_decode_static_scratch, per-device handles it looks up once (the device
 *   addresses of that word and array, SM counts, kernel attributes), and the stream and
 *   two events pa_mixed_step creates per device and host thread (freed by
 *   pa_release_thread_resources).  cudaDeviceReset invalidates those handles: do not
 *   call the library on a device after resetting it in the same process.
 * Streams.  `stream` is a cudaStream_t (NULL = legacy default stream).  Every call only
 *   enqueues work on it and returns without synchronising.
 * Errors.  A call returns PA_OK or a PA_ERR_* code.  Arguments are validated on the
 *   host before anything is enqueued; on an error nothing is launched and
 *   pa_last_error_string() (thread-local) says why.  Data-dependent faults found by the
 *   kernels (a block id outside the pool, a slot outside the pool, a context longer
 *   than its table) never trap: the offending access is skipped or reads zeros, and a
 *   bit is set in the device status word read by pa_get_status() (or in the word the
 *   caller gave the call's stream with pa_set_stream_status).
 * Supported shapes.  head_dim in {64, 128}; block_size in {16, 32};
 *   num_q_heads / num_kv_heads in {1, 2, 4, 8, 16}.  dtype PA_F32, PA_F16, PA_BF16 for
 *   cache writes, copies and decode; PA_F16 and PA_BF16 for chunked prefill.
 */
#ifndef PAGED_KV_CACHE_PA_H_
#define PAGED_KV_CACHE_PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { PA_F32 = 0, PA_F16 = 1, PA_BF16 = 2 } pa_dtype;

/* return codes */
#define PA_OK 0
#define PA_ERR_INVALID_ARG 1 /* null/misaligned pointer, bad size, inconsistent shapes */
#define PA_ERR_UNSUPPORTED 2 /* a head_dim, block_size, group size or dtype not built */
#define PA_ERR_WORKSPACE 3   /* workspace smaller than the *_workspace_bytes() figure */
#define PA_ERR_CUDA 4        /* the CUDA runtime refused a launch or a query */
#define PA_ERR_NO_BLOCKS 5   /* the block manager lacks free blocks (pa_block_manager.h) */

/* bits of the device status word */
#define PA_STATUS_BAD_BLOCK 0x1   /* a block id outside [0, num_blocks) was met */
#define PA_STATUS_BAD_SLOT 0x2    /* a slot outside [0, num_blocks * block_size) */
#define PA_STATUS_BAD_CONTEXT 0x4 /* context < 0, or longer than max_ctx / its table */
#define PA_STATUS_TIMEOUT 0x8     /* a pipeline wait in a kernel gave up (never expected) */
#define PA_STATUS_RANGE 0x10      /* reserved: no longer set (pa_prefill_chunk computes V
                                     values outside fp16's range exactly) */

/* Library version: major * 10000 + minor * 100 + patch. */
int pa_version(void);

/* Why the last call on this thread failed ("" after a success). */
const char* pa_last_error_string(void);

/* Reads the current device's status word into *status and clears it.  Synchronises
 * the device.  Returns PA_ERR_CUDA if the device cannot be reached.  Bits of calls on a
 * stream with a word of its own (pa_set_stream_status) do not appear here. */
int pa_get_status(int32_t* status);

/*
 * pa_set_stream_status -- gives the calls on one stream a status word of their own.
 *
 * The device-wide word read by pa_get_status() is shared by every caller on the device,
 * and reading it clears the bits of all of them.  After this call, the kernels of every
 * call enqueued on `stream` (a cudaStream_t of the current device; NULL = the legacy
 * default stream) OR their PA_STATUS_* bits into `*status` instead: an int32 in DEVICE
 * memory, 4-byte aligned, owned by the caller, which the library never reads or clears
 * (the caller reads and zeroes it, e.g. with cudaMemcpyAsync / cudaMemsetAsync on the
 * same stream).  Registering a stream again replaces its word; status = NULL removes the
 * stream's entry.  Remove it before destroying the stream (a later stream may get the
 * same handle).  A call enqueued on a stream picks its word when it is made.  The work
 * pa_mixed_step runs on its own stream reports to the word of the caller's `stream`.
 * At most 64 (device, stream) entries exist at a time: PA_ERR_UNSUPPORTED beyond.
 * Returns PA_ERR_INVALID_ARG for a misaligned word, PA_ERR_CUDA without a device.
 */
int pa_set_stream_status(void* stream, int32_t* status);

/*
 * pa_release_thread_resources -- destroys the stream and the two events pa_mixed_step
 * created for the calling host thread (one set per device it ran on).  Call it before a
 * thread that used pa_mixed_step exits, or whenever it is done with the library; a later
 * pa_mixed_step creates them again.  No work of the thread's pa_mixed_step calls may
 * still be pending when it is called (synchronise their streams first).  Returns
 * PA_ERR_CUDA if a handle could not be destroyed (the others are destroyed regardless).
 */
int pa_release_thread_resources(void);

/* Self-test of the kernels' bounded waits: launches one CTA on `stream` (cudaStream_t,
 * may be null) that waits on a shared-memory mbarrier nothing ever arrives on, with the
 * wait function every pipeline in this library uses, given up after `timeout_us`
 * microseconds (1 .. 2,000,000) instead of the library's 2 s.  The kernel then sets
 * PA_STATUS_TIMEOUT in the status word (the stream's own word if it has one) and returns:
 * the device stays usable, and pa_get_status() reports the bit.  No other effect.  Returns PA_ERR_INVALID_ARG for a
 * timeout out of range, PA_ERR_CUDA if the launch fails. */
int pa_selftest_wait_timeout(int timeout_us, void* stream);

/*
 * pa_slot_mapping -- physical slot of every new token of a step.
 *
 * Blocks are allocated one at a time as a sequence grows, and each new token goes to
 * the slot its position maps to through the table ("PagedAttention: a block table for
 * the KV cache", page cited above).  Sequence b appends the tokens cu_q_lens[b] ..
 * cu_q_lens[b+1]-1 of the step (one for a decode, a chunk for a prefill); they are the
 * last positions of its context, so token t sits at position
 *     pos = context_lens[b] - (cu_q_lens[b+1] - cu_q_lens[b]) + (t - cu_q_lens[b])
 * and gets slot = block_tables[b][pos / block_size] * block_size + pos % block_size.
 *
 *   slots         int64 [num_tokens], written
 *   block_tables  int32 [num_seqs, max_blocks_per_seq]
 *   cu_q_lens     int32 [num_seqs + 1], cu_q_lens[0] = 0, cu_q_lens[num_seqs] = num_tokens
 *   context_lens  int32 [num_seqs]
 * A token whose position falls outside its table or whose block id is outside the pool
 * gets slot -1 and sets a status bit.  Bit-exact.
 */
int pa_slot_mapping(int64_t* slots, const int32_t* block_tables, int max_blocks_per_seq,
                    const int32_t* cu_q_lens, const int32_t* context_lens, int num_seqs,
                    int num_tokens, int block_size, int num_blocks, void* stream);

/*
 * pa_reshape_and_cache -- writes the new tokens' K and V into their slots.
 *
 *   k_new, v_new      [num_tokens, num_kv_heads, head_dim] of `dtype`
 *   k_cache, v_cache  [num_blocks, num_kv_heads, block_size, head_dim] of `dtype`
 *   slot_mapping      int64 [num_tokens]; a negative slot marks padding and is skipped;
 *                     a slot >= num_blocks * block_size is skipped and sets a status bit
 * Slots must be distinct within a call.  A bit copy: bit-exact.
 */
int pa_reshape_and_cache(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                         const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                         int head_dim, int block_size, int num_blocks, pa_dtype dtype,
                         void* stream);

/*
 * pa_cache_append -- slot mapping and cache write of a step's new tokens in one launch.
 *
 * Computes every new token's slot exactly as pa_slot_mapping does and writes its K and
 * V there exactly as pa_reshape_and_cache does, without a slot array round trip.
 *
 *   k_new, v_new    [num_tokens, num_kv_heads, head_dim] of `dtype`, token t of sequence b
 *                   at row cu_q_lens[b] + (t - cu_q_lens[b])
 *   slots           int64 [num_tokens] receiving the slots (-1 for a rejected token), or
 *                   NULL
 *   max_q           bound on every sequence's new-token count cu_q_lens[b+1]-cu_q_lens[b]
 * Other arguments as in pa_slot_mapping and pa_reshape_and_cache.  Bit-exact.
 */
int pa_cache_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                    int64_t* slots, const int32_t* block_tables, int max_blocks_per_seq,
                    const int32_t* cu_q_lens, const int32_t* context_lens, int num_seqs,
                    int num_tokens, int max_q, int num_kv_heads, int head_dim, int block_size,
                    int num_blocks, pa_dtype dtype, void* stream);

/*
 * pa_copy_blocks -- copy-on-write of shared blocks.
 *
 * Sequences may share physical blocks; a shared block is copied only when one of them
 * must append to it ("KV Cache in Serving Engines", section "Sharing Blocks";
 * "PagedAttention and Continuous Batching Explained (2026)", "Sharing").  For every
 * pair (src, dst) and every layer, block dst of the K and the V cache becomes a copy
 * of block src.
 *
 *   k_caches, v_caches  HOST arrays of `num_layers` DEVICE pointers, each a cache as in
 *                       pa_reshape_and_cache (num_layers <= 256)
 *   pairs               int32 [num_pairs, 2] (src, dst), device
 * Destinations must be distinct and must not appear as a source in the same call.  A
 * pair with an id outside [0, num_blocks) is skipped and sets a status bit.  Bit-exact.
 */
int pa_copy_blocks(void* const* k_caches, void* const* v_caches, int num_layers,
                   const int32_t* pairs, int num_pairs, int num_kv_heads, int head_dim,
                   int block_size, int num_blocks, pa_dtype dtype, void* stream);

/*
 * pa_swap_blocks -- whole-block copies between two pools, for pre-emption by swapping a
 * sequence's blocks to host memory and back ("Continuous batching and paged attention",
 * section "Why they depend on each other": recompute versus swap to host memory).
 *
 * For every pair (src, dst) and every layer, block dst of the destination K and V pools
 * becomes a copy of block src of the source pools.  Typically one side is the device
 * pool and the other a host pool of the same geometry in page-locked memory, which the
 * kernel reads or writes directly through the unified address space (over the
 * chip-to-chip link on Grace systems); device-to-device pools work as well.
 *
 *   src_k, src_v, dst_k, dst_v  HOST arrays of `num_layers` pool pointers (num_layers <=
 *                   128), each [blocks, num_kv_heads, block_size, head_dim] of `dtype`,
 *                   16-byte aligned, in this device's memory or in page-locked host
 *                   memory (pageable memory is rejected)
 *   pairs           int32 [num_pairs, 2] (src block, dst block), device or page-locked
 *                   host memory; the block manager's pa_bm_swap_out / pa_bm_swap_in emit
 *                   them
 *   src_num_blocks, dst_num_blocks  blocks in each pool; a pair outside them is skipped
 *                   and sets PA_STATUS_BAD_BLOCK
 * Destinations must be distinct.  Asynchronous on `stream`; the host side must not be
 * read (swap-out) or reused (swap-in) before the stream reaches this point.  Bit-exact.
 */
int pa_swap_blocks(void* const* src_k, void* const* src_v, void* const* dst_k,
                   void* const* dst_v, int num_layers, const int32_t* pairs, int num_pairs,
                   int num_kv_heads, int head_dim, int block_size, int src_num_blocks,
                   int dst_num_blocks, pa_dtype dtype, void* stream);

/*
 * pa_decode_workspace_bytes -- bytes of device workspace pa_decode needs for these
 * sizes (the split-KV partial results and the work list).  max_ctx bounds every
 * context length of the call.
 */
size_t pa_decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                 int head_dim, int max_ctx, int block_size);

/*
 * pa_decode -- paged decode attention: one query token per sequence.
 *
 * For sequence b and query head i, with kv head h = i / (num_q_heads / num_kv_heads):
 *     out[b][i] = sum_j softmax_j(scale * q[b][i] . K_b[j][h]) * V_b[j][h]
 * over the context positions j < context_lens[b], where K_b and V_b are reached through
 * row b of the block table.  This is the same attention as over a contiguous cache
 * ("PagedAttention and Continuous Batching Explained (2026)", FAQ "Is PagedAttention a
 * different attention algorithm?").  Long contexts are split into partitions whose
 * partial results are merged by log-sum-exp rescaling.
 *
 *   out           [num_seqs, num_q_heads, head_dim] of out_dtype (dtype or PA_F32)
 *   q             [num_seqs, num_q_heads, head_dim] of dtype
 *   k/v_cache     [num_blocks, num_kv_heads, block_size, head_dim] of dtype
 *   block_tables  int32 [num_seqs, max_blocks_per_seq]
 *   context_lens  int32 [num_seqs]; every entry must be <= max_ctx and <=
 *                 max_blocks_per_seq * block_size (longer ones are clamped and set a
 *                 status bit); a sequence with context 0 gets a zero output
 *   workspace     device scratch of at least pa_decode_workspace_bytes(...) bytes; its
 *                 contents need no initialisation and are overwritten
 * Accumulation is fp32.  Two calls that share a workspace must not overlap in time.
 */
int pa_decode(void* out, pa_dtype out_dtype, const void* q, const void* k_cache,
              const void* v_cache, const int32_t* block_tables, int max_blocks_per_seq,
              const int32_t* context_lens, int max_ctx, int num_seqs, int num_q_heads,
              int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
              pa_dtype dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * pa_decode_append -- one decode step: write each sequence's new token into the cache,
 * then pa_decode.
 *
 * Equivalent to pa_cache_append with one new token per sequence (row b of k_new / v_new
 * is sequence b's token, at position context_lens[b] - 1; its slot is written to
 * slots[b] if slots is not null) followed by pa_decode on the same arguments: the same
 * cache bytes, slots and outputs.  Inside one call the library knows that the cache write
 * touches nothing the decode's work planning reads, so the planning runs beside the
 * cache write instead of after it.  This is one decode step as the pages describe it:
 * the new token's K and V join the cache kept for every token seen so far, in the block
 * its position maps to through the table, and the token attends over the whole context
 * ("PagedAttention and Continuous Batching Explained (2026)", sections "Why the KV cache
 * is the problem" and "PagedAttention: a block table for the KV cache").
 *
 *   k_new / v_new  [num_seqs, num_kv_heads, head_dim] of dtype, 16-byte aligned
 *   slots          int64 [num_seqs] or null
 * Every other argument, error and status bit as in pa_decode and pa_cache_append (a
 * context length below 1 has no position for the new token: PA_STATUS_BAD_CONTEXT).
 */
int pa_decode_append(void* out, pa_dtype out_dtype, const void* q, const void* k_new,
                     const void* v_new, void* k_cache, void* v_cache, int64_t* slots,
                     const int32_t* block_tables, int max_blocks_per_seq,
                     const int32_t* context_lens, int max_ctx, int num_seqs, int num_q_heads,
                     int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
                     pa_dtype dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * pa_decode_shared_prefix -- pa_decode for a batch in which some sequences share one
 * physical prefix.
 *
 * Sequences may point their tables at the same physical blocks when they share a prompt
 * prefix ("Continuous batching, paged attention, prefix caching", section "Prefix
 * caching": the server keeps one physical copy and points both block tables at it).
 * The result is the same attention as pa_decode's, within the same error bound (the
 * two differ in summation order and rounding, not in what they compute); the work
 * differs: the prefix's attention is computed once per KV head for all the sequences
 * reading it, as one dense contraction of all their query groups with the prefix's K/V on
 * the tensor cores, and merged with each sequence's own remaining context by log-sum-exp
 * rescaling.  The prefix's K/V are read from HBM once instead of once per sequence.  In
 * the prefix's P V, P is one fp16 term for fp16 caches (unit roundoff 2^-11) and a pair
 * of bf16 hi + lo terms for bf16 caches (relative error 2^-17), V as stored.
 *
 *   prefix_blocks  int32 [prefix_len / block_size], the prefix's physical blocks, device
 *   prefix_len     tokens of the prefix, a multiple of block_size
 *   sharers        int32 [num_sharers], distinct indices of the sequences (rows of
 *                  block_tables) whose first prefix_len tokens are that prefix; each must
 *                  have context_lens >= prefix_len (else PA_STATUS_BAD_CONTEXT) and its
 *                  table must start with prefix_blocks (not checked); an index outside
 *                  [0, num_seqs) sets PA_STATUS_BAD_CONTEXT and is skipped
 *   workspace      at least pa_decode_shared_prefix_workspace_bytes(...) bytes
 * Other arguments as in pa_decode; dtype PA_F16 or PA_BF16.  num_sharers = 0 (or
 * prefix_len = 0) is a plain decode.
 */
size_t pa_decode_shared_prefix_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                               int head_dim, int max_ctx, int block_size,
                                               int num_sharers, int prefix_len);
int pa_decode_shared_prefix(void* out, pa_dtype out_dtype, const void* q, const void* k_cache,
                            const void* v_cache, const int32_t* block_tables,
                            int max_blocks_per_seq, const int32_t* context_lens, int max_ctx,
                            int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                            int block_size, int num_blocks, const int32_t* prefix_blocks,
                            int prefix_len, const int32_t* sharers, int num_sharers, float scale,
                            pa_dtype dtype, void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * pa_decode_static_scratch -- pa_decode for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this call; it exists for integration.  A caller that
 * has handed all of the GPU's memory to its own pool (a serving engine typically sizes
 * its KV-block pool to fill the device) or that must not call cudaMalloc/cudaFree on its
 * path (they can synchronise the device) has no workspace to pass.  This call takes the
 * same arguments as pa_decode minus the workspace and computes the same result, using a
 * 32 MiB array compiled into the library as its scratch.  It allocates nothing.
 *
 *   Limit.   Sizes whose pa_decode_workspace_bytes(...) exceeds 32 MiB are rejected
 *            with PA_ERR_WORKSPACE before anything is launched (for example 256
 *            sequences of up to 8192 tokens with 32 query heads of 128 fit; 248
 *            sequences of up to 131072 tokens do not).
 *   Memory.  Every GPU that loads the library reserves the 32 MiB until the process
 *            exits.  The first call on each device looks up the array's device address
 *            (cudaGetSymbolAddress) and keeps it for the later calls; make that first
 *            call before any stream capture.  A device reset invalidates the kept address
 *            (see "Memory" above: do not use the library after cudaDeviceReset).
 *   Sharing. All calls on a device share the one array and it keeps the last call's
 *            contents; each call rewrites what it reads, so nothing has to be cleared
 *            between calls.  Calls that overlap in time on the GPU (different streams,
 *            or different host threads) race on the array and give wrong results:
 *            serialise them.
 */
int pa_decode_static_scratch(void* out, pa_dtype out_dtype, const void* q, const void* k_cache,
                             const void* v_cache, const int32_t* block_tables,
                             int max_blocks_per_seq, const int32_t* context_lens, int max_ctx,
                             int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                             int block_size, int num_blocks, float scale, pa_dtype dtype,
                             void* stream);

/*
 * pa_prefill_workspace_bytes -- bytes of device workspace pa_prefill_chunk needs.
 */
size_t pa_prefill_workspace_bytes(int num_seqs, int num_tokens, int max_q, int num_q_heads,
                                  int num_kv_heads, int head_dim, int max_ctx,
                                  int block_size);

/*
 * pa_prefill_chunk -- causal attention of a chunk of prompt tokens over paged context.
 *
 * Chunked prefill splits a long prompt into pieces processed in separate steps next to
 * decodes ("PagedAttention and Continuous Batching Explained (2026)", section "Chunked
 * prefill").  Sequence b owns query rows cu_q_lens[b] .. cu_q_lens[b+1]-1; its context
 * holds context_lens[b] tokens INCLUDING the chunk, whose K/V must already be in the
 * cache (call pa_reshape_and_cache first).  Query i of the chunk sits at position
 * context_lens[b] - chunk_len + i and attends to positions 0 .. that position:
 *     out[t][i] = sum_{j <= pos(t)} softmax_j(scale * q[t][i] . K_b[j][h]) * V_b[j][h]
 *
 *   out           [num_tokens, num_q_heads, head_dim] of out_dtype (dtype or PA_F32)
 *   q             [num_tokens, num_q_heads, head_dim] of dtype (PA_F16 or PA_BF16)
 *   cu_q_lens     int32 [num_seqs + 1]; max_q >= every chunk length
 *   context_lens  int32 [num_seqs]; chunk_len <= context_lens[b] <= max_ctx
 *   workspace     device scratch of pa_prefill_workspace_bytes(...) bytes (may be 0)
 * QK^T and PV run on the tensor cores with fp32 accumulation.  P and V enter the PV
 * product in fp16 (unit roundoff 2^-11; bf16's 2^-8 alone would not meet a 2e-3 bound):
 * bf16 V values are converted to fp16 in shared memory, which is exact for magnitudes
 * from 2^-14 up to 65520 (below 2^-14 they become fp16 subnormals, within 2^-25).  The
 * work items (sequence, KV head, group of query rows) that meet a V value of 65520 or
 * more are computed again in the same call with V in bf16 and P as two bf16 terms (hi +
 * lo, a relative error of at most 2^-18 per probability), as pa_decode computes them.
 */
int pa_prefill_chunk(void* out, pa_dtype out_dtype, const void* q, const void* k_cache,
                     const void* v_cache, const int32_t* block_tables, int max_blocks_per_seq,
                     const int32_t* cu_q_lens, const int32_t* context_lens, int num_seqs,
                     int num_tokens, int max_q, int max_ctx, int num_q_heads, int num_kv_heads,
                     int head_dim, int block_size, int num_blocks, float scale, pa_dtype dtype,
                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * pa_mixed_step -- one serving step of a batch that mixes decodes and prefill chunks.
 *
 * Prefill and decode share one batch ("KV Cache in Serving Engines", section "New
 * Problem: Long Prefills Pause Decoding"; "Continuous batching, paged attention, prefix
 * caching", section "Throughput against latency"): here the decode half streams K/V from
 * HBM while the prefill half keeps the tensor cores busy, so the two run side by side on
 * disjoint SMs instead of one after the other.  The result is that of
 *     pa_decode_append(decode batch), then
 *     pa_cache_append(prefill batch's new tokens) + pa_prefill_chunk(prefill batch):
 * the same cache bytes, slots and outputs.  The decode runs on `stream`, its attention
 * kernel on about 58% of the SMs; the prefill runs on a stream of the library's own that
 * waits for the work enqueued on `stream` before the call, and `stream` waits for it
 * before any later work (so the call is stream-ordered as usual, under graph capture
 * too).  That stream and its two events are created on the first call per device and
 * host thread and kept for the next ones; pa_release_thread_resources destroys them.
 * The two batches must not share sequences.
 *
 *   dec   the decode batch: one new token per sequence (row b of k_new / v_new), as in
 *         pa_decode_append; null or num_seqs = 0 for none
 *   pre   the prefill batch: num_tokens new tokens in chunks cu_q_lens, as in
 *         pa_cache_append + pa_prefill_chunk; null or num_seqs = 0 for none
 * Errors and status bits as in those calls (the message names pa_mixed_step).
 */
typedef struct {
  void* out;                   /* [num_seqs, num_q_heads, head_dim] of out_dtype */
  pa_dtype out_dtype;          /* dtype or PA_F32 */
  const void* q;               /* [num_seqs, num_q_heads, head_dim] of dtype */
  const void* k_new;           /* [num_seqs, num_kv_heads, head_dim] of dtype */
  const void* v_new;
  int64_t* slots;              /* int64 [num_seqs] or null */
  const int32_t* block_tables; /* int32 [num_seqs, max_blocks_per_seq] */
  int max_blocks_per_seq;
  const int32_t* context_lens; /* int32 [num_seqs], the new token included */
  int max_ctx;
  int num_seqs;
  void* workspace;             /* pa_decode_workspace_bytes(...) bytes */
  size_t workspace_bytes;
} pa_decode_batch;

typedef struct {
  void* out;                   /* [num_tokens, num_q_heads, head_dim] of out_dtype */
  pa_dtype out_dtype;
  const void* q;               /* [num_tokens, num_q_heads, head_dim] of dtype */
  const void* k_new;           /* [num_tokens, num_kv_heads, head_dim] of dtype */
  const void* v_new;
  int64_t* slots;              /* int64 [num_tokens] or null */
  const int32_t* block_tables;
  int max_blocks_per_seq;
  const int32_t* cu_q_lens;    /* int32 [num_seqs + 1] */
  const int32_t* context_lens; /* int32 [num_seqs], the chunk included */
  int max_q;
  int max_ctx;
  int num_seqs;
  int num_tokens;
  void* workspace;             /* pa_prefill_workspace_bytes(...) bytes */
  size_t workspace_bytes;
} pa_prefill_batch;

int pa_mixed_step(const pa_decode_batch* dec, const pa_prefill_batch* pre, void* k_cache,
                  void* v_cache, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                  int num_blocks, float scale, pa_dtype dtype, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_KV_CACHE_PA_H_ */
