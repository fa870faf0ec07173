/*
 * pa_testing.h -- entry points of libpagedattn.so that exist for tests of its internals.
 *
 * They are not part of the serving interface (pa.h) and may change with the kernels.
 * Every convention of pa.h (layouts, device pointers, streams, errors, status bits)
 * applies.
 */
#ifndef PAGED_KV_CACHE_PA_TESTING_H_
#define PAGED_KV_CACHE_PA_TESTING_H_

#include <stddef.h>
#include <stdint.h>

#include "pa.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * pa_testing_decode_partitions -- pa_decode with the split-KV partition length fixed by
 * the caller.
 *
 * pa_decode cuts each context into partitions whose length it picks on the device from
 * the whole batch, and merges their partial softmax results by log-sum-exp rescaling.
 * The pages define only the attention itself ("PagedAttention and Continuous Batching
 * Explained (2026)", FAQ "Is PagedAttention a different attention algorithm?": the same
 * result as attention over a contiguous cache), so the result may not depend on how a
 * context is partitioned.  This call lets a test choose the partitioning: every context
 * is cut into partitions of `part_blocks` whole blocks (the last one shorter), so that
 * one sequence of n blocks can be run with any partition count from ceil(n / 128) up to
 * n (one block per partition).
 *
 *   part_blocks    1 .. 128 blocks per partition (PA_ERR_INVALID_ARG otherwise)
 *   workspace      at least pa_testing_decode_workspace_bytes(..., part_blocks) bytes
 * Every other argument as in pa_decode.  Same kernels, same result up to the rounding of
 * a different summation order.
 */
size_t pa_testing_decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                         int head_dim, int max_ctx, int block_size,
                                         int part_blocks);
int pa_testing_decode_partitions(void* out, pa_dtype out_dtype, const void* q,
                                 const void* k_cache, const void* v_cache,
                                 const int32_t* block_tables, int max_blocks_per_seq,
                                 const int32_t* context_lens, int max_ctx, int num_seqs,
                                 int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                 int num_blocks, float scale, pa_dtype dtype, int part_blocks,
                                 void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_KV_CACHE_PA_TESTING_H_ */
