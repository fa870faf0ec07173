// Host-side declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

// Records a failure for pa_last_error_string() and returns `code`.
int fail(int code, const char* fmt, ...);
// Empties pa_last_error_string() at the start of an entry point.
void clear_error();

// Device address of the current device's status word (nullptr if unavailable).
int32_t* device_status_word();
// The status word the kernels of a call enqueued on `stream` write: the caller's word
// registered for that stream by pa_set_stream_status, else the device's.
int32_t* status_word(void* stream);

// Streaming-multiprocessor count of the current device (cached per device).
int sm_count();

// Encodes a 2-D TMA descriptor over a K or V cache viewed as rows of head_dim elements
// ([num_blocks * num_kv_heads * block_size, head_dim]); each box is block_size rows by
// 64 elements with the 128-byte swizzle.  Returns a CUresult.
int encode_cache_map(CUtensorMap* map, const void* cache, pa_dtype dtype, int num_blocks,
                     int num_kv_heads, int block_size, int head_dim);

// Encodes a 3-D TMA descriptor over query rows [tokens, num_q_heads, head_dim] for one
// KV head's group: box = 64 elements x group heads x rows_per_box tokens.
int encode_query_map(CUtensorMap* map, const void* q, pa_dtype dtype, int num_tokens,
                     int num_q_heads, int head_dim, int group, int rows_per_box);

inline size_t dtype_bytes(pa_dtype dt) { return dt == PA_F32 ? 4 : 2; }

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ----------------------------------------------------------------------------------
// cache operations (pa_cache_ops.cu)
// ----------------------------------------------------------------------------------
cudaError_t launch_slot_mapping(int64_t* slots, const int32_t* block_tables, int max_blocks,
                                const int32_t* cu_q_lens, const int32_t* context_lens,
                                int num_seqs, int num_tokens, int block_size, int num_blocks,
                                int32_t* status, cudaStream_t stream);

cudaError_t launch_reshape_and_cache(const void* k_new, const void* v_new, void* k_cache,
                                     void* v_cache, const int64_t* slots, int num_tokens,
                                     int num_kv_heads, int head_dim, int block_size,
                                     int num_blocks, size_t elem_bytes, int32_t* status,
                                     cudaStream_t stream);

cudaError_t launch_cache_append(const void* k_new, const void* v_new, void* k_cache,
                                void* v_cache, int64_t* slots, const int32_t* block_tables,
                                int max_blocks, const int32_t* cu_q_lens,
                                const int32_t* context_lens, int num_seqs, int num_tokens,
                                int max_q, int num_kv_heads, int head_dim, int block_size,
                                int num_blocks, size_t elem_bytes, int32_t* status,
                                cudaStream_t stream);

constexpr int kMaxCopyLayers = 256;
constexpr int kMaxSwapLayers = 128;
cudaError_t launch_swap_blocks(void* const* src_k, void* const* src_v, void* const* dst_k,
                               void* const* dst_v, int num_layers, const int32_t* pairs,
                               int num_pairs, size_t block_bytes, int src_blocks,
                               int dst_blocks, int32_t* status, cudaStream_t stream);

cudaError_t launch_copy_blocks(void* const* k_caches, void* const* v_caches, int num_layers,
                               const int32_t* pairs, int num_pairs, size_t block_bytes,
                               int num_blocks, int32_t* status, cudaStream_t stream);

// ----------------------------------------------------------------------------------
// decode (pa_decode.cu)
// ----------------------------------------------------------------------------------

// Split-KV work planning.  A sequence's context is cut into partitions of
// `part_tokens` tokens (a multiple of the block size, chosen on the device from the
// batch's total context so that about kTargetUnits (partition, KV head) units exist);
// the partial results of a multi-partition sequence are merged by a third kernel.
#ifndef PA_DECODE_TARGET_UNITS
#define PA_DECODE_TARGET_UNITS 2048
#endif
constexpr int kTargetUnits = PA_DECODE_TARGET_UNITS;
constexpr int kMinPartBlocks = 2;
constexpr int kMaxPartBlocks = 128;

// One split-KV partition of one sequence, as the plan kernel describes it.
struct PartRec {
  int b;           // sequence
  int p;           // partition index within the sequence
  int tok0;        // first context position of the partition
  int ntok;        // positions in the partition (1 .. part_tokens)
  int part_start;  // global index of the sequence's first partition
  int nparts;      // partitions of the sequence
  int pad0, pad1;
};

struct DecodeWorkspace {
  int* header;        // [0] unit counter, [1] units, [2] part_tokens, [3] partitions,
                      // [4] sequences to merge
  int* part_start;    // [num_seqs + 1] first partition index of each sequence
  int* seq_flags;     // [num_seqs] 1 for a sequence reading the shared prefix (or null)
  int* merge_seqs;    // [num_seqs] the sequences whose partials the merge combines
  PartRec* parts;     // [max_parts] partitions, largest first
  float2* part_ml;    // [max_parts * num_q_heads] (running max in log2 units, sum)
  float* part_acc;    // [max_parts * num_q_heads * head_dim] unnormalised outputs
};

// A prefix of `prefix_len` tokens held once and read by every sequence listed in
// `sharers`: its attention is computed once per KV head for all of them, in `splits`
// pieces of `split_tokens` tokens, into partial slots the plan reserves ahead of each
// sharer's own partitions.  num_sharers = 0 for a plain decode.
struct PrefixPlan {
  const int32_t* sharers;
  const int32_t* prefix_blocks;
  int num_sharers, prefix_len, splits, split_tokens;
  // set at launch: own partitions a sharer may have so that, with its `splits` prefix
  // partials, the merge takes every partial of it in one round (<= 0: no limit)
  int max_own_parts;
};

// forced_psz > 0: every partition has that many tokens (the testing entry point)
size_t decode_max_parts(int num_seqs, int num_kv_heads, int max_ctx, int block_size,
                        int forced_psz = 0);
size_t decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                              int max_ctx, int block_size, long long extra_slots = 0,
                              int forced_psz = 0);
DecodeWorkspace carve_decode_workspace(void* ws, int num_seqs, int num_q_heads,
                                       int num_kv_heads, int head_dim, int max_ctx,
                                       int block_size, long long extra_slots = 0,
                                       int forced_psz = 0);
// Splits of a shared prefix: about two CTAs per SM of work, in whole 128-token tiles.
PrefixPlan plan_prefix(int num_sharers, int prefix_len, int group, int num_kv_heads);

struct DecodeArgs {
  void* out;
  pa_dtype out_dtype;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  int max_blocks;
  const int32_t* context_lens;
  int max_ctx;
  int num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks;
  float scale;
  pa_dtype dtype;
  DecodeWorkspace ws;
  int32_t* status;
  PrefixPlan prefix;  // num_sharers = 0: no shared prefix
  // The plan kernel may run beside the kernel launched just before it on the stream and
  // wait for it only before it exits: set when that kernel is known not to write what the
  // plan reads (context lengths, sharers) nor the output rows it zeroes.
  bool plan_wait_late = false;
  // at most this many CTAs for the attention kernel (0: one per SM), leaving the other SMs
  // to work running beside it on another stream
  int max_ctas = 0;
  // tokens per split-KV partition, a multiple of the block size (0: chosen on the device
  // from the batch); set only by the testing entry point
  int forced_part_tokens = 0;
};

// Attention of a shared prefix for all of its sharers (pa_shared_prefix.cu): writes
// their prefix partials into the slots the decode plan reserved.
int launch_shared_prefix(const DecodeArgs& a, cudaStream_t stream);

// Launches the plan, attention and merge kernels.  Returns PA_OK or a PA_ERR_* code (after
// recording the reason).
int launch_decode(const DecodeArgs& a, cudaStream_t stream);

// ----------------------------------------------------------------------------------
// chunked prefill (pa_prefill.cu)
// ----------------------------------------------------------------------------------
struct PrefillArgs {
  void* out;
  pa_dtype out_dtype;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  int max_blocks;
  const int32_t* cu_q_lens;
  const int32_t* context_lens;
  int num_seqs, num_tokens, max_q, max_ctx;
  int num_q_heads, num_kv_heads, head_dim, block_size, num_blocks;
  float scale;
  pa_dtype dtype;
  void* workspace;
  size_t workspace_bytes;
  int32_t* status;
};

size_t prefill_workspace_bytes(int num_seqs, int num_tokens, int max_q, int num_q_heads,
                               int num_kv_heads, int head_dim, int max_ctx, int block_size);
int launch_prefill(const PrefillArgs& a, cudaStream_t stream);

}  // namespace pa
