// Bit-exact cache operations: slot mapping, cache write (reshape_and_cache) and
// copy-on-write block copies.  All three are pure data movement bounded by HBM (or, at
// decode sizes, by launch latency); each thread moves 16-byte vectors.
#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_launch.h"

namespace pa {
namespace {

// One warp per sequence; its lanes walk the sequence's new tokens.  Token t of
// sequence b (cu_q_lens[b] <= t < cu_q_lens[b+1]) is the matching tail position of the
// sequence's context.
__global__ void __launch_bounds__(256) slot_mapping_kernel(
    int64_t* __restrict__ slots, const int32_t* __restrict__ block_tables, int max_blocks,
    const int32_t* __restrict__ cu_q_lens, const int32_t* __restrict__ context_lens,
    int num_seqs, int num_tokens, int block_size, int num_blocks, int32_t* status) {
  griddep_wait();
  griddep_launch_dependents();
  const int b = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (b >= num_seqs) return;
  const int first = __ldg(cu_q_lens + b);
  const int n_new = __ldg(cu_q_lens + b + 1) - first;
  const long long ctx = __ldg(context_lens + b);
  const int32_t* row = block_tables + (size_t)b * max_blocks;
  for (int i = lane; i < n_new; i += 32) {
    const long long t = (long long)first + i;
    if (t < 0 || t >= num_tokens) {
      flag_status(status, PA_STATUS_BAD_CONTEXT);
      continue;
    }
    const long long pos = ctx - n_new + i;
    if (pos < 0 || pos >= (long long)max_blocks * block_size) {
      flag_status(status, PA_STATUS_BAD_CONTEXT);
      slots[t] = -1;
      continue;
    }
    const int blk = __ldg(row + pos / block_size);
    if (blk < 0 || blk >= num_blocks) {
      flag_status(status, PA_STATUS_BAD_BLOCK);
      slots[t] = -1;
      continue;
    }
    slots[t] = (int64_t)blk * block_size + pos % block_size;
  }
}

// One thread per 16-byte chunk of one (token, KV head) row; K and V move together.
__global__ void reshape_and_cache_kernel(const uint4* __restrict__ k_new,
                                         const uint4* __restrict__ v_new, uint4* __restrict__ k_cache,
                                         uint4* __restrict__ v_cache,
                                         const int64_t* __restrict__ slots, int num_tokens,
                                         int num_kv_heads, int chunks_per_row, int block_size,
                                         long long num_slots, int32_t* status) {
  griddep_wait();
  griddep_launch_dependents();
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long per_token = (long long)num_kv_heads * chunks_per_row;
  if (i >= (long long)num_tokens * per_token) return;
  const long long t = i / per_token;
  const int rem = (int)(i - t * per_token);
  const int h = rem / chunks_per_row;
  const int c = rem - h * chunks_per_row;
  const long long slot = __ldg(slots + t);
  if (slot < 0) return;  // padding token
  if (slot >= num_slots) {
    if (rem == 0) flag_status(status, PA_STATUS_BAD_SLOT);
    return;
  }
  const long long blk = slot / block_size, off = slot - blk * block_size;
  const long long dst = ((blk * num_kv_heads + h) * block_size + off) * chunks_per_row + c;
  const long long src = i;
  k_cache[dst] = __ldg(k_new + src);
  v_cache[dst] = __ldg(v_new + src);
}

// Slot mapping fused with the cache write: CTA (x, b) takes up to kAppendTokens new
// tokens of sequence b, computes their slots, then moves their K and V rows in 16-byte
// chunks with all of its threads.
constexpr int kAppendTokens = 8;

__global__ void __launch_bounds__(256) cache_append_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new, uint4* __restrict__ k_cache,
    uint4* __restrict__ v_cache, int64_t* __restrict__ slots_out,
    const int32_t* __restrict__ block_tables, int max_blocks, const int32_t* __restrict__ cu_q_lens,
    const int32_t* __restrict__ context_lens, int num_tokens, int num_kv_heads,
    int chunks_per_row, int block_size, int num_blocks, int32_t* status) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ long long s_slot[kAppendTokens];
  const int b = blockIdx.y;
  // no cu_q_lens: one new token per sequence, token b for sequence b (a decode step)
  const int first = cu_q_lens != nullptr ? __ldg(cu_q_lens + b) : b;
  const int n_new = cu_q_lens != nullptr ? __ldg(cu_q_lens + b + 1) - first : 1;
  const int i0 = blockIdx.x * kAppendTokens;
  if (i0 >= n_new) return;
  const int nt = min(kAppendTokens, n_new - i0);
  if (threadIdx.x < nt) {
    const int i = i0 + threadIdx.x;
    const long long t = (long long)first + i;
    long long slot = -1;
    const long long pos = (long long)__ldg(context_lens + b) - n_new + i;
    if (t < 0 || t >= num_tokens || pos < 0 || pos >= (long long)max_blocks * block_size) {
      flag_status(status, PA_STATUS_BAD_CONTEXT);
    } else {
      const int blk = __ldg(block_tables + (size_t)b * max_blocks + pos / block_size);
      if (blk < 0 || blk >= num_blocks)
        flag_status(status, PA_STATUS_BAD_BLOCK);
      else
        slot = (long long)blk * block_size + pos % block_size;
    }
    s_slot[threadIdx.x] = slot;
    if (slots_out != nullptr && t >= 0 && t < num_tokens) slots_out[t] = slot;
  }
  __syncthreads();
  const int per_tok = num_kv_heads * chunks_per_row;
  for (int c = threadIdx.x; c < nt * per_tok; c += blockDim.x) {
    const int ti = c / per_tok, rem = c - ti * per_tok;
    const long long slot = s_slot[ti];
    if (slot < 0) continue;
    const int h = rem / chunks_per_row, cc = rem - h * chunks_per_row;
    const long long blk = slot / block_size, off = slot - blk * block_size;
    const long long dst = ((blk * num_kv_heads + h) * block_size + off) * chunks_per_row + cc;
    const long long src = ((long long)(first + i0 + ti) * num_kv_heads + h) * chunks_per_row + cc;
    k_cache[dst] = __ldg(k_new + src);
    v_cache[dst] = __ldg(v_new + src);
  }
}

struct LayerPtrs {
  uint4* k[kMaxCopyLayers];
  uint4* v[kMaxCopyLayers];
};

// One CTA per (pair, layer, K-or-V); the CTA copies one whole block (all KV heads).
__global__ void __launch_bounds__(256) copy_blocks_kernel(const __grid_constant__ LayerPtrs ptrs,
                                                          const int32_t* __restrict__ pairs,
                                                          int chunks_per_block, int num_blocks,
                                                          int32_t* status) {
  griddep_wait();
  griddep_launch_dependents();
  const int pair = blockIdx.x, layer = blockIdx.y;
  const int src = __ldg(pairs + 2 * pair), dst = __ldg(pairs + 2 * pair + 1);
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0 && blockIdx.z == 0) flag_status(status, PA_STATUS_BAD_BLOCK);
    return;
  }
  uint4* base = blockIdx.z == 0 ? ptrs.k[layer] : ptrs.v[layer];
  const uint4* s = base + (size_t)src * chunks_per_block;
  uint4* d = base + (size_t)dst * chunks_per_block;
  for (int c = threadIdx.x; c < chunks_per_block; c += blockDim.x) d[c] = __ldg(s + c);
}

struct SwapPtrs {
  const uint4* src_k[kMaxSwapLayers];
  const uint4* src_v[kMaxSwapLayers];
  uint4* dst_k[kMaxSwapLayers];
  uint4* dst_v[kMaxSwapLayers];
};

// Whole-block copies from one pool to another (device memory or pinned host memory
// reached through the unified address space): one CTA per (pair, layer, K-or-V).
__global__ void __launch_bounds__(256) swap_blocks_kernel(const __grid_constant__ SwapPtrs ptrs,
                                                          const int32_t* __restrict__ pairs,
                                                          int chunks_per_block, int src_blocks,
                                                          int dst_blocks, int32_t* status) {
  griddep_wait();
  griddep_launch_dependents();
  const int pair = blockIdx.x, layer = blockIdx.y;
  const int src = pairs[2 * pair], dst = pairs[2 * pair + 1];
  if (src < 0 || src >= src_blocks || dst < 0 || dst >= dst_blocks) {
    if (threadIdx.x == 0 && blockIdx.z == 0) flag_status(status, PA_STATUS_BAD_BLOCK);
    return;
  }
  const uint4* s = (blockIdx.z == 0 ? ptrs.src_k[layer] : ptrs.src_v[layer]) +
                   (size_t)src * chunks_per_block;
  uint4* d = (blockIdx.z == 0 ? ptrs.dst_k[layer] : ptrs.dst_v[layer]) +
             (size_t)dst * chunks_per_block;
  // four independent 16-byte loads in flight per thread: host memory is far away
  int c = threadIdx.x;
  for (; c + 3 * blockDim.x < chunks_per_block; c += 4 * blockDim.x) {
    const uint4 a = s[c], b = s[c + blockDim.x], e = s[c + 2 * blockDim.x],
                f = s[c + 3 * blockDim.x];
    d[c] = a;
    d[c + blockDim.x] = b;
    d[c + 2 * blockDim.x] = e;
    d[c + 3 * blockDim.x] = f;
  }
  for (; c < chunks_per_block; c += blockDim.x) d[c] = s[c];
}

}  // namespace

cudaError_t launch_swap_blocks(void* const* src_k, void* const* src_v, void* const* dst_k,
                               void* const* dst_v, int num_layers, const int32_t* pairs,
                               int num_pairs, size_t block_bytes, int src_blocks,
                               int dst_blocks, int32_t* status, cudaStream_t stream) {
  SwapPtrs ptrs;
  for (int l = 0; l < num_layers; ++l) {
    ptrs.src_k[l] = static_cast<const uint4*>(src_k[l]);
    ptrs.src_v[l] = static_cast<const uint4*>(src_v[l]);
    ptrs.dst_k[l] = static_cast<uint4*>(dst_k[l]);
    ptrs.dst_v[l] = static_cast<uint4*>(dst_v[l]);
  }
  return launch_pdl(swap_blocks_kernel, dim3(num_pairs, num_layers, 2), dim3(256), 0, stream,
                    ptrs, pairs, (int)(block_bytes / 16), src_blocks, dst_blocks, status);
}

cudaError_t launch_slot_mapping(int64_t* slots, const int32_t* block_tables, int max_blocks,
                                const int32_t* cu_q_lens, const int32_t* context_lens,
                                int num_seqs, int num_tokens, int block_size, int num_blocks,
                                int32_t* status, cudaStream_t stream) {
  const int warps_per_cta = 8;
  return launch_pdl(slot_mapping_kernel, dim3((num_seqs + warps_per_cta - 1) / warps_per_cta),
                    dim3(32 * warps_per_cta), 0, stream, slots, block_tables, max_blocks,
                    cu_q_lens, context_lens, num_seqs, num_tokens, block_size, num_blocks, status);
}

cudaError_t launch_reshape_and_cache(const void* k_new, const void* v_new, void* k_cache,
                                     void* v_cache, const int64_t* slots, int num_tokens,
                                     int num_kv_heads, int head_dim, int block_size,
                                     int num_blocks, size_t elem_bytes, int32_t* status,
                                     cudaStream_t stream) {
  const int chunks_per_row = (int)(head_dim * elem_bytes / 16);
  const long long total = (long long)num_tokens * num_kv_heads * chunks_per_row;
  const int threads = 256;
  const long long grid = (total + threads - 1) / threads;
  if (grid > 0x7fffffffll) return cudaErrorInvalidValue;
  return launch_pdl(reshape_and_cache_kernel, dim3((unsigned)grid), dim3(threads), 0, stream,
                    static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
                    static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), slots,
                    num_tokens, num_kv_heads, chunks_per_row, block_size,
                    (long long)num_blocks * block_size, status);
}

cudaError_t launch_cache_append(const void* k_new, const void* v_new, void* k_cache,
                                void* v_cache, int64_t* slots, const int32_t* block_tables,
                                int max_blocks, const int32_t* cu_q_lens,
                                const int32_t* context_lens, int num_seqs, int num_tokens,
                                int max_q, int num_kv_heads, int head_dim, int block_size,
                                int num_blocks, size_t elem_bytes, int32_t* status,
                                cudaStream_t stream) {
  const int chunks_per_row = (int)(head_dim * elem_bytes / 16);
  const int gx = (max_q + kAppendTokens - 1) / kAppendTokens;
  if (num_seqs > 65535) return cudaErrorInvalidValue;
  return launch_pdl(cache_append_kernel, dim3(gx, num_seqs), dim3(256), 0, stream,
                    static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
                    static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), slots,
                    block_tables, max_blocks, cu_q_lens, context_lens, num_tokens, num_kv_heads,
                    chunks_per_row, block_size, num_blocks, status);
}

cudaError_t launch_copy_blocks(void* const* k_caches, void* const* v_caches, int num_layers,
                               const int32_t* pairs, int num_pairs, size_t block_bytes,
                               int num_blocks, int32_t* status, cudaStream_t stream) {
  LayerPtrs ptrs;
  for (int l = 0; l < num_layers; ++l) {
    ptrs.k[l] = static_cast<uint4*>(k_caches[l]);
    ptrs.v[l] = static_cast<uint4*>(v_caches[l]);
  }
  for (int l = num_layers; l < kMaxCopyLayers; ++l) ptrs.k[l] = ptrs.v[l] = nullptr;
  if (num_pairs > 0x7fffffff || num_layers > 65535) return cudaErrorInvalidValue;
  return launch_pdl(copy_blocks_kernel, dim3(num_pairs, num_layers, 2), dim3(256), 0, stream, ptrs,
                    pairs, (int)(block_bytes / 16), num_blocks, status);
}

}  // namespace pa
