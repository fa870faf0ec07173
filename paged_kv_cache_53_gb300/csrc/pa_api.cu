// C-ABI entry points: host-side validation, error reporting, the device status word,
// TMA descriptor encoding, and dispatch to the kernels' launchers.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "pa.h"
#include "pa_device.cuh"
#include "pa_testing.h"
#include "pa_internal.h"

namespace pa {

namespace {

thread_local char g_error[512] = "";

constexpr int kMaxDevices = 64;
__device__ int32_t g_status_word;  // one per device that loads the library

int32_t* g_status_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};
std::mutex g_mutex;

// Caller-owned status words registered per (device, stream) by pa_set_stream_status.
struct StreamStatus {
  int dev;
  cudaStream_t stream;
  int32_t* word;
};
constexpr int kMaxStreamStatus = 64;
StreamStatus g_stream_status[kMaxStreamStatus];
int g_num_stream_status = 0;                 // entries in use (under g_mutex)
std::atomic<int> g_stream_status_used{0};    // the same count, read without the lock

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_dtype(int dt) { return dt == PA_F32 || dt == PA_F16 || dt == PA_BF16; }

bool supported_group(int g) { return g == 1 || g == 2 || g == 4 || g == 8 || g == 16; }

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return g_encode;
}

CUtensorMapDataType tma_dtype(pa_dtype dt) {
  switch (dt) {
    case PA_F16: return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    case PA_BF16: return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    default: return CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  }
}

// Checks shared by every attention / cache call.
int check_cache_geometry(const char* fn, int num_kv_heads, int head_dim, int block_size,
                         int num_blocks, int dtype) {
  if (!valid_dtype(dtype)) return fail(PA_ERR_INVALID_ARG, "%s: unknown dtype %d", fn, dtype);
  if (num_kv_heads <= 0 || num_blocks <= 0 || head_dim <= 0 || block_size <= 0)
    return fail(PA_ERR_INVALID_ARG, "%s: sizes must be positive (kv_heads=%d blocks=%d)", fn,
                num_kv_heads, num_blocks);
  if (head_dim != 64 && head_dim != 128)
    return fail(PA_ERR_UNSUPPORTED, "%s: head_dim %d not built (64, 128)", fn, head_dim);
  if (block_size != 16 && block_size != 32)
    return fail(PA_ERR_UNSUPPORTED, "%s: block_size %d not built (16, 32)", fn, block_size);
  const long long rows = (long long)num_blocks * num_kv_heads * block_size;
  if (rows >= (1ll << 31))
    return fail(PA_ERR_INVALID_ARG, "%s: num_blocks * num_kv_heads * block_size = %lld >= 2^31",
                fn, rows);
  return PA_OK;
}

// The address a kernel on the current device uses for `p`: device or managed memory of
// this device as is, page-locked host memory through its device mapping; null for
// pageable host memory or another device's memory.
void* device_view(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged)
    return at.device == current_device() ? const_cast<void*>(p) : nullptr;
  if (at.type == cudaMemoryTypeHost) return at.devicePointer;
  return nullptr;
}

}  // namespace

void clear_error() { g_error[0] = '\0'; }

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_error, sizeof(g_error), fmt, ap);
  va_end(ap);
  return code;
}

int32_t* device_status_word() {
  const int dev = current_device();
  if (dev < 0) return nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_status_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<int32_t*>(p);
  }
  return g_status_ptr[dev];
}

int32_t* status_word(void* stream) {
  if (g_stream_status_used.load(std::memory_order_acquire) > 0) {
    const int dev = current_device();
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    std::lock_guard<std::mutex> lock(g_mutex);
    for (int i = 0; i < g_num_stream_status; ++i)
      if (g_stream_status[i].dev == dev && g_stream_status[i].stream == s)
        return g_stream_status[i].word;
  }
  return device_status_word();
}

int sm_count() {
  const int dev = current_device();
  if (dev < 0) return 0;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_sm_count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

int encode_cache_map(CUtensorMap* map, const void* cache, pa_dtype dtype, int num_blocks,
                     int num_kv_heads, int block_size, int head_dim) {
  auto enc = encoder();
  if (enc == nullptr) return CUDA_ERROR_NOT_FOUND;
  const cuuint64_t dims[2] = {(cuuint64_t)head_dim,
                              (cuuint64_t)num_blocks * num_kv_heads * block_size};
  const cuuint64_t strides[1] = {(cuuint64_t)head_dim * dtype_bytes(dtype)};
  const cuuint32_t box[2] = {64, (cuuint32_t)block_size};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, tma_dtype(dtype), 2, const_cast<void*>(cache), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

int encode_query_map(CUtensorMap* map, const void* q, pa_dtype dtype, int num_tokens,
                     int num_q_heads, int head_dim, int group, int rows_per_box) {
  auto enc = encoder();
  if (enc == nullptr) return CUDA_ERROR_NOT_FOUND;
  const size_t e = dtype_bytes(dtype);
  const cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)num_q_heads,
                              (cuuint64_t)num_tokens};
  const cuuint64_t strides[2] = {(cuuint64_t)head_dim * e, (cuuint64_t)num_q_heads * head_dim * e};
  const cuuint32_t box[3] = {64, (cuuint32_t)group, (cuuint32_t)rows_per_box};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, tma_dtype(dtype), 3, const_cast<void*>(q), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

namespace {
// One thread waits on an mbarrier initialised for one arrival that never comes.
__global__ void selftest_wait_kernel(uint64_t timeout_ns, int32_t* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(smem_addr(&bar), 1);
  fence_mbar_init();
  if (!mbar_wait(smem_addr(&bar), 0, timeout_ns)) flag_status(status, PA_STATUS_TIMEOUT);
}
}  // namespace

cudaError_t launch_selftest_wait(uint64_t timeout_ns, int32_t* status, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(timeout_ns, status);
  return cudaGetLastError();
}

}  // namespace pa

using namespace pa;

extern "C" {

int pa_version(void) { return 100; }

const char* pa_last_error_string(void) { return g_error; }

int pa_selftest_wait_timeout(int timeout_us, void* stream) {
  pa::clear_error();
  if (timeout_us < 1 || timeout_us > 2000000)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_selftest_wait_timeout: timeout_us %d outside [1, 2e6]",
                    timeout_us);
  int32_t* st = pa::status_word(stream);
  if (st == nullptr) return pa::fail(PA_ERR_CUDA, "pa_selftest_wait_timeout: no usable device");
  const cudaError_t e = pa::launch_selftest_wait((uint64_t)timeout_us * 1000ull, st,
                                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess)
    return pa::fail(PA_ERR_CUDA, "pa_selftest_wait_timeout: %s", cudaGetErrorString(e));
  return PA_OK;
}

int pa_set_stream_status(void* stream, int32_t* status) {
  g_error[0] = '\0';
  const int dev = current_device();
  if (dev < 0) return fail(PA_ERR_CUDA, "pa_set_stream_status: no usable CUDA device");
  if (status != nullptr && (reinterpret_cast<uintptr_t>(status) & 3u))
    return fail(PA_ERR_INVALID_ARG, "pa_set_stream_status: status word must be 4-byte aligned");
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lock(g_mutex);
  int found = -1;
  for (int i = 0; i < g_num_stream_status; ++i)
    if (g_stream_status[i].dev == dev && g_stream_status[i].stream == s) found = i;
  if (status == nullptr) {  // remove the entry (keeping the others packed)
    if (found >= 0) {
      g_stream_status[found] = g_stream_status[g_num_stream_status - 1];
      --g_num_stream_status;
    }
  } else if (found >= 0) {
    g_stream_status[found].word = status;
  } else {
    if (g_num_stream_status == kMaxStreamStatus)
      return fail(PA_ERR_UNSUPPORTED, "pa_set_stream_status: more than %d streams registered",
                  kMaxStreamStatus);
    g_stream_status[g_num_stream_status++] = StreamStatus{dev, s, status};
  }
  g_stream_status_used.store(g_num_stream_status, std::memory_order_release);
  return PA_OK;
}

int pa_get_status(int32_t* status) {
  g_error[0] = '\0';
  if (status == nullptr) return fail(PA_ERR_INVALID_ARG, "pa_get_status: null output pointer");
  int32_t* p = device_status_word();
  if (p == nullptr) return fail(PA_ERR_CUDA, "pa_get_status: no usable CUDA device");
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(status, p, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(p, 0, sizeof(int32_t)) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess)
    return fail(PA_ERR_CUDA, "pa_get_status: %s", cudaGetErrorString(cudaGetLastError()));
  return PA_OK;
}

int pa_slot_mapping(int64_t* slots, const int32_t* block_tables, int max_blocks_per_seq,
                    const int32_t* cu_q_lens, const int32_t* context_lens, int num_seqs,
                    int num_tokens, int block_size, int num_blocks, void* stream) {
  g_error[0] = '\0';
  if (num_seqs < 0 || num_tokens < 0)
    return fail(PA_ERR_INVALID_ARG, "pa_slot_mapping: negative sizes");
  if (num_tokens == 0) return PA_OK;
  if (num_seqs == 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 || block_size <= 0)
    return fail(PA_ERR_INVALID_ARG, "pa_slot_mapping: tokens without sequences or blocks");
  if (!slots || !block_tables || !cu_q_lens || !context_lens)
    return fail(PA_ERR_INVALID_ARG, "pa_slot_mapping: null pointer");
  int32_t* st = status_word(stream);
  if (st == nullptr) return fail(PA_ERR_CUDA, "pa_slot_mapping: no usable CUDA device");
  cudaError_t e = launch_slot_mapping(slots, block_tables, max_blocks_per_seq, cu_q_lens,
                                      context_lens, num_seqs, num_tokens, block_size, num_blocks,
                                      st, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "pa_slot_mapping: %s", cudaGetErrorString(e));
  return PA_OK;
}

int pa_reshape_and_cache(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                         const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                         int head_dim, int block_size, int num_blocks, pa_dtype dtype,
                         void* stream) {
  g_error[0] = '\0';
  if (num_tokens < 0) return fail(PA_ERR_INVALID_ARG, "pa_reshape_and_cache: num_tokens < 0");
  int rc = check_cache_geometry("pa_reshape_and_cache", num_kv_heads, head_dim, block_size,
                                num_blocks, dtype);
  if (rc != PA_OK) return rc;
  if (num_tokens == 0) return PA_OK;
  if (!k_new || !v_new || !k_cache || !v_cache || !slot_mapping)
    return fail(PA_ERR_INVALID_ARG, "pa_reshape_and_cache: null pointer");
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(PA_ERR_INVALID_ARG, "pa_reshape_and_cache: K/V pointers must be 16-byte aligned");
  int32_t* st = status_word(stream);
  if (st == nullptr) return fail(PA_ERR_CUDA, "pa_reshape_and_cache: no usable CUDA device");
  cudaError_t e = launch_reshape_and_cache(k_new, v_new, k_cache, v_cache, slot_mapping,
                                           num_tokens, num_kv_heads, head_dim, block_size,
                                           num_blocks, dtype_bytes(dtype), st,
                                           static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess)
    return fail(PA_ERR_CUDA, "pa_reshape_and_cache: %s", cudaGetErrorString(e));
  return PA_OK;
}

int pa_cache_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                    int64_t* slots, const int32_t* block_tables, int max_blocks_per_seq,
                    const int32_t* cu_q_lens, const int32_t* context_lens, int num_seqs,
                    int num_tokens, int max_q, int num_kv_heads, int head_dim, int block_size,
                    int num_blocks, pa_dtype dtype, void* stream) {
  g_error[0] = '\0';
  if (num_tokens < 0 || num_seqs < 0 || max_q < 0)
    return fail(PA_ERR_INVALID_ARG, "pa_cache_append: negative sizes");
  int rc = check_cache_geometry("pa_cache_append", num_kv_heads, head_dim, block_size, num_blocks,
                                dtype);
  if (rc != PA_OK) return rc;
  if (num_tokens == 0 || num_seqs == 0 || max_q == 0) return PA_OK;
  if (max_blocks_per_seq <= 0)
    return fail(PA_ERR_INVALID_ARG, "pa_cache_append: max_blocks_per_seq <= 0");
  if (!k_new || !v_new || !k_cache || !v_cache || !block_tables || !cu_q_lens || !context_lens)
    return fail(PA_ERR_INVALID_ARG, "pa_cache_append: null pointer");
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(PA_ERR_INVALID_ARG, "pa_cache_append: K/V pointers must be 16-byte aligned");
  int32_t* st = status_word(stream);
  if (st == nullptr) return fail(PA_ERR_CUDA, "pa_cache_append: no usable CUDA device");
  cudaError_t e = launch_cache_append(k_new, v_new, k_cache, v_cache, slots, block_tables,
                                      max_blocks_per_seq, cu_q_lens, context_lens, num_seqs,
                                      num_tokens, max_q, num_kv_heads, head_dim, block_size,
                                      num_blocks, dtype_bytes(dtype), st,
                                      static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "pa_cache_append: %s", cudaGetErrorString(e));
  return PA_OK;
}

int pa_copy_blocks(void* const* k_caches, void* const* v_caches, int num_layers,
                   const int32_t* pairs, int num_pairs, int num_kv_heads, int head_dim,
                   int block_size, int num_blocks, pa_dtype dtype, void* stream) {
  g_error[0] = '\0';
  if (num_pairs < 0 || num_layers < 0)
    return fail(PA_ERR_INVALID_ARG, "pa_copy_blocks: negative sizes");
  int rc = check_cache_geometry("pa_copy_blocks", num_kv_heads, head_dim, block_size, num_blocks,
                                dtype);
  if (rc != PA_OK) return rc;
  if (num_pairs == 0 || num_layers == 0) return PA_OK;
  if (num_layers > kMaxCopyLayers)
    return fail(PA_ERR_UNSUPPORTED, "pa_copy_blocks: %d layers > %d", num_layers, kMaxCopyLayers);
  if (!k_caches || !v_caches || !pairs)
    return fail(PA_ERR_INVALID_ARG, "pa_copy_blocks: null pointer");
  for (int l = 0; l < num_layers; ++l) {
    if (!k_caches[l] || !v_caches[l] || !aligned16(k_caches[l]) || !aligned16(v_caches[l]))
      return fail(PA_ERR_INVALID_ARG, "pa_copy_blocks: layer %d cache pointer null or unaligned",
                  l);
  }
  int32_t* st = status_word(stream);
  if (st == nullptr) return fail(PA_ERR_CUDA, "pa_copy_blocks: no usable CUDA device");
  const size_t block_bytes = (size_t)num_kv_heads * block_size * head_dim * dtype_bytes(dtype);
  cudaError_t e = launch_copy_blocks(k_caches, v_caches, num_layers, pairs, num_pairs,
                                     block_bytes, num_blocks, st,
                                     static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "pa_copy_blocks: %s", cudaGetErrorString(e));
  return PA_OK;
}

int pa_swap_blocks(void* const* src_k, void* const* src_v, void* const* dst_k,
                   void* const* dst_v, int num_layers, const int32_t* pairs, int num_pairs,
                   int num_kv_heads, int head_dim, int block_size, int src_num_blocks,
                   int dst_num_blocks, pa_dtype dtype, void* stream) {
  g_error[0] = '\0';
  if (num_pairs < 0 || num_layers < 0)
    return fail(PA_ERR_INVALID_ARG, "pa_swap_blocks: negative sizes");
  int rc = check_cache_geometry("pa_swap_blocks", num_kv_heads, head_dim, block_size,
                                src_num_blocks, dtype);
  if (rc != PA_OK) return rc;
  rc = check_cache_geometry("pa_swap_blocks", num_kv_heads, head_dim, block_size,
                            dst_num_blocks, dtype);
  if (rc != PA_OK) return rc;
  if (num_pairs == 0 || num_layers == 0) return PA_OK;
  if (num_layers > kMaxSwapLayers)
    return fail(PA_ERR_UNSUPPORTED, "pa_swap_blocks: %d layers > %d", num_layers, kMaxSwapLayers);
  if (!src_k || !src_v || !dst_k || !dst_v || !pairs)
    return fail(PA_ERR_INVALID_ARG, "pa_swap_blocks: null pointer");
  int32_t* st = status_word(stream);
  if (st == nullptr) return fail(PA_ERR_CUDA, "pa_swap_blocks: no usable CUDA device");
  void* views[4][kMaxSwapLayers];
  void* const* in[4] = {src_k, src_v, dst_k, dst_v};
  for (int a = 0; a < 4; ++a)
    for (int l = 0; l < num_layers; ++l) {
      if (!in[a][l] || !aligned16(in[a][l]))
        return fail(PA_ERR_INVALID_ARG, "pa_swap_blocks: layer %d pool pointer null or unaligned",
                    l);
      views[a][l] = device_view(in[a][l]);
      if (views[a][l] == nullptr)
        return fail(PA_ERR_INVALID_ARG,
                    "pa_swap_blocks: layer %d pool is neither this device's memory nor "
                    "page-locked host memory",
                    l);
    }
  const int32_t* pv = static_cast<const int32_t*>(device_view(pairs));
  if (pv == nullptr || (reinterpret_cast<uintptr_t>(pairs) & 3u))
    return fail(PA_ERR_INVALID_ARG,
                "pa_swap_blocks: pairs must be device or page-locked host memory, 4-byte aligned");
  const size_t block_bytes = (size_t)num_kv_heads * block_size * head_dim * dtype_bytes(dtype);
  cudaError_t e = launch_swap_blocks(views[0], views[1], views[2], views[3], num_layers, pv,
                                     num_pairs, block_bytes, src_num_blocks, dst_num_blocks, st,
                                     static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "pa_swap_blocks: %s", cudaGetErrorString(e));
  return PA_OK;
}

size_t pa_decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                 int max_ctx, int block_size) {
  if (num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || max_ctx < 0 ||
      block_size <= 0)
    return 0;
  return decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, max_ctx,
                                block_size);
}

}  // extern "C"

// Checks pa_decode's arguments (naming `who` in errors) and fills the launch arguments.
static int decode_args(const char* who, void* out, pa_dtype out_dtype, const void* q,
                       const void* k_cache, const void* v_cache, const int32_t* block_tables,
                       int max_blocks_per_seq, const int32_t* context_lens, int max_ctx,
                       int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                       int block_size, int num_blocks, float scale, pa_dtype dtype,
                       void* workspace, size_t workspace_bytes, void* stream, DecodeArgs& a) {
  int rc = check_cache_geometry(who, num_kv_heads, head_dim, block_size, num_blocks, dtype);
  if (rc != PA_OK) return rc;
  if (num_seqs < 0 || max_ctx < 0 || num_q_heads <= 0)
    return fail(PA_ERR_INVALID_ARG, "%s: negative sizes", who);
  if (!valid_dtype(out_dtype) || (out_dtype != dtype && out_dtype != PA_F32))
    return fail(PA_ERR_INVALID_ARG, "%s: out_dtype must equal dtype or be PA_F32", who);
  if (num_q_heads % num_kv_heads != 0)
    return fail(PA_ERR_INVALID_ARG, "%s: num_q_heads %d not a multiple of num_kv_heads %d", who,
                num_q_heads, num_kv_heads);
  if (!supported_group(num_q_heads / num_kv_heads))
    return fail(PA_ERR_UNSUPPORTED, "%s: group size %d not built (1, 2, 4, 8, 16)", who,
                num_q_heads / num_kv_heads);
  if (max_blocks_per_seq <= 0) return fail(PA_ERR_INVALID_ARG, "%s: max_blocks_per_seq <= 0", who);
  if (!(scale == scale)) return fail(PA_ERR_INVALID_ARG, "%s: scale is NaN", who);
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !workspace)
    return fail(PA_ERR_INVALID_ARG, "%s: null pointer", who);
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(workspace))
    return fail(PA_ERR_INVALID_ARG, "%s: out/q/caches/workspace must be 16-byte aligned", who);
  const size_t need = decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                             max_ctx, block_size);
  if (workspace_bytes < need)
    return fail(PA_ERR_WORKSPACE, "%s: workspace %zu bytes < %zu needed", who, workspace_bytes,
                need);
  int32_t* st = status_word(stream);
  if (st == nullptr) return fail(PA_ERR_CUDA, "%s: no usable CUDA device", who);
  a.out = out;
  a.out_dtype = out_dtype;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.max_blocks = max_blocks_per_seq;
  a.context_lens = context_lens;
  a.max_ctx = max_ctx;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.scale = scale;
  a.dtype = dtype;
  a.ws = carve_decode_workspace(workspace, num_seqs, num_q_heads, num_kv_heads, head_dim, max_ctx,
                                block_size);
  a.status = st;
  a.prefix = PrefixPlan{};
  return PA_OK;
}

// The cache write of one new token per sequence (row b of k_new / v_new for sequence b),
// then the decode.  The cache write neither reads nor writes what the decode's plan uses:
// the plan builds the work list beside it and waits for it only before it exits.
static int launch_decode_append(const char* who, DecodeArgs& a, const void* k_new,
                                const void* v_new, int64_t* slots, cudaStream_t s) {
  const cudaError_t e = launch_cache_append(
      k_new, v_new, const_cast<void*>(a.k_cache), const_cast<void*>(a.v_cache), slots,
      a.block_tables, a.max_blocks, nullptr, a.context_lens, a.num_seqs, a.num_seqs, 1,
      a.num_kv_heads, a.head_dim, a.block_size, a.num_blocks, dtype_bytes(a.dtype), a.status, s);
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "%s: %s", who, cudaGetErrorString(e));
  a.plan_wait_late = true;
  return launch_decode(a, s);
}

extern "C" {

int pa_decode(void* out, pa_dtype out_dtype, const void* q, const void* k_cache,
              const void* v_cache, const int32_t* block_tables, int max_blocks_per_seq,
              const int32_t* context_lens, int max_ctx, int num_seqs, int num_q_heads,
              int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
              pa_dtype dtype, void* workspace, size_t workspace_bytes, void* stream) {
  g_error[0] = '\0';
  if (num_seqs == 0 && max_ctx >= 0 && num_q_heads > 0 &&
      check_cache_geometry("pa_decode", num_kv_heads, head_dim, block_size, num_blocks, dtype) ==
          PA_OK)
    return PA_OK;
  DecodeArgs a;
  const int rc = decode_args("pa_decode", out, out_dtype, q, k_cache, v_cache, block_tables,
                             max_blocks_per_seq, context_lens, max_ctx, num_seqs, num_q_heads,
                             num_kv_heads, head_dim, block_size, num_blocks, scale, dtype,
                             workspace, workspace_bytes, stream, a);
  if (rc != PA_OK) return rc;
  return launch_decode(a, static_cast<cudaStream_t>(stream));
}

int pa_decode_append(void* out, pa_dtype out_dtype, const void* q, const void* k_new,
                     const void* v_new, void* k_cache, void* v_cache, int64_t* slots,
                     const int32_t* block_tables, int max_blocks_per_seq,
                     const int32_t* context_lens, int max_ctx, int num_seqs, int num_q_heads,
                     int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
                     pa_dtype dtype, void* workspace, size_t workspace_bytes, void* stream) {
  g_error[0] = '\0';
  if (num_seqs == 0 && max_ctx >= 0 && num_q_heads > 0 &&
      check_cache_geometry("pa_decode_append", num_kv_heads, head_dim, block_size, num_blocks,
                           dtype) == PA_OK)
    return PA_OK;
  if (num_seqs > 0 && (!k_new || !v_new))
    return fail(PA_ERR_INVALID_ARG, "pa_decode_append: null pointer");
  if (num_seqs > 0 && (!aligned16(k_new) || !aligned16(v_new)))
    return fail(PA_ERR_INVALID_ARG, "pa_decode_append: K/V pointers must be 16-byte aligned");
  DecodeArgs a;
  int rc = decode_args("pa_decode_append", out, out_dtype, q, k_cache, v_cache, block_tables,
                       max_blocks_per_seq, context_lens, max_ctx, num_seqs, num_q_heads,
                       num_kv_heads, head_dim, block_size, num_blocks, scale, dtype, workspace,
                       workspace_bytes, stream, a);
  if (rc != PA_OK) return rc;
  return launch_decode_append("pa_decode_append", a, k_new, v_new, slots,
                              static_cast<cudaStream_t>(stream));
}

// Partial slots the prefix's splits add to the decode workspace (none without sharers,
// which also leaves the workspace without per-sequence prefix flags).
static long long prefix_slots(const PrefixPlan& pp) {
  return pp.num_sharers > 0 ? (long long)pp.num_sharers * pp.splits : 0;
}

size_t pa_decode_shared_prefix_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                               int head_dim, int max_ctx, int block_size,
                                               int num_sharers, int prefix_len) {
  if (num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || max_ctx < 0 ||
      block_size <= 0 || num_sharers < 0 || prefix_len < 0 || num_q_heads % num_kv_heads != 0)
    return 0;
  const PrefixPlan pp =
      plan_prefix(num_sharers, prefix_len, num_q_heads / num_kv_heads, num_kv_heads);
  return decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, max_ctx,
                                block_size, prefix_slots(pp));
}

int pa_decode_shared_prefix(void* out, pa_dtype out_dtype, const void* q, const void* k_cache,
                            const void* v_cache, const int32_t* block_tables,
                            int max_blocks_per_seq, const int32_t* context_lens, int max_ctx,
                            int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                            int block_size, int num_blocks, const int32_t* prefix_blocks,
                            int prefix_len, const int32_t* sharers, int num_sharers, float scale,
                            pa_dtype dtype, void* workspace, size_t workspace_bytes,
                            void* stream) {
  g_error[0] = '\0';
  int rc = check_cache_geometry("pa_decode_shared_prefix", num_kv_heads, head_dim, block_size,
                                num_blocks, dtype);
  if (rc != PA_OK) return rc;
  if (dtype == PA_F32)
    return fail(PA_ERR_UNSUPPORTED, "pa_decode_shared_prefix: fp16/bf16 only (tensor cores)");
  if (num_seqs < 0 || max_ctx < 0 || num_q_heads <= 0 || num_sharers < 0 || prefix_len < 0)
    return fail(PA_ERR_INVALID_ARG, "pa_decode_shared_prefix: negative sizes");
  if (num_seqs == 0) return PA_OK;
  if (!valid_dtype(out_dtype) || (out_dtype != dtype && out_dtype != PA_F32))
    return fail(PA_ERR_INVALID_ARG,
                "pa_decode_shared_prefix: out_dtype must equal dtype or be PA_F32");
  if (num_q_heads % num_kv_heads != 0 || !supported_group(num_q_heads / num_kv_heads))
    return fail(PA_ERR_UNSUPPORTED, "pa_decode_shared_prefix: group size not built");
  if (max_blocks_per_seq <= 0)
    return fail(PA_ERR_INVALID_ARG, "pa_decode_shared_prefix: max_blocks_per_seq <= 0");
  if (prefix_len % block_size != 0 || prefix_len > max_ctx)
    return fail(PA_ERR_INVALID_ARG,
                "pa_decode_shared_prefix: prefix_len %d must be a multiple of the block size "
                "and <= max_ctx",
                prefix_len);
  if (!(scale == scale)) return fail(PA_ERR_INVALID_ARG, "pa_decode_shared_prefix: scale is NaN");
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !workspace ||
      (num_sharers > 0 && prefix_len > 0 && (!sharers || !prefix_blocks)))
    return fail(PA_ERR_INVALID_ARG, "pa_decode_shared_prefix: null pointer");
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(workspace))
    return fail(PA_ERR_INVALID_ARG,
                "pa_decode_shared_prefix: out/q/caches/workspace must be 16-byte aligned");
  const size_t need = pa_decode_shared_prefix_workspace_bytes(
      num_seqs, num_q_heads, num_kv_heads, head_dim, max_ctx, block_size, num_sharers,
      prefix_len);
  if (workspace_bytes < need)
    return fail(PA_ERR_WORKSPACE, "pa_decode_shared_prefix: workspace %zu bytes < %zu needed",
                workspace_bytes, need);
  int32_t* st = status_word(stream);
  if (st == nullptr) return fail(PA_ERR_CUDA, "pa_decode_shared_prefix: no usable CUDA device");
  DecodeArgs a;
  a.out = out;
  a.out_dtype = out_dtype;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.max_blocks = max_blocks_per_seq;
  a.context_lens = context_lens;
  a.max_ctx = max_ctx;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.scale = scale;
  a.dtype = dtype;
  a.prefix = plan_prefix(num_sharers, prefix_len, num_q_heads / num_kv_heads, num_kv_heads);
  a.prefix.sharers = sharers;
  a.prefix.prefix_blocks = prefix_blocks;
  a.ws = carve_decode_workspace(workspace, num_seqs, num_q_heads, num_kv_heads, head_dim, max_ctx,
                                block_size, prefix_slots(a.prefix));
  a.status = st;
  return launch_decode(a, static_cast<cudaStream_t>(stream));
}

size_t pa_testing_decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                         int head_dim, int max_ctx, int block_size,
                                         int part_blocks) {
  if (num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || max_ctx < 0 ||
      block_size <= 0 || part_blocks < 1 || part_blocks > kMaxPartBlocks)
    return 0;
  return decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, max_ctx,
                                block_size, 0, part_blocks * block_size);
}

int pa_testing_decode_partitions(void* out, pa_dtype out_dtype, const void* q,
                                 const void* k_cache, const void* v_cache,
                                 const int32_t* block_tables, int max_blocks_per_seq,
                                 const int32_t* context_lens, int max_ctx, int num_seqs,
                                 int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                 int num_blocks, float scale, pa_dtype dtype, int part_blocks,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  g_error[0] = '\0';
  const char* who = "pa_testing_decode_partitions";
  if (part_blocks < 1 || part_blocks > kMaxPartBlocks)
    return fail(PA_ERR_INVALID_ARG, "%s: part_blocks %d outside [1, %d]", who, part_blocks,
                kMaxPartBlocks);
  if (num_seqs == 0) return PA_OK;
  // the plain checks with the default workspace size, then the forced size's own
  DecodeArgs a;
  const size_t need = pa_testing_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads,
                                                        head_dim, max_ctx, block_size,
                                                        part_blocks);
  if (need == 0) return fail(PA_ERR_INVALID_ARG, "%s: bad sizes", who);
  if (workspace_bytes < need)
    return fail(PA_ERR_WORKSPACE, "%s: workspace %zu bytes < %zu needed", who, workspace_bytes,
                need);
  const int rc = decode_args(who, out, out_dtype, q, k_cache, v_cache, block_tables,
                             max_blocks_per_seq, context_lens, max_ctx, num_seqs, num_q_heads,
                             num_kv_heads, head_dim, block_size, num_blocks, scale, dtype,
                             workspace, ~size_t(0), stream, a);
  if (rc != PA_OK) return rc;
  a.forced_part_tokens = part_blocks * block_size;
  a.ws = carve_decode_workspace(workspace, num_seqs, num_q_heads, num_kv_heads, head_dim, max_ctx,
                                block_size, 0, a.forced_part_tokens);
  return launch_decode(a, static_cast<cudaStream_t>(stream));
}

size_t pa_prefill_workspace_bytes(int num_seqs, int num_tokens, int max_q, int num_q_heads,
                                  int num_kv_heads, int head_dim, int max_ctx, int block_size) {
  if (num_seqs <= 0 || num_tokens < 0 || max_q < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
      head_dim <= 0 || max_ctx < 0 || block_size <= 0)
    return 0;
  return prefill_workspace_bytes(num_seqs, num_tokens, max_q, num_q_heads, num_kv_heads, head_dim,
                                 max_ctx, block_size);
}

}  // extern "C"

// Checks pa_prefill_chunk's arguments (naming `who` in errors) and fills the launch
// arguments.  *empty is set when there is nothing to do (no sequences or tokens).
static int prefill_args(const char* who, void* out, pa_dtype out_dtype, const void* q,
                        const void* k_cache, const void* v_cache, const int32_t* block_tables,
                        int max_blocks_per_seq, const int32_t* cu_q_lens,
                        const int32_t* context_lens, int num_seqs, int num_tokens, int max_q,
                        int max_ctx, int num_q_heads, int num_kv_heads, int head_dim,
                        int block_size, int num_blocks, float scale, pa_dtype dtype,
                        void* workspace, size_t workspace_bytes, void* stream, PrefillArgs& a,
                        bool* empty) {
  *empty = false;
  int rc = check_cache_geometry(who, num_kv_heads, head_dim, block_size, num_blocks, dtype);
  if (rc != PA_OK) return rc;
  if (dtype == PA_F32)
    return fail(PA_ERR_UNSUPPORTED, "%s: fp32 runs on decode only (f16/bf16 here)", who);
  if (num_seqs < 0 || num_tokens < 0 || max_q < 0 || max_ctx < 0 || num_q_heads <= 0)
    return fail(PA_ERR_INVALID_ARG, "%s: negative sizes", who);
  if (num_seqs == 0 || num_tokens == 0) {
    *empty = true;
    return PA_OK;
  }
  if (!valid_dtype(out_dtype) || (out_dtype != dtype && out_dtype != PA_F32))
    return fail(PA_ERR_INVALID_ARG, "%s: out_dtype must equal dtype or be PA_F32", who);
  if (num_q_heads % num_kv_heads != 0)
    return fail(PA_ERR_INVALID_ARG, "%s: num_q_heads %d not a multiple of num_kv_heads %d", who,
                num_q_heads, num_kv_heads);
  if (!supported_group(num_q_heads / num_kv_heads))
    return fail(PA_ERR_UNSUPPORTED, "%s: group size %d not built", who, num_q_heads / num_kv_heads);
  if (max_blocks_per_seq <= 0 || max_q <= 0)
    return fail(PA_ERR_INVALID_ARG, "%s: max_blocks_per_seq and max_q must be > 0", who);
  if (!(scale == scale)) return fail(PA_ERR_INVALID_ARG, "%s: scale is NaN", who);
  if (!out || !q || !k_cache || !v_cache || !block_tables || !cu_q_lens || !context_lens)
    return fail(PA_ERR_INVALID_ARG, "%s: null pointer", who);
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(PA_ERR_INVALID_ARG, "%s: out/q/caches must be 16-byte aligned", who);
  const size_t need = prefill_workspace_bytes(num_seqs, num_tokens, max_q, num_q_heads,
                                              num_kv_heads, head_dim, max_ctx, block_size);
  if (need > 0 && (workspace == nullptr || !aligned16(workspace)))
    return fail(PA_ERR_INVALID_ARG, "%s: workspace null or unaligned", who);
  if (workspace_bytes < need)
    return fail(PA_ERR_WORKSPACE, "%s: workspace %zu bytes < %zu needed", who, workspace_bytes,
                need);
  int32_t* st = status_word(stream);
  if (st == nullptr) return fail(PA_ERR_CUDA, "%s: no usable CUDA device", who);
  a.out = out;
  a.out_dtype = out_dtype;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.max_blocks = max_blocks_per_seq;
  a.cu_q_lens = cu_q_lens;
  a.context_lens = context_lens;
  a.num_seqs = num_seqs;
  a.num_tokens = num_tokens;
  a.max_q = max_q;
  a.max_ctx = max_ctx;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.scale = scale;
  a.dtype = dtype;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.status = st;
  return PA_OK;
}

// Share of the SMs the decode's attention kernel takes in a mixed step: it stays bound by
// HBM on ~58% of them (2.74 against 2.70 ms on the mixed workload's decode batch), and the
// prefill's tensor-core work fills the rest (the step 2.85 ms against 3.13 ms in turn).
constexpr int kMixedDecodePercent = 58;

// A stream of the library's own per device and host thread, for work that runs beside the
// caller's stream, with the two events that fork it from and join it to that stream.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

static thread_local SideStream t_side[64];  // per device, for this host thread

static int side_stream(const char* who, SideStream** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
    return fail(PA_ERR_CUDA, "%s: no usable CUDA device", who);
  SideStream& x = t_side[dev];
  if (x.stream == nullptr) {
    if (cudaStreamCreateWithFlags(&x.stream, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&x.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&x.join, cudaEventDisableTiming) != cudaSuccess)
      return fail(PA_ERR_CUDA, "%s: %s", who, cudaGetErrorString(cudaGetLastError()));
  }
  *out = &x;
  return PA_OK;
}

// A prefill batch's cache write (its chunks' new tokens), then its attention.
static int launch_prefill_append(const char* who, const PrefillArgs& a, const void* k_new,
                                 const void* v_new, int64_t* slots, cudaStream_t s) {
  const cudaError_t e = launch_cache_append(
      k_new, v_new, const_cast<void*>(a.k_cache), const_cast<void*>(a.v_cache), slots,
      a.block_tables, a.max_blocks, a.cu_q_lens, a.context_lens, a.num_seqs, a.num_tokens,
      a.max_q, a.num_kv_heads, a.head_dim, a.block_size, a.num_blocks, dtype_bytes(a.dtype),
      a.status, s);
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "%s: %s", who, cudaGetErrorString(e));
  return launch_prefill(a, s);
}

extern "C" {

int pa_prefill_chunk(void* out, pa_dtype out_dtype, const void* q, const void* k_cache,
                     const void* v_cache, const int32_t* block_tables, int max_blocks_per_seq,
                     const int32_t* cu_q_lens, const int32_t* context_lens, int num_seqs,
                     int num_tokens, int max_q, int max_ctx, int num_q_heads, int num_kv_heads,
                     int head_dim, int block_size, int num_blocks, float scale, pa_dtype dtype,
                     void* workspace, size_t workspace_bytes, void* stream) {
  g_error[0] = '\0';
  PrefillArgs a;
  bool empty = false;
  const int rc = prefill_args("pa_prefill_chunk", out, out_dtype, q, k_cache, v_cache,
                              block_tables, max_blocks_per_seq, cu_q_lens, context_lens, num_seqs,
                              num_tokens, max_q, max_ctx, num_q_heads, num_kv_heads, head_dim,
                              block_size, num_blocks, scale, dtype, workspace, workspace_bytes,
                              stream, a, &empty);
  if (rc != PA_OK || empty) return rc;
  return launch_prefill(a, static_cast<cudaStream_t>(stream));
}

int pa_mixed_step(const pa_decode_batch* dec, const pa_prefill_batch* pre, void* k_cache,
                  void* v_cache, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                  int num_blocks, float scale, pa_dtype dtype, void* stream) {
  g_error[0] = '\0';
  const char* who = "pa_mixed_step";
  const bool has_dec = dec != nullptr && dec->num_seqs != 0;
  const bool has_pre = pre != nullptr && (pre->num_seqs != 0 || pre->num_tokens != 0);
  if (has_dec && dec->num_seqs > 0 && (!dec->k_new || !dec->v_new))
    return fail(PA_ERR_INVALID_ARG, "%s: decode batch: null pointer", who);
  if (has_dec && dec->num_seqs > 0 && (!aligned16(dec->k_new) || !aligned16(dec->v_new)))
    return fail(PA_ERR_INVALID_ARG, "%s: decode batch: K/V pointers must be 16-byte aligned", who);
  if (has_pre && pre->num_tokens > 0 && (!pre->k_new || !pre->v_new))
    return fail(PA_ERR_INVALID_ARG, "%s: prefill batch: null pointer", who);
  if (has_pre && pre->num_tokens > 0 && (!aligned16(pre->k_new) || !aligned16(pre->v_new)))
    return fail(PA_ERR_INVALID_ARG, "%s: prefill batch: K/V pointers must be 16-byte aligned", who);
  DecodeArgs da;
  if (has_dec) {
    const int rc = decode_args(who, dec->out, dec->out_dtype, dec->q, k_cache, v_cache,
                               dec->block_tables, dec->max_blocks_per_seq, dec->context_lens,
                               dec->max_ctx, dec->num_seqs, num_q_heads, num_kv_heads, head_dim,
                               block_size, num_blocks, scale, dtype, dec->workspace,
                               dec->workspace_bytes, stream, da);
    if (rc != PA_OK) return rc;
  }
  PrefillArgs pa_args;
  bool pre_empty = true;
  if (has_pre) {
    const int rc = prefill_args(who, pre->out, pre->out_dtype, pre->q, k_cache, v_cache,
                                pre->block_tables, pre->max_blocks_per_seq, pre->cu_q_lens,
                                pre->context_lens, pre->num_seqs, pre->num_tokens, pre->max_q,
                                pre->max_ctx, num_q_heads, num_kv_heads, head_dim, block_size,
                                num_blocks, scale, dtype, pre->workspace, pre->workspace_bytes,
                                stream, pa_args, &pre_empty);
    if (rc != PA_OK) return rc;
  }
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!has_dec && pre_empty) return PA_OK;
  if (!has_dec) return launch_prefill_append(who, pa_args, pre->k_new, pre->v_new, pre->slots, s);
  if (pre_empty) return launch_decode_append(who, da, dec->k_new, dec->v_new, dec->slots, s);
  // both: the decode on the caller's stream, launched first so that its attention kernel
  // holds its share of the SMs before the prefill's CTAs take the rest
  SideStream* side = nullptr;
  int rc = side_stream(who, &side);
  if (rc != PA_OK) return rc;
  if (cudaEventRecord(side->fork, s) != cudaSuccess ||
      cudaStreamWaitEvent(side->stream, side->fork, 0) != cudaSuccess)
    return fail(PA_ERR_CUDA, "%s: %s", who, cudaGetErrorString(cudaGetLastError()));
  da.max_ctas = std::max(1, sm_count() * kMixedDecodePercent / 100);
  rc = launch_decode_append(who, da, dec->k_new, dec->v_new, dec->slots, s);
  // the side stream is joined back even when a launch failed, so that `stream` never
  // runs ahead of work already enqueued beside it
  const int rc2 = launch_prefill_append(who, pa_args, pre->k_new, pre->v_new, pre->slots,
                                        side->stream);
  if (cudaEventRecord(side->join, side->stream) != cudaSuccess ||
      cudaStreamWaitEvent(s, side->join, 0) != cudaSuccess)
    return fail(PA_ERR_CUDA, "%s: %s", who, cudaGetErrorString(cudaGetLastError()));
  return rc != PA_OK ? rc : rc2;
}

int pa_release_thread_resources(void) {
  g_error[0] = '\0';
  int cur = 0;
  const bool restore = cudaGetDevice(&cur) == cudaSuccess;
  int rc = PA_OK;
  for (int dev = 0; dev < 64; ++dev) {
    SideStream& x = t_side[dev];
    if (x.stream == nullptr && x.fork == nullptr && x.join == nullptr) continue;
    // each handle is destroyed with its own device current
    if (cudaSetDevice(dev) != cudaSuccess ||
        (x.stream != nullptr && cudaStreamDestroy(x.stream) != cudaSuccess) ||
        (x.fork != nullptr && cudaEventDestroy(x.fork) != cudaSuccess) ||
        (x.join != nullptr && cudaEventDestroy(x.join) != cudaSuccess))
      rc = fail(PA_ERR_CUDA, "pa_release_thread_resources: %s",
                cudaGetErrorString(cudaGetLastError()));
    x = SideStream{};
  }
  if (restore) cudaSetDevice(cur);
  return rc;
}

}  // extern "C"
