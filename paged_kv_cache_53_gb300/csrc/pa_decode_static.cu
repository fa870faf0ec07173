// pa_decode_static_scratch: pa_decode without a caller-provided workspace.
//
// Some callers cannot allocate device memory for a workspace: an engine that hands the
// whole GPU to its KV-block pool and caching allocator at start-up has no free memory
// to give, and a caller on a latency-critical path cannot afford cudaMalloc/cudaFree,
// which may synchronise the device.  This entry point takes its split-KV scratch from a
// fixed array compiled into the library instead, so it allocates nothing.
#include <mutex>

#include "pa.h"
#include "pa_internal.h"

namespace pa {
namespace {

// The scratch array.  Every GPU that loads the library reserves these bytes until the
// process exits.  In host code its name is only a host-side stand-in: its device
// address comes from cudaGetSymbolAddress below.
constexpr size_t kStaticScratchBytes = 32ull << 20;  // 32 MiB
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxScratchDevices = 64;
void* g_scratch_addr[kMaxScratchDevices] = {};
std::mutex g_scratch_mutex;

// Device address of the scratch array on the current device, looked up once per device.
void* scratch_address(int* err) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices) {
    *err = (int)(e != cudaSuccess ? e : cudaErrorInvalidDevice);
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) {
      *err = (int)e;
      return nullptr;
    }
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace
}  // namespace pa

extern "C" int pa_decode_static_scratch(void* out, pa_dtype out_dtype, const void* q,
                                        const void* k_cache, const void* v_cache,
                                        const int32_t* block_tables, int max_blocks_per_seq,
                                        const int32_t* context_lens, int max_ctx, int num_seqs,
                                        int num_q_heads, int num_kv_heads, int head_dim,
                                        int block_size, int num_blocks, float scale,
                                        pa_dtype dtype, void* stream) {
  if (num_seqs > 0 && num_q_heads > 0 && num_kv_heads > 0 && head_dim > 0 && max_ctx >= 0 &&
      block_size > 0) {
    const size_t need = pa_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                  max_ctx, block_size);
    if (need > pa::kStaticScratchBytes)
      return pa::fail(PA_ERR_WORKSPACE,
                      "pa_decode_static_scratch: these sizes need %zu bytes of scratch, more "
                      "than the library's fixed %zu-byte array; use pa_decode with a workspace",
                      need, pa::kStaticScratchBytes);
  }
  int err = 0;
  void* scratch = pa::scratch_address(&err);
  if (scratch == nullptr)
    return pa::fail(PA_ERR_CUDA, "pa_decode_static_scratch: cannot locate the scratch array: %s",
                    cudaGetErrorString((cudaError_t)err));
  return pa_decode(out, out_dtype, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                   context_lens, max_ctx, num_seqs, num_q_heads, num_kv_heads, head_dim,
                   block_size, num_blocks, scale, dtype, scratch, pa::kStaticScratchBytes,
                   stream);
}
