// Chunked-prefill attention (causal query chunk over paged context) for sm_103a.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

size_t prefill_workspace_bytes(int, int, int, int, int, int, int, int) { return 0; }

int launch_prefill(const PrefillArgs&, cudaStream_t) {
  return fail(PA_ERR_UNSUPPORTED, "pa_prefill_chunk: not built yet");
}

}  // namespace pa
