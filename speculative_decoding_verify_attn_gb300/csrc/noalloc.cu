// spec_verify_attn_noalloc: verify attention for callers that cannot allocate device memory.
//
// Some callers must not allocate on their hot path: a serving engine that reserved all of HBM for
// its KV cache and weights at start-up, a plugin inside a host framework that owns every device
// allocation, or a decode loop that cannot afford cudaMalloc/cudaFree (both synchronize the
// device).  Such callers cannot hand spec_verify_attn a workspace of their own, so this entry
// point uses a fixed scratch array compiled into the library instead.
//
// The array is a file-scope __device__ variable: every GPU that loads the library holds its
// SPEC_NOALLOC_SCRATCH_BYTES until the process exits.  Host code cannot use the symbol itself as
// a device address (on the host it only names a shadow), so every call looks the array's device
// address up with cudaGetSymbolAddress in the context current on the calling thread.  The address
// is not cached: it belongs to one context, and a caller may switch contexts (its own driver-API
// context, or a new primary context after cudaDeviceReset) between calls, where a cached address
// would point at memory the new context does not map.  After the first call in a context the
// lookup is a host-side table read.  Calls share the array; calls that overlap on the GPU race.
#include <cuda_runtime.h>

#include "spec_verify.h"

namespace {

static __device__ __align__(256) unsigned char g_verify_scratch[SPEC_NOALLOC_SCRATCH_BYTES];

// Device address of g_verify_scratch in the calling thread's current context.
int scratch_for_current_context(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_verify_scratch) != cudaSuccess || p == nullptr) return SPEC_ERR_CUDA;
  *out = p;
  return SPEC_OK;
}

}  // namespace

extern "C" int spec_verify_attn_noalloc(const spec_attn_args* args, spec_stream_t stream) {
  if (!args) return SPEC_ERR_INVALID_ARG;
  const size_t need = spec_verify_attn_workspace(args);
  if (need == 0) return SPEC_ERR_INVALID_ARG;
  if (need > SPEC_NOALLOC_SCRATCH_BYTES) return SPEC_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  const int st = scratch_for_current_context(&scratch);
  if (st != SPEC_OK) return st;
  spec_attn_args a = *args;
  a.workspace = scratch;
  a.workspace_bytes = SPEC_NOALLOC_SCRATCH_BYTES;
  return spec_verify_attn(&a, stream);
}
