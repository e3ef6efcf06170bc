// quest_static_scratch.cu - quest_decode_static: the fused decode step for callers that
// cannot allocate device memory.
//
// quest_decode needs a caller-provided workspace.  Some callers cannot provide one: code
// that runs where it does not own the device allocator (a plugin or extension hosted by a
// runtime that hands it tensors but forbids it to call cudaMalloc, an engine that allows no
// allocation once it has started serving, a binding from a language with no device
// allocator of its own).  For them this file keeps the scratch in the library itself: a
// fixed-size array in device global memory, declared at file scope, which every GPU that
// loads the library holds until the process exits.  The caller still passes the cache,
// the query and the output buffers; nothing here calls cudaMalloc, cudaFree or any other
// routine that allocates.
#include <cstdio>

#include "quest_internal.h"

namespace {

// Largest workspace quest_decode_static can serve (bytes).
constexpr size_t kStaticScratchBytes = size_t(16) << 20;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// In host code `g_static_scratch` names a host-side stand-in, not device memory: its
// device address (on the current device) is looked up on every call, so that a context
// torn down and rebuilt (which reloads the module) never leaves a stale address behind.
// The lookup is not a stream operation and costs well under a microsecond.
int scratch_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
  if (e != cudaSuccess || !p)
    return quest::set_last_error(QUEST_ERR_CUDA, "cudaGetSymbolAddress(static scratch) failed");
  *out = p;
  return QUEST_OK;
}

}  // namespace

extern "C" int quest_decode_static(const quest_cache_t* cache, const void* q, int32_t top_k,
                                   void* out, float* lse, int32_t* idx_out, int32_t* count_out,
                                   int32_t* status_out, quest_stream_t stream) {
  size_t need = 0, zeroed = 0;
  int rc = quest::decode_workspace_requirement(cache, top_k, &need, &zeroed);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cache->batch == 0) {  // nothing to do: the status reads OK, as after any good call
    if (status_out) {
      const cudaError_t e = cudaMemsetAsync(status_out, 0, 4 * sizeof(int32_t), s);
      if (e != cudaSuccess) return quest::set_last_error(QUEST_ERR_CUDA, cudaGetErrorString(e));
    }
    return QUEST_OK;
  }
  if (need > kStaticScratchBytes) {
    char msg[160];
    snprintf(msg, sizeof(msg),
             "this cache and top_k need %zu bytes of scratch; the static scratch holds %zu",
             need, kStaticScratchBytes);
    return quest::set_last_error(QUEST_ERR_WORKSPACE, msg);
  }
  void* ws = nullptr;
  if ((rc = scratch_address(&ws))) return rc;
  // The array keeps whatever the previous call left: clear the header (status word and
  // counters), the arrival counters, the ready flags and the key rows before this call
  // uses them.
  cudaError_t e = cudaMemsetAsync(ws, 0, zeroed, s);
  if (e != cudaSuccess) return quest::set_last_error(QUEST_ERR_CUDA, cudaGetErrorString(e));
  rc = quest_decode(cache, q, top_k, out, lse, idx_out, count_out, ws, kStaticScratchBytes,
                    nullptr, stream);
  if (rc) return rc;
  if (status_out) {
    e = cudaMemcpyAsync(status_out, ws, 4 * sizeof(int32_t), cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return quest::set_last_error(QUEST_ERR_CUDA, cudaGetErrorString(e));
  }
  return QUEST_OK;
}
