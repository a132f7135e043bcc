// gdn_chunk_prefill_noalloc: chunked prefill for callers that cannot allocate device memory.
//
// The prefill needs scratch memory (post-conv activations, the tensor-core path's chunk
// tiles), which gdn_chunk_prefill takes from a caller-provided workspace.  Some callers
// cannot provide one: code running inside a CUDA-graph capture that must not call
// cudaMalloc, plug-ins handed only input and output pointers by a host framework, or
// allocators that forbid allocations outside start-up.  This entry point uses instead a
// file-scope device array of fixed size, GDN_NOALLOC_SCRATCH_BYTES, that every GPU which
// loads the library holds until the process exits.  It never calls cudaMalloc, cudaFree or
// any allocating routine.
//
// The array's name is only a host-side stand-in in host code, so its device address is
// obtained with cudaGetSymbolAddress, once per device, with that device current, on the first
// call made on that device, and cached for the life of the process (a device reset that
// destroys the context makes the cached address stale; the header tells callers not to call
// this entry point again on that device).
#include <mutex>

#include "common.cuh"

static __device__ __align__(256) unsigned char g_gdn_noalloc_scratch[GDN_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (nullptr on failure).
void* noalloc_scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_gdn_noalloc_scratch) != cudaSuccess || !p) return nullptr;
    g_noalloc_ptr[dev] = p;
  }
  return g_noalloc_ptr[dev];
}

}  // namespace

extern "C" {

gdn_status gdn_chunk_prefill_noalloc(const gdn_dims* dims, const gdn_opts* opts, const void* q,
                                     const void* k, const void* v, const void* a, const void* b,
                                     const float* A_log, const float* dt_bias,
                                     const void* conv_weight, const void* conv_bias,
                                     float* state, void* conv_state,
                                     const int32_t* state_slots, void* out, void* stream) {
  const size_t need = gdn_prefill_workspace_size(dims, opts);
  if (need > GDN_NOALLOC_SCRATCH_BYTES) return GDN_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    scratch = noalloc_scratch_on_current_device();
    if (!scratch) return GDN_ERR_CUDA;
  }
  return gdn_chunk_prefill(dims, opts, q, k, v, a, b, A_log, dt_bias, conv_weight, conv_bias,
                           state, conv_state, state_slots, out, scratch,
                           need > 0 ? (size_t)GDN_NOALLOC_SCRATCH_BYTES : 0, stream);
}

}  // extern "C"
