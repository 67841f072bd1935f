// gla_bwd_scratch.cu -- the library's own fixed workspace for the tensor-core
// backward (gla_chunk_bwd_fixed_workspace).
//
// Some callers cannot call cudaMalloc at the point where they need a gradient:
// code running inside a caching allocator's own callbacks, real-time threads
// that must not block on the driver's allocator lock, or embedders whose memory
// is fully reserved up front.  For them the workspace is a file-scope static
// device array of kBwdFixedWorkspaceBytes (384 MiB), which comes with this
// translation unit's module instead of being allocated at run time.
//
// Placement: with CUDA's lazy module loading (CUDA_MODULE_LOADING=LAZY, the
// default of current toolkits) the module that holds the array is loaded, and
// the 384 MiB reserved on a GPU, only when the entry point first asks for the
// array's address on that GPU; with eager loading every process that loads
// libgla.so reserves it on every GPU it uses, forward-only users included.
// Once placed, the array stays until the process exits.
#include <mutex>

#include "gla_internal.cuh"

namespace gla {

static __device__ __align__(256) uint8_t g_bwd_fixed_workspace[kBwdFixedWorkspaceBytes];

namespace {
constexpr int kMaxScratchDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxScratchDevices] = {};
}  // namespace

// The array's device address on the current GPU.  In host code the array's
// name denotes a host-side stand-in, not device memory, so the address comes
// from cudaGetSymbolAddress: once per device (the first call on that device,
// with it current), then from the cache.  On failure returns nullptr with *err
// set, and clears the runtime's last error so that a later, unrelated launch
// check does not report it.
void* bwd_fixed_workspace(cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxScratchDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_bwd_fixed_workspace);
    if (*err != cudaSuccess) {
      (void)cudaGetLastError();
      return nullptr;
    }
    g_scratch_ptr[dev] = p;
  }
  *err = cudaSuccess;
  return g_scratch_ptr[dev];
}

}  // namespace gla
