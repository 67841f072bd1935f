// gla_bwd_scratch.cu -- the library's own fixed workspace for the tensor-core
// backward (gla_chunk_bwd_fixed_workspace).
//
// A file-scope static device array: the device memory comes with this
// translation unit's module, so nothing is allocated at run time.  The module
// holds nothing else, and it is loaded (and the array placed on the GPU) only
// when the entry point first asks for the array's address, so callers of the
// rest of the library do not carry it.
#include "gla_internal.cuh"

namespace gla {

static __device__ __align__(256) uint8_t g_bwd_fixed_workspace[kBwdFixedWorkspaceBytes];

void* bwd_fixed_workspace(cudaError_t* err) {
  void* p = nullptr;
  *err = cudaGetSymbolAddress(&p, g_bwd_fixed_workspace);
  return *err == cudaSuccess ? p : nullptr;
}

}  // namespace gla
