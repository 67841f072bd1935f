// gla_chunk_tc.cu -- placeholder until the tensor-core prefill kernel lands.
#include "gla_internal.cuh"

namespace gla {
bool chunk_tc_supported(const ChunkArgs&) { return false; }
cudaError_t launch_chunk_tc(const ChunkArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace gla
