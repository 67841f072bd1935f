// gla_chunk_bwd_head_f32.cu -- the chunked backward for the per-head gate, fp32 q, k, v, d_out
// (the kernels are in gla_chunk_bwd.cuh).
#include "gla_chunk_bwd.cuh"

namespace gla {

cudaError_t launch_chunk_bwd_head_f32(const ChunkBwdArgs& a, cudaStream_t stream) {
  return launch_bwd<float, false>(a, stream);
}

}  // namespace gla
