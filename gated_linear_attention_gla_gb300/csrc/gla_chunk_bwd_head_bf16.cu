// gla_chunk_bwd_head_bf16.cu -- the chunked backward for the per-head gate, bf16 q, k, v, d_out
// (the kernels are in gla_chunk_bwd.cuh).
#include "gla_chunk_bwd.cuh"

namespace gla {

cudaError_t launch_chunk_bwd_head_bf16(const ChunkBwdArgs& a, cudaStream_t stream) {
  return launch_bwd<__nv_bfloat16, false>(a, stream);
}

}  // namespace gla
