// gla_internal.cuh -- declarations shared by the translation units of libgla.so.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace gla {

// Bits of the per-GPU device status word (see gla_status_sync in gla.h).
enum : unsigned {
  kDevBadSeqlens = 1u << 0,  // a cu_seqlens entry was out of order or out of range
  kDevTimeout = 1u << 1,     // a bounded mbarrier wait gave up
  kDevLayout = 1u << 2,      // a kernel's shared-memory window was not 1024-byte aligned
  // (kDevBadSeqlens also flags a decode slot index outside the state pool)
};

// Log-decays below -kGateClamp are raised to it before in-chunk cumulative
// sums, so that differences of sums stay finite (exp(-30) ~ 9.4e-14).
constexpr float kGateClamp = 30.0f;

struct ChunkArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  float scale;
  const float* init_state;
  void* out;
  float* final_state;
  const int32_t* cu_seqlens;
  int B, H, T, dk, dv, chunk;
  bool fp32_io;      // q, k, v (and out) fp32
  bool fp32_out;     // out fp32 with bf16 q, k, v
  bool vector_gate;
  bool out_reversed;  // token t of a sequence of len tokens stored at row len - 1 - t
                      // (tensor-core kernels only; the backward's reversed runs)
  // per-head tensor-core kernel only (the backward's dg terms): when dot_out is
  // set, dot_out[row, h] += dot_sign * sum_j out[row, h, j] * dot_rows[row, h, j]
  // (fp32 output values; dot_rows bf16 with the output's layout)
  const void* dot_rows;
  float* dot_out;
  float dot_sign;
  unsigned* status;   // device status word
};

struct DecodeArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  float scale;
  float* state;           // [N, H, dk, dv], or a pool of num_slots pages when slots is set
  const int32_t* slots;   // device [N]: the pool page of sequence n (-1: skip it), or null
  int num_slots;
  unsigned* status;       // device status word (slot out of range)
  void* out;
  // the mixer steps after the readout (each null = skipped): self-augmentation
  // weights [H, dk], head RMSNorm weights [H, dv] and eps, output gate [N, H, dv]
  const float* aug;
  const float* norm_w;
  float eps;
  const void* z;
  int N, H, dk, dv;
  bool fp32_io;
  bool fp32_out;
  bool vector_gate;
};

struct EpilogueArgs {
  void* out;              // [rows, H, dv], updated in place
  const void* q;          // [rows, H, dk] (with aug)
  const void* k;
  const void* v;          // [rows, H, dv] (with aug)
  const float* aug;       // [H, dk] or null
  const float* norm_w;    // [H, dv] or null
  float eps;
  const void* z;          // [rows, H, dv] or null
  long long rows;
  int H, dk, dv;
  bool fp32_io;           // q, k, v, z fp32 (else bf16)
  bool fp32_out;          // out fp32 (else bf16)
};

struct ChunkBwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  float scale;
  const float* init_state;  // [B, H, dk, dv] or null
  const void* d_out;        // [rows, H, dv]
  const float* d_final;     // [B, H, dk, dv] or null
  void* dq;
  void* dk;
  void* dv;
  float* dg;                // g's shape, or null
  float* d_init;            // [B, H, dk, dv] or null
  const int32_t* cu_seqlens;
  int B, H, T;
  int dk_size, dv_size;
  bool fp32_io;
  bool fp32_out;
  bool vector_gate;
  bool skip_dv;             // the CUDA-core kernels leave dv to another path
  unsigned* status;
};

// Wall-time limit of the tensor-core prefill kernels' hand-off waits, read at
// each launch (process-wide; set by gla_set_wait_limit_ns, default 2 s).  Their
// teardown drains keep the default.
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;
uint64_t handoff_wait_limit_ns();

// Kernel launchers (one per translation unit).  They assume validated arguments
// and a non-empty problem, and return the launch error.
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_epilogue(const EpilogueArgs& a, cudaStream_t stream);
cudaError_t launch_chunk_simt(const ChunkArgs& a, cudaStream_t stream);
bool chunk_tc_supported(const ChunkArgs& a);
cudaError_t launch_chunk_tc(const ChunkArgs& a, cudaStream_t stream);
bool chunk_tc_vec_supported(const ChunkArgs& a);
// with `mix`, the mixer's steps after the readout run inside the kernel (the
// fields other than aug, norm_w, eps and z are ignored)
cudaError_t launch_chunk_tc_vec(const ChunkArgs& a, cudaStream_t stream,
                                const EpilogueArgs* mix = nullptr);
// the chunked backward, one launcher per (gate, I/O dtype)
cudaError_t launch_chunk_bwd_head_bf16(const ChunkBwdArgs& a, cudaStream_t stream);
cudaError_t launch_chunk_bwd_head_f32(const ChunkBwdArgs& a, cudaStream_t stream);
cudaError_t launch_chunk_bwd_chan_bf16(const ChunkBwdArgs& a, cudaStream_t stream);
cudaError_t launch_chunk_bwd_chan_f32(const ChunkBwdArgs& a, cudaStream_t stream);
// the backward on the tensor cores, bf16, with chunk_bwd_tc_workspace(B, H,
// rows, dk, dv, vector_gate) bytes of workspace: per-head gate (d_k, d_v in
// {64, 128}), every gradient from three prefill runs; per-key-channel gate
// (d_k = d_v = 128), dv from one run of the per-key-channel prefill (dq, dk on
// the CUDA cores)
bool chunk_bwd_tc_supported(int dk, int dv, bool fp32_io, bool vector_gate);
size_t chunk_bwd_tc_workspace(int B, int H, long long rows, int dk, int dv, bool vector_gate);
cudaError_t launch_chunk_bwd_tc(const ChunkBwdArgs& a, void* workspace, cudaStream_t stream);
cudaError_t launch_chunk_bwd_tc_vec_dv(const ChunkBwdArgs& a, void* workspace,
                                       cudaStream_t stream);
// the fixed device workspace of gla_chunk_bwd_fixed_workspace (a static array;
// its address, or null with *err set)
constexpr size_t kBwdFixedWorkspaceBytes = 384ull << 20;
void* bwd_fixed_workspace(cudaError_t* err);

// ---------------------------------------------------------------------------
// Small device helpers shared by the kernels.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Sequence bounds for sequence s: dense batches own rows [s*T, s*T+T); packed
// batches read cu_seqlens.  Returns false (and flags the status word) for a
// malformed entry.
__device__ __forceinline__ bool seq_bounds(const int32_t* cu, int s, int B, int T,
                                           long long* start, int* len, unsigned* status) {
  if (cu == nullptr) {
    *start = (long long)s * T;
    *len = T;
    return true;
  }
  const int a = __ldg(cu + s), b = __ldg(cu + s + 1);
  const int first = __ldg(cu), last = __ldg(cu + B);
  if (first != 0 || last != T || a < 0 || b < a || b > T) {
    if (status) atomicOr(status, kDevBadSeqlens);
    return false;
  }
  *start = a;
  *len = b - a;
  return true;
}

}  // namespace gla
