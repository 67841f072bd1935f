// gla_chunk_simt.cu -- chunked GLA prefill on the fp32 CUDA cores.
//
// Method: the chunked form of the "i14 Laplace 3B on AWS Trainium2" page
// (section "Challenge 1", Figure 3), generalised to per-token log-decays.
// Inside a chunk of n tokens, with G_t the running sum of the (clamped) gate
// from the chunk start through token t (per key channel for the vector gate):
//     o_t   = scale * ( sum_{j<=t} (q_t . (k_j * exp(G_t - G_j))) v_j
//                       + (q_t * exp(G_t)) S )
//     S'    = diag(exp(G_{n-1})) S + sum_j (k_j * exp(G_{n-1} - G_j))^T v_j
//
// This is the full-precision path: every product and sum is fp32 with accurate
// expf, so it serves fp32 I/O (the 1e-5 tolerance case), any chunk size up to
// 128, and the per-key-channel gate.  It is not the throughput path for bf16.
//
// Decomposition: one CTA per (sequence, head, 64-wide slice of dv); 8 warps.
// The chunk's K, V-slice and cumulative gates sit in shared memory as fp32;
// each warp produces one output row at a time (scores across lanes, then
// columns across lanes); the state slice S[dk][64] stays in shared memory for
// the whole sequence and is advanced once per chunk by all threads.
#include "gla_internal.cuh"

namespace gla {
namespace {

constexpr int kSimtThreads = 256;
constexpr int kSimtWarps = kSimtThreads / 32;
constexpr int kSlice = 64;  // dv columns per CTA

template <int DK, int CH, bool VEC>
struct SimtSmem {
  static constexpr int kKs = CH * (DK + 1);              // K chunk, padded rows
  static constexpr int kGs = VEC ? CH * (DK + 1) : CH;   // cumulative gates
  static constexpr int kVs = CH * kSlice;                // V slice
  static constexpr int kS = DK * kSlice;                 // state slice
  static constexpr int kQw = kSimtWarps * DK;            // q row per warp
  static constexpr int kQt = kSimtWarps * DK;            // q * exp(G_t) per warp
  static constexpr int kPw = kSimtWarps * CH;            // score row per warp
  static constexpr int kGa = VEC ? DK : 1;               // chunk-total decay
  static constexpr int kFloats = kKs + kGs + kVs + kS + kQw + kQt + kPw + kGa;
  static constexpr size_t kBytes = sizeof(float) * (size_t)kFloats;
};

// Inclusive prefix sum of x[0..n) (n <= CH) by one warp, in place in shared memory.
template <int CH>
__device__ __forceinline__ void warp_scan_inplace(float* x, int n, int lane) {
  constexpr int PER = (CH + 31) / 32;
  float v[PER];
  float run = 0.f;
#pragma unroll
  for (int r = 0; r < PER; ++r) {
    const int t = lane * PER + r;
    run += (t < n) ? x[t] : 0.f;
    v[r] = run;
  }
  float incl = run;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  const float excl = incl - run;
#pragma unroll
  for (int r = 0; r < PER; ++r) {
    const int t = lane * PER + r;
    if (t < n) x[t] = v[r] + excl;
  }
}

template <typename IO, typename OUT, int DK, int CH, bool VEC>
__global__ void __launch_bounds__(kSimtThreads, 1)
chunk_simt_kernel(const IO* __restrict__ q, const IO* __restrict__ k,
                  const IO* __restrict__ v, const float* __restrict__ g, float scale,
                  const float* __restrict__ init_state, OUT* __restrict__ out,
                  float* __restrict__ final_state, const int32_t* __restrict__ cu_seqlens,
                  int B, int H, int T, int DV, unsigned* status) {
  using L = SimtSmem<DK, CH, VEC>;
  extern __shared__ float smem[];
  float* Ks = smem;
  float* Gs = Ks + L::kKs;
  float* Vs = Gs + L::kGs;
  float* S = Vs + L::kVs;
  float* Qw = S + L::kS;
  float* Qt = Qw + L::kQw;
  float* Pw = Qt + L::kQt;
  float* Ga = Pw + L::kPw;
  constexpr int KP = DK + 1;

  const int nslices = DV / kSlice;
  const int slice = blockIdx.x % nslices;
  const int h = (blockIdx.x / nslices) % H;
  const int s = blockIdx.x / (nslices * H);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int col0 = slice * kSlice;

  long long start;
  int len;
  if (!seq_bounds(cu_seqlens, s, B, T, &start, &len, status)) return;

  // state slice <- initial state (or zero)
  const size_t st_off = ((size_t)s * H + h) * (size_t)DK * DV;
  for (int idx = tid; idx < DK * kSlice; idx += kSimtThreads) {
    const int d = idx / kSlice, j = idx % kSlice;
    S[idx] = init_state ? init_state[st_off + (size_t)d * DV + col0 + j] : 0.f;
  }

  for (int c0 = 0; c0 < len; c0 += CH) {
    const int n = min(CH, len - c0);
    const long long base = start + c0;
    __syncthreads();  // previous chunk fully consumed
    for (int idx = tid; idx < n * DK; idx += kSimtThreads) {
      const int t = idx / DK, d = idx % DK;
      Ks[t * KP + d] = to_f32(k[((base + t) * H + h) * DK + d]);
    }
    for (int idx = tid; idx < n * kSlice; idx += kSimtThreads) {
      const int t = idx / kSlice, j = idx % kSlice;
      Vs[idx] = to_f32(v[((base + t) * H + h) * (long long)DV + col0 + j]);
    }
    if constexpr (VEC) {
      for (int idx = tid; idx < n * DK; idx += kSimtThreads) {
        const int t = idx / DK, d = idx % DK;
        Gs[t * KP + d] = fmaxf(g[((base + t) * H + h) * DK + d], -kGateClamp);
      }
      __syncthreads();
      for (int d = tid; d < DK; d += kSimtThreads) {
        float run = 0.f;
        for (int t = 0; t < n; ++t) {
          run += Gs[t * KP + d];
          Gs[t * KP + d] = run;
        }
      }
    } else {
      for (int t = tid; t < n; t += kSimtThreads)
        Gs[t] = fmaxf(g[(base + t) * H + h], -kGateClamp);
      __syncthreads();
      if (warp == 0) warp_scan_inplace<CH>(Gs, n, lane);
    }
    __syncthreads();

    // ---- outputs: one row per warp at a time --------------------------------
    float* qw = Qw + warp * DK;
    float* qt = Qt + warp * DK;
    float* pw = Pw + warp * CH;
    for (int i = warp; i < n; i += kSimtWarps) {
      for (int d = lane; d < DK; d += 32) {
        const float qd = to_f32(q[((base + i) * H + h) * DK + d]);
        qw[d] = qd;
        qt[d] = qd * expf(VEC ? Gs[i * KP + d] : Gs[i]);
      }
      __syncwarp();
      for (int t = lane; t <= i; t += 32) {
        float acc = 0.f;
        if constexpr (VEC) {
#pragma unroll 8
          for (int d = 0; d < DK; ++d)
            acc = fmaf(qw[d] * Ks[t * KP + d], expf(Gs[i * KP + d] - Gs[t * KP + d]), acc);
        } else {
#pragma unroll 8
          for (int d = 0; d < DK; ++d) acc = fmaf(qw[d], Ks[t * KP + d], acc);
          acc *= expf(Gs[i] - Gs[t]);
        }
        pw[t] = acc;
      }
      __syncwarp();
#pragma unroll
      for (int jj = 0; jj < kSlice / 32; ++jj) {
        const int j = lane + 32 * jj;
        float acc = 0.f;
        for (int t = 0; t <= i; ++t) acc = fmaf(pw[t], Vs[t * kSlice + j], acc);
#pragma unroll 8
        for (int d = 0; d < DK; ++d) acc = fmaf(qt[d], S[d * kSlice + j], acc);
        out[((base + i) * H + h) * (long long)DV + col0 + j] = from_f32<OUT>(scale * acc);
      }
      __syncwarp();
    }
    __syncthreads();

    // ---- state step: S <- diag(exp G_last) S + (K * exp(G_last - G))^T V ------
    if constexpr (VEC) {
      for (int d = tid; d < DK; d += kSimtThreads) Ga[d] = expf(Gs[(n - 1) * KP + d]);
    } else {
      if (tid == 0) Ga[0] = expf(Gs[n - 1]);
    }
    for (int idx = tid; idx < n * DK; idx += kSimtThreads) {
      const int t = idx / DK, d = idx % DK;
      const float glast = VEC ? Gs[(n - 1) * KP + d] : Gs[n - 1];
      const float gt = VEC ? Gs[t * KP + d] : Gs[t];
      Ks[t * KP + d] *= expf(glast - gt);
    }
    __syncthreads();
    for (int idx = tid; idx < DK * kSlice; idx += kSimtThreads) {
      const int d = idx / kSlice, j = idx % kSlice;
      float acc = (VEC ? Ga[d] : Ga[0]) * S[idx];
      for (int t = 0; t < n; ++t) acc = fmaf(Ks[t * KP + d], Vs[t * kSlice + j], acc);
      S[idx] = acc;
    }
  }
  __syncthreads();
  if (final_state) {
    for (int idx = tid; idx < DK * kSlice; idx += kSimtThreads) {
      const int d = idx / kSlice, j = idx % kSlice;
      final_state[st_off + (size_t)d * DV + col0 + j] = S[idx];
    }
  }
}

template <typename IO, typename OUT, int DK, int CH, bool VEC>
cudaError_t launch_cfg(const ChunkArgs& a, cudaStream_t stream) {
  using L = SimtSmem<DK, CH, VEC>;
  auto kern = chunk_simt_kernel<IO, OUT, DK, CH, VEC>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)L::kBytes);
  if (e != cudaSuccess) return e;
  const long long ctas = (long long)a.B * a.H * (a.dv / kSlice);
  kern<<<(unsigned)ctas, kSimtThreads, L::kBytes, stream>>>(
      (const IO*)a.q, (const IO*)a.k, (const IO*)a.v, a.g, a.scale, a.init_state, (OUT*)a.out,
      a.final_state, a.cu_seqlens, a.B, a.H, a.T, a.dv, a.status);
  return cudaGetLastError();
}

template <typename IO, typename OUT, int DK, bool VEC>
cudaError_t launch_chunk(const ChunkArgs& a, cudaStream_t stream) {
  switch (a.chunk) {
    case 16: return launch_cfg<IO, OUT, DK, 16, VEC>(a, stream);
    case 32: return launch_cfg<IO, OUT, DK, 32, VEC>(a, stream);
    case 64: return launch_cfg<IO, OUT, DK, 64, VEC>(a, stream);
    default: return launch_cfg<IO, OUT, DK, 128, VEC>(a, stream);
  }
}

template <typename IO, typename OUT>
cudaError_t launch_io(const ChunkArgs& a, cudaStream_t stream) {
  if (a.dk == 128)
    return a.vector_gate ? launch_chunk<IO, OUT, 128, true>(a, stream)
                         : launch_chunk<IO, OUT, 128, false>(a, stream);
  if (a.dk == 96)
    return a.vector_gate ? launch_chunk<IO, OUT, 96, true>(a, stream)
                         : launch_chunk<IO, OUT, 96, false>(a, stream);
  return a.vector_gate ? launch_chunk<IO, OUT, 64, true>(a, stream)
                       : launch_chunk<IO, OUT, 64, false>(a, stream);
}

}  // namespace

cudaError_t launch_chunk_simt(const ChunkArgs& a, cudaStream_t stream) {
  if (a.fp32_io) return launch_io<float, float>(a, stream);
  if (a.fp32_out) return launch_io<__nv_bfloat16, float>(a, stream);
  return launch_io<__nv_bfloat16, __nv_bfloat16>(a, stream);
}

}  // namespace gla
