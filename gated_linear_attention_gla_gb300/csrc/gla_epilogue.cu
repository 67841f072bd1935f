// gla_epilogue.cu -- the mixer's steps after the readout, over a finished
// output o (in place).
//
// Method: the "GLA mixer" paragraph of the "i14 Laplace 3B on AWS Trainium2"
// page, the steps that follow the readout, per token and head:
//     o += sigmoid(q . (aug * k)) * v                 (self-augmentation)
//     o  = o / sqrt(mean_j o_j^2 + eps) * w[h]        (head RMSNorm)
//     o *= silu(z)                                    (output gate)
// each step optional.  One warp per (token, head): the two dot products are
// warp reductions, every lane owns dv / 32 columns.  A pure stream over o, q,
// k, v and z (HBM-bound); the decode kernel fuses the same steps instead.
#include "gla_internal.cuh"

namespace gla {
namespace {

constexpr int kEpiWarps = 8;

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

template <typename IO, typename OUT, int DK, int DV>
__global__ void __launch_bounds__(kEpiWarps * 32)
epilogue_kernel(OUT* __restrict__ out, const IO* __restrict__ q, const IO* __restrict__ k,
                const IO* __restrict__ v, const float* __restrict__ aug,
                const float* __restrict__ norm_w, float eps, const IO* __restrict__ z,
                long long units, int H) {
  constexpr int PER = DV / 32;  // columns per lane
  const int lane = threadIdx.x & 31;
  const long long unit = (long long)blockIdx.x * kEpiWarps + (threadIdx.x >> 5);  // row * H + h
  if (unit >= units) return;
  const int h = (int)(unit % H);
  float o[PER];
#pragma unroll
  for (int c = 0; c < PER; ++c) o[c] = to_f32(out[unit * DV + lane + 32 * c]);
  if (aug != nullptr) {
    float s = 0.f;
#pragma unroll
    for (int i = lane; i < DK; i += 32)
      s += to_f32(q[unit * DK + i]) * __ldg(aug + h * DK + i) * to_f32(k[unit * DK + i]);
    s = warp_sum(s);
    const float gate = 1.f / (1.f + expf(-s));
#pragma unroll
    for (int c = 0; c < PER; ++c) o[c] = fmaf(gate, to_f32(v[unit * DV + lane + 32 * c]), o[c]);
  }
  if (norm_w != nullptr) {
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < PER; ++c) ss += o[c] * o[c];
    ss = warp_sum(ss);
    const float r = rsqrtf(ss / DV + eps);
#pragma unroll
    for (int c = 0; c < PER; ++c) o[c] *= r * __ldg(norm_w + h * DV + lane + 32 * c);
  }
  if (z != nullptr) {
#pragma unroll
    for (int c = 0; c < PER; ++c) {
      const float zz = to_f32(z[unit * DV + lane + 32 * c]);
      o[c] *= zz / (1.f + expf(-zz));
    }
  }
#pragma unroll
  for (int c = 0; c < PER; ++c) out[unit * DV + lane + 32 * c] = from_f32<OUT>(o[c]);
}

template <typename IO, typename OUT, int DK>
cudaError_t launch_dv(const EpilogueArgs& a, cudaStream_t stream) {
  const long long units = a.rows * a.H;
  const unsigned grid = (unsigned)((units + kEpiWarps - 1) / kEpiWarps);
#define GLA_EPI(DV)                                                                          \
  epilogue_kernel<IO, OUT, DK, DV><<<grid, kEpiWarps * 32, 0, stream>>>(                     \
      (OUT*)a.out, (const IO*)a.q, (const IO*)a.k, (const IO*)a.v, a.aug, a.norm_w, a.eps,   \
      (const IO*)a.z, units, a.H)
  if (a.dv == 192) GLA_EPI(192);
  else if (a.dv == 128) GLA_EPI(128);
  else GLA_EPI(64);
#undef GLA_EPI
  return cudaGetLastError();
}

template <typename IO, typename OUT>
cudaError_t launch_io(const EpilogueArgs& a, cudaStream_t stream) {
  if (a.dk == 128) return launch_dv<IO, OUT, 128>(a, stream);
  if (a.dk == 96) return launch_dv<IO, OUT, 96>(a, stream);
  return launch_dv<IO, OUT, 64>(a, stream);
}

}  // namespace

cudaError_t launch_epilogue(const EpilogueArgs& a, cudaStream_t stream) {
  if (a.fp32_io) return launch_io<float, float>(a, stream);
  if (a.fp32_out) return launch_io<__nv_bfloat16, float>(a, stream);
  return launch_io<__nv_bfloat16, __nv_bfloat16>(a, stream);
}

}  // namespace gla
