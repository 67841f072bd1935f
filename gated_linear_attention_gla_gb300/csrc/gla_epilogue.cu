// gla_epilogue.cu -- the mixer's steps after the readout, over a finished
// output o (in place).
//
// Method: the "GLA mixer" paragraph of the "i14 Laplace 3B on AWS Trainium2"
// page, the steps that follow the readout, per token and head:
//     o += sigmoid(q . (aug * k)) * v                 (self-augmentation)
//     o  = o / sqrt(mean_j o_j^2 + eps) * w[h]        (head RMSNorm)
//     o *= silu(z)                                    (output gate)
// each step optional.  Sixteen lanes per (token, head): the two dot products
// are reductions over those lanes, every lane owns dv / 16 adjacent columns
// (and dk / 16 key channels), so each tensor is read as one contiguous span
// per unit.  A pure
// stream over o, q, k, v and z (HBM-bound); the decode kernel fuses the same
// steps instead.
#include "gla_internal.cuh"

namespace gla {
namespace {

constexpr int kEpiWarps = 8;



// N consecutive elements as fp32: 16-, 8- or 4-byte loads for even N (the
// caller's tensors are 16-byte aligned and every run starts on a multiple of
// its own size), element loads for odd N.
template <int N, typename T>
__device__ __forceinline__ void load_run(const T* __restrict__ p, float (&x)[N]) {
  if constexpr (N % 2 != 0) {  // odd runs (dk = 96: three channels a lane)
#pragma unroll
    for (int i = 0; i < N; ++i) x[i] = to_f32(__ldg(p + i));
  } else if constexpr (sizeof(T) == 4) {
    if constexpr (N % 4 == 0) {
#pragma unroll
      for (int i = 0; i < N; i += 4) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(p + i));
        x[i] = v.x; x[i + 1] = v.y; x[i + 2] = v.z; x[i + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < N; i += 2) {
        const float2 v = __ldg(reinterpret_cast<const float2*>(p + i));
        x[i] = v.x; x[i + 1] = v.y;
      }
    }
  } else {  // bf16: pairs in 32-bit words
    if constexpr (N % 8 == 0) {
#pragma unroll
      for (int i = 0; i < N; i += 8) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(p + i));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          x[i + 2 * e] = __uint_as_float(w[e] << 16);
          x[i + 2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
        }
      }
    } else if constexpr (N % 4 == 0) {
#pragma unroll
      for (int i = 0; i < N; i += 4) {
        const uint2 v = __ldg(reinterpret_cast<const uint2*>(p + i));
        x[i] = __uint_as_float(v.x << 16);
        x[i + 1] = __uint_as_float(v.x & 0xffff0000u);
        x[i + 2] = __uint_as_float(v.y << 16);
        x[i + 3] = __uint_as_float(v.y & 0xffff0000u);
      }
    } else {
#pragma unroll
      for (int i = 0; i < N; i += 2) {
        const unsigned v = __ldg(reinterpret_cast<const unsigned*>(p + i));
        x[i] = __uint_as_float(v << 16);
        x[i + 1] = __uint_as_float(v & 0xffff0000u);
      }
    }
  }
}

template <int N, typename T>
__device__ __forceinline__ void store_run(T* __restrict__ p, const float (&x)[N]) {
  if constexpr (sizeof(T) == 4 && N % 4 == 0) {
#pragma unroll
    for (int i = 0; i < N; i += 4)
      *reinterpret_cast<float4*>(p + i) = make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]);
  } else if constexpr (sizeof(T) == 4) {
#pragma unroll
    for (int i = 0; i < N; i += 2)
      *reinterpret_cast<float2*>(p + i) = make_float2(x[i], x[i + 1]);
  } else if constexpr (N % 8 == 0) {
#pragma unroll
    for (int i = 0; i < N; i += 8) {
      auto pack = [&](int e) {
        return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x[i + 2 * e])) |
               ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x[i + 2 * e + 1])) << 16);
      };
      *reinterpret_cast<uint4*>(p + i) = make_uint4(pack(0), pack(1), pack(2), pack(3));
    }
  } else {
#pragma unroll
    for (int i = 0; i < N; i += 2) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(x[i], x[i + 1]);
      *reinterpret_cast<__nv_bfloat162*>(p + i) = b;
    }
  }
}

// kEpiLanes lanes per (row, head), two units a warp: lane l of a unit owns the
// dv / kEpiLanes adjacent columns from l * dv / kEpiLanes and the dk /
// kEpiLanes adjacent key channels from l * dk / kEpiLanes, read and written as
// runs (16-byte vectors at d = 128 in bf16; each unit's access is one
// contiguous span).
constexpr int kEpiLanes = 16;

// sum over the kEpiLanes lanes of a unit (an aligned group of the warp)
__device__ __forceinline__ float unit_sum(float x) {
#pragma unroll
  for (int off = kEpiLanes / 2; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

template <typename IO, typename OUT, int DK, int DV>
__global__ void __launch_bounds__(kEpiWarps * 32)
epilogue_kernel(OUT* __restrict__ out, const IO* __restrict__ q, const IO* __restrict__ k,
                const IO* __restrict__ v, const float* __restrict__ aug,
                const float* __restrict__ norm_w, float eps, const IO* __restrict__ z,
                long long units, int H) {
  constexpr int PER = DV / kEpiLanes;   // columns per lane
  constexpr int PK = DK / kEpiLanes;    // key channels per lane
  static_assert(DV % kEpiLanes == 0 && DK % kEpiLanes == 0, "whole runs");
  const int lane = (threadIdx.x & 31) % kEpiLanes;
  const long long unit0 = (long long)blockIdx.x * kEpiWarps * (32 / kEpiLanes) +
                          (threadIdx.x >> 5) * (32 / kEpiLanes) + (threadIdx.x & 31) / kEpiLanes;
  // a unit past the end still joins its warp's shuffles, on unit 0's data, and
  // stores nothing
  const bool valid = unit0 < units;
  const long long unit = valid ? unit0 : 0;  // row * H + h
  const int h = (int)(unit % H);
  const long long ob = unit * DV + lane * PER;
  const long long kb = unit * DK + lane * PK;
  // every load of the row first, so that they are all in flight together
  float o[PER], vv[PER], zz[PER], w[PER], qv[PK], kv[PK], av[PK];
  load_run<PER>(out + ob, o);
  if (aug != nullptr) {
    load_run<PK>(q + kb, qv);
    load_run<PK>(k + kb, kv);
    load_run<PK>(aug + h * DK + lane * PK, av);
    load_run<PER>(v + ob, vv);
  }
  if (norm_w != nullptr) load_run<PER>(norm_w + h * DV + lane * PER, w);
  if (z != nullptr) load_run<PER>(z + ob, zz);
  if (aug != nullptr) {
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < PK; ++i) s = fmaf(qv[i] * av[i], kv[i], s);
    s = unit_sum(s);
    const float gate = 1.f / (1.f + expf(-s));
#pragma unroll
    for (int c = 0; c < PER; ++c) o[c] = fmaf(gate, vv[c], o[c]);
  }
  if (norm_w != nullptr) {
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < PER; ++c) ss = fmaf(o[c], o[c], ss);
    ss = unit_sum(ss);
    const float r = rsqrtf(ss / DV + eps);
#pragma unroll
    for (int c = 0; c < PER; ++c) o[c] *= r * w[c];
  }
  if (z != nullptr) {
#pragma unroll
    for (int c = 0; c < PER; ++c) o[c] *= zz[c] / (1.f + expf(-zz[c]));
  }
  if (valid) store_run<PER>(out + ob, o);
}

template <typename IO, typename OUT, int DK>
cudaError_t launch_dv(const EpilogueArgs& a, cudaStream_t stream) {
  const long long units = a.rows * a.H;
  const long long per_cta = (long long)kEpiWarps * (32 / kEpiLanes);
  const unsigned grid = (unsigned)((units + per_cta - 1) / per_cta);
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
