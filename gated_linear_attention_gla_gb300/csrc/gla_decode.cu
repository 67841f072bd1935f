// gla_decode.cu -- one-token recurrent decode step over N concurrent sequences.
//
// Method: the "GLA mixer" recurrence of the "i14 Laplace 3B on AWS Trainium2"
// page applied to one token per sequence, each sequence owning a fixed-size
// fp32 state page (section "Inference optimization on Trainium2"):
//     S'[i][j] = exp(g[i]) * S[i][j] + k[i] * v[j]      (written back in place)
//     o[j]     = scale * sum_i q[i] * S'[i][j]
//
// The step is a pure stream over the state: 2 * 4 * dk * dv bytes of state
// read-modify-write per (sequence, head) against ~3 * 2 * d bytes of inputs,
// about 0.5 flop per byte, so HBM bandwidth bounds it.  One CTA owns one
// (sequence, head) page:
//   * threads are laid out so that a warp reads whole 512-byte state rows with
//     128-bit loads (dv / 4 threads per row, fully coalesced);
//   * every thread issues all of its state loads before any use, so each SM
//     keeps ~128 KB of reads in flight;
//   * loads and stores carry streaming (evict-first) cache hints: the state
//     is touched once per step;
//   * q . S' is accumulated per column in registers across the rows a thread
//     owns, then reduced over the row groups through shared memory;
//   * optionally the mixer's steps after the readout follow in the same CTA
//     (the page's paragraph "GLA mixer"): o += sigmoid(q . (aug * k)) v, the
//     head RMSNorm over the dv columns, o *= silu(z) -- one thread per column.
#include "gla_internal.cuh"

namespace gla {
namespace {

// threads per CTA: dv / 4 threads per state row times 8 (dv = 192) or more rows
__host__ __device__ constexpr int decode_threads(int dv) { return dv == 192 ? 384 : 256; }

template <typename IO> struct Vec4In;
template <> struct Vec4In<float> {
  static __device__ __forceinline__ float4 load(const float* p) {
    return __ldg(reinterpret_cast<const float4*>(p));
  }
};
template <> struct Vec4In<__nv_bfloat16> {
  static __device__ __forceinline__ float4 load(const __nv_bfloat16* p) {
    const uint2 raw = __ldg(reinterpret_cast<const uint2*>(p));
    __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
    __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
    float2 a = __bfloat1622float2(lo), b = __bfloat1622float2(hi);
    return make_float4(a.x, a.y, b.x, b.y);
  }
};

template <typename IO, typename OUT, int DK, int DV, bool VEC>
__global__ void __launch_bounds__(decode_threads(DV), 2)
decode_kernel(const IO* __restrict__ q, const IO* __restrict__ k, const IO* __restrict__ v,
              const float* __restrict__ g, float scale, float* __restrict__ state,
              const int32_t* __restrict__ slots, int num_slots, unsigned* status, int H,
              OUT* __restrict__ out, const float* __restrict__ aug,
              const float* __restrict__ norm_w, float eps, const IO* __restrict__ z) {
  constexpr int TPR = DV / 4;                   // threads per state row
  constexpr int THREADS = decode_threads(DV);
  constexpr int RPP = THREADS / TPR;            // rows per pass
  constexpr int PASSES = DK / RPP;              // state float4 loads per thread
  static_assert(THREADS % TPR == 0 && DK % RPP == 0 && THREADS >= DK && THREADS >= DV,
                "tile shape");

  __shared__ float s_q[DK];
  __shared__ float s_k[DK];
  __shared__ float s_a[VEC ? DK : 1];
  __shared__ float s_red[RPP][DV];
  __shared__ float s_p[DK];              // q_i aug_i k_i (self-augmentation)
  __shared__ float s_ws[THREADS / 32];   // per-warp sums of o^2 (RMSNorm)

  const long long unit = blockIdx.x;  // n * H + h
  const int tid = threadIdx.x;
  const int col4 = tid % TPR;
  const int row0 = tid / TPR;

  // the state page: unit itself, or head h of pool page slots[n]
  long long page = unit;
  if (slots != nullptr) {
    const long long n = unit / H;
    const int slot = __ldg(slots + n);
    if (slot < 0) return;  // a padding row: no state, no output
    if (slot >= num_slots) {
      if (tid == 0) atomicOr(status, kDevBadSeqlens);
      return;
    }
    page = (long long)slot * H + (unit - n * H);
  }
  float4* S = reinterpret_cast<float4*>(state + page * (long long)(DK * DV));

  // Issue every state load of this thread first (PASSES x 16 bytes in flight).
  float4 s[PASSES];
#pragma unroll
  for (int p = 0; p < PASSES; ++p)
    s[p] = __ldcs(S + (row0 + p * RPP) * TPR + col4);

  if (tid < DK) {
    s_q[tid] = to_f32(q[unit * DK + tid]);
    s_k[tid] = to_f32(k[unit * DK + tid]);
    if constexpr (VEC) s_a[tid] = expf(__ldg(g + unit * DK + tid));
    if (aug) s_p[tid] = s_q[tid] * __ldg(aug + (unit % H) * DK + tid) * s_k[tid];
  }
  const float4 vv = Vec4In<IO>::load(v + unit * DV + col4 * 4);
  float a_scalar = 1.0f;
  if constexpr (!VEC) a_scalar = expf(__ldg(g + unit));
  __syncthreads();

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int p = 0; p < PASSES; ++p) {
    const int i = row0 + p * RPP;
    const float a = VEC ? s_a[i] : a_scalar;
    const float ki = s_k[i], qi = s_q[i];
    float4 x = s[p];
    x.x = fmaf(a, x.x, ki * vv.x);
    x.y = fmaf(a, x.y, ki * vv.y);
    x.z = fmaf(a, x.z, ki * vv.z);
    x.w = fmaf(a, x.w, ki * vv.w);
    __stcs(S + i * TPR + col4, x);
    acc.x = fmaf(qi, x.x, acc.x);
    acc.y = fmaf(qi, x.y, acc.y);
    acc.z = fmaf(qi, x.z, acc.z);
    acc.w = fmaf(qi, x.w, acc.w);
  }
  *reinterpret_cast<float4*>(&s_red[row0][col4 * 4]) = acc;
  __syncthreads();
  float o = 0.f;
  if (tid < DV) {
#pragma unroll
    for (int r = 0; r < RPP; ++r) o += s_red[r][tid];
    o *= scale;
  }
  // the mixer's steps after the readout (uniform branches: every thread takes them)
  const int h = (int)(unit % H);
  if (aug) {
    float s = 0.f;
#pragma unroll 8
    for (int i = 0; i < DK; ++i) s += s_p[i];
    if (tid < DV) o = fmaf(1.f / (1.f + expf(-s)), to_f32(v[unit * DV + tid]), o);
  }
  if (norm_w) {
    float x = (tid < DV) ? o * o : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    if ((tid & 31) == 0) s_ws[tid >> 5] = x;
    __syncthreads();
    float ss = 0.f;
#pragma unroll
    for (int w = 0; w < THREADS / 32; ++w) ss += s_ws[w];
    if (tid < DV) o *= rsqrtf(ss / DV + eps) * __ldg(norm_w + h * DV + tid);
  }
  if (z && tid < DV) {
    const float zz = to_f32(z[unit * DV + tid]);
    o *= zz / (1.f + expf(-zz));
  }
  if (tid < DV) out[unit * DV + tid] = from_f32<OUT>(o);
}

template <typename IO, typename OUT, int DK, int DV>
cudaError_t launch_typed(const DecodeArgs& a, cudaStream_t stream) {
  const long long units = (long long)a.N * a.H;
  const dim3 grid((unsigned)units);
  if (a.vector_gate)
    decode_kernel<IO, OUT, DK, DV, true><<<grid, decode_threads(DV), 0, stream>>>(
        (const IO*)a.q, (const IO*)a.k, (const IO*)a.v, a.g, a.scale, a.state, a.slots,
        a.num_slots, a.status, a.H, (OUT*)a.out, a.aug, a.norm_w, a.eps, (const IO*)a.z);
  else
    decode_kernel<IO, OUT, DK, DV, false><<<grid, decode_threads(DV), 0, stream>>>(
        (const IO*)a.q, (const IO*)a.k, (const IO*)a.v, a.g, a.scale, a.state, a.slots,
        a.num_slots, a.status, a.H, (OUT*)a.out, a.aug, a.norm_w, a.eps, (const IO*)a.z);
  return cudaGetLastError();
}

template <typename IO, typename OUT, int DK>
cudaError_t launch_dv(const DecodeArgs& a, cudaStream_t stream) {
  if (a.dv == 192) return launch_typed<IO, OUT, DK, 192>(a, stream);
  if (a.dv == 128) return launch_typed<IO, OUT, DK, 128>(a, stream);
  return launch_typed<IO, OUT, DK, 64>(a, stream);
}

template <typename IO, typename OUT>
cudaError_t launch_io(const DecodeArgs& a, cudaStream_t stream) {
  if (a.dk == 128) return launch_dv<IO, OUT, 128>(a, stream);
  if (a.dk == 96) return launch_dv<IO, OUT, 96>(a, stream);
  return launch_dv<IO, OUT, 64>(a, stream);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  if (a.fp32_io) return launch_io<float, float>(a, stream);
  if (a.fp32_out) return launch_io<__nv_bfloat16, float>(a, stream);
  return launch_io<__nv_bfloat16, __nv_bfloat16>(a, stream);
}

}  // namespace gla
