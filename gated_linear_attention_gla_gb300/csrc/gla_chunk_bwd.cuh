// gla_chunk_bwd.cuh -- the gradient of chunked GLA on the fp32 CUDA cores.
//
// Method: reverse mode through the recurrence of the "i14 Laplace 3B on AWS
// Trainium2" page (section "i14 and the Laplace 3B architecture", paragraph
// "GLA mixer"), in the chunked form of its section "Challenge 1" (Figure 3);
// the page trains the chunked layer and notes that its backward pass is
// unrolled over the chunks like the forward.  With Sbar_t = dL/dS_t:
//     Sbar_t = scale q_t^T do_t + diag(exp g_{t+1}) Sbar_{t+1}
//     dq_t = scale S_t do_t^T     dk_t = Sbar_t v_t^T     dv_t = k_t Sbar_t
// Inside a chunk (G_t = running sum of the clamped gate from the chunk start,
// G_L its last value, S the state entering the chunk, R = the gradient that
// reaches the chunk's last state from the chunks after it):
//     dq_t = scale (sum_{u<=t} (do_t.v_u) k_u e^{G_t-G_u} + e^{G_t} S do_t^T)
//     dk_t = scale sum_{u>=t} (do_u.v_t) q_u e^{G_u-G_t} + e^{G_L-G_t} R v_t^T
//     dv_t = scale sum_{u>=t} (q_u.(k_t e^{G_u-G_t})) do_u + (k_t e^{G_L-G_t}) R
//     S <- diag(e^{G_L}) S + sum_u (k_u e^{G_L-G_u})^T v_u       (forward)
//     R <- diag(e^{G_L}) R + scale sum_u (q_u e^{G_u})^T do_u     (backward)
// and the initial state's gradient is R after the first chunk.  Every decay
// factor above is at most 1, so nothing overflows for any chunk length.
//
// The gate's gradient uses dg_t[i] = sum_{u>=t} (q_u[i] dq_u[i] - k_u[i]
// dk_u[i]) + sum_j S_T[i][j] dS_T[i][j] (reverse mode of the same recurrence,
// summed over a suffix; summed over i for the per-head gate), so it needs no
// stored states: the dg output buffer first collects the per-token terms and
// is then summed from the end.
//
// Four launches, none of them needing scratch memory:
//   bwd_dq_kernel  forward sweep, one CTA per (sequence, head, 32 key rows):
//                  dq, the q*dq terms and the final-state term of dg
//   bwd_dk_kernel  reverse sweep, one CTA per (sequence, head, 32 key rows):
//                  dk, d_init, the k*dk terms; for the per-key-channel gate
//                  also the suffix sums (the CTA owns its columns of dg)
//   bwd_dv_kernel  reverse sweep, one CTA per (sequence, head, 64 value
//                  columns): dv
//   bwd_dg_scan_kernel  per-head gate only: suffix sums of dg, one warp per
//                  (sequence, head)
// The key-row and value-column splits keep every output owned by one CTA;
// only the per-head gate's dg terms are summed across CTAs (fp32 atomics, so
// its last bits depend on the order of arrival).
//
// Chunks are 64 tokens; every operand tile sits in shared memory as fp32 and
// each thread accumulates a register tile of rows ty + 16 m, columns tx + 16 n.
//
// The templates are instantiated per (gate, I/O dtype) in four translation
// units (gla_chunk_bwd_{head,chan}_{bf16,f32}.cu) so that they compile in
// parallel; the gradients' dtype (bf16 or fp32) is a run-time choice.
#pragma once
#include "gla_internal.cuh"

namespace gla {
namespace {

constexpr int kBwdThreads = 256;
constexpr int kC = 64;    // tokens per chunk
constexpr int kIS = 32;   // key rows per CTA (dq and dk kernels)
constexpr int kJS = 64;   // value columns per CTA (dv kernel)
constexpr int kLDP = kC + 1;
constexpr float kLog2e = 1.4426950408889634f;

// Store a gradient element as fp32 or (rounded to nearest-even) bf16.
__device__ __forceinline__ void store_grad(void* p, long long idx, float x, bool f32) {
  if (f32)
    static_cast<float*>(p)[idx] = x;
  else
    static_cast<__nv_bfloat16*>(p)[idx] = __float2bfloat16_rn(x);
}

// dst[t][c] (row stride ld) <- src rows base + t, columns c0 + c of a [rows, H, D]
// tensor, for t < kC and c < W; rows past n are zero.
template <int W, typename IO>
__device__ __forceinline__ void load_tile(float* dst, int ld, const IO* __restrict__ src,
                                          long long base, int n, int H, int h, int D, int c0) {
  for (int idx = threadIdx.x; idx < kC * W; idx += kBwdThreads) {
    const int t = idx / W, c = idx - t * W;
    dst[t * ld + c] =
        t < n ? to_f32(src[((base + t) * H + h) * (long long)D + c0 + c]) : 0.f;
  }
}

// G[t][c] <- log2(e) * sum_{s<=t} max(g_s, -clamp) for the chunk's tokens, per
// key channel c0 + c (W columns, row stride ld) or per head (W = 1).  Rows past
// n repeat the last sum.  Two barriers inside.
template <int W, bool VEC>
__device__ __forceinline__ void load_gate(float* G, int ld, const float* __restrict__ g,
                                          long long base, int n, int H, int h, int DK, int c0) {
  for (int idx = threadIdx.x; idx < kC * W; idx += kBwdThreads) {
    const int t = idx / W, c = idx - t * W;
    float x = 0.f;
    if (t < n) {
      const float raw = VEC ? g[((base + t) * H + h) * (long long)DK + c0 + c]
                            : g[(base + t) * H + h];
      x = fmaxf(raw, -kGateClamp) * kLog2e;
    }
    G[t * ld + c] = x;
  }
  __syncthreads();
  if (threadIdx.x < W) {
    float v[kC];
#pragma unroll
    for (int t = 0; t < kC; ++t) v[t] = G[t * ld + threadIdx.x];
    float run = 0.f;
#pragma unroll
    for (int t = 0; t < kC; ++t) {
      run += v[t];
      G[t * ld + threadIdx.x] = run;
    }
  }
  __syncthreads();
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

// Sum over the 16 lanes that share a tile row (lanes 0-15 or 16-31).
__device__ __forceinline__ float row_sum16(float x) {
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

// P[a][b] = dO_a . V_b for b <= a (the later token a, the earlier b), times
// exp(G_a - G_b) for the per-head gate; zero above the diagonal.  The same
// matrix serves dq (rows t, columns u <= t) and dk (rows u, columns t <= u).
template <int DV, bool VEC>
__device__ __forceinline__ void make_p(float* sP, const float* sDO, const float* sV,
                                       const float* sG) {
  constexpr int LDV = DV + 1;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};
#pragma unroll 4
  for (int j = 0; j < DV; ++j) {
    float a[4], b[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) a[m] = sDO[(ty + 16 * m) * LDV + j];
#pragma unroll
    for (int c = 0; c < 4; ++c) b[c] = sV[(tx + 16 * c) * LDV + j];
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[m][c] = fmaf(a[m], b[c], acc[m][c]);
  }
#pragma unroll
  for (int m = 0; m < 4; ++m)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int r = ty + 16 * m, col = tx + 16 * c;
      float p = 0.f;
      if (col <= r) p = VEC ? acc[m][c] : acc[m][c] * exp2f(sG[r] - sG[col]);
      sP[r * kLDP + col] = p;
    }
}

// ---------------------------------------------------------------------------
// dq (forward sweep over the chunks)
// ---------------------------------------------------------------------------
template <int DK, int DV, bool VEC>
struct DqSmem {
  static constexpr int LDV = DV + 1;
  static constexpr int GW = VEC ? kIS : 1;
  static constexpr int kFloats =
      2 * kC * LDV + 2 * kC * kIS + kC * GW + kC * kLDP + kIS * LDV;
  static constexpr size_t kBytes = sizeof(float) * (size_t)kFloats;
};

template <typename IO, int DK, int DV, bool VEC>
__global__ void __launch_bounds__(kBwdThreads, 1)
bwd_dq_kernel(const IO* __restrict__ q, const IO* __restrict__ k, const IO* __restrict__ v,
              const float* __restrict__ g, float scale, const float* __restrict__ init_state,
              const IO* __restrict__ d_out, const float* __restrict__ d_final,
              void* __restrict__ dq, bool out_f32, float* __restrict__ dg,
              const int32_t* __restrict__ cu, int B, int H, int T, unsigned* status) {
  using L = DqSmem<DK, DV, VEC>;
  constexpr int LDV = L::LDV, GW = L::GW, NS = DK / kIS, TN = DV / 16;
  extern __shared__ float sm[];
  float* sDO = sm;               // [kC][LDV]
  float* sV = sDO + kC * LDV;    // [kC][LDV]
  float* sK = sV + kC * LDV;     // [kC][kIS]: k, then k * exp(G_L - G)
  float* sQ = sK + kC * kIS;     // [kC][kIS]
  float* sG = sQ + kC * kIS;     // [kC][GW]
  float* sP = sG + kC * GW;      // [kC][kLDP]
  float* sS = sP + kC * kLDP;    // [kIS][LDV]: the state's rows i0 .. i0 + 31

  const int slice = blockIdx.x % NS;
  const int h = (blockIdx.x / NS) % H;
  const int s = blockIdx.x / (NS * H);
  const int i0 = slice * kIS;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  long long start;
  int len;
  if (!seq_bounds(cu, s, B, T, &start, &len, status)) return;
  const size_t st_off = ((size_t)s * H + h) * (size_t)DK * DV;

  for (int idx = tid; idx < kIS * DV; idx += kBwdThreads) {
    const int i = idx / DV, j = idx - i * DV;
    sS[i * LDV + j] = init_state ? init_state[st_off + (size_t)(i0 + i) * DV + j] : 0.f;
  }

  for (int c0 = 0; c0 < len; c0 += kC) {
    const int n = min(kC, len - c0);
    const long long base = start + c0;
    __syncthreads();  // the previous chunk is consumed
    load_tile<DV>(sDO, LDV, d_out, base, n, H, h, DV, 0);
    load_tile<DV>(sV, LDV, v, base, n, H, h, DV, 0);
    load_tile<kIS>(sK, kIS, k, base, n, H, h, DK, i0);
    if (dg) load_tile<kIS>(sQ, kIS, q, base, n, H, h, DK, i0);
    load_gate<GW, VEC>(sG, GW, g, base, n, H, h, DK, i0);
    make_p<DV, VEC>(sP, sDO, sV, sG);
    __syncthreads();

    // dq[t][i]: rows t = ty + 16 m, key rows i = tx + 16 c
    {
      float intra[4][2] = {}, inter[4][2] = {};
      if constexpr (VEC) {
        float gt[4][2];
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
          for (int c = 0; c < 2; ++c) gt[m][c] = sG[(ty + 16 * m) * kIS + tx + 16 * c];
#pragma unroll 2
        for (int u = 0; u < kC; ++u) {
          float a[4], b[2], gu[2];
#pragma unroll
          for (int m = 0; m < 4; ++m) a[m] = sP[(ty + 16 * m) * kLDP + u];
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            b[c] = sK[u * kIS + tx + 16 * c];
            gu[c] = sG[u * kIS + tx + 16 * c];
          }
#pragma unroll
          for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              const float e = (u <= ty + 16 * m) ? exp2f(gt[m][c] - gu[c]) : 0.f;
              intra[m][c] = fmaf(a[m] * b[c], e, intra[m][c]);
            }
        }
      } else {
#pragma unroll 4
        for (int u = 0; u < kC; ++u) {
          float a[4], b[2];
#pragma unroll
          for (int m = 0; m < 4; ++m) a[m] = sP[(ty + 16 * m) * kLDP + u];
#pragma unroll
          for (int c = 0; c < 2; ++c) b[c] = sK[u * kIS + tx + 16 * c];
#pragma unroll
          for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int c = 0; c < 2; ++c) intra[m][c] = fmaf(a[m], b[c], intra[m][c]);
        }
      }
#pragma unroll 4
      for (int j = 0; j < DV; ++j) {
        float a[4], b[2];
#pragma unroll
        for (int m = 0; m < 4; ++m) a[m] = sDO[(ty + 16 * m) * LDV + j];
#pragma unroll
        for (int c = 0; c < 2; ++c) b[c] = sS[(tx + 16 * c) * LDV + j];
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
          for (int c = 0; c < 2; ++c) inter[m][c] = fmaf(a[m], b[c], inter[m][c]);
      }
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int t = ty + 16 * m;
        float xs = 0.f;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int i = tx + 16 * c;
          if (t < n) {
            const float e = exp2f(VEC ? sG[t * kIS + i] : sG[t]);
            const float d = scale * fmaf(e, inter[m][c], intra[m][c]);
            const long long row = (base + t) * H + h;
            store_grad(dq, row * DK + i0 + i, d, out_f32);
            const float x = sQ[t * kIS + i] * d;
            if (VEC && dg) dg[row * DK + i0 + i] = x;
            xs += x;
          }
        }
        if (!VEC && dg) {  // every lane of the warp takes part in the shuffles
          xs = row_sum16(xs);
          if (tx == 0 && t < n) atomicAdd(dg + (base + t) * H + h, xs);
        }
      }
    }
    __syncthreads();

    // state step: S <- diag(exp G_L) S + (K exp(G_L - G))^T V
    for (int idx = tid; idx < kC * kIS; idx += kBwdThreads) {
      const int u = idx / kIS, i = idx - u * kIS;
      const float gl = VEC ? sG[(n - 1) * kIS + i] : sG[n - 1];
      const float gu = VEC ? sG[u * kIS + i] : sG[u];
      sK[idx] = u < n ? sK[idx] * exp2f(gl - gu) : 0.f;
    }
    __syncthreads();
    {
      float acc[2][TN] = {};
#pragma unroll 4
      for (int u = 0; u < kC; ++u) {
        float a[2], b[TN];
#pragma unroll
        for (int r = 0; r < 2; ++r) a[r] = sK[u * kIS + ty + 16 * r];
#pragma unroll
        for (int c = 0; c < TN; ++c) b[c] = sV[u * LDV + tx + 16 * c];
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
          for (int c = 0; c < TN; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int i = ty + 16 * r;
        const float el = exp2f(VEC ? sG[(n - 1) * kIS + i] : sG[n - 1]);
#pragma unroll
        for (int c = 0; c < TN; ++c) {
          float* p = sS + i * LDV + tx + 16 * c;
          *p = fmaf(el, *p, acc[r][c]);
        }
      }
    }
  }

  // the final state's part of dg: sum_j S_T[i][j] dS_T[i][j], at the last token
  if (dg && d_final && len > 0) {
    __syncthreads();
    const int lane = tid & 31, warp = tid >> 5;
    const long long last = start + len - 1;
    for (int i = warp; i < kIS; i += kBwdThreads / 32) {
      float acc = 0.f;
      for (int j = lane; j < DV; j += 32)
        acc = fmaf(sS[i * LDV + j], d_final[st_off + (size_t)(i0 + i) * DV + j], acc);
      acc = warp_sum(acc);
      if (lane == 0) {
        if (VEC)
          dg[(last * H + h) * DK + i0 + i] += acc;
        else
          atomicAdd(dg + last * H + h, acc);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// dk, d_init (reverse sweep)
// ---------------------------------------------------------------------------
template <int DK, int DV, bool VEC>
struct DkSmem {
  static constexpr int LDV = DV + 1;
  static constexpr int GW = VEC ? kIS : 1;
  static constexpr int kFloats =
      2 * kC * LDV + 2 * kC * kIS + kC * GW + kC * kLDP + kIS * LDV + (VEC ? kC * kIS : 0);
  static constexpr size_t kBytes = sizeof(float) * (size_t)kFloats;
};

template <typename IO, int DK, int DV, bool VEC>
__global__ void __launch_bounds__(kBwdThreads, 1)
bwd_dk_kernel(const IO* __restrict__ q, const IO* __restrict__ k, const IO* __restrict__ v,
              const float* __restrict__ g, float scale, const IO* __restrict__ d_out,
              const float* __restrict__ d_final, void* __restrict__ dk_out,
              bool out_f32, float* __restrict__ dg, float* __restrict__ d_init,
              const int32_t* __restrict__ cu, int B, int H, int T, unsigned* status) {
  using L = DkSmem<DK, DV, VEC>;
  constexpr int LDV = L::LDV, GW = L::GW, NS = DK / kIS, TN = DV / 16;
  extern __shared__ float sm[];
  float* sDO = sm;               // [kC][LDV]
  float* sV = sDO + kC * LDV;    // [kC][LDV]
  float* sQ = sV + kC * LDV;     // [kC][kIS]: q, then q * exp(G)
  float* sK = sQ + kC * kIS;     // [kC][kIS]
  float* sG = sK + kC * kIS;     // [kC][GW]
  float* sP = sG + kC * GW;      // [kC][kLDP]
  float* sR = sP + kC * kLDP;    // [kIS][LDV]: rows i0 .. i0 + 31 of the carried gradient
  float* sX = sR + kIS * LDV;    // [kC][kIS]: dg terms (per-key-channel gate)

  const int slice = blockIdx.x % NS;
  const int h = (blockIdx.x / NS) % H;
  const int s = blockIdx.x / (NS * H);
  const int i0 = slice * kIS;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  long long start;
  int len;
  if (!seq_bounds(cu, s, B, T, &start, &len, status)) return;
  const size_t st_off = ((size_t)s * H + h) * (size_t)DK * DV;

  for (int idx = tid; idx < kIS * DV; idx += kBwdThreads) {
    const int i = idx / DV, j = idx - i * DV;
    sR[i * LDV + j] = d_final ? d_final[st_off + (size_t)(i0 + i) * DV + j] : 0.f;
  }
  float carry = 0.f;  // per-key-channel gate: thread i < kIS carries column i's suffix sum

  for (int c0 = ((len - 1) / kC) * kC; c0 >= 0 && len > 0; c0 -= kC) {
    const int n = min(kC, len - c0);
    const long long base = start + c0;
    __syncthreads();
    load_tile<DV>(sDO, LDV, d_out, base, n, H, h, DV, 0);
    load_tile<DV>(sV, LDV, v, base, n, H, h, DV, 0);
    load_tile<kIS>(sQ, kIS, q, base, n, H, h, DK, i0);
    if (dg) load_tile<kIS>(sK, kIS, k, base, n, H, h, DK, i0);
    load_gate<GW, VEC>(sG, GW, g, base, n, H, h, DK, i0);
    make_p<DV, VEC>(sP, sDO, sV, sG);
    __syncthreads();

    // dk[t][i]: rows t = ty + 16 m, key rows i = tx + 16 c
    {
      float intra[4][2] = {}, inter[4][2] = {};
      if constexpr (VEC) {
        float gt[4][2];
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
          for (int c = 0; c < 2; ++c) gt[m][c] = sG[(ty + 16 * m) * kIS + tx + 16 * c];
#pragma unroll 2
        for (int u = 0; u < kC; ++u) {
          float a[4], b[2], gu[2];
#pragma unroll
          for (int m = 0; m < 4; ++m) a[m] = sP[u * kLDP + ty + 16 * m];
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            b[c] = sQ[u * kIS + tx + 16 * c];
            gu[c] = sG[u * kIS + tx + 16 * c];
          }
#pragma unroll
          for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              const float e = (u >= ty + 16 * m) ? exp2f(gu[c] - gt[m][c]) : 0.f;
              intra[m][c] = fmaf(a[m] * b[c], e, intra[m][c]);
            }
        }
      } else {
#pragma unroll 4
        for (int u = 0; u < kC; ++u) {
          float a[4], b[2];
#pragma unroll
          for (int m = 0; m < 4; ++m) a[m] = sP[u * kLDP + ty + 16 * m];
#pragma unroll
          for (int c = 0; c < 2; ++c) b[c] = sQ[u * kIS + tx + 16 * c];
#pragma unroll
          for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int c = 0; c < 2; ++c) intra[m][c] = fmaf(a[m], b[c], intra[m][c]);
        }
      }
#pragma unroll 4
      for (int j = 0; j < DV; ++j) {
        float a[4], b[2];
#pragma unroll
        for (int m = 0; m < 4; ++m) a[m] = sV[(ty + 16 * m) * LDV + j];
#pragma unroll
        for (int c = 0; c < 2; ++c) b[c] = sR[(tx + 16 * c) * LDV + j];
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
          for (int c = 0; c < 2; ++c) inter[m][c] = fmaf(a[m], b[c], inter[m][c]);
      }
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int t = ty + 16 * m;
        float xs = 0.f;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int i = tx + 16 * c;
          float x = 0.f;
          if (t < n) {
            const float gl = VEC ? sG[(n - 1) * kIS + i] : sG[n - 1];
            const float gt = VEC ? sG[t * kIS + i] : sG[t];
            const float d = fmaf(scale, intra[m][c], exp2f(gl - gt) * inter[m][c]);
            const long long row = (base + t) * H + h;
            store_grad(dk_out, row * DK + i0 + i, d, out_f32);
            if (dg) {
              x = -sK[t * kIS + i] * d;
              if (VEC) x += dg[row * DK + i0 + i];  // the q * dq term (and the final-state term)
            }
          }
          if (VEC) sX[t * kIS + i] = x;
          xs += x;
        }
        if (!VEC && dg) {
          xs = row_sum16(xs);
          if (tx == 0 && t < n) atomicAdd(dg + (base + t) * H + h, xs);
        }
      }
    }
    __syncthreads();

    // per-key-channel gate: suffix sums down column i, carried across chunks
    if (VEC && dg && tid < kIS) {
      float run = carry;
      for (int t = n - 1; t >= 0; --t) {
        run += sX[t * kIS + tid];
        dg[((base + t) * H + h) * DK + i0 + tid] = run;
      }
      carry = run;
    }

    // R <- diag(exp G_L) R + scale (Q exp(G))^T dO
    for (int idx = tid; idx < kC * kIS; idx += kBwdThreads) {
      const int u = idx / kIS, i = idx - u * kIS;
      sQ[idx] *= exp2f(VEC ? sG[u * kIS + i] : sG[u]);
    }
    __syncthreads();
    {
      float acc[2][TN] = {};
#pragma unroll 4
      for (int u = 0; u < kC; ++u) {
        float a[2], b[TN];
#pragma unroll
        for (int r = 0; r < 2; ++r) a[r] = sQ[u * kIS + ty + 16 * r];
#pragma unroll
        for (int c = 0; c < TN; ++c) b[c] = sDO[u * LDV + tx + 16 * c];
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
          for (int c = 0; c < TN; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int i = ty + 16 * r;
        const float el = exp2f(VEC ? sG[(n - 1) * kIS + i] : sG[n - 1]);
#pragma unroll
        for (int c = 0; c < TN; ++c) {
          float* p = sR + i * LDV + tx + 16 * c;
          *p = fmaf(el, *p, scale * acc[r][c]);
        }
      }
    }
  }
  __syncthreads();
  if (d_init) {
    for (int idx = tid; idx < kIS * DV; idx += kBwdThreads) {
      const int i = idx / DV, j = idx - i * DV;
      d_init[st_off + (size_t)(i0 + i) * DV + j] = sR[i * LDV + j];
    }
  }
}

// ---------------------------------------------------------------------------
// dv (reverse sweep)
// ---------------------------------------------------------------------------
template <int DK, int DV, bool VEC>
struct DvSmem {
  static constexpr int LDK = DK + 1;
  static constexpr int GW = VEC ? LDK : 1;
  static constexpr int kFloats = 2 * kC * LDK + kC * kJS + kC * GW + kC * kLDP + DK * kJS;
  static constexpr size_t kBytes = sizeof(float) * (size_t)kFloats;
};

template <typename IO, int DK, int DV, bool VEC>
__global__ void __launch_bounds__(kBwdThreads, 1)
bwd_dv_kernel(const IO* __restrict__ q, const IO* __restrict__ k, const float* __restrict__ g,
              float scale, const IO* __restrict__ d_out, const float* __restrict__ d_final,
              void* __restrict__ dv_out, bool out_f32, const int32_t* __restrict__ cu, int B,
              int H, int T, unsigned* status) {
  using L = DvSmem<DK, DV, VEC>;
  constexpr int LDK = L::LDK, GW = L::GW, NS = DV / kJS, TR = DK / 16;
  extern __shared__ float sm[];
  float* sQ = sm;                // [kC][LDK]: q, then q * exp(G)
  float* sK = sQ + kC * LDK;     // [kC][LDK]: k, then k * exp(G_L - G)
  float* sDO = sK + kC * LDK;    // [kC][kJS]
  float* sG = sDO + kC * kJS;    // [kC][GW]
  float* sM = sG + kC * GW;      // [kC][kLDP]
  float* sR = sM + kC * kLDP;    // [DK][kJS]: columns j0 .. j0 + 63 of the carried gradient

  const int slice = blockIdx.x % NS;
  const int h = (blockIdx.x / NS) % H;
  const int s = blockIdx.x / (NS * H);
  const int j0 = slice * kJS;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  long long start;
  int len;
  if (!seq_bounds(cu, s, B, T, &start, &len, status)) return;
  const size_t st_off = ((size_t)s * H + h) * (size_t)DK * DV;

  for (int idx = tid; idx < DK * kJS; idx += kBwdThreads) {
    const int i = idx / kJS, j = idx - i * kJS;
    sR[idx] = d_final ? d_final[st_off + (size_t)i * DV + j0 + j] : 0.f;
  }

  for (int c0 = ((len - 1) / kC) * kC; c0 >= 0 && len > 0; c0 -= kC) {
    const int n = min(kC, len - c0);
    const long long base = start + c0;
    __syncthreads();
    load_tile<DK>(sQ, LDK, q, base, n, H, h, DK, 0);
    load_tile<DK>(sK, LDK, k, base, n, H, h, DK, 0);
    load_tile<kJS>(sDO, kJS, d_out, base, n, H, h, DV, j0);
    if constexpr (VEC)
      load_gate<DK, true>(sG, LDK, g, base, n, H, h, DK, 0);
    else
      load_gate<1, false>(sG, 1, g, base, n, H, h, DK, 0);

    // M[u][t] = q_u . (k_t exp(G_u - G_t)) for t <= u: rows u = ty + 16 m, columns t = tx + 16 c
    {
      float acc[4][4] = {};
      if constexpr (VEC) {
#pragma unroll 2
        for (int i = 0; i < DK; ++i) {
          float a[4], b[4], gu[4], gt[4];
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            a[m] = sQ[(ty + 16 * m) * LDK + i];
            gu[m] = sG[(ty + 16 * m) * LDK + i];
          }
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            b[c] = sK[(tx + 16 * c) * LDK + i];
            gt[c] = sG[(tx + 16 * c) * LDK + i];
          }
#pragma unroll
          for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const float e = (tx + 16 * c <= ty + 16 * m) ? exp2f(gu[m] - gt[c]) : 0.f;
              acc[m][c] = fmaf(a[m] * b[c], e, acc[m][c]);
            }
        }
      } else {
#pragma unroll 4
        for (int i = 0; i < DK; ++i) {
          float a[4], b[4];
#pragma unroll
          for (int m = 0; m < 4; ++m) a[m] = sQ[(ty + 16 * m) * LDK + i];
#pragma unroll
          for (int c = 0; c < 4; ++c) b[c] = sK[(tx + 16 * c) * LDK + i];
#pragma unroll
          for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[m][c] = fmaf(a[m], b[c], acc[m][c]);
        }
      }
#pragma unroll
      for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int u = ty + 16 * m, t = tx + 16 * c;
          float x = 0.f;
          if (t <= u) x = VEC ? acc[m][c] : acc[m][c] * exp2f(sG[u] - sG[t]);
          sM[u * kLDP + t] = x;
        }
    }
    __syncthreads();
    // K <- K exp(G_L - G), Q <- Q exp(G)
    for (int idx = tid; idx < kC * DK; idx += kBwdThreads) {
      const int u = idx / DK, i = idx - u * DK;
      const float gl = VEC ? sG[(n - 1) * LDK + i] : sG[n - 1];
      const float gu = VEC ? sG[u * LDK + i] : sG[u];
      sK[u * LDK + i] *= exp2f(gl - gu);
      sQ[u * LDK + i] *= exp2f(gu);
    }
    __syncthreads();

    // dv[t][j] = scale sum_u M[u][t] dO[u][j] + sum_i Kd[t][i] R[i][j]
    {
      float acc[4][4] = {};
#pragma unroll 4
      for (int u = 0; u < kC; ++u) {
        float a[4], b[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) a[m] = sM[u * kLDP + ty + 16 * m];
#pragma unroll
        for (int c = 0; c < 4; ++c) b[c] = sDO[u * kJS + tx + 16 * c];
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[m][c] = fmaf(a[m], b[c], acc[m][c]);
      }
#pragma unroll
      for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[m][c] *= scale;
#pragma unroll 4
      for (int i = 0; i < DK; ++i) {
        float a[4], b[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) a[m] = sK[(ty + 16 * m) * LDK + i];
#pragma unroll
        for (int c = 0; c < 4; ++c) b[c] = sR[i * kJS + tx + 16 * c];
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[m][c] = fmaf(a[m], b[c], acc[m][c]);
      }
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int t = ty + 16 * m;
        if (t < n) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            store_grad(dv_out, ((base + t) * H + h) * (long long)DV + j0 + tx + 16 * c,
                       acc[m][c], out_f32);
        }
      }
    }
    __syncthreads();

    // R <- diag(exp G_L) R + scale (Q exp(G))^T dO: rows i = ty + 16 r
    {
      float acc[TR][4] = {};
#pragma unroll 4
      for (int u = 0; u < kC; ++u) {
        float a[TR], b[4];
#pragma unroll
        for (int r = 0; r < TR; ++r) a[r] = sQ[u * LDK + ty + 16 * r];
#pragma unroll
        for (int c = 0; c < 4; ++c) b[c] = sDO[u * kJS + tx + 16 * c];
#pragma unroll
        for (int r = 0; r < TR; ++r)
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
      }
#pragma unroll
      for (int r = 0; r < TR; ++r) {
        const int i = ty + 16 * r;
        const float el = exp2f(VEC ? sG[(n - 1) * LDK + i] : sG[n - 1]);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float* p = sR + i * kJS + tx + 16 * c;
          *p = fmaf(el, *p, scale * acc[r][c]);
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// per-head gate: dg_t <- sum_{u >= t} dg_u within each sequence (in place)
// ---------------------------------------------------------------------------
constexpr int kScanWarps = 8;
constexpr int kScanPer = 8;  // tokens per lane per pass

__global__ void __launch_bounds__(kScanWarps * 32)
bwd_dg_scan_kernel(float* __restrict__ dg, const int32_t* __restrict__ cu, int B, int H, int T,
                   unsigned* status) {
  const int lane = threadIdx.x & 31;
  const long long unit = (long long)blockIdx.x * kScanWarps + (threadIdx.x >> 5);
  if (unit >= (long long)B * H) return;
  const int s = (int)(unit / H), h = (int)(unit % H);
  long long start;
  int len;
  if (!seq_bounds(cu, s, B, T, &start, &len, status)) return;
  constexpr int kSpan = 32 * kScanPer;
  float carry = 0.f;
  for (int end = len; end > 0; end -= kSpan) {
    const int lo = end - kSpan;  // may be negative: those tokens do not exist
    float x[kScanPer];
#pragma unroll
    for (int r = 0; r < kScanPer; ++r) {
      const int t = lo + kScanPer * lane + r;
      x[r] = (t >= 0 && t < end) ? dg[(start + t) * H + h] : 0.f;
    }
    float suf = 0.f;
#pragma unroll
    for (int r = kScanPer - 1; r >= 0; --r) {
      suf += x[r];
      x[r] = suf;
    }
    float incl = suf;  // sum over this lane and every later lane
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_down_sync(0xffffffffu, incl, off);
      if (lane + off < 32) incl += y;
    }
    const float later = incl - suf + carry;
#pragma unroll
    for (int r = 0; r < kScanPer; ++r) {
      const int t = lo + kScanPer * lane + r;
      if (t >= 0 && t < end) dg[(start + t) * H + h] = x[r] + later;
    }
    carry += __shfl_sync(0xffffffffu, incl, 0);
  }
}

// ---------------------------------------------------------------------------
// launch
// ---------------------------------------------------------------------------
template <typename K>
cudaError_t set_smem(K kern, size_t bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <typename IO, int DK, int DV, bool VEC>
cudaError_t launch_shape(const ChunkBwdArgs& a, cudaStream_t stream) {
  const long long pairs = (long long)a.B * a.H;
  cudaError_t e;
  if (a.dg && !VEC) {
    const long long rows = a.cu_seqlens ? (long long)a.T : (long long)a.B * a.T;
    e = cudaMemsetAsync(a.dg, 0, sizeof(float) * (size_t)(rows * a.H), stream);
    if (e != cudaSuccess) return e;
  }
  {
    using L = DqSmem<DK, DV, VEC>;
    auto kern = bwd_dq_kernel<IO, DK, DV, VEC>;
    if ((e = set_smem(kern, L::kBytes)) != cudaSuccess) return e;
    kern<<<(unsigned)(pairs * (DK / kIS)), kBwdThreads, L::kBytes, stream>>>(
        (const IO*)a.q, (const IO*)a.k, (const IO*)a.v, a.g, a.scale, a.init_state,
        (const IO*)a.d_out, a.d_final, a.dq, a.fp32_out, a.dg, a.cu_seqlens, a.B, a.H, a.T, a.status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  {
    using L = DkSmem<DK, DV, VEC>;
    auto kern = bwd_dk_kernel<IO, DK, DV, VEC>;
    if ((e = set_smem(kern, L::kBytes)) != cudaSuccess) return e;
    kern<<<(unsigned)(pairs * (DK / kIS)), kBwdThreads, L::kBytes, stream>>>(
        (const IO*)a.q, (const IO*)a.k, (const IO*)a.v, a.g, a.scale, (const IO*)a.d_out,
        a.d_final, a.dk, a.fp32_out, a.dg, a.d_init, a.cu_seqlens, a.B, a.H, a.T, a.status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  {
    using L = DvSmem<DK, DV, VEC>;
    auto kern = bwd_dv_kernel<IO, DK, DV, VEC>;
    if ((e = set_smem(kern, L::kBytes)) != cudaSuccess) return e;
    kern<<<(unsigned)(pairs * (DV / kJS)), kBwdThreads, L::kBytes, stream>>>(
        (const IO*)a.q, (const IO*)a.k, a.g, a.scale, (const IO*)a.d_out, a.d_final,
        a.dv, a.fp32_out, a.cu_seqlens, a.B, a.H, a.T, a.status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (a.dg && !VEC) {
    const unsigned grid = (unsigned)((pairs + kScanWarps - 1) / kScanWarps);
    bwd_dg_scan_kernel<<<grid, kScanWarps * 32, 0, stream>>>(a.dg, a.cu_seqlens, a.B, a.H, a.T,
                                                              a.status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <typename IO, int DK, bool VEC>
cudaError_t launch_dv(const ChunkBwdArgs& a, cudaStream_t stream) {
  if (a.dv_size == 192) return launch_shape<IO, DK, 192, VEC>(a, stream);
  if (a.dv_size == 128) return launch_shape<IO, DK, 128, VEC>(a, stream);
  return launch_shape<IO, DK, 64, VEC>(a, stream);
}

// All head sizes of one (I/O dtype, gate) pair.
template <typename IO, bool VEC>
cudaError_t launch_bwd(const ChunkBwdArgs& a, cudaStream_t stream) {
  if (a.dk_size == 128) return launch_dv<IO, 128, VEC>(a, stream);
  if (a.dk_size == 96) return launch_dv<IO, 96, VEC>(a, stream);
  return launch_dv<IO, 64, VEC>(a, stream);
}

}  // namespace
}  // namespace gla
