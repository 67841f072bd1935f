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
//   bwd_dg_scan_kernel  per-head gate only: suffix sums of dg, one CTA per
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
constexpr int kLDP = kC + 4;  // P and M rows: 16-byte aligned, 4 banks apart
constexpr float kLog2e = 1.4426950408889634f;

// Store a gradient element as fp32 or (rounded to nearest-even) bf16.
__device__ __forceinline__ void store_grad(void* p, long long idx, float x, bool f32) {
  if (f32)
    static_cast<float*>(p)[idx] = x;
  else
    static_cast<__nv_bfloat16*>(p)[idx] = __float2bfloat16_rn(x);
}

// Four consecutive floats into shared memory: one 128-bit store where the row
// stride keeps them 16-byte aligned, else four scalar stores.
__device__ __forceinline__ void store4(float* d, float4 x, int ld) {
  if ((ld & 3) == 0) {
    *reinterpret_cast<float4*>(d) = x;
  } else {
    d[0] = x.x;
    d[1] = x.y;
    d[2] = x.z;
    d[3] = x.w;
  }
}

// A chunk's tile of a [rows, H, D] tensor -- rows base .. base + kC - 1,
// columns c0 .. c0 + W - 1 -- fetched as 16-byte vectors into registers, so
// that the next chunk's loads are in flight while this chunk is computed, and
// then put into shared memory as fp32 (row stride ld).  Rows past n are zero.
// Every row and column offset is a multiple of 16 bytes (checked by the host:
// 16-byte-aligned tensors, d a multiple of 32).
template <typename IO, int W>
struct TileFetch {
  static constexpr int VE = 16 / (int)sizeof(IO);  // elements per vector
  static constexpr int VPR = W / VE;               // vectors per row
  static constexpr int NV = kC * VPR;
  static constexpr int PER = (NV + kBwdThreads - 1) / kBwdThreads;
  static_assert(W % VE == 0, "tile width must be whole vectors");
  uint4 r[PER];

  __device__ __forceinline__ void fetch(const IO* __restrict__ src, long long base, int n,
                                        int H, int h, int D, int c0) {
#pragma unroll
    for (int p = 0; p < PER; ++p) {
      const int idx = threadIdx.x + p * kBwdThreads;
      const int t = idx / VPR, cv = idx - t * VPR;
      r[p] = make_uint4(0u, 0u, 0u, 0u);
      if (idx < NV && t < n)
        r[p] = __ldg(reinterpret_cast<const uint4*>(
            src + ((base + t) * H + h) * (long long)D + c0 + cv * VE));
    }
  }

  __device__ __forceinline__ void put(float* dst, int ld) const {
#pragma unroll
    for (int p = 0; p < PER; ++p) {
      const int idx = threadIdx.x + p * kBwdThreads;
      if (idx < NV) {
        const int t = idx / VPR, cv = idx - t * VPR;
        float* d = dst + t * ld + cv * VE;
        if constexpr (sizeof(IO) == 4) {
          store4(d, make_float4(__uint_as_float(r[p].x), __uint_as_float(r[p].y),
                                __uint_as_float(r[p].z), __uint_as_float(r[p].w)), ld);
        } else {
          // bf16 -> fp32 is exact: the bf16 bits are the high half of the float
          store4(d, make_float4(__uint_as_float(r[p].x << 16),
                                __uint_as_float(r[p].x & 0xffff0000u),
                                __uint_as_float(r[p].y << 16),
                                __uint_as_float(r[p].y & 0xffff0000u)), ld);
          store4(d + 4, make_float4(__uint_as_float(r[p].z << 16),
                                    __uint_as_float(r[p].z & 0xffff0000u),
                                    __uint_as_float(r[p].w << 16),
                                    __uint_as_float(r[p].w & 0xffff0000u)), ld);
        }
      }
    }
  }
};

// The chunk's log-decays: per key channel (W columns from c0, fetched like a
// tile) or per head (one value per token, strided by H).  put() stores them
// raw; gate_scan() turns them into running sums.
template <bool VEC, int W>
struct GateFetch {
  TileFetch<float, VEC ? W : 4> vec;
  float one;

  __device__ __forceinline__ void fetch(const float* __restrict__ g, long long base, int n,
                                        int H, int h, int DK, int c0) {
    if constexpr (VEC) {
      vec.fetch(g, base, n, H, h, DK, c0);
    } else {
      one = 0.f;
      if ((int)threadIdx.x < n) one = __ldg(g + (base + threadIdx.x) * H + h);
    }
  }

  __device__ __forceinline__ void put(float* G, int ld) const {
    if constexpr (VEC)
      vec.put(G, ld);
    else if (threadIdx.x < kC)
      G[threadIdx.x] = one;
  }
};

// G[t][c] <- log2(e) * sum_{s<=t} max(g_s, -clamp) down each of W columns
// (row stride ld), in place over the raw values that put() stored.  Rows past
// the chunk's end hold 0 and so repeat the last sum.
template <int W>
__device__ __forceinline__ void gate_scan(float* G, int ld) {
  if (threadIdx.x < W) {
    float v[kC];
#pragma unroll
    for (int t = 0; t < kC; ++t) v[t] = G[t * ld + threadIdx.x];
    float run = 0.f;
#pragma unroll
    for (int t = 0; t < kC; ++t) {
      run += fmaxf(v[t], -kGateClamp) * kLog2e;
      G[t * ld + threadIdx.x] = run;
    }
  }
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

// ---------------------------------------------------------------------------
// Register-tile products over shared memory.  Thread (tx, ty) = (tid % 16,
// tid / 16).  Row strides are multiples of 4 floats (16-byte rows) and, where
// 16 lanes read 16 different rows, 4 modulo 32, so that those 128-bit reads
// fall in distinct banks; the reads that all lanes of a half-warp share are
// broadcasts.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float4 ld4(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
__device__ __forceinline__ float2 ld2(const float* p) {
  return *reinterpret_cast<const float2*>(p);
}
__device__ __forceinline__ float comp(const float4& x, int i) {
  return i == 0 ? x.x : i == 1 ? x.y : i == 2 ? x.z : x.w;
}

// acc[m][n] += sum_k A[ty + 16 m][k] B[tx + 16 n][k]   (K a multiple of 4)
template <int TM, int TN>
__device__ __forceinline__ void gemm_nt(float (&acc)[TM][TN], const float* A, int lda,
                                        const float* B, int ldb, int K) {
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const float* pa = A + ty * lda;
  const float* pb = B + tx * ldb;
  float4 a[2][TM], b[2][TN];  // fragments of step k and k + 4, loaded one step ahead
#pragma unroll
  for (int m = 0; m < TM; ++m) a[0][m] = ld4(pa + 16 * m * lda);
#pragma unroll
  for (int n = 0; n < TN; ++n) b[0][n] = ld4(pb + 16 * n * ldb);
#pragma unroll 2
  for (int k = 0; k < K; k += 4) {
    const int cur = (k >> 2) & 1;
    if (k + 4 < K) {
#pragma unroll
      for (int m = 0; m < TM; ++m) a[cur ^ 1][m] = ld4(pa + 16 * m * lda + k + 4);
#pragma unroll
      for (int n = 0; n < TN; ++n) b[cur ^ 1][n] = ld4(pb + 16 * n * ldb + k + 4);
    }
#pragma unroll
    for (int m = 0; m < TM; ++m)
#pragma unroll
      for (int n = 0; n < TN; ++n) {
        acc[m][n] = fmaf(a[cur][m].x, b[cur][n].x, acc[m][n]);
        acc[m][n] = fmaf(a[cur][m].y, b[cur][n].y, acc[m][n]);
        acc[m][n] = fmaf(a[cur][m].z, b[cur][n].z, acc[m][n]);
        acc[m][n] = fmaf(a[cur][m].w, b[cur][n].w, acc[m][n]);
      }
  }
}

// acc[m][n] += sum_k A[ty + 16 m][k] B[k][tx + 16 n]   (K a multiple of 4)
template <int TM, int TN>
__device__ __forceinline__ void gemm_nn(float (&acc)[TM][TN], const float* A, int lda,
                                        const float* B, int ldb, int K) {
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll 2
  for (int k = 0; k < K; k += 4) {
    float4 a[TM];
#pragma unroll
    for (int m = 0; m < TM; ++m) a[m] = ld4(A + (ty + 16 * m) * lda + k);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      float b[TN];
#pragma unroll
      for (int n = 0; n < TN; ++n) b[n] = B[(k + kk) * ldb + tx + 16 * n];
#pragma unroll
      for (int m = 0; m < TM; ++m)
#pragma unroll
        for (int n = 0; n < TN; ++n) acc[m][n] = fmaf(comp(a[m], kk), b[n], acc[m][n]);
    }
  }
}

// Column of element n of a thread's row when every thread owns runs of four
// adjacent columns, the runs of a half-warp side by side: 4 tx + 64 (n / 4) + n % 4.
__device__ __forceinline__ int col4(int n) {
  return 4 * (threadIdx.x & 15) + 64 * (n >> 2) + (n & 3);
}

// acc[m][n] += sum_k A[k][TM ty + m] B[k][col4(n)]   (TM even, TN a multiple of 4)
template <int TM, int TN>
__device__ __forceinline__ void gemm_tn(float (&acc)[TM][TN], const float* A, int lda,
                                        const float* B, int ldb, int K) {
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll 4
  for (int k = 0; k < K; ++k) {
    float a[TM];
    float4 b[TN / 4];
#pragma unroll
    for (int m = 0; m < TM; m += 2) {
      const float2 x = ld2(A + k * lda + TM * ty + m);
      a[m] = x.x;
      a[m + 1] = x.y;
    }
#pragma unroll
    for (int n = 0; n < TN / 4; ++n) b[n] = ld4(B + k * ldb + 4 * tx + 64 * n);
#pragma unroll
    for (int m = 0; m < TM; ++m)
#pragma unroll
      for (int n = 0; n < TN; ++n) acc[m][n] = fmaf(a[m], comp(b[n >> 2], n & 3), acc[m][n]);
  }
}

// acc[m][n] += sum_k A[TM ty + m][k] B[k][col4(n)]   (K a multiple of 4, TN of 4)
template <int TM, int TN>
__device__ __forceinline__ void gemm_nn4(float (&acc)[TM][TN], const float* A, int lda,
                                         const float* B, int ldb, int K) {
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll 2
  for (int k = 0; k < K; k += 4) {
    float4 a[TM];
#pragma unroll
    for (int m = 0; m < TM; ++m) a[m] = ld4(A + (TM * ty + m) * lda + k);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      float4 b[TN / 4];
#pragma unroll
      for (int n = 0; n < TN / 4; ++n) b[n] = ld4(B + (k + kk) * ldb + 4 * tx + 64 * n);
#pragma unroll
      for (int m = 0; m < TM; ++m)
#pragma unroll
        for (int n = 0; n < TN; ++n)
          acc[m][n] = fmaf(comp(a[m], kk), comp(b[n >> 2], n & 3), acc[m][n]);
    }
  }
}

// P[a][b] = dO_a . V_b for b <= a (the later token a, the earlier b), times
// exp(G_a - G_b) for the per-head gate; zero above the diagonal.  The same
// matrix serves dq (rows t, columns u <= t) and dk (rows u, columns t <= u).
template <int DV, bool VEC>
__device__ __forceinline__ void make_p(float* sP, const float* sDO, const float* sV,
                                       const float* sG) {
  constexpr int LDV = DV + 4;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};
  gemm_nt<4, 4>(acc, sDO, LDV, sV, LDV, DV);
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
  static constexpr int LDV = DV + 4;  // 16-byte rows, 4 banks apart
  static constexpr int GW = VEC ? kIS : 1;
  static constexpr int kFloats =
      2 * kC * LDV + 2 * kC * kIS + kC * GW + kC * kLDP + kIS * LDV + (VEC ? kC * kIS : 0);
  static constexpr size_t kBytes = sizeof(float) * (size_t)kFloats;
};

// Per-key-channel gate: the in-chunk decays e^{G_t[i] - G_u[i]} of pairs in
// different 16-token sub-blocks are split at a sub-block boundary b between
// them, e^{G_t - G_b} e^{G_b - G_u} (both factors <= 1), so that one factor
// folds into the operand rows and the other into the result, one exp per
// (row, channel, sub-block); only pairs inside one sub-block take an exp each.
// Thread rows t = ty + 16 m lie in sub-block m.
constexpr int kSub = 16;

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
  float* sKh = sS + kIS * LDV;   // [kC][kIS]: k e^{G_b - G} to its sub-block's end b (VEC)

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

  TileFetch<IO, DV> fDO, fV;
  TileFetch<IO, kIS> fK, fQ;
  GateFetch<VEC, kIS> fG;
  auto fetch = [&](int c) {
    const int n = min(kC, len - c);
    const long long base = start + c;
    fDO.fetch(d_out, base, n, H, h, DV, 0);
    fV.fetch(v, base, n, H, h, DV, 0);
    fK.fetch(k, base, n, H, h, DK, i0);
    if (dg) fQ.fetch(q, base, n, H, h, DK, i0);
    fG.fetch(g, base, n, H, h, DK, i0);
  };
  if (len > 0) fetch(0);

  for (int c0 = 0; c0 < len; c0 += kC) {
    const int n = min(kC, len - c0);
    const long long base = start + c0;
    __syncthreads();  // the previous chunk is consumed
    fDO.put(sDO, LDV);
    fV.put(sV, LDV);
    fK.put(sK, kIS);
    if (dg) fQ.put(sQ, kIS);
    fG.put(sG, GW);
    __syncthreads();
    if (c0 + kC < len) fetch(c0 + kC);  // in flight during this chunk
    gate_scan<GW>(sG, GW);
    __syncthreads();
    make_p<DV, VEC>(sP, sDO, sV, sG);
    __syncthreads();

    // dq[t][i]: rows t = ty + 16 m, key rows i = tx + 16 c
    {
      float intra[4][2] = {}, inter[4][2] = {};
      if constexpr (VEC) {
        // u in an earlier sub-block: through that sub-block's last token b
        for (int idx = tid; idx < kC * kIS; idx += kBwdThreads) {
          const int u = idx / kIS, i = idx - u * kIS;
          sKh[idx] = sK[idx] * exp2f(sG[(u | (kSub - 1)) * kIS + i] - sG[u * kIS + i]);
        }
        __syncthreads();
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int t = ty + 16 * m;
          float gt[2];
#pragma unroll
          for (int c = 0; c < 2; ++c) gt[c] = sG[t * kIS + tx + 16 * c];
#pragma unroll
          for (int bu = 0; bu < m; ++bu) {
            float part[2] = {0.f, 0.f};
#pragma unroll 4
            for (int uu = 0; uu < kSub; ++uu) {
              const int u = kSub * bu + uu;
              const float a = sP[t * kLDP + u];
#pragma unroll
              for (int c = 0; c < 2; ++c) part[c] = fmaf(a, sKh[u * kIS + tx + 16 * c], part[c]);
            }
            const int b = kSub * bu + kSub - 1;
#pragma unroll
            for (int c = 0; c < 2; ++c)
              intra[m][c] =
                  fmaf(part[c], exp2f(gt[c] - sG[b * kIS + tx + 16 * c]), intra[m][c]);
          }
          // u in t's own sub-block, u <= t: one exp each (P is zero past t)
#pragma unroll 4
          for (int uu = 0; uu < kSub; ++uu) {
            const int u = kSub * m + uu;
            const float a = sP[t * kLDP + u];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              const float e = u <= t ? exp2f(gt[c] - sG[u * kIS + tx + 16 * c]) : 0.f;
              intra[m][c] = fmaf(a * sK[u * kIS + tx + 16 * c], e, intra[m][c]);
            }
          }
        }
      } else {
        gemm_nn<4, 2>(intra, sP, kLDP, sK, kIS, kC);
      }
      gemm_nt<4, 2>(inter, sDO, LDV, sS, LDV, DV);
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
      // rows i = 2 ty + r, columns col4(c)
      float acc[2][TN] = {};
      gemm_tn<2, TN>(acc, sK, kIS, sV, LDV, kC);
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int i = 2 * ty + r;
        const float el = exp2f(VEC ? sG[(n - 1) * kIS + i] : sG[n - 1]);
#pragma unroll
        for (int c = 0; c < TN; ++c) {
          float* p = sS + i * LDV + col4(c);
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
  static constexpr int LDV = DV + 4;  // 16-byte rows, 4 banks apart
  static constexpr int GW = VEC ? kIS : 1;
  static constexpr int kFloats = 2 * kC * LDV + 2 * kC * kIS + kC * GW + kC * kLDP +
                                kIS * LDV + (VEC ? 2 * kC * kIS : 0);
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
  float* sQh = sX + kC * kIS;    // [kC][kIS]: q e^{G - G_b} from the boundary b before its sub-block

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

  TileFetch<IO, DV> fDO, fV;
  TileFetch<IO, kIS> fQ, fK;
  GateFetch<VEC, kIS> fG;
  auto fetch = [&](int c) {
    const int n = min(kC, len - c);
    const long long base = start + c;
    fDO.fetch(d_out, base, n, H, h, DV, 0);
    fV.fetch(v, base, n, H, h, DV, 0);
    fQ.fetch(q, base, n, H, h, DK, i0);
    if (dg) fK.fetch(k, base, n, H, h, DK, i0);
    fG.fetch(g, base, n, H, h, DK, i0);
  };
  const int last_c0 = len > 0 ? ((len - 1) / kC) * kC : -1;
  if (len > 0) fetch(last_c0);

  for (int c0 = last_c0; c0 >= 0; c0 -= kC) {
    const int n = min(kC, len - c0);
    const long long base = start + c0;
    __syncthreads();
    fDO.put(sDO, LDV);
    fV.put(sV, LDV);
    fQ.put(sQ, kIS);
    if (dg) fK.put(sK, kIS);
    fG.put(sG, GW);
    __syncthreads();
    if (c0 > 0) fetch(c0 - kC);  // in flight during this chunk
    gate_scan<GW>(sG, GW);
    __syncthreads();
    make_p<DV, VEC>(sP, sDO, sV, sG);
    __syncthreads();

    // dk[t][i]: rows t = ty + 16 m, key rows i = tx + 16 c
    {
      float intra[4][2] = {}, inter[4][2] = {};
      if constexpr (VEC) {
        // u in a later sub-block: through the token b just before that sub-block
        for (int idx = kSub * kIS + tid; idx < kC * kIS; idx += kBwdThreads) {
          const int u = idx / kIS, i = idx - u * kIS;
          sQh[idx] = sQ[idx] * exp2f(sG[u * kIS + i] - sG[((u & ~(kSub - 1)) - 1) * kIS + i]);
        }
        __syncthreads();
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int t = ty + 16 * m;
          float gt[2];
#pragma unroll
          for (int c = 0; c < 2; ++c) gt[c] = sG[t * kIS + tx + 16 * c];
#pragma unroll
          for (int bu = m + 1; bu < 4; ++bu) {
            float part[2] = {0.f, 0.f};
#pragma unroll 4
            for (int uu = 0; uu < kSub; ++uu) {
              const int u = kSub * bu + uu;
              const float a = sP[u * kLDP + t];
#pragma unroll
              for (int c = 0; c < 2; ++c) part[c] = fmaf(a, sQh[u * kIS + tx + 16 * c], part[c]);
            }
            const int b = kSub * bu - 1;
#pragma unroll
            for (int c = 0; c < 2; ++c)
              intra[m][c] =
                  fmaf(part[c], exp2f(sG[b * kIS + tx + 16 * c] - gt[c]), intra[m][c]);
          }
          // u in t's own sub-block, u >= t: one exp each (P[u][t] is zero for u < t)
#pragma unroll 4
          for (int uu = 0; uu < kSub; ++uu) {
            const int u = kSub * m + uu;
            const float a = sP[u * kLDP + t];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              const float e = u >= t ? exp2f(sG[u * kIS + tx + 16 * c] - gt[c]) : 0.f;
              intra[m][c] = fmaf(a * sQ[u * kIS + tx + 16 * c], e, intra[m][c]);
            }
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
      gemm_nt<4, 2>(inter, sV, LDV, sR, LDV, DV);
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
      // rows i = 2 ty + r, columns col4(c)
      float acc[2][TN] = {};
      gemm_tn<2, TN>(acc, sQ, kIS, sDO, LDV, kC);
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int i = 2 * ty + r;
        const float el = exp2f(VEC ? sG[(n - 1) * kIS + i] : sG[n - 1]);
#pragma unroll
        for (int c = 0; c < TN; ++c) {
          float* p = sR + i * LDV + col4(c);
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
  static constexpr int LDK = DK + 4;              // 16-byte rows, 4 banks apart
  static constexpr int GW = VEC ? DK + 1 : 1;     // gate rows (scalar reads only)
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

  TileFetch<IO, DK> fQ, fK;
  TileFetch<IO, kJS> fDO;
  GateFetch<VEC, DK> fG;
  auto fetch = [&](int c) {
    const int n = min(kC, len - c);
    const long long base = start + c;
    fQ.fetch(q, base, n, H, h, DK, 0);
    fK.fetch(k, base, n, H, h, DK, 0);
    fDO.fetch(d_out, base, n, H, h, DV, j0);
    fG.fetch(g, base, n, H, h, DK, 0);
  };
  const int last_c0 = len > 0 ? ((len - 1) / kC) * kC : -1;
  if (len > 0) fetch(last_c0);

  for (int c0 = last_c0; c0 >= 0; c0 -= kC) {
    const int n = min(kC, len - c0);
    const long long base = start + c0;
    __syncthreads();
    fQ.put(sQ, LDK);
    fK.put(sK, LDK);
    fDO.put(sDO, kJS);
    fG.put(sG, GW);
    __syncthreads();
    if (c0 > 0) fetch(c0 - kC);  // in flight during this chunk
    gate_scan<VEC ? DK : 1>(sG, GW);
    __syncthreads();

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
            gu[m] = sG[(ty + 16 * m) * GW + i];
          }
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            b[c] = sK[(tx + 16 * c) * LDK + i];
            gt[c] = sG[(tx + 16 * c) * GW + i];
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
        gemm_nt<4, 4>(acc, sQ, LDK, sK, LDK, DK);
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
      const float gl = VEC ? sG[(n - 1) * GW + i] : sG[n - 1];
      const float gu = VEC ? sG[u * GW + i] : sG[u];
      sK[u * LDK + i] *= exp2f(gl - gu);
      sQ[u * LDK + i] *= exp2f(gu);
    }
    __syncthreads();

    // dv[t][j] = scale sum_u M[u][t] dO[u][j] + sum_i Kd[t][i] R[i][j]:
    // rows t = 4 ty + m, columns j = 4 tx + c
    {
      float acc[4][4] = {};
      gemm_tn<4, 4>(acc, sM, kLDP, sDO, kJS, kC);
#pragma unroll
      for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[m][c] *= scale;
      gemm_nn4<4, 4>(acc, sK, LDK, sR, kJS, DK);
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int t = 4 * ty + m;
        if (t < n) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            store_grad(dv_out, ((base + t) * H + h) * (long long)DV + j0 + 4 * tx + c,
                       acc[m][c], out_f32);
        }
      }
    }
    __syncthreads();

    // R <- diag(exp G_L) R + scale (Q exp(G))^T dO: rows i = TR ty + r, columns 4 tx + c
    {
      float acc[TR][4] = {};
      gemm_tn<TR, 4>(acc, sQ, LDK, sDO, kJS, kC);
#pragma unroll
      for (int r = 0; r < TR; ++r) {
        const int i = TR * ty + r;
        const float el = exp2f(VEC ? sG[(n - 1) * GW + i] : sG[n - 1]);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float* p = sR + i * kJS + 4 * tx + c;
          *p = fmaf(el, *p, scale * acc[r][c]);
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// per-head gate: dg_t <- sum_{u >= t} dg_u within each sequence (in place)
// ---------------------------------------------------------------------------
constexpr int kScanThreads = 256;
constexpr int kScanPer = 8;  // tokens per thread per pass

// Suffix sums of dg over the len tokens of one (sequence, head), in place, by
// one CTA of kScanThreads threads (warp_total: kScanThreads / 32 floats of
// shared memory).  A pass covers the last kScanThreads * kScanPer tokens not
// yet summed: thread i holds kScanPer consecutive tokens (later tokens in
// higher threads), sums them from the back, and adds the totals of every later
// thread (warp shuffles, then the warps' totals through shared memory) and of
// every later pass (the carry).
__device__ __forceinline__ void dg_suffix_scan_cta(float* __restrict__ dg, long long start,
                                                   int len, int H, int h, float* warp_total) {
  constexpr int kWarps = kScanThreads / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int kSpan = kScanThreads * kScanPer;
  float carry = 0.f;
  for (int end = len; end > 0; end -= kSpan) {
    const int lo = end - kSpan;  // may be negative: those tokens do not exist
    float x[kScanPer];
#pragma unroll
    for (int r = 0; r < kScanPer; ++r) {
      const int t = lo + kScanPer * (int)threadIdx.x + r;
      x[r] = (t >= 0) ? dg[(start + t) * H + h] : 0.f;
    }
    float suf = 0.f;
#pragma unroll
    for (int r = kScanPer - 1; r >= 0; --r) {
      suf += x[r];
      x[r] = suf;
    }
    float incl = suf;  // sum over this thread and the later lanes of its warp
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_down_sync(0xffffffffu, incl, off);
      if (lane + off < 32) incl += y;
    }
    if (lane == 0) warp_total[warp] = incl;
    __syncthreads();
    float later_warps = 0.f, pass_total = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float v = warp_total[w];
      pass_total += v;
      if (w > warp) later_warps += v;
    }
    const float later = incl - suf + later_warps + carry;
#pragma unroll
    for (int r = 0; r < kScanPer; ++r) {
      const int t = lo + kScanPer * (int)threadIdx.x + r;
      if (t >= 0) dg[(start + t) * H + h] = x[r] + later;
    }
    carry += pass_total;
    __syncthreads();  // warp_total is rewritten by the next pass
  }
}

// One CTA per (sequence, head).
__global__ void __launch_bounds__(kScanThreads)
bwd_dg_scan_kernel(float* __restrict__ dg, const int32_t* __restrict__ cu, int B, int H, int T,
                   unsigned* status) {
  __shared__ float warp_total[kScanThreads / 32];
  const long long unit = blockIdx.x;
  if (unit >= (long long)B * H) return;  // whole CTA
  const int s = (int)(unit / H), h = (int)(unit % H);
  long long start;
  int len;
  if (!seq_bounds(cu, s, B, T, &start, &len, status)) return;  // whole CTA
  dg_suffix_scan_cta(dg, start, len, H, h, warp_total);
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
  if (!a.skip_dv) {
    using L = DvSmem<DK, DV, VEC>;
    auto kern = bwd_dv_kernel<IO, DK, DV, VEC>;
    if ((e = set_smem(kern, L::kBytes)) != cudaSuccess) return e;
    kern<<<(unsigned)(pairs * (DV / kJS)), kBwdThreads, L::kBytes, stream>>>(
        (const IO*)a.q, (const IO*)a.k, a.g, a.scale, (const IO*)a.d_out, a.d_final,
        a.dv, a.fp32_out, a.cu_seqlens, a.B, a.H, a.T, a.status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (a.dg && !VEC) {
    bwd_dg_scan_kernel<<<(unsigned)pairs, kScanThreads, 0, stream>>>(a.dg, a.cu_seqlens, a.B,
                                                                      a.H, a.T, a.status);
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
