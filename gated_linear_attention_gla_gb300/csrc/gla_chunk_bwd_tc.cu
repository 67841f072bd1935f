// gla_chunk_bwd_tc.cu -- the backward for the per-head gate on the tensor
// cores: three runs of the tcgen05 prefill kernel.
//
// Method: reverse mode through the recurrence of the "i14 Laplace 3B on AWS
// Trainium2" page (paragraph "GLA mixer"), chunked as in its section
// "Challenge 1".  The gradient of a linear recurrence is the same kind of
// recurrence with the roles of its operands exchanged (fp64 check: 1e-15):
//   dq:  S^T_t = e^{g_t} S^T_{t-1} + v_t^T k_t,  dq_t = scale do_t S^T_t
//        -- the prefill with (q, k, v) = (do, v, k) and initial state S_0^T;
//        its final state is S_T^T.
//   dk, dv: with Sbar_t = dL/dS_t = scale q_t^T do_t + e^{g_{t+1}} Sbar_{t+1},
//        R_t = Sbar_t / scale obeys the prefill recurrence backwards in time,
//        with key q, value do, initial state dS_T / scale and, at reversed
//        position tau, the gate of the following token (g_{len - tau}; 0 at
//        tau = 0).  Then dk_t = scale v_t R_t^T -- the prefill with (q, k, v) =
//        (v, do, q) on the reversed sequence, state R^T -- and dv_t = scale
//        k_t R_t -- the prefill with (q, k, v) = (k, q, do), state R, whose
//        final state is R_0, so d_init = scale e^{g_0} R_0.
//   dg:  dg_t = sum_{u >= t} sum_i (q_u[i] dq_u[i] - k_u[i] dk_u[i])
//               + sum_ij S_T[i][j] dS_T[i][j].
// The prefill kernel reads tokens in order, so a prepare pass writes the
// reversed (and gate-shifted) copies into the caller's workspace.  Each run
// stores its gradient straight into the caller's buffer in the gradients'
// dtype (the dk and dv runs back in token order: row len - 1 - tau for
// reversed position tau), and the dq and dk runs add dg's per-token terms
// q . dq and -k . dk, formed from their fp32 outputs, to dg (zeroed first).  A
// tail pass adds the final-state term, takes the suffix sums and scales
// d_init.  Launches: prepare, 3 x prefill, and the tail when dg or d_init is
// wanted (plus a memset of dg).
#include "gla_chunk_bwd.cuh"

namespace gla {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kBlocksPerPair = 32;  // CTAs per (sequence, head) for the copy passes
constexpr int kTcDK = 128, kTcDV = 128;

__device__ __forceinline__ void pair_and_block(int H, int* s, int* h, int* blk) {
  const int pair = blockIdx.x / kBlocksPerPair;
  *blk = blockIdx.x % kBlocksPerPair;
  *s = pair / H;
  *h = pair % H;
}

// tokens [t0, t1) of a sequence of len tokens for copy block blk
__device__ __forceinline__ void block_range(int len, int blk, int* t0, int* t1) {
  const int per = (len + kBlocksPerPair - 1) / kBlocksPerPair;
  *t0 = min(len, blk * per);
  *t1 = min(len, *t0 + per);
}

// Reversed copies of q, k, v, do (token t of a sequence to position len-1-t),
// the gate shifted by one token (position tau holds g of natural token
// len - tau, position 0 holds 0), S_0^T, dS_T / scale and its transpose.
// The head sizes are template parameters so that the per-vector index
// arithmetic divides by constants.
template <int DK, int DV>
__global__ void __launch_bounds__(kCopyThreads)
bwd_tc_prep_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                   const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ d_out,
                   const float* __restrict__ g, float inv_scale,
                   const float* __restrict__ init_state, const float* __restrict__ d_final,
                   __nv_bfloat16* __restrict__ rq, __nv_bfloat16* __restrict__ rk,
                   __nv_bfloat16* __restrict__ rv, __nv_bfloat16* __restrict__ rdo,
                   float* __restrict__ rg, float* __restrict__ s0t, float* __restrict__ dfs,
                   float* __restrict__ dfst, const int32_t* __restrict__ cu, int B, int H,
                   int T, unsigned* status) {
  int s, h, blk;
  pair_and_block(H, &s, &h, &blk);
  long long start;
  int len;
  if (!seq_bounds(cu, s, B, T, &start, &len, status)) return;
  int t0, t1;
  block_range(len, blk, &t0, &t1);
  // 16-byte vectors: a token's q and k rows (DK / 8 each), then its v and do
  // rows (DV / 8 each); eight vectors a thread in flight at a time
  constexpr int VK = DK / 8, VV = DV / 8;
  constexpr int VPT = 2 * VK + 2 * VV;
  constexpr int kBatch = 8;
  // vector c of a token: its tensor (0 q, 1 k, 2 v, 3 do), index in the row, row width
  auto which = [&](int c, int* w, int* e, int* width) {
    if (c < 2 * VK) {
      *w = c / VK; *e = c % VK; *width = DK;
    } else {
      c -= 2 * VK;
      *w = 2 + c / VV; *e = c % VV; *width = DV;
    }
  };
  auto src_of = [&](int w) { return w == 0 ? q : w == 1 ? k : w == 2 ? v : d_out; };
  auto dst_of = [&](int w) { return w == 0 ? rq : w == 1 ? rk : w == 2 ? rv : rdo; };
  const int nvec = (t1 - t0) * VPT;
  for (int base = threadIdx.x; base < nvec; base += kCopyThreads * kBatch) {
    uint4 r[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int idx = base + b * kCopyThreads;
      if (idx < nvec) {
        const int t = t0 + idx / VPT;
        int w, e, width;
        which(idx % VPT, &w, &e, &width);
        const long long src = (start + t) * H + h;
        r[b] = __ldg(reinterpret_cast<const uint4*>(src_of(w) + src * width) + e);
      }
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int idx = base + b * kCopyThreads;
      if (idx < nvec) {
        const int t = t0 + idx / VPT;
        int w, e, width;
        which(idx % VPT, &w, &e, &width);
        const long long dst = (start + (len - 1 - t)) * H + h;
        reinterpret_cast<uint4*>(dst_of(w) + dst * width)[e] = r[b];
      }
    }
  }
  for (int t = t0 + threadIdx.x; t < t1; t += kCopyThreads)
    rg[(start + (len - 1 - t)) * H + h] = t + 1 < len ? __ldg(g + (start + t + 1) * H + h) : 0.f;
  // the states: 32 x 32 tiles spread over the blocks of the pair, transposed through
  // shared memory so that reads and writes are both row-contiguous
  __shared__ float tile[2][32][33];
  const size_t off = ((size_t)s * H + h) * (size_t)DK * DV;
  const int kTiles = (DK / 32) * (DV / 32);
  for (int tt = blk; tt < kTiles; tt += kBlocksPerPair) {
    const int ti = (tt / (DV / 32)) * 32, tj = (tt % (DV / 32)) * 32;
    const int r = threadIdx.x / 32, c = threadIdx.x % 32;  // 8 rows of 32 per pass
    __syncthreads();
    for (int rr = r; rr < 32; rr += kCopyThreads / 32) {
      const size_t e = off + (size_t)(ti + rr) * DV + tj + c;
      tile[0][rr][c] = init_state ? __ldg(init_state + e) : 0.f;
      if (d_final) {
        const float x = __ldg(d_final + e) * inv_scale;
        dfs[e] = x;
        tile[1][rr][c] = x;
      }
    }
    __syncthreads();
    for (int rr = r; rr < 32; rr += kCopyThreads / 32) {
      const size_t e = off + (size_t)(tj + rr) * DK + ti + c;  // row j, column i
      if (init_state) s0t[e] = tile[0][c][rr];
      if (d_final) dfst[e] = tile[1][c][rr];
    }
  }
}

__device__ __forceinline__ float warp_sum32(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

// The per-(sequence, head) tail of the backward, one CTA each: the final-state
// term of dg, sum_ij S_T[i][j] dS_T[i][j] = scale sum_e S_T^T[e] (dS_T /
// scale)^T[e] (both transposed copies in the workspace, read in order), added
// at the last token; the suffix sums of dg (whose per-token terms q.dq - k.dk
// the dq and dk runs have added); and d_init = scale e^{g_0} R_0 from the dv
// run's final state, in place.
__global__ void __launch_bounds__(kScanThreads)
bwd_tc_tail_kernel(const float* __restrict__ g, float scale, const float* __restrict__ stt,
                   const float* __restrict__ dfst, float* __restrict__ dg,
                   float* __restrict__ d_init, const int32_t* __restrict__ cu, int B, int H,
                   int T, int DK, int DV, unsigned* status) {
  __shared__ float red[kScanThreads / 32];
  __shared__ float warp_total[kScanThreads / 32];
  const long long unit = blockIdx.x;
  if (unit >= (long long)B * H) return;  // whole CTA
  const int s = (int)(unit / H), h = (int)(unit % H);
  long long start;
  int len;
  if (!seq_bounds(cu, s, B, T, &start, &len, status)) return;  // whole CTA
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const size_t st_off = ((size_t)s * H + h) * (size_t)DK * DV;
  const int kPer = DK * DV / 4 / kScanThreads;  // float4 a thread: 4, 8 or 16
  constexpr int kBatch = 4;                     // loads in flight (a divisor of kPer)
  if (dg && stt && dfst && len > 0) {
    float acc = 0.f;
#pragma unroll 1
    for (int b = 0; b < kPer; b += kBatch) {
      float4 x[kBatch], y[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int e = (b + u) * kScanThreads + threadIdx.x;
        x[u] = __ldg(reinterpret_cast<const float4*>(stt + st_off) + e);
        y[u] = __ldg(reinterpret_cast<const float4*>(dfst + st_off) + e);
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u)
        acc = fmaf(x[u].x, y[u].x, fmaf(x[u].y, y[u].y, fmaf(x[u].z, y[u].z,
                                                               fmaf(x[u].w, y[u].w, acc))));
    }
    acc = warp_sum32(acc);
    if (lane == 0) red[warp] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
      float c_t = 0.f;
      for (int w = 0; w < kScanThreads / 32; ++w) c_t += red[w];
      dg[(start + len - 1) * H + h] += scale * c_t;
    }
    __syncthreads();  // the scan reads that token
  }
  if (dg) dg_suffix_scan_cta(dg, start, len, H, h, warp_total);
  if (d_init) {
    const float f = len > 0 ? scale * expf(fmaxf(__ldg(g + start * H + h), -kGateClamp)) : scale;
    float4* p = reinterpret_cast<float4*>(d_init + st_off);
#pragma unroll 1
    for (int b = 0; b < kPer; b += kBatch) {
      float4 x[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) x[u] = p[(b + u) * kScanThreads + threadIdx.x];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        x[u].x *= f; x[u].y *= f; x[u].z *= f; x[u].w *= f;
        p[(b + u) * kScanThreads + threadIdx.x] = x[u];
      }
    }
  }
}

// Per-key-channel gate (dv only): reversed copies of q, k and do, the gate
// rows (one value per key channel) shifted by one token, and dS_T / scale.
__global__ void __launch_bounds__(kCopyThreads)
bwd_tc_prep_vec_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                       const __nv_bfloat16* __restrict__ d_out, const float* __restrict__ g,
                       float inv_scale, const float* __restrict__ d_final,
                       __nv_bfloat16* __restrict__ rq, __nv_bfloat16* __restrict__ rk,
                       __nv_bfloat16* __restrict__ rdo, float* __restrict__ rg,
                       float* __restrict__ dfs, const int32_t* __restrict__ cu, int B, int H,
                       int T, unsigned* status) {
  int s, h, blk;
  pair_and_block(H, &s, &h, &blk);
  long long start;
  int len;
  if (!seq_bounds(cu, s, B, T, &start, &len, status)) return;
  int t0, t1;
  block_range(len, blk, &t0, &t1);
  // 16-byte vectors of a token: q, k, do rows (bf16, 16 each) and its gate row
  // (fp32, 32); eight vectors a thread in flight at a time
  constexpr int VB = kTcDK / 8, VG = kTcDK / 4;
  constexpr int VPT = 3 * VB + VG;
  constexpr int kBatch = 8;
  static_assert(kTcDK == kTcDV, "one row width");
  auto src_of = [&](int c, long long row) -> const uint4* {
    if (c < 3 * VB) {
      const __nv_bfloat16* b = c < VB ? q : c < 2 * VB ? k : d_out;
      return reinterpret_cast<const uint4*>(b + row * kTcDK) + c % VB;
    }
    // the gate of the following token (none for the last one)
    return reinterpret_cast<const uint4*>(g + (row + H) * kTcDK) + (c - 3 * VB);
  };
  auto dst_of = [&](int c, long long row) -> uint4* {
    if (c < 3 * VB) {
      __nv_bfloat16* b = c < VB ? rq : c < 2 * VB ? rk : rdo;
      return reinterpret_cast<uint4*>(b + row * kTcDK) + c % VB;
    }
    return reinterpret_cast<uint4*>(rg + row * kTcDK) + (c - 3 * VB);
  };
  const int nvec = (t1 - t0) * VPT;
  for (int base = threadIdx.x; base < nvec; base += kCopyThreads * kBatch) {
    uint4 r[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int idx = base + b * kCopyThreads;
      if (idx < nvec) {
        const int t = t0 + idx / VPT, c = idx % VPT;
        const bool last_gate = c >= 3 * VB && t + 1 >= len;
        r[b] = last_gate ? make_uint4(0u, 0u, 0u, 0u) : __ldg(src_of(c, (start + t) * H + h));
      }
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int idx = base + b * kCopyThreads;
      if (idx < nvec) {
        const int t = t0 + idx / VPT, c = idx % VPT;
        *dst_of(c, (start + (len - 1 - t)) * H + h) = r[b];
      }
    }
  }
  if (d_final) {
    const size_t off = ((size_t)s * H + h) * (size_t)kTcDK * kTcDV;
    constexpr int kPer = kTcDK * kTcDV / 4 / kBlocksPerPair;
    const float4* src = reinterpret_cast<const float4*>(d_final + off) + blk * kPer;
    float4* dst = reinterpret_cast<float4*>(dfs + off) + blk * kPer;
    for (int e = threadIdx.x; e < kPer; e += kCopyThreads) {
      float4 x = __ldg(src + e);
      x.x *= inv_scale; x.y *= inv_scale; x.z *= inv_scale; x.w *= inv_scale;
      dst[e] = x;
    }
  }
}

// Workspace sections, each starting on a 256-byte boundary.
struct TcWorkspace {
  size_t rq, rk, rv, rdo, rg, s0t, dfs, dfst, stt, total;
};

TcWorkspace workspace_layout(int B, int H, long long rows, int DK, int DV) {
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const size_t tok = (size_t)rows * H;
  const size_t st = (size_t)B * H * DK * DV * 4;
  TcWorkspace w;
  size_t o = 0;
  w.rq = o;    o += up(tok * DK * 2);
  w.rk = o;    o += up(tok * DK * 2);
  w.rv = o;    o += up(tok * DV * 2);
  w.rdo = o;   o += up(tok * DV * 2);
  w.rg = o;    o += up(tok * 4);
  w.s0t = o;   o += up(st);
  w.dfs = o;   o += up(st);
  w.dfst = o;  o += up(st);
  w.stt = o;   o += up(st);
  w.total = o;
  return w;
}

// Per-key-channel gate: the workspace of the dv run.
struct TcVecWorkspace {
  size_t rq, rk, rdo, rg, dfs, total;
};

TcVecWorkspace vec_workspace_layout(int B, int H, long long rows) {
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const size_t tok = (size_t)rows * H;
  TcVecWorkspace w;
  size_t o = 0;
  w.rq = o;   o += up(tok * kTcDK * 2);
  w.rk = o;   o += up(tok * kTcDK * 2);
  w.rdo = o;  o += up(tok * kTcDV * 2);
  w.rg = o;   o += up(tok * kTcDK * 4);
  w.dfs = o;  o += up((size_t)B * H * kTcDK * kTcDV * 4);
  w.total = o;
  return w;
}

}  // namespace

bool chunk_bwd_tc_supported(int dk, int dv, bool fp32_io, bool vector_gate) {
  if (fp32_io) return false;
  // per-key-channel gate: dv's run on the d = 128 per-key-channel kernel;
  // per-head gate: every run's head sizes (d_k, d_v exchanged) are ones the
  // per-head kernel takes as key and value sizes
  if (vector_gate) return dk == kTcDK && dv == kTcDV;
  return (dk == 64 || dk == 128) && (dv == 64 || dv == 128);
}

size_t chunk_bwd_tc_workspace(int B, int H, long long rows, int dk, int dv, bool vector_gate) {
  return vector_gate ? vec_workspace_layout(B, H, rows).total
                     : workspace_layout(B, H, rows, dk, dv).total;
}

cudaError_t launch_chunk_bwd_tc_vec_dv(const ChunkBwdArgs& a, void* workspace,
                                       cudaStream_t stream) {
  const long long rows = a.cu_seqlens ? (long long)a.T : (long long)a.B * a.T;
  const TcVecWorkspace w = vec_workspace_layout(a.B, a.H, rows);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto bf = [&](size_t off) { return reinterpret_cast<__nv_bfloat16*>(ws + off); };
  auto fl = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };
  const unsigned grid = (unsigned)((long long)a.B * a.H * kBlocksPerPair);
  bwd_tc_prep_vec_kernel<<<grid, kCopyThreads, 0, stream>>>(
      (const __nv_bfloat16*)a.q, (const __nv_bfloat16*)a.k, (const __nv_bfloat16*)a.d_out, a.g,
      1.f / a.scale, a.d_final, bf(w.rq), bf(w.rk), bf(w.rdo), fl(w.rg), fl(w.dfs),
      a.cu_seqlens, a.B, a.H, a.T, a.status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // dv (reversed): the per-key-channel prefill of (k, q, do) with dS_T / scale,
  // stored back in token order and in the gradients' dtype
  ChunkArgs c{};
  c.q = bf(w.rk); c.k = bf(w.rq); c.v = bf(w.rdo); c.g = fl(w.rg);
  c.scale = a.scale; c.init_state = a.d_final ? fl(w.dfs) : nullptr;
  c.out = a.dv; c.out_reversed = true;
  c.final_state = nullptr; c.cu_seqlens = a.cu_seqlens;
  c.B = a.B; c.H = a.H; c.T = a.T; c.dk = kTcDK; c.dv = kTcDV; c.chunk = 128;
  c.fp32_io = false; c.fp32_out = a.fp32_out; c.vector_gate = true; c.status = a.status;
  return launch_chunk_tc_vec(c, stream);
}

cudaError_t launch_chunk_bwd_tc(const ChunkBwdArgs& a, void* workspace, cudaStream_t stream) {
  const long long rows = a.cu_seqlens ? (long long)a.T : (long long)a.B * a.T;
  const int DK = a.dk_size, DV = a.dv_size;
  const TcWorkspace w = workspace_layout(a.B, a.H, rows, DK, DV);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto bf = [&](size_t off) { return reinterpret_cast<__nv_bfloat16*>(ws + off); };
  auto fl = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };
  const unsigned grid = (unsigned)((long long)a.B * a.H * kBlocksPerPair);

  auto prep = DK == 64 ? (DV == 64 ? bwd_tc_prep_kernel<64, 64> : bwd_tc_prep_kernel<64, 128>)
                       : (DV == 64 ? bwd_tc_prep_kernel<128, 64> : bwd_tc_prep_kernel<128, 128>);
  prep<<<grid, kCopyThreads, 0, stream>>>(
      (const __nv_bfloat16*)a.q, (const __nv_bfloat16*)a.k, (const __nv_bfloat16*)a.v,
      (const __nv_bfloat16*)a.d_out, a.g, 1.f / a.scale, a.init_state, a.d_final, bf(w.rq),
      bf(w.rk), bf(w.rv), bf(w.rdo), fl(w.rg), fl(w.s0t), fl(w.dfs), fl(w.dfst), a.cu_seqlens,
      a.B, a.H, a.T, a.status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  // dg's per-token terms arrive from the dq and the dk run (one CTA per 64-wide
  // output slice each) as fp32 atomics
  if (a.dg) {
    if ((e = cudaMemsetAsync(a.dg, 0, sizeof(float) * (size_t)(rows * a.H), stream)) !=
        cudaSuccess)
      return e;
  }
  ChunkArgs c{};
  c.scale = a.scale; c.cu_seqlens = a.cu_seqlens; c.B = a.B; c.H = a.H; c.T = a.T;
  c.chunk = 128; c.fp32_io = false; c.fp32_out = a.fp32_out; c.vector_gate = false;
  c.status = a.status;
  // dq: the prefill of (do, v, k) with S_0^T, stored in dq's dtype, adding
  // q . dq to dg; its final state S_T^T feeds dg's final-state term
  c.q = a.d_out; c.k = a.v; c.v = a.k; c.g = a.g;
  c.init_state = a.init_state ? fl(w.s0t) : nullptr;
  c.out = a.dq;
  c.final_state = (a.dg && a.d_final) ? fl(w.stt) : nullptr;
  c.dot_rows = a.dg ? a.q : nullptr; c.dot_out = a.dg; c.dot_sign = 1.f;
  c.dk = DV; c.dv = DK;
  if ((e = launch_chunk_tc(c, stream)) != cudaSuccess) return e;
  // dk (reversed): the prefill of (v, do, q) with (dS_T / scale)^T, stored back
  // in token order, adding -k . dk to dg
  c.q = bf(w.rv); c.k = bf(w.rdo); c.v = bf(w.rq); c.g = fl(w.rg);
  c.init_state = a.d_final ? fl(w.dfst) : nullptr;
  c.out = a.dk; c.out_reversed = true;
  c.final_state = nullptr;
  c.dot_rows = a.dg ? a.k : nullptr; c.dot_out = a.dg; c.dot_sign = -1.f;
  c.dk = DV; c.dv = DK;
  if ((e = launch_chunk_tc(c, stream)) != cudaSuccess) return e;
  // dv (reversed): the prefill of (k, q, do) with dS_T / scale, stored back in
  // token order; final state R_0
  c.q = bf(w.rk); c.k = bf(w.rq); c.v = bf(w.rdo); c.g = fl(w.rg);
  c.init_state = a.d_final ? fl(w.dfs) : nullptr;
  c.out = a.dv; c.out_reversed = true;
  c.final_state = a.d_init;
  c.dot_rows = nullptr; c.dot_out = nullptr;
  c.dk = DK; c.dv = DV;
  if ((e = launch_chunk_tc(c, stream)) != cudaSuccess) return e;

  if (a.dg || a.d_init) {
    bwd_tc_tail_kernel<<<(unsigned)((long long)a.B * a.H), kScanThreads, 0, stream>>>(
        a.g, a.scale, (a.dg && a.d_final) ? fl(w.stt) : nullptr,
        a.d_final ? fl(w.dfst) : nullptr, a.dg, a.d_init, a.cu_seqlens, a.B, a.H, a.T, DK, DV,
        a.status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace gla
