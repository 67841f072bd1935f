// gla_chunk_tc_vec.cu -- chunked GLA prefill with a per-key-channel gate on the
// 5th-generation tensor cores.
//
// Method: the chunked form of the "i14 Laplace 3B on AWS Trainium2" page
// (section "Challenge 1", Figure 3) with the gate extended to one log-decay
// per key channel (row i of the state decays by exp(g_t,i)).  For a chunk of
// C = 128 tokens, G_t,i = sum of g over the chunk up to and including t in
// channel i, L the chunk's last token:
//     S_next = diag(exp G_L) S + Kt^T V,            Kt_j = k_j * exp(G_L - G_j)   (<= 1)
//     o_t    = scale * ( (q_t * exp G_t) S + sum_{j<=t} A_tj V_j ),
//     A_tj   = sum_i q_ti k_ji exp(G_ti - G_ji) = Q'_t . Kt_j,  Q'_t = q_t * exp(G_t - G_L)
// so with S' = diag(exp G_L) S the output is o = scale * (Q' S' + causal(Q' Kt^T) V):
// the decay moves into the operands (Kt serves the state update and the
// scores) and no per-row factor remains.  Q' <= exp(span) with span =
// max_i (G_0,i - G_L,i); while span stays below 2^100 every operand is a
// normal bf16 number.  A chunk with a wider span ("wide": several resets or
// very strong decay) is processed token by token on the CUDA cores instead,
// with the state in registers (exact, slow, rare).
//
// One CTA owns one (sequence, head) with the full d_v = 128 and walks the
// chunks in order.  The state S (128 x 128 fp32) lives in tensor memory.
// Per chunk, bf16 x bf16 -> fp32 contractions:
//     MMA1  A  = Q' Kt^T          M=128 (t) N=128 (j) K=128 (i)  hi and lo of Kt
//     MMA3  O  = Q' S'_bf16       M=128 (t) N=128     K=128 (i)
//     MMA4  S += Kt^T V           M=128 (i) N=128     K=128 (t)  hi and lo of Kt
//     MMA2  O += P' V             M=128 (t) N=128     K=128 (j)  P' in TMEM, plus
//                                                               the diagonal lo part
// P' = causal(A) is rounded to bf16 once, except on the four 32 x 32 diagonal
// blocks, which also carry a lo part (as in the per-head kernel).
//
// Roles (16 warps):
//   warp 0       producer: TMA loads of g (fp32 [128 x 128], 64 KB), Q, K, V
//   warp 1       TMEM allocator; issues every MMA
//   warps 4..7   mask group: P' from A (thread t = token row t), then the
//                output of the previous chunk
//   warps 8..15  gate group: in-chunk prefix sums of g per channel, Q' and
//                Kt (hi in place over K, lo in its own tile); then the state
//                pass (S <- diag(exp G_L) S in TMEM, its bf16 copy S');
//                wide chunks and the final state
// Buffers (single, except O): g, Q, K, Kt_lo, V, S' in shared memory; A/P',
// O (two, by parity of the chunk's index among the tensor-core chunks), S in
// TMEM.  Every mbarrier wait is bounded in wall time; on timeout the kernel
// flags the device status word, stops issuing work, releases TMEM and
// returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "gla_internal.cuh"
#include "gla_sm100.cuh"

namespace gla {
namespace {

using namespace sm100;

constexpr int kC = 128;        // chunk (tokens)
constexpr int kD = 128;        // d_k = d_v
constexpr int kThreads = 512;  // 16 warps
constexpr int kMaskWarps = 4;
constexpr int kGateWarps = 8;
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitLimitNs = kDefaultWaitLimitNs;  // the drains' limit (2 s)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kWideSpan = 100.f;  // log2 span above which a chunk is processed token by token

// shared memory map; the dynamic shared memory base must be 1024-byte aligned
constexpr uint32_t kPanel = kC * 128;             // 16 KB: 128 rows x 128 B
constexpr uint32_t kTile = 2 * kPanel;            // 32 KB: 128 x 128 bf16, two 64-column panels
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kTile;         // Kt hi in place after the gate pass
constexpr uint32_t kOffKlo = kOffK + kTile;       // Kt lo; wide chunks: reduction scratch
constexpr uint32_t kOffV = kOffKlo + kTile;
constexpr uint32_t kOffSb = kOffV + kTile;        // S' bf16: row i (K), 128 columns (N)
constexpr uint32_t kOffG = kOffSb + kTile;        // g: [128 tokens][128 channels] fp32
constexpr uint32_t kGBytes = kC * kD * 4;
constexpr uint32_t kOffPart = kOffG + kGBytes;    // 4 x 128 fp32 partial sums of g
constexpr uint32_t kOffWide = kOffPart + 4 * kD * 4;  // 4 ints: wide flags by chunk % 4
constexpr uint32_t kOffVote = kOffWide + 16;          // 2 ints: the gate group's wide votes
constexpr uint32_t kOffBar = kOffVote + 16;
constexpr uint32_t kBarBytes = 256;
constexpr uint32_t kOffMisc = kOffBar + kBarBytes;    // tmem base, abort flag
constexpr uint32_t kSmemBytes = kOffMisc + 16;
static_assert(kSmemBytes <= 232448, "shared memory budget");

// TMEM column map
constexpr uint32_t kColA = 0;     // A = Q' Kt^T (fp32), then P' (bf16 pairs) and its diagonal lo
constexpr uint32_t kColO = 128;   // 2 x 128: O by tensor-core chunk parity
constexpr uint32_t kColS = 384;   // 128: the running state, fp32

enum Bar {
  kGFull = 0, kGEmpty, kQKFull, kQKEmpty, kVFull, kVEmpty, kScaled0, kScaled1, kSbReady,
  kAFull, kPFull0, kPFull1, kSFull, kOFull0, kOFull1, kOFree0, kOFree1, kAck0, kAck1,
  kGateSync, kDrain, kNumBars
};
static_assert(kNumBars * 8 <= kBarBytes, "barrier area");

constexpr uint32_t kIdQK = idesc_bf16(128, 128, false, false);
constexpr uint32_t kIdQS = idesc_bf16(128, 128, false, true);
constexpr uint32_t kIdKV = idesc_bf16(128, 128, true, true);
constexpr uint32_t kIdPV = idesc_bf16(128, 128, false, true);

struct VecParams {
  float scale;
  const float* init_state;
  void* out;
  float* final_state;
  const int32_t* cu_seqlens;
  int B, H, T;
  int out_v8;        // out is 32-byte aligned: 256-bit stores
  int out_reversed;  // token t of a sequence stored at row len - 1 - t
  unsigned* status;
  uint64_t wait_ns;  // limit of the hand-off waits (the drain keeps kWaitLimitNs)
  // MIX kernels: the mixer's steps after the readout, each skipped when null --
  // self-augmentation weights [H, 128], head RMSNorm weights [H, 128] and eps,
  // output gate z [rows, H, 128] (bf16)
  const float* aug;
  const float* norm_w;
  float eps;
  const __nv_bfloat16* z;
};

// logistic sigmoid and SiLU with the fast exponential and reciprocal (the
// mixer's gate runs once per output element; 1 / inf = 0 gives the limits)
// 2^x by the hardware approximation (PTX ex2.approx.ftz): for the operand
// scaling, whose exponents stay within [-100, 100] on the tensor-core chunks, so
// that no result is subnormal; it gives the same bits as exp2f there and skips
// exp2f's handling of the ranges outside.
__device__ __forceinline__ float ex2_(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float sigmoidf_(float x) { return __fdividef(1.f, 1.f + __expf(-x)); }
__device__ __forceinline__ float siluf_(float x) { return __fdividef(x, 1.f + __expf(-x)); }

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Byte offset of the bf16 pair (row, columns 2p, 2p + 1) in a 128-row tile of
// two 64-column panels, 128-byte swizzled (the TMA SWIZZLE_128B layout).
__device__ __forceinline__ uint32_t pair_offset(uint32_t row, uint32_t p) {
  const uint32_t col = 2 * p;
  return (col >> 6) * kPanel + sw128_offset(row, (col & 63) >> 3) + (col & 7) * 2;
}

// P' of token row r (lane quadrant q4) from A in TMEM, in place: block cb (32
// fp32 columns) becomes 16 columns of bf16 pairs at 16 cb (read by then), the
// lo part of the row's diagonal block goes to 64 + 16 q4, the other lo blocks
// are zero.  Plain causal mask (diagonal kept); diag_add is added to the
// row's diagonal entry (the mixer's self-augmentation term, 0 without it).
__device__ __forceinline__ void build_p(uint32_t a_row, int q4, int r, float diag_add) {
  uint32_t a[32], dlo[16];
  tmem_ld_32x32b_x32(a_row, a);
#pragma unroll 1
  for (int cb = 0; cb < 4; ++cb) {
    uint32_t pk[16];
    if (cb > q4) {
#pragma unroll
      for (int e = 0; e < 16; ++e) pk[e] = 0u;
    } else if (cb < q4) {
      tmem_ld_wait_x32(a);
#pragma unroll
      for (int e = 0; e < 16; ++e)
        pk[e] = pack_bf16x2(__uint_as_float(a[2 * e]), __uint_as_float(a[2 * e + 1]));
      tmem_ld_32x32b_x32(a_row + 32 * (cb + 1), a);
    } else {
      tmem_ld_wait_x32(a);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int j = 32 * cb + 2 * e;
        const float x0 = j <= r ? __uint_as_float(a[2 * e]) + (j == r ? diag_add : 0.f) : 0.f;
        const float x1 =
            j + 1 <= r ? __uint_as_float(a[2 * e + 1]) + (j + 1 == r ? diag_add : 0.f) : 0.f;
        pk[e] = pack_bf16x2(x0, x1);
        dlo[e] = pack_bf16x2(x0 - bf16lo(pk[e]), x1 - bf16hi(pk[e]));
      }
    }
    tmem_st_32x32b_x16(a_row + 16 * cb, pk);
  }
#pragma unroll 1
  for (int b = 0; b < 4; ++b) {
    if (b == q4) {
      tmem_st_32x32b_x16(a_row + 64 + 16 * b, dlo);
    } else {
      uint32_t z[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) z[e] = 0u;
      tmem_st_32x32b_x16(a_row + 64 + 16 * b, z);
    }
  }
}

template <bool OUTF32, bool MIX>
__global__ void __launch_bounds__(kThreads, 1)
chunk_tc_vec_kernel(const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmG, const VecParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  // the layout assumes a 1024-byte aligned base (the 128-byte swizzle atoms)
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicOr(p.status, kDevLayout);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  volatile int* wide_ring = reinterpret_cast<volatile int*>(smem + kOffWide);
  int* vote = reinterpret_cast<int*>(smem + kOffVote);
  float* gsm = reinterpret_cast<float*>(smem + kOffG);
  float* part = reinterpret_cast<float*>(smem + kOffPart);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x % p.H;
  const int s = blockIdx.x / p.H;

  long long start;
  int len;
  if (!seq_bounds(p.cu_seqlens, s, p.B, p.T, &start, &len, p.status)) return;
  const int nch = (len + kC - 1) / kC;
  const bool packed = p.cu_seqlens != nullptr;

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      uint32_t cnt = 1;
      if (i == kPFull0 || i == kPFull1 || i == kOFree0 || i == kOFree1) cnt = kMaskWarps;
      if (i == kScaled0 || i == kScaled1 || i == kSbReady || i == kGateSync) cnt = kGateWarps;
      // the issuer and the mask warps acknowledge each chunk's flags
      if (i == kAck0 || i == kAck1) cnt = 1 + kMaskWarps;
      // with the mixer, the mask warps also read a chunk's Q' and Kt rows
      if (MIX && i == kQKEmpty) cnt = 1 + kMaskWarps;
      mbar_init(&bars[i], cnt);
    }
    *abort_flag = 0;
    vote[0] = vote[1] = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmG);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sbase = smem_u32(smem);

  // a hand-off wait: gives up once the CTA is aborting, or after p.wait_ns
  // (then it starts the abort)
  auto wait = [&](int b, uint32_t parity) -> bool {
    if (*abort_flag) return false;
    if (mbar_try_wait(&bars[b], parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
      if (mbar_try_wait(&bars[b], parity)) return true;
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > p.wait_ns) {
        *abort_flag = 1;
        atomicOr(p.status, kDevTimeout);
        return false;
      }
    }
  };
  // the same, decided for the whole warp (full-warp roles never split on a wait)
  auto wait_w = [&](int b, uint32_t parity) -> bool {
    return __all_sync(0xffffffffu, wait(b, parity));
  };
  auto ph = [](int k) -> uint32_t { return static_cast<uint32_t>(k) & 1u; };
  auto warp_arrive = [&](int b) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[b]);
  };

  // the TMA transactions the producer started on kGFull, kQKFull, kVFull (one
  // per chunk each), for the teardown drain
  int issued_g = 0, issued_qk = 0, issued_v = 0;
  bool mma_issued = false;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const int bidx = packed ? 0 : s;
      for (int c = 0; c < nch; ++c) {
        const int row = packed ? (int)(start + (long long)c * kC) : c * kC;
        if (c >= 1 && !wait(kGEmpty, ph(c - 1))) break;
        mbar_arrive_expect_tx(&bars[kGFull], kGBytes);
        tma_load_4d(gsm, &tmG, &bars[kGFull], 0, h, row, bidx);
        ++issued_g;
        if (c >= 1 && !wait(kQKEmpty, ph(c - 1))) break;
        mbar_arrive_expect_tx(&bars[kQKFull], 2 * kTile);
#pragma unroll
        for (int pn = 0; pn < 2; ++pn) {
          tma_load_4d(smem + kOffQ + pn * kPanel, &tmQ, &bars[kQKFull], pn * 64, h, row, bidx);
          tma_load_4d(smem + kOffK + pn * kPanel, &tmK, &bars[kQKFull], pn * 64, h, row, bidx);
        }
        ++issued_qk;
        if (c >= 1 && !wait(kVEmpty, ph(c - 1))) break;
        mbar_arrive_expect_tx(&bars[kVFull], kTile);
#pragma unroll
        for (int pn = 0; pn < 2; ++pn)
          tma_load_4d(smem + kOffV + pn * kPanel, &tmV, &bars[kVFull], pn * 64, h, row, bidx);
        ++issued_v;
        // every tile is single-buffered, so chunk c + 1's loads can only be issued
        // once chunk c has released them: fetch its tiles into L2 now, so that
        // those loads then wait for L2 rather than HBM
        if (c + 1 < nch) {
          const int nrow = row + kC;
          tma_prefetch_l2_4d(&tmG, 0, h, nrow, bidx);
#pragma unroll
          for (int pn = 0; pn < 2; ++pn) {
            tma_prefetch_l2_4d(&tmQ, pn * 64, h, nrow, bidx);
            tma_prefetch_l2_4d(&tmK, pn * 64, h, nrow, bidx);
            tma_prefetch_l2_4d(&tmV, pn * 64, h, nrow, bidx);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Per tensor-core chunk (index n among them): MMA1, MMA3, MMA4, then MMA2.
    // The whole warp waits and forms the descriptors; one elected lane issues.
    const uint64_t qd = sdesc_sw128(sbase + kOffQ, 16, 1024);
    const uint64_t kd = sdesc_sw128(sbase + kOffK, 16, 1024);
    const uint64_t kld = sdesc_sw128(sbase + kOffKlo, 16, 1024);
    const uint64_t ktd = sdesc_sw128(sbase + kOffK, kPanel, 1024);    // Kt^T (MN-major)
    const uint64_t ktld = sdesc_sw128(sbase + kOffKlo, kPanel, 1024);
    const uint64_t sd = sdesc_sw128(sbase + kOffSb, kPanel, 1024);
    const uint64_t vd = sdesc_sw128(sbase + kOffV, kPanel, 1024);
    int n = 0;
    for (int c = 0; c < nch; ++c) {
      if (!wait_w(kScaled0 + (c & 1), ph(c >> 1))) break;
      const bool wide = wide_ring[c & 3] != 0;
      warp_arrive(kAck0 + (c & 1));
      if (wide) continue;  // processed by the gate group
      const int ob = n & 1;
      tc_fence_after();
      if (elect_one_sync()) {
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
          mma_bf16(tmem + kColA, desc_add(qd, off), desc_add(kd, off), kIdQK, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
          mma_bf16(tmem + kColA, desc_add(qd, off), desc_add(kld, off), kIdQK, 1);
        }
        mma_commit(&bars[kAFull]);
      }
      __syncwarp();
      mma_issued = true;
      if (!wait_w(kSbReady, ph(n))) break;
      if (n >= 2 && !wait_w(kOFree0 + ob, ph((n >> 1) - 1))) break;  // output(n-2) read O
      tc_fence_after();
      if (elect_one_sync()) {
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_bf16(tmem + kColO + ob * kD, desc_add(qd, (kk >> 2) * kPanel + (kk & 3) * 32),
                   desc_add(sd, kk * 2048), kIdQS, kk > 0);
      }
      __syncwarp();
      if (!wait_w(kVFull, ph(c))) break;
      tc_fence_after();
      if (elect_one_sync()) {
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_bf16(tmem + kColS, desc_add(ktd, kk * 2048), desc_add(vd, kk * 2048), kIdKV, 1);
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_bf16(tmem + kColS, desc_add(ktld, kk * 2048), desc_add(vd, kk * 2048), kIdKV, 1);
        mma_commit(&bars[kSFull]);    // S complete; S' no longer read
        mma_commit(&bars[kQKEmpty]);  // Q', Kt hi and lo no longer read
      }
      __syncwarp();
      if (!wait_w(kPFull0 + ob, ph(n >> 1))) break;
      tc_fence_after();
      const uint32_t a_p = tmem + kColA;
      if (elect_one_sync()) {
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_bf16_tmem_a(tmem + kColO + ob * kD, a_p + 8 * kk, desc_add(vd, kk * 2048), kIdPV, 1);
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_bf16_tmem_a(tmem + kColO + ob * kD, a_p + 64 + 8 * kk, desc_add(vd, kk * 2048),
                          kIdPV, 1);
        mma_commit(&bars[kOFull0 + ob]);
        mma_commit(&bars[kVEmpty]);  // V no longer read
      }
      __syncwarp();
      ++n;
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ mask group
    const int q4 = warp & 3;
    const int r = 32 * q4 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
    const float scale = p.scale;
    // q . (aug * k) of this thread's token row from the scaled tiles: Q' (bf16)
    // times Kt hi + lo, 128 channels in 16-byte groups
    auto aug_dot = [&]() -> float {
      const float* ah = p.aug + (size_t)h * kD;
      float acc = 0.f;
#pragma unroll 1
      for (int pn = 0; pn < 2; ++pn) {
#pragma unroll
        for (int ci = 0; ci < 8; ++ci) {
          const uint32_t o = pn * kPanel + sw128_offset(r, ci);
          const uint4 qv = *reinterpret_cast<const uint4*>(smem + kOffQ + o);
          const uint4 kh = *reinterpret_cast<const uint4*>(smem + kOffK + o);
          const uint4 kl = *reinterpret_cast<const uint4*>(smem + kOffKlo + o);
          const float4 a0 = __ldg(reinterpret_cast<const float4*>(ah + 64 * pn + 8 * ci));
          const float4 a1 = __ldg(reinterpret_cast<const float4*>(ah + 64 * pn + 8 * ci + 4));
          const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
          const uint32_t hw[4] = {kh.x, kh.y, kh.z, kh.w};
          const uint32_t lw[4] = {kl.x, kl.y, kl.z, kl.w};
          const float aw[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            acc = fmaf(bf16lo(qw[e]) * aw[2 * e], bf16lo(hw[e]) + bf16lo(lw[e]), acc);
            acc = fmaf(bf16hi(qw[e]) * aw[2 * e + 1], bf16hi(hw[e]) + bf16hi(lw[e]), acc);
          }
        }
      }
      return acc;
    };
    // the mixer's row steps for 16 columns of the output: head RMSNorm weight
    // (rstd already applied) and the SiLU output gate
    auto mix_cols = [&](float (&o)[16], int col0, bool gate, const uint4 z0, const uint4 z1) {
      if (p.norm_w) {
        const float4* w4 = reinterpret_cast<const float4*>(p.norm_w + (size_t)h * kD + col0);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float4 w = __ldg(w4 + j);
          o[4 * j] *= w.x; o[4 * j + 1] *= w.y; o[4 * j + 2] *= w.z; o[4 * j + 3] *= w.w;
        }
      }
      if (gate) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const uint4 zz = j == 0 ? z0 : z1;
          const uint32_t zw[4] = {zz.x, zz.y, zz.z, zz.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float z0 = bf16lo(zw[e]), z1 = bf16hi(zw[e]);
            o[8 * j + 2 * e] *= siluf_(z0);
            o[8 * j + 2 * e + 1] *= siluf_(z1);
          }
        }
      }
    };
    auto output = [&](int c, int n) -> bool {
      const int ob = n & 1;
      const int nrows = min(kC, len - c * kC);
      const long long tok = (long long)c * kC + r;  // stored only while r < nrows
      const long long orow = start + (p.out_reversed ? len - 1 - tok : tok);
      const size_t off = ((size_t)orow * p.H + h) * kD;
      // with the mixer: the gate's whole z row is requested first (its latency
      // overlaps the wait for O and the RMS pass), then the row's RMS over all
      // 128 columns (a first pass over O)
      const bool gate = MIX && p.z != nullptr && r < nrows;
      uint4 zq[MIX ? kD / 8 : 1];
      if constexpr (MIX) {
#pragma unroll
        for (int j = 0; j < kD / 8; ++j)
          zq[j] = gate ? __ldg(reinterpret_cast<const uint4*>(p.z + off) + j)
                       : make_uint4(0u, 0u, 0u, 0u);
      }
      if (!wait_w(kOFull0 + ob, ph(n >> 1))) return false;
      tc_fence_after();
      float rstd = 1.f;
      if constexpr (MIX) {
        if (p.norm_w) {
          float ss = 0.f;
#pragma unroll 1
          for (int part = 0; part < kD / 16; ++part) {
            uint32_t v[16];
            tmem_ld_32x32b_x16(tmem + lane_off + kColO + ob * kD + 16 * part, v);
            tmem_ld_wait_x16(v);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float o = scale * __uint_as_float(v[j]);
              ss = fmaf(o, o, ss);
            }
          }
          rstd = rsqrtf(ss * (1.f / kD) + p.eps);
        }
      }
      auto store_part = [&](int part, const uint4 z0, const uint4 z1) {
        uint32_t v[16];
        tmem_ld_32x32b_x16(tmem + lane_off + kColO + ob * kD + 16 * part, v);
        tmem_ld_wait_x16(v);
        if (part == kD / 16 - 1) {
          tc_fence_before();
          warp_arrive(kOFree0 + ob);
        }
        float o[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) o[j] = scale * rstd * __uint_as_float(v[j]);
        if constexpr (MIX) mix_cols(o, 16 * part, gate, z0, z1);
        if (r < nrows) {
          if constexpr (OUTF32) {
            float* dst = static_cast<float*>(p.out) + off + 16 * part;
            if (p.out_v8) {
#pragma unroll
              for (int j = 0; j < 2; ++j)
                st_global_v8(dst + 8 * j, __float_as_uint(o[8 * j]), __float_as_uint(o[8 * j + 1]),
                             __float_as_uint(o[8 * j + 2]), __float_as_uint(o[8 * j + 3]),
                             __float_as_uint(o[8 * j + 4]), __float_as_uint(o[8 * j + 5]),
                             __float_as_uint(o[8 * j + 6]), __float_as_uint(o[8 * j + 7]));
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                reinterpret_cast<float4*>(dst)[j] =
                    make_float4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
            }
          } else {
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + off + 16 * part;
            uint32_t w[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) w[j] = pack_bf16x2(o[2 * j], o[2 * j + 1]);
            if (p.out_v8) {
              st_global_v8(dst, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
            } else {
              reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
              reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
            }
          }
        }
      };
      if constexpr (MIX) {
        // unrolled, so that the z words stay in registers
#pragma unroll
        for (int part = 0; part < kD / 16; ++part) store_part(part, zq[2 * part], zq[2 * part + 1]);
      } else {
#pragma unroll 1
        for (int part = 0; part < kD / 16; ++part)
          store_part(part, make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u));
      }
      return true;
    };
    // iteration c: P' of chunk c (tensor-core chunks), then the output of the
    // previous tensor-core chunk
    int n = 0, pending_c = -1;
    for (int c = 0; c <= nch; ++c) {
      bool tc = false;
      if (c < nch) {
        if (!wait_w(kScaled0 + (c & 1), ph(c >> 1))) break;
        tc = wide_ring[c & 3] == 0;
        warp_arrive(kAck0 + (c & 1));
        float diag_add = 0.f;
        if constexpr (MIX) {
          // self-augmentation: sigmoid(q . (aug * k)) v enters through P''s
          // diagonal (o = scale (Q' S' + P' V)); q_i k_i = Q'_i Kt_i, the decay
          // factors cancel within a token
          if (tc && p.aug) diag_add = sigmoidf_(aug_dot()) / scale;
          warp_arrive(kQKEmpty);  // done with this chunk's Q' and Kt rows
          if (tc && p.z) {
            const long long tok = (long long)c * kC + r;
            if (r < min(kC, len - c * kC)) {
              const long long orow = start + (p.out_reversed ? len - 1 - tok : tok);
              const __nv_bfloat16* zr = p.z + ((size_t)orow * p.H + h) * kD;
              prefetch_l2(zr);
              prefetch_l2(zr + 64);
            }
          }
        }
        if (tc) {
          if (!wait_w(kAFull, ph(n))) break;
          tc_fence_after();
          build_p(tmem + lane_off + kColA, q4, r, diag_add);
          tmem_st_wait();
          tc_fence_before();
          warp_arrive(kPFull0 + (n & 1));
        }
      }
      if (pending_c >= 0 && !output(pending_c, n - 1)) break;
      pending_c = -1;
      if (tc) {
        pending_c = c;
        ++n;
      }
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------ gate group
    const int gw = warp - 8;
    // gate pass mapping: channel pair pr (channels 2 pr, 2 pr + 1), tokens
    // 32 rg .. 32 rg + 31
    const int pr = 32 * (gw & 1) + lane;
    const int rg = gw >> 1;
    // state mapping: row i (TMEM lane quadrant = warp % 4), columns 64 hf ..
    const int q4 = warp & 3;
    const int hf = gw >> 2;
    const int si = 32 * q4 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
    const size_t st_off =
        (((size_t)s * p.H + h) * kD + (size_t)si) * kD + (size_t)(64 * hf);
    uint8_t* sb = smem + kOffSb;
    const float* init_row = p.init_state ? p.init_state + st_off : nullptr;
    float* final_row = p.final_state ? p.final_state + st_off : nullptr;

    // barrier of the gate group: an mbarrier with a bounded wait, so a group
    // that is aborting cannot hang the others
    int gk = 0;
    auto group_sync = [&]() -> bool {
      warp_arrive(kGateSync);
      return wait_w(kGateSync, ph(gk++));
    };

    // S rows of this thread (64 columns) between TMEM and registers
    auto s_load = [&](float (&sv)[64], bool from_init) {
      if (from_init) {
#pragma unroll
        for (int j = 0; j < 64; j += 4) {
          const float4 x = init_row ? __ldg(reinterpret_cast<const float4*>(init_row + j))
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
          sv[j] = x.x; sv[j + 1] = x.y; sv[j + 2] = x.z; sv[j + 3] = x.w;
        }
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t v[16];
          tmem_ld_32x32b_x16(tmem + lane_off + kColS + 64 * hf + 16 * q, v);
          tmem_ld_wait_x16(v);
#pragma unroll
          for (int j = 0; j < 16; ++j) sv[16 * q + j] = __uint_as_float(v[j]);
        }
      }
    };
    auto s_store = [&](const float (&sv)[64]) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = __float_as_uint(sv[16 * q + j]);
        tmem_st_32x32b_x16(tmem + lane_off + kColS + 64 * hf + 16 * q, v);
      }
      tmem_st_wait();
    };

    // A wide chunk, token by token: S <- diag(exp g_t) S + k_t^T v_t, o_t = scale q_t S.
    // Row sums over the 128 state rows: a butterfly over the warp's 32 rows,
    // then the four row-quadrant warps through shared memory (the Kt lo tile
    // is free in a wide chunk).
    auto wide_chunk = [&](int c, float (&sv)[64]) -> bool {
      const int nrows = min(kC, len - c * kC);
      float* red = reinterpret_cast<float*>(smem + kOffKlo);  // [2][4][128]
      const uint8_t* qs = smem + kOffQ;
      const uint8_t* ks = smem + kOffK;
      const uint8_t* vs = smem + kOffV + hf * kPanel;
#pragma unroll 1
      for (int t = 0; t < nrows; ++t) {
        const float gi = fmaxf(gsm[t * kD + si], -kGateClamp);
        const float a = exp2f(gi * kLog2e);
        const uint32_t eoff = (si >> 6) * kPanel + sw128_offset(t, (si & 63) >> 3) + (si & 7) * 2;
        const float kv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(ks + eoff));
        const float qv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(qs + eoff));
        float* rb = red + (t & 1) * 4 * kD;
        // 32 columns at a time: update S, multiply by q, then reduce-scatter
        // the products over the warp's 32 rows (lane l ends with column l)
#pragma unroll
        for (int grp = 0; grp < 2; ++grp) {
          float pv[32];
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            const uint4 raw = *reinterpret_cast<const uint4*>(vs + sw128_offset(t, 4 * grp + cc));
            const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int j = 8 * cc + 2 * e;
              float& s0 = sv[32 * grp + j];
              float& s1 = sv[32 * grp + j + 1];
              s0 = fmaf(a, s0, kv * bf16lo(w4[e]));
              s1 = fmaf(a, s1, kv * bf16hi(w4[e]));
              pv[j] = qv * s0;
              pv[j + 1] = qv * s1;
            }
          }
#pragma unroll
          for (int rd = 0; rd < 5; ++rd) {
            const int keep_n = 16 >> rd;
            const int bit = 16 >> rd;
            const bool upper = (lane & bit) != 0;
#pragma unroll
            for (int x = 0; x < 16; ++x) {
              if (x < keep_n) {
                const float send = upper ? pv[x] : pv[x + keep_n];
                const float keep = upper ? pv[x + keep_n] : pv[x];
                pv[x] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
              }
            }
          }
          rb[q4 * kD + 64 * hf + 32 * grp + lane] = pv[0];
        }
        if (!group_sync()) return false;
        if (q4 == 0) {
          const long long tok = (long long)c * kC + t;
          const long long orow = start + (p.out_reversed ? len - 1 - tok : tok);
          float ov[2];
#pragma unroll
          for (int grp = 0; grp < 2; ++grp) {
            const int col = 64 * hf + 32 * grp + lane;
            float o = 0.f;
#pragma unroll
            for (int w = 0; w < 4; ++w) o += rb[w * kD + col];
            ov[grp] = o * p.scale;
          }
          if constexpr (MIX) {
            // the mixer's steps on this token: both warps of the row quadrant
            // recompute what needs all 128 columns (the augmentation dot and
            // the RMS) from the same shared data, so they agree exactly
            const uint8_t* vall = smem + kOffV;
            auto elem = [&](const uint8_t* tile, int ch) -> float {  // bf16 (t, ch)
              const uint32_t eo = (ch >> 6) * kPanel + sw128_offset(t, (ch & 63) >> 3) + (ch & 7) * 2;
              return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(tile + eo));
            };
            float sg = 0.f;
            if (p.aug) {
              float sa = 0.f;
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int ch = 4 * lane + i;
                sa = fmaf(elem(qs, ch) * __ldg(p.aug + (size_t)h * kD + ch), elem(ks, ch), sa);
              }
#pragma unroll
              for (int m = 16; m >= 1; m >>= 1) sa += __shfl_xor_sync(0xffffffffu, sa, m);
              sg = sigmoidf_(sa);
#pragma unroll
              for (int grp = 0; grp < 2; ++grp) ov[grp] += sg * elem(vall, 64 * hf + 32 * grp + lane);
            }
            float rs = 1.f;
            if (p.norm_w) {
              float ss = 0.f;
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int col = 32 * i + lane;
                float o = 0.f;
#pragma unroll
                for (int w = 0; w < 4; ++w) o += rb[w * kD + col];
                o = o * p.scale + sg * (p.aug ? elem(vall, col) : 0.f);
                ss = fmaf(o, o, ss);
              }
#pragma unroll
              for (int m = 16; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
              rs = rsqrtf(ss * (1.f / kD) + p.eps);
            }
#pragma unroll
            for (int grp = 0; grp < 2; ++grp) {
              const int col = 64 * hf + 32 * grp + lane;
              ov[grp] *= rs;
              if (p.norm_w) ov[grp] *= __ldg(p.norm_w + (size_t)h * kD + col);
              if (p.z) {
                const float zv =
                    __bfloat162float(p.z[((size_t)orow * p.H + h) * kD + col]);
                ov[grp] *= siluf_(zv);
              }
            }
          }
#pragma unroll
          for (int grp = 0; grp < 2; ++grp) {
            const int col = 64 * hf + 32 * grp + lane;
            const size_t off = ((size_t)orow * p.H + h) * kD + col;
            if constexpr (OUTF32)
              static_cast<float*>(p.out)[off] = ov[grp];
            else
              static_cast<__nv_bfloat16*>(p.out)[off] = __float2bfloat16_rn(ov[grp]);
          }
        }
      }
      return true;
    };

    int n = 0;           // tensor-core chunks so far
    bool s_in_tmem = false;  // S lives in TMEM (else: the initial state in global memory)
    bool last_tc = false;    // the latest S update was an MMA4 (wait for SFull)
    bool ok = true;
    for (int c = 0; c < nch && ok; ++c) {
      const int nrows = min(kC, len - c * kC);
      if (!wait_w(kGFull, ph(c))) { ok = false; break; }
      // pass 1: this thread's partial sums of g (two channels, 32 tokens)
      float sum0 = 0.f, sum1 = 0.f;
#pragma unroll 8
      for (int t = 32 * rg; t < 32 * rg + 32; ++t) {
        if (t < nrows) {
          const float2 gv = *reinterpret_cast<const float2*>(gsm + t * kD + 2 * pr);
          sum0 += fmaxf(gv.x, -kGateClamp);
          sum1 += fmaxf(gv.y, -kGateClamp);
        }
      }
      part[rg * kD + 2 * pr] = sum0;
      part[rg * kD + 2 * pr + 1] = sum1;
      if (!group_sync()) { ok = false; break; }
      float off0 = 0.f, off1 = 0.f, tot0 = 0.f, tot1 = 0.f;
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const float a0 = part[x * kD + 2 * pr], a1 = part[x * kD + 2 * pr + 1];
        if (x < rg) { off0 += a0; off1 += a1; }
        tot0 += a0;
        tot1 += a1;
      }
      // per-channel totals for the state pass (row si), read before the
      // partials are rewritten (the next write follows two more barriers)
      float totr = 0.f;
#pragma unroll
      for (int x = 0; x < 4; ++x) totr += part[x * kD + si];
      const float GL0 = tot0 * kLog2e, GL1 = tot1 * kLog2e;
      // wide: some channel's decay over the chunk exceeds 2^-100
      if (-GL0 > kWideSpan || -GL1 > kWideSpan) atomicOr(&vote[c & 1], 1);
      if (!group_sync()) { ok = false; break; }
      const bool wide = *reinterpret_cast<volatile int*>(&vote[c & 1]) != 0;
      // the consumers have read the flags of chunk c - 2: its ring entry and
      // its parity's phase of the chunk barrier may be reused
      if (c >= 2 && !wait_w(kAck0 + (c & 1), ph((c - 2) >> 1))) { ok = false; break; }
      if (tid == 256) wide_ring[c & 3] = wide ? 1 : 0;
      if (!wide) {
        // state pass first: S <- diag(exp G_L) S in TMEM, S' = its bf16 copy.  It
        // needs only the previous chunk's MMA4, so it runs while Q and K land.
        if (last_tc && !wait_w(kSFull, ph(n - 1))) { ok = false; break; }
        tc_fence_after();
        float sv[64];
        s_load(sv, !s_in_tmem);
        const float dec = exp2f(totr * kLog2e);
#pragma unroll
        for (int j = 0; j < 64; ++j) sv[j] *= dec;
        s_store(sv);
#pragma unroll
        for (int cc = 0; cc < 8; ++cc)
          *reinterpret_cast<uint4*>(sb + hf * kPanel + sw128_offset(si, cc)) =
              make_uint4(pack_bf16x2(sv[8 * cc], sv[8 * cc + 1]),
                         pack_bf16x2(sv[8 * cc + 2], sv[8 * cc + 3]),
                         pack_bf16x2(sv[8 * cc + 4], sv[8 * cc + 5]),
                         pack_bf16x2(sv[8 * cc + 6], sv[8 * cc + 7]));
        fence_proxy_async_smem();
        tc_fence_before();
        warp_arrive(kSbReady);
        if (!wait_w(kQKFull, ph(c))) { ok = false; break; }
        // pass 2: Q' = q exp(G - G_L) in place, Kt = k exp(G_L - G) as hi (in
        // place) + lo; rows past the sequence end are zeroed
        float G0 = off0 * kLog2e, G1 = off1 * kLog2e;
#pragma unroll 8
        for (int t = 32 * rg; t < 32 * rg + 32; ++t) {
          const uint32_t eo = pair_offset(t, pr);
          uint32_t qo = 0u, kh = 0u, kl = 0u;
          if (t < nrows) {
            const float2 gv = *reinterpret_cast<const float2*>(gsm + t * kD + 2 * pr);
            G0 += fmaxf(gv.x, -kGateClamp) * kLog2e;
            G1 += fmaxf(gv.y, -kGateClamp) * kLog2e;
            const uint32_t qraw = *reinterpret_cast<const uint32_t*>(smem + kOffQ + eo);
            const uint32_t kraw = *reinterpret_cast<const uint32_t*>(smem + kOffK + eo);
            qo = pack_bf16x2(bf16lo(qraw) * ex2_(G0 - GL0), bf16hi(qraw) * ex2_(G1 - GL1));
            const float k0 = bf16lo(kraw) * ex2_(GL0 - G0), k1 = bf16hi(kraw) * ex2_(GL1 - G1);
            kh = pack_bf16x2(k0, k1);
            kl = pack_bf16x2(k0 - bf16lo(kh), k1 - bf16hi(kh));
          }
          *reinterpret_cast<uint32_t*>(smem + kOffQ + eo) = qo;
          *reinterpret_cast<uint32_t*>(smem + kOffK + eo) = kh;
          *reinterpret_cast<uint32_t*>(smem + kOffKlo + eo) = kl;
        }
        fence_proxy_async_smem();
        if (!group_sync()) { ok = false; break; }  // every thread is done with g
        if (tid == 256) {
          mbar_arrive(&bars[kGEmpty]);
          vote[c & 1] = 0;  // read by all before the last barrier; next used by chunk c + 2
        }
        warp_arrive(kScaled0 + (c & 1));
        s_in_tmem = true;
        last_tc = true;
        ++n;
      } else {
        if (!wait_w(kQKFull, ph(c))) { ok = false; break; }
        warp_arrive(kScaled0 + (c & 1));
        if (last_tc && !wait_w(kSFull, ph(n - 1))) { ok = false; break; }
        if (!wait_w(kVFull, ph(c))) { ok = false; break; }
        tc_fence_after();
        float sv[64];
        s_load(sv, !s_in_tmem);
        if (!wide_chunk(c, sv)) { ok = false; break; }
        s_store(sv);
        tc_fence_before();
        if (!group_sync()) { ok = false; break; }  // every thread is done with g, Q, K, V
        if (tid == 256) {
          mbar_arrive(&bars[kGEmpty]);
          mbar_arrive(&bars[kQKEmpty]);
          mbar_arrive(&bars[kVEmpty]);
          vote[c & 1] = 0;
        }
        s_in_tmem = true;
        last_tc = false;
      }
    }
    // the final state
    if (ok && !*abort_flag) {
      if (last_tc && !wait_w(kSFull, ph(n - 1))) ok = false;
      if (ok && final_row) {
        tc_fence_after();
        float sv[64];
        s_load(sv, !s_in_tmem);
#pragma unroll
        for (int j = 0; j < 64; j += 4)
          *reinterpret_cast<float4*>(final_row + j) = make_float4(sv[j], sv[j + 1], sv[j + 2], sv[j + 3]);
      }
    }
  }

  // Teardown, also after an abort: every copy into this CTA's shared memory and
  // every MMA (with its commits' barrier arrivals) lands before the CTA ends.
  if (warp == 0 && lane == 0) {
    if (issued_g > 0) (void)mbar_wait_bounded(&bars[kGFull], (issued_g - 1) & 1, kWaitLimitNs);
    if (issued_qk > 0) (void)mbar_wait_bounded(&bars[kQKFull], (issued_qk - 1) & 1, kWaitLimitNs);
    if (issued_v > 0) (void)mbar_wait_bounded(&bars[kVFull], (issued_v - 1) & 1, kWaitLimitNs);
  }
  if (warp == 1 && mma_issued) {
    // the lane that issued the MMAs commits them to the drain barrier
    if (elect_one_sync()) mma_commit(&bars[kDrain]);
    __syncwarp();
    (void)mbar_wait_bounded(&bars[kDrain], 0u, kWaitLimitNs);
  }
  if (__any_sync(0xffffffffu, *abort_flag != 0)) {
    // a role that gave up may have left tensor-memory accesses unwaited
    tmem_ld_wait();
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// [nb][rows][H][d] viewed as 4-D {d, H, rows, nb}: bf16 tiles of 128 rows x 64
// columns (128-byte swizzle), or fp32 tiles of 128 rows x 128 columns (no swizzle).
bool make_map(CUtensorMap* map, const void* base, bool fp32, int d, int H, long long rows, int nb) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t es = fp32 ? 4 : 2;
  const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)rows, (cuuint64_t)nb};
  const cuuint64_t strides[3] = {(cuuint64_t)d * es, (cuuint64_t)H * d * es,
                                 (cuuint64_t)rows * H * d * es};
  const cuuint32_t box[4] = {fp32 ? (cuuint32_t)kD : 64u, 1, (cuuint32_t)kC, 1};
  const cuuint32_t el[4] = {1, 1, 1, 1};
  return fn(map, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
            const_cast<void*>(base), dims, strides, box, el, CU_TENSOR_MAP_INTERLEAVE_NONE,
            fp32 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool chunk_tc_vec_supported(const ChunkArgs& a) {
  return !a.fp32_io && a.vector_gate && a.chunk == kC && a.dk == kD && a.dv == kD;
}

cudaError_t launch_chunk_tc_vec(const ChunkArgs& a, cudaStream_t stream, const EpilogueArgs* mix) {
  const bool packed = a.cu_seqlens != nullptr;
  const long long rows = a.T;
  const int nb = packed ? 1 : a.B;
  CUtensorMap mq, mk, mv, mg;
  if (!make_map(&mq, a.q, false, a.dk, a.H, rows, nb) ||
      !make_map(&mk, a.k, false, a.dk, a.H, rows, nb) ||
      !make_map(&mv, a.v, false, a.dv, a.H, rows, nb) ||
      !make_map(&mg, a.g, true, a.dk, a.H, rows, nb))
    return cudaErrorInvalidValue;
  VecParams p;
  p.scale = a.scale; p.init_state = a.init_state; p.out = a.out;
  p.final_state = a.final_state; p.cu_seqlens = a.cu_seqlens;
  p.B = a.B; p.H = a.H; p.T = a.T; p.status = a.status;
  p.wait_ns = handoff_wait_limit_ns();
  p.out_v8 = (reinterpret_cast<uintptr_t>(a.out) & 31) == 0;
  p.out_reversed = a.out_reversed;
  p.aug = mix ? mix->aug : nullptr;
  p.norm_w = mix ? mix->norm_w : nullptr;
  p.eps = mix ? mix->eps : 0.f;
  p.z = mix ? static_cast<const __nv_bfloat16*>(mix->z) : nullptr;
  const long long ctas = (long long)a.B * a.H;
  auto launch = [&](auto kern) -> cudaError_t {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)ctas, kThreads, kSmemBytes, stream>>>(mq, mk, mv, mg, p);
    return cudaGetLastError();
  };
  if (a.fp32_out)
    return mix ? launch(chunk_tc_vec_kernel<true, true>) : launch(chunk_tc_vec_kernel<true, false>);
  return mix ? launch(chunk_tc_vec_kernel<false, true>) : launch(chunk_tc_vec_kernel<false, false>);
}

}  // namespace gla
