// gla_chunk_tc.cu -- chunked GLA prefill on the 5th-generation tensor cores.
//
// Method: the chunked form of the "i14 Laplace 3B on AWS Trainium2" page
// (section "Challenge 1", Figure 3) with per-token log-decays g.  For a chunk
// of C = 128 tokens, G_t = the sum of g over the chunk up to and including t
// (log2 units) and L the chunk's last token:
//     U      = K^T (W V),            W_j = 2^{G_L - G_j}  (<= 1)
//     S_c    = 2^{G_L} S_{c-1} + U
//     o_t    = scale * 2^{G_t - G_L} * ( Q S' + P' V )_t,   S' = 2^{G_L} S_{c-1},
//     P'_tj  = (Q K^T)_tj W_j   for j <= t (causal mask, diagonal kept),
// exact while the chunk's decay span 2^{G_0 - G_L} stays inside 2^96; a wider
// ("wide") chunk takes the explicit form
//     o_t    = scale * ( 2^{G_t} (Q S_{c-1})_t + sum_{j<=t} (Q K^T)_tj 2^{G_t - G_j} V_j ).
//
// Precision: every operand is either exact in bf16 (Q, K, V) or split into a
// bf16 hi part and a bf16 lo part (the rest) that both enter the contraction:
// W V (state update), S' (inter-chunk readout) and P' (intra-chunk readout).
// What remains is fp32 accumulation.  (With S' rounded once to bf16, heads
// whose state decays slowly -- the fixed schedule's last heads -- lose about
// 2 % of the output's RMS; with hi + lo they keep about 1e-3.)
//
// One CTA owns one (sequence, head, 64-wide slice of dv) and walks the chunks
// in order.  The chain that makes a chunk wait for the previous one is cut to
// its arithmetic core: the chunk's own update U = K^T (W V) goes into a TMEM
// accumulator of its own (double-buffered), independent of the state, and the
// state itself lives in registers of the state group, S <- 2^{G_L} S + U.
// Five tcgen05 contractions per chunk, bf16 x bf16 -> fp32 in TMEM:
//     MMA1  A   = Q K^T                  M=128 (t)  N=128 (j)  K=dk   issuer A
//     MMA4  U   = K^T (W V)hi + lo       M=128 (i)  N=64       K=128  issuer C
//     MMA3  O   = Q S'hi + Q S'lo        M=128 (t)  N=64       K=dk   issuer B
//     MMA2  O  += P'hi V + P'lo V        M=128 (t)  N=64       K=128  issuer B (A in TMEM)
// Each issuer waits only for its own operands.
//
// Roles (16 warps):
//   warp 0       producer: the TMA loads of a 2-stage Q/K ring and a 2-buffer
//                V ring (lane 0; the first two chunks' before anything else),
//                prefix sums of g and the chunk's flags (all lanes)
//   warp 1       issuer A (MMA1), TMEM allocation
//   warp 2       issuer B (MMA3, then MMA2)
//   warp 3       issuer C (MMA4)
//   warps 4..7   mask group: P' of chunk c from A (thread = token row; hi and
//                lo written in place over each 32-column block of A), then the
//                output of chunk c - 1
//   warps 8..15  state group: the W V split of chunk c + 1, then the state
//                step S_c = 2^{G_L} S_{c-1} + U_c (registers) and S'_c (bf16
//                hi + lo) for chunk c + 1, or the final state; two warps per
//                TMEM lane quadrant, 32 of the 64 columns each
// TMEM: A/P' 2 x 128 (chunk parity), O 2 x 64, U 2 x 64 = 512 columns.
// Shared memory: the gate ring and barriers first, then from 3 KB on the
// 1024-aligned tiles: Q/K ring 2 x 64 KB, V 2 x 16 KB, (W V) hi/lo 32 KB,
// S' hi/lo 32 KB -- 227 KB.  Every mbarrier wait is bounded in wall time; on
// timeout the kernel flags the device status word, stops issuing work, lets
// its copies and contractions land, releases TMEM and returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "gla_internal.cuh"
#include "gla_sm100.cuh"

// Timing probes: a build may define GLA_TRACE_POINT(kernel, event, iteration)
// to record when roles pass their hand-offs; by default it is nothing.
#ifndef GLA_TRACE_POINT
#define GLA_TRACE_POINT(kern, ev, it) ((void)0)
#endif

namespace gla {
namespace {

using namespace sm100;

constexpr int kC = 128;        // chunk (tokens)
constexpr int kDK = 128;       // key head size of the tiles (d_k = 64, 96 run zero-padded)
constexpr int kDVS = 64;       // value columns per CTA
constexpr int kThreads = 512;  // 16 warps
constexpr int kMaskWarps = 4;
constexpr int kStateWarps = 8;
constexpr uint64_t kWaitLimitNs = kDefaultWaitLimitNs;  // the drains' limit (2 s)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kWideSpan = 96.f;      // log2 chunk decay span above which a chunk is "wide"
constexpr int kSlots = 3;              // gate ring: chunks c (mask), c + 1 (state), c + 2

// shared memory map: small state first, tiles from the first 1024-byte boundary
// gate slot (floats): arr[128] (W_j on a plain chunk, G_j on a wide one) | total, wide
constexpr int kSlotFloats = 132;
constexpr uint32_t kOffGate = 0;
constexpr uint32_t kOffBar = kOffGate + kSlots * kSlotFloats * 4;
constexpr uint32_t kBarBytes = 320;
constexpr uint32_t kOffMisc = kOffBar + kBarBytes;  // tmem base, abort flag
constexpr uint32_t kOffTiles = (kOffMisc + 16 + 1023) & ~1023u;
constexpr uint32_t kPanel = kC * 128;                  // 128 rows x 128 B
constexpr uint32_t kQBytes = kPanel * (kDK / 64);      // 32 KB
constexpr uint32_t kQKStage = 2 * kQBytes;             // 64 KB
constexpr uint32_t kTile = kPanel;                     // 16 KB: 128 rows x 64 columns bf16
constexpr uint32_t kOffQK = kOffTiles;                 // 2 stages
constexpr uint32_t kOffV = kOffQK + 2 * kQKStage;      // 2 buffers
constexpr uint32_t kOffWVhi = kOffV + 2 * kTile;
constexpr uint32_t kOffWVlo = kOffWVhi + kTile;
constexpr uint32_t kOffShi = kOffWVlo + kTile;         // dk rows x 128 B
constexpr uint32_t kOffSlo = kOffShi + kTile;
constexpr uint32_t kSmemBytes = kOffSlo + kTile;
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffBar % 8 == 0 && kOffTiles % 1024 == 0, "alignment");

// TMEM column map
constexpr uint32_t kColA = 0;      // 2 x 128: A = Q K^T (fp32), then P' (bf16 hi / lo) in place
constexpr uint32_t kColO = 256;    // 2 x 64: O = Q S' + P' V, per chunk parity
constexpr uint32_t kColU = 384;    // 2 x 64: U = K^T (W V), per chunk parity
constexpr uint32_t kTmemCols = 512;

enum Bar {
  kQKFull0 = 0, kQKEmpty0 = 2, kVFull0 = 4, kVEmpty0 = 6, kAFull0 = 8, kAFree0 = 10,
  kPFull0 = 12, kO3Full0 = 14, kOFull0 = 16, kOFree0 = 18, kUFull0 = 20, kUFree0 = 22,
  kVtFull = 24, kVtFree, kSReady, kSFree, kGReady0, kGFree0 = kGReady0 + kSlots,
  kDrain = kGFree0 + kSlots, kNumBars = kDrain + 3
};
static_assert(kNumBars * 8 <= kBarBytes, "barrier area");

constexpr uint32_t kIdQK = idesc_bf16(128, 128, false, false);
constexpr uint32_t kIdQS = idesc_bf16(128, kDVS, false, true);
constexpr uint32_t kIdKV = idesc_bf16(kDK, kDVS, true, true);
constexpr uint32_t kIdPV = idesc_bf16(128, kDVS, false, true);

struct TcParams {
  const float* g;
  float scale;
  const float* init_state;
  void* out;
  float* final_state;
  const int32_t* cu_seqlens;
  int B, H, T, DK, DV, nslices;  // DK = 64, 96 run as 128 with zero channels DK..127
  int out_v8;        // out is 32-byte aligned: 256-bit stores
  int out_reversed;  // token t of a sequence stored at row len - 1 - t
  // DOT kernels: dot_out[row, h] += dot_sign * (out row . dot_rows row), the
  // fp32 output against a bf16 tensor of the output's layout
  const __nv_bfloat16* dot_rows;
  float* dot_out;
  float dot_sign;
  unsigned* status;
  uint64_t wait_ns;  // limit of the hand-off waits (the drain keeps kWaitLimitNs)
};

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }
__device__ __forceinline__ uint32_t ph(int k) { return static_cast<uint32_t>(k) & 1u; }

// Bounded mbarrier wait that also gives up once the CTA is aborting: one
// inline test, then an out-of-line loop (kept out of line to keep the
// kernel's code small).
__device__ __noinline__ bool wait_bar_slow(uint64_t* bar, uint32_t parity,
                                           volatile int* abort_flag, unsigned* status,
                                           uint64_t limit_ns) {
  if (*abort_flag) return false;
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      atomicOr(status, kDevTimeout);
      return false;
    }
  }
}
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity,
                                         volatile int* abort_flag, unsigned* status,
                                         uint64_t limit_ns) {
  if (!*abort_flag && mbar_try_wait(bar, parity)) return true;
  return wait_bar_slow(bar, parity, abort_flag, status, limit_ns);
}

// Teardown: wait (bounded) until the last of `issued` transactions counted on
// `bar` has landed, so that no copy into shared memory is in flight at exit.
__device__ __forceinline__ void drain_bar(uint64_t* bar, int issued) {
  if (issued > 0) (void)mbar_wait_bounded(bar, (uint32_t)(issued - 1) & 1u, kWaitLimitNs);
}

// P' of token row r from A = Q K^T in TMEM, in place: the fp32 32-column block
// cb (tokens j = 32 cb .. 32 cb + 31) becomes its bf16 hi pairs in columns
// 32 cb .. 32 cb + 15 and its lo pairs in 32 cb + 16 .. 32 cb + 31, so no block
// overwrites another before it is read.  Not WIDE: P'_rj = A_rj W_j on the
// causal part (W is zero past the chunk's last valid token); WIDE: the
// explicit decays 2^{G_r - G_j} for j <= r (arr holds G).  Blocks past the
// row's own are zero and never read.
template <bool WIDE>
__device__ __forceinline__ void build_p(uint32_t a_row, int q4, int r, float G2r,
                                        const float* arr) {
  uint32_t a[32];
  tmem_ld_32x32b_x32(a_row, a);
#pragma unroll 1
  for (int cb = 0; cb < 4; ++cb) {
    if (cb <= q4) {
      tmem_ld_wait_x32(a);
      const bool diag = cb == q4;
      const float4* w4 = reinterpret_cast<const float4*>(arr + 32 * cb);
      // half h: columns 16 h .. 16 h + 15 of the block -> hi pairs at 8 h, lo
      // pairs at 16 + 8 h (columns whose A values are already in registers);
      // then the next block's same half is loaded into the freed registers
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t hi[8], lo[8];
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4) {
          const int e = 16 * hf + 4 * e4;
          const float4 wv = w4[4 * hf + e4];
          const float wa[4] = {wv.x, wv.y, wv.z, wv.w};
          float x[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int j = 32 * cb + e + i;
            const float av = __uint_as_float(a[e + i]);
            if constexpr (WIDE) {
              x[i] = j <= r ? av * exp2f(G2r - wa[i]) : 0.f;
            } else {
              x[i] = (diag && j > r) ? 0.f : av * wa[i];
            }
          }
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const uint32_t h2 = pack_bf16x2(x[2 * i], x[2 * i + 1]);
            hi[2 * e4 + i] = h2;
            lo[2 * e4 + i] = pack_bf16x2(x[2 * i] - bf16lo(h2), x[2 * i + 1] - bf16hi(h2));
          }
        }
        if (cb < q4)
          tmem_ld_32x32b_x16(a_row + 32 * (cb + 1) + 16 * hf,
                             *reinterpret_cast<uint32_t(*)[16]>(a + 16 * hf));
        tmem_st_32x32b_x8(a_row + 32 * cb + 8 * hf, hi);
        tmem_st_32x32b_x8(a_row + 32 * cb + 16 + 8 * hf, lo);
      }
    } else {
      uint32_t z[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) z[e] = 0u;
      tmem_st_32x32b_x16(a_row + 32 * cb, z);
      tmem_st_32x32b_x16(a_row + 32 * cb + 16, z);
    }
  }
}

template <bool OUTF32, bool DOT>
__global__ void __launch_bounds__(kThreads, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const TcParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  // the tiles need 1024-byte alignment (128-byte swizzle) and the layout fills
  // the whole budget, so a window that does not start aligned is refused
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicOr(p.status, kDevLayout);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  float* gate_ring = reinterpret_cast<float*>(smem + kOffGate);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nsl = p.nslices;
  const int sl = blockIdx.x % nsl;
  const int h = (blockIdx.x / nsl) % p.H;
  const int s = blockIdx.x / (nsl * p.H);
  const int nks = p.DK / 16;  // k-steps over the key channels

  long long start;
  int len;
  // all threads agree (same s): either every thread returns here or none does
  if (!seq_bounds(p.cu_seqlens, s, p.B, p.T, &start, &len, p.status)) return;
  const int nch = (len + kC - 1) / kC;
  const bool packed = p.cu_seqlens != nullptr;

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      uint32_t cnt = 1;
      if (i == kPFull0 || i == kPFull0 + 1 || i == kOFree0 || i == kOFree0 + 1) cnt = kMaskWarps;
      if (i == kUFree0 || i == kUFree0 + 1 || i == kVtFull || i == kSReady) cnt = kStateWarps;
      // the three issuers each commit once they are done with a Q/K stage
      if (i == kQKEmpty0 || i == kQKEmpty0 + 1) cnt = 3;
      // a V buffer is free once MMA2 has run and the state group has split it
      if (i == kVEmpty0 || i == kVEmpty0 + 1) cnt = 1 + kStateWarps;
      if (i >= kGFree0 && i < kGFree0 + kSlots) cnt = kMaskWarps + kStateWarps;
      mbar_init(&bars[i], cnt);
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = __shfl_sync(0xffffffffu, *tmem_slot, 0);  // warp-uniform
  const uint32_t sbase = smem_u32(smem);
  if (tid == 0) GLA_TRACE_POINT(0, 30, 0);

  auto wait = [&](int b, uint32_t parity) -> bool {
    return wait_bar(&bars[b], parity, abort_flag, p.status, p.wait_ns);
  };
  auto wait_w = [&](int b, uint32_t parity) -> bool {
    return __all_sync(0xffffffffu, wait(b, parity));
  };
  // One arrival for the whole warp, after every lane's prior writes and fences
  // (__syncwarp orders them before lane 0's release-arrive).
  auto warp_arrive = [&](int b) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[b]);
  };
  auto slot_of = [&](int c) -> float* { return gate_ring + (c % kSlots) * kSlotFloats; };

  int issued_qk[2] = {0, 0}, issued_v[2] = {0, 0};
  bool mma_issued = false;

  if (warp == 0) {
    // ------------------------------------------- producer: gate sums and TMA
    // All lanes: prefix sums of g for chunk c (lane l owns tokens 4l .. 4l+3)
    // into the gate ring; lane 0: the TMA loads of chunk c.  The gate values
    // are read when their chunk comes up and prefetched into L2 three chunks
    // ahead.
    const int bidx = packed ? 0 : s;
    auto prefetch_gates = [&](int c) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int t = c * kC + 4 * lane + i;
        if (c < nch && t < len) prefetch_l2(p.g + (start + t) * p.H + h);
      }
    };
    // lane 0: the TMA loads of chunk c (after its ring stages are free)
    auto issue_loads = [&](int c) -> bool {
      const int st = c & 1;
      const int row = packed ? (int)(start + (long long)c * kC) : c * kC;
      if (c >= 2 && !wait(kQKEmpty0 + st, ph((c >> 1) - 1))) return false;
      uint8_t* q_s = smem + kOffQK + st * kQKStage;
      uint8_t* k_s = q_s + kQBytes;
      mbar_arrive_expect_tx(&bars[kQKFull0 + st], kQKStage);
#pragma unroll
      for (int pn = 0; pn < kDK / 64; ++pn) {
        tma_load_4d(q_s + pn * kPanel, &tmQ, &bars[kQKFull0 + st], pn * 64, h, row, bidx);
        tma_load_4d(k_s + pn * kPanel, &tmK, &bars[kQKFull0 + st], pn * 64, h, row, bidx);
      }
      ++issued_qk[st];
      GLA_TRACE_POINT(0, 1, c);
      if (c >= 2 && !wait(kVEmpty0 + st, ph((c >> 1) - 1))) return false;
      mbar_arrive_expect_tx(&bars[kVFull0 + st], kTile);
      tma_load_4d(smem + kOffV + st * kTile, &tmV, &bars[kVFull0 + st], sl * kDVS, h, row, bidx);
      ++issued_v[st];
      GLA_TRACE_POINT(0, 2, c);
      return true;
    };
    // the first two chunks' tiles need no free stage: start them before the gates
    if (lane == 0)
      for (int c = 0; c < 2 && c < nch; ++c) (void)issue_loads(c);
    for (int c = 0; c < 3; ++c) prefetch_gates(c);
    for (int c = 0; c < nch; ++c) {
      float gv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int t = c * kC + 4 * lane + i;
        gv[i] = t < len ? fmaxf(__ldg(p.g + (start + t) * p.H + h), -kGateClamp) : 0.f;
      }
      prefetch_gates(c + 3);
      bool ok = true;
      if (c >= kSlots && !wait(kGFree0 + c % kSlots, ph(c / kSlots - 1))) ok = false;
      if (__any_sync(0xffffffffu, !ok)) break;
      float run[4];
      run[0] = gv[0];
#pragma unroll
      for (int i = 1; i < 4; ++i) run[i] = run[i - 1] + gv[i];
      float incl = run[3];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
      }
      const float excl = incl - run[3];
      const float total = __shfl_sync(0xffffffffu, incl, 31) * kLog2e;
      float G2[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) G2[i] = (excl + run[i]) * kLog2e;
      const float first = __shfl_sync(0xffffffffu, G2[0], 0);
      const bool wide = first - total > kWideSpan;
      const int n = min(kC, len - c * kC);
      float arr[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        arr[i] = wide ? G2[i] : ((4 * lane + i < n) ? exp2f(total - G2[i]) : 0.f);
      float* slot = slot_of(c);
      *reinterpret_cast<float4*>(slot + 4 * lane) = make_float4(arr[0], arr[1], arr[2], arr[3]);
      if (lane == 0) {
        slot[128] = total;
        slot[129] = wide ? 1.f : 0.f;
      }
      warp_arrive(kGReady0 + c % kSlots);
      if (lane == 0) {
        GLA_TRACE_POINT(0, 0, c);
        if (c >= 2) ok = issue_loads(c);
      }
      if (__any_sync(0xffffffffu, !ok)) break;
    }
  } else if (warp == 1) {
    // ------------------------------------------------- issuer A: MMA1 A = Q K^T
    // (the whole warp waits and forms the descriptors; one lane issues)
    for (int c = 0; c < nch; ++c) {
      const int st = c & 1;
      if (!wait_w(kQKFull0 + st, ph(c >> 1))) break;
      if (c >= 2 && !wait_w(kAFree0 + st, ph((c >> 1) - 1))) break;
      tc_fence_after();
      GLA_TRACE_POINT(0, 3, c);
      const uint32_t q_s = sbase + kOffQK + st * kQKStage;
      const uint64_t qd = sdesc_sw128(q_s, 16, 1024), kd = sdesc_sw128(q_s + kQBytes, 16, 1024);
      if (elect_one_sync()) {
        for (int kk = 0; kk < nks; ++kk) {
          const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
          mma_bf16(tmem + kColA + st * 128, desc_add(qd, off), desc_add(kd, off), kIdQK, kk > 0);
        }
        mma_commit(&bars[kAFull0 + st]);
        mma_commit(&bars[kQKEmpty0 + st]);
      }
      __syncwarp();
      mma_issued = true;
    }
  } else if (warp == 2) {
    // ---------------------- issuer B: MMA3 O = Q S', then MMA2 O += P' V
    for (int c = 0; c < nch; ++c) {
      const int st = c & 1;
      if (!wait_w(kQKFull0 + st, ph(c >> 1))) break;
      if (!wait_w(kSReady, ph(c))) break;  // S'_{c-1} hi / lo in shared memory
      if (c >= 2 && !wait_w(kOFree0 + st, ph((c >> 1) - 1))) break;  // output(c-2) read O
      tc_fence_after();
      GLA_TRACE_POINT(0, 4, c);
      const uint32_t q_s = sbase + kOffQK + st * kQKStage;
      const uint64_t qd = sdesc_sw128(q_s, 16, 1024);
      const uint64_t hd = sdesc_sw128(sbase + kOffShi, kPanel, 1024);
      const uint64_t ld = sdesc_sw128(sbase + kOffSlo, kPanel, 1024);
      if (elect_one_sync()) {
        for (int kk = 0; kk < nks; ++kk) {
          const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
          mma_bf16(tmem + kColO + st * kDVS, desc_add(qd, off), desc_add(hd, kk * 2048), kIdQS,
                   kk > 0);
        }
        for (int kk = 0; kk < nks; ++kk) {
          const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
          mma_bf16(tmem + kColO + st * kDVS, desc_add(qd, off), desc_add(ld, kk * 2048), kIdQS,
                   1);
        }
        mma_commit(&bars[kO3Full0 + st]);
        mma_commit(&bars[kSFree]);
        mma_commit(&bars[kQKEmpty0 + st]);
      }
      __syncwarp();
      mma_issued = true;
      // MMA2: P' (A operand in TMEM: hi / lo pairs in place) times the raw V
      if (!wait_w(kPFull0 + st, ph(c >> 1))) break;
      if (!wait_w(kVFull0 + st, ph(c >> 1))) break;
      tc_fence_after();
      GLA_TRACE_POINT(0, 5, c);
      const uint32_t a_p = tmem + kColA + st * 128;
      const uint64_t vd = sdesc_sw128(sbase + kOffV + st * kTile, kPanel, 1024);
      if (elect_one_sync()) {
#pragma unroll
        for (int pass = 0; pass < 2; ++pass)
#pragma unroll
          for (int kk = 0; kk < kC / 16; ++kk)
            mma_bf16_tmem_a(tmem + kColO + st * kDVS, a_p + 32 * (kk >> 1) + 16 * pass + 8 * (kk & 1),
                            desc_add(vd, kk * 2048), kIdPV, 1);
        mma_commit(&bars[kOFull0 + st]);
        mma_commit(&bars[kAFree0 + st]);
        mma_commit(&bars[kVEmpty0 + st]);
      }
      __syncwarp();
    }
  } else if (warp == 3) {
    // -------------------------------------- issuer C: MMA4 U = K^T (W V)
    for (int c = 0; c < nch; ++c) {
      const int st = c & 1;
      if (!wait_w(kQKFull0 + st, ph(c >> 1))) break;
      if (!wait_w(kVtFull, ph(c))) break;  // (W V) hi / lo of chunk c
      if (c >= 2 && !wait_w(kUFree0 + st, ph((c >> 1) - 1))) break;
      tc_fence_after();
      GLA_TRACE_POINT(0, 6, c);
      const uint32_t k_s = sbase + kOffQK + st * kQKStage + kQBytes;
      const uint64_t kd = sdesc_sw128(k_s, kPanel, 1024);
      const uint64_t hd = sdesc_sw128(sbase + kOffWVhi, kPanel, 1024);
      const uint64_t ld = sdesc_sw128(sbase + kOffWVlo, kPanel, 1024);
      if (elect_one_sync()) {
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_bf16(tmem + kColU + st * kDVS, desc_add(kd, kk * 2048), desc_add(hd, kk * 2048),
                   kIdKV, kk > 0);
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_bf16(tmem + kColU + st * kDVS, desc_add(kd, kk * 2048), desc_add(ld, kk * 2048),
                   kIdKV, 1);
        mma_commit(&bars[kUFull0 + st]);
        mma_commit(&bars[kVtFree]);
        mma_commit(&bars[kQKEmpty0 + st]);
      }
      __syncwarp();
      mma_issued = true;
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ mask group
    const int q4 = warp & 3;
    const int r = 32 * q4 + lane;         // token row
    const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
    const float scale = p.scale;

    // this thread's output row of chunk c (valid while r < n)
    auto out_row = [&](int c) -> long long {
      const long long tok = (long long)c * kC + r;
      return start + (p.out_reversed ? len - 1 - tok : tok);
    };

    // output of chunk c: o = scale f_t O[c & 1] (f_t = 2^{G_t - G_L} = 1 / W_t on
    // a plain chunk, 1 on a wide one, whose O carries the decay already)
    auto output = [&](int c, float f) -> bool {
      const int n = min(kC, len - c * kC);
      const bool valid = r < n;
      const long long orow = out_row(c);
      const size_t off = ((size_t)(valid ? orow : start) * p.H + h) * p.DV + (size_t)sl * kDVS;
      const float s1 = valid ? scale * f : 0.f;
      const int b = c & 1;
      if constexpr (DOT) {
        uint4 pr[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          pr[j] = valid ? __ldg(reinterpret_cast<const uint4*>(p.dot_rows + off) + j)
                        : make_uint4(0u, 0u, 0u, 0u);
        if (!wait_w(kOFull0 + b, ph(c >> 1))) return false;  // MMA2(c)
        tc_fence_after();
        float dot = 0.f;
#pragma unroll
        for (int part = 0; part < 4; ++part) {
          uint32_t v[16];
          tmem_ld_32x32b_x16(tmem + lane_off + kColO + b * kDVS + 16 * part, v);
          tmem_ld_wait_x16(v);
          if (part == 3) {
            tc_fence_before();
            warp_arrive(kOFree0 + b);
          }
          float o[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) o[j] = s1 * __uint_as_float(v[j]);
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const uint4 q = pr[2 * part + j];
            const uint32_t bw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              dot = fmaf(o[8 * j + 2 * e], bf16lo(bw[e]),
                         fmaf(o[8 * j + 2 * e + 1], bf16hi(bw[e]), dot));
          }
          if (valid) {
            if constexpr (OUTF32) {
              float* dst = static_cast<float*>(p.out) + off + 16 * part;
#pragma unroll
              for (int j = 0; j < 4; ++j)
                reinterpret_cast<float4*>(dst)[j] =
                    make_float4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
            } else {
              __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + off + 16 * part;
              uint32_t w[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) w[j] = pack_bf16x2(o[2 * j], o[2 * j + 1]);
              reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
              reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
            }
          }
        }
        if (valid) atomicAdd(p.dot_out + (size_t)orow * p.H + h, p.dot_sign * dot);
        return true;
      }
      if (!wait_w(kOFull0 + b, ph(c >> 1))) return false;  // MMA2(c)
      tc_fence_after();
      if (warp == 4 && lane == 0) GLA_TRACE_POINT(0, 9, c);
      for (int part = 0; part < 2; ++part) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem + lane_off + kColO + b * kDVS + 32 * part, v);
        tmem_ld_wait_x32(v);
        if (part == 1) {
          tc_fence_before();
          warp_arrive(kOFree0 + b);
        }
        if (valid) {
          if constexpr (OUTF32) {
            float* dst = static_cast<float*>(p.out) + off + 32 * part;
#pragma unroll
            for (int j = 0; j < 8; ++j)
              reinterpret_cast<float4*>(dst)[j] = make_float4(
                  s1 * __uint_as_float(v[4 * j]), s1 * __uint_as_float(v[4 * j + 1]),
                  s1 * __uint_as_float(v[4 * j + 2]), s1 * __uint_as_float(v[4 * j + 3]));
          } else {
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + off + 32 * part;
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
              w[j] = pack_bf16x2(s1 * __uint_as_float(v[2 * j]),
                                 s1 * __uint_as_float(v[2 * j + 1]));
            if (p.out_v8) {
              st_global_v8(dst, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
              st_global_v8(dst + 16, w[8], w[9], w[10], w[11], w[12], w[13], w[14], w[15]);
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                reinterpret_cast<uint4*>(dst)[j] =
                    make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
            }
          }
        }
      }
      return true;
    };

    // iteration c: P' of chunk c, then the output of chunk c - 1 (its MMA2 ran
    // while this P' was built)
    float fprev = 1.f;
    for (int c = 0; c <= nch; ++c) {
      float f = 1.f;
      if (c < nch) {
        const int b = c & 1;
        if (!wait_w(kGReady0 + c % kSlots, ph(c / kSlots))) break;
        const float* slot = slot_of(c);
        const float ar = slot[r];
        const bool wide = slot[129] != 0.f;
        if (!wait_w(kAFull0 + b, ph(c >> 1))) break;
        tc_fence_after();
        const uint32_t a_row = tmem + lane_off + kColA + b * 128;
        if (warp == 4 && lane == 0) GLA_TRACE_POINT(0, 7, c);
        // the tensor-memory accesses stay warp-uniform (.sync.aligned)
        if (wide) {
          build_p<true>(a_row, q4, r, ar, slot);
        } else {
          build_p<false>(a_row, q4, r, 0.f, slot);
        }
        warp_arrive(kGFree0 + c % kSlots);
        if (wide) {
          // O = Q S_{c-1} so far: row t times 2^{G_t} before MMA2 adds P V
          if (!wait_w(kO3Full0 + b, ph(c >> 1))) break;
          tc_fence_after();
          const float e = exp2f(ar);
          const uint32_t o_row = tmem + lane_off + kColO + b * kDVS;
#pragma unroll 1
          for (int part = 0; part < 4; ++part) {
            uint32_t v[16];
            tmem_ld_32x32b_x16(o_row + 16 * part, v);
            tmem_ld_wait_x16(v);
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = __float_as_uint(e * __uint_as_float(v[j]));
            tmem_st_32x32b_x16(o_row + 16 * part, v);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        warp_arrive(kPFull0 + b);
        // the row factor of this chunk's output (written next iteration), off
        // the path from the A wait to P'-ready
        f = wide ? 1.f : (ar != 0.f ? 1.f / ar : 0.f);
        if (warp == 4 && lane == 0) GLA_TRACE_POINT(0, 8, c);
      }
      if (c >= 1 && !output(c - 1, fprev)) break;
      fprev = f;
    }
  } else {
    // ----------------------------------------------------------- state group
    const int q4 = warp & 3;
    const int hh = (warp - 8) >> 2;       // which 32 of the 64 state / V columns
    const int r = 32 * q4 + lane;         // state row i (key channel), token row for W V
    const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
    // state rows past the key head size (d_k = 64, 96) stay zero: their K
    // channels are the zero columns the TMA fills in
    const bool row_ok = r < p.DK;
    const size_t st_off = ((size_t)s * p.H + h) * (size_t)p.DK * p.DV +
                          (size_t)(row_ok ? r : 0) * p.DV + (size_t)sl * kDVS + 32 * hh;
    float S[32];
    if (p.init_state && row_ok) {
      const float4* src = reinterpret_cast<const float4*>(p.init_state + st_off);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 x = __ldg(src + j);
        S[4 * j] = x.x; S[4 * j + 1] = x.y; S[4 * j + 2] = x.z; S[4 * j + 3] = x.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) S[j] = 0.f;
    }

    // W V split of chunk c (token row r, V columns 32 hh .. +31) into bf16 hi
    // and lo, once MMA4(c - 1) is done with the single (W V) buffer
    auto split_wv = [&](int c) -> bool {
      const int b = c & 1;
      const int n = min(kC, len - c * kC);
      if (!wait_w(kGReady0 + c % kSlots, ph(c / kSlots))) return false;
      const float* slot = slot_of(c);
      const float total = slot[128];
      const bool wide = slot[129] != 0.f;
      const float w = r < n ? (wide ? exp2f(total - slot[r]) : slot[r]) : 0.f;
      if (!wait_w(kVFull0 + b, ph(c >> 1))) return false;
      if (c >= 1 && !wait_w(kVtFree, ph(c - 1))) return false;
      if (warp == 8 && lane == 0) GLA_TRACE_POINT(0, 11, c);
      const uint8_t* v_s = smem + kOffV + b * kTile;
      uint8_t* hi_s = smem + kOffWVhi;
      uint8_t* lo_s = smem + kOffWVlo;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t o = sw128_offset(r, 4 * hh + q);
        const uint4 raw = *reinterpret_cast<const uint4*>(v_s + o);
        const uint32_t in[4] = {raw.x, raw.y, raw.z, raw.w};
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x0 = w * bf16lo(in[e]), x1 = w * bf16hi(in[e]);
          hi[e] = pack_bf16x2(x0, x1);
          lo[e] = pack_bf16x2(x0 - bf16lo(hi[e]), x1 - bf16hi(hi[e]));
        }
        *reinterpret_cast<uint4*>(hi_s + o) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(lo_s + o) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      fence_proxy_async_smem();
      warp_arrive(kVtFull);
      warp_arrive(kVEmpty0 + b);  // the V tile is also MMA2's; this group is done with it
      if (warp == 8 && lane == 0) GLA_TRACE_POINT(0, 12, c);
      return true;
    };

    // S' = f S as bf16 hi + lo into the S' tile (row r, columns 32 hh .. +31),
    // once MMA3 of the previous chunk is done with it
    auto store_sp = [&](int c, float f) -> bool {
      uint32_t hw[16], lw[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float x0 = f * S[2 * e], x1 = f * S[2 * e + 1];
        hw[e] = pack_bf16x2(x0, x1);
        lw[e] = pack_bf16x2(x0 - bf16lo(hw[e]), x1 - bf16hi(hw[e]));
      }
      if (c >= 0 && !wait_w(kSFree, ph(c))) return false;  // MMA3(c) read S'_{c-1}
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t o = sw128_offset(r, 4 * hh + q);
        *reinterpret_cast<uint4*>(smem + kOffShi + o) =
            make_uint4(hw[4 * q], hw[4 * q + 1], hw[4 * q + 2], hw[4 * q + 3]);
        *reinterpret_cast<uint4*>(smem + kOffSlo + o) =
            make_uint4(lw[4 * q], lw[4 * q + 1], lw[4 * q + 2], lw[4 * q + 3]);
      }
      fence_proxy_async_smem();
      warp_arrive(kSReady);
      if (warp == 8 && lane == 0) GLA_TRACE_POINT(0, 14, c + 1);
      return true;
    };

    bool ok = true;
    // iteration c: the split of chunk c + 1 (MMA4(c + 1) needs it), then the
    // state step with U_c and the S' tile for chunk c + 1 (c = -1: the initial
    // state)
    for (int c = -1; c < nch && ok; ++c) {
      if (c + 1 < nch && !split_wv(c + 1)) { ok = false; break; }
      if (c >= 0) {
        const int b = c & 1;
        const float decay = exp2f(slot_of(c)[128]);
        if (!wait_w(kUFull0 + b, ph(c >> 1))) { ok = false; break; }
        if (warp == 8 && lane == 0) GLA_TRACE_POINT(0, 13, c);
        tc_fence_after();
        uint32_t u[32];
        tmem_ld_32x32b_x32(tmem + lane_off + kColU + b * kDVS + 32 * hh, u);
        tmem_ld_wait_x32(u);
#pragma unroll
        for (int j = 0; j < 32; ++j) S[j] = fmaf(decay, S[j], __uint_as_float(u[j]));
        tc_fence_before();
        warp_arrive(kUFree0 + b);
      }
      if (c + 1 < nch) {
        const float* nslot = slot_of(c + 1);
        const float f = nslot[129] != 0.f ? 1.f : exp2f(nslot[128]);
        if (!store_sp(c, f)) { ok = false; break; }
      }
      if (c >= 0) warp_arrive(kGFree0 + c % kSlots);
    }
    if (ok && p.final_state && row_ok) {
      float4* dst = reinterpret_cast<float4*>(p.final_state + st_off);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        dst[j] = make_float4(S[4 * j], S[4 * j + 1], S[4 * j + 2], S[4 * j + 3]);
    }
  }

  // Teardown, also after an abort: every copy into this CTA's shared memory and
  // every MMA (with its commits' barrier arrivals) lands before the CTA ends.
  if (warp == 0 && lane == 0) {
    for (int st = 0; st < 2; ++st) {
      drain_bar(&bars[kQKFull0 + st], issued_qk[st]);
      drain_bar(&bars[kVFull0 + st], issued_v[st]);
    }
  }
  if (warp >= 1 && warp <= 3 && mma_issued) {
    // the lane that issued this warp's MMAs commits them to the drain barrier
    if (elect_one_sync()) mma_commit(&bars[kDrain + warp - 1]);
    __syncwarp();
    (void)mbar_wait_bounded(&bars[kDrain + warp - 1], 0u, kWaitLimitNs);
  }
  if (__any_sync(0xffffffffu, *abort_flag != 0)) {
    // a role that gave up may have left tensor-memory accesses unwaited
    tmem_ld_wait();
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0) GLA_TRACE_POINT(0, 31, 0);
  if (warp == 1) {
    __syncwarp();
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

// bf16 tensor [nb][rows][H][d] viewed as 4-D {d, H, rows, nb}; box {64, 1, 128, 1}.
bool make_map(CUtensorMap* map, const void* base, int d, int H, long long rows, int nb) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)rows, (cuuint64_t)nb};
  const cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2,
                                 (cuuint64_t)rows * H * d * 2};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)kC, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool chunk_tc_supported(const ChunkArgs& a) {
  return !a.fp32_io && !a.vector_gate && a.chunk == kC &&
         (a.dk == 64 || a.dk == 96 || a.dk == kDK) &&
         (a.dv == 64 || a.dv == 128 || a.dv == 192);
}

cudaError_t launch_chunk_tc(const ChunkArgs& a, cudaStream_t stream) {
  // dense: [B][T][H][d]; packed: one batch of T rows
  const bool packed = a.cu_seqlens != nullptr;
  const long long rows = a.T;
  const int nb = packed ? 1 : a.B;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, a.q, a.dk, a.H, rows, nb) || !make_map(&mk, a.k, a.dk, a.H, rows, nb) ||
      !make_map(&mv, a.v, a.dv, a.H, rows, nb))
    return cudaErrorInvalidValue;
  TcParams p;
  p.g = a.g; p.scale = a.scale; p.init_state = a.init_state; p.out = a.out;
  p.final_state = a.final_state; p.cu_seqlens = a.cu_seqlens;
  p.B = a.B; p.H = a.H; p.T = a.T; p.DK = a.dk; p.DV = a.dv; p.nslices = a.dv / kDVS;
  p.status = a.status;
  p.wait_ns = handoff_wait_limit_ns();
  p.out_v8 = (reinterpret_cast<uintptr_t>(a.out) & 31) == 0;
  p.out_reversed = a.out_reversed;
  p.dot_rows = static_cast<const __nv_bfloat16*>(a.dot_rows);
  p.dot_out = a.dot_out;
  p.dot_sign = a.dot_sign;
  const long long ctas = (long long)a.B * a.H * p.nslices;
  auto run = [&](auto kern) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)ctas, kThreads, kSmemBytes, stream>>>(mq, mk, mv, p);
    return cudaGetLastError();
  };
  if (a.dot_out)
    return a.fp32_out ? run(chunk_tc_kernel<true, true>) : run(chunk_tc_kernel<false, true>);
  return a.fp32_out ? run(chunk_tc_kernel<true, false>) : run(chunk_tc_kernel<false, false>);
}

}  // namespace gla
