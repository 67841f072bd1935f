// gla_chunk_tc.cu -- chunked GLA prefill on the 5th-generation tensor cores.
//
// Method: the chunked form of the "i14 Laplace 3B on AWS Trainium2" page
// (section "Challenge 1", Figure 3) with per-token log-decays g.  For a chunk
// of C = 128 tokens, G_t = sum of g over the chunk up to and including t, and
// L the chunk's last token:
//     S_next = exp(G_L) S + K^T (W V),     W_j = exp(G_L - G_j)  (<= 1)
//     o_t    = scale * ( sum_{j<=t} A_tj exp(G_t - G_j) V_j + exp(G_t) (Q S)_t )
// with A = Q K^T.  Writing exp(G_t - G_j) = exp(G_t - G_L) W_j, the
// intra-chunk term becomes exp(G_t - G_L) * (causal(A) . (W V))_t: the same
// decayed values W V that update the state also serve the output, and the
// mask is a plain causal mask.  This is exact while the chunk's decay span
// exp(G_0 - G_L) stays inside 2^96 (so W V and the row factor stay in the
// normal bf16/fp32 range); a chunk with a wider span takes the explicit path:
// P = A * exp(G_t - G_j) on the causal part, times the raw V.
//
// Since exp(G_t) = exp(G_t - G_L) exp(G_L), the whole output row is
//     o_t = scale * exp(G_t - G_L) * ( Q S' + causal(A) (W V) )_t,  S' = exp(G_L) S
// and the two contractions share one accumulator.
//
// Head sizes: d_k = 128, or 64 and 96 run as 128 (the TMA fills the channels
// past d_k with zeros -- for d_k = 64 the whole second 64-channel panel lies
// outside the tensor -- so those state rows stay zero and are never stored);
// d_v = 64, 128 or 192 (one CTA per 64-wide slice).
//
// One CTA owns one (sequence, head, 64-wide slice of dv) and walks the chunks
// in order.  The state slice S (dk x 64, fp32) lives in tensor memory (TMEM)
// for the whole sequence: the state group scales it by exp(G_L) in place (its
// bf16 copy is S') and the chunk's K^T (W V) accumulates into it.  Four
// tcgen05 contractions per chunk, bf16 x bf16 -> fp32 in TMEM:
//     MMA1  A   = Q K^T              M=128 (t) N=128 (j) K=dk  A,B smem K-major
//     MMA4  S  += K^T (W V)          M=dk (i)  N=64      K=128 A,B smem MN-major
//     MMA3  O   = Q S'               M=128 (t) N=64      K=dk  B smem MN-major
//     MMA2  O  += P' (W V)           M=128 (t) N=64      K=128 A = P' in TMEM,
//                                                                three passes
// O is double-buffered by chunk parity, so MMA2 of a chunk never waits for
// the previous chunk's output to be read.  A wide chunk keeps S' = S and the
// mask group scales O's row t by exp(G_t) between MMA3 and MMA2.
// W V is carried as two bf16 tiles, hi + lo (hi = W V rounded, lo = the
// rest), and MMA2 takes both passes; MMA4 takes the lo pass only while the
// decay still to come over the next two chunks is at least 2^-16 (else the
// final state sees this chunk's rounding shrunk below 2^-25).  P' = causal(A) is
// rounded to bf16 once, except on the four 32 x 32 diagonal blocks, where the
// largest terms of a row sit under strong decay: there P' also has a lo part,
// taken in a third MMA2 pass against (W V)_hi.  P' overwrites A in TMEM:
// block b (32 fp32 columns) becomes 16 columns of bf16 pairs at column 16 b,
// and the diagonal lo parts fill columns 64 .. 127 (block b at 64 + 16 b,
// zero off the row's own diagonal block); every fp32 block a row needs is
// read by then.
//
// Resources and their release points (the chunk pipeline):
//   Q, K tiles      2-stage ring, free once MMA1 and MMA3/MMA4 of the chunk
//                   have run (one commit from each issuer)
//   V tile          single buffer, free once the W V split has read it (wide
//                   chunks: once MMA2 has run)
//   (W V) hi, lo    2 buffers each, free once MMA2 (and MMA4) have run
//   S'              1 buffer, bf16 (B operand of MMA3), rewritten once MMA4
//                   (issued after MMA3) has completed
//   O               2 buffers in TMEM, free once the output has read them
// Roles (16 warps):
//   warp 0       producer: prefix sums of g and the chunk's flags (all lanes,
//                into a 3-slot ring), then the TMA loads (lane 0)
//   warp 1       TMEM allocator; issues MMA1
//   warp 2       issues MMA2
//   warp 3       issues MMA3 then MMA4 (the state chain)
// Each MMA issuer waits only for its own operands, so no chain holds up
// another one's issue.
//   warps 4..7   mask group: P' from A (thread t owns token row t), then the
//                output of the previous chunk (256-bit stores when the output
//                is 32-byte aligned)
//   warps 8..15  state group: W V split, in-place decay of S, the bf16 copy of
//                S (S') for MMA3, the final state; two warps per TMEM lane
//                quadrant, each owning 32 of the 64 state columns
// TMEM: A/P' 2x128, O 2x64, S 64 (columns 384..447 unused) of 512.  Every
// mbarrier wait is bounded in wall time; on timeout the kernel flags the
// device status word, stops issuing work, releases TMEM and returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "gla_internal.cuh"
#include "gla_sm100.cuh"

namespace gla {
namespace {

using namespace sm100;

constexpr int kC = 128;        // chunk (tokens)
constexpr int kDK = 128;       // key head size of the tiles (d_k = 64, 96 run zero-padded)
constexpr int kDVS = 64;       // value columns per CTA
constexpr int kThreads = 512;  // 16 warps
constexpr int kMaskWarps = 4;
constexpr int kStateWarps = 8;
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kWideSpan = 96.f;      // log2 chunk decay span above which a chunk is "wide"
constexpr float kLoCutoff = -16.f;     // log2 decay still to come below which MMA4 skips lo
constexpr int kSlots = 3;              // gate ring: chunks c (mask), c + 1 (split), c + 2 (gate)

// shared memory map (offsets from the 1024-byte-aligned base)
constexpr uint32_t kPanel = kC * 128;                 // 128 rows x 128 B
constexpr uint32_t kQBytes = kPanel * (kDK / 64);     // 32 KB
constexpr uint32_t kKBytes = kPanel * (kDK / 64);     // 32 KB
constexpr uint32_t kQKStage = kQBytes + kKBytes;      // 64 KB
constexpr uint32_t kTile = kPanel;                    // 16 KB: 128 rows x 64 columns bf16
constexpr uint32_t kOffV = 2 * kQKStage;
constexpr uint32_t kOffVhi = kOffV + kTile;           // 2 buffers
constexpr uint32_t kOffVlo = kOffVhi + 2 * kTile;     // 2 buffers
constexpr uint32_t kOffSb = kOffVlo + 2 * kTile;      // dk rows x 128 B
// gate slot (floats): G2[128] | total, wide, need_lo, -
constexpr int kSlotG2 = 0, kSlotTotal = 128, kSlotWide = 129, kSlotNeedLo = 130, kSlotFloats = 132;
constexpr uint32_t kOffGate = kOffSb + kDK * 128;
constexpr uint32_t kOffBar = kOffGate + kSlots * kSlotFloats * 4;
constexpr uint32_t kBarBytes = 320;
constexpr uint32_t kOffMisc = kOffBar + kBarBytes;    // tmem base, abort flag
constexpr uint32_t kSmemUsed = kOffMisc + 16;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;     // alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffBar % 8 == 0 && kOffGate % 16 == 0, "alignment");

// TMEM column map
constexpr uint32_t kColA = 0;      // 2 x 128: A = Q K^T (fp32), then P' (bf16 pairs) in place
constexpr uint32_t kColO = 256;    // 2 x 64: O = Q S' + P' (W V), per chunk parity
constexpr uint32_t kColS = 448;    // 64: the running state slice, fp32

enum Bar {
  kQKFull0 = 0, kQKFull1, kQKEmpty0, kQKEmpty1, kVFull, kVEmpty, kAFull0, kAFull1,
  kAFree0, kAFree1, kPFull0, kPFull1, kVtFull0, kVtFull1, kVtFree0, kVtFree1, kSFull, kSReady,
  kO3Full0, kO3Full1, kOFull0, kOFull1, kOFree0, kOFree1, kStateSync, kGReady0,
  kGFree0 = kGReady0 + kSlots, kNumBars = kGFree0 + kSlots
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
};

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// P' of token row r (lane quadrant q4) from A = Q K^T in TMEM, in place.  A
// row is read one 32-column block at a time, the next block's load in flight;
// P' of block cb goes to columns 16 cb .. 16 cb + 15 (already read), and the
// lo part of the row's diagonal block to 64 + 16 q4 (the other three lo
// blocks are zero).  WIDE: explicit decay exp(G_t - G_j) <= 1 on the causal
// part (G2s: the chunk's log2 prefix sums); otherwise the plain causal mask.
// The two variants are separate bodies so that neither pays for the other.
template <bool WIDE>
__device__ __forceinline__ void build_p_body(uint32_t a_row, int q4, int r, float G2,
                                             const float* G2s) {
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
      for (int e = 0; e < 16; ++e) {
        float x0 = __uint_as_float(a[2 * e]), x1 = __uint_as_float(a[2 * e + 1]);
        if constexpr (WIDE) {
          x0 *= exp2f(G2 - G2s[32 * cb + 2 * e]);
          x1 *= exp2f(G2 - G2s[32 * cb + 2 * e + 1]);
        }
        pk[e] = pack_bf16x2(x0, x1);
      }
      tmem_ld_32x32b_x32(a_row + 32 * (cb + 1), a);
    } else {
      // diagonal block: causal mask (diagonal kept), bf16 hi + lo
      tmem_ld_wait_x32(a);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int j = 32 * cb + 2 * e;
        float x0 = j <= r ? __uint_as_float(a[2 * e]) : 0.f;
        float x1 = j + 1 <= r ? __uint_as_float(a[2 * e + 1]) : 0.f;
        if constexpr (WIDE) {
          x0 = j <= r ? x0 * exp2f(G2 - G2s[j]) : 0.f;
          x1 = j + 1 <= r ? x1 * exp2f(G2 - G2s[j + 1]) : 0.f;
        }
        pk[e] = pack_bf16x2(x0, x1);
        dlo[e] = pack_bf16x2(x0 - bf16lo(pk[e]), x1 - bf16hi(pk[e]));
      }
    }
    tmem_st_32x32b_x16(a_row + 16 * cb, pk);
  }
#pragma unroll
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
__device__ __forceinline__ void build_p(uint32_t a_row, int q4, int r, float G2) {
  build_p_body<false>(a_row, q4, r, G2, nullptr);
}
// wide chunks are rare: their variant stays out of line
__device__ __noinline__ void build_p_wide(uint32_t a_row, int q4, int r, float G2,
                                          const float* G2s) {
  build_p_body<true>(a_row, q4, r, G2, G2s);
}

template <bool OUTF32, bool DOT>
__global__ void __launch_bounds__(kThreads, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  float* gate_ring = reinterpret_cast<float*>(smem + kOffGate);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nsl = p.nslices;
  const int sl = blockIdx.x % nsl;
  const int h = (blockIdx.x / nsl) % p.H;
  const int s = blockIdx.x / (nsl * p.H);

  long long start;
  int len;
  // all threads agree (same s): either every thread returns here or none does
  if (!seq_bounds(p.cu_seqlens, s, p.B, p.T, &start, &len, p.status)) return;
  const int nch = (len + kC - 1) / kC;
  const bool packed = p.cu_seqlens != nullptr;

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      // group barriers take one arrival per warp (see warp_arrive)
      uint32_t cnt = 1;
      if (i == kPFull0 || i == kPFull1 || i == kOFree0 || i == kOFree1) cnt = kMaskWarps;
      if (i == kVtFull0 || i == kVtFull1 || i == kSReady || i == kStateSync) cnt = kStateWarps;
      // both MMA issuers that read Q and K commit to the stage's empty barrier
      if (i == kQKEmpty0 || i == kQKEmpty1) cnt = 2;
      // gate slots are released by both groups and the MMA2 issuer
      if (i >= kGFree0 && i < kGFree0 + kSlots) cnt = kMaskWarps + kStateWarps + 1;
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
  const uint32_t tmem = *tmem_slot;
  const uint32_t sbase = smem_u32(smem);

  auto wait = [&](int b, uint32_t parity) -> bool {
    if (*abort_flag) return false;
    if (mbar_wait_bounded(&bars[b], parity, kWaitLimitNs)) return true;
    *abort_flag = 1;
    atomicOr(p.status, kDevTimeout);
    return false;
  };
  // the same, decided for the whole warp (full-warp roles never split on a wait)
  auto wait_w = [&](int b, uint32_t parity) -> bool {
    return __all_sync(0xffffffffu, wait(b, parity));
  };
  // parity of the k-th completion (k = 0, 1, ...) of a barrier
  auto ph = [](int k) -> uint32_t { return static_cast<uint32_t>(k) & 1u; };
  // One arrival for the whole warp, after every lane's prior writes and fences
  // (__syncwarp orders them before lane 0's release-arrive).
  auto warp_arrive = [&](int b) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[b]);
  };
  auto slot_of = [&](int c) -> float* { return gate_ring + (c % kSlots) * kSlotFloats; };

  if (warp == 0) {
    // ------------------------------------------- producer: gate sums and TMA
    // All lanes: prefix sums of g for chunk c (lane l owns tokens 4l .. 4l+3)
    // into the gate ring; lane 0: the TMA loads of chunk c.
    // raw values: the clamp is applied where they are used, an iteration or more
    // later, so that nothing waits for these loads in the iteration that issues them
    auto load4 = [&](int c, float (&gv)[4]) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int t = c * kC + 4 * lane + i;
        gv[i] = (c < nch && t < len) ? __ldg(p.g + (start + t) * p.H + h) : 0.f;
      }
    };
    auto clamp4 = [](const float (&x)[4]) {
      return fmaxf(x[0], -kGateClamp) + fmaxf(x[1], -kGateClamp) + fmaxf(x[2], -kGateClamp) +
             fmaxf(x[3], -kGateClamp);
    };
    // sum over the warp of a per-lane value
    auto warp_sum = [&](float x) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
      return x;
    };
    const int bidx = packed ? 0 : s;
    // The totals of g over chunks c + 1 and c + 2 decide whether MMA4(c) needs the
    // lo half of W V (the final state sees chunk c's rounding scaled by the decay
    // still to come).  g is loaded three chunks ahead, so that those sums never
    // wait for a load issued in the same iteration (this warp's gate sums and TMA
    // issues pace every other role).
    float gnext[4], gnext2[4], gnext3[4];
    load4(0, gnext);
    load4(1, gnext2);
    load4(2, gnext3);
    for (int c = 0; c < nch; ++c) {
      bool ok = true;
      float gv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        gv[i] = gnext[i];
        gnext[i] = gnext2[i];
        gnext2[i] = gnext3[i];
      }
      load4(c + 3, gnext3);
      const float rest = warp_sum(clamp4(gnext)) + warp_sum(clamp4(gnext2));
      if (c >= kSlots && !wait(kGFree0 + c % kSlots, ph(c / kSlots - 1))) ok = false;
      if (__any_sync(0xffffffffu, !ok)) break;
      float* slot = slot_of(c);
#pragma unroll
      for (int i = 0; i < 4; ++i) gv[i] = fmaxf(gv[i], -kGateClamp);
      float run[4];
      run[0] = gv[0];
#pragma unroll
      for (int i = 1; i < 4; ++i) run[i] = run[i - 1] + gv[i];
      float incl = run[3];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      const float excl = incl - run[3];
      const float total = __shfl_sync(0xffffffffu, incl, 31) * kLog2e;
      float G2[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) G2[i] = (excl + run[i]) * kLog2e;
      *reinterpret_cast<float4*>(slot + kSlotG2 + 4 * lane) =
          make_float4(G2[0], G2[1], G2[2], G2[3]);
      const float first = __shfl_sync(0xffffffffu, G2[0], 0);
      if (lane == 0) {
        slot[kSlotTotal] = total;
        slot[kSlotWide] = (first - total > kWideSpan) ? 1.f : 0.f;
        slot[kSlotNeedLo] = (rest * kLog2e < kLoCutoff) ? 0.f : 1.f;
      }
      warp_arrive(kGReady0 + c % kSlots);
      if (lane == 0) {
        const int st = c & 1;
        const int row = packed ? (int)(start + (long long)c * kC) : c * kC;
        if (c >= 2 && !wait(kQKEmpty0 + st, ph((c >> 1) - 1))) ok = false;
        if (ok) {
          uint8_t* q_s = smem + st * kQKStage;
          uint8_t* k_s = q_s + kQBytes;
          mbar_arrive_expect_tx(&bars[kQKFull0 + st], kQKStage);
#pragma unroll
          for (int pn = 0; pn < kDK / 64; ++pn) {
            tma_load_4d(q_s + pn * kPanel, &tmQ, &bars[kQKFull0 + st], pn * 64, h, row, bidx);
            tma_load_4d(k_s + pn * kPanel, &tmK, &bars[kQKFull0 + st], pn * 64, h, row, bidx);
          }
        }
        if (ok && c >= 1 && !wait(kVEmpty, ph(c - 1))) ok = false;
        if (ok) {
          mbar_arrive_expect_tx(&bars[kVFull], kTile);
          tma_load_4d(smem + kOffV, &tmV, &bars[kVFull], sl * kDVS, h, row, bidx);
        }
      }
      if (__any_sync(0xffffffffu, !ok)) break;
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA1 issuer
    if (lane == 0) {
      for (int c = 0; c < nch; ++c) {
        const int st = c & 1;
        const uint32_t q_s = sbase + st * kQKStage;
        const uint32_t k_s = q_s + kQBytes;
        if (!wait(kQKFull0 + st, ph(c >> 1))) break;
        if (c >= 2 && !wait(kAFree0 + st, ph((c >> 1) - 1))) break;
        tc_fence_after();
        const uint64_t qd = sdesc_sw128(q_s, 16, 1024), kd = sdesc_sw128(k_s, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kDK / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
          mma_bf16(tmem + kColA + st * 128, desc_add(qd, off), desc_add(kd, off), kIdQK, kk > 0);
        }
        mma_commit(&bars[kAFull0 + st]);
        mma_commit(&bars[kQKEmpty0 + st]);  // this issuer is done with Q(c), K(c)
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------- MMA back: 2
    if (lane == 0) {
      for (int c = 0; c < nch; ++c) {
        const int st = c & 1;
        // one P' barrier per chunk parity: the mask group may finish P' of chunk
        // c + 1 before this wait (P' of chunk c + 2 needs MMA2(c) first)
        if (!wait(kPFull0 + st, ph(c >> 1))) break;
        if (!wait(kO3Full0 + st, ph(c >> 1))) break;  // MMA3(c) first, then accumulate
        if (!wait(kVtFull0 + st, ph(c >> 1))) break;  // W V (and V) of chunk c ready
        tc_fence_after();
        const bool wide = slot_of(c)[kSlotWide] != 0.f;
        mbar_arrive(&bars[kGFree0 + c % kSlots]);
        const uint32_t a_p = tmem + kColA + st * 128;  // P': k-step kk at column 8 kk
        // P' hi at column 8 kk, the diagonal lo parts at 64 + 8 kk; B is the raw V
        // on a wide chunk, else (W V) hi and lo
        const uint64_t hd =
            sdesc_sw128(wide ? sbase + kOffV : sbase + kOffVhi + st * kTile, kPanel, 1024);
        const uint64_t ld = sdesc_sw128(sbase + kOffVlo + st * kTile, kPanel, 1024);
        const uint32_t d = tmem + kColO + st * kDVS;
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_bf16_tmem_a(d, a_p + 8 * kk, desc_add(hd, kk * 2048), kIdPV, 1);
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_bf16_tmem_a(d, a_p + 64 + 8 * kk, desc_add(hd, kk * 2048), kIdPV, 1);
        if (!wide) {
#pragma unroll
          for (int kk = 0; kk < kC / 16; ++kk)
            mma_bf16_tmem_a(d, a_p + 8 * kk, desc_add(ld, kk * 2048), kIdPV, 1);
        }
        mma_commit(&bars[kOFull0 + st]);
        mma_commit(&bars[kAFree0 + st]);   // A/P' buffer
        mma_commit(&bars[kVtFree0 + st]);  // (W V) hi/lo buffers
        if (wide) mma_commit(&bars[kVEmpty]);
      }
    }
  } else if (warp == 3) {
    // ---------------------------------------------------- MMA3 / MMA4 issuer
    // MMA3(c) (O = Q S') first, so that MMA2 can follow early, then MMA4(c)
    // (S += K^T (W V)); the commit after MMA4 covers both.
    if (lane == 0) {
      const uint32_t sb = sbase + kOffSb;
      for (int c = 0; c < nch; ++c) {
        const int st = c & 1;
        const uint32_t q_s = sbase + st * kQKStage;
        const uint32_t k_s = q_s + kQBytes;
        if (!wait(kQKFull0 + st, ph(c >> 1))) break;
        if (!wait(kVtFull0 + st, ph(c >> 1))) break;
        if (!wait(kSReady, ph(c))) break;  // S' in smem, exp(G_L) S_{c-1} in TMEM
        if (c >= 2 && !wait(kOFree0 + st, ph((c >> 1) - 1))) break;  // output(c-2) read O
        // slot c stays until MMA2(c) has run, which needs this warp's MMA3(c)
        if (!wait(kGReady0 + c % kSlots, ph(c / kSlots))) break;
        const bool need_lo = slot_of(c)[kSlotNeedLo] != 0.f;
        tc_fence_after();
        {
          const uint64_t qd = sdesc_sw128(q_s, 16, 1024), sd = sdesc_sw128(sb, kPanel, 1024);
#pragma unroll
          for (int kk = 0; kk < kDK / 16; ++kk)
            mma_bf16(tmem + kColO + st * kDVS, desc_add(qd, (kk >> 2) * kPanel + (kk & 3) * 32),
                     desc_add(sd, kk * 2048), kIdQS, kk > 0);
        }
        mma_commit(&bars[kO3Full0 + st]);  // O = Q S' written
        {
          const uint64_t kd = sdesc_sw128(k_s, kPanel, 1024);
          const uint64_t hd = sdesc_sw128(sbase + kOffVhi + st * kTile, kPanel, 1024);
          const uint64_t ld = sdesc_sw128(sbase + kOffVlo + st * kTile, kPanel, 1024);
#pragma unroll
          for (int kk = 0; kk < kC / 16; ++kk)
            mma_bf16(tmem + kColS, desc_add(kd, kk * 2048), desc_add(hd, kk * 2048), kIdKV, 1);
          if (need_lo) {
#pragma unroll
            for (int kk = 0; kk < kC / 16; ++kk)
              mma_bf16(tmem + kColS, desc_add(kd, kk * 2048), desc_add(ld, kk * 2048), kIdKV, 1);
          }
        }
        mma_commit(&bars[kSFull]);          // S = S_c, and S' no longer read
        mma_commit(&bars[kQKEmpty0 + st]);  // this issuer is done with Q(c), K(c)
      }
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ mask group
    const int q4 = warp & 3;
    const int r = 32 * q4 + lane;         // token row
    const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
    const float scale = p.scale;

    // one 16-column part of an output row: to the output's dtype and stored
    auto store_part = [&](size_t off, int part, const float* o) {
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
    };

    // this thread's output row of chunk c (valid while r < n)
    auto out_row = [&](int c) -> long long {
      const long long tok = (long long)c * kC + r;
      return start + (p.out_reversed ? len - 1 - tok : tok);
    };

    // output of chunk c: o = scale f_t O[c & 1], f_t = exp(G_t - G_L) (1 on wide
    // chunks, whose O carries the decay already)
    auto output = [&](int c, float f) -> bool {
      const int n = min(kC, len - c * kC);
      const long long orow = out_row(c);
      const size_t off = ((size_t)orow * p.H + h) * p.DV + (size_t)sl * kDVS;
      const float s1 = scale * f;
      if constexpr (DOT) {
        // the row's 64 partner values, loaded before MMA2 is waited for
        uint4 pr[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          pr[j] = r < n ? __ldg(reinterpret_cast<const uint4*>(p.dot_rows + off) + j)
                        : make_uint4(0u, 0u, 0u, 0u);
        if (!wait_w(kOFull0 + (c & 1), ph(c >> 1))) return false;  // MMA2(c)
        tc_fence_after();
        float dot = 0.f;
#pragma unroll
        for (int part = 0; part < 4; ++part) {
          uint32_t v[16];
          tmem_ld_32x32b_x16(tmem + lane_off + kColO + (c & 1) * kDVS + 16 * part, v);
          tmem_ld_wait();
          if (part == 3) {
            tc_fence_before();
            warp_arrive(kOFree0 + (c & 1));
          }
          float o[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) o[j] = s1 * __uint_as_float(v[j]);
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const uint4 b = pr[2 * part + j];
            const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              dot = fmaf(o[8 * j + 2 * e], bf16lo(bw[e]),
                         fmaf(o[8 * j + 2 * e + 1], bf16hi(bw[e]), dot));
          }
          if (r < n) store_part(off, part, o);
        }
        if (r < n) atomicAdd(p.dot_out + (size_t)orow * p.H + h, p.dot_sign * dot);
        return true;
      }
      if (!wait_w(kOFull0 + (c & 1), ph(c >> 1))) return false;  // MMA2(c)
      tc_fence_after();
#pragma unroll 1
      for (int part = 0; part < 4; ++part) {
        uint32_t v[16];
        tmem_ld_32x32b_x16(tmem + lane_off + kColO + (c & 1) * kDVS + 16 * part, v);
        tmem_ld_wait();
        if (part == 3) {
          tc_fence_before();
          warp_arrive(kOFree0 + (c & 1));
        }
        float o[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) o[j] = s1 * __uint_as_float(v[j]);
        if (r < n) store_part(off, part, o);
      }
      return true;
    };

    // iteration c: P' of chunk c, then the output of chunk c - 1 (its MMA2 ran
    // while this P' was built)
    float fprev = 1.f;
    for (int c = 0; c <= nch; ++c) {
      float f = 1.f;
      if (c < nch) {
        if constexpr (DOT) {
          // chunk c's partner rows into L2, an iteration before output(c) reads them
          if (r < len - c * kC) {
            const __nv_bfloat16* row =
                p.dot_rows + ((size_t)out_row(c) * p.H + h) * p.DV + (size_t)sl * kDVS;
            prefetch_l2(row);
            prefetch_l2(row + kDVS - 8);
          }
        }
        const int st = c & 1;
        const float* slot = slot_of(c);
        if (!wait_w(kGReady0 + c % kSlots, ph(c / kSlots))) break;
        const float G2 = slot[kSlotG2 + r];
        const float total = slot[kSlotTotal];
        const bool wide = slot[kSlotWide] != 0.f;
        f = wide ? 1.f : exp2f(G2 - total);
        if (!wait_w(kAFull0 + st, ph(c >> 1))) break;
        tc_fence_after();
        const uint32_t a_row = tmem + lane_off + kColA + st * 128;
        if (wide) {
          build_p_wide(a_row, q4, r, G2, slot + kSlotG2);
          // O = Q S_{c-1} so far: scale row t by exp(G_t) before MMA2 adds P V
          if (!wait_w(kO3Full0 + st, ph(c >> 1))) break;
          tc_fence_after();
          const float e = exp2f(G2);
          const uint32_t o_row = tmem + lane_off + kColO + st * kDVS;
#pragma unroll 1
          for (int part = 0; part < 4; ++part) {
            uint32_t v[16];
            tmem_ld_32x32b_x16(o_row + 16 * part, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = __float_as_uint(e * __uint_as_float(v[j]));
            tmem_st_32x32b_x16(o_row + 16 * part, v);
          }
        } else {
          build_p(a_row, q4, r, G2);
        }
        tmem_st_wait();
        tc_fence_before();
        warp_arrive(kPFull0 + st);
        warp_arrive(kGFree0 + c % kSlots);
      }
      if (c >= 1 && !output(c - 1, fprev)) break;
      fprev = f;
    }
  } else {
    // ----------------------------------------------------------- state group
    const int q4 = warp & 3;
    const int half = (warp - 8) >> 2;     // which 32 of the 64 state / V columns
    const int r = 32 * q4 + lane;         // state row i (key channel), token row for W V
    const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
    // state rows past the key head size (d_k = 64, 96) stay zero: their K
    // channels are the zero columns the TMA fills in
    const bool row_ok = r < p.DK;
    const size_t st_off = ((size_t)s * p.H + h) * (size_t)p.DK * p.DV +
                          (size_t)(row_ok ? r : 0) * p.DV + (size_t)sl * kDVS + 32 * half;
    uint8_t* sb_row = smem + kOffSb;
    float* final_row = (p.final_state && row_ok) ? p.final_state + st_off : nullptr;
    const float* init_row = (p.init_state && row_ok) ? p.init_state + st_off : nullptr;

    int nsync = 0;  // completions of the group barrier so far
    // W V split of chunk c (this thread: token row r, V columns 32 half .. +31)
    // into bf16 hi and lo (buffers c & 1).  Returns the chunk's total log2 decay.
    auto split_wv = [&](int c, float& total, bool& wide) -> bool {
      const int n = min(kC, len - c * kC);
      if (!wait_w(kGReady0 + c % kSlots, ph(c / kSlots))) return false;
      const float* slot = slot_of(c);
      const float G2r = slot[kSlotG2 + r];
      total = slot[kSlotTotal];
      wide = slot[kSlotWide] != 0.f;
      warp_arrive(kGFree0 + c % kSlots);
      // MMA2(c-2) done; MMA4(c-2) is done too (its S was passed before this call)
      if (c >= 2 && !wait_w(kVtFree0 + (c & 1), ph((c >> 1) - 1))) return false;
      if (!wait_w(kVFull, ph(c))) return false;
      const uint8_t* v_s = smem + kOffV;
      uint8_t* hi_s = smem + kOffVhi + (c & 1) * kTile;
      uint8_t* lo_s = smem + kOffVlo + (c & 1) * kTile;
      const float w = (r < n) ? exp2f(total - G2r) : 0.f;
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        const uint32_t off = sw128_offset(r, 4 * half + cc);
        const uint4 raw = *reinterpret_cast<const uint4*>(v_s + off);
        const uint32_t in[4] = {raw.x, raw.y, raw.z, raw.w};
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x0 = w * bf16lo(in[e]), x1 = w * bf16hi(in[e]);
          hi[e] = pack_bf16x2(x0, x1);
          lo[e] = pack_bf16x2(x0 - bf16lo(hi[e]), x1 - bf16hi(hi[e]));
        }
        *reinterpret_cast<uint4*>(hi_s + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(lo_s + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      fence_proxy_async_smem();
      if (!wide) {
        // the raw V tile is no longer needed (a wide chunk keeps it for MMA2)
        // all of the group is done with it (an mbarrier with a bounded wait, so a
        // group that is aborting cannot hang the others)
        warp_arrive(kStateSync);
        if (!wait_w(kStateSync, ph(nsync++))) return false;
        if (warp == 8 && lane == 0) mbar_arrive(&bars[kVEmpty]);
      }
      warp_arrive(kVtFull0 + (c & 1));
      return true;
    };

    // One pass over this thread's 32 columns of S_c (c = -1: the initial state).
    // Not last: exp(G_L(c+1)) S_c back into TMEM for MMA4(c+1), and its bf16
    // copy S' for MMA3(c+1) (S_c itself when chunk c+1 is wide).  Last: S_c out
    // to the final state.
    auto pass_state = [&](int c, float decay, bool last, bool next_wide) {
#pragma unroll 1
      for (int q = 0; q < 2; ++q) {  // 16 columns at a time
        uint32_t v[16];
        if (c < 0) {
#pragma unroll
          for (int j = 0; j < 16; j += 4) {
            const float4 x = init_row
                                 ? __ldg(reinterpret_cast<const float4*>(init_row + 16 * q + j))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
            v[j] = __float_as_uint(x.x); v[j + 1] = __float_as_uint(x.y);
            v[j + 2] = __float_as_uint(x.z); v[j + 3] = __float_as_uint(x.w);
          }
        } else {
          tmem_ld_32x32b_x16(tmem + lane_off + kColS + 32 * half + 16 * q, v);
          tmem_ld_wait();
        }
        if (last) {
          if (final_row) {
            float4* dst = reinterpret_cast<float4*>(final_row) + 4 * q;
#pragma unroll
            for (int j = 0; j < 4; ++j)
              dst[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                   __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
          }
        } else {
          float sv[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float x = __uint_as_float(v[j]);
            v[j] = __float_as_uint(decay * x);
            sv[j] = next_wide ? x : __uint_as_float(v[j]);
          }
#pragma unroll
          for (int cc = 0; cc < 2; ++cc)
            *reinterpret_cast<uint4*>(sb_row + sw128_offset(r, 4 * half + 2 * q + cc)) =
                make_uint4(pack_bf16x2(sv[8 * cc], sv[8 * cc + 1]),
                           pack_bf16x2(sv[8 * cc + 2], sv[8 * cc + 3]),
                           pack_bf16x2(sv[8 * cc + 4], sv[8 * cc + 5]),
                           pack_bf16x2(sv[8 * cc + 6], sv[8 * cc + 7]));
          tmem_st_32x32b_x16(tmem + lane_off + kColS + 32 * half + 16 * q, v);
        }
      }
      if (!last) tmem_st_wait();
    };

    if (nch == 0) {
      // empty sequence: the final state is the initial state
      if (final_row) {
#pragma unroll 4
        for (int j = 0; j < 32; ++j) final_row[j] = init_row ? init_row[j] : 0.f;
      }
    }
    // iteration c: the W V split of chunk c + 1 first (MMA4(c+1) needs it
    // together with S_c), then the pass over S_c
    for (int c = -1; c < nch; ++c) {
      const bool last = c + 1 == nch;
      float next_total = 0.f;
      bool next_wide = false;
      if (!last && !split_wv(c + 1, next_total, next_wide)) break;
      if (c >= 0) {
        if (!wait_w(kSFull, ph(c))) break;  // S = S_c; MMA3(c) has read S'
        tc_fence_after();
      }
      pass_state(c, last ? 1.f : exp2f(next_total), last, next_wide);
      if (!last) {
        fence_proxy_async_smem();
        tc_fence_before();
        warp_arrive(kSReady);
      }
    }
  }

  if (*abort_flag) {
    // give copies and MMAs that may still be in flight time to land
#pragma unroll 1
    for (int i = 0; i < 1000; ++i) __nanosleep(1000);
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
