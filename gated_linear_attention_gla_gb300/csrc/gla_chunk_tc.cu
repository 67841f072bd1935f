// gla_chunk_tc.cu -- chunked GLA prefill on the 5th-generation tensor cores.
//
// Method: the chunked form of the "i14 Laplace 3B on AWS Trainium2" page
// (section "Challenge 1", Figure 3) with per-token log-decays g.  For a chunk
// of C = 128 tokens, G_t = sum of g over the chunk up to and including t:
//     A   = Q K^T                                       (C x C)
//     P   = A * exp(G_t - G_j) for j <= t, 0 above       (decay-masked, causal)
//     O   = scale * ( P V + diag(exp G_t) Q S )          (intra + running state)
//     S'  = exp(G_last) S + K^T diag(exp(G_last - G_j)) V
//
// One CTA owns one (sequence, head, 64-wide slice of dv) and walks the
// sequence's chunks in order.  The state slice S (dk x 64, fp32) lives in
// tensor memory (TMEM) for the whole sequence: before each chunk the state
// group scales it by exp(G_last) in place, and the chunk's K^T (W V) product
// accumulates straight into it.  Four tensor-core contractions per chunk, all
// bf16 x bf16 -> fp32 into TMEM:
//     MMA1  A   = Q K^T           M=128 (t) N=128 (j) K=dk   A,B K-major
//     MMA4  S  += K^T (W V)       M=dk (i)  N=64      K=128  A,B MN-major
//     MMA3  O2  = Q S_bf16        M=128 (t) N=64      K=dk   B MN-major
//     MMA2  O1  = P V             M=128 (t) N=64      K=128  B MN-major
// W V (W_j = exp(G_last - G_j)) is rounded to bf16 as hi + lo.  The lo term
// only matters through the final state, and only while enough of it survives
// the decay still to come: a chunk whose remaining decay to the end of the
// sequence is below 2^-16 (known two chunks ahead) skips it.  MMA3 reads the
// state through a bf16 copy in shared memory.
//
// The only true recurrence is S_c = exp(G_last) S_{c-1} + dS_c; everything
// else in a chunk overlaps its neighbours.  Roles (16 warps):
//   warp 0       TMA producer: Q, K (two 64-column panels) and the V slice of
//                each chunk into a 2-stage ring, 128-byte swizzled
//   warp 1       TMEM allocator; issues MMA1, MMA4, MMA3 (the "front")
//   warp 2       issues MMA2 (the "back"), so P V never blocks the state chain
//   warp 3       gate warp: prefix sums of g and the per-column decay factors,
//                two chunks ahead, into a 6-slot ring
//   warps 4..11  mask group: the decay-masked P (written over the chunk's K
//                tile, dead once MMA4 has run), then the output of the previous
//                chunk; two warps per TMEM lane quadrant (warp % 4), one for the
//                even and one for the odd 32-column blocks of P and one
//                32-column half of the output
//   warps 12..15 state group: W V split, the in-place decay of S, the bf16
//                copy of S for MMA3, the final state
// TMEM: A 2x128, O1 64, O2 2x64, S 64 = 512 columns.  Every wait on an
// mbarrier is bounded in wall time; on timeout the kernel flags the device
// status word, stops issuing work, releases TMEM and returns.
//
// Decay mask: for a column block (32 columns) strictly below the diagonal
// block of row t, exp(G_t - G_j) = exp(G_t - G_e) * exp(G_e - G_j) with e the
// block's last column; both factors are <= 1 because g <= 0, so the product
// costs two multiplies and cannot overflow.  On the diagonal block the
// reference is the block's first column s, exp(G_s - G_j) >= 1, used when the
// block's decay span is below 2^64; otherwise each element takes its own exp.
#include <cudaTypedefs.h>

#include <mutex>

#include "gla_internal.cuh"
#include "gla_sm100.cuh"

namespace gla {
namespace {

using namespace sm100;

constexpr int kC = 128;        // chunk (tokens)
constexpr int kDK = 128;       // key head size handled by this kernel
constexpr int kDVS = 64;       // value columns per CTA
constexpr int kThreads = 512;  // 16 warps
constexpr int kMaskWarps = 8;
constexpr int kStateWarps = 4;
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kSpanLimit = 64.f;     // log2 span allowed for the diagonal factorization
constexpr float kLoCutoff = -16.f;     // log2 of the remaining decay below which lo is dropped
constexpr int kLookahead = 2;          // chunks the gate warp runs ahead
constexpr int kSlots = 6;              // gate ring depth (>= kLookahead + 3)

// shared memory map (offsets from the 1024-byte-aligned base)
constexpr uint32_t kPanel = kC * 128;                 // 128 rows x 128 B
constexpr uint32_t kQBytes = kPanel * (kDK / 64);     // 32 KB
constexpr uint32_t kKBytes = kPanel * (kDK / 64);     // 32 KB
constexpr uint32_t kVBytes = kPanel;                  // 16 KB (64 columns)
constexpr uint32_t kStageBytes = kQBytes + kKBytes + kVBytes;
constexpr uint32_t kOffVhi = 2 * kStageBytes;
constexpr uint32_t kOffVlo = kOffVhi + kVBytes;
constexpr uint32_t kOffSb = kOffVlo + kVBytes;        // dk rows x 128 B
// gate slot (floats): G2[128] | total, need_lo, -, - | wE[128] | wS[128] | diag_ok[4]
constexpr int kSlotG2 = 0, kSlotTotal = 128, kSlotNeedLo = 129, kSlotWE = 132, kSlotWS = 260,
              kSlotDiag = 388, kSlotFloats = 392;
constexpr uint32_t kOffGate = kOffSb + kDK * 128;
constexpr uint32_t kOffBar = kOffGate + kSlots * kSlotFloats * 4;
constexpr uint32_t kOffMisc = kOffBar + 256;          // tmem base, abort flag
constexpr uint32_t kSmemUsed = kOffMisc + 64;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;     // alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");

// TMEM column map
constexpr uint32_t kColA = 0;      // 2 x 128
constexpr uint32_t kColO1 = 256;   // 64
constexpr uint32_t kColO2 = 320;   // 2 x 64
constexpr uint32_t kColS = 448;    // 64: the running state slice, fp32

enum Bar {
  kFull0 = 0, kFull1, kEmpty0, kEmpty1, kAFull0, kAFull1, kAFree0, kAFree1,
  kPFull, kVtFull, kSFull, kSReady, kSbFull, kSbFree, kOFull, kO1Free,
  kO2Free0, kO2Free1, kO2Full0, kO2Full1, kGReady0, kGFree0 = kGReady0 + kSlots,
  kNumBars = kGFree0 + kSlots
};
static_assert(kNumBars * 8 <= 256, "barrier area");

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
  int B, H, T, DV, nslices;
  unsigned* status;
};

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

template <bool OUTF32>
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
      if (i == kAFree0 || i == kAFree1 || i == kPFull || i == kO1Free || i == kO2Free0 ||
          i == kO2Free1)
        cnt = kMaskWarps;
      if (i == kVtFull || i == kSReady || i == kSbFull) cnt = kStateWarps;
      if (i == kEmpty0 || i == kEmpty1) cnt = 2;  // MMA3 (front) and MMA2 (back) done
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
  const uint32_t tmem = *tmem_slot;
  const uint32_t sbase = smem_u32(smem);

  auto wait = [&](int b, uint32_t parity) -> bool {
    if (*abort_flag) return false;
    if (mbar_wait_bounded(&bars[b], parity, kWaitLimitNs)) return true;
    *abort_flag = 1;
    atomicOr(p.status, kDevTimeout);
    return false;
  };
  // parity of the k-th completion (k = 0, 1, ...) of a barrier
  auto ph = [](int k) -> uint32_t { return static_cast<uint32_t>(k) & 1u; };
  // One arrival for the whole warp, after every lane's prior writes and fences
  // (__syncwarp orders them before lane 0's release-arrive).
  auto warp_arrive = [&](int b) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[b]);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      for (int c = 0; c < nch; ++c) {
        const int st = c & 1;
        if (c >= 2 && !wait(kEmpty0 + st, ph((c >> 1) - 1))) break;
        uint8_t* q_s = smem + st * kStageBytes;
        uint8_t* k_s = q_s + kQBytes;
        uint8_t* v_s = k_s + kKBytes;
        const int row = packed ? (int)(start + (long long)c * kC) : c * kC;
        const int bidx = packed ? 0 : s;
        mbar_arrive_expect_tx(&bars[kFull0 + st], kStageBytes);
#pragma unroll
        for (int pn = 0; pn < kDK / 64; ++pn) {
          tma_load_4d(q_s + pn * kPanel, &tmQ, &bars[kFull0 + st], pn * 64, h, row, bidx);
          tma_load_4d(k_s + pn * kPanel, &tmK, &bars[kFull0 + st], pn * 64, h, row, bidx);
        }
        tma_load_4d(v_s, &tmV, &bars[kFull0 + st], sl * kDVS, h, row, bidx);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------- MMA front: 1, 4, 3
    // Order: MMA1(0); then per chunk c: MMA4(c), MMA3(c), MMA1(c+1), so the
    // next chunk's Q K^T never sits in the tensor pipe ahead of the state chain.
    if (lane == 0) {
      const uint32_t sb = sbase + kOffSb, vhi = sbase + kOffVhi, vlo = sbase + kOffVlo;
      auto mma1 = [&](int c) -> bool {
        const int st = c & 1;
        const uint32_t q_s = sbase + st * kStageBytes;
        const uint32_t k_s = q_s + kQBytes;
        if (!wait(kFull0 + st, ph(c >> 1))) return false;
        if (c >= 2 && !wait(kAFree0 + st, ph((c >> 1) - 1))) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kDK / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
          mma_bf16(tmem + kColA + st * 128, sdesc_sw128(q_s + off, 16, 1024),
                   sdesc_sw128(k_s + off, 16, 1024), kIdQK, kk > 0);
        }
        return true;
      };
      bool ok = nch == 0 || mma1(0);
      for (int c = 0; c < nch && ok; ++c) {
        const int st = c & 1;
        const uint32_t q_s = sbase + st * kStageBytes;
        const uint32_t k_s = q_s + kQBytes;
        if (!wait(kVtFull, ph(c))) break;
        if (!wait(kSReady, ph(c))) break;  // S holds exp(G_last) S_{c-1}
        tc_fence_after();
        const bool need_lo = gate_ring[(c % kSlots) * kSlotFloats + kSlotNeedLo] != 0.f;
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_bf16(tmem + kColS, sdesc_sw128(k_s + kk * 2048, kPanel, 1024),
                   sdesc_sw128(vhi + kk * 2048, kPanel, 1024), kIdKV, 1);
        if (need_lo) {
#pragma unroll
          for (int kk = 0; kk < kC / 16; ++kk)
            mma_bf16(tmem + kColS, sdesc_sw128(k_s + kk * 2048, kPanel, 1024),
                     sdesc_sw128(vlo + kk * 2048, kPanel, 1024), kIdKV, 1);
        }
        mma_commit(&bars[kSFull]);         // S = S_c
        mma_commit(&bars[kAFull0 + st]);  // A ready and K no longer read: P may overwrite K
        if (!wait(kSbFull, ph(c))) break;
        if (c >= 2 && !wait(kO2Free0 + st, ph((c >> 1) - 1))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kDK / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
          mma_bf16(tmem + kColO2 + st * kDVS, sdesc_sw128(q_s + off, 16, 1024),
                   sdesc_sw128(sb + kk * 2048, kPanel, 1024), kIdQS, kk > 0);
        }
        mma_commit(&bars[kSbFree]);        // S_{c-1} (bf16) read
        mma_commit(&bars[kO2Full0 + st]);  // O2(c) complete
        mma_commit(&bars[kEmpty0 + st]);   // Q(c) no longer read
        if (c + 1 < nch) ok = mma1(c + 1);
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------- MMA back: 2
    if (lane == 0) {
      for (int c = 0; c < nch; ++c) {
        const int st = c & 1;
        const uint32_t p_s = sbase + st * kStageBytes + kQBytes;  // P over the K tile
        const uint32_t v_s = p_s + kKBytes;
        if (!wait(kPFull, ph(c))) break;
        if (c >= 1 && !wait(kO1Free, ph(c - 1))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
          mma_bf16(tmem + kColO1, sdesc_sw128(p_s + off, 16, 1024),
                   sdesc_sw128(v_s + kk * 2048, kPanel, 1024), kIdPV, kk > 0);
        }
        mma_commit(&bars[kOFull]);
        mma_commit(&bars[kEmpty0 + st]);
      }
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------- gate warp
    // lane l owns tokens 4l .. 4l+3 of each chunk
    auto load4 = [&](int c, float (&gv)[4]) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int t = c * kC + 4 * lane + i;
        gv[i] = (c < nch && t < len) ? fmaxf(__ldg(p.g + (start + t) * p.H + h), -kGateClamp)
                                     : 0.f;
      }
    };
    float totals[kLookahead + 1];  // chunk totals (log2) of chunks c-kLookahead .. c
#pragma unroll
    for (int i = 0; i <= kLookahead; ++i) totals[i] = 0.f;
    // publish chunk d: remaining decay after it decides whether MMA4 needs lo
    auto publish = [&](int d, float remaining) {
      float* slot = gate_ring + (d % kSlots) * kSlotFloats;
      if (lane == 0) slot[kSlotNeedLo] = (remaining < kLoCutoff) ? 0.f : 1.f;
      warp_arrive(kGReady0 + d % kSlots);
    };
    float gnext[4];
    load4(0, gnext);
    bool ok = true;
    for (int c = 0; c < nch; ++c) {
      float gv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) gv[i] = gnext[i];
      load4(c + 1, gnext);
      if (c >= kSlots && !wait(kGFree0 + c % kSlots, ph(c / kSlots - 1))) { ok = false; break; }
      float* slot = gate_ring + (c % kSlots) * kSlotFloats;
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
      *reinterpret_cast<float4*>(slot + kSlotG2 + 4 * lane) = make_float4(G2[0], G2[1], G2[2], G2[3]);
      // block of my columns: 32 * (lane / 8) .. +31; its first column is lane 8k's
      // first token, its last column is lane 8k+7's last token
      const float Gb = __shfl_sync(0xffffffffu, G2[0], lane & ~7);
      const float Ge = __shfl_sync(0xffffffffu, G2[3], lane | 7);
      float wE[4], wS[4], span = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        wE[i] = exp2f(Ge - G2[i]);
        wS[i] = exp2f(Gb - G2[i]);
        span = fmaxf(span, fabsf(Gb - G2[i]));
      }
      *reinterpret_cast<float4*>(slot + kSlotWE + 4 * lane) = make_float4(wE[0], wE[1], wE[2], wE[3]);
      *reinterpret_cast<float4*>(slot + kSlotWS + 4 * lane) = make_float4(wS[0], wS[1], wS[2], wS[3]);
#pragma unroll
      for (int off = 1; off < 8; off <<= 1)
        span = fmaxf(span, __shfl_xor_sync(0xffffffffu, span, off));
      if ((lane & 7) == 0) reinterpret_cast<int*>(slot)[kSlotDiag + (lane >> 3)] =
          span < kSpanLimit ? 1 : 0;
      if (lane == 0) slot[kSlotTotal] = total;
#pragma unroll
      for (int i = 0; i < kLookahead; ++i) totals[i] = totals[i + 1];
      totals[kLookahead] = total;
      if (c >= kLookahead) {
        float rem = 0.f;
#pragma unroll
        for (int i = 1; i <= kLookahead; ++i) rem += totals[i];
        publish(c - kLookahead, rem);
      }
    }
    if (ok && !*abort_flag) {
      // the last kLookahead chunks: the remaining decay is known exactly
      for (int d = max(0, nch - kLookahead); d < nch; ++d) {
        float rem = 0.f;
#pragma unroll
        for (int i = 0; i <= kLookahead; ++i) {
          const int chunk = nch - 1 - kLookahead + i;  // totals[i] belongs to this chunk
          if (chunk > d) rem += totals[i];
        }
        publish(d, rem);
      }
    }
  } else if (warp < 12) {
    // ------------------------------------------------------------ mask group
    const int q4 = warp & 3;
    const int mh = (warp - 4) >> 2;       // column-block parity, and output half
    const int r = 32 * q4 + lane;         // token row
    const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
    const float scale = p.scale;

    // output of chunk c: o = scale (O1 + exp(G_t) O2[c & 1]), columns 32 mh .. +31,
    // in two 16-column passes
    auto output = [&](int c, float G2t) -> bool {
      if (!wait(kOFull, ph(c))) return false;                  // MMA2(c): O1
      if (!wait(kO2Full0 + (c & 1), ph(c >> 1))) return false; // MMA3(c): O2
      tc_fence_after();
      const int n = min(kC, len - c * kC);
      const float se = scale * exp2f(G2t);
      const long long rowbase = start + (long long)c * kC;
      const size_t off =
          ((size_t)(rowbase + r) * p.H + h) * p.DV + (size_t)sl * kDVS + 32 * mh;
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        uint32_t o1[16], o2[16];
        tmem_ld_32x32b_x16(tmem + lane_off + kColO1 + 32 * mh + 16 * part, o1);
        tmem_ld_32x32b_x16(tmem + lane_off + kColO2 + (c & 1) * kDVS + 32 * mh + 16 * part, o2);
        tmem_ld_wait();
        if (part == 1) {
          tc_fence_before();
          warp_arrive(kO1Free);
          warp_arrive(kO2Free0 + (c & 1));
        }
        float o[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          o[j] = fmaf(se, __uint_as_float(o2[j]), scale * __uint_as_float(o1[j]));
        if (r < n) {
          if constexpr (OUTF32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + off) + 4 * part;
#pragma unroll
            for (int j = 0; j < 4; ++j)
              dst[j] = make_float4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
          } else {
            uint4* dst =
                reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + off) + 2 * part;
#pragma unroll
            for (int j = 0; j < 2; ++j)
              dst[j] = make_uint4(pack_bf16x2(o[8 * j], o[8 * j + 1]),
                                  pack_bf16x2(o[8 * j + 2], o[8 * j + 3]),
                                  pack_bf16x2(o[8 * j + 4], o[8 * j + 5]),
                                  pack_bf16x2(o[8 * j + 6], o[8 * j + 7]));
          }
        }
      }
      return true;
    };

    float G2prev = 0.f;
    bool ok = true;
    for (int c = 0; c < nch; ++c) {
      const int st = c & 1;
      const float* slot = gate_ring + (c % kSlots) * kSlotFloats;
      uint8_t* p_s = smem + st * kStageBytes + kQBytes;  // P over the K tile
      if (!wait(kGReady0 + c % kSlots, ph(c / kSlots))) { ok = false; break; }
      const float G2 = slot[kSlotG2 + r];
      if (!wait(kAFull0 + st, ph(c >> 1))) { ok = false; break; }
      tc_fence_after();
      // this warp's blocks: cb = mh and cb = mh + 2; blocks above the diagonal
      // block (cb > q4) are zero and need no TMEM read
      const uint32_t a_base = tmem + lane_off + kColA + st * 128;
      const float* G2s = slot + kSlotG2;
      uint32_t a[2][32];
#pragma unroll
      for (int i = 0; i < 2; ++i)
        if (mh + 2 * i <= q4) tmem_ld_32x32b_x32(a_base + 32 * (mh + 2 * i), a[i]);
      tmem_ld_wait();
      tc_fence_before();
      warp_arrive(kAFree0 + st);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int cb = mh + 2 * i;
        uint32_t pk[16];
        if (cb < q4 || (cb == q4 && reinterpret_cast<const int*>(slot)[kSlotDiag + cb] != 0)) {
          // factorised decay: u (per row and block) times w (per column)
          const bool diag = (cb == q4);
          const float u = exp2f(G2 - (diag ? G2s[32 * cb] : G2s[32 * cb + 31]));
          const float* wv = slot + (diag ? kSlotWS : kSlotWE) + 32 * cb;
#pragma unroll
          for (int jj = 0; jj < 32; jj += 4) {
            const float4 w4 = *reinterpret_cast<const float4*>(wv + jj);
            const int j = 32 * cb + jj;
            float p0 = __uint_as_float(a[i][jj]) * (u * w4.x);
            float p1 = __uint_as_float(a[i][jj + 1]) * (u * w4.y);
            float p2 = __uint_as_float(a[i][jj + 2]) * (u * w4.z);
            float p3 = __uint_as_float(a[i][jj + 3]) * (u * w4.w);
            if (diag) {
              p0 = (j <= r) ? p0 : 0.f;
              p1 = (j + 1 <= r) ? p1 : 0.f;
              p2 = (j + 2 <= r) ? p2 : 0.f;
              p3 = (j + 3 <= r) ? p3 : 0.f;
            }
            pk[jj / 2] = pack_bf16x2(p0, p1);
            pk[jj / 2 + 1] = pack_bf16x2(p2, p3);
          }
        } else if (cb == q4) {
          // diagonal block with a decay span too wide to factorise: one exp each
#pragma unroll
          for (int jj = 0; jj < 32; jj += 2) {
            const int j = 32 * cb + jj;
            const float p0 = (j <= r) ? __uint_as_float(a[i][jj]) * exp2f(G2 - G2s[j]) : 0.f;
            const float p1 =
                (j + 1 <= r) ? __uint_as_float(a[i][jj + 1]) * exp2f(G2 - G2s[j + 1]) : 0.f;
            pk[jj / 2] = pack_bf16x2(p0, p1);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) pk[e] = 0u;
        }
        uint8_t* panel = p_s + (cb >> 1) * kPanel;
#pragma unroll
        for (int m = 0; m < 4; ++m)
          *reinterpret_cast<uint4*>(panel + sw128_offset(r, (cb & 1) * 4 + m)) =
              make_uint4(pk[4 * m], pk[4 * m + 1], pk[4 * m + 2], pk[4 * m + 3]);
      }
      fence_proxy_async_smem();
      warp_arrive(kPFull);
      // output of the previous chunk (its MMA2 ran while P was built)
      if (c >= 1) {
        ok = output(c - 1, G2prev);
        warp_arrive(kGFree0 + (c - 1) % kSlots);
        if (!ok) break;
      }
      G2prev = G2;
    }
    if (ok && nch >= 1 && output(nch - 1, G2prev))
      warp_arrive(kGFree0 + (nch - 1) % kSlots);
  } else {
    // ----------------------------------------------------------- state group
    const int q4 = warp & 3;
    const int r = 32 * q4 + lane;         // state row i (key channel), token row for W V
    const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
    const size_t st_off = ((size_t)s * p.H + h) * (size_t)kDK * p.DV + (size_t)r * p.DV +
                          (size_t)sl * kDVS;
    uint8_t* sb_row = smem + kOffSb;

    // S_c (in TMEM) -> bf16 copy for MMA3 (optional) and, scaled by `decay`,
    // back into TMEM for the next MMA4 (optional) or to the final state.
    auto pass_state = [&](float decay, bool to_sb, bool rescale, float* final_row) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {  // 16 columns at a time
        uint32_t v[16];
        tmem_ld_32x32b_x16(tmem + lane_off + kColS + 16 * q, v);
        tmem_ld_wait();
        if (to_sb) {
#pragma unroll
          for (int cc = 0; cc < 2; ++cc)
            *reinterpret_cast<uint4*>(sb_row + sw128_offset(r, 2 * q + cc)) = make_uint4(
                pack_bf16x2(__uint_as_float(v[8 * cc]), __uint_as_float(v[8 * cc + 1])),
                pack_bf16x2(__uint_as_float(v[8 * cc + 2]), __uint_as_float(v[8 * cc + 3])),
                pack_bf16x2(__uint_as_float(v[8 * cc + 4]), __uint_as_float(v[8 * cc + 5])),
                pack_bf16x2(__uint_as_float(v[8 * cc + 6]), __uint_as_float(v[8 * cc + 7])));
        }
        if (final_row) {
          float4* dst = reinterpret_cast<float4*>(final_row) + 4 * q;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            dst[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                 __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
        }
        if (rescale) {
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = __float_as_uint(decay * __uint_as_float(v[j]));
          tmem_st_32x32b_x16(tmem + lane_off + kColS + 16 * q, v);
        }
      }
      if (rescale) tmem_st_wait();
    };

    // W V split of chunk c into bf16 hi (+ lo); thread r handles token row r.
    // Returns the chunk's total log2 decay through `total`.
    auto split_wv = [&](int c, float& total) -> bool {
      const int st = c & 1;
      const int n = min(kC, len - c * kC);
      if (!wait(kGReady0 + c % kSlots, ph(c / kSlots))) return false;
      const float* slot = gate_ring + (c % kSlots) * kSlotFloats;
      const float G2r = slot[kSlotG2 + r];
      total = slot[kSlotTotal];
      const bool need_lo = slot[kSlotNeedLo] != 0.f;
      warp_arrive(kGFree0 + c % kSlots);
      if (!wait(kFull0 + st, ph(c >> 1))) return false;
      const uint8_t* v_s = smem + st * kStageBytes + kQBytes + kKBytes;
      const float w = (r < n) ? exp2f(total - G2r) : 0.f;
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        const uint32_t off = sw128_offset(r, cc);
        const uint4 raw = *reinterpret_cast<const uint4*>(v_s + off);
        const uint32_t in[4] = {raw.x, raw.y, raw.z, raw.w};
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x0 = w * bf16lo(in[e]), x1 = w * bf16hi(in[e]);
          hi[e] = pack_bf16x2(x0, x1);
          lo[e] = pack_bf16x2(x0 - bf16lo(hi[e]), x1 - bf16hi(hi[e]));
        }
        *reinterpret_cast<uint4*>(smem + kOffVhi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        if (need_lo)
          *reinterpret_cast<uint4*>(smem + kOffVlo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      fence_proxy_async_smem();
      warp_arrive(kVtFull);
      return true;
    };

    bool ok = true;
    float* final_row = p.final_state ? p.final_state + st_off : nullptr;
    if (nch == 0) {
      // empty sequence: the final state is the initial state
      if (final_row) {
#pragma unroll 4
        for (int j = 0; j < kDVS; ++j) final_row[j] = p.init_state ? p.init_state[st_off + j] : 0.f;
      }
    } else {
      // S_{-1} = initial state: bf16 copy for MMA3(0); TMEM gets exp(G_last(0)) S_{-1}
      float total = 0.f;
      ok = split_wv(0, total);
      if (ok) {
        const float decay = exp2f(total);
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // 16 columns at a time
          uint32_t v[16];
#pragma unroll
          for (int j = 0; j < 16; j += 4) {
            const float4 x = p.init_state
                                 ? __ldg(reinterpret_cast<const float4*>(p.init_state + st_off +
                                                                         16 * q + j))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
            v[j] = __float_as_uint(x.x); v[j + 1] = __float_as_uint(x.y);
            v[j + 2] = __float_as_uint(x.z); v[j + 3] = __float_as_uint(x.w);
          }
#pragma unroll
          for (int cc = 0; cc < 2; ++cc)
            *reinterpret_cast<uint4*>(sb_row + sw128_offset(r, 2 * q + cc)) = make_uint4(
                pack_bf16x2(__uint_as_float(v[8 * cc]), __uint_as_float(v[8 * cc + 1])),
                pack_bf16x2(__uint_as_float(v[8 * cc + 2]), __uint_as_float(v[8 * cc + 3])),
                pack_bf16x2(__uint_as_float(v[8 * cc + 4]), __uint_as_float(v[8 * cc + 5])),
                pack_bf16x2(__uint_as_float(v[8 * cc + 6]), __uint_as_float(v[8 * cc + 7])));
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = __float_as_uint(decay * __uint_as_float(v[j]));
          tmem_st_32x32b_x16(tmem + lane_off + kColS + 16 * q, v);
        }
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        warp_arrive(kSbFull);
        warp_arrive(kSReady);
      }
      for (int c = 0; c < nch && ok; ++c) {
        if (!wait(kSFull, ph(c))) { ok = false; break; }  // S = S_c
        tc_fence_after();
        if (c + 1 < nch) {
          // W V of the next chunk first (the W V buffers are free now)
          if (!split_wv(c + 1, total)) { ok = false; break; }
          if (!wait(kSbFree, ph(c))) { ok = false; break; }  // MMA3(c) has read S_{c-1}
          pass_state(exp2f(total), true, true, nullptr);
          fence_proxy_async_smem();
          tc_fence_before();
          warp_arrive(kSbFull);
          warp_arrive(kSReady);
        } else {
          pass_state(1.f, false, false, final_row);
        }
      }
    }
  }

  if (*abort_flag) {
    // give copies and MMAs that may still be in flight time to land
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
  return !a.fp32_io && !a.vector_gate && a.chunk == kC && a.dk == kDK &&
         (a.dv == 64 || a.dv == 128);
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
  p.B = a.B; p.H = a.H; p.T = a.T; p.DV = a.dv; p.nslices = a.dv / kDVS;
  p.status = a.status;
  const long long ctas = (long long)a.B * a.H * p.nslices;
  if (a.fp32_out) {
    auto kern = chunk_tc_kernel<true>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)ctas, kThreads, kSmemBytes, stream>>>(mq, mk, mv, p);
  } else {
    auto kern = chunk_tc_kernel<false>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)ctas, kThreads, kSmemBytes, stream>>>(mq, mk, mv, p);
  }
  return cudaGetLastError();
}

}  // namespace gla
