// gla_chunk_split.cu -- chunked GLA prefill in two passes on the 5th-generation
// tensor cores: a state pass that walks each (sequence, head)'s chunks in order,
// and an output pass whose (sequence, head, chunk) tiles are independent.
//
// Method: the chunked form of the "i14 Laplace 3B on AWS Trainium2" page
// (section "Challenge 1", Figure 3): the intra-chunk parts of all chunks can run
// in parallel and only the state update is sequential.  With G_t the sum of the
// log-decays over the chunk up to and including token t (in log2 units) and L
// the chunk's last token:
//     S_c    = 2^{G_L} S_{c-1} + K^T (W V),        W_j = 2^{G_L - G_j}  (<= 1)
//     o_t    = scale * 2^{G_t - G_L} * ( Q S' + P' V )_t,   S' = 2^{G_L} S_{c-1},
//     P'_tj  = (Q K^T)_tj W_j   for j <= t (causal mask, diagonal kept).
// This is exact while the chunk's decay span 2^{G_first - G_L} stays inside
// 2^96; a wider chunk takes the explicit form
//     o_t    = scale * ( 2^{G_t} (Q S_{c-1})_t + sum_{j<=t} (Q K^T)_tj 2^{G_t - G_j} V_j ).
//
// Chunks are aligned to the END of each sequence: chunk c covers tokens
// [off + 128 c, off + 128 c + 128) with off = len - 128 * nch, so every chunk
// but the first holds 128 tokens (the first holds 1 to 128).  The chunking
// changes only the rounding of the result.
//
// Pass 1, chunk_state_kernel -- one CTA per (sequence, head, 64 value columns).
//   For each chunk: U = K^T (W V) on tcgen05 (W V as bf16 hi + lo, so U is
//   exact to fp32 accumulation), S = 2^{G_L} S + U in registers (fp32), and for
//   the NEXT chunk c + 1 the tile S'_c = 2^{G_L(c+1)} S_c (S_c itself when chunk
//   c + 1 is wide) written into the output rows of chunk c + 1, which that
//   chunk's output later overwrites: the library needs no workspace.  The tile
//   is stored in block floating point: per state row and 64 value columns an
//   exponent E (the smallest with |x| < 2^E) and int16 mantissas
//   m = round(x 2^{14 - E}); E's eight bits replace the lowest bit of the row's
//   first eight mantissas.  That is 2^-14 of the row's largest value, against
//   bf16's 2^-8 of each value, in the 2 bytes per value the output rows offer.
//   The last chunk's state goes to the final state (fp32).
// Pass 2, chunk_out_kernel -- persistent CTAs over (sequence, head, chunk,
//   value slice) tiles.  Per tile: the staged state tile (chunk 0: the initial
//   state, converted directly) decoded into bf16 hi + lo; MMA1 A = Q K^T;
//   P' = A W (or the explicit decays) as bf16 hi + lo in TMEM; MMA3
//   O = Q S'hi + Q S'lo; MMA2 O += P'hi V + P'lo V (V exact); the output row
//   scale * 2^{G_t - G_L} O_t.  With every operand exact or split into hi + lo,
//   the only roundings left are the fp32 accumulations and the state tile's
//   block format.
// When the final state overwrites the initial state (the same buffer), the
// output pass runs its chunk-0 tiles first, then the state pass, then the rest.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "gla_internal.cuh"
#include "gla_sm100.cuh"

namespace gla {
namespace {

using namespace sm100;

constexpr int kC = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kWideSpan = 96.f;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr uint32_t kPanel = kC * 128;             // 128 rows x 128 B = 16 KB
constexpr int kBfpMant = 14;                      // |mantissa| <= 2^14
constexpr int kBfpEmin = -100;

struct SplitParams {
  const float* g;
  float scale;
  const float* init_state;
  void* out;
  float* final_state;
  const int32_t* cu_seqlens;
  int B, H, T, DK, DV;
  int dvs;           // output-pass slice width (64 or 128); also fixes the staging layout
  int osz;           // bytes per output element (2 or 4)
  int out_v8;        // out is 32-byte aligned: 256-bit stores
  int out_reversed;  // token t of a sequence stored at row len - 1 - t
  // output pass, DOT variant: dot_out[row, h] += dot_sign * (out row . dot_rows row)
  const __nv_bfloat16* dot_rows;
  float* dot_out;
  float dot_sign;
  int mode;          // output pass: 0 every chunk, 1 chunk 0 only, 2 chunks >= 1 only
  unsigned* status;
};

// ------------------------------------------------------------ shared helpers
__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// first output row of the 128-row block chunk c (c >= 1, a full chunk) occupies
__device__ __forceinline__ long long block_row(long long start, int len, int off, int c,
                                               bool reversed) {
  const long long t0 = (long long)off + (long long)c * kC;
  return reversed ? start + len - kC - t0 : start + t0;
}

// bf16 column of value column j in the staging layout: the tile of output
// slice j / dvs sits at the start of that slice's own output bytes
__device__ __forceinline__ int stage_col(int j, int dvs, int osz) {
  return (osz / 2) * dvs * (j / dvs) + (j % dvs);
}

// Bounded mbarrier wait that also gives up once the CTA is aborting.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity,
                                         volatile int* abort_flag, unsigned* status) {
  if (*abort_flag) return false;
  if (mbar_try_wait(bar, parity, 20000u)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity, 20000u)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      atomicOr(status, kDevTimeout);
      return false;
    }
  }
}

// On abort: wait (bounded) until the last of `issued` transactions counted on
// `bar` has landed, so that no copy into shared memory is in flight when the
// CTA exits.
__device__ __forceinline__ void drain_bar(uint64_t* bar, int issued) {
  if (issued > 0) (void)mbar_wait_bounded(bar, (uint32_t)(issued - 1) & 1u, kWaitLimitNs);
}

__device__ __forceinline__ uint32_t ph(int k) { return static_cast<uint32_t>(k) & 1u; }

// ===================================================================== pass 1
constexpr int kStThreads = 384;  // 12 warps
constexpr int kStStages = 3;
constexpr int kStSW = 64;        // value columns per CTA
constexpr int kStSlots = 4;
constexpr int kStSlotFloats = 132;  // G2[128] | total, wide, -, -
// stage: K (two 64-channel panels) | V, overwritten by (W V) hi | (W V) lo
constexpr uint32_t kStOffK = 0, kStOffV = 2 * kPanel, kStOffLo = 3 * kPanel;
constexpr uint32_t kStStageBytes = 4 * kPanel;  // 64 KB
constexpr uint32_t kStOffSlots = kStStages * kStStageBytes;
constexpr uint32_t kStOffBar = kStOffSlots + kStSlots * kStSlotFloats * 4;
enum StBar {
  kStKVFull = 0, kStKVEmpty = kStKVFull + kStStages, kStWVReady = kStKVEmpty + kStStages,
  kStUFull = kStWVReady + kStStages, kStUFree = kStUFull + 2, kStGReady = kStUFree + 2,
  kStGFree = kStGReady + kStSlots, kStDrain = kStGFree + kStSlots, kStNumBars
};
constexpr uint32_t kStOffMisc = kStOffBar + kStNumBars * 8;
constexpr uint32_t kStSmemBytes = kStOffMisc + 16 + 1024;
static_assert(kStSmemBytes <= 232448, "shared memory budget");
constexpr uint32_t kStTmemCols = 128;  // U, double-buffered, 64 columns each
constexpr uint32_t kIdKV = idesc_bf16(128, kStSW, true, true);

__global__ void __launch_bounds__(kStThreads, 1)
chunk_state_kernel(const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const SplitParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kStOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kStOffMisc + 4);
  float* slots = reinterpret_cast<float*>(smem + kStOffSlots);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nsl = p.DV / kStSW;
  const int sl = blockIdx.x % nsl;
  const int h = (blockIdx.x / nsl) % p.H;
  const int s = blockIdx.x / (nsl * p.H);
  long long start;
  int len;
  if (!seq_bounds(p.cu_seqlens, s, p.B, p.T, &start, &len, p.status)) return;
  const int nch = (len + kC - 1) / kC;
  const int off = len - kC * nch;
  const bool packed = p.cu_seqlens != nullptr;

  if (tid == 0) {
    for (int i = 0; i < kStNumBars; ++i) {
      uint32_t cnt = 1;
      if (i >= kStWVReady && i < kStWVReady + kStStages) cnt = 4;
      if (i == kStUFree || i == kStUFree + 1) cnt = 4;
      if (i >= kStGFree && i < kStGFree + kStSlots) cnt = 8;  // split (4) + scan (4) warps
      mbar_init(&bars[i], cnt);
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kStTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sbase = smem_u32(smem);

  auto wait = [&](int b, uint32_t parity) -> bool {
    return wait_bar(&bars[b], parity, abort_flag, p.status);
  };
  auto wait_w = [&](int b, uint32_t parity) -> bool {
    return __all_sync(0xffffffffu, wait(b, parity));
  };
  auto warp_arrive = [&](int b) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[b]);
  };
  auto slot_of = [&](int c) -> float* { return slots + (c % kStSlots) * kStSlotFloats; };

  int issued[kStStages] = {0, 0, 0};  // producer lane 0: loads per stage barrier
  bool mma_issued = false;

  if (warp == 0) {
    // ----------------------------------------------- producer: gate sums, TMA
    const int bidx = packed ? 0 : s;
    auto load4 = [&](int c, float (&gv)[4]) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int t = off + c * kC + 4 * lane + i;
        gv[i] = (c < nch && t >= 0) ? __ldg(p.g + (start + t) * p.H + h) : 0.f;
      }
    };
    float gnext[4];
    load4(0, gnext);
    for (int c = 0; c < nch; ++c) {
      float gv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) gv[i] = fmaxf(gnext[i], -kGateClamp);
      load4(c + 1, gnext);
      bool ok = true;
      if (c >= kStSlots && !wait(kStGFree + c % kStSlots, ph(c / kStSlots - 1))) ok = false;
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
      float* slot = slot_of(c);
      float G2[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) G2[i] = (excl + run[i]) * kLog2e;
      *reinterpret_cast<float4*>(slot + 4 * lane) = make_float4(G2[0], G2[1], G2[2], G2[3]);
      const int pad = c == 0 ? -off : 0;  // first valid row of the chunk
      const float first = __shfl_sync(0xffffffffu, G2[pad & 3], pad >> 2);
      if (lane == 0) {
        slot[128] = total;
        slot[129] = (first - total > kWideSpan) ? 1.f : 0.f;
      }
      warp_arrive(kStGReady + c % kStSlots);
      if (lane == 0) {
        const int st = c % kStStages;
        const int row = (int)((packed ? start : 0) + off + (long long)c * kC);
        if (c >= kStStages && !wait(kStKVEmpty + st, ph(c / kStStages - 1))) ok = false;
        if (ok) {
          uint8_t* stage = smem + st * kStStageBytes;
          mbar_arrive_expect_tx(&bars[kStKVFull + st], 3 * kPanel);
          tma_load_4d(stage + kStOffK, &tmK, &bars[kStKVFull + st], 0, h, row, bidx);
          tma_load_4d(stage + kStOffK + kPanel, &tmK, &bars[kStKVFull + st], 64, h, row, bidx);
          tma_load_4d(stage + kStOffV, &tmV, &bars[kStKVFull + st], sl * kStSW, h, row, bidx);
          ++issued[st];
        }
      }
      if (__any_sync(0xffffffffu, !ok)) break;
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA: U = K^T (W V)
    if (lane == 0) {
      for (int c = 0; c < nch; ++c) {
        const int st = c % kStStages, b = c & 1;
        if (!wait(kStKVFull + st, ph(c / kStStages))) break;
        if (!wait(kStWVReady + st, ph(c / kStStages))) break;
        if (c >= 2 && !wait(kStUFree + b, ph(c / 2 - 1))) break;
        tc_fence_after();
        const uint32_t stage = sbase + st * kStStageBytes;
        const uint64_t kd = sdesc_sw128(stage + kStOffK, kPanel, 1024);
        const uint64_t hd = sdesc_sw128(stage + kStOffV, kPanel, 1024);
        const uint64_t ld = sdesc_sw128(stage + kStOffLo, kPanel, 1024);
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_bf16(tmem + kStSW * b, desc_add(kd, kk * 2048), desc_add(hd, kk * 2048), kIdKV,
                   kk > 0);
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_bf16(tmem + kStSW * b, desc_add(kd, kk * 2048), desc_add(ld, kk * 2048), kIdKV, 1);
        mma_commit(&bars[kStUFull + b]);
        mma_commit(&bars[kStKVEmpty + st]);
        mma_issued = true;
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // --------------------------------------- (W V) hi / lo, token row r each
    const int r = 32 * (warp - 4) + lane;
    for (int c = 0; c < nch; ++c) {
      const int st = c % kStStages;
      if (!wait_w(kStGReady + c % kStSlots, ph(c / kStSlots))) break;
      const float* slot = slot_of(c);
      const float G2r = slot[r], total = slot[128];
      if (!wait_w(kStKVFull + st, ph(c / kStStages))) break;
      const bool valid = off + c * kC + r >= 0;
      const float w = valid ? exp2f(total - G2r) : 0.f;
      uint8_t* v_s = smem + st * kStStageBytes + kStOffV;
      uint8_t* lo_s = smem + st * kStStageBytes + kStOffLo;
#pragma unroll 2
      for (int cc = 0; cc < 8; ++cc) {
        const uint32_t o = sw128_offset(r, cc);
        const uint4 raw = *reinterpret_cast<const uint4*>(v_s + o);
        const uint32_t in[4] = {raw.x, raw.y, raw.z, raw.w};
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x0 = w * bf16lo(in[e]), x1 = w * bf16hi(in[e]);
          hi[e] = pack_bf16x2(x0, x1);
          lo[e] = pack_bf16x2(x0 - bf16lo(hi[e]), x1 - bf16hi(hi[e]));
        }
        *reinterpret_cast<uint4*>(v_s + o) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(lo_s + o) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      fence_proxy_async_smem();
      warp_arrive(kStWVReady + st);
      warp_arrive(kStGFree + c % kStSlots);
    }
  } else if (warp >= 8) {
    // -------------------------- scan: state row i, 64 value columns, registers
    const int q4 = warp & 3;
    const int i = 32 * q4 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
    const bool row_ok = i < p.DK;
    const size_t st_off = ((size_t)s * p.H + h) * (size_t)p.DK * p.DV +
                          (size_t)(row_ok ? i : 0) * p.DV + (size_t)sl * kStSW;
    float S[kStSW];
    if (p.init_state && row_ok) {
      const float4* src = reinterpret_cast<const float4*>(p.init_state + st_off);
#pragma unroll
      for (int j = 0; j < kStSW / 4; ++j) {
        const float4 x = __ldg(src + j);
        S[4 * j] = x.x; S[4 * j + 1] = x.y; S[4 * j + 2] = x.z; S[4 * j + 3] = x.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < kStSW; ++j) S[j] = 0.f;
    }
    const int col0 = stage_col(sl * kStSW, p.dvs, p.osz);
    bool ok = true;
    for (int c = 0; c < nch && ok; ++c) {
      const int b = c & 1;
      if (!wait_w(kStGReady + c % kStSlots, ph(c / kStSlots))) { ok = false; break; }
      const float decay = exp2f(slot_of(c)[128]);
      if (!wait_w(kStUFull + b, ph(c >> 1))) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t u[32];
        tmem_ld_32x32b_x32(tmem + lane_off + kStSW * b + 32 * half, u);
        tmem_ld_wait_x32(u);
#pragma unroll
        for (int j = 0; j < 32; ++j)
          S[32 * half + j] = fmaf(decay, S[32 * half + j], __uint_as_float(u[j]));
      }
      tc_fence_before();
      warp_arrive(kStUFree + b);
      if (c + 1 < nch) {
        if (!wait_w(kStGReady + (c + 1) % kStSlots, ph((c + 1) / kStSlots))) { ok = false; break; }
        const float* nslot = slot_of(c + 1);
        const float f = nslot[129] != 0.f ? 1.f : exp2f(nslot[128]);
        // S'_c for chunk c + 1 in block floating point
        float mx = 0.f;
#pragma unroll
        for (int j = 0; j < kStSW; ++j) mx = fmaxf(mx, fabsf(f * S[j]));
        int E = (int)((__float_as_uint(mx) >> 23) & 0xffu) - 126;
        E = min(max(E, kBfpEmin), 127);
        const float up = __uint_as_float((uint32_t)(kBfpMant - E + 127) << 23);  // 2^(14 - E)
        const uint32_t ebits = (uint32_t)(E + 128);
        if (row_ok) {
          const long long row = block_row(start, len, off, c + 1, p.out_reversed) + i;
          uint8_t* dst = static_cast<uint8_t*>(p.out) +
                         ((size_t)row * p.H + h) * (size_t)p.DV * p.osz + 2 * (size_t)col0;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int j = 8 * q + 2 * e;
              int m0 = __float2int_rn(f * S[j] * up);
              int m1 = __float2int_rn(f * S[j + 1] * up);
              if (q == 0) {
                m0 = (m0 & ~1) | (int)((ebits >> (2 * e)) & 1u);
                m1 = (m1 & ~1) | (int)((ebits >> (2 * e + 1)) & 1u);
              }
              w[e] = ((uint32_t)m0 & 0xffffu) | ((uint32_t)m1 << 16);
            }
            reinterpret_cast<uint4*>(dst)[q] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      warp_arrive(kStGFree + c % kStSlots);
    }
    if (ok && p.final_state && row_ok) {
      float4* dst = reinterpret_cast<float4*>(p.final_state + st_off);
#pragma unroll
      for (int j = 0; j < kStSW / 4; ++j)
        dst[j] = make_float4(S[4 * j], S[4 * j + 1], S[4 * j + 2], S[4 * j + 3]);
    }
  }

  if (*abort_flag) {
    // let every copy into this CTA's shared memory and every MMA land first
    if (warp == 0 && lane == 0)
      for (int st = 0; st < kStStages; ++st) drain_bar(&bars[kStKVFull + st], issued[st]);
    if (warp == 1 && lane == 0 && mma_issued) {
      mma_commit(&bars[kStDrain]);
      (void)mbar_wait_bounded(&bars[kStDrain], 0u, kWaitLimitNs);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kStTmemCols);
  }
}

// ===================================================================== pass 2
constexpr int kOutThreads = 512;  // 16 warps
constexpr int kOutSlots = 4;
// slot: G2[128] | W[128] | ints: c, s, h, sl, pad, wide, has_state, done, bidx,
//       row coordinate (TMA), block row lo / hi (output rows), total (float)
constexpr int kSlotW = 128, kSlotI = 256, kSlotWords = 272;
enum SlotField {
  kFc = 0, kFs, kFh, kFsl, kFpad, kFwide, kFstate, kFdone, kFbidx, kFrow, kFblo, kFbhi, kFtotal
};

template <int DVS>
struct OutLayout {
  static constexpr int kPanels = DVS / 64;
  static constexpr uint32_t kQ = 0;                               // 2 buffers x 32 KB
  static constexpr uint32_t kK = kQ + 2 * 2 * kPanel;             // 32 KB
  static constexpr uint32_t kV = kK + 2 * kPanel;                 // DVS/64 panels
  static constexpr uint32_t kShi = kV + kPanels * kPanel;         // staged tile / S' hi
  static constexpr uint32_t kSlo = kShi + kPanels * kPanel;       // S' lo
  static constexpr uint32_t kSlots = kSlo + kPanels * kPanel;
  static constexpr uint32_t kBar = kSlots + kOutSlots * kSlotWords * 4;
  static constexpr uint32_t kMisc = kBar + 64 * 8;
  static constexpr uint32_t kSmem = kMisc + 16 + 1024;
  static_assert(kSmem <= 232448, "shared memory budget");
};

enum OutBar {
  kQFull = 0, kQEmpty = 2, kKFull = 4, kKEmpty, kVFull, kVEmpty, kSRaw, kSFull, kSEmpty,
  kAFull = 11, kAFree = 13, kPFull = 15, kO3Full = 17, kOFull = 19, kOFree = 21,
  kGReady = 23, kGFree = kGReady + kOutSlots, kDrainO = kGFree + kOutSlots, kOutNumBars
};
static_assert(kOutNumBars <= 64, "barrier area");

// the tile sequence of one CTA: tiles blockIdx.x, + gridDim.x, ... of the
// call's (sequence, head, chunk, slice) tiles; dense batches in chunk-major
// order (all heads of a chunk position together), packed ones per sequence
struct TileWalk {
  const int32_t* cu;
  unsigned* status;
  int B, H, T, nsl, mode;
  long long next_idx;
  // packed: the sequence the walk is in and the index of its first tile
  int seq;
  long long seq_base;
  bool bad;

  __device__ __forceinline__ void init(const SplitParams& p, int nslices) {
    cu = p.cu_seqlens; status = p.status; B = p.B; H = p.H; T = p.T; mode = p.mode;
    nsl = nslices; next_idx = blockIdx.x; seq = 0; seq_base = 0; bad = false;
  }
  __device__ void chunk_range(int nch, int& c0, int& c1) const {
    c0 = mode == 2 ? 1 : 0;
    c1 = mode == 1 ? min(nch, 1) : nch;
    if (c1 < c0) c1 = c0;
  }
  // next tile: (s, c, h, sl, start, len); false when the walk is over
  __device__ __forceinline__ bool next(int& s, int& c, int& h, int& sl, long long& start,
                                      int& len) {
    const long long idx = next_idx;
    next_idx += gridDim.x;
    const long long per = (long long)H * nsl;
    if (cu == nullptr) {
      const int nch = (T + kC - 1) / kC;
      int c0, c1;
      chunk_range(nch, c0, c1);
      const long long per_c = per * B;
      if (idx >= per_c * (c1 - c0)) return false;
      c = c0 + (int)(idx / per_c);
      const long long rem = idx % per_c;
      s = (int)(rem / per);
      h = (int)((rem / nsl) % H);
      sl = (int)(rem % nsl);
      start = (long long)s * T;
      len = T;
      return true;
    }
    if (bad) return false;
    if (__ldg(cu) != 0 || __ldg(cu + B) != T) {
      bad = true;
      atomicOr(status, kDevBadSeqlens);
      return false;
    }
    while (seq < B) {
      const int a = __ldg(cu + seq), b = __ldg(cu + seq + 1);
      if (a < 0 || b < a || b > T) {
        bad = true;
        atomicOr(status, kDevBadSeqlens);
        return false;
      }
      const int nch = (b - a + kC - 1) / kC;
      int c0, c1;
      chunk_range(nch, c0, c1);
      const long long n = per * (c1 - c0);
      if (idx < seq_base + n) {
        const long long local = idx - seq_base;
        c = c0 + (int)(local / per);
        h = (int)((local / nsl) % H);
        sl = (int)(local % nsl);
        s = seq;
        start = a;
        len = b - a;
        return true;
      }
      seq_base += n;
      ++seq;
    }
    return false;
  }
};

// P' of token row r from A = Q K^T in TMEM, in place: hi of 32-column block cb
// at columns 16 cb .. 16 cb + 15, lo at 64 + 16 cb.  Not WIDE: P'_rj = A_rj W_j
// on the causal part (W is zero before the first valid token); WIDE: the
// explicit decays 2^{G_r - G_j} for pad <= j <= r.  A lo block overwrites
// fp32 columns of block 2 + cb / 2, so it is stored once that block has been
// read (blocks past the row's own are zero and never read).
template <bool WIDE>
__device__ __forceinline__ void build_p(uint32_t a_row, int q4, int r, float G2r,
                                        const float* W, const float* G2s, int pad) {
  uint32_t a[32];
  uint32_t lo0[16], lo1[16], lo2[16];
  uint32_t z[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) z[e] = 0u;
  tmem_ld_32x32b_x32(a_row, a);
#pragma unroll
  for (int cb = 0; cb < 4; ++cb) {
    uint32_t hi[16], lo[16];
    if (cb <= q4) {
      tmem_ld_wait_x32(a);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int j = 32 * cb + 2 * e;
        float x0 = __uint_as_float(a[2 * e]), x1 = __uint_as_float(a[2 * e + 1]);
        if constexpr (WIDE) {
          x0 = (j <= r && j >= pad) ? x0 * exp2f(G2r - G2s[j]) : 0.f;
          x1 = (j + 1 <= r && j + 1 >= pad) ? x1 * exp2f(G2r - G2s[j + 1]) : 0.f;
        } else {
          x0 = j <= r ? x0 * W[j] : 0.f;
          x1 = j + 1 <= r ? x1 * W[j + 1] : 0.f;
        }
        hi[e] = pack_bf16x2(x0, x1);
        lo[e] = pack_bf16x2(x0 - bf16lo(hi[e]), x1 - bf16hi(hi[e]));
      }
      if (cb < q4) tmem_ld_32x32b_x32(a_row + 32 * (cb + 1), a);
      tmem_st_32x32b_x16(a_row + 16 * cb, hi);
    } else {
      tmem_st_32x32b_x16(a_row + 16 * cb, z);
#pragma unroll
      for (int e = 0; e < 16; ++e) lo[e] = 0u;
    }
    // lo parts: block cb's lo lands on fp32 block 2 + cb / 2
    if (cb == 0) {
#pragma unroll
      for (int e = 0; e < 16; ++e) lo0[e] = lo[e];
      if (q4 < 2) tmem_st_32x32b_x16(a_row + 64, lo0);
    } else if (cb == 1) {
#pragma unroll
      for (int e = 0; e < 16; ++e) lo1[e] = lo[e];
      if (q4 < 2) tmem_st_32x32b_x16(a_row + 80, lo1);
    } else if (cb == 2) {
#pragma unroll
      for (int e = 0; e < 16; ++e) lo2[e] = lo[e];
      if (q4 >= 2) {  // block 2 has been read
        tmem_st_32x32b_x16(a_row + 64, lo0);
        tmem_st_32x32b_x16(a_row + 80, lo1);
      }
      if (q4 < 3) tmem_st_32x32b_x16(a_row + 96, lo2);
    } else {
      if (q4 == 3) tmem_st_32x32b_x16(a_row + 96, lo2);  // block 3 has been read
      tmem_st_32x32b_x16(a_row + 112, lo);
    }
  }
}

template <int DVS, bool OUTF32, bool DOT>
__global__ void __launch_bounds__(kOutThreads, 1)
chunk_out_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmS,
                 const SplitParams p) {
  using Lay = OutLayout<DVS>;
  constexpr int kPanels = Lay::kPanels;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lay::kMisc + 4);
  uint32_t* slots = reinterpret_cast<uint32_t*>(smem + Lay::kSlots);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nsl = p.DV / DVS;
  const int nks = p.DK / 16;  // k-steps over the key channels
  const bool packed = p.cu_seqlens != nullptr;

  if (tid == 0) {
    for (int i = 0; i < kOutNumBars; ++i) {
      uint32_t cnt = 1;
      if (i == kSFull) cnt = 4;
      if (i == kPFull || i == kPFull + 1 || i == kOFree || i == kOFree + 1) cnt = 4;
      // P' (4), output (4) and state-tile (4) warps, the MMA issuer and the V loader
      if (i >= kGFree && i < kGFree + kOutSlots) cnt = 14;
      mbar_init(&bars[i], cnt);
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmS);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sbase = smem_u32(smem);
  // TMEM: A / P' per tile parity at columns 0 and 128, O at 256 and 256 + DVS
  auto colA = [](int b) -> uint32_t { return 128u * b; };
  auto colO = [](int b) -> uint32_t { return 256u + DVS * b; };

  auto wait = [&](int b, uint32_t parity) -> bool {
    return wait_bar(&bars[b], parity, abort_flag, p.status);
  };
  auto wait_w = [&](int b, uint32_t parity) -> bool {
    return __all_sync(0xffffffffu, wait(b, parity));
  };
  auto warp_arrive = [&](int b) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[b]);
  };
  auto slot_of = [&](int k) -> uint32_t* { return slots + (k % kOutSlots) * kSlotWords; };
  auto sf = [](const uint32_t* sl, int f) -> int { return (int)sl[kSlotI + f]; };

  int issued_q[2] = {0, 0}, issued_k = 0, issued_s = 0, issued_v = 0;
  bool mma_issued = false;

  if (warp == 0) {
    // --------------------------- producer: tiles, gate sums, Q / K / S' loads
    TileWalk walk;
    walk.init(p, nsl);
    int ns, nc, nh, nsl_i, nlen;
    long long nstart;
    bool have = walk.next(ns, nc, nh, nsl_i, nstart, nlen);
    float gnext[4];
    auto load4 = [&](bool valid, int c, long long st, int ln, int hh, float (&gv)[4]) {
      const int nch = (ln + kC - 1) / kC, off = ln - kC * nch;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int t = off + c * kC + 4 * lane + i;
        gv[i] = (valid && t >= 0) ? __ldg(p.g + (st + t) * p.H + hh) : 0.f;
      }
    };
    load4(have, nc, nstart, nlen, nh, gnext);
    int k = 0;
    for (;; ++k) {
      bool ok = true;
      if (k >= kOutSlots && !wait(kGFree + k % kOutSlots, ph(k / kOutSlots - 1))) ok = false;
      if (__any_sync(0xffffffffu, !ok)) break;
      uint32_t* slot = slot_of(k);
      if (!have) {
        if (lane == 0) slot[kSlotI + kFdone] = 1u;
        warp_arrive(kGReady + k % kOutSlots);
        break;
      }
      const int s = ns, c = nc, h = nh, sl = nsl_i, len = nlen;
      const long long start = nstart;
      float gv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) gv[i] = fmaxf(gnext[i], -kGateClamp);
      have = walk.next(ns, nc, nh, nsl_i, nstart, nlen);
      load4(have, nc, nstart, nlen, nh, gnext);

      const int nch = (len + kC - 1) / kC, off = len - kC * nch;
      const int pad = c == 0 ? -off : 0;
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
      float G2[4], Wv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        G2[i] = (excl + run[i]) * kLog2e;
        Wv[i] = (4 * lane + i >= pad) ? exp2f(total - G2[i]) : 0.f;
      }
      const float first = __shfl_sync(0xffffffffu, G2[pad & 3], pad >> 2);
      const bool wide = first - total > kWideSpan;
      float* fslot = reinterpret_cast<float*>(slot);
      *reinterpret_cast<float4*>(fslot + 4 * lane) = make_float4(G2[0], G2[1], G2[2], G2[3]);
      *reinterpret_cast<float4*>(fslot + kSlotW + 4 * lane) =
          make_float4(Wv[0], Wv[1], Wv[2], Wv[3]);
      const int bidx = packed ? 0 : s;
      const int row = (int)((packed ? start : 0) + off + (long long)c * kC);
      const bool has_state = c > 0 || p.init_state != nullptr;
      const long long brow = c > 0 ? block_row(start, len, off, c, p.out_reversed) : 0;
      if (lane == 0) {
        uint32_t* si = slot + kSlotI;
        si[kFc] = c; si[kFs] = s; si[kFh] = h; si[kFsl] = sl; si[kFpad] = pad;
        si[kFwide] = wide; si[kFstate] = has_state; si[kFdone] = 0; si[kFbidx] = bidx;
        si[kFrow] = (uint32_t)row;
        si[kFblo] = (uint32_t)(brow & 0xffffffffll);
        si[kFbhi] = (uint32_t)(brow >> 32);
        fslot[kSlotI + kFtotal] = total;
      }
      warp_arrive(kGReady + k % kOutSlots);
      if (lane == 0) {
        const int qb = k & 1;
        // Q(k): buffer k & 1, free once MMA3(k - 2) has run
        if (k >= 2 && !wait(kQEmpty + qb, ph((k >> 1) - 1))) ok = false;
        if (ok) {
          uint8_t* q_s = smem + Lay::kQ + qb * 2 * kPanel;
          const int np = (p.DK + 63) / 64;
          mbar_arrive_expect_tx(&bars[kQFull + qb], np * kPanel);
          for (int pn = 0; pn < np; ++pn)
            tma_load_4d(q_s + pn * kPanel, &tmQ, &bars[kQFull + qb], pn * 64, h, row, bidx);
          ++issued_q[qb];
        }
        // K(k): one buffer, free once MMA1(k - 1) has run
        if (ok && k >= 1 && !wait(kKEmpty, ph(k - 1))) ok = false;
        if (ok) {
          uint8_t* k_s = smem + Lay::kK;
          const int np = (p.DK + 63) / 64;
          mbar_arrive_expect_tx(&bars[kKFull], np * kPanel);
          for (int pn = 0; pn < np; ++pn)
            tma_load_4d(k_s + pn * kPanel, &tmK, &bars[kKFull], pn * 64, h, row, bidx);
          ++issued_k;
        }
        // the staged state tile of a chunk >= 1, once MMA3(k - 1) has run
        if (ok && c > 0) {
          if (k >= 1 && !wait(kSEmpty, ph(k - 1))) ok = false;
          if (ok) {
            uint8_t* s_s = smem + Lay::kShi;
            const int x0 = (p.osz / 2) * DVS * sl;
            mbar_arrive_expect_tx(&bars[kSRaw], kPanels * p.DK * 128);
            for (int pn = 0; pn < kPanels; ++pn)
              tma_load_4d(s_s + pn * kPanel, &tmS, &bars[kSRaw], x0 + 64 * pn, h,
                          packed ? (int)brow : (int)(brow - (long long)s * p.T),
                          bidx);
            ++issued_s;
          }
        }
      }
      if (__any_sync(0xffffffffu, !ok)) break;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idQK = idesc_bf16(128, 128, false, false);
      const uint32_t idQS = idesc_bf16(128, DVS, false, true);
      const uint32_t idPV = idesc_bf16(128, DVS, false, true);
      bool prev_state = false;
      for (int k = 0;; ++k) {
        if (!wait(kGReady + k % kOutSlots, ph(k / kOutSlots))) break;
        const uint32_t* slot = slot_of(k);
        const bool done = sf(slot, kFdone) != 0;
        const bool has_state = sf(slot, kFstate) != 0;
        mbar_arrive(&bars[kGFree + k % kOutSlots]);
        const int qb = k & 1, b = k & 1;
        if (!done) {
          // MMA1: A(k) = Q K^T
          if (!wait(kQFull + qb, ph(k >> 1))) break;
          if (!wait(kKFull, ph(k))) break;
          if (k >= 2 && !wait(kAFree + b, ph((k >> 1) - 1))) break;
          tc_fence_after();
          const uint32_t q_s = sbase + Lay::kQ + qb * 2 * kPanel;
          const uint64_t qd = sdesc_sw128(q_s, 16, 1024);
          const uint64_t kd = sdesc_sw128(sbase + Lay::kK, 16, 1024);
          for (int kk = 0; kk < nks; ++kk) {
            const uint32_t o = (kk >> 2) * kPanel + (kk & 3) * 32;
            mma_bf16(tmem + colA(b), desc_add(qd, o), desc_add(kd, o), idQK, kk > 0);
          }
          mma_commit(&bars[kAFull + b]);
          mma_commit(&bars[kKEmpty]);
          mma_issued = true;
        }
        // MMA2 of the previous tile: O(k-1) += P'hi V + P'lo V
        if (k >= 1) {
          const int pb = (k - 1) & 1;
          if (!wait(kPFull + pb, ph((k - 1) >> 1))) break;
          if (!wait(kVFull, ph(k - 1))) break;
          tc_fence_after();
          const uint32_t a_p = tmem + colA(pb);
          const uint64_t vd = sdesc_sw128(sbase + Lay::kV, kPanel, 1024);
#pragma unroll
          for (int pass = 0; pass < 2; ++pass)
#pragma unroll
            for (int kk = 0; kk < kC / 16; ++kk)
              mma_bf16_tmem_a(tmem + colO(pb), a_p + 64 * pass + 8 * kk,
                              desc_add(vd, kk * 2048), idPV,
                              (prev_state || pass > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&bars[kOFull + pb]);
          mma_commit(&bars[kVEmpty]);
          mma_commit(&bars[kAFree + pb]);
          mma_issued = true;
        }
        if (done) break;
        // MMA3: O(k) = Q S'hi + Q S'lo
        if (!wait(kSFull, ph(k))) break;
        if (k >= 2 && !wait(kOFree + b, ph((k >> 1) - 1))) break;
        tc_fence_after();
        if (has_state) {
          const uint32_t q_s = sbase + Lay::kQ + qb * 2 * kPanel;
          const uint64_t qd = sdesc_sw128(q_s, 16, 1024);
          const uint64_t hd = sdesc_sw128(sbase + Lay::kShi, kPanel, 1024);
          const uint64_t ld = sdesc_sw128(sbase + Lay::kSlo, kPanel, 1024);
          for (int kk = 0; kk < nks; ++kk) {
            const uint32_t o = (kk >> 2) * kPanel + (kk & 3) * 32;
            mma_bf16(tmem + colO(b), desc_add(qd, o), desc_add(hd, kk * 2048), idQS, kk > 0);
          }
          for (int kk = 0; kk < nks; ++kk) {
            const uint32_t o = (kk >> 2) * kPanel + (kk & 3) * 32;
            mma_bf16(tmem + colO(b), desc_add(qd, o), desc_add(ld, kk * 2048), idQS, 1);
          }
        }
        mma_commit(&bars[kO3Full + b]);
        mma_commit(&bars[kSEmpty]);
        mma_commit(&bars[kQEmpty + qb]);
        prev_state = has_state;
      }
    }
  } else if (warp == 2) {
    // ----------------------------------------------------------- V loader
    for (int k = 0;; ++k) {
      if (!wait_w(kGReady + k % kOutSlots, ph(k / kOutSlots))) break;
      const uint32_t* slot = slot_of(k);
      const bool done = sf(slot, kFdone) != 0;
      const int h = sf(slot, kFh), sl = sf(slot, kFsl), row = sf(slot, kFrow),
                bidx = sf(slot, kFbidx);
      bool ok = true;
      if (lane == 0 && !done) {
        if (k >= 1 && !wait(kVEmpty, ph(k - 1))) ok = false;
        if (ok) {
          mbar_arrive_expect_tx(&bars[kVFull], kPanels * kPanel);
          for (int pn = 0; pn < kPanels; ++pn)
            tma_load_4d(smem + Lay::kV + pn * kPanel, &tmV, &bars[kVFull], sl * DVS + 64 * pn,
                        h, row, bidx);
          ++issued_v;
        }
      }
      warp_arrive(kGFree + k % kOutSlots);
      if (done || __any_sync(0xffffffffu, !ok)) break;
    }
  } else if (warp >= 4 && warp < 8) {
    // ----------------------------------------------------------- P' builders
    const int q4 = warp & 3;
    const int r = 32 * q4 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
    for (int k = 0;; ++k) {
      if (!wait_w(kGReady + k % kOutSlots, ph(k / kOutSlots))) break;
      const uint32_t* slot = slot_of(k);
      if (sf(slot, kFdone)) {
        warp_arrive(kGFree + k % kOutSlots);
        break;
      }
      const float* fslot = reinterpret_cast<const float*>(slot);
      const int pad = sf(slot, kFpad);
      const bool wide = sf(slot, kFwide) != 0, has_state = sf(slot, kFstate) != 0;
      const float G2r = fslot[r];
      const int b = k & 1;
      if (!wait_w(kAFull + b, ph(k >> 1))) break;
      tc_fence_after();
      const uint32_t a_row = tmem + lane_off + colA(b);
      // Rows before the sequence (r < pad) come out zero on both paths: W_j is
      // zero for j < pad, and the explicit path keeps pad <= j <= r.  The
      // tensor-memory accesses stay warp-uniform (.sync.aligned).
      if (wide) {
        build_p<true>(a_row, q4, r, G2r, fslot + kSlotW, fslot, pad);
      } else {
        build_p<false>(a_row, q4, r, G2r, fslot + kSlotW, fslot, pad);
      }
      if (wide && has_state) {
        // O = Q S so far: row t times 2^{G_t} before MMA2 adds the intra-chunk part
        if (!wait_w(kO3Full + b, ph(k >> 1))) break;
        tc_fence_after();
        const float e = r >= pad ? exp2f(G2r) : 0.f;
        const uint32_t o_row = tmem + lane_off + colO(b);
#pragma unroll 1
        for (int part = 0; part < DVS / 16; ++part) {
          uint32_t v[16];
          tmem_ld_32x32b_x16(o_row + 16 * part, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = __float_as_uint(e * __uint_as_float(v[j]));
          tmem_st_32x32b_x16(o_row + 16 * part, v);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      warp_arrive(kPFull + b);
      warp_arrive(kGFree + k % kOutSlots);
    }
  } else if (warp >= 8 && warp < 12) {
    // -------------------------------------------------------------- output
    const int q4 = warp & 3;
    const int r = 32 * q4 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
    for (int k = 0;; ++k) {
      if (!wait_w(kGReady + k % kOutSlots, ph(k / kOutSlots))) break;
      const uint32_t* slot = slot_of(k);
      if (sf(slot, kFdone)) {
        warp_arrive(kGFree + k % kOutSlots);
        break;
      }
      const float* fslot = reinterpret_cast<const float*>(slot);
      const int c = sf(slot, kFc), h = sf(slot, kFh), sl = sf(slot, kFsl),
                pad = sf(slot, kFpad), s = sf(slot, kFs);
      const bool wide = sf(slot, kFwide) != 0;
      const float total = fslot[kSlotI + kFtotal];
      const float G2r = fslot[r];
      const float s1 = p.scale * (wide ? 1.f : exp2f(G2r - total));
      const bool valid = r >= pad;
      // this row's output row in the tensor
      long long start;
      int len;
      if (packed) {
        start = __ldg(p.cu_seqlens + s);
        len = __ldg(p.cu_seqlens + s + 1) - (int)start;
      } else {
        start = (long long)s * p.T;
        len = p.T;
      }
      const int nch = (len + kC - 1) / kC, off = len - kC * nch;
      const long long tok = (long long)off + (long long)c * kC + r;
      const long long orow = start + (p.out_reversed ? len - 1 - tok : tok);
      const size_t base = ((size_t)(valid ? orow : start) * p.H + h) * p.DV + (size_t)sl * DVS;
      const int b = k & 1;
      if constexpr (DOT) {
        uint4 pr[DVS / 8];
#pragma unroll
        for (int j = 0; j < DVS / 8; ++j)
          pr[j] = valid ? __ldg(reinterpret_cast<const uint4*>(p.dot_rows + base) + j)
                        : make_uint4(0u, 0u, 0u, 0u);
        if (!wait_w(kOFull + b, ph(k >> 1))) break;
        tc_fence_after();
        float dot = 0.f;
#pragma unroll
        for (int part = 0; part < DVS / 16; ++part) {
          uint32_t v[16];
          tmem_ld_32x32b_x16(tmem + lane_off + colO(b) + 16 * part, v);
          tmem_ld_wait();
          if (part == DVS / 16 - 1) {
            tc_fence_before();
            warp_arrive(kOFree + b);
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
              float* dst = static_cast<float*>(p.out) + base + 16 * part;
#pragma unroll
              for (int j = 0; j < 4; ++j)
                reinterpret_cast<float4*>(dst)[j] =
                    make_float4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
            } else {
              __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + base + 16 * part;
              uint32_t w[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) w[j] = pack_bf16x2(o[2 * j], o[2 * j + 1]);
              reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
              reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
            }
          }
        }
        if (valid) atomicAdd(p.dot_out + (size_t)orow * p.H + h, p.dot_sign * dot);
      } else {
        if (!wait_w(kOFull + b, ph(k >> 1))) break;
        tc_fence_after();
#pragma unroll 1
        for (int part = 0; part < DVS / 32; ++part) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tmem + lane_off + colO(b) + 32 * part, v);
          tmem_ld_wait_x32(v);
          if (part == DVS / 32 - 1) {
            tc_fence_before();
            warp_arrive(kOFree + b);
          }
          if (valid) {
            if constexpr (OUTF32) {
              float* dst = static_cast<float*>(p.out) + base + 32 * part;
              if (p.out_v8) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  st_global_v8(dst + 8 * j, __float_as_uint(s1 * __uint_as_float(v[8 * j])),
                               __float_as_uint(s1 * __uint_as_float(v[8 * j + 1])),
                               __float_as_uint(s1 * __uint_as_float(v[8 * j + 2])),
                               __float_as_uint(s1 * __uint_as_float(v[8 * j + 3])),
                               __float_as_uint(s1 * __uint_as_float(v[8 * j + 4])),
                               __float_as_uint(s1 * __uint_as_float(v[8 * j + 5])),
                               __float_as_uint(s1 * __uint_as_float(v[8 * j + 6])),
                               __float_as_uint(s1 * __uint_as_float(v[8 * j + 7])));
              } else {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  reinterpret_cast<float4*>(dst)[j] = make_float4(
                      s1 * __uint_as_float(v[4 * j]), s1 * __uint_as_float(v[4 * j + 1]),
                      s1 * __uint_as_float(v[4 * j + 2]), s1 * __uint_as_float(v[4 * j + 3]));
              }
            } else {
              __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + base + 32 * part;
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
      }
      warp_arrive(kGFree + k % kOutSlots);
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------ state-tile warps
    // The tile S' (dk rows x DVS columns) as bf16 hi + lo in the MN-major
    // operand layout: decoded in place from the staged block-floating-point
    // tile (chunks >= 1), or converted from the fp32 initial state (chunk 0).
    const int i = 32 * (warp - 12) + lane;  // state row (key channel)
    int nraw = 0;
    for (int k = 0;; ++k) {
      if (!wait_w(kGReady + k % kOutSlots, ph(k / kOutSlots))) break;
      const uint32_t* slot = slot_of(k);
      if (sf(slot, kFdone)) {
        warp_arrive(kGFree + k % kOutSlots);
        break;
      }
      const float* fslot = reinterpret_cast<const float*>(slot);
      const int c = sf(slot, kFc), s = sf(slot, kFs), h = sf(slot, kFh), sl = sf(slot, kFsl);
      const bool wide = sf(slot, kFwide) != 0, has_state = sf(slot, kFstate) != 0;
      const float total = fslot[kSlotI + kFtotal];
      uint8_t* hi_s = smem + Lay::kShi;
      uint8_t* lo_s = smem + Lay::kSlo;
      bool ok = true;
      if (c > 0) {
        if (!wait_w(kSRaw, ph(nraw++))) break;
        if (i < p.DK) {
#pragma unroll 1
          for (int pn = 0; pn < kPanels; ++pn) {
            uint8_t* hp = hi_s + pn * kPanel;
            uint8_t* lp = lo_s + pn * kPanel;
            const uint4 c0 = *reinterpret_cast<const uint4*>(hp + sw128_offset(i, 0));
            const uint32_t w0[4] = {c0.x, c0.y, c0.z, c0.w};
            int ebits = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e)
              ebits |= (int)((w0[e] & 1u) << (2 * e)) | (int)(((w0[e] >> 16) & 1u) << (2 * e + 1));
            const int E = ebits - 128;
            const float down = __uint_as_float((uint32_t)(E - kBfpMant + 127) << 23);
#pragma unroll 2
            for (int q = 0; q < 8; ++q) {
              const uint32_t o = sw128_offset(i, q);
              const uint4 raw = *reinterpret_cast<const uint4*>(hp + o);
              const uint32_t in[4] = {raw.x, raw.y, raw.z, raw.w};
              uint32_t hw[4], lw[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float x0 = (float)(int16_t)(in[e] & 0xffffu) * down;
                const float x1 = (float)(int16_t)(in[e] >> 16) * down;
                hw[e] = pack_bf16x2(x0, x1);
                lw[e] = pack_bf16x2(x0 - bf16lo(hw[e]), x1 - bf16hi(hw[e]));
              }
              *reinterpret_cast<uint4*>(hp + o) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
              *reinterpret_cast<uint4*>(lp + o) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
          }
        }
      } else {
        // chunk 0: the initial state, decayed over the chunk unless it is wide
        // (nothing to write without one); either way the previous tile's MMA3
        // must be done with the buffers, which also keeps these warps at most
        // one tile ahead of it
        if (k >= 1 && !wait_w(kSEmpty, ph(k - 1))) break;
        if (has_state && i < p.DK) {
          const float f = wide ? 1.f : exp2f(total);
          const float* src = p.init_state + (((size_t)s * p.H + h) * p.DK + i) * p.DV +
                             (size_t)sl * DVS;
#pragma unroll 1
          for (int pn = 0; pn < kPanels; ++pn) {
#pragma unroll 2
            for (int q = 0; q < 8; ++q) {
              const float4 a = __ldg(reinterpret_cast<const float4*>(src + 64 * pn + 8 * q));
              const float4 bq = __ldg(reinterpret_cast<const float4*>(src + 64 * pn + 8 * q + 4));
              const float x[8] = {f * a.x, f * a.y, f * a.z, f * a.w,
                                  f * bq.x, f * bq.y, f * bq.z, f * bq.w};
              uint32_t hw[4], lw[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                hw[e] = pack_bf16x2(x[2 * e], x[2 * e + 1]);
                lw[e] = pack_bf16x2(x[2 * e] - bf16lo(hw[e]), x[2 * e + 1] - bf16hi(hw[e]));
              }
              const uint32_t o = sw128_offset(i, q);
              *reinterpret_cast<uint4*>(hi_s + pn * kPanel + o) =
                  make_uint4(hw[0], hw[1], hw[2], hw[3]);
              *reinterpret_cast<uint4*>(lo_s + pn * kPanel + o) =
                  make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
          }
        }
      }
      if (!ok) break;
      fence_proxy_async_smem();
      warp_arrive(kSFull);
      warp_arrive(kGFree + k % kOutSlots);
    }
  }

  if (*abort_flag) {
    if (warp == 0 && lane == 0) {
      drain_bar(&bars[kQFull], issued_q[0]);
      drain_bar(&bars[kQFull + 1], issued_q[1]);
      drain_bar(&bars[kKFull], issued_k);
      drain_bar(&bars[kSRaw], issued_s);
    }
    if (warp == 2 && lane == 0) drain_bar(&bars[kVFull], issued_v);
    if (warp == 1 && lane == 0 && mma_issued) {
      mma_commit(&bars[kDrainO]);
      (void)mbar_wait_bounded(&bars[kDrainO], 0u, kWaitLimitNs);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
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

// A bf16 view [nb][rows][H][d] of `base` (row pitch H * pitch_elems elements,
// head pitch pitch_elems) as the 4-D tensor {d, H, rows, nb}; box {64, 1,
// box_rows, 1}, 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, int d, int pitch_elems, int H,
              long long rows, int nb, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)rows, (cuuint64_t)nb};
  const cuuint64_t strides[3] = {(cuuint64_t)pitch_elems * 2, (cuuint64_t)H * pitch_elems * 2,
                                 (cuuint64_t)rows * H * pitch_elems * 2};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

template <typename K>
cudaError_t set_smem(K kern, uint32_t bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <int DVS>
cudaError_t launch_out(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                       const CUtensorMap& ms, const SplitParams& p, bool f32, bool dot,
                       unsigned grid, cudaStream_t stream) {
  using Lay = OutLayout<DVS>;
  auto run = [&](auto kern) {
    cudaError_t e = set_smem(kern, Lay::kSmem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kOutThreads, Lay::kSmem, stream>>>(mq, mk, mv, ms, p);
    return cudaGetLastError();
  };
  if (dot)
    return f32 ? run(chunk_out_kernel<DVS, true, true>) : run(chunk_out_kernel<DVS, false, true>);
  return f32 ? run(chunk_out_kernel<DVS, true, false>) : run(chunk_out_kernel<DVS, false, false>);
}

}  // namespace

bool chunk_split_supported(const ChunkArgs& a) {
  return !a.fp32_io && !a.vector_gate && a.chunk == kC &&
         (a.dk == 64 || a.dk == 96 || a.dk == 128) &&
         (a.dv == 64 || a.dv == 128 || a.dv == 192);
}

cudaError_t launch_chunk_split(const ChunkArgs& a, cudaStream_t stream) {
  const bool packed = a.cu_seqlens != nullptr;
  const long long rows = a.T;
  const int nb = packed ? 1 : a.B;
  const int dvs = a.dv == 128 ? 128 : 64;
  const int osz = a.fp32_out ? 4 : 2;
  CUtensorMap mq, mk, mv, ms;
  if (!make_map(&mq, a.q, a.dk, a.dk, a.H, rows, nb, kC) ||
      !make_map(&mk, a.k, a.dk, a.dk, a.H, rows, nb, kC) ||
      !make_map(&mv, a.v, a.dv, a.dv, a.H, rows, nb, kC) ||
      !make_map(&ms, a.out, a.dv * osz / 2, a.dv * osz / 2, a.H, rows, nb, a.dk))
    return cudaErrorInvalidValue;
  SplitParams p;
  p.g = a.g; p.scale = a.scale; p.init_state = a.init_state; p.out = a.out;
  p.final_state = a.final_state; p.cu_seqlens = a.cu_seqlens;
  p.B = a.B; p.H = a.H; p.T = a.T; p.DK = a.dk; p.DV = a.dv;
  p.dvs = dvs; p.osz = osz;
  p.out_v8 = (reinterpret_cast<uintptr_t>(a.out) & 31) == 0;
  p.out_reversed = a.out_reversed;
  p.dot_rows = static_cast<const __nv_bfloat16*>(a.dot_rows);
  p.dot_out = a.dot_out;
  p.dot_sign = a.dot_sign;
  p.status = a.status;
  p.mode = 0;

  // output-pass grid: one CTA per SM, or fewer when the call has fewer tiles
  const int nsl_out = a.dv / dvs;
  long long tiles_bound;
  if (packed) {
    tiles_bound = ((long long)a.T / kC + a.B) * a.H * nsl_out;
  } else {
    tiles_bound = (long long)a.B * ((a.T + kC - 1) / kC) * a.H * nsl_out;
  }
  const unsigned out_grid =
      (unsigned)std::max<long long>(1, std::min<long long>(tiles_bound, num_sms()));
  const bool f32 = a.fp32_out, dot = a.dot_out != nullptr;
  auto out_pass = [&](int mode) -> cudaError_t {
    SplitParams q = p;
    q.mode = mode;
    return dvs == 128 ? launch_out<128>(mq, mk, mv, ms, q, f32, dot, out_grid, stream)
                      : launch_out<64>(mq, mk, mv, ms, q, f32, dot, out_grid, stream);
  };
  auto state_pass = [&]() -> cudaError_t {
    cudaError_t e = set_smem(chunk_state_kernel, kStSmemBytes);
    if (e != cudaSuccess) return e;
    const long long ctas = (long long)a.B * a.H * (a.dv / kStSW);
    chunk_state_kernel<<<(unsigned)ctas, kStThreads, kStSmemBytes, stream>>>(mk, mv, p);
    return cudaGetLastError();
  };
  const bool alias = a.init_state != nullptr && a.init_state == a.final_state;
  cudaError_t e;
  if (tiles_bound == 0) return state_pass();
  if (alias) {
    if ((e = out_pass(1)) != cudaSuccess) return e;
    if ((e = state_pass()) != cudaSuccess) return e;
    return out_pass(2);
  }
  if ((e = state_pass()) != cudaSuccess) return e;
  return out_pass(0);
}

}  // namespace gla
