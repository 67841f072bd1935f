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
// sequence's chunks in order; the state slice S (dk x 64, fp32) never leaves
// the SM.  Four tensor-core contractions per chunk, all bf16 x bf16 -> fp32
// into tensor memory (TMEM):
//     MMA1  A   = Q K^T          M=128 (t) N=128 (j) K=dk   A,B K-major
//     MMA3  O2  = Q S_bf16       M=128 (t) N=64      K=dk   B MN-major
//     MMA4  dS  = K^T (Vhi+Vlo)  M=dk (i)  N=64      K=128  A,B MN-major
//     MMA2  O1  = P V            M=128 (t) N=64      K=128  B MN-major
// The decayed values W V (W = exp(G_last - G_j)) are split into two bf16
// terms hi + lo, so the state update keeps ~16 significant bits of each
// product instead of 8 (the final state is held to 1e-3 of its RMS).  The
// running state is kept in fp32 registers of the compute warps (thread i owns
// row i) and fed to MMA3 through a bf16 copy in shared memory.
//
// Warp roles (192 threads):
//   warp 0      TMA producer: Q, K (two 64-column panels each) and the V slice
//               of each chunk into a 2-stage ring, 128-byte swizzled
//   warp 1      TMEM allocator and single-thread MMA issuer
//   warps 2..5  compute: gate prefix sums, W V split, decay mask of A into P
//               (written over the chunk's Q tile), state update, output
// Every wait on an mbarrier is bounded; on timeout the kernel flags the
// device status word, stops issuing work, releases TMEM and returns.
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
constexpr int kThreads = 192;
constexpr int kComputeThreads = 128;
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr float kLog2e = 1.4426950408889634f;

// shared memory map (offsets from the 1024-byte-aligned base)
constexpr uint32_t kPanel = kC * 128;                 // 128 rows x 128 B
constexpr uint32_t kQBytes = kPanel * (kDK / 64);     // 32 KB
constexpr uint32_t kKBytes = kPanel * (kDK / 64);     // 32 KB
constexpr uint32_t kVBytes = kPanel;                  // 16 KB (64 columns)
constexpr uint32_t kStageBytes = kQBytes + kKBytes + kVBytes;
constexpr uint32_t kOffVhi = 2 * kStageBytes;
constexpr uint32_t kOffVlo = kOffVhi + kVBytes;
constexpr uint32_t kOffSb = kOffVlo + kVBytes;        // dk rows x 128 B
constexpr uint32_t kOffG = kOffSb + kDK * 128;        // float G2[128]
constexpr uint32_t kOffRed = kOffG + kC * 4;          // 4 warp totals
constexpr uint32_t kOffBar = kOffRed + 64;
constexpr uint32_t kOffMisc = kOffBar + 256;          // tmem base, abort flag
constexpr uint32_t kSmemUsed = kOffMisc + 64;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;     // alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");

// TMEM column map
constexpr uint32_t kColA = 0;     // two 128-column buffers
constexpr uint32_t kColO1 = 256;
constexpr uint32_t kColO2 = 320;
constexpr uint32_t kColDS = 384;

enum Bar {
  kFull0 = 0, kFull1, kEmpty0, kEmpty1, kAFull0, kAFull1, kAFree0, kAFree1,
  kPFull, kVtFull, kDsFull, kDsFree, kSbFull, kOFull, kOFree, kNumBars
};

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
  float* Gs = reinterpret_cast<float*>(smem + kOffG);
  float* red = reinterpret_cast<float*>(smem + kOffRed);

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
      uint32_t cnt = 1;
      if (i == kAFree0 || i == kAFree1 || i == kPFull || i == kVtFull || i == kDsFree ||
          i == kSbFull || i == kOFree)
        cnt = kComputeThreads;
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      for (int c = 0; c < nch; ++c) {
        const int st = c & 1;
        if (c >= 2 && !wait(kEmpty0 + st, ((c >> 1) + 1) & 1)) break;
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
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t sb = sbase + kOffSb, vhi = sbase + kOffVhi, vlo = sbase + kOffVlo;
      for (int c = 0; c < nch; ++c) {
        const int st = c & 1, ab = c & 1;
        const uint32_t q_s = sbase + st * kStageBytes;
        const uint32_t k_s = q_s + kQBytes;
        const uint32_t v_s = k_s + kKBytes;
        if (!wait(kFull0 + st, (c >> 1) & 1)) break;
        if (c >= 2 && !wait(kAFree0 + ab, ((c >> 1) + 1) & 1)) break;
        tc_fence_after();
        // MMA1: A = Q K^T
#pragma unroll
        for (int kk = 0; kk < kDK / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
          mma_bf16(tmem + kColA + ab * 128, sdesc_sw128(q_s + off, 16, 1024),
                   sdesc_sw128(k_s + off, 16, 1024), kIdQK, kk > 0);
        }
        // MMA3: O2 = Q S_{c-1}
        if (!wait(kSbFull, c & 1)) break;
        if (c >= 1 && !wait(kOFree, (c - 1) & 1)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kDK / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
          mma_bf16(tmem + kColO2, sdesc_sw128(q_s + off, 16, 1024),
                   sdesc_sw128(sb + kk * 2048, kPanel, 1024), kIdQS, kk > 0);
        }
        mma_commit(&bars[kAFull0 + ab]);
        // MMA4: dS = K^T (Vhi + Vlo)
        if (!wait(kVtFull, c & 1)) break;
        if (c >= 1 && !wait(kDsFree, (c - 1) & 1)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_bf16(tmem + kColDS, sdesc_sw128(k_s + kk * 2048, kPanel, 1024),
                   sdesc_sw128(vhi + kk * 2048, kPanel, 1024), kIdKV, kk > 0);
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_bf16(tmem + kColDS, sdesc_sw128(k_s + kk * 2048, kPanel, 1024),
                   sdesc_sw128(vlo + kk * 2048, kPanel, 1024), kIdKV, 1);
        mma_commit(&bars[kDsFull]);
        // MMA2: O1 = P V   (P was written over this stage's Q tile)
        if (!wait(kPFull, c & 1)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
          mma_bf16(tmem + kColO1, sdesc_sw128(q_s + off, 16, 1024),
                   sdesc_sw128(v_s + kk * 2048, kPanel, 1024), kIdPV, kk > 0);
        }
        mma_commit(&bars[kOFull]);
        mma_commit(&bars[kEmpty0 + st]);
      }
    }
  } else {
    // ------------------------------------------------------------ compute
    const int q4 = warp & 3;              // TMEM lane quadrant of this warp
    const int r = 32 * q4 + lane;         // token row (A, O) / state row (dS)
    const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
    const size_t st_off = ((size_t)s * p.H + h) * (size_t)kDK * p.DV + (size_t)r * p.DV +
                          (size_t)sl * kDVS;
    float S[kDVS];
    if (p.init_state) {
      const float4* src = reinterpret_cast<const float4*>(p.init_state + st_off);
#pragma unroll
      for (int j = 0; j < kDVS / 4; ++j) {
        const float4 v = __ldg(src + j);
        S[4 * j] = v.x; S[4 * j + 1] = v.y; S[4 * j + 2] = v.z; S[4 * j + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < kDVS; ++j) S[j] = 0.f;
    }
    auto write_sb = [&]() {
      const uint32_t row_addr = sbase + kOffSb;
#pragma unroll
      for (int cc = 0; cc < 8; ++cc)
        st_shared_v4(row_addr + sw128_offset(r, cc), pack_bf16x2(S[8 * cc], S[8 * cc + 1]),
                     pack_bf16x2(S[8 * cc + 2], S[8 * cc + 3]),
                     pack_bf16x2(S[8 * cc + 4], S[8 * cc + 5]),
                     pack_bf16x2(S[8 * cc + 6], S[8 * cc + 7]));
      fence_proxy_async_smem();
      mbar_arrive(&bars[kSbFull]);
    };
    write_sb();

    auto load_g = [&](int c) -> float {
      const int t = c * kC + r;
      if (c >= nch || t >= len) return 0.f;
      return fmaxf(__ldg(p.g + (start + t) * p.H + h), -kGateClamp);
    };
    float g_next = load_g(0);
    const float scale = p.scale;

    for (int c = 0; c < nch; ++c) {
      const int st = c & 1, ab = c & 1;
      const int n = min(kC, len - c * kC);
      const uint32_t q_s = sbase + st * kStageBytes;
      const uint32_t v_s = q_s + kQBytes + kKBytes;
      const long long rowbase = start + (long long)c * kC;

      // (1) gate prefix sum over the chunk (g = 0 beyond the sequence end)
      const float gcur = g_next;
      g_next = load_g(c + 1);
      float incl = gcur;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      if (lane == 31) red[q4] = incl;
      named_bar_sync(1, kComputeThreads);
      float prefix = 0.f, total = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float tw = red[w];
        if (w < q4) prefix += tw;
        total += tw;
      }
      const float G2 = (incl + prefix) * kLog2e;   // log2 of the decay from chunk start
      const float G2last = total * kLog2e;
      Gs[r] = G2;
      named_bar_sync(1, kComputeThreads);

      // (2) W V split into bf16 hi + lo (rows beyond the sequence get W = 0)
      if (!wait(kFull0 + st, (c >> 1) & 1)) break;
      {
        const float w = (r < n) ? exp2f(G2last - G2) : 0.f;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          const uint32_t off = sw128_offset(r, cc);
          const uint4 raw = ld_shared_v4(v_s + off);
          const uint32_t in[4] = {raw.x, raw.y, raw.z, raw.w};
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = unpack_bf16x2(in[e]);
            const float x0 = w * f.x, x1 = w * f.y;
            hi[e] = pack_bf16x2(x0, x1);
            const float2 hf = unpack_bf16x2(hi[e]);
            lo[e] = pack_bf16x2(x0 - hf.x, x1 - hf.y);
          }
          st_shared_v4(sbase + kOffVhi + off, hi[0], hi[1], hi[2], hi[3]);
          st_shared_v4(sbase + kOffVlo + off, lo[0], lo[1], lo[2], lo[3]);
        }
        fence_proxy_async_smem();
        mbar_arrive(&bars[kVtFull]);
      }

      // (3) P = decay-masked A, written over the stage's Q tile (K-major)
      if (!wait(kAFull0 + ab, (c >> 1) & 1)) break;
      tc_fence_after();
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t pk[16];
        if (cb <= q4) {
          uint32_t a[32];
          tmem_ld_32x32b_x32(tmem + lane_off + kColA + ab * 128 + 32 * cb, a);
          tmem_ld_wait();
#pragma unroll
          for (int jj = 0; jj < 32; jj += 2) {
            const int j = 32 * cb + jj;
            const float p0 = (j <= r) ? __uint_as_float(a[jj]) * exp2f(G2 - Gs[j]) : 0.f;
            const float p1 =
                (j + 1 <= r) ? __uint_as_float(a[jj + 1]) * exp2f(G2 - Gs[j + 1]) : 0.f;
            pk[jj / 2] = pack_bf16x2(p0, p1);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) pk[e] = 0u;
        }
        const uint32_t panel = q_s + (cb >> 1) * kPanel;
#pragma unroll
        for (int m = 0; m < 4; ++m)
          st_shared_v4(panel + sw128_offset(r, (cb & 1) * 4 + m), pk[4 * m], pk[4 * m + 1],
                       pk[4 * m + 2], pk[4 * m + 3]);
      }
      tc_fence_before();
      mbar_arrive(&bars[kAFree0 + ab]);
      fence_proxy_async_smem();
      mbar_arrive(&bars[kPFull]);

      // (4) state: S = exp(G_last) S + dS (thread r owns state row r)
      if (!wait(kDsFull, c & 1)) break;
      tc_fence_after();
      {
        const float decay = exp2f(G2last);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t d[32];
          tmem_ld_32x32b_x32(tmem + lane_off + kColDS + 32 * half, d);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j)
            S[32 * half + j] = fmaf(decay, S[32 * half + j], __uint_as_float(d[j]));
        }
        tc_fence_before();
        mbar_arrive(&bars[kDsFree]);
        if (c + 1 < nch) write_sb();
      }

      // (5) output o = scale (O1 + exp(G_t) O2)
      if (!wait(kOFull, c & 1)) break;
      tc_fence_after();
      {
        const float eg = exp2f(G2);
        float o[kDVS];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t a1[32], a2[32];
          tmem_ld_32x32b_x32(tmem + lane_off + kColO1 + 32 * half, a1);
          tmem_ld_32x32b_x32(tmem + lane_off + kColO2 + 32 * half, a2);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j)
            o[32 * half + j] =
                scale * fmaf(eg, __uint_as_float(a2[j]), __uint_as_float(a1[j]));
        }
        tc_fence_before();
        mbar_arrive(&bars[kOFree]);
        if (r < n) {
          const size_t off = ((size_t)(rowbase + r) * p.H + h) * p.DV + (size_t)sl * kDVS;
          if constexpr (OUTF32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + off);
#pragma unroll
            for (int j = 0; j < kDVS / 4; ++j)
              dst[j] = make_float4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + off);
#pragma unroll
            for (int j = 0; j < kDVS / 8; ++j)
              dst[j] = make_uint4(pack_bf16x2(o[8 * j], o[8 * j + 1]),
                                  pack_bf16x2(o[8 * j + 2], o[8 * j + 3]),
                                  pack_bf16x2(o[8 * j + 4], o[8 * j + 5]),
                                  pack_bf16x2(o[8 * j + 6], o[8 * j + 7]));
          }
        }
      }
    }
    if (p.final_state && !*abort_flag) {
      float4* dst = reinterpret_cast<float4*>(p.final_state + st_off);
#pragma unroll
      for (int j = 0; j < kDVS / 4; ++j)
        dst[j] = make_float4(S[4 * j], S[4 * j + 1], S[4 * j + 2], S[4 * j + 3]);
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
