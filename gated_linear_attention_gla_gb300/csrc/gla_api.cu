// gla_api.cu -- the C ABI of libgla.so: argument checks, dispatch, status word.
//
// Every check below runs on the host before anything is enqueued, so a call
// that returns an error has launched nothing.  Only cu_seqlens (a device
// array) is checked on the device; see seq_bounds() in gla_internal.cuh.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <atomic>
#include <cstring>
#include <mutex>

#include "gla.h"
#include "gla_internal.cuh"

namespace {

// One status word per GPU.  It is a static __device__ variable, so the library
// allocates nothing; kernels receive its address as a parameter.
__device__ unsigned g_status_word;

constexpr int kMaxDevices = 64;
std::mutex g_status_mutex;
unsigned* g_status_ptr[kMaxDevices] = {};

// Address of the current GPU's status word (nullptr and *err set on failure).
unsigned* status_word(cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_status_mutex);
  if (g_status_ptr[dev] == nullptr) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_status_word);
    if (*err != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<unsigned*>(p);
  }
  return g_status_ptr[dev];
}

bool aligned(const void* p, uintptr_t bytes) {
  return (reinterpret_cast<uintptr_t>(p) & (bytes - 1)) == 0;
}

// key head sizes 64, 96, 128; value head sizes 64, 128, 192 (96 x 192 is the
// Laplace 3B head of the "i14 Laplace 3B" page)
bool dk_ok(int d) { return d == 64 || d == 96 || d == 128; }
bool dv_ok(int d) { return d == 64 || d == 128 || d == 192; }

bool flags_ok(unsigned flags) {
  return (flags & ~(GLA_FLAG_FP32_IO | GLA_FLAG_VECTOR_GATE | GLA_FLAG_FP32_OUT)) == 0u;
}

// [a, a + na) and [b, b + nb) overlap (byte ranges).
bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

constexpr long long kMaxElems = 1ll << 40;  // per tensor; keeps index arithmetic exact

thread_local cudaError_t g_last_cuda_error = cudaSuccess;
// the text of the calling thread's most recent non-CUDA failure that carries
// one (empty: the most recent failure was a CUDA error, or there was none)
thread_local char g_last_text[192] = "";

// Map a CUDA result to a status, remembering the error for gla_last_error_string.
gla_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return GLA_OK;
  g_last_cuda_error = e;
  g_last_text[0] = '\0';
  return GLA_ERR_CUDA;
}

std::atomic<uint64_t> g_wait_limit_ns{0};  // 0: the default

}  // namespace

namespace gla {
uint64_t handoff_wait_limit_ns() {
  const uint64_t v = g_wait_limit_ns.load(std::memory_order_relaxed);
  return v != 0 ? v : kDefaultWaitLimitNs;
}
}  // namespace gla

extern "C" {

const char* gla_version(void) { return "0.1.0"; }

uint64_t gla_set_wait_limit_ns(uint64_t nanoseconds) {
  return g_wait_limit_ns.exchange(nanoseconds, std::memory_order_relaxed);
}

const char* gla_last_error_string(void) {
  if (g_last_text[0] != '\0') return g_last_text;
  return g_last_cuda_error == cudaSuccess ? "no error" : cudaGetErrorString(g_last_cuda_error);
}

const char* gla_chunk_fwd_kernel(int dk, int dv, int chunk, unsigned flags) {
  if (!flags_ok(flags) || !dk_ok(dk) || !dv_ok(dv)) return nullptr;
  if (chunk != 16 && chunk != 32 && chunk != 64 && chunk != 128) return nullptr;
  gla::ChunkArgs a{};
  a.dk = dk; a.dv = dv; a.chunk = chunk;
  a.fp32_io = (flags & GLA_FLAG_FP32_IO) != 0;
  a.fp32_out = a.fp32_io || (flags & GLA_FLAG_FP32_OUT) != 0;
  a.vector_gate = (flags & GLA_FLAG_VECTOR_GATE) != 0;
  return (gla::chunk_tc_supported(a) || gla::chunk_tc_vec_supported(a)) ? "tensor_core"
                                                                        : "cuda_core";
}

const char* gla_status_string(gla_status status) {
  switch (status) {
    case GLA_OK: return "ok";
    case GLA_ERR_INVALID_ARG: return "invalid argument";
    case GLA_ERR_UNSUPPORTED: return "unsupported configuration";
    case GLA_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case GLA_ERR_CUDA: return "CUDA error";
    case GLA_ERR_TIMEOUT: return "on-device wait timed out";
  }
  return "unknown status";
}

}  // extern "C"

namespace {

// gla_chunk_fwd, and with `mixer` (its aug / norm_w / eps / z; q, k, v, out and
// the sizes are taken from the call) the mixer's steps after the readout as a
// second launch over out.
gla_status chunk_fwd_impl(const void* q, const void* k, const void* v, const float* g,
                          float scale, const float* init_state, void* out,
                          float* final_state, const int32_t* cu_seqlens, int B, int H, int T,
                          int dk, int dv, int chunk, gla_stream_t stream, unsigned flags,
                          const gla::EpilogueArgs* mixer) {
  if (!flags_ok(flags) || B < 0 || H < 0 || T < 0 || !std::isfinite(scale))
    return GLA_ERR_INVALID_ARG;
  if (!dk_ok(dk) || !dv_ok(dv)) return GLA_ERR_UNSUPPORTED;
  if (chunk != 16 && chunk != 32 && chunk != 64 && chunk != 128) return GLA_ERR_UNSUPPORTED;
  const bool fp32 = (flags & GLA_FLAG_FP32_IO) != 0;
  const bool f32out = fp32 || (flags & GLA_FLAG_FP32_OUT) != 0;
  const bool vec = (flags & GLA_FLAG_VECTOR_GATE) != 0;
  if (B == 0 || H == 0) return GLA_OK;

  const long long rows = cu_seqlens ? (long long)T : (long long)B * T;
  const long long esz = fp32 ? 4 : 2;
  const long long osz = f32out ? 4 : 2;
  const long long qk_elems = rows * H * dk, v_elems = rows * H * dv;
  const long long st_elems = (long long)B * H * dk * dv;
  if (qk_elems > kMaxElems || v_elems > kMaxElems || st_elems > kMaxElems)
    return GLA_ERR_INVALID_ARG;
  if ((long long)B * H * (dv / 64) > 0x7fffffffll) return GLA_ERR_INVALID_ARG;

  if (rows > 0 && (!q || !k || !v || !g || !out)) return GLA_ERR_INVALID_ARG;
  if (cu_seqlens == nullptr && B > 0 && T == 0 && final_state == nullptr) return GLA_OK;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(init_state, 16) || !aligned(final_state, 16) ||
      !aligned(g, vec ? 16 : 4) || !aligned(cu_seqlens, 4))
    return GLA_ERR_MISALIGNED;
  // out must not overlap any input; final_state may equal init_state exactly.
  const size_t out_b = (size_t)(v_elems * osz);
  const size_t v_b = (size_t)(v_elems * esz);
  const size_t qk_b = (size_t)(qk_elems * esz);
  const size_t g_b = (size_t)(rows * H * (vec ? dk : 1) * 4);
  const size_t st_b = (size_t)(st_elems * 4);
  if (overlap(out, out_b, q, qk_b) || overlap(out, out_b, k, qk_b) ||
      overlap(out, out_b, v, v_b) || overlap(out, out_b, g, g_b) ||
      overlap(out, out_b, init_state, st_b) || overlap(out, out_b, final_state, st_b))
    return GLA_ERR_INVALID_ARG;
  if (final_state != init_state && overlap(final_state, st_b, init_state, st_b))
    return GLA_ERR_INVALID_ARG;
  if (overlap(final_state, st_b, q, qk_b) || overlap(final_state, st_b, k, qk_b) ||
      overlap(final_state, st_b, v, v_b) || overlap(final_state, st_b, g, g_b))
    return GLA_ERR_INVALID_ARG;
  if (mixer) {
    if (!std::isfinite(mixer->eps) || mixer->eps < 0.f) return GLA_ERR_INVALID_ARG;
    if (!aligned(mixer->aug, 16) || !aligned(mixer->norm_w, 16) || !aligned(mixer->z, 16))
      return GLA_ERR_MISALIGNED;
    const size_t aug_b = mixer->aug ? (size_t)H * dk * 4 : 0;
    const size_t w_b = mixer->norm_w ? (size_t)H * dv * 4 : 0;
    const size_t z_b = mixer->z ? v_b : 0;
    if (overlap(out, out_b, mixer->aug, aug_b) || overlap(out, out_b, mixer->norm_w, w_b) ||
        overlap(out, out_b, mixer->z, z_b) || overlap(final_state, st_b, mixer->z, z_b) ||
        overlap(final_state, st_b, mixer->aug, aug_b) ||
        overlap(final_state, st_b, mixer->norm_w, w_b))
      return GLA_ERR_INVALID_ARG;
    if (!mixer->aug && !mixer->norm_w && !mixer->z) mixer = nullptr;  // nothing to apply
  }

  cudaError_t err;
  unsigned* status = status_word(&err);
  if (!status) return cuda_status(err);

  gla::ChunkArgs a{};
  a.q = q; a.k = k; a.v = v; a.g = g; a.scale = scale;
  a.init_state = init_state; a.out = out; a.final_state = final_state;
  a.cu_seqlens = cu_seqlens;
  a.B = B; a.H = H; a.T = T; a.dk = dk; a.dv = dv; a.chunk = chunk;
  a.fp32_io = fp32; a.fp32_out = f32out; a.vector_gate = vec; a.status = status;

  // bf16 I/O with chunk 128 runs on the tensor cores whenever that kernel covers
  // the shape; if it cannot be launched the call fails (no quiet substitution).
  // The per-key-channel tensor-core kernel applies the mixer's steps itself
  // (its CTAs own whole output rows); the other kernels are followed by the
  // epilogue pass.
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  bool mixed = false;
  if (rows > 0 && gla::chunk_tc_supported(a)) {
    err = gla::launch_chunk_tc(a, s);
  } else if (rows > 0 && gla::chunk_tc_vec_supported(a)) {
    err = gla::launch_chunk_tc_vec(a, s, mixer);
    mixed = mixer != nullptr;
  } else {
    err = gla::launch_chunk_simt(a, s);
  }
  if (err == cudaSuccess && mixer && !mixed && rows > 0) {
    gla::EpilogueArgs e = *mixer;
    e.out = out; e.q = q; e.k = k; e.v = v; e.rows = rows; e.H = H; e.dk = dk; e.dv = dv;
    e.fp32_io = fp32; e.fp32_out = f32out;
    err = gla::launch_epilogue(e, s);
  }
  return cuda_status(err);
}

}  // namespace

extern "C" {

gla_status gla_chunk_fwd(const void* q, const void* k, const void* v, const float* g,
                         float scale, const float* init_state, void* out,
                         float* final_state, const int32_t* cu_seqlens, int B, int H, int T,
                         int dk, int dv, int chunk, gla_stream_t stream, unsigned flags) {
  return chunk_fwd_impl(q, k, v, g, scale, init_state, out, final_state, cu_seqlens, B, H, T,
                        dk, dv, chunk, stream, flags, nullptr);
}

gla_status gla_chunk_fwd_mixer(const void* q, const void* k, const void* v, const float* g,
                               float scale, const float* init_state, void* out,
                               float* final_state, const int32_t* cu_seqlens, int B, int H,
                               int T, int dk, int dv, int chunk, const float* aug,
                               const float* norm_w, float eps, const void* z,
                               gla_stream_t stream, unsigned flags) {
  gla::EpilogueArgs m{};
  m.aug = aug; m.norm_w = norm_w; m.eps = eps; m.z = z;
  return chunk_fwd_impl(q, k, v, g, scale, init_state, out, final_state, cu_seqlens, B, H, T,
                        dk, dv, chunk, stream, flags, &m);
}

size_t gla_chunk_bwd_workspace_size(int B, int H, int T, int dk, int dv, int packed,
                                    unsigned flags) {
  if (!flags_ok(flags) || B <= 0 || H <= 0 || T < 0) return 0;
  const bool fp32 = (flags & GLA_FLAG_FP32_IO) != 0;
  const bool vec = (flags & GLA_FLAG_VECTOR_GATE) != 0;
  if (!gla::chunk_bwd_tc_supported(dk, dv, fp32, vec)) return 0;
  const long long rows = packed ? (long long)T : (long long)B * T;
  if (rows * H * dk > kMaxElems) return 0;
  return gla::chunk_bwd_tc_workspace(B, H, rows, dk, dv, vec);
}

static_assert(GLA_BWD_FIXED_WORKSPACE_BYTES == gla::kBwdFixedWorkspaceBytes,
              "the header states the fixed workspace's size");

}  // extern "C"

namespace {

// gla_chunk_bwd's checks and launches; with check_only, returns after the checks.
gla_status chunk_bwd_impl(const void* q, const void* k, const void* v, const float* g,
                          float scale, const float* init_state, const void* d_out,
                          const float* d_final_state, void* dq, void* dk_out, void* dv_out,
                          float* dg, float* d_init_state, const int32_t* cu_seqlens, int B,
                          int H, int T, int dk, int dv, void* workspace, size_t workspace_bytes,
                          gla_stream_t stream, unsigned flags, bool check_only) {
  if (!flags_ok(flags) || B < 0 || H < 0 || T < 0 || !std::isfinite(scale))
    return GLA_ERR_INVALID_ARG;
  if (!dk_ok(dk) || !dv_ok(dv)) return GLA_ERR_UNSUPPORTED;
  const bool fp32 = (flags & GLA_FLAG_FP32_IO) != 0;
  const bool f32out = fp32 || (flags & GLA_FLAG_FP32_OUT) != 0;
  const bool vec = (flags & GLA_FLAG_VECTOR_GATE) != 0;
  if (B == 0 || H == 0) return GLA_OK;

  const long long rows = cu_seqlens ? (long long)T : (long long)B * T;
  const long long esz = fp32 ? 4 : 2, osz = f32out ? 4 : 2;
  const long long qk_elems = rows * H * dk, v_elems = rows * H * dv;
  const long long st_elems = (long long)B * H * dk * dv;
  if (qk_elems > kMaxElems || v_elems > kMaxElems || st_elems > kMaxElems)
    return GLA_ERR_INVALID_ARG;
  if ((long long)B * H * (dk / 32) > 0x7fffffffll) return GLA_ERR_INVALID_ARG;
  if (rows > 0 && (!q || !k || !v || !g || !d_out || !dq || !dk_out || !dv_out))
    return GLA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(d_out, 16) ||
      !aligned(dq, 16) || !aligned(dk_out, 16) || !aligned(dv_out, 16) ||
      !aligned(init_state, 16) || !aligned(d_final_state, 16) || !aligned(d_init_state, 16) ||
      !aligned(dg, 16) || !aligned(g, vec ? 16 : 4) || !aligned(cu_seqlens, 4) ||
      !aligned(workspace, 256))
    return GLA_ERR_MISALIGNED;
  // every output is disjoint from every input and from the other outputs
  const size_t qk_b = (size_t)(qk_elems * esz), v_b = (size_t)(v_elems * esz);
  const size_t dqk_b = (size_t)(qk_elems * osz), dv_b = (size_t)(v_elems * osz);
  const size_t g_b = (size_t)(rows * H * (vec ? dk : 1) * 4);
  const size_t st_b = (size_t)(st_elems * 4);
  const void* in_p[] = {q, k, v, g, d_out, init_state, d_final_state, cu_seqlens};
  const size_t in_b[] = {qk_b, qk_b, v_b, g_b, v_b, st_b, st_b,
                         cu_seqlens ? (size_t)(B + 1) * 4 : 0};
  // the tensor-core path runs when it covers the call and the workspace is large enough
  const size_t ws_need = gla::chunk_bwd_tc_supported(dk, dv, fp32, vec)
                             ? gla::chunk_bwd_tc_workspace(B, H, rows, dk, dv, vec)
                             : 0;
  const bool use_tc = rows > 0 && ws_need > 0 && workspace != nullptr && workspace_bytes >= ws_need;
  const void* out_p[] = {dq, dk_out, dv_out, dg, d_init_state, use_tc ? workspace : nullptr};
  const size_t out_b[] = {dqk_b, dqk_b, dv_b, g_b, st_b, ws_need};
  for (int o = 0; o < 6; ++o) {
    for (int i = 0; i < 8; ++i)
      if (overlap(out_p[o], out_b[o], in_p[i], in_b[i])) return GLA_ERR_INVALID_ARG;
    for (int o2 = o + 1; o2 < 6; ++o2)
      if (overlap(out_p[o], out_b[o], out_p[o2], out_b[o2])) return GLA_ERR_INVALID_ARG;
  }
  if (check_only || (rows == 0 && d_init_state == nullptr)) return GLA_OK;

  cudaError_t err;
  unsigned* status = status_word(&err);
  if (!status) return cuda_status(err);
  gla::ChunkBwdArgs a;
  a.q = q; a.k = k; a.v = v; a.g = g; a.scale = scale; a.init_state = init_state;
  a.d_out = d_out; a.d_final = d_final_state; a.dq = dq; a.dk = dk_out; a.dv = dv_out;
  a.dg = rows > 0 ? dg : nullptr; a.d_init = d_init_state; a.cu_seqlens = cu_seqlens;
  a.B = B; a.H = H; a.T = T; a.dk_size = dk; a.dv_size = dv;
  a.fp32_io = fp32; a.fp32_out = f32out; a.vector_gate = vec; a.status = status;
  a.skip_dv = false;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (use_tc && !vec) {
    err = gla::launch_chunk_bwd_tc(a, workspace, s);
  } else if (use_tc) {
    // per-key-channel gate: dq, dk (and dg, d_init) on the CUDA cores, dv on the tensor cores
    a.skip_dv = true;
    err = gla::launch_chunk_bwd_chan_bf16(a, s);
    if (err == cudaSuccess) err = gla::launch_chunk_bwd_tc_vec_dv(a, workspace, s);
  } else if (vec)
    err = fp32 ? gla::launch_chunk_bwd_chan_f32(a, s) : gla::launch_chunk_bwd_chan_bf16(a, s);
  else
    err = fp32 ? gla::launch_chunk_bwd_head_f32(a, s) : gla::launch_chunk_bwd_head_bf16(a, s);
  return cuda_status(err);
}

}  // namespace

extern "C" {

gla_status gla_chunk_bwd(const void* q, const void* k, const void* v, const float* g,
                         float scale, const float* init_state, const void* d_out,
                         const float* d_final_state, void* dq, void* dk_out, void* dv_out,
                         float* dg, float* d_init_state, const int32_t* cu_seqlens, int B,
                         int H, int T, int dk, int dv, void* workspace, size_t workspace_bytes,
                         gla_stream_t stream, unsigned flags) {
  return chunk_bwd_impl(q, k, v, g, scale, init_state, d_out, d_final_state, dq, dk_out, dv_out,
                        dg, d_init_state, cu_seqlens, B, H, T, dk, dv, workspace,
                        workspace_bytes, stream, flags, false);
}

gla_status gla_chunk_bwd_fixed_workspace(const void* q, const void* k, const void* v,
                                         const float* g, float scale, const float* init_state,
                                         const void* d_out, const float* d_final_state,
                                         void* dq, void* dk_out, void* dv_out, float* dg,
                                         float* d_init_state, const int32_t* cu_seqlens, int B,
                                         int H, int T, int dk, int dv, gla_stream_t stream,
                                         unsigned flags) {
  // every argument check first, exactly as gla_chunk_bwd makes them
  const gla_status st =
      chunk_bwd_impl(q, k, v, g, scale, init_state, d_out, d_final_state, dq, dk_out, dv_out,
                     dg, d_init_state, cu_seqlens, B, H, T, dk, dv, nullptr, 0, stream, flags,
                     true);
  if (st != GLA_OK) return st;
  // The library's buffer is used (and its module loaded) only when the
  // tensor-core path covers the call; a call whose workspace need exceeds the
  // buffer is rejected before anything is enqueued.
  void* ws = nullptr;
  if (B > 0 && H > 0 && T > 0) {
    const size_t need = gla_chunk_bwd_workspace_size(B, H, T, dk, dv, cu_seqlens != nullptr,
                                                     flags);
    if (need > gla::kBwdFixedWorkspaceBytes) {
      std::snprintf(g_last_text, sizeof(g_last_text),
                    "gla_chunk_bwd_fixed_workspace: the call needs %zu bytes of workspace, "
                    "the fixed buffer holds %zu",
                    need, gla::kBwdFixedWorkspaceBytes);
      return GLA_ERR_UNSUPPORTED;
    }
    if (need > 0) {
      cudaError_t err;
      ws = gla::bwd_fixed_workspace(&err);
      if (!ws) return cuda_status(err);
    }
  }
  return gla_chunk_bwd(q, k, v, g, scale, init_state, d_out, d_final_state, dq, dk_out, dv_out,
                       dg, d_init_state, cu_seqlens, B, H, T, dk, dv, ws,
                       ws ? gla::kBwdFixedWorkspaceBytes : 0, stream, flags);
}

namespace {

// The decode step over N sequences whose state pages are either the N pages of
// `state` (slots == nullptr) or pages slots[n] of a pool of num_slots pages.
gla_status decode_common(const void* q, const void* k, const void* v, const float* g,
                         float scale, float* state, int num_slots, const int32_t* slots,
                         void* out, int N, int H, int dk, int dv, const float* aug,
                         const float* norm_w, float eps, const void* z, gla_stream_t stream,
                         unsigned flags) {
  if (!flags_ok(flags) || N < 0 || H < 0 || !std::isfinite(scale) || !std::isfinite(eps) ||
      eps < 0.f)
    return GLA_ERR_INVALID_ARG;
  if (!dk_ok(dk) || !dv_ok(dv)) return GLA_ERR_UNSUPPORTED;
  if (slots && num_slots < 0) return GLA_ERR_INVALID_ARG;
  if (N == 0 || H == 0) return GLA_OK;
  const long long units = (long long)N * H;
  const long long pages = slots ? (long long)num_slots * H : units;
  if (units > 0x7fffffffll || pages * dk * dv > kMaxElems) return GLA_ERR_INVALID_ARG;
  if (!q || !k || !v || !g || !state || !out) return GLA_ERR_INVALID_ARG;
  const bool fp32 = (flags & GLA_FLAG_FP32_IO) != 0;
  const bool f32out = fp32 || (flags & GLA_FLAG_FP32_OUT) != 0;
  const bool vec = (flags & GLA_FLAG_VECTOR_GATE) != 0;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(state, 16) || !aligned(g, 4) || !aligned(slots, 4))
    return GLA_ERR_MISALIGNED;
  const long long esz = fp32 ? 4 : 2;
  const size_t st_b = (size_t)(pages * dk * dv * 4);
  const size_t out_b = (size_t)(units * dv * (f32out ? 4 : 2));
  const size_t v_b = (size_t)(units * dv * esz);
  const size_t qk_b = (size_t)(units * dk * esz);
  const size_t g_b = (size_t)(units * (vec ? dk : 1) * 4);
  const size_t sl_b = slots ? (size_t)N * 4 : 0;
  if (overlap(out, out_b, state, st_b) || overlap(out, out_b, q, qk_b) ||
      overlap(out, out_b, k, qk_b) || overlap(out, out_b, v, v_b) ||
      overlap(out, out_b, g, g_b) || overlap(state, st_b, q, qk_b) ||
      overlap(state, st_b, k, qk_b) || overlap(state, st_b, v, v_b) ||
      overlap(state, st_b, g, g_b) || overlap(out, out_b, slots, sl_b) ||
      overlap(state, st_b, slots, sl_b))
    return GLA_ERR_INVALID_ARG;
  if (!aligned(aug, 4) || !aligned(norm_w, 4) || !aligned(z, (uintptr_t)esz))
    return GLA_ERR_MISALIGNED;
  const size_t z_b = z ? (size_t)(units * dv * esz) : 0;
  if (overlap(out, out_b, z, z_b) || overlap(state, st_b, z, z_b) ||
      overlap(out, out_b, aug, aug ? (size_t)H * dk * 4 : 0) ||
      overlap(out, out_b, norm_w, norm_w ? (size_t)H * dv * 4 : 0) ||
      overlap(state, st_b, aug, aug ? (size_t)H * dk * 4 : 0) ||
      overlap(state, st_b, norm_w, norm_w ? (size_t)H * dv * 4 : 0))
    return GLA_ERR_INVALID_ARG;

  cudaError_t err = cudaSuccess;
  unsigned* status = nullptr;
  if (slots) {
    status = status_word(&err);
    if (!status) return cuda_status(err);
  }
  gla::DecodeArgs a;
  a.q = q; a.k = k; a.v = v; a.g = g; a.scale = scale;
  a.state = state; a.slots = slots; a.num_slots = num_slots; a.status = status; a.out = out;
  a.aug = aug; a.norm_w = norm_w; a.eps = eps; a.z = z;
  a.N = N; a.H = H; a.dk = dk; a.dv = dv;
  a.fp32_io = fp32; a.fp32_out = f32out; a.vector_gate = vec;
  return cuda_status(gla::launch_decode(a, reinterpret_cast<cudaStream_t>(stream)));
}

}  // namespace

gla_status gla_decode_step(const void* q, const void* k, const void* v, const float* g,
                           float scale, float* state_inout, void* out, int N, int H, int dk,
                           int dv, gla_stream_t stream, unsigned flags) {
  return decode_common(q, k, v, g, scale, state_inout, 0, nullptr, out, N, H, dk, dv, nullptr,
                       nullptr, 0.f, nullptr, stream, flags);
}

gla_status gla_decode_step_slots(const void* q, const void* k, const void* v, const float* g,
                                 float scale, float* state_pool, int num_slots,
                                 const int32_t* slots, void* out, int N, int H, int dk, int dv,
                                 gla_stream_t stream, unsigned flags) {
  if (!slots) return GLA_ERR_INVALID_ARG;
  return decode_common(q, k, v, g, scale, state_pool, num_slots, slots, out, N, H, dk, dv,
                       nullptr, nullptr, 0.f, nullptr, stream, flags);
}

gla_status gla_decode_step_mixer(const void* q, const void* k, const void* v, const float* g,
                                 float scale, float* state, int num_slots, const int32_t* slots,
                                 void* out, int N, int H, int dk, int dv, const float* aug,
                                 const float* norm_w, float eps, const void* z,
                                 gla_stream_t stream, unsigned flags) {
  if (slots == nullptr && num_slots != 0) return GLA_ERR_INVALID_ARG;
  return decode_common(q, k, v, g, scale, state, num_slots, slots, out, N, H, dk, dv, aug,
                       norm_w, eps, z, stream, flags);
}

gla_status gla_mixer_epilogue(void* out, const void* q, const void* k, const void* v,
                              const float* aug, const float* norm_w, float eps, const void* z,
                              int rows, int H, int dk, int dv, gla_stream_t stream,
                              unsigned flags) {
  if ((flags & ~(GLA_FLAG_FP32_IO | GLA_FLAG_FP32_OUT)) != 0u || rows < 0 || H < 0 ||
      !std::isfinite(eps) || eps < 0.f)
    return GLA_ERR_INVALID_ARG;
  if (!dk_ok(dk) || !dv_ok(dv)) return GLA_ERR_UNSUPPORTED;
  if (rows == 0 || H == 0) return GLA_OK;
  const long long units = (long long)rows * H;
  if (units * dk > kMaxElems || units * dv > kMaxElems) return GLA_ERR_INVALID_ARG;
  if (!out || (aug && (!q || !k || !v))) return GLA_ERR_INVALID_ARG;
  const bool fp32 = (flags & GLA_FLAG_FP32_IO) != 0;
  const bool f32out = fp32 || (flags & GLA_FLAG_FP32_OUT) != 0;
  const size_t esz = fp32 ? 4 : 2, osz = f32out ? 4 : 2;
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) ||
      !aligned(z, 16) || !aligned(aug, 16) || !aligned(norm_w, 16))
    return GLA_ERR_MISALIGNED;
  const size_t out_b = (size_t)(units * dv) * osz;
  const size_t qk_b = aug ? (size_t)(units * dk) * esz : 0;
  const size_t v_b = aug ? (size_t)(units * dv) * esz : 0;
  const size_t z_b = z ? (size_t)(units * dv) * esz : 0;
  if (overlap(out, out_b, q, qk_b) || overlap(out, out_b, k, qk_b) ||
      overlap(out, out_b, v, v_b) || overlap(out, out_b, z, z_b) ||
      overlap(out, out_b, aug, aug ? (size_t)H * dk * 4 : 0) ||
      overlap(out, out_b, norm_w, norm_w ? (size_t)H * dv * 4 : 0))
    return GLA_ERR_INVALID_ARG;
  if (!aug && !norm_w && !z) return GLA_OK;
  gla::EpilogueArgs a;
  a.out = out; a.q = q; a.k = k; a.v = v; a.aug = aug; a.norm_w = norm_w; a.eps = eps; a.z = z;
  a.rows = rows; a.H = H; a.dk = dk; a.dv = dv; a.fp32_io = fp32; a.fp32_out = f32out;
  return cuda_status(gla::launch_epilogue(a, reinterpret_cast<cudaStream_t>(stream)));
}

gla_status gla_status_sync(gla_stream_t stream) {
  cudaError_t err = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_status(err);
  unsigned* p = status_word(&err);
  if (!p) return cuda_status(err);
  unsigned word = 0;
  err = cudaMemcpy(&word, p, sizeof(word), cudaMemcpyDeviceToHost);
  if (err != cudaSuccess) return cuda_status(err);
  if (word != 0 && (err = cudaMemset(p, 0, sizeof(unsigned))) != cudaSuccess)
    return cuda_status(err);
  if (word & gla::kDevTimeout) return GLA_ERR_TIMEOUT;
  if (word & gla::kDevLayout) return GLA_ERR_UNSUPPORTED;
  if (word & gla::kDevBadSeqlens) return GLA_ERR_INVALID_ARG;
  return GLA_OK;
}

}  // extern "C"
