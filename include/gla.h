/*
 * gla.h -- C ABI of libgla.so: gated linear attention (GLA) on one NVIDIA
 * GB300 (sm_103a).
 *
 * The method (the "i14 Laplace 3B on AWS Trainium2" blog page, section
 * "i14 and the Laplace 3B architecture", paragraph "GLA mixer"): every head
 * keeps a dk x dv matrix state S that decays and absorbs one rank-1
 * key/value write per token, and the query reads the state after the write:
 *
 *     S_t = diag(exp g_t) S_{t-1} + k_t^T v_t
 *     o_t = scale * q_t S_t
 *
 * g_t is a log-decay, either one value per (token, head) -- the page's
 * "Simple GLA" with a per-head decay -- or one value per (token, head, key
 * channel), where row i of S decays by exp(g_t[i]).
 *
 * Entry points:
 *   gla_chunk_fwd    prefill: the chunked form of the same page's section
 *                    "Challenge 1" (Figure 3) -- per chunk a causal Q K^T
 *                    weighted by the decays, times V, plus the carried-in
 *                    state's share, then one state step with the chunk's
 *                    total decay; emits the final state.
 *   gla_decode_step  one token for each of N concurrent sequences, each with a
 *                    fixed-size state page updated in place (section
 *                    "Inference optimization on Trainium2": one fixed page per
 *                    sequence); gla_decode_step_slots takes the pages from a
 *                    pool by slot index (for padded, graph-replayed batches).
 *   gla_mixer_epilogue, gla_chunk_fwd_mixer, gla_decode_step_mixer
 *                    the mixer's steps after the readout (self-augmentation,
 *                    head RMSNorm, SiLU output gate): over a finished output,
 *                    after a prefill in one call, fused into the decode step.
 *   gla_chunk_bwd    the gradient of the prefill (dq, dk, dv, dg and the
 *                    initial state's gradient) for training;
 *                    gla_chunk_bwd_workspace_size sizes its tensor-core path's
 *                    workspace, gla_chunk_bwd_fixed_workspace runs it on a
 *                    buffer of the library's own.
 *   gla_status_sync, gla_status_string, gla_last_error_string, gla_version,
 *   gla_chunk_fwd_kernel, gla_set_wait_limit_ns
 *                    diagnostics.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *     never allocates or frees device memory; it keeps one device status word
 *     per GPU and the fixed backward workspace (static __device__ variables)
 *     and no other state.
 *   - Calls are asynchronous on `stream` (0 = legacy default stream).  Host-side
 *     argument checks happen before anything is enqueued: a call that returns
 *     an error has launched nothing and written nothing.
 *   - Layouts are dense, row-major, token-major ("[B, T, H, d]": d fastest).
 *   - bf16 is IEEE-style bfloat16 (1-8-7); outputs are rounded to nearest even
 *     from fp32.  States are always fp32.  Accumulation is fp32.
 *   - Errors detected on the device (a malformed cu_seqlens, an internal wait
 *     that ran out) set bits in the status word; the affected (sequence, head)
 *     writes nothing.  gla_status_sync() reports and clears them.
 *   - Thread safety: calls may come from any host thread; the device status
 *     word is shared by all streams of a GPU.
 */
#ifndef GLA_H_
#define GLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream; declared here so that this header
 * needs no CUDA header. */
typedef struct CUstream_st *gla_stream_t;

typedef enum gla_status {
    GLA_OK = 0,
    GLA_ERR_INVALID_ARG = 1,  /* null pointer, negative size, bad flags, bad cu_seqlens */
    GLA_ERR_UNSUPPORTED = 2,  /* valid but not implemented: head size, chunk size */
    GLA_ERR_MISALIGNED = 3,   /* a tensor pointer is not 16-byte aligned */
    GLA_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed */
    GLA_ERR_TIMEOUT = 5       /* a bounded on-device wait gave up (reported by gla_status_sync) */
} gla_status;

/* flags */
#define GLA_FLAG_FP32_IO (1u << 0)     /* q, k, v and out are fp32 (default bf16) */
#define GLA_FLAG_VECTOR_GATE (1u << 1) /* g has one value per key channel (default per head) */
#define GLA_FLAG_FP32_OUT (1u << 2)    /* out is fp32 while q, k, v stay bf16; the bf16 output of
                                          the same call is exactly this result rounded to
                                          nearest-even (same kernels, only the store differs) */

/*
 * gla_chunk_fwd -- chunked prefill over a batch of sequences.
 *
 * Source: "i14 Laplace 3B" page, section "Challenge 1: Using native PyTorch
 * on Trainium for GLA" (chunked intra-chunk output, chunked state update,
 * Figure 3), with the recurrence of the "GLA mixer" paragraph.  Chunks start
 * at each sequence start; the last chunk of a sequence may be partial.  The
 * chunk size changes only the rounding, not the result.
 *
 * Arguments
 *   q, k        [B, T, H, dk] (dense) or [R, H, dk] (packed), bf16 or fp32
 *   v           [B, T, H, dv] or [R, H, dv], same dtype as q
 *   g           fp32 log-decay, [B, T, H] / [R, H], or with
 *               GLA_FLAG_VECTOR_GATE [B, T, H, dk] / [R, H, dk].  Values must be
 *               <= 0 or -inf; values below -30 act as -30 (exp(-30) ~ 1e-13).
 *   scale       readout scale (finite), usually dk^-0.5
 *   init_state  fp32 [B, H, dk, dv] state before the first token, or NULL (zeros)
 *   out         [B, T, H, dv] / [R, H, dv], same dtype as q (fp32 with
 *               GLA_FLAG_FP32_OUT); must not overlap any input
 *   final_state fp32 [B, H, dk, dv] state after the last token, or NULL (not
 *               written).  May alias init_state exactly (in-place update).
 *   cu_seqlens  NULL for a dense batch of B sequences of T tokens; otherwise a
 *               DEVICE int32 [B+1] array of packed sequence offsets with
 *               cu_seqlens[0] = 0, non-decreasing, cu_seqlens[B] = T = R (the
 *               number of packed token rows).  Checked on the device: a
 *               violation sets GLA_ERR_INVALID_ARG in the status word and the
 *               offending sequence writes nothing.
 *   B, H, T     batch (or number of packed sequences), heads, tokens per
 *               sequence (or packed rows).  B, H, T >= 0; with T = 0 (or empty
 *               sequences) final_state receives init_state (or zeros).
 *   dk, dv      head sizes: dk 64, 96 or 128; dv 64, 128 or 192
 *   chunk       tokens per chunk: 128 (tensor-core path for bf16 I/O: the
 *               per-head gate with every head size above -- dk = 64 and 96
 *               run zero-padded to 128 --, the per-key-channel gate with
 *               dk = dv = 128), or 16, 32, 64 (fp32 SIMT path); fp32 I/O and
 *               the other head sizes take the SIMT path
 *   stream      CUDA stream
 *   flags       GLA_FLAG_* bits; 0 = bf16 I/O, per-head gate
 *
 * Alignment: q, k, v, out, init_state, final_state must be 16-byte aligned; g
 * 4-byte aligned (16-byte with GLA_FLAG_VECTOR_GATE).
 */
gla_status gla_chunk_fwd(const void *q, const void *k, const void *v, const float *g,
                         float scale, const float *init_state, void *out,
                         float *final_state, const int32_t *cu_seqlens, int B, int H,
                         int T, int dk, int dv, int chunk, gla_stream_t stream,
                         unsigned flags);

/*
 * gla_decode_step -- one recurrent step for N concurrent sequences.
 *
 * Source: "i14 Laplace 3B" page, paragraph "GLA mixer" (the recurrence, one
 * token) and section "Inference optimization on Trainium2" (decode over many
 * concurrent sequences, one fixed state page per sequence).
 *
 * For every (n, h): S <- diag(exp g) S + k^T v (in place), o <- scale * q S.
 *
 * Arguments
 *   q, k         [N, H, dk], bf16 or fp32 (GLA_FLAG_FP32_IO)
 *   v            [N, H, dv], same dtype
 *   g            fp32 [N, H], or [N, H, dk] with GLA_FLAG_VECTOR_GATE; -inf allowed
 *   scale        readout scale
 *   state_inout  fp32 [N, H, dk, dv], read and overwritten in place
 *   out          [N, H, dv], same dtype as q (fp32 with GLA_FLAG_FP32_OUT)
 *   N, H         sequences and heads (>= 0; 0 does nothing)
 *   dk, dv       dk 64, 96 or 128; dv 64, 128 or 192
 * Alignment: every pointer 16-byte aligned except g (4-byte).
 */
gla_status gla_decode_step(const void *q, const void *k, const void *v, const float *g,
                           float scale, float *state_inout, void *out, int N, int H,
                           int dk, int dv, gla_stream_t stream, unsigned flags);

/*
 * gla_decode_step_slots -- the decode step with the states held in a pool of
 * pages, sequence n using page slots[n].
 *
 * Source: as gla_decode_step; the page's serving setup keeps one fixed state
 * page per sequence in a pool that the token mixer reads and writes (section
 * "Inference optimization on Trainium2").  Indexing the pool lets sequences
 * arrive and leave without moving state, and lets a batch be padded to a
 * fixed width (for CUDA-graph replay) with rows that do nothing.
 *
 * Arguments: as gla_decode_step, except
 *   state_pool   fp32 [num_slots, H, dk, dv]; page slots[n] is read and
 *                overwritten in place for sequence n
 *   num_slots    pages in the pool (>= 0)
 *   slots        DEVICE int32 [N]: the page of each row.  -1 marks a padding
 *                row: its state is not touched and its out row not written.
 *                The slots of one call must be distinct (two rows on one page
 *                race).  A slot >= num_slots is reported by gla_status_sync
 *                as GLA_ERR_INVALID_ARG and that row does nothing.
 * Returns GLA_ERR_INVALID_ARG for a null slots pointer; alignment as
 * gla_decode_step (slots 4-byte aligned).
 */
gla_status gla_decode_step_slots(const void *q, const void *k, const void *v, const float *g,
                                 float scale, float *state_pool, int num_slots,
                                 const int32_t *slots, void *out, int N, int H, int dk, int dv,
                                 gla_stream_t stream, unsigned flags);

/*
 * gla_mixer_epilogue -- the mixer's steps after the readout, in place over a
 * finished output (for instance the out of gla_chunk_fwd).
 *
 * Source: "i14 Laplace 3B" page, paragraph "GLA mixer": a self-augmentation
 * adds the value gated by the query dotted with a learned per-key-channel
 * rescaling of the key; the per-head outputs pass a head RMSNorm (one weight
 * per decay tier); the result is gated by SiLU of the gate stream.  Per token
 * and head, each step skipped when its pointer is null:
 *     o += sigmoid(sum_i q_i aug[h][i] k_i) * v
 *     o  = o / sqrt(mean_j o_j^2 + eps) * norm_w[h][j]
 *     o *= z / (1 + exp(-z))
 *
 * Arguments
 *   out          [rows, H, dv] bf16 (fp32 with GLA_FLAG_FP32_OUT), in place
 *   q, k         [rows, H, dk], v [rows, H, dv]: bf16 (fp32 with
 *                GLA_FLAG_FP32_IO); needed only with aug
 *   aug          fp32 [H, dk] or NULL
 *   norm_w       fp32 [H, dv] or NULL (a tier's heads carry equal rows)
 *   eps          >= 0, added to the mean square
 *   z            [rows, H, dv], q's dtype, or NULL
 *   rows, H      token rows and heads (>= 0); dk, dv as gla_chunk_fwd
 *   flags        GLA_FLAG_FP32_IO, GLA_FLAG_FP32_OUT only
 * Alignment: every pointer 16-byte aligned.  out must not overlap any input.
 */
gla_status gla_mixer_epilogue(void *out, const void *q, const void *k, const void *v,
                              const float *aug, const float *norm_w, float eps, const void *z,
                              int rows, int H, int dk, int dv, gla_stream_t stream,
                              unsigned flags);

/*
 * gla_chunk_fwd_mixer -- gla_chunk_fwd followed by the mixer's steps after the
 * readout (as gla_mixer_epilogue) on its output, in one call: the prefill, then
 * a second launch over `out` (a pass at ~70 % of HBM bandwidth).  Arguments:
 * those of gla_chunk_fwd, plus aug, norm_w, eps and z as for
 * gla_mixer_epilogue (z shaped like out, in q's dtype); each step is skipped
 * when its pointer is NULL.  Alignment: as gla_chunk_fwd, and aug, norm_w, z
 * 16-byte aligned.
 */
gla_status gla_chunk_fwd_mixer(const void *q, const void *k, const void *v, const float *g,
                               float scale, const float *init_state, void *out,
                               float *final_state, const int32_t *cu_seqlens, int B, int H,
                               int T, int dk, int dv, int chunk, const float *aug,
                               const float *norm_w, float eps, const void *z,
                               gla_stream_t stream, unsigned flags);

/*
 * gla_decode_step_mixer -- the decode step with the mixer's steps after the
 * readout fused into it (one CTA owns a head's whole output row).
 *
 * Arguments: as gla_decode_step_slots (slots NULL: state is [N, H, dk, dv]
 * and num_slots must be 0), plus aug, norm_w, eps and z as for
 * gla_mixer_epilogue (z [N, H, dv] in q's dtype).  Each step is skipped when
 * its pointer is NULL.
 */
gla_status gla_decode_step_mixer(const void *q, const void *k, const void *v, const float *g,
                                 float scale, float *state, int num_slots,
                                 const int32_t *slots, void *out, int N, int H, int dk, int dv,
                                 const float *aug, const float *norm_w, float eps,
                                 const void *z, gla_stream_t stream, unsigned flags);

/*
 * gla_chunk_bwd -- the gradient of gla_chunk_fwd (training), for a loss whose
 * gradients with respect to out and final_state are d_out and d_final_state.
 *
 * Source: "i14 Laplace 3B" page, section "Challenge 1" (the chunked layer is
 * trained; its backward pass runs over the chunks like the forward) with the
 * recurrence of the "GLA mixer" paragraph.  Reverse mode through
 * S_t = diag(exp g_t) S_{t-1} + k_t^T v_t, o_t = scale q_t S_t: with
 * Sbar_t = dL/dS_t = scale q_t^T do_t + diag(exp g_{t+1}) Sbar_{t+1},
 *     dq_t = scale S_t do_t^T      dk_t = Sbar_t v_t^T      dv_t = k_t Sbar_t
 *     dg_t[i] = exp(g_t[i]) sum_j S_{t-1}[i][j] Sbar_t[i][j]  (summed over i
 *               for the per-head gate)
 *     d_init = diag(exp g_0) Sbar_0
 * computed chunk by chunk (64 tokens) in fp32.  The gate is clamped at -30 as
 * in the forward; dg is the gradient with respect to the clamped gate.
 *
 * Arguments
 *   q, k, v, g, scale, init_state, cu_seqlens, B, H, T, dk, dv
 *                 exactly as passed to gla_chunk_fwd
 *   d_out         [B, T, H, dv] / [R, H, dv], q's dtype: dL/d out
 *   d_final_state fp32 [B, H, dk, dv] dL/d final_state, or NULL (zero)
 *   dq, dk_out    [.., H, dk]; dv_out [.., H, dv]: q's dtype, fp32 with
 *                 GLA_FLAG_FP32_OUT (the bf16 results are these rounded to
 *                 nearest-even)
 *   dg            fp32, g's shape, or NULL (not computed).  With the per-head
 *                 gate its terms are summed across CTAs with fp32 atomics, so
 *                 its last bits may vary from run to run.
 *   d_init_state  fp32 [B, H, dk, dv], or NULL (not written)
 *   workspace     device scratch owned by the caller, or NULL; with at least
 *                 gla_chunk_bwd_workspace_size(...) bytes (256-byte aligned),
 *                 bf16 I/O and dk, dv each 64 or 128 (the per-key-channel
 *                 gate: dk = dv = 128), the call uses the tensor cores:
 *                 the gradient of the recurrence is the same recurrence with
 *                 its operands exchanged -- dq is the prefill of (d_out, v, k),
 *                 dk and dv are prefills of (v, d_out, q) and (k, q, d_out) run
 *                 backwards in time.  Per-head gate: the tcgen05 prefill kernel
 *                 runs three times between a reversing pass and a tail pass
 *                 (dg's final-state term and suffix sums, d_init's factor);
 *                 each run stores its gradient straight into dq, dk_out or
 *                 dv_out, and the dq and dk runs add dg's per-token terms
 *                 with fp32 atomics.  Per-key-channel gate: dv is one reversed run of the
 *                 per-key-channel tcgen05 prefill (whose decay falls on the
 *                 state's rows, as dv's does); dq and dk, whose decays fall on
 *                 the value side, stay on the CUDA cores.  Tensor-core results
 *                 have the prefill's accuracy (bf16 operands, fp32
 *                 accumulation).  Otherwise (or with a smaller workspace) the
 *                 fp32 CUDA-core kernels run.
 *   flags         GLA_FLAG_FP32_IO, GLA_FLAG_VECTOR_GATE, GLA_FLAG_FP32_OUT
 * The outputs and the workspace must not overlap one another or any input.
 * Empty sequences write d_init_state = d_final_state (or zeros).
 * Alignment: as gla_chunk_fwd; every output 16-byte aligned.
 */
gla_status gla_chunk_bwd(const void *q, const void *k, const void *v, const float *g,
                         float scale, const float *init_state, const void *d_out,
                         const float *d_final_state, void *dq, void *dk_out, void *dv_out,
                         float *dg, float *d_init_state, const int32_t *cu_seqlens, int B,
                         int H, int T, int dk, int dv, void *workspace,
                         size_t workspace_bytes, gla_stream_t stream, unsigned flags);

/*
 * gla_chunk_bwd_fixed_workspace -- gla_chunk_bwd for callers that cannot
 * allocate device memory when they need the gradient (code running inside a
 * caching allocator's callbacks, real-time threads that must not take the
 * driver's allocation lock, embedders whose memory is reserved up front): the
 * tensor-core path takes its workspace from a fixed device buffer inside the
 * library, so the call allocates nothing (no cudaMalloc, no cudaFree, no
 * allocating library routine).  The pages have no counterpart of this entry
 * point; it is a deployment convenience.
 *
 * The buffer is a static device array of GLA_BWD_FIXED_WORKSPACE_BYTES
 * (384 MiB).  With CUDA's lazy module loading (CUDA_MODULE_LOADING=LAZY, the
 * default) it is placed on a GPU the first time this function needs it there;
 * with eager loading every process that loads libgla.so reserves it on every
 * GPU it uses, forward-only users included.  Once placed it stays until the
 * process exits.  The first call that needs it on a device looks up its
 * device address (cudaGetSymbolAddress) and caches it: make that first call
 * before capturing any stream into a CUDA graph.  If the buffer cannot be
 * placed (not enough free memory when the module loads), the call returns
 * GLA_ERR_CUDA with the runtime's reason in gla_last_error_string(), and the
 * runtime's last-error state is cleared so that later calls are not charged
 * with it.
 *
 * Sizes: a call whose workspace need (gla_chunk_bwd_workspace_size) exceeds
 * the buffer is rejected with GLA_ERR_UNSUPPORTED before anything is enqueued,
 * and gla_last_error_string() states the need and the limit (with d_k = d_v =
 * 128 and 16 heads the buffer covers about 20,000 tokens, e.g. ten sequences
 * of 2,048);
 * such a call can go to gla_chunk_bwd with workspace = NULL, which runs the
 * CUDA-core kernels and needs no workspace either.  Calls that the tensor-core
 * path does not cover (fp32 I/O, other head sizes) need no workspace and run
 * on the CUDA cores as with gla_chunk_bwd.
 *
 * Sharing: every call on a GPU uses the same buffer, and a call overwrites
 * what the previous one left there (each call writes every workspace byte it
 * reads, so nothing depends on earlier contents).  Calls that overlap in time
 * on the GPU race on it: issue them on one stream, or synchronise between them.
 * Arguments, results and errors otherwise as gla_chunk_bwd.
 */
#define GLA_BWD_FIXED_WORKSPACE_BYTES ((size_t)384 << 20)
gla_status gla_chunk_bwd_fixed_workspace(const void *q, const void *k, const void *v,
                                         const float *g, float scale, const float *init_state,
                                         const void *d_out, const float *d_final_state,
                                         void *dq, void *dk_out, void *dv_out, float *dg,
                                         float *d_init_state, const int32_t *cu_seqlens, int B,
                                         int H, int T, int dk, int dv, gla_stream_t stream,
                                         unsigned flags);

/*
 * gla_chunk_bwd_workspace_size -- bytes of device workspace with which
 * gla_chunk_bwd takes its tensor-core path for these sizes and flags, or 0 when
 * that path does not cover them (the call then runs on the CUDA cores and
 * needs no workspace).  `packed` != 0: T counts packed rows (cu_seqlens given).
 * Pure host function.
 */
size_t gla_chunk_bwd_workspace_size(int B, int H, int T, int dk, int dv, int packed,
                                    unsigned flags);

/*
 * gla_chunk_fwd_kernel -- which kernel gla_chunk_fwd runs for a non-empty call
 * with these head sizes, chunk size and flags: "tensor_core" (a tcgen05
 * kernel: per-head or per-key-channel gate), "cuda_core" (the fp32 CUDA-core
 * kernel), or NULL when the call would be rejected.  Pure host function:
 * launches nothing.
 */
const char *gla_chunk_fwd_kernel(int dk, int dv, int chunk, unsigned flags);

/* Static English text for a status code (never NULL). */
const char *gla_status_string(gla_status status);

/*
 * gla_status_sync -- wait for `stream`, then read and clear the current GPU's
 * device status word.  Returns GLA_ERR_CUDA if the stream reports a CUDA error,
 * otherwise the most severe device-side status seen since the last call
 * (GLA_ERR_TIMEOUT over GLA_ERR_UNSUPPORTED over GLA_ERR_INVALID_ARG over
 * GLA_OK).  GLA_ERR_UNSUPPORTED here means a tensor-core kernel found its
 * shared-memory window not 1024-byte aligned and wrote nothing.
 */
gla_status gla_status_sync(gla_stream_t stream);

/* Text of the calling thread's most recent failure: the CUDA error behind a
 * GLA_ERR_CUDA, or the size limit behind gla_chunk_bwd_fixed_workspace's
 * GLA_ERR_UNSUPPORTED (thread-local storage, never NULL; "no error" if there
 * was none). */
const char *gla_last_error_string(void);

/*
 * gla_set_wait_limit_ns -- the wall-time limit of the waits with which the
 * warp roles of the tensor-core prefill kernels (gla_chunk_fwd, the mixer and
 * backward calls that run them) hand chunks to one another; 0 restores the
 * default, 2 s.  Process-wide, read at each launch; returns the previous
 * setting (0 = the default).  A wait that runs out makes the kernel stop
 * issuing work, let its own copies and matrix products land (with the default
 * limit), release its tensor memory and return: gla_status_sync then reports
 * GLA_ERR_TIMEOUT and the call's outputs are undefined.  For tests of that
 * path: a limit shorter than a chunk's hand-offs (about a microsecond) makes
 * the next call fail that way, and the call after the default is restored
 * runs normally.  The pages have no counterpart (failure handling is the
 * library's own).
 */
uint64_t gla_set_wait_limit_ns(uint64_t nanoseconds);

/* Library version, "major.minor.patch". */
const char *gla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GLA_H_ */
