/*
 * gla_oracle.c -- TEST INFRASTRUCTURE, not part of the product path.
 *
 * A plain, slow, fp64 CPU statement of gated linear attention (GLA), written
 * from the "i14 Laplace 3B on AWS Trainium2" blog page (section "i14 and the
 * Laplace 3B architecture", paragraph "GLA mixer", and section "Challenge 1:
 * Using native PyTorch on Trainium for GLA", Figure 3).  Only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg may load this library.
 * It shares no code, header or constant with the CUDA library.
 *
 * What is computed (the page's equation images were lost; the prose fixes the
 * shape of each step, and the gate is generalised to a per-token log-decay):
 *
 *   S_t = diag(exp g_t) S_{t-1} + k_t^T v_t      (the old state shrinks by the
 *                                                 head's decay and the token's
 *                                                 key/value pair is added as a
 *                                                 rank-one matrix)
 *   o_t = scale * q_t S_t                        (the query reads the state
 *                                                 once this token is in it)
 *
 * g_t is either one number per (token, head) -- every row of S decays alike,
 * the page's Simple GLA -- or one number per (token, head, key channel), in
 * which case row i of S (key channel i) decays by exp(g_t[i]).
 *
 * Layouts (all fp64, row-major, "token-major"):
 *   q, k   [R, H, dk]      v, out [R, H, dv]
 *   g      [R, H]          (scalar gate)   or [R, H, dk] (vector gate)
 *   states [NS, H, dk, dv]
 * R is the number of token rows: B*T for a dense batch (sequence s owns rows
 * s*T .. s*T+T-1), or cu_seqlens[NS] for a packed batch (sequence s owns rows
 * cu_seqlens[s] .. cu_seqlens[s+1]-1).  NS is B in both cases.
 *
 * Three entry points:
 *   gla_oracle_recurrent_f64  token-by-token recurrence (the definition)
 *   gla_oracle_chunked_f64    the page's chunked form: per chunk, causal
 *                             attention with decay weights inside the chunk
 *                             plus what the carried-in state contributes,
 *                             then one state step with the chunk's total decay
 *   gla_oracle_decode_step_f64 one recurrent step for N independent states
 *   gla_oracle_backward_f64   the gradient of the recurrence (reverse mode)
 *
 * Return value: 0 on success, -1 on a bad argument (nothing is written).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* exp of the log-decay that token row `row` applies to key channel i of head h. */
static double decay_factor(const double *g, int vector_gate, long row, int H, int h,
                           int dk, int i)
{
    if (vector_gate)
        return exp(g[((size_t)row * H + h) * dk + i]);
    return exp(g[(size_t)row * H + h]);
}

/* First row and length of sequence s. */
static int seq_bounds(const int32_t *cu_seqlens, int s, int T, long *start, long *len)
{
    if (cu_seqlens) {
        *start = cu_seqlens[s];
        *len = (long)cu_seqlens[s + 1] - (long)cu_seqlens[s];
        if (*len < 0)
            return -1;
    } else {
        *start = (long)s * T;
        *len = T;
    }
    return 0;
}

static int check_args(const void *q, const void *k, const void *v, const void *g,
                      const void *out, const int32_t *cu_seqlens, int B, int H, int T,
                      int dk, int dv)
{
    if (!q || !k || !v || !g || !out)
        return -1;
    if (B < 0 || H < 0 || T < 0 || dk <= 0 || dv <= 0)
        return -1;
    if (cu_seqlens) {
        if (cu_seqlens[0] != 0)
            return -1;
        for (int s = 0; s < B; ++s)
            if (cu_seqlens[s + 1] < cu_seqlens[s])
                return -1;
    }
    return 0;
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/* ------------------------------------------------------------------------- */
/* The recurrence, one token at a time.                                      */
/* ------------------------------------------------------------------------- */
int gla_oracle_recurrent_f64(const double *q, const double *k, const double *v,
                             const double *g, int vector_gate, double scale,
                             const double *init_state, double *out,
                             double *final_state, const int32_t *cu_seqlens, int B,
                             int H, int T, int dk, int dv, int nthreads)
{
    if (check_args(q, k, v, g, out, cu_seqlens, B, H, T, dk, dv))
        return -1;
    set_threads(nthreads);
    const long pairs = (long)B * H;
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
    for (long p = 0; p < pairs; ++p) {
        const int s = (int)(p / H), h = (int)(p % H);
        long start, len;
        if (seq_bounds(cu_seqlens, s, T, &start, &len)) {
            failed |= 1;
            continue;
        }
        double *S = (double *)malloc(sizeof(double) * (size_t)dk * dv);
        if (!S) {
            failed |= 1;
            continue;
        }
        const size_t state_off = (size_t)p * dk * dv;
        if (init_state)
            memcpy(S, init_state + state_off, sizeof(double) * (size_t)dk * dv);
        else
            memset(S, 0, sizeof(double) * (size_t)dk * dv);

        for (long t = 0; t < len; ++t) {
            const long row = start + t;
            const double *qt = q + ((size_t)row * H + h) * dk;
            const double *kt = k + ((size_t)row * H + h) * dk;
            const double *vt = v + ((size_t)row * H + h) * dv;
            double *ot = out + ((size_t)row * H + h) * dv;
            /* S <- diag(exp g_t) S + k_t^T v_t */
            for (int i = 0; i < dk; ++i) {
                const double a = decay_factor(g, vector_gate, row, H, h, dk, i);
                for (int j = 0; j < dv; ++j)
                    S[(size_t)i * dv + j] = a * S[(size_t)i * dv + j] + kt[i] * vt[j];
            }
            /* o_t <- scale * q_t S */
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i)
                    acc += qt[i] * S[(size_t)i * dv + j];
                ot[j] = scale * acc;
            }
        }
        if (final_state)
            memcpy(final_state + state_off, S, sizeof(double) * (size_t)dk * dv);
        free(S);
    }
    return failed ? -1 : 0;
}

/* ------------------------------------------------------------------------- */
/* The chunked form.                                                         */
/*                                                                           */
/* Within a chunk holding tokens 0..n-1 (relative to the chunk start):       */
/*   D(j, t)[i] = prod_{u=j+1..t} exp(g_u[i])   decay from token j to t      */
/*   E(t)[i]    = prod_{u=0..t}   exp(g_u[i])   decay from the chunk start   */
/*   o_t = scale * ( sum_{j<=t} (q_t . (k_j * D(j,t))) v_j                   */
/*                   + (q_t * E(t)) S_prev )                                 */
/*   S_next = diag(E(n-1)) S_prev + sum_j (k_j * D(j, n-1))^T v_j            */
/* The decays are running products of exp(g), so g = -inf gives exactly 0.  */
/* Chunks restart at each sequence start; the last chunk may be partial.     */
/* ------------------------------------------------------------------------- */
int gla_oracle_chunked_f64(const double *q, const double *k, const double *v,
                           const double *g, int vector_gate, double scale,
                           const double *init_state, double *out, double *final_state,
                           const int32_t *cu_seqlens, int B, int H, int T, int dk, int dv,
                           int chunk, int nthreads)
{
    if (check_args(q, k, v, g, out, cu_seqlens, B, H, T, dk, dv) || chunk <= 0)
        return -1;
    set_threads(nthreads);
    const long pairs = (long)B * H;
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
    for (long p = 0; p < pairs; ++p) {
        const int s = (int)(p / H), h = (int)(p % H);
        long start, len;
        if (seq_bounds(cu_seqlens, s, T, &start, &len)) {
            failed |= 1;
            continue;
        }
        const size_t SD = (size_t)dk * dv;
        double *S = (double *)malloc(sizeof(double) * SD);
        double *Snew = (double *)malloc(sizeof(double) * SD);
        double *D = (double *)malloc(sizeof(double) * (size_t)dk);  /* D(j,t) for one t */
        double *E = (double *)malloc(sizeof(double) * (size_t)dk);  /* E(t) */
        double *acc = (double *)malloc(sizeof(double) * (size_t)dv);
        if (!S || !Snew || !D || !E || !acc) {
            free(S); free(Snew); free(D); free(E); free(acc);
            failed |= 1;
            continue;
        }
        if (init_state)
            memcpy(S, init_state + (size_t)p * SD, sizeof(double) * SD);
        else
            memset(S, 0, sizeof(double) * SD);

        for (long c0 = 0; c0 < len; c0 += chunk) {
            const long n = (len - c0 < chunk) ? (len - c0) : chunk;
            const long base = start + c0;
            /* outputs of the chunk */
            for (long t = 0; t < n; ++t) {
                const long rt = base + t;
                const double *qt = q + ((size_t)rt * H + h) * dk;
                for (int j = 0; j < dv; ++j)
                    acc[j] = 0.0;
                /* intra-chunk: walk j from t down to 0, extending D(j,t) by one gate */
                for (int i = 0; i < dk; ++i)
                    D[i] = 1.0;
                for (long jj = t; jj >= 0; --jj) {
                    if (jj < t)
                        for (int i = 0; i < dk; ++i)
                            D[i] *= decay_factor(g, vector_gate, base + jj + 1, H, h, dk, i);
                    const double *kj = k + ((size_t)(base + jj) * H + h) * dk;
                    const double *vj = v + ((size_t)(base + jj) * H + h) * dv;
                    double score = 0.0;
                    for (int i = 0; i < dk; ++i)
                        score += qt[i] * kj[i] * D[i];
                    for (int j = 0; j < dv; ++j)
                        acc[j] += score * vj[j];
                }
                /* inter-chunk: the state at the chunk start, decayed to token t */
                for (int i = 0; i < dk; ++i) {
                    E[i] = 1.0;
                    for (long u = 0; u <= t; ++u)
                        E[i] *= decay_factor(g, vector_gate, base + u, H, h, dk, i);
                }
                for (int i = 0; i < dk; ++i) {
                    const double qe = qt[i] * E[i];
                    for (int j = 0; j < dv; ++j)
                        acc[j] += qe * S[(size_t)i * dv + j];
                }
                double *ot = out + ((size_t)rt * H + h) * dv;
                for (int j = 0; j < dv; ++j)
                    ot[j] = scale * acc[j];
            }
            /* state step over the whole chunk */
            for (int i = 0; i < dk; ++i) {
                E[i] = 1.0;
                for (long u = 0; u < n; ++u)
                    E[i] *= decay_factor(g, vector_gate, base + u, H, h, dk, i);
            }
            for (int i = 0; i < dk; ++i)
                for (int j = 0; j < dv; ++j)
                    Snew[(size_t)i * dv + j] = E[i] * S[(size_t)i * dv + j];
            for (int i = 0; i < dk; ++i)
                D[i] = 1.0;
            for (long jj = n - 1; jj >= 0; --jj) {
                if (jj < n - 1)
                    for (int i = 0; i < dk; ++i)
                        D[i] *= decay_factor(g, vector_gate, base + jj + 1, H, h, dk, i);
                const double *kj = k + ((size_t)(base + jj) * H + h) * dk;
                const double *vj = v + ((size_t)(base + jj) * H + h) * dv;
                for (int i = 0; i < dk; ++i) {
                    const double kd = kj[i] * D[i];
                    for (int j = 0; j < dv; ++j)
                        Snew[(size_t)i * dv + j] += kd * vj[j];
                }
            }
            double *tmp = S;
            S = Snew;
            Snew = tmp;
        }
        if (final_state)
            memcpy(final_state + (size_t)p * SD, S, sizeof(double) * SD);
        free(S); free(Snew); free(D); free(E); free(acc);
    }
    return failed ? -1 : 0;
}

/* ------------------------------------------------------------------------- */
/* One decode step for N independent sequences (the serving form: one token */
/* per sequence, each sequence owning a fixed-size state page).              */
/*   q, k [N, H, dk]  v, out [N, H, dv]  g [N, H] or [N, H, dk]               */
/*   state [N, H, dk, dv], updated in place.                                 */
/* ------------------------------------------------------------------------- */
int gla_oracle_decode_step_f64(const double *q, const double *k, const double *v,
                               const double *g, int vector_gate, double scale,
                               double *state, double *out, int N, int H, int dk, int dv,
                               int nthreads)
{
    if (!q || !k || !v || !g || !state || !out || N < 0 || H < 0 || dk <= 0 || dv <= 0)
        return -1;
    set_threads(nthreads);
    const long pairs = (long)N * H;
#pragma omp parallel for schedule(static)
    for (long p = 0; p < pairs; ++p) {
        const int h = (int)(p % H);
        const long row = p / H;
        double *S = state + (size_t)p * dk * dv;
        const double *qt = q + (size_t)p * dk;
        const double *kt = k + (size_t)p * dk;
        const double *vt = v + (size_t)p * dv;
        for (int i = 0; i < dk; ++i) {
            const double a = decay_factor(g, vector_gate, row, H, h, dk, i);
            for (int j = 0; j < dv; ++j)
                S[(size_t)i * dv + j] = a * S[(size_t)i * dv + j] + kt[i] * vt[j];
        }
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int i = 0; i < dk; ++i)
                acc += qt[i] * S[(size_t)i * dv + j];
            out[(size_t)p * dv + j] = scale * acc;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* The gradient of the recurrence (reverse mode, one token at a time).       */
/*                                                                           */
/* For a loss L with dL/do_t = d_out[t] and dL/dS_final = d_final (zero when */
/* absent), let Sbar_t = dL/dS_t, the gradient reaching the state after      */
/* token t through every later readout and step.  Going backwards:           */
/*   Sbar_t      = scale * q_t^T do_t + diag(exp g_{t+1}) Sbar_{t+1}          */
/*                 (Sbar at the last token starts from d_final)              */
/*   dq_t        = scale * S_t do_t^T           (forward sweep)              */
/*   dk_t        = Sbar_t v_t^T                                              */
/*   dv_t        = k_t Sbar_t                                                */
/*   dg_t[i]     = exp(g_t[i]) * sum_j S_{t-1}[i][j] * Sbar_t[i][j]          */
/*                 (summed over i for the per-head gate)                     */
/*   d_init      = diag(exp g_0) Sbar_0                                      */
/* S_{t-1} is needed in reverse order: the forward sweep keeps the state at  */
/* the start of every BWD_SEGMENT tokens, and the reverse sweep recomputes   */
/* one segment's states from its checkpoint before walking it backwards.     */
/* No gate clamping: this is the exact gradient of the recurrence above.     */
/* ------------------------------------------------------------------------- */
#define BWD_SEGMENT 64

int gla_oracle_backward_f64(const double *q, const double *k, const double *v,
                            const double *g, int vector_gate, double scale,
                            const double *init_state, const double *d_out,
                            const double *d_final, double *dq, double *dk_out,
                            double *dv_out, double *dg, double *d_init,
                            const int32_t *cu_seqlens, int B, int H, int T, int dk, int dv,
                            int nthreads)
{
    if (check_args(q, k, v, g, d_out, cu_seqlens, B, H, T, dk, dv) || !dq || !dk_out ||
        !dv_out || !dg)
        return -1;
    set_threads(nthreads);
    const long pairs = (long)B * H;
    const size_t SD = (size_t)dk * dv;
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
    for (long p = 0; p < pairs; ++p) {
        const int s = (int)(p / H), h = (int)(p % H);
        long start, len;
        if (seq_bounds(cu_seqlens, s, T, &start, &len)) {
            failed |= 1;
            continue;
        }
        const long nseg = (len + BWD_SEGMENT - 1) / BWD_SEGMENT;
        /* ckpt[m] = state before token m * BWD_SEGMENT; seg[r] = S_{t0 + r - 1} */
        double *ckpt = (double *)malloc(sizeof(double) * SD * (size_t)(nseg + 1));
        double *seg = (double *)malloc(sizeof(double) * SD * (BWD_SEGMENT + 1));
        double *Sbar = (double *)malloc(sizeof(double) * SD);
        double *S = (double *)malloc(sizeof(double) * SD);
        if (!ckpt || !seg || !Sbar || !S) {
            free(ckpt); free(seg); free(Sbar); free(S);
            failed |= 1;
            continue;
        }
        if (init_state)
            memcpy(S, init_state + (size_t)p * SD, sizeof(double) * SD);
        else
            memset(S, 0, sizeof(double) * SD);

        /* forward sweep: checkpoints and dq_t = scale * S_t do_t^T */
        for (long t = 0; t < len; ++t) {
            if (t % BWD_SEGMENT == 0)
                memcpy(ckpt + SD * (size_t)(t / BWD_SEGMENT), S, sizeof(double) * SD);
            const long row = start + t;
            const double *kt = k + ((size_t)row * H + h) * dk;
            const double *vt = v + ((size_t)row * H + h) * dv;
            const double *dot = d_out + ((size_t)row * H + h) * dv;
            double *dqt = dq + ((size_t)row * H + h) * dk;
            for (int i = 0; i < dk; ++i) {
                const double a = decay_factor(g, vector_gate, row, H, h, dk, i);
                double acc = 0.0;
                for (int j = 0; j < dv; ++j) {
                    S[(size_t)i * dv + j] = a * S[(size_t)i * dv + j] + kt[i] * vt[j];
                    acc += S[(size_t)i * dv + j] * dot[j];
                }
                dqt[i] = scale * acc;
            }
        }

        /* reverse sweep */
        if (d_final)
            memcpy(Sbar, d_final + (size_t)p * SD, sizeof(double) * SD);
        else
            memset(Sbar, 0, sizeof(double) * SD);
        for (long m = nseg - 1; m >= 0; --m) {
            const long t0 = m * BWD_SEGMENT;
            const long t1 = (t0 + BWD_SEGMENT < len) ? t0 + BWD_SEGMENT : len;
            /* seg[0] = S_{t0-1} (the checkpoint), seg[r] = S_{t0+r-1} */
            memcpy(seg, ckpt + SD * (size_t)m, sizeof(double) * SD);
            for (long t = t0; t < t1 - 1; ++t) {
                const long row = start + t;
                const double *kt = k + ((size_t)row * H + h) * dk;
                const double *vt = v + ((size_t)row * H + h) * dv;
                const double *prev = seg + SD * (size_t)(t - t0);
                double *next = seg + SD * (size_t)(t - t0 + 1);
                for (int i = 0; i < dk; ++i) {
                    const double a = decay_factor(g, vector_gate, row, H, h, dk, i);
                    for (int j = 0; j < dv; ++j)
                        next[(size_t)i * dv + j] = a * prev[(size_t)i * dv + j] + kt[i] * vt[j];
                }
            }
            for (long t = t1 - 1; t >= t0; --t) {
                const long row = start + t;
                const double *qt = q + ((size_t)row * H + h) * dk;
                const double *kt = k + ((size_t)row * H + h) * dk;
                const double *vt = v + ((size_t)row * H + h) * dv;
                const double *dot = d_out + ((size_t)row * H + h) * dv;
                const double *Sprev = seg + SD * (size_t)(t - t0);   /* S_{t-1} */
                double *dkt = dk_out + ((size_t)row * H + h) * dk;
                double *dvt = dv_out + ((size_t)row * H + h) * dv;
                /* Sbar <- Sbar_t: add this token's readout */
                for (int i = 0; i < dk; ++i)
                    for (int j = 0; j < dv; ++j)
                        Sbar[(size_t)i * dv + j] += scale * qt[i] * dot[j];
                for (int i = 0; i < dk; ++i) {
                    double acc = 0.0;
                    for (int j = 0; j < dv; ++j)
                        acc += Sbar[(size_t)i * dv + j] * vt[j];
                    dkt[i] = acc;
                }
                for (int j = 0; j < dv; ++j) {
                    double acc = 0.0;
                    for (int i = 0; i < dk; ++i)
                        acc += kt[i] * Sbar[(size_t)i * dv + j];
                    dvt[j] = acc;
                }
                double gsum = 0.0;
                for (int i = 0; i < dk; ++i) {
                    const double a = decay_factor(g, vector_gate, row, H, h, dk, i);
                    double acc = 0.0;
                    for (int j = 0; j < dv; ++j)
                        acc += Sprev[(size_t)i * dv + j] * Sbar[(size_t)i * dv + j];
                    if (vector_gate)
                        dg[((size_t)row * H + h) * dk + i] = a * acc;
                    else
                        gsum += a * acc;
                    /* Sbar <- diag(exp g_t) Sbar: the gradient reaching S_{t-1} */
                    for (int j = 0; j < dv; ++j)
                        Sbar[(size_t)i * dv + j] *= a;
                }
                if (!vector_gate)
                    dg[(size_t)row * H + h] = gsum;
            }
        }
        if (d_init)
            memcpy(d_init + (size_t)p * SD, Sbar, sizeof(double) * SD);
        free(ckpt); free(seg); free(Sbar); free(S);
    }
    return failed ? -1 : 0;
}

/* Number of threads OpenMP would use (1 without OpenMP). */
int gla_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
