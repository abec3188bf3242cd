/*
 * Lightning-attention oracle: plain, slow, fp64 CPU code.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file; it exists so the tests, the smoke check and the CPU baseline of
 * the benchmark have an independent statement of what the GPU kernels must
 * compute.  It shares no code, header, table or constant with the CUDA path.
 *
 * What is computed (MiniMax-01 technical report, CSDN full translation,
 * §2.2.1 "Lightning Attention"):
 *   - eq. 4, the causal "left product": O = [(Q K^T) (.) M] V with
 *     M_ts = 1 when t >= s and 0 otherwise;
 *   - eq. 5, the "right product" recursion kv_t = kv_{t-1} + k_t^T v_t,
 *     o_t = q_t kv_t, starting from kv_0 = 0;
 *   - the per-head exponential decay that the same report's Fig. 12 caption
 *     calls the diagonal decay matrix, and that the K3 report reading notes
 *     ("solution idea one: a positional decay term", RetNet style) describe:
 *     the weight of key/value u seen from query t is lambda_h^(t-u).
 * With the decay, the two forms become
 *     quadratic:  o_t = sum_{u<=t} lambda^(t-u) (q_t . k_u) v_u
 *     recurrent:  kv_t = lambda kv_{t-1} + k_t^T v_t,  o_t = q_t kv_t
 * and the state after the last token is sum_u lambda^(L-1-u) k_u^T v_u.
 * A sequence may continue from a cached state S0 (the prefix KV cache of
 * §3.3.1): S0 = sum over the earlier tokens u' < 0 of lambda^(-1-u') k^T v,
 * so kv_{-1} = S0 in the recursion and the left product gains the earlier
 * tokens' terms, sum_{u'<0} lambda^(t-u') (q_t . k_u') v_u' =
 * lambda^(t+1) q_t S0.  Without a cached state S0 = 0.
 * Normalisation, SiLU and gating are left out, as the report's derivation
 * does (§2.2.1).  Packed inputs ("data packing", §3.2) are independent
 * sequences: the state restarts from zero at every sequence start.
 *
 * Layouts (row-major, fp64):
 *   q, k, v, out   [T, H, d]       token-major, T = cu_seqlens[nseq]
 *   lam            [H]             per-head decay lambda_h in (0, 1]
 *   cu_seqlens     [nseq + 1]      sequence s is tokens [cu[s], cu[s+1])
 *   state          [nseq, H, d, d] state[s][h][i][j] = sum_u w_u k_u[i] v_u[j]
 *   initial_state  [nseq, H, d, d] cached state S0 per sequence (nullable)
 *
 * Parity pins for every function here live in the CPU test suite (hand
 * examples, closed forms, the agreement of the two independent forms,
 * exact rational brute force, packing and continuation invariants).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static int check_cu(const int32_t *cu, int nseq)
{
    if (nseq < 0 || cu == NULL) return 1;
    if (cu[0] != 0) return 1;
    for (int s = 0; s < nseq; ++s)
        if (cu[s + 1] < cu[s]) return 1;
    return 0;
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/* Number of threads OpenMP will use for the next parallel region. */
int la_oracle_max_threads(int nthreads)
{
#ifdef _OPENMP
    set_threads(nthreads);
    return omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/*
 * Quadratic ("left product", eq. 4) form, with the decay mask
 * M_tu = lambda^(t-u) for t >= u and 0 above the diagonal.
 * For every (sequence, head): S = Q K^T, P = S (.) M, O = P V, plus
 * lambda^(t+1) q_t S0 for a cached state S0 (initial_state, nullable).
 * head_sel (nullable) restricts the work to heads with head_sel[h] != 0;
 * rows of other heads are left untouched.  O(L^2 d) per (sequence, head).
 */
int la_oracle_quadratic(const double *q, const double *k, const double *v,
                        const double *lam, const int32_t *cu, int nseq,
                        int H, int d, const uint8_t *head_sel,
                        const double *initial_state, double *out, int nthreads)
{
    if (check_cu(cu, nseq) || H <= 0 || d <= 0) return 1;
    set_threads(nthreads);
    const long row = (long)H * d;
    const long npairs = (long)nseq * H;
#pragma omp parallel for schedule(dynamic, 1)
    for (long p = 0; p < npairs; ++p) {
        const int s = (int)(p / H), h = (int)(p % H);
        if (head_sel && !head_sel[h]) continue;
        const long t0 = cu[s], L = cu[s + 1] - cu[s];
        const double la = lam[h];
        for (long t = 0; t < L; ++t) {
            const double *qt = q + (t0 + t) * row + (long)h * d;
            double *ot = out + (t0 + t) * row + (long)h * d;
            for (int j = 0; j < d; ++j) ot[j] = 0.0;
            for (long u = 0; u <= t; ++u) {
                const double *ku = k + (t0 + u) * row + (long)h * d;
                const double *vu = v + (t0 + u) * row + (long)h * d;
                double s_tu = 0.0;                     /* (Q K^T)_tu */
                for (int i = 0; i < d; ++i) s_tu += qt[i] * ku[i];
                const double m_tu = pow(la, (double)(t - u)); /* decay mask */
                const double p_tu = s_tu * m_tu;
                for (int j = 0; j < d; ++j) ot[j] += p_tu * vu[j];
            }
            if (initial_state) {  /* the earlier tokens, through S0 */
                const double *s0 = initial_state + ((long)s * H + h) * d * d;
                const double w = pow(la, (double)(t + 1));
                for (int j = 0; j < d; ++j) {
                    double acc = 0.0;
                    for (int i = 0; i < d; ++i) acc += qt[i] * s0[(long)i * d + j];
                    ot[j] += w * acc;
                }
            }
        }
    }
    return 0;
}

/*
 * Recurrent ("right product", eq. 5) form with decay:
 *   kv <- lambda kv + k_t^T v_t ;  o_t = q_t kv   (update, then read),
 * kv starting at zero for every sequence, or at its cached state S0 when
 * initial_state is given.  Writes out (nullable) and the state after each
 * sequence's last token (nullable; S0 for an empty sequence).  O(L d^2) per
 * (sequence, head).  head_sel as in la_oracle_quadratic.
 */
int la_oracle_recurrent(const double *q, const double *k, const double *v,
                        const double *lam, const int32_t *cu, int nseq,
                        int H, int d, const uint8_t *head_sel,
                        const double *initial_state, double *out,
                        double *final_state, int nthreads)
{
    if (check_cu(cu, nseq) || H <= 0 || d <= 0) return 1;
    set_threads(nthreads);
    const long row = (long)H * d;
    const long npairs = (long)nseq * H;
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (long p = 0; p < npairs; ++p) {
        const int s = (int)(p / H), h = (int)(p % H);
        if (head_sel && !head_sel[h]) continue;
        double *kv = (double *)calloc((size_t)d * d, sizeof(double));
        if (!kv) {
#pragma omp atomic write
            err = 2;
            continue;
        }
        if (initial_state)
            memcpy(kv, initial_state + ((long)s * H + h) * d * d,
                   sizeof(double) * (size_t)d * d);
        const long t0 = cu[s], L = cu[s + 1] - cu[s];
        const double la = lam[h];
        for (long t = 0; t < L; ++t) {
            const double *qt = q + (t0 + t) * row + (long)h * d;
            const double *kt = k + (t0 + t) * row + (long)h * d;
            const double *vt = v + (t0 + t) * row + (long)h * d;
            for (int i = 0; i < d; ++i)
                for (int j = 0; j < d; ++j)
                    kv[(long)i * d + j] = la * kv[(long)i * d + j] + kt[i] * vt[j];
            if (out) {
                double *ot = out + (t0 + t) * row + (long)h * d;
                for (int j = 0; j < d; ++j) {
                    double acc = 0.0;
                    for (int i = 0; i < d; ++i) acc += qt[i] * kv[(long)i * d + j];
                    ot[j] = acc;
                }
            }
        }
        if (final_state)
            memcpy(final_state + ((long)s * H + h) * d * d, kv,
                   sizeof(double) * (size_t)d * d);
        free(kv);
    }
    return err;
}

/*
 * One decode step (the recurrent form applied to a single new token per
 * sequence, continuing from a cached state):
 *   state[b][h] <- lambda_h state[b][h] + k_b^T v_b ;  o_b = q_b state[b][h].
 * q, k, v, out: [batch, H, d]; state: [batch, H, d, d], updated in place.
 */
int la_oracle_decode(const double *q, const double *k, const double *v,
                     const double *lam, double *state, int batch, int H, int d,
                     double *out, int nthreads)
{
    if (batch < 0 || H <= 0 || d <= 0) return 1;
    set_threads(nthreads);
    const long npairs = (long)batch * H;
#pragma omp parallel for schedule(static)
    for (long p = 0; p < npairs; ++p) {
        const int h = (int)(p % H);
        const double *qb = q + p * d, *kb = k + p * d, *vb = v + p * d;
        double *kv = state + p * d * d;
        const double la = lam[h];
        for (int i = 0; i < d; ++i)
            for (int j = 0; j < d; ++j)
                kv[(long)i * d + j] = la * kv[(long)i * d + j] + kb[i] * vb[j];
        for (int j = 0; j < d; ++j) {
            double acc = 0.0;
            for (int i = 0; i < d; ++i) acc += qb[i] * kv[(long)i * d + j];
            out[p * d + j] = acc;
        }
    }
    return 0;
}

/*
 * Gradients of the quadratic form (training, §2.2.1 and the report's TGS
 * measurements of §2.2.2): for a loss with dL/do_t = dout_t,
 *   dq_t = sum_{u<=t} lambda^(t-u) (dout_t . v_u) k_u
 *   dk_u = sum_{t>=u} lambda^(t-u) (dout_t . v_u) q_t
 *   dv_u = sum_{t>=u} lambda^(t-u) (q_t . k_u) dout_t
 * per sequence and head (zero state at every sequence start), written out
 * term by term from o_t = sum_{u<=t} lambda^(t-u) (q_t . k_u) v_u.
 * All arrays [T, H, d]; dq, dk, dv are overwritten.  O(L^2 d) per
 * (sequence, head).
 */
int la_oracle_backward(const double *q, const double *k, const double *v,
                       const double *lam, const int32_t *cu, int nseq, int H,
                       int d, const double *dout, double *dq, double *dk,
                       double *dv, int nthreads)
{
    if (check_cu(cu, nseq) || H <= 0 || d <= 0) return 1;
    set_threads(nthreads);
    const long row = (long)H * d;
    const long npairs = (long)nseq * H;
#pragma omp parallel for schedule(dynamic, 1)
    for (long p = 0; p < npairs; ++p) {
        const int s = (int)(p / H), h = (int)(p % H);
        const long t0 = cu[s], L = cu[s + 1] - cu[s];
        const double la = lam[h];
        for (long t = 0; t < L; ++t)
            for (int j = 0; j < d; ++j) {
                const long o = (t0 + t) * row + (long)h * d + j;
                dq[o] = 0.0;
                dk[o] = 0.0;
                dv[o] = 0.0;
            }
        for (long t = 0; t < L; ++t) {
            const double *qt = q + (t0 + t) * row + (long)h * d;
            const double *gt = dout + (t0 + t) * row + (long)h * d;
            double *dqt = dq + (t0 + t) * row + (long)h * d;
            for (long u = 0; u <= t; ++u) {
                const double *ku = k + (t0 + u) * row + (long)h * d;
                const double *vu = v + (t0 + u) * row + (long)h * d;
                double *dku = dk + (t0 + u) * row + (long)h * d;
                double *dvu = dv + (t0 + u) * row + (long)h * d;
                const double w = pow(la, (double)(t - u));
                double g_v = 0.0, q_k = 0.0;   /* dout_t . v_u, q_t . k_u */
                for (int i = 0; i < d; ++i) {
                    g_v += gt[i] * vu[i];
                    q_k += qt[i] * ku[i];
                }
                for (int i = 0; i < d; ++i) {
                    dqt[i] += w * g_v * ku[i];
                    dku[i] += w * g_v * qt[i];
                    dvu[i] += w * q_k * gt[i];
                }
            }
        }
    }
    return 0;
}

/*
 * Channel-wise decay (the K3 report reading notes, "gated DeltaNet ...
 * changes the scalar decay to a channel-wise decay, which can fall back to
 * the uniform one"; the decay acts on the key channels, the dimension Q and
 * K share): lam_cw[h][i] is the decay of key channel i of head h, so
 *   quadratic:  o_t = sum_{u<=t} (sum_i q_t[i] k_u[i] lam_i^(t-u)) v_u
 *   recurrent:  kv_t[i][j] = lam_i kv_{t-1}[i][j] + k_t[i] v_t[j],
 *               o_t = q_t kv_t
 * starting from zero (or initial_state) at every sequence start.  With all
 * lam_i equal these are la_oracle_quadratic / la_oracle_recurrent.
 */
int la_oracle_quadratic_cw(const double *q, const double *k, const double *v,
                           const double *lam_cw, const int32_t *cu, int nseq, int H,
                           int d, const double *initial_state, double *out, int nthreads)
{
    if (check_cu(cu, nseq) || H <= 0 || d <= 0) return 1;
    set_threads(nthreads);
    const long row = (long)H * d;
    const long npairs = (long)nseq * H;
#pragma omp parallel for schedule(dynamic, 1)
    for (long p = 0; p < npairs; ++p) {
        const int s = (int)(p / H), h = (int)(p % H);
        const double *la = lam_cw + (long)h * d;
        const long t0 = cu[s], L = cu[s + 1] - cu[s];
        for (long t = 0; t < L; ++t) {
            const double *qt = q + (t0 + t) * row + (long)h * d;
            double *ot = out + (t0 + t) * row + (long)h * d;
            for (int j = 0; j < d; ++j) ot[j] = 0.0;
            for (long u = 0; u <= t; ++u) {
                const double *ku = k + (t0 + u) * row + (long)h * d;
                const double *vu = v + (t0 + u) * row + (long)h * d;
                double s_tu = 0.0;  /* sum_i q_t[i] k_u[i] lam_i^(t-u) */
                for (int i = 0; i < d; ++i) s_tu += qt[i] * ku[i] * pow(la[i], (double)(t - u));
                for (int j = 0; j < d; ++j) ot[j] += s_tu * vu[j];
            }
            if (initial_state) {  /* the earlier tokens, through S0 */
                const double *s0 = initial_state + ((long)s * H + h) * d * d;
                for (int j = 0; j < d; ++j) {
                    double acc = 0.0;
                    for (int i = 0; i < d; ++i)
                        acc += qt[i] * pow(la[i], (double)(t + 1)) * s0[(long)i * d + j];
                    ot[j] += acc;
                }
            }
        }
    }
    return 0;
}

int la_oracle_recurrent_cw(const double *q, const double *k, const double *v,
                           const double *lam_cw, const int32_t *cu, int nseq, int H,
                           int d, const double *initial_state, double *out,
                           double *final_state, int nthreads)
{
    if (check_cu(cu, nseq) || H <= 0 || d <= 0) return 1;
    set_threads(nthreads);
    const long row = (long)H * d;
    const long npairs = (long)nseq * H;
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (long p = 0; p < npairs; ++p) {
        const int s = (int)(p / H), h = (int)(p % H);
        const double *la = lam_cw + (long)h * d;
        double *kv = (double *)calloc((size_t)d * d, sizeof(double));
        if (!kv) {
#pragma omp atomic write
            err = 2;
            continue;
        }
        if (initial_state)
            memcpy(kv, initial_state + ((long)s * H + h) * d * d, sizeof(double) * (size_t)d * d);
        const long t0 = cu[s], L = cu[s + 1] - cu[s];
        for (long t = 0; t < L; ++t) {
            const double *qt = q + (t0 + t) * row + (long)h * d;
            const double *kt = k + (t0 + t) * row + (long)h * d;
            const double *vt = v + (t0 + t) * row + (long)h * d;
            for (int i = 0; i < d; ++i)
                for (int j = 0; j < d; ++j)
                    kv[(long)i * d + j] = la[i] * kv[(long)i * d + j] + kt[i] * vt[j];
            if (out) {
                double *ot = out + (t0 + t) * row + (long)h * d;
                for (int j = 0; j < d; ++j) {
                    double acc = 0.0;
                    for (int i = 0; i < d; ++i) acc += qt[i] * kv[(long)i * d + j];
                    ot[j] = acc;
                }
            }
        }
        if (final_state)
            memcpy(final_state + ((long)s * H + h) * d * d, kv, sizeof(double) * (size_t)d * d);
        free(kv);
    }
    return err;
}

/* One decode step with channel-wise decay: state[i][j] <- lam_i state[i][j]
 * + k[i] v[j], o = q state (after the update). */
int la_oracle_decode_cw(const double *q, const double *k, const double *v,
                        const double *lam_cw, double *state, int batch, int H, int d,
                        double *out, int nthreads)
{
    if (batch < 0 || H <= 0 || d <= 0) return 1;
    set_threads(nthreads);
    const long npairs = (long)batch * H;
#pragma omp parallel for schedule(static)
    for (long p = 0; p < npairs; ++p) {
        const int h = (int)(p % H);
        const double *qb = q + p * d, *kb = k + p * d, *vb = v + p * d;
        const double *la = lam_cw + (long)h * d;
        double *kv = state + p * d * d;
        for (int i = 0; i < d; ++i)
            for (int j = 0; j < d; ++j)
                kv[(long)i * d + j] = la[i] * kv[(long)i * d + j] + kb[i] * vb[j];
        for (int j = 0; j < d; ++j) {
            double acc = 0.0;
            for (int i = 0; i < d; ++i) acc += qb[i] * kv[(long)i * d + j];
            out[p * d + j] = acc;
        }
    }
    return 0;
}
