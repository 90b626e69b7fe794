/*
 * kda_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU restatement of Kimi Delta Attention (KDA), the gated
 * delta rule with a per-channel decay.  It exists so that the CUDA path can be
 * checked against something obviously correct; nothing in the product path may
 * call it.  It shares no code, header or constant with the CUDA library.
 *
 * Source of every step: "はじめての自然言語処理 -- Kimi K3" (ogis-ri.co.jp),
 * section 3.1 "KDA (Kimi Delta Attention)":
 *   - the state S_t is d_k x d_v, q_t and k_t are d_k vectors, v_t a d_v vector,
 *     alpha_t a d_k vector of per-channel retention factors in (0,1), beta_t a
 *     scalar write strength in (0,1), and the read-out is o_t = S_t^T q_t
 *     (the shapes list and the read-out paragraph);
 *   - the delta rule written out in four steps, in this order (the paragraph
 *     that decomposes the delta rule, "S_t^-, v^_t, e_t, S_t"):
 *         S^-  = Diag(alpha_t) S_{t-1}          (forget, per key channel)
 *         vhat = (S^-)^T k_t                    (read with the current key)
 *         e    = v_t - vhat                     (the "delta")
 *         S_t  = S^- + beta_t k_t e^T           (write the correction only)
 *     which folds into S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1}
 *     + beta_t k_t v_t^T, the report's equation (1).
 *   - alpha_t = exp(g_t) with g_t the per-channel log decay (the lower-bound
 *     paragraph of the same section).
 * Readings taken where the page is silent: o_t uses S_t after the write of
 * token t (the intra-chunk mask there is i <= j, inclusive); no scale is applied
 * to q; q and k are used exactly as given (their L2 normalisation is the
 * caller's job); each packed sequence starts its own recurrence.
 *
 * Layouts (all row-major, double):
 *   q, k, g : [tokens][H][dk]     v, out : [tokens][H][dv]     beta : [tokens][H]
 *   states  : [N][H][dk][dv]      cu     : int64 [N+1] token offsets
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>

/* One token of the recurrence on one (sequence, head) state, in place.
 * e is caller scratch of dv doubles. */
static void kda_oracle_token(double *S, int64_t dk, int64_t dv,
                             const double *q, const double *k, const double *v,
                             const double *g, double beta, double *o, double *e)
{
    int64_t i, j;
    /* forget: S <- Diag(exp g) S  (alpha scales the key channel, i.e. row i) */
    for (i = 0; i < dk; ++i) {
        const double a = exp(g[i]);
        for (j = 0; j < dv; ++j) S[i * dv + j] *= a;
    }
    /* read with the current key: vhat = S^T k, then e = v - vhat */
    for (j = 0; j < dv; ++j) e[j] = 0.0;
    for (i = 0; i < dk; ++i)
        for (j = 0; j < dv; ++j) e[j] += S[i * dv + j] * k[i];
    for (j = 0; j < dv; ++j) e[j] = v[j] - e[j];
    /* write the correction: S <- S + beta k e^T */
    for (i = 0; i < dk; ++i) {
        const double bk = beta * k[i];
        for (j = 0; j < dv; ++j) S[i * dv + j] += bk * e[j];
    }
    /* read-out with the updated state: o = S^T q */
    for (j = 0; j < dv; ++j) o[j] = 0.0;
    for (i = 0; i < dk; ++i)
        for (j = 0; j < dv; ++j) o[j] += S[i * dv + j] * q[i];
}

/* Prefill / resume: runs the recurrence for every (sequence n, head h) unit
 * u = n*H + h with unit_begin <= u < unit_end.  s0 may be NULL (zero start);
 * sT may be NULL (final state not wanted).  Returns 0, or -1 if scratch could
 * not be allocated. */
int kda_oracle_forward(const double *q, const double *k, const double *v,
                       const double *g, const double *beta, const double *s0,
                       const int64_t *cu, int64_t N, int64_t H, int64_t dk,
                       int64_t dv, double *out, double *sT,
                       int64_t unit_begin, int64_t unit_end)
{
    double *S = (double *)malloc((size_t)(dk * dv + dv) * sizeof(double));
    if (!S) return -1;
    double *e = S + dk * dv;
    for (int64_t u = unit_begin; u < unit_end && u < N * H; ++u) {
        const int64_t n = u / H, h = u % H;
        const double *init = s0 ? s0 + (n * H + h) * dk * dv : NULL;
        for (int64_t x = 0; x < dk * dv; ++x) S[x] = init ? init[x] : 0.0;
        for (int64_t t = cu[n]; t < cu[n + 1]; ++t) {
            const int64_t row = t * H + h;
            kda_oracle_token(S, dk, dv, q + row * dk, k + row * dk,
                             v + row * dv, g + row * dk, beta[row],
                             out + row * dv, e);
        }
        if (sT) {
            double *dst = sT + (n * H + h) * dk * dv;
            for (int64_t x = 0; x < dk * dv; ++x) dst[x] = S[x];
        }
    }
    free(S);
    return 0;
}

/* Decode: one token per row n, applied in place to the state slot
 * pool[slot(n)][h], slot(n) = idx ? idx[n] : n.  Inputs are [N][H][d] rows. */
int kda_oracle_decode_step(const double *q, const double *k, const double *v,
                           const double *g, const double *beta, double *pool,
                           const int64_t *idx, int64_t N, int64_t H, int64_t dk,
                           int64_t dv, double *out, int64_t unit_begin,
                           int64_t unit_end)
{
    double *e = (double *)malloc((size_t)dv * sizeof(double));
    if (!e) return -1;
    for (int64_t u = unit_begin; u < unit_end && u < N * H; ++u) {
        const int64_t n = u / H, h = u % H;
        const int64_t slot = idx ? idx[n] : n;
        const int64_t row = n * H + h;
        kda_oracle_token(pool + (slot * H + h) * dk * dv, dk, dv,
                         q + row * dk, k + row * dk, v + row * dv,
                         g + row * dk, beta[row], out + row * dv, e);
    }
    free(e);
    return 0;
}
