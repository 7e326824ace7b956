/*
 * gdn_oracle.c -- plain fp64 CPU oracle for the Gated DeltaNet layer core.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or helper with the CUDA
 * library.
 *
 * What it computes, and where that is defined:
 *   - The gate from A_log and dt_bias, the beta sigmoid, q/k L2 norm and
 *     grouped value heads are the ingredients the JevAny page lists for the
 *     chunked GDN kernel ("Add opt-in fused Qwen3.5 inference kernels",
 *     section Summary).  The pages print no formula; the exact gate, beta and
 *     recurrence are the plain reading of the gated delta rule:
 *         g_t    = -exp(A_log) * softplus(a_t + dt_bias)
 *         beta_t = sigmoid(b_t)
 *         S_t    = exp(g_t) S_{t-1} + k_t (beta_t (v_t - exp(g_t) S_{t-1}^T k_t))^T
 *         o_t    = S_t^T q_t / sqrt(Dk)
 *     with S held as Dk x Dv ("HKV" state layout, pegainfer page, sections
 *     Summary and Correctness), q/k L2-normalised, and value head h reading
 *     key/query head h / (Hv/Hk).
 *   - Packed variable-length sequences with optional initial states, final
 *     states returned (pegainfer page, Correctness: chunked vs unchunked
 *     prefill, T = 1, 2, 63, 64, 65, 127, 128 boundaries).
 *   - The optional fused gated RMSNorm after the core (JevAny page, Summary):
 *         y = o / sqrt(mean(o^2) + eps) * w * silu(z), per (token, head).
 *
 * Two fp64 forms of the same core are given:
 *   gdn_oracle_core          the definition, token by token;
 *   gdn_oracle_core_chunked  the chunked (WY/UT) algebra, chunk length C,
 *                            written from the token form (delta_i = U_i).
 * The first is the oracle; the second is checked against it, in plain fp64
 * loops, as a second route through the chunked algebra.
 *
 * No fast-math; build with -ffp-contract=off so x86 and Arm agree.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* softplus(x) = log(1 + e^x), written so that e^x never overflows. */
double gdn_oracle_softplus(double x)
{
    if (x > 30.0)
        return x + log1p(exp(-x));
    return log1p(exp(x));
}

double gdn_oracle_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* Per-token prep: gate, beta and L2-normalised q/k.
 *   q, k  [T, hk, dk]      a, b [T, hv]      A_log, dt_bias [hv]
 *   g, beta [T, hv]        qn, kn [T, hk, dk]
 * l2_eps sits inside the square root: x / sqrt(sum x^2 + l2_eps). */
void gdn_oracle_prep(int64_t T, int hk, int hv, int dk,
                     const double *q, const double *k,
                     const double *a, const double *b,
                     const double *A_log, const double *dt_bias, double l2_eps,
                     double *g, double *beta, double *qn, double *kn)
{
    for (int64_t t = 0; t < T; ++t) {
        for (int h = 0; h < hv; ++h) {
            double x = a[t * hv + h] + dt_bias[h];
            g[t * hv + h] = -exp(A_log[h]) * gdn_oracle_softplus(x);
            beta[t * hv + h] = gdn_oracle_sigmoid(b[t * hv + h]);
        }
        for (int h = 0; h < hk; ++h) {
            const double *qs = q + (t * hk + h) * dk;
            const double *ks = k + (t * hk + h) * dk;
            double sq = 0.0, sk = 0.0;
            for (int i = 0; i < dk; ++i) {
                sq += qs[i] * qs[i];
                sk += ks[i] * ks[i];
            }
            double rq = 1.0 / sqrt(sq + l2_eps), rk = 1.0 / sqrt(sk + l2_eps);
            for (int i = 0; i < dk; ++i) {
                qn[(t * hk + h) * dk + i] = qs[i] * rq;
                kn[(t * hk + h) * dk + i] = ks[i] * rk;
            }
        }
    }
}

/* Gated RMSNorm over one row of length dv, in place:
 *   o <- o / sqrt(mean(o^2) + eps) * w * z * sigmoid(z). */
static void gated_rmsnorm_row(int dv, double *o, const double *z, const double *w, double eps)
{
    double ss = 0.0;
    for (int j = 0; j < dv; ++j)
        ss += o[j] * o[j];
    double r = 1.0 / sqrt(ss / dv + eps);
    for (int j = 0; j < dv; ++j)
        o[j] = o[j] * r * w[j] * (z[j] * gdn_oracle_sigmoid(z[j]));
}

void gdn_oracle_gated_rmsnorm(int64_t rows, int dv, double *o, const double *z,
                              const double *w, double eps)
{
    for (int64_t r = 0; r < rows; ++r)
        gated_rmsnorm_row(dv, o + r * dv, z + r * dv, w, eps);
}

static int set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
    return nthreads;
#else
    (void)nthreads;
    return 1;
#endif
}

/* The token-by-token recurrence (the definition).
 *   cu [N+1]; g, beta [T, hv]; qn, kn [T, hk, dk]; v [T, hv, dv]
 *   init_state [N, hv, dk, dv] or NULL (zeros)
 *   out [T, hv, dv] (pre-norm o_t); final_state [N, hv, dk, dv]
 * Returns 0, or -1 on a bad argument or allocation failure. */
int gdn_oracle_core(int num_seqs, const int32_t *cu, int hk, int hv, int dk, int dv,
                    const double *g, const double *beta, const double *qn,
                    const double *kn, const double *v, const double *init_state,
                    double *out, double *final_state, int nthreads)
{
    if (hk <= 0 || hv <= 0 || hv % hk != 0 || dk <= 0 || dv <= 0)
        return -1;
    const int group = hv / hk;
    const double scale = 1.0 / sqrt((double)dk);
    const int64_t units = (int64_t)num_seqs * hv;
    int err = 0;
    nthreads = set_threads(nthreads);
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 1) reduction(| : err)
    for (int64_t u = 0; u < units; ++u) {
        const int n = (int)(u / hv), h = (int)(u % hv), hq = h / group;
        double *S = (double *)malloc(sizeof(double) * (size_t)dk * dv);
        double *kv = (double *)malloc(sizeof(double) * (size_t)dv);
        if (!S || !kv) {
            free(S);
            free(kv);
            err |= 1;
            continue;
        }
        const size_t ssz = (size_t)dk * dv;
        if (init_state)
            memcpy(S, init_state + (size_t)u * ssz, sizeof(double) * ssz);
        else
            memset(S, 0, sizeof(double) * ssz);
        for (int64_t t = cu[n]; t < cu[n + 1]; ++t) {
            const double eg = exp(g[t * hv + h]);
            const double bt = beta[t * hv + h];
            const double *kt = kn + (t * hk + hq) * dk;
            const double *qt = qn + (t * hk + hq) * dk;
            const double *vt = v + (t * hv + h) * dv;
            /* S <- e^g S */
            for (size_t e = 0; e < ssz; ++e)
                S[e] *= eg;
            /* delta = beta (v - S^T k), with S already decayed */
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i)
                    acc += S[(size_t)i * dv + j] * kt[i];
                kv[j] = bt * (vt[j] - acc);
            }
            /* S <- S + k delta^T */
            for (int i = 0; i < dk; ++i)
                for (int j = 0; j < dv; ++j)
                    S[(size_t)i * dv + j] += kt[i] * kv[j];
            /* o = S^T q / sqrt(dk), from the updated state */
            double *ot = out + (t * hv + h) * dv;
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i)
                    acc += S[(size_t)i * dv + j] * qt[i];
                ot[j] = acc * scale;
            }
        }
        memcpy(final_state + (size_t)u * ssz, S, sizeof(double) * ssz);
        free(S);
        free(kv);
    }
    return err ? -1 : 0;
}

/* The chunked (WY/UT) form of the same core, in fp64, chunk length C.
 * Per chunk with start state S0 and in-chunk cumulative gate G_i:
 *   A_ij = beta_i e^{G_i - G_j} (k_i . k_j)        (j < i)
 *   Tm   = (I + A)^{-1}                            (forward substitution)
 *   W    = Tm diag(beta e^G) K,  Ut = Tm diag(beta) V,  U = Ut - W S0
 *   o_i  = scale (e^{G_i} q_i^T S0 + sum_{j<=i} e^{G_i - G_j} (q_i . k_j) U_j)
 *   S    = e^{G_last} S0 + sum_j e^{G_last - G_j} k_j U_j^T
 * Chunks restart at every sequence start; the last chunk may be short. */
int gdn_oracle_core_chunked(int num_seqs, const int32_t *cu, int hk, int hv, int dk, int dv,
                            int C, const double *g, const double *beta, const double *qn,
                            const double *kn, const double *v, const double *init_state,
                            double *out, double *final_state, int nthreads)
{
    if (hk <= 0 || hv <= 0 || hv % hk != 0 || dk <= 0 || dv <= 0 || C <= 0)
        return -1;
    const int group = hv / hk;
    const double scale = 1.0 / sqrt((double)dk);
    const int64_t units = (int64_t)num_seqs * hv;
    int err = 0;
    nthreads = set_threads(nthreads);
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 1) reduction(| : err)
    for (int64_t u = 0; u < units; ++u) {
        const int n = (int)(u / hv), h = (int)(u % hv), hq = h / group;
        const size_t ssz = (size_t)dk * dv;
        double *S = (double *)malloc(sizeof(double) * ssz);
        double *G = (double *)malloc(sizeof(double) * C);
        double *A = (double *)malloc(sizeof(double) * (size_t)C * C);
        double *Tm = (double *)malloc(sizeof(double) * (size_t)C * C);
        double *W = (double *)malloc(sizeof(double) * (size_t)C * dk);
        double *U = (double *)malloc(sizeof(double) * (size_t)C * dv);
        double *Snew = (double *)malloc(sizeof(double) * ssz);
        if (!S || !G || !A || !Tm || !W || !U || !Snew) {
            free(S); free(G); free(A); free(Tm); free(W); free(U); free(Snew);
            err |= 1;
            continue;
        }
        if (init_state)
            memcpy(S, init_state + (size_t)u * ssz, sizeof(double) * ssz);
        else
            memset(S, 0, sizeof(double) * ssz);
        for (int64_t c0 = cu[n]; c0 < cu[n + 1]; c0 += C) {
            const int L = (int)((cu[n + 1] - c0) < C ? (cu[n + 1] - c0) : C);
#define KN(i) (kn + ((c0 + (i)) * hk + hq) * dk)
#define QN(i) (qn + ((c0 + (i)) * hk + hq) * dk)
#define VV(i) (v + ((c0 + (i)) * hv + h) * dv)
#define BT(i) (beta[(c0 + (i)) * hv + h])
            double run = 0.0;
            for (int i = 0; i < L; ++i) {
                run += g[(c0 + i) * hv + h];
                G[i] = run;
            }
            /* A (strictly lower) */
            for (int i = 0; i < L; ++i)
                for (int j = 0; j < L; ++j) {
                    double val = 0.0;
                    if (j < i) {
                        double dot = 0.0;
                        for (int e = 0; e < dk; ++e)
                            dot += KN(i)[e] * KN(j)[e];
                        val = BT(i) * exp(G[i] - G[j]) * dot;
                    }
                    A[i * C + j] = val;
                }
            /* Tm = (I + A)^{-1}: row i of Tm is e_i - sum_{j<i} A_ij Tm_j */
            for (int i = 0; i < L; ++i) {
                for (int l = 0; l < L; ++l)
                    Tm[i * C + l] = (i == l) ? 1.0 : 0.0;
                for (int j = 0; j < i; ++j) {
                    double aij = A[i * C + j];
                    for (int l = 0; l <= j; ++l)
                        Tm[i * C + l] -= aij * Tm[j * C + l];
                }
            }
            /* W = Tm diag(beta e^G) K;  U = Tm diag(beta) V - W S0 */
            for (int i = 0; i < L; ++i) {
                for (int e = 0; e < dk; ++e) {
                    double acc = 0.0;
                    for (int j = 0; j <= i; ++j)
                        acc += Tm[i * C + j] * BT(j) * exp(G[j]) * KN(j)[e];
                    W[(size_t)i * dk + e] = acc;
                }
                for (int c = 0; c < dv; ++c) {
                    double acc = 0.0;
                    for (int j = 0; j <= i; ++j)
                        acc += Tm[i * C + j] * BT(j) * VV(j)[c];
                    double ws = 0.0;
                    for (int e = 0; e < dk; ++e)
                        ws += W[(size_t)i * dk + e] * S[(size_t)e * dv + c];
                    U[(size_t)i * dv + c] = acc - ws;
                }
            }
            /* outputs */
            for (int i = 0; i < L; ++i) {
                double *ot = out + ((c0 + i) * hv + h) * dv;
                for (int c = 0; c < dv; ++c) {
                    double inter = 0.0;
                    for (int e = 0; e < dk; ++e)
                        inter += QN(i)[e] * S[(size_t)e * dv + c];
                    double intra = 0.0;
                    for (int j = 0; j <= i; ++j) {
                        double qk = 0.0;
                        for (int e = 0; e < dk; ++e)
                            qk += QN(i)[e] * KN(j)[e];
                        intra += exp(G[i] - G[j]) * qk * U[(size_t)j * dv + c];
                    }
                    ot[c] = scale * (exp(G[i]) * inter + intra);
                }
            }
            /* state at the end of the chunk */
            const double Gl = G[L - 1];
            for (int e = 0; e < dk; ++e)
                for (int c = 0; c < dv; ++c) {
                    double acc = exp(Gl) * S[(size_t)e * dv + c];
                    for (int j = 0; j < L; ++j)
                        acc += exp(Gl - G[j]) * KN(j)[e] * U[(size_t)j * dv + c];
                    Snew[(size_t)e * dv + c] = acc;
                }
            memcpy(S, Snew, sizeof(double) * ssz);
#undef KN
#undef QN
#undef VV
#undef BT
        }
        memcpy(final_state + (size_t)u * ssz, S, sizeof(double) * ssz);
        free(S); free(G); free(A); free(Tm); free(W); free(U); free(Snew);
    }
    return err ? -1 : 0;
}

/* Full prefill: prep, token-by-token core, optional gated RMSNorm.
 * z == NULL skips the norm.  Returns 0 or -1. */
int gdn_oracle_prefill(int num_seqs, const int32_t *cu, int hk, int hv, int dk, int dv,
                       const double *q, const double *k, const double *v,
                       const double *a, const double *b,
                       const double *A_log, const double *dt_bias, double l2_eps,
                       const double *init_state, const double *z, const double *norm_w,
                       double eps, double *out, double *final_state, int nthreads)
{
    if (num_seqs < 0 || hk <= 0 || hv <= 0 || hv % hk != 0)
        return -1;
    const int64_t T = num_seqs > 0 ? cu[num_seqs] : 0;
    double *g = (double *)malloc(sizeof(double) * (size_t)(T * hv + 1));
    double *be = (double *)malloc(sizeof(double) * (size_t)(T * hv + 1));
    double *qn = (double *)malloc(sizeof(double) * (size_t)(T * hk * dk + 1));
    double *kn = (double *)malloc(sizeof(double) * (size_t)(T * hk * dk + 1));
    int rc = -1;
    if (g && be && qn && kn) {
        gdn_oracle_prep(T, hk, hv, dk, q, k, a, b, A_log, dt_bias, l2_eps, g, be, qn, kn);
        rc = gdn_oracle_core(num_seqs, cu, hk, hv, dk, dv, g, be, qn, kn, v, init_state,
                             out, final_state, nthreads);
        if (rc == 0 && z)
            gdn_oracle_gated_rmsnorm(T * hv, dv, out, z, norm_w, eps);
    }
    free(g); free(be); free(qn); free(kn);
    return rc;
}

/* One decode step: every sequence gets one token; state updated in place.
 *   q, k [B, hk, dk]; v [B, hv, dv]; a, b [B, hv]; state [B, hv, dk, dv]
 *   out [B, hv, dv]; z [B, hv, dv] or NULL. */
int gdn_oracle_decode_step(int batch, int hk, int hv, int dk, int dv,
                           const double *q, const double *k, const double *v,
                           const double *a, const double *b,
                           const double *A_log, const double *dt_bias, double l2_eps,
                           double *state, const double *z, const double *norm_w, double eps,
                           double *out, int nthreads)
{
    if (batch < 0 || hk <= 0 || hv <= 0 || hv % hk != 0)
        return -1;
    int32_t *cu = (int32_t *)malloc(sizeof(int32_t) * (size_t)(batch + 1));
    if (!cu)
        return -1;
    for (int i = 0; i <= batch; ++i)
        cu[i] = i;
    int rc = gdn_oracle_prefill(batch, cu, hk, hv, dk, dv, q, k, v, a, b, A_log, dt_bias,
                                l2_eps, state, z, norm_w, eps, out, state, nthreads);
    free(cu);
    return rc;
}
