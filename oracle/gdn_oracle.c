/*
 * Gated DeltaNet recurrence: CPU oracle in fp64.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously correct
 * statement of what the GPU library computes.  Only the test-suite, the
 * smoke check and the CPU-baseline leg of the benchmark load it; the product
 * path never does.  It shares no code, header or constant with the CUDA
 * library.
 *
 * Source of the method: "Optimizing on-device inference for Apple Silicon"
 * (Perplexity blog), section "Qwen creates three workload shapes": each Gated
 * DeltaNet layer squeezes history into a fixed-size recurrent state; a learned
 * gate decides how much of the old state is kept and a delta update writes
 * the current token in, token after token.  The same section says prefill may
 * evaluate this either by scanning tokens or by regrouping the updates into
 * blocks.  Section "Keep recurrent state on chip" fixes the state (and its
 * gate) as fp32 on the device; this oracle carries it in fp64.
 *
 * Per sequence n and value head h, with S (dv x dk) starting at init_state
 * (or zero), for each token t:
 *     alpha_t = exp(log_alpha_t)
 *     S <- alpha_t * S * (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *     o_t  = S q_t                                   (post-update state)
 * and final_state = S after the last token.  The sequential scan below uses
 * the algebraically identical expanded form
 *     S <- alpha_t S + beta_t (v_t - alpha_t S k_t) k_t^T .
 * Value head h reads query/key head h / (hv / hk).
 *
 * Query/key preparation (optional, qk_norm != 0): the pages' decode path fuses
 * "query and key preparation" into its kernels ("Optimizing on-device
 * inference for Apple Silicon", section "Reduce intermediate and state
 * traffic"); the benchmark spec describes q and k as L2-normalised with q
 * scaled by 1/sqrt(dk).  With qk_norm each head vector x of q and k is
 * replaced by x / sqrt(sum_j x_j^2 + 1e-6) before the recurrence; in every
 * case q is then multiplied by q_scale (1 leaves q as given).
 *
 * Gates from raw inputs (optional, gate_scale != NULL): the pages' kernels
 * carry "the state and its gate" in fp32 ("Keep recurrent state on chip") but
 * print no gate formula.  The configured workloads draw the gates as
 *     log_alpha = -c softplus(x + b),   beta = sigmoid(y),
 * with x, y ~ N(0, 1) and (c, b) = (0.5, 2) for the model-shaped layers or
 * (1, 0) for the tiny case.  Our reading of "computing the gates" is that map
 * with one (c_h, b_h) per value head h: the log_alpha and beta arrays then
 * hold the raw per-token projections a and y, gate_scale[h] = c_h >= 0 and
 * gate_bias[h] = b_h, and per token
 *     log_alpha = -c_h log(1 + e^{a + b_h}),   beta = 1 / (1 + e^{-y}),
 * evaluated here in fp64 (softplus(x) as max(x, 0) + log(1 + e^{-|x|}), which
 * neither overflows nor loses the small-x tail).
 *
 * Layouts (row-major): q,k [T, hk, dk]; v [T, hv, dv]; log_alpha, beta
 * [T, hv]; state [n_seqs, hv, dv, dk] (row = value index); out [T, hv, dv];
 * gate_scale, gate_bias [hv].
 * cu_seqlens [n_seqs + 1] holds token offsets of the packed sequences.
 *
 * Return value: 0 on success, a negative number for invalid arguments.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static int check_common(int n_seqs, const int32_t *cu, int hk, int hv, int dk, int dv)
{
    if (n_seqs < 0 || hk <= 0 || hv <= 0 || dk <= 0 || dv <= 0) return -1;
    if (hv % hk != 0) return -2;
    if (n_seqs > 0 && cu == NULL) return -3;
    for (int n = 0; n < n_seqs; ++n)
        if (cu[n + 1] < cu[n]) return -4;
    return 0;
}

/* Query/key preparation of one token (see the header), in fp64. */
static void prep_qk(const float *q, const float *k, int dk, int qk_norm, double q_scale,
                    double *qd, double *kd)
{
    double sq = 0.0, sk = 0.0;
    for (int j = 0; j < dk; ++j) {
        qd[j] = (double)q[j];
        kd[j] = (double)k[j];
        sq += qd[j] * qd[j];
        sk += kd[j] * kd[j];
    }
    const double fq = q_scale * (qk_norm ? 1.0 / sqrt(sq + 1e-6) : 1.0);
    const double fk = qk_norm ? 1.0 / sqrt(sk + 1e-6) : 1.0;
    for (int j = 0; j < dk; ++j) {
        qd[j] *= fq;
        kd[j] *= fk;
    }
}

/* The gates of one token of value head h (see the header): finished gates as given, or computed from the
 * raw inputs when gate_scale is not NULL. */
static void token_gates(const float *la, const float *bt, size_t idx, int h, const float *gate_scale,
                        const float *gate_bias, double *log_alpha, double *beta)
{
    if (!gate_scale) {
        *log_alpha = (double)la[idx];
        *beta = (double)bt[idx];
        return;
    }
    const double x = (double)la[idx] + (double)gate_bias[h];
    const double softplus = (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x)));
    *log_alpha = -(double)gate_scale[h] * softplus;
    *beta = 1.0 / (1.0 + exp(-(double)bt[idx]));
}

/* One token of the recurrence on one (sequence, head) state, fp64. */
static void token_update(double *S, int dk, int dv, const double *q, const double *k,
                         const float *v, double log_alpha, double beta, double *o,
                         double *sk)
{
    const double alpha = exp(log_alpha);   /* log_alpha = -inf gives alpha = 0 */
    for (int i = 0; i < dv; ++i) {
        double acc = 0.0;
        for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * k[j];
        sk[i] = acc;
    }
    for (int i = 0; i < dv; ++i) {
        const double u = beta * ((double)v[i] - alpha * sk[i]);
        for (int j = 0; j < dk; ++j)
            S[(size_t)i * dk + j] = alpha * S[(size_t)i * dk + j] + u * k[j];
    }
    for (int i = 0; i < dv; ++i) {
        double acc = 0.0;
        for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * q[j];
        o[i] = acc;
    }
}

int gdn_oracle_prefill(int n_seqs, const int32_t *cu_seqlens, int hk, int hv, int dk, int dv,
                       const float *q, const float *k, const float *v,
                       const float *log_alpha, const float *beta,
                       const double *init_state, double *out, double *final_state,
                       int qk_norm, double q_scale, const float *gate_scale, const float *gate_bias,
                       int n_threads)
{
    int rc = check_common(n_seqs, cu_seqlens, hk, hv, dk, dv);
    if (rc) return rc;
    if ((gate_scale == NULL) != (gate_bias == NULL)) return -6;
    const int group = hv / hk;
    const long n_units = (long)n_seqs * hv;
    if (n_threads <= 0) n_threads = 1;
    int failed = 0;

#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads)
    for (long unit = 0; unit < n_units; ++unit) {
        const int n = (int)(unit / hv), h = (int)(unit % hv), hq = h / group;
        double *S = (double *)malloc(sizeof(double) * ((size_t)dv * dk + 2 * (size_t)dv + 2 * (size_t)dk));
        if (!S) { failed = 1; continue; }
        double *sk = S + (size_t)dv * dk, *o = sk + dv, *qd = o + dv, *kd = qd + dk;
        const size_t soff = ((size_t)n * hv + h) * dv * dk;
        if (init_state) memcpy(S, init_state + soff, sizeof(double) * dv * dk);
        else memset(S, 0, sizeof(double) * dv * dk);
        for (int t = cu_seqlens[n]; t < cu_seqlens[n + 1]; ++t) {
            prep_qk(q + ((size_t)t * hk + hq) * dk, k + ((size_t)t * hk + hq) * dk, dk, qk_norm, q_scale, qd, kd);
            double la_t, b_t;
            token_gates(log_alpha, beta, (size_t)t * hv + h, h, gate_scale, gate_bias, &la_t, &b_t);
            token_update(S, dk, dv, qd, kd, v + ((size_t)t * hv + h) * dv, la_t, b_t, o, sk);
            if (out) memcpy(out + ((size_t)t * hv + h) * dv, o, sizeof(double) * dv);
        }
        if (final_state) memcpy(final_state + soff, S, sizeof(double) * dv * dk);
        free(S);
    }
    return failed ? -10 : 0;
}

/*
 * One decode step: the same token update applied to n independent states
 * (a batch of one token each), in place.  q,k [n, hk, dk]; v [n, hv, dv];
 * log_alpha, beta [n, hv] (raw a, y with gate_scale / gate_bias [hv], as for
 * the prefill); state [n, hv, dv, dk]; out [n, hv, dv].
 */
int gdn_oracle_decode_step(int n, int hk, int hv, int dk, int dv, double *state,
                           const float *q, const float *k, const float *v,
                           const float *log_alpha, const float *beta, double *out,
                           int qk_norm, double q_scale, const float *gate_scale, const float *gate_bias,
                           int n_threads)
{
    if (n < 0 || hk <= 0 || hv <= 0 || dk <= 0 || dv <= 0 || hv % hk) return -1;
    if ((gate_scale == NULL) != (gate_bias == NULL)) return -6;
    const int group = hv / hk;
    const long n_units = (long)n * hv;
    if (n_threads <= 0) n_threads = 1;
    int failed = 0;
#pragma omp parallel for schedule(static) num_threads(n_threads)
    for (long unit = 0; unit < n_units; ++unit) {
        const int b = (int)(unit / hv), h = (int)(unit % hv), hq = h / group;
        double *tmp = (double *)malloc(sizeof(double) * (2 * (size_t)dv + 2 * (size_t)dk));
        if (!tmp) { failed = 1; continue; }
        double *qd = tmp + 2 * (size_t)dv, *kd = qd + dk;
        double *S = state + ((size_t)b * hv + h) * dv * dk;
        prep_qk(q + ((size_t)b * hk + hq) * dk, k + ((size_t)b * hk + hq) * dk, dk, qk_norm, q_scale, qd, kd);
        double la_t, b_t;
        token_gates(log_alpha, beta, (size_t)b * hv + h, h, gate_scale, gate_bias, &la_t, &b_t);
        token_update(S, dk, dv, qd, kd, v + ((size_t)b * hv + h) * dv, la_t, b_t, tmp + dv, tmp);
        if (out) memcpy(out + ((size_t)b * hv + h) * dv, tmp + dv, sizeof(double) * dv);
        free(tmp);
    }
    return failed ? -10 : 0;
}

/*
 * The blocked ("chunked") evaluation of the same recurrence, in fp64, used
 * only to pin the two readings of the method against each other.
 *
 * The pages say the updates may be regrouped into blocks that expose matrix
 * work ("Qwen creates three workload shapes") but print no algorithm; this is
 * our derivation.  Inside a chunk of L tokens with local index i and the
 * running log-decay g_i = sum_{j<=i} log_alpha_j, unrolling the recurrence
 * gives S_i = e^{g_i} S0 + sum_{j<=i} e^{g_i-g_j} u_j k_j^T, where u_j are the
 * per-token delta vectors.  Substituting into u_i = beta_i (v_i - alpha_i
 * S_{i-1} k_i) yields the unit lower-triangular system
 *     (I + A) U = diag(beta) V - diag(beta e^g) K S0^T,
 *     A_ij = beta_i e^{g_i - g_j} k_i.k_j   (j < i),
 * solved here as U = Ut - W S0^T with T = (I + A)^-1 (forward substitution),
 * W = T diag(beta e^g) K and Ut = T diag(beta) V.  Then
 *     O   = diag(e^g) Q S0^T + (M o Q K^T) U,  M_ij = e^{g_i - g_j} (j <= i)
 *     S_L = e^{g_L} S0 + U^T diag(e^{g_L - g_j}) K .
 * Decay factors are always exponentials of differences g_i - g_j <= 0.
 * The chunk never straddles a sequence boundary; a sequence's last chunk may
 * be shorter than `chunk`.  Gates must be finite here.
 */
int gdn_oracle_prefill_chunked(int n_seqs, const int32_t *cu_seqlens, int hk, int hv, int dk,
                               int dv, const float *q, const float *k, const float *v,
                               const float *log_alpha, const float *beta,
                               const double *init_state, double *out, double *final_state,
                               int chunk, int qk_norm, double q_scale, int n_threads)
{
    int rc = check_common(n_seqs, cu_seqlens, hk, hv, dk, dv);
    if (rc) return rc;
    if (chunk <= 0) return -5;
    const int group = hv / hk;
    const long n_units = (long)n_seqs * hv;
    const int C = chunk;
    if (n_threads <= 0) n_threads = 1;
    int failed = 0;

#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads)
    for (long unit = 0; unit < n_units; ++unit) {
        const int n = (int)(unit / hv), h = (int)(unit % hv), hq = h / group;
        const size_t nS = (size_t)dv * dk;
        /* S, Snew, g, A, T, W, Ut, U, Kc, Qc, Vc, tmp */
        size_t need = 2 * nS + C + 2 * (size_t)C * C + (size_t)C * dk * 3 + (size_t)C * dv * 3;
        double *mem = (double *)malloc(sizeof(double) * need);
        if (!mem) { failed = 1; continue; }
        double *S = mem, *Sn = S + nS, *g = Sn + nS, *A = g + C, *Tm = A + (size_t)C * C;
        double *W = Tm + (size_t)C * C, *Kc = W + (size_t)C * dk, *Qc = Kc + (size_t)C * dk;
        double *Ut = Qc + (size_t)C * dk, *U = Ut + (size_t)C * dv, *Vc = U + (size_t)C * dv;
        const size_t soff = ((size_t)n * hv + h) * nS;
        if (init_state) memcpy(S, init_state + soff, sizeof(double) * nS);
        else memset(S, 0, sizeof(double) * nS);

        for (int t0 = cu_seqlens[n]; t0 < cu_seqlens[n + 1]; t0 += C) {
            const int L = (cu_seqlens[n + 1] - t0 < C) ? cu_seqlens[n + 1] - t0 : C;
            double bet[L > 0 ? L : 1];
            for (int i = 0; i < L; ++i) {
                const size_t t = (size_t)t0 + i;
                prep_qk(q + (t * hk + hq) * dk, k + (t * hk + hq) * dk, dk, qk_norm, q_scale,
                        Qc + (size_t)i * dk, Kc + (size_t)i * dk);
                for (int j = 0; j < dv; ++j) Vc[(size_t)i * dv + j] = v[(t * hv + h) * dv + j];
                g[i] = (i ? g[i - 1] : 0.0) + (double)log_alpha[t * hv + h];
                bet[i] = beta[t * hv + h];
            }
            /* A (strictly lower) */
            for (int i = 0; i < L; ++i)
                for (int j = 0; j < L; ++j) {
                    double a = 0.0;
                    if (j < i) {
                        double kk = 0.0;
                        for (int d = 0; d < dk; ++d) kk += Kc[(size_t)i * dk + d] * Kc[(size_t)j * dk + d];
                        a = bet[i] * exp(g[i] - g[j]) * kk;
                    }
                    A[(size_t)i * L + j] = a;
                }
            /* T = (I + A)^-1 by forward substitution, one column at a time */
            for (int c = 0; c < L; ++c)
                for (int i = 0; i < L; ++i) {
                    double x = (i == c) ? 1.0 : 0.0;
                    for (int j = 0; j < i; ++j) x -= A[(size_t)i * L + j] * Tm[(size_t)j * L + c];
                    Tm[(size_t)i * L + c] = x;
                }
            /* W = T diag(beta e^g) K ; Ut = T diag(beta) V */
            for (int i = 0; i < L; ++i) {
                for (int d = 0; d < dk; ++d) {
                    double acc = 0.0;
                    for (int j = 0; j < L; ++j)
                        acc += Tm[(size_t)i * L + j] * bet[j] * exp(g[j]) * Kc[(size_t)j * dk + d];
                    W[(size_t)i * dk + d] = acc;
                }
                for (int d = 0; d < dv; ++d) {
                    double acc = 0.0;
                    for (int j = 0; j < L; ++j) acc += Tm[(size_t)i * L + j] * bet[j] * Vc[(size_t)j * dv + d];
                    Ut[(size_t)i * dv + d] = acc;
                }
            }
            /* U = Ut - W S0^T */
            for (int i = 0; i < L; ++i)
                for (int e = 0; e < dv; ++e) {
                    double acc = 0.0;
                    for (int d = 0; d < dk; ++d) acc += W[(size_t)i * dk + d] * S[(size_t)e * dk + d];
                    U[(size_t)i * dv + e] = Ut[(size_t)i * dv + e] - acc;
                }
            /* O = diag(e^g) Q S0^T + (M o Q K^T) U */
            if (out)
                for (int i = 0; i < L; ++i)
                    for (int e = 0; e < dv; ++e) {
                        double acc = 0.0;
                        for (int d = 0; d < dk; ++d) acc += Qc[(size_t)i * dk + d] * S[(size_t)e * dk + d];
                        acc *= exp(g[i]);
                        for (int j = 0; j <= i; ++j) {
                            double qk = 0.0;
                            for (int d = 0; d < dk; ++d) qk += Qc[(size_t)i * dk + d] * Kc[(size_t)j * dk + d];
                            acc += exp(g[i] - g[j]) * qk * U[(size_t)j * dv + e];
                        }
                        out[(((size_t)t0 + i) * hv + h) * dv + e] = acc;
                    }
            /* S_L = e^{g_L} S0 + U^T diag(e^{g_L - g}) K */
            const double gl = g[L - 1];
            for (int e = 0; e < dv; ++e)
                for (int d = 0; d < dk; ++d) {
                    double acc = exp(gl) * S[(size_t)e * dk + d];
                    for (int j = 0; j < L; ++j)
                        acc += U[(size_t)j * dv + e] * exp(gl - g[j]) * Kc[(size_t)j * dk + d];
                    Sn[(size_t)e * dk + d] = acc;
                }
            memcpy(S, Sn, sizeof(double) * nS);
        }
        if (final_state) memcpy(final_state + soff, S, sizeof(double) * nS);
        free(mem);
    }
    return failed ? -10 : 0;
}

int gdn_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
