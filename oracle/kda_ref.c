/*
 * kda_ref.c -- fp64 CPU oracle for Kimi Delta Attention (KDA).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes (the definition, token by token, in double precision):
 *
 *   Per head, the state S is a d_k x d_v matrix ("Kimi K3" blog, section
 *   "Kimi Delta Attention": q_t, k_t in R^{d_k}, v_t in R^{d_v},
 *   S_t in R^{d_k x d_v}, read-out o_t = S_t^T q_t).
 *
 *   The recurrence is applied in the two-stage form given on the same page
 *   (sub-sections "Decay Old Memory" and "Apply Delta-Rule Update"):
 *
 *       Sbar  = Diag(alpha_t) S_{t-1}          (row i scaled by alpha_t[i])
 *       v_old = Sbar^T k_t
 *       S_t   = Sbar + beta_t k_t (v_t - v_old)^T
 *       o_t   = S_t^T q_t
 *
 *   which the page states is the product form
 *       S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T.
 *   alpha_t is passed as its natural logarithm (log_alpha), one value per
 *   (token, head, key channel); beta_t is one scalar per (token, head).
 *
 * Packed variable-length batches: sequence n owns tokens
 * [cu_seqlens[n], cu_seqlens[n+1]) of the packed token axis; each sequence
 * starts from its own initial state S0[n] (zeros when S0 is NULL) and ends
 * in S_final[n].
 *
 * Layouts (row-major, contiguous):
 *   q, k        [T_total, H, dk]   float (exactly the stored values, widened)
 *   v           [T_total, H, dv]   float
 *   log_alpha   [T_total, H, dk]   float
 *   beta        [T_total, H]       float
 *   S0          [n_seq, H, dk, dv] double, or NULL
 *   O           [T_total, Hs, dv]  double, or NULL        (Hs = h1 - h0)
 *   S_final     [n_seq, Hs, dk, dv] double, or NULL
 * Only heads h0 <= h < h1 are computed (so a bounded sample of a large
 * workload can be checked head by head).  Work is spread over
 * (sequence, head) pairs with OpenMP when it is available.
 *
 * Optional prologue (kda_ref_prefill_prologue): the parameter-free steps of
 * the Kimi Linear layer in front of the operator ("Kimi K3: the manos, the
 * mythos, the legendos", section "Kimi Linear": q and k are L2-normalised;
 * "LLM architecture at trillion scale", section "The KDA update, in plain
 * words": the log-decay stays inside (-5, 0)).  Per (token, head), in double:
 *     q <- q / sqrt(sum q^2 + 1e-6),   k <- k / sqrt(sum k^2 + 1e-6)
 *     log_alpha = clamp(-softplus(gate), -5, -1e-4),  softplus(a) = log(1 + e^a)
 *     beta = 1 / (1 + e^(-beta_logit))
 * where the inputs log_alpha / beta then hold gate / beta_logit.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int kda_ref_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static double prologue_unit_scale(const float* x, int n) {
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += (double)x[i] * (double)x[i];
    return 1.0 / sqrt(ss + 1e-6);
}
static double prologue_log_alpha(double a) {
    const double lg = -log1p(exp(a));                 /* -softplus(a) */
    return lg < -5.0 ? -5.0 : (lg > -1e-4 ? -1e-4 : lg);
}
static double prologue_beta(double b) { return 1.0 / (1.0 + exp(-b)); }

/* The prologue alone, for its own checks: x [n_rows, d] -> x_hat; gate -> log_alpha;
   beta_logit -> beta (each output array may be NULL). */
void kda_ref_prologue(const float* x, int n_rows, int d, double* x_hat, const float* gate, int n_gate,
                      double* log_alpha, const float* beta_logit, int n_beta, double* beta) {
    if (x && x_hat)
        for (int r = 0; r < n_rows; ++r) {
            const double sc = prologue_unit_scale(x + (size_t)r * d, d);
            for (int i = 0; i < d; ++i) x_hat[(size_t)r * d + i] = sc * (double)x[(size_t)r * d + i];
        }
    if (gate && log_alpha)
        for (int i = 0; i < n_gate; ++i) log_alpha[i] = prologue_log_alpha((double)gate[i]);
    if (beta_logit && beta)
        for (int i = 0; i < n_beta; ++i) beta[i] = prologue_beta((double)beta_logit[i]);
}

/* One (sequence, head) pair: S is dk*dv doubles of scratch owned by the caller,
   tok is 3 dk + dv doubles (the current token's q, k, log-decay and v). */
static void run_one(const float* q, const float* k, const float* v,
                    const float* log_alpha, const float* beta, int prologue,
                    const double* S0_nh, int64_t bos, int64_t eos, int h, int H,
                    int dk, int dv, int hs, int Hs, double* O, double* Sf_nh,
                    double* S, double* x, double* tok) {
    if (S0_nh)
        memcpy(S, S0_nh, sizeof(double) * (size_t)dk * dv);
    else
        memset(S, 0, sizeof(double) * (size_t)dk * dv);

    for (int64_t t = bos; t < eos; ++t) {
        /* This token's inputs, widened to double (after the prologue when asked). */
        const float* q32 = q + ((size_t)t * H + h) * dk;
        const float* k32 = k + ((size_t)t * H + h) * dk;
        const float* g32 = log_alpha + ((size_t)t * H + h) * dk;
        const float* v32 = v + ((size_t)t * H + h) * dv;
        double* qt = tok;
        double* kt = tok + dk;
        double* gt = tok + 2 * dk;
        double* vt = tok + 3 * dk;
        const double qs = prologue ? prologue_unit_scale(q32, dk) : 1.0;
        const double ks = prologue ? prologue_unit_scale(k32, dk) : 1.0;
        for (int i = 0; i < dk; ++i) {
            qt[i] = qs * (double)q32[i];
            kt[i] = ks * (double)k32[i];
            gt[i] = prologue ? prologue_log_alpha((double)g32[i]) : (double)g32[i];
        }
        for (int j = 0; j < dv; ++j) vt[j] = (double)v32[j];
        const double b_in = (double)beta[(size_t)t * H + h];
        const double bt = prologue ? prologue_beta(b_in) : b_in;

        /* Decay old memory: row i of S times alpha_t[i]. */
        for (int i = 0; i < dk; ++i) {
            const double a = exp((double)gt[i]);
            double* Si = S + (size_t)i * dv;
            for (int j = 0; j < dv; ++j) Si[j] *= a;
        }
        /* v_old = Sbar^T k_t. */
        for (int j = 0; j < dv; ++j) x[j] = 0.0;
        for (int i = 0; i < dk; ++i) {
            const double ki = (double)kt[i];
            const double* Si = S + (size_t)i * dv;
            for (int j = 0; j < dv; ++j) x[j] += Si[j] * ki;
        }
        /* Delta-rule write: S += k_t (beta_t (v_t - v_old))^T. */
        for (int j = 0; j < dv; ++j) x[j] = bt * ((double)vt[j] - x[j]);
        for (int i = 0; i < dk; ++i) {
            const double ki = (double)kt[i];
            double* Si = S + (size_t)i * dv;
            for (int j = 0; j < dv; ++j) Si[j] += ki * x[j];
        }
        /* Read-out o_t = S_t^T q_t (after the write). */
        if (O) {
            double* ot = O + ((size_t)t * Hs + hs) * dv;
            for (int j = 0; j < dv; ++j) ot[j] = 0.0;
            for (int i = 0; i < dk; ++i) {
                const double qi = (double)qt[i];
                const double* Si = S + (size_t)i * dv;
                for (int j = 0; j < dv; ++j) ot[j] += Si[j] * qi;
            }
        }
    }
    if (Sf_nh) memcpy(Sf_nh, S, sizeof(double) * (size_t)dk * dv);
}

/* Returns 0 on success, -1 on a bad argument, -2 when out of host memory. */
static int prefill_any(const float* q, const float* k, const float* v,
                       const float* log_alpha, const float* beta, int prologue, const double* S0,
                       const int64_t* cu_seqlens, int n_seq, int H, int dk, int dv,
                       int h0, int h1, double* O, double* S_final, int n_threads) {
    if (!q || !k || !v || !log_alpha || !beta || !cu_seqlens) return -1;
    if (n_seq < 0 || H <= 0 || dk <= 0 || dv <= 0) return -1;
    if (h0 < 0 || h1 > H || h0 >= h1) return -1;
    for (int n = 0; n < n_seq; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
    const int Hs = h1 - h0;
    const int64_t units = (int64_t)n_seq * Hs;
    int fail = 0;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel
#endif
    {
        double* S = (double*)malloc(sizeof(double) * ((size_t)dk * dv + dv + 3 * (size_t)dk + dv));
        if (!S) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            fail = 1;
        }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t u = 0; u < units; ++u) {
            if (!S) continue;
            const int n = (int)(u / Hs);
            const int hs = (int)(u % Hs);
            const int h = h0 + hs;
            const double* S0_nh = S0 ? S0 + ((size_t)n * H + h) * dk * dv : NULL;
            double* Sf_nh = S_final ? S_final + ((size_t)n * Hs + hs) * dk * dv : NULL;
            run_one(q, k, v, log_alpha, beta, prologue, S0_nh, cu_seqlens[n], cu_seqlens[n + 1],
                    h, H, dk, dv, hs, Hs, O, Sf_nh, S, S + (size_t)dk * dv, S + (size_t)dk * dv + dv);
        }
        free(S);
    }
    (void)n_threads;
    return fail ? -2 : 0;
}

int kda_ref_prefill(const float* q, const float* k, const float* v,
                    const float* log_alpha, const float* beta, const double* S0,
                    const int64_t* cu_seqlens, int n_seq, int H, int dk, int dv,
                    int h0, int h1, double* O, double* S_final, int n_threads) {
    return prefill_any(q, k, v, log_alpha, beta, 0, S0, cu_seqlens, n_seq, H, dk, dv, h0, h1, O, S_final,
                       n_threads);
}

/* As kda_ref_prefill, with q, k unnormalised and gate / beta_logit in place of
   log_alpha / beta (the prologue above). */
int kda_ref_prefill_prologue(const float* q, const float* k, const float* v,
                             const float* gate, const float* beta_logit, const double* S0,
                             const int64_t* cu_seqlens, int n_seq, int H, int dk, int dv,
                             int h0, int h1, double* O, double* S_final, int n_threads) {
    return prefill_any(q, k, v, gate, beta_logit, 1, S0, cu_seqlens, n_seq, H, dk, dv, h0, h1, O, S_final,
                       n_threads);
}
