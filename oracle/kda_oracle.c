/*
 * KDA oracle in plain C, fp64.  TEST INFRASTRUCTURE ONLY: the CUDA library
 * never links, loads or calls this file; only the tests, the package's smoke
 * check and the benchmark's CPU-baseline leg do.
 *
 * It computes Kimi Delta Attention for one (sequence, head) problem at a
 * time, token by token, exactly as the Kimi K3 technical report states it:
 *
 *   gate   (section 2.1.1, Eq. 5 with the bias of Eq. 2 inside the logit):
 *          g_t = g_min * Sigmoid(exp(A_h) * (z_t + b_h)),  alpha_t = exp(g_t)
 *   update (section 2.1.1, Eq. 1; the decay is applied before the delta rule):
 *          S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *   output (Eq. 1):  o_t = scale * S_t^T q_t   (scale = 1 in the report)
 *
 * The update is evaluated in the expanded form
 *          S' = Diag(alpha_t) S_{t-1};  S_t = S' + beta_t k_t (v_t - S'^T k_t)^T,
 * which equals Eq. 1 term by term.  Inputs are fp32 values (bf16 inputs are
 * passed upcast, which is exact) and are read into fp64.  S is d_k x d_v,
 * row-major (row = key channel, column = value channel).
 *
 * Problems are independent and run in parallel with OpenMP.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int64_t T, dk, dv;
    const float *q, *k, *v, *z; /* token t, channel c at p[t * stride + c] */
    int64_t stride_q, stride_k, stride_v, stride_z;
    const float *beta; /* token t at beta[t * stride_beta] */
    int64_t stride_beta;
    const float *bias; /* [dk] */
    double A_log, g_min, scale;
    const double *S0; /* [dk * dv] or NULL (zero state) */
    double *o;        /* [T * dv] output */
    double *S;        /* [dk * dv] final state (also the running state) */
    const double *g_direct; /* optional [T * dk] log-decay; when set, z/bias/A_log are ignored */
} kda_oracle_problem;

/* Eq. 5: bounded log-decay of one channel. */
double kda_oracle_gate1(double z, double b, double A_log, double g_min) {
    double x = exp(A_log) * (z + b);
    return g_min / (1.0 + exp(-x));
}

static void run_problem(const kda_oracle_problem *P) {
    const int64_t dk = P->dk, dv = P->dv;
    double *S = P->S;
    double *alpha = (double *)malloc(sizeof(double) * (size_t)dk);
    double *kk = (double *)malloc(sizeof(double) * (size_t)dk);
    double *qq = (double *)malloc(sizeof(double) * (size_t)dk);
    double *p = (double *)malloc(sizeof(double) * (size_t)dv);

    if (P->S0) memcpy(S, P->S0, sizeof(double) * (size_t)(dk * dv));
    else memset(S, 0, sizeof(double) * (size_t)(dk * dv));

    for (int64_t t = 0; t < P->T; ++t) {
        const float *qt = P->q + t * P->stride_q;
        const float *kt = P->k + t * P->stride_k;
        const float *vt = P->v + t * P->stride_v;
        const double beta = (double)P->beta[t * P->stride_beta];
        for (int64_t c = 0; c < dk; ++c) {
            double g;
            if (P->g_direct) g = P->g_direct[t * dk + c];
            else g = kda_oracle_gate1((double)P->z[t * P->stride_z + c], (double)P->bias[c],
                                      P->A_log, P->g_min);
            alpha[c] = exp(g);
            kk[c] = (double)kt[c];
            qq[c] = (double)qt[c];
        }
        /* decay: S' = Diag(alpha) S */
        for (int64_t c = 0; c < dk; ++c)
            for (int64_t j = 0; j < dv; ++j) S[c * dv + j] *= alpha[c];
        /* p = S'^T k */
        for (int64_t j = 0; j < dv; ++j) p[j] = 0.0;
        for (int64_t c = 0; c < dk; ++c)
            for (int64_t j = 0; j < dv; ++j) p[j] += S[c * dv + j] * kk[c];
        /* delta update: S = S' + k (beta (v - p))^T */
        for (int64_t j = 0; j < dv; ++j) p[j] = beta * ((double)vt[j] - p[j]);
        for (int64_t c = 0; c < dk; ++c)
            for (int64_t j = 0; j < dv; ++j) S[c * dv + j] += kk[c] * p[j];
        /* output: o_t = scale * S^T q */
        double *ot = P->o + t * dv;
        for (int64_t j = 0; j < dv; ++j) ot[j] = 0.0;
        for (int64_t c = 0; c < dk; ++c)
            for (int64_t j = 0; j < dv; ++j) ot[j] += S[c * dv + j] * qq[c];
        for (int64_t j = 0; j < dv; ++j) ot[j] *= P->scale;
    }
    free(alpha);
    free(kk);
    free(qq);
    free(p);
}

/* Runs n independent problems with up to nthreads OpenMP threads; returns the
 * number of threads used. */
int kda_oracle_run(int64_t n, const kda_oracle_problem *probs, int nthreads) {
    int used = 1;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel num_threads(nthreads)
    {
#pragma omp single
        {
#ifdef _OPENMP
            used = omp_get_num_threads();
#endif
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < n; ++i) run_problem(&probs[i]);
    }
    return used;
}

int kda_oracle_problem_size(void) { return (int)sizeof(kda_oracle_problem); }
