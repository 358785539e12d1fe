/*
 * Float64 CPU oracle for linear attention with a diagonal-plus-low-rank decay.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may call this code; it
 * exists so that tests, the smoke check and the benchmark's CPU baseline can
 * compare the CUDA path against a plain, slow, obviously correct definition.
 * It shares no code, header or constant with the CUDA library.
 *
 * What it computes (per batch b, head h), serially token by token, with the
 * state S in R^{dk x dv} (column convention, decay acting from the left):
 *
 *   GENERIC  S_t = (D_t - A_t B_t^T) S_{t-1} + K_t V_t^T,   D_t = Diag(exp(decay_t))
 *            -- the general recurrence of "Householder-Diagonalized Linear
 *               Attention" (HDLA), Key design 3, displayed equation.
 *   GDN      S_t = exp(g_t) (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
 *            -- the Gated DeltaNet token update of "HLA: Expressive Hybrid
 *               Linear Attention via Chunk-Wise Dynamic Mixing", Prerequisites
 *               (Gated DeltaNet) and Method step 1, in the column convention.
 *   HDLA     P_t = (I - beta_t k_t k_t^T) Diag(lambda_t) (I - beta_t k_t k_t^T),
 *            applied literally as the three steps of the test-time-training
 *            reading (erase, diagonal forget, delta-rule write):
 *              S <- S - beta k (k^T S)
 *              S <- Diag(lambda) S
 *              S <- S - beta k (k^T S) + beta k v^T
 *            -- HDLA page, Key design 2 (displayed equation and the TTT
 *               paragraph that follows it).
 *
 * Readout (all modes): o_t = S_t^T q_t with S_t the state AFTER token t's
 * update (the problem statement o_t = S_t^T q_t; no 1/sqrt(dk) factor).
 *
 * Layouts (row-major, float64):
 *   q [B,H,T,dk]; k [B,H,T,dk]; v [B,H,T,dv]
 *   decay: GDN [B,H,T] (log gate g); HDLA/GENERIC [B,H,T,dk] (log lambda)
 *   beta [B,H,T]                      (GDN, HDLA)
 *   A, Bm [B,H,T,r,dk]; K [B,H,T,p,dk]; V [B,H,T,p,dv]   (GENERIC; row i of
 *   the [r,dk] block is column i of A_t)
 *   S0, ST [B,H,dk,dv] (S0 may be NULL = zero; ST may be NULL)
 *   o [B,H,T,dv]
 *
 * Each column of S evolves on its own (the decay acts from the left), so the
 * work is split over (b, h, block of 16 state columns) with OpenMP.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_MODE_GDN 1
#define ORACLE_MODE_HDLA 2
#define ORACLE_MODE_GENERIC 3
#define ORACLE_COLS 16

typedef struct {
    int mode, T, dk, dv, r, p;
    const double *q, *k, *v, *decay, *beta, *A, *Bm, *K, *V, *S0;
    double *o, *ST;
} head_args;

/* Runs one head over state columns [c0, c0+nc). S is dk x nc, w is max(r,1) x nc. */
static void run_columns(const head_args* a, int c0, int nc, double* S, double* w)
{
    const int T = a->T, dk = a->dk, dv = a->dv, r = a->r, p = a->p;
    for (int i = 0; i < dk; ++i)
        for (int n = 0; n < nc; ++n)
            S[i * nc + n] = a->S0 ? a->S0[(size_t)i * dv + c0 + n] : 0.0;

    for (int t = 0; t < T; ++t) {
        const double* qt = a->q + (size_t)t * dk;
        if (a->mode == ORACLE_MODE_GENERIC) {
            const double* At = a->A ? a->A + (size_t)t * r * dk : NULL;
            const double* Bt = a->Bm ? a->Bm + (size_t)t * r * dk : NULL;
            const double* lt = a->decay + (size_t)t * dk;
            /* w = B_t^T S */
            for (int i = 0; i < r; ++i)
                for (int n = 0; n < nc; ++n) {
                    double s = 0.0;
                    for (int c = 0; c < dk; ++c) s += Bt[(size_t)i * dk + c] * S[c * nc + n];
                    w[i * nc + n] = s;
                }
            /* S = D_t S - A_t w + K_t V_t^T */
            for (int c = 0; c < dk; ++c) {
                const double d = exp(lt[c]);
                for (int n = 0; n < nc; ++n) {
                    double s = d * S[c * nc + n];
                    for (int i = 0; i < r; ++i) s -= At[(size_t)i * dk + c] * w[i * nc + n];
                    for (int l = 0; l < p; ++l)
                        s += a->K[((size_t)t * p + l) * dk + c] * a->V[((size_t)t * p + l) * dv + c0 + n];
                    S[c * nc + n] = s;
                }
            }
        } else {
            const double* kt = a->k + (size_t)t * dk;
            const double* vt = a->v + (size_t)t * dv;
            const double bt = a->beta[t];
            if (a->mode == ORACLE_MODE_GDN) {
                const double gate = exp(a->decay[t]);
                for (int n = 0; n < nc; ++n) {
                    double s = 0.0;
                    for (int c = 0; c < dk; ++c) s += kt[c] * S[c * nc + n];
                    w[n] = s;
                }
                for (int c = 0; c < dk; ++c)
                    for (int n = 0; n < nc; ++n)
                        S[c * nc + n] = gate * (S[c * nc + n] - bt * kt[c] * w[n])
                                        + bt * kt[c] * vt[c0 + n];
            } else { /* HDLA, three literal steps */
                const double* lt = a->decay + (size_t)t * dk;
                /* 1: erase  S <- (I - beta k k^T) S */
                for (int n = 0; n < nc; ++n) {
                    double s = 0.0;
                    for (int c = 0; c < dk; ++c) s += kt[c] * S[c * nc + n];
                    w[n] = s;
                }
                for (int c = 0; c < dk; ++c)
                    for (int n = 0; n < nc; ++n) S[c * nc + n] -= bt * kt[c] * w[n];
                /* 2: diagonal forget  S <- Diag(lambda) S */
                for (int c = 0; c < dk; ++c) {
                    const double lam = exp(lt[c]);
                    for (int n = 0; n < nc; ++n) S[c * nc + n] *= lam;
                }
                /* 3: delta-rule write  S <- S - beta k (k^T S - v^T) */
                for (int n = 0; n < nc; ++n) {
                    double s = 0.0;
                    for (int c = 0; c < dk; ++c) s += kt[c] * S[c * nc + n];
                    w[n] = s - vt[c0 + n];
                }
                for (int c = 0; c < dk; ++c)
                    for (int n = 0; n < nc; ++n) S[c * nc + n] -= bt * kt[c] * w[n];
            }
        }
        /* o_t = S_t^T q_t */
        double* ot = a->o + (size_t)t * dv + c0;
        for (int n = 0; n < nc; ++n) {
            double s = 0.0;
            for (int c = 0; c < dk; ++c) s += S[c * nc + n] * qt[c];
            ot[n] = s;
        }
    }
    if (a->ST)
        for (int i = 0; i < dk; ++i)
            for (int n = 0; n < nc; ++n) a->ST[(size_t)i * dv + c0 + n] = S[i * nc + n];
}

/* Returns 0 on success, a negative code on bad arguments. */
int oracle_forward(int mode, int B, int H, int T, int dk, int dv, int r, int p,
                   const double* q, const double* k, const double* v,
                   const double* decay, const double* beta,
                   const double* A, const double* Bm, const double* K, const double* V,
                   const double* S0, double* o, double* ST, int nthreads)
{
    if (B < 0 || H < 0 || T < 0 || dk <= 0 || dv <= 0) return -1;
    if (mode != ORACLE_MODE_GDN && mode != ORACLE_MODE_HDLA && mode != ORACLE_MODE_GENERIC) return -2;
    if (mode == ORACLE_MODE_GENERIC) {
        if (r < 0 || p < 0) return -3;
        if (T > 0 && (!decay || !q || (r > 0 && (!A || !Bm)) || (p > 0 && (!K || !V)))) return -4;
    } else {
        if (T > 0 && (!q || !k || !v || !decay || !beta)) return -4;
    }
    if (T > 0 && !o) return -4;

    const int nblk = (dv + ORACLE_COLS - 1) / ORACLE_COLS;
    const long ntask = (long)B * H * nblk;
    const int rw = r > 1 ? r : 1;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif

#pragma omp parallel
    {
        double* S = (double*)malloc(sizeof(double) * (size_t)dk * ORACLE_COLS);
        double* w = (double*)malloc(sizeof(double) * (size_t)rw * ORACLE_COLS);
#pragma omp for schedule(dynamic, 1)
        for (long task = 0; task < ntask; ++task) {
            const long bh = task / nblk;
            const int blk = (int)(task % nblk);
            const int c0 = blk * ORACLE_COLS;
            const int nc = (dv - c0) < ORACLE_COLS ? (dv - c0) : ORACLE_COLS;
            const size_t tk = (size_t)bh * T;
            head_args a;
            a.mode = mode; a.T = T; a.dk = dk; a.dv = dv; a.r = r; a.p = p;
            a.q = q ? q + tk * dk : NULL;
            a.k = k ? k + tk * dk : NULL;
            a.v = v ? v + tk * dv : NULL;
            a.decay = decay ? decay + tk * (mode == ORACLE_MODE_GDN ? 1 : dk) : NULL;
            a.beta = beta ? beta + tk : NULL;
            a.A = A ? A + tk * r * dk : NULL;
            a.Bm = Bm ? Bm + tk * r * dk : NULL;
            a.K = K ? K + tk * p * dk : NULL;
            a.V = V ? V + tk * p * dv : NULL;
            a.S0 = S0 ? S0 + (size_t)bh * dk * dv : NULL;
            a.o = o ? o + tk * dv : NULL;
            a.ST = ST ? ST + (size_t)bh * dk * dv : NULL;
            run_columns(&a, c0, nc, S, w);
        }
        free(S);
        free(w);
    }
    return 0;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
