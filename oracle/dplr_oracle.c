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

/*
 * Reverse mode of the same serial recurrence: the gradients of a scalar loss
 *   L = sum_t do_t . o_t + sum(dST * S_T)
 * with respect to every input, given the upstream gradients do [B,H,T,dv] and
 * dST [B,H,dk,dv] (NULL = zero). TEST INFRASTRUCTURE ONLY, like the forward.
 *
 * The forward pass is re-run and every state S_0 .. S_T of a head is kept
 * (T+1 blocks of dk x dv doubles, so this is for small problems only); then the
 * tokens are walked backwards with the adjoint state dS (the gradient of L with
 * respect to S_t):
 *   readout   o_t = S_t^T q_t      dq_t = S_t do_t,  dS += q_t do_t^T
 *   update    S_t = F_t(S_{t-1})   each mode's update differentiated step by
 *             step (the same steps as the forward), dS <- dF_t^T(dS)
 * and dS0 is the final dS. Outputs (same layouts as the inputs, NULL = not
 * wanted): dq, dk, dv, ddecay, dbeta, dA, dBm, dK, dV, dS0.
 */
typedef struct {
    int mode, T, dk, dv, r, p;
    const double *q, *k, *v, *decay, *beta, *A, *Bm, *K, *V, *S0, *dO, *dST;
    double *dq, *dk_, *dv_, *ddecay, *dbeta, *dA, *dB, *dK, *dV, *dS0;
} head_bwd;

/* One token's forward update of the whole state (dk x dv), from Sp into Sn. */
static void step_forward(const head_bwd* a, int t, const double* Sp, double* Sn, double* w)
{
    const int dk = a->dk, dv = a->dv, r = a->r, p = a->p;
    if (a->mode == ORACLE_MODE_GENERIC) {
        const double* At = a->A + (size_t)t * r * dk;
        const double* Bt = a->Bm + (size_t)t * r * dk;
        const double* lt = a->decay + (size_t)t * dk;
        for (int i = 0; i < r; ++i)
            for (int n = 0; n < dv; ++n) {
                double s = 0.0;
                for (int c = 0; c < dk; ++c) s += Bt[(size_t)i * dk + c] * Sp[(size_t)c * dv + n];
                w[(size_t)i * dv + n] = s;
            }
        for (int c = 0; c < dk; ++c)
            for (int n = 0; n < dv; ++n) {
                double s = exp(lt[c]) * Sp[(size_t)c * dv + n];
                for (int i = 0; i < r; ++i) s -= At[(size_t)i * dk + c] * w[(size_t)i * dv + n];
                for (int l = 0; l < p; ++l)
                    s += a->K[((size_t)t * p + l) * dk + c] * a->V[((size_t)t * p + l) * dv + n];
                Sn[(size_t)c * dv + n] = s;
            }
        return;
    }
    const double* kt = a->k + (size_t)t * dk;
    const double* vt = a->v + (size_t)t * dv;
    const double bt = a->beta[t];
    memcpy(Sn, Sp, sizeof(double) * (size_t)dk * dv);
    if (a->mode == ORACLE_MODE_GDN) {
        const double gate = exp(a->decay[t]);
        for (int n = 0; n < dv; ++n) {
            double s = 0.0;
            for (int c = 0; c < dk; ++c) s += kt[c] * Sp[(size_t)c * dv + n];
            w[n] = s;
        }
        for (int c = 0; c < dk; ++c)
            for (int n = 0; n < dv; ++n)
                Sn[(size_t)c * dv + n] = gate * (Sp[(size_t)c * dv + n] - bt * kt[c] * w[n]) + bt * kt[c] * vt[n];
        return;
    }
    const double* lt = a->decay + (size_t)t * dk;   /* HDLA: erase, forget, erase + write */
    for (int n = 0; n < dv; ++n) {
        double s = 0.0;
        for (int c = 0; c < dk; ++c) s += kt[c] * Sn[(size_t)c * dv + n];
        w[n] = s;
    }
    for (int c = 0; c < dk; ++c)
        for (int n = 0; n < dv; ++n) Sn[(size_t)c * dv + n] -= bt * kt[c] * w[n];
    for (int c = 0; c < dk; ++c)
        for (int n = 0; n < dv; ++n) Sn[(size_t)c * dv + n] *= exp(lt[c]);
    for (int n = 0; n < dv; ++n) {
        double s = 0.0;
        for (int c = 0; c < dk; ++c) s += kt[c] * Sn[(size_t)c * dv + n];
        w[n] = s - vt[n];
    }
    for (int c = 0; c < dk; ++c)
        for (int n = 0; n < dv; ++n) Sn[(size_t)c * dv + n] -= bt * kt[c] * w[n];
}

/* Backward of an erase-and-write step  Sout = Sin - beta k (k^T Sin - u)^T  (u = v, or 0 for a pure erase):
 * given dOut, adds to dk, dbeta (and du when wanted) and writes dIn. */
static void erase_write_bwd(int dk, int dv, const double* kt, double bt, const double* Sin, const double* u,
                            const double* dOut, double* dIn, double* dkt, double* dbt, double* dut, double* tmp)
{
    /* z = k^T Sin - u,  g = k^T dOut (both dv) */
    double* z = tmp;
    double* g = tmp + dv;
    for (int n = 0; n < dv; ++n) {
        double s = 0.0, h = 0.0;
        for (int c = 0; c < dk; ++c) {
            s += kt[c] * Sin[(size_t)c * dv + n];
            h += kt[c] * dOut[(size_t)c * dv + n];
        }
        z[n] = s - (u ? u[n] : 0.0);
        g[n] = h;
    }
    /* dbeta -= sum_n g_n z_n;  dk_c -= beta (sum_n dOut[c][n] z_n + sum_n Sin[c][n] g_n);  du += beta g */
    double db = 0.0;
    for (int n = 0; n < dv; ++n) db += g[n] * z[n];
    *dbt -= db;
    for (int c = 0; c < dk; ++c) {
        double s = 0.0;
        for (int n = 0; n < dv; ++n) s += dOut[(size_t)c * dv + n] * z[n] + Sin[(size_t)c * dv + n] * g[n];
        dkt[c] -= bt * s;
    }
    if (dut)
        for (int n = 0; n < dv; ++n) dut[n] += bt * g[n];
    for (int c = 0; c < dk; ++c)
        for (int n = 0; n < dv; ++n) dIn[(size_t)c * dv + n] = dOut[(size_t)c * dv + n] - bt * kt[c] * g[n];
}

static void run_head_bwd(const head_bwd* a, double* states, double* work)
{
    const int T = a->T, dk = a->dk, dv = a->dv, r = a->r, p = a->p;
    const size_t SS = (size_t)dk * dv;
    double* w = work;                         /* max(r,1) x dv */
    double* dS = w + (size_t)(r > 1 ? r : 1) * dv;
    double* dT = dS + SS;                     /* scratch state-sized blocks */
    double* S1 = dT + SS;
    double* S2 = S1 + SS;
    double* tmp = S2 + SS;                    /* 2 dv + r dv */
    for (size_t e = 0; e < SS; ++e) states[e] = a->S0 ? a->S0[e] : 0.0;
    for (int t = 0; t < T; ++t) step_forward(a, t, states + (size_t)t * SS, states + (size_t)(t + 1) * SS, w);
    for (size_t e = 0; e < SS; ++e) dS[e] = a->dST ? a->dST[e] : 0.0;

    for (int t = T - 1; t >= 0; --t) {
        const double* St = states + (size_t)(t + 1) * SS;
        const double* Sp = states + (size_t)t * SS;
        const double* qt = a->q + (size_t)t * dk;
        const double* dot = a->dO + (size_t)t * dv;
        /* readout */
        if (a->dq)
            for (int c = 0; c < dk; ++c) {
                double s = 0.0;
                for (int n = 0; n < dv; ++n) s += St[(size_t)c * dv + n] * dot[n];
                a->dq[(size_t)t * dk + c] = s;
            }
        for (int c = 0; c < dk; ++c)
            for (int n = 0; n < dv; ++n) dS[(size_t)c * dv + n] += qt[c] * dot[n];

        if (a->mode == ORACLE_MODE_GENERIC) {
            const double* At = a->A + (size_t)t * r * dk;
            const double* Bt = a->Bm + (size_t)t * r * dk;
            const double* lt = a->decay + (size_t)t * dk;
            double* dW = tmp;   /* r x dv */
            for (int i = 0; i < r; ++i)
                for (int n = 0; n < dv; ++n) {
                    double s = 0.0, h = 0.0;
                    for (int c = 0; c < dk; ++c) {
                        s += Bt[(size_t)i * dk + c] * Sp[(size_t)c * dv + n];
                        h += At[(size_t)i * dk + c] * dS[(size_t)c * dv + n];
                    }
                    w[(size_t)i * dv + n] = s;      /* W = B^T S_{t-1} */
                    dW[(size_t)i * dv + n] = -h;    /* dW = -A^T dS */
                }
            for (int c = 0; c < dk; ++c) {
                const double lam = exp(lt[c]);
                double dd = 0.0;
                for (int n = 0; n < dv; ++n) dd += dS[(size_t)c * dv + n] * Sp[(size_t)c * dv + n];
                if (a->ddecay) a->ddecay[(size_t)t * dk + c] = lam * dd;
                for (int i = 0; i < r; ++i) {
                    double sa = 0.0, sb = 0.0;
                    for (int n = 0; n < dv; ++n) {
                        sa += dS[(size_t)c * dv + n] * w[(size_t)i * dv + n];
                        sb += Sp[(size_t)c * dv + n] * dW[(size_t)i * dv + n];
                    }
                    if (a->dA) a->dA[((size_t)t * r + i) * dk + c] = -sa;
                    if (a->dB) a->dB[((size_t)t * r + i) * dk + c] = sb;
                }
                for (int l = 0; l < p; ++l) {
                    double s = 0.0;
                    for (int n = 0; n < dv; ++n) s += dS[(size_t)c * dv + n] * a->V[((size_t)t * p + l) * dv + n];
                    if (a->dK) a->dK[((size_t)t * p + l) * dk + c] = s;
                }
            }
            for (int l = 0; l < p; ++l)
                for (int n = 0; n < dv; ++n) {
                    double s = 0.0;
                    for (int c = 0; c < dk; ++c) s += dS[(size_t)c * dv + n] * a->K[((size_t)t * p + l) * dk + c];
                    if (a->dV) a->dV[((size_t)t * p + l) * dv + n] = s;
                }
            /* dS_{t-1} = D dS + B dW */
            for (int c = 0; c < dk; ++c)
                for (int n = 0; n < dv; ++n) {
                    double s = exp(lt[c]) * dS[(size_t)c * dv + n];
                    for (int i = 0; i < r; ++i) s += Bt[(size_t)i * dk + c] * dW[(size_t)i * dv + n];
                    dT[(size_t)c * dv + n] = s;
                }
            memcpy(dS, dT, sizeof(double) * SS);
            continue;
        }
        const double* kt = a->k + (size_t)t * dk;
        const double* vt = a->v + (size_t)t * dv;
        const double bt = a->beta[t];
        double* dkt = tmp + 2 * (size_t)dv;   /* dk */
        double* dvt = dkt + dk;               /* dv */
        double dbt = 0.0;
        for (int c = 0; c < dk; ++c) dkt[c] = 0.0;
        for (int n = 0; n < dv; ++n) dvt[n] = 0.0;
        if (a->mode == ORACLE_MODE_GDN) {
            /* S_t = e^g X + beta k v^T with X = S_{t-1} - beta k (k^T S_{t-1})^T */
            const double gate = exp(a->decay[t]);
            memcpy(S1, Sp, sizeof(double) * SS);
            for (int n = 0; n < dv; ++n) {
                double s = 0.0;
                for (int c = 0; c < dk; ++c) s += kt[c] * Sp[(size_t)c * dv + n];
                w[n] = s;
            }
            for (int c = 0; c < dk; ++c)
                for (int n = 0; n < dv; ++n) S1[(size_t)c * dv + n] -= bt * kt[c] * w[n];   /* X */
            double dg = 0.0;
            for (size_t e = 0; e < SS; ++e) dg += dS[e] * S1[e];
            if (a->ddecay) a->ddecay[t] = gate * dg;
            /* the write beta k v^T */
            for (int n = 0; n < dv; ++n) {
                double s = 0.0;
                for (int c = 0; c < dk; ++c) s += kt[c] * dS[(size_t)c * dv + n];
                dvt[n] += bt * s;
                dbt += s * vt[n];
            }
            for (int c = 0; c < dk; ++c) {
                double s = 0.0;
                for (int n = 0; n < dv; ++n) s += dS[(size_t)c * dv + n] * vt[n];
                dkt[c] += bt * s;
            }
            for (size_t e = 0; e < SS; ++e) dT[e] = gate * dS[e];   /* dX */
            erase_write_bwd(dk, dv, kt, bt, Sp, NULL, dT, dS, dkt, &dbt, NULL, tmp);
        } else {
            /* HDLA: S1 = erase(S_{t-1}), S2 = Diag(lambda) S1, S_t = erase_write(S2, v) */
            const double* lt = a->decay + (size_t)t * dk;
            memcpy(S1, Sp, sizeof(double) * SS);
            for (int n = 0; n < dv; ++n) {
                double s = 0.0;
                for (int c = 0; c < dk; ++c) s += kt[c] * Sp[(size_t)c * dv + n];
                w[n] = s;
            }
            for (int c = 0; c < dk; ++c)
                for (int n = 0; n < dv; ++n) S1[(size_t)c * dv + n] -= bt * kt[c] * w[n];
            for (int c = 0; c < dk; ++c)
                for (int n = 0; n < dv; ++n) S2[(size_t)c * dv + n] = exp(lt[c]) * S1[(size_t)c * dv + n];
            erase_write_bwd(dk, dv, kt, bt, S2, vt, dS, dT, dkt, &dbt, dvt, tmp);   /* dT = dS2 */
            for (int c = 0; c < dk; ++c) {
                const double lam = exp(lt[c]);
                double dd = 0.0;
                for (int n = 0; n < dv; ++n) dd += dT[(size_t)c * dv + n] * S1[(size_t)c * dv + n];
                if (a->ddecay) a->ddecay[(size_t)t * dk + c] = lam * dd;
                for (int n = 0; n < dv; ++n) dT[(size_t)c * dv + n] *= lam;   /* dS1 */
            }
            erase_write_bwd(dk, dv, kt, bt, Sp, NULL, dT, dS, dkt, &dbt, NULL, tmp);
        }
        if (a->dk_) memcpy(a->dk_ + (size_t)t * dk, dkt, sizeof(double) * dk);
        if (a->dv_) memcpy(a->dv_ + (size_t)t * dv, dvt, sizeof(double) * dv);
        if (a->dbeta) a->dbeta[t] = dbt;
    }
    if (a->dS0) memcpy(a->dS0, dS, sizeof(double) * SS);
}

int oracle_backward(int mode, int B, int H, int T, int dk, int dv, int r, int p,
                    const double* q, const double* k, const double* v,
                    const double* decay, const double* beta,
                    const double* A, const double* Bm, const double* K, const double* V,
                    const double* S0, const double* dO, const double* dST,
                    double* dq, double* dk_, double* dv_, double* ddecay, double* dbeta,
                    double* dA, double* dBm, double* dK, double* dV, double* dS0, int nthreads)
{
    if (B < 0 || H < 0 || T < 0 || dk <= 0 || dv <= 0) return -1;
    if (mode != ORACLE_MODE_GDN && mode != ORACLE_MODE_HDLA && mode != ORACLE_MODE_GENERIC) return -2;
    if (mode == ORACLE_MODE_GENERIC) {
        if (r < 0 || p < 0) return -3;
        if (T > 0 && (!decay || !q || (r > 0 && (!A || !Bm)) || (p > 0 && (!K || !V)))) return -4;
    } else {
        r = 1;
        p = 0;
        if (T > 0 && (!q || !k || !v || !decay || !beta)) return -4;
    }
    if (T > 0 && !dO) return -4;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    const size_t SS = (size_t)dk * dv;
    const long nheads = (long)B * H;
    const int rw = r > 1 ? r : 1;
#pragma omp parallel
    {
        double* states = (double*)malloc(sizeof(double) * SS * ((size_t)T + 1));
        double* work = (double*)malloc(sizeof(double) * ((size_t)rw * dv + 4 * SS + 3 * (size_t)dv + (size_t)rw * dv + dk));
#pragma omp for schedule(dynamic, 1)
        for (long bh = 0; bh < nheads; ++bh) {
            const size_t tk = (size_t)bh * T;
            const int gd = mode == ORACLE_MODE_GDN;
            head_bwd a;
            a.mode = mode; a.T = T; a.dk = dk; a.dv = dv; a.r = r; a.p = p;
            a.q = q ? q + tk * dk : NULL;
            a.k = k ? k + tk * dk : NULL;
            a.v = v ? v + tk * dv : NULL;
            a.decay = decay ? decay + tk * (gd ? 1 : dk) : NULL;
            a.beta = beta ? beta + tk : NULL;
            a.A = A ? A + tk * r * dk : NULL;
            a.Bm = Bm ? Bm + tk * r * dk : NULL;
            a.K = K ? K + tk * p * dk : NULL;
            a.V = V ? V + tk * p * dv : NULL;
            a.S0 = S0 ? S0 + (size_t)bh * SS : NULL;
            a.dO = dO ? dO + tk * dv : NULL;
            a.dST = dST ? dST + (size_t)bh * SS : NULL;
            a.dq = dq ? dq + tk * dk : NULL;
            a.dk_ = dk_ ? dk_ + tk * dk : NULL;
            a.dv_ = dv_ ? dv_ + tk * dv : NULL;
            a.ddecay = ddecay ? ddecay + tk * (gd ? 1 : dk) : NULL;
            a.dbeta = dbeta ? dbeta + tk : NULL;
            a.dA = dA ? dA + tk * r * dk : NULL;
            a.dB = dBm ? dBm + tk * r * dk : NULL;
            a.dK = dK ? dK + tk * p * dk : NULL;
            a.dV = dV ? dV + tk * p * dv : NULL;
            a.dS0 = dS0 ? dS0 + (size_t)bh * SS : NULL;
            if (states && work) run_head_bwd(&a, states, work);
        }
        free(states);
        free(work);
    }
    return 0;
}

/*
 * HLA's query-conditioned composition of chunk transitions ("HLA: Expressive Hybrid Linear Attention via
 * Chunk-Wise Dynamic Mixing", Method steps 1, 2, 4 and 5), on the Gated DeltaNet token update above.
 * TEST INFRASTRUCTURE ONLY, like the rest of this file.
 *
 * The sequence is cut into chunks of L tokens (the last may be shorter). Each chunk j has the exact affine
 * summary S -> A_j S + B_j of its token updates (A_j the product of its P_t, B_j its state from zero). For query
 * token i in chunk c, with gates w_ij (j < c; the gates of the current and later chunks are not used), gates
 * below `theta` set to zero:
 *   S_i = 0;  for j = 0 .. c-1:  S_i = ((1 - w_ij) I + w_ij A_j) S_i + w_ij B_j
 *   then the tokens of chunk c up to i, one by one (the causal prefix of the current chunk),
 *   o_i = S_i^T q_i.
 * Layouts: q, k [B,H,T,dk]; v [B,H,T,dv]; g, beta [B,H,T]; W [B,H,T,N] with N = ceil(T / L); o [B,H,T,dv].
 */
static void gdn_token(int dk, int dv, const double* kt, const double* vt, double gt, double bt, double* S, double* w)
{
    const double gate = exp(gt);
    for (int n = 0; n < dv; ++n) {
        double s = 0.0;
        for (int c = 0; c < dk; ++c) s += kt[c] * S[(size_t)c * dv + n];
        w[n] = s;
    }
    for (int c = 0; c < dk; ++c)
        for (int n = 0; n < dv; ++n)
            S[(size_t)c * dv + n] = gate * (S[(size_t)c * dv + n] - bt * kt[c] * w[n]) + (vt ? bt * kt[c] * vt[n] : 0.0);
}

int oracle_hla(int B, int H, int T, int dk, int dv, int L, double theta,
               const double* q, const double* k, const double* v, const double* g, const double* beta,
               const double* W, double* o, int nthreads)
{
    if (B < 0 || H < 0 || T < 0 || dk <= 0 || dv <= 0 || L <= 0) return -1;
    if (T > 0 && (!q || !k || !v || !g || !beta || !W || !o)) return -4;
    const int N = (T + L - 1) / L;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    const long nheads = (long)B * H;
    const size_t SS = (size_t)dk * dv, AA = (size_t)dk * dk;
#pragma omp parallel
    {
        double* Am = (double*)malloc(sizeof(double) * AA * (N > 0 ? N : 1));   /* A_j */
        double* Bm = (double*)malloc(sizeof(double) * SS * (N > 0 ? N : 1));   /* B_j */
        double* S = (double*)malloc(sizeof(double) * SS);
        double* X = (double*)malloc(sizeof(double) * (AA > SS ? AA : SS));
        double* w = (double*)malloc(sizeof(double) * (dk > dv ? dk : dv));
#pragma omp for schedule(dynamic, 1)
        for (long bh = 0; bh < nheads; ++bh) {
            const size_t tk = (size_t)bh * T;
            /* chunk summaries: A_j by applying the token updates (no write) to the identity, B_j from zero */
            for (int j = 0; j < N; ++j) {
                double* A = Am + (size_t)j * AA;
                double* Bj = Bm + (size_t)j * SS;
                for (int r = 0; r < dk; ++r)
                    for (int c = 0; c < dk; ++c) A[(size_t)r * dk + c] = r == c ? 1.0 : 0.0;
                memset(Bj, 0, sizeof(double) * SS);
                for (int t = j * L; t < T && t < (j + 1) * L; ++t) {
                    gdn_token(dk, dk, k + (tk + t) * dk, NULL, g[tk + t], beta[tk + t], A, w);
                    gdn_token(dk, dv, k + (tk + t) * dk, v + (tk + t) * dv, g[tk + t], beta[tk + t], Bj, w);
                }
            }
            for (int i = 0; i < T; ++i) {
                const int c = i / L;
                memset(S, 0, sizeof(double) * SS);
                for (int j = 0; j < c; ++j) {
                    double wij = W[(tk + i) * N + j];
                    if (wij < theta) wij = 0.0;
                    if (wij == 0.0) continue;   /* (1 - 0) I: the state passes unchanged */
                    const double* A = Am + (size_t)j * AA;
                    const double* Bj = Bm + (size_t)j * SS;
                    for (int r = 0; r < dk; ++r)
                        for (int n = 0; n < dv; ++n) {
                            double s = 0.0;
                            for (int c2 = 0; c2 < dk; ++c2) s += A[(size_t)r * dk + c2] * S[(size_t)c2 * dv + n];
                            X[(size_t)r * dv + n] = (1.0 - wij) * S[(size_t)r * dv + n] + wij * (s + Bj[(size_t)r * dv + n]);
                        }
                    memcpy(S, X, sizeof(double) * SS);
                }
                for (int t = c * L; t <= i; ++t)
                    gdn_token(dk, dv, k + (tk + t) * dk, v + (tk + t) * dv, g[tk + t], beta[tk + t], S, w);
                for (int n = 0; n < dv; ++n) {
                    double s = 0.0;
                    for (int c2 = 0; c2 < dk; ++c2) s += S[(size_t)c2 * dv + n] * q[(tk + i) * dk + c2];
                    o[(tk + i) * dv + n] = s;
                }
            }
        }
        free(Am); free(Bm); free(S); free(X); free(w);
    }
    return 0;
}

/*
 * Gated DeltaProduct-style stacked Householders ("Householder-Diagonalized Linear Attention", research
 * background and the computation table: GDP with n_h = 2, 3, r_ab = r_kv = n_h): per token the gate once, then
 * n_h delta-rule steps, each an erase and a write with its own key, value and beta:
 *   S <- e^{g_t} S;  for h = 1 .. n_h:  S <- S - beta_{t,h} k_{t,h} (k_{t,h}^T S - v_{t,h}^T)
 * then o_t = S^T q_t. TEST INFRASTRUCTURE ONLY, like the rest of this file.
 * Layouts: q [B,H,T,dk]; k [B,H,T,nh,dk]; v [B,H,T,nh,dv]; g [B,H,T]; beta [B,H,T,nh]; S0, ST [B,H,dk,dv].
 */
int oracle_gdp(int B, int H, int T, int dk, int dv, int nh, const double* q, const double* k, const double* v,
               const double* g, const double* beta, const double* S0, double* o, double* ST, int nthreads)
{
    if (B < 0 || H < 0 || T < 0 || dk <= 0 || dv <= 0 || nh <= 0) return -1;
    if (T > 0 && (!q || !k || !v || !g || !beta || !o)) return -4;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    const long nheads = (long)B * H;
    const size_t SS = (size_t)dk * dv;
#pragma omp parallel
    {
        double* S = (double*)malloc(sizeof(double) * SS);
        double* w = (double*)malloc(sizeof(double) * dv);
#pragma omp for schedule(dynamic, 1)
        for (long bh = 0; bh < nheads; ++bh) {
            const size_t tk = (size_t)bh * T;
            for (size_t e = 0; e < SS; ++e) S[e] = S0 ? S0[(size_t)bh * SS + e] : 0.0;
            for (int t = 0; t < T; ++t) {
                const double gate = exp(g[tk + t]);
                for (size_t e = 0; e < SS; ++e) S[e] *= gate;
                for (int h = 0; h < nh; ++h) {
                    const double* kt = k + ((tk + t) * nh + h) * dk;
                    const double* vt = v + ((tk + t) * nh + h) * dv;
                    const double bt = beta[(tk + t) * nh + h];
                    for (int n = 0; n < dv; ++n) {
                        double s = 0.0;
                        for (int c = 0; c < dk; ++c) s += kt[c] * S[(size_t)c * dv + n];
                        w[n] = s - vt[n];
                    }
                    for (int c = 0; c < dk; ++c)
                        for (int n = 0; n < dv; ++n) S[(size_t)c * dv + n] -= bt * kt[c] * w[n];
                }
                for (int n = 0; n < dv; ++n) {
                    double s = 0.0;
                    for (int c = 0; c < dk; ++c) s += S[(size_t)c * dv + n] * q[(tk + t) * dk + c];
                    o[(tk + t) * dv + n] = s;
                }
            }
            if (ST)
                for (size_t e = 0; e < SS; ++e) ST[(size_t)bh * SS + e] = S[e];
        }
        free(S);
        free(w);
    }
    return 0;
}
