// Backward of the chunkwise DPLR forward: the gradients of a scalar loss with respect to every input, given
// the upstream gradients dO of the outputs and dS_T of the final state. The chunk-wise algorithm of
// "Householder-Diagonalized Linear Attention" (Key design 3) exists for chunk-parallel training; its backward
// reuses the same WY factors.
//
// Three passes over blocks of cb tokens (cb = the largest power of two with cb max(r, p) <= 32 in the generic form
// of the mode: 32 for GDN, 16 for HDLA):
//   1. the forward again, with the fp32 chunk-map and scan kernels at WY blocks of cb tokens, keeping the state
//      before every block (the checkpoints S_{j-1});
//   2. the block-boundary state gradients, backwards over the blocks with the transposed maps of pass 1:
//         dS_{j-1} = P_j^T dS_j + Q'_j^T dO_j,    dS_{nb} = dS_T,   dS0 = dS_{-1} ... (the gradient of S0)
//   3. every block in parallel: given S_{j-1}, dS_j and the block's dO, the gradients of its inputs through the
//      block's WY algebra (below), then through the decay scaling and the mode's factor construction.
//
// Pass 3 in the generic form S_t = D_t S_{t-1} - A_t (B_t^T S_{t-1}) + K_t V_t^T, with the block's decay-scaled
// factors (anchor a = G_C / 2, as in the forward) A~, B~, K~, Q~, its Gram blocks L = strict(B~ A~^T),
// G = strict(B~ K~^T), QA = incl(Q~ A~^T), QK = incl(Q~ K~^T), M = (I + L)^{-1}, the scaled state S0 = e^a S_{j-1}
// and the block's forward quantities H = B~ S0 + G V, E = M H:
//   dS^ = e^a dS_j          dE = -A~ dS^ - QA^T dO          dH = M^T dE
//   dA~ = -E dS^T + dQA^T Q~ + dL^T B~        dQA = incl(-dO E^T),   dL = strict(-dH E^T)
//   dB~ = dH S0^T + dG K~ + dL A~             dG  = strict(dH V^T),  dQK = incl(dO V^T)
//   dK~ = V dS^T + dQK^T Q~ + dG^T B~         dV  = K~ dS^ + QK^T dO + G^T dH
//   dQ~ = dO S0^T + dQA A~ + dQK K~
// then dA = e^{a - G_t} dA~ (and likewise for B, K, q), and the cumulative log-decay collects
//   dG_t = -sum A~ dA~ - sum K~ dK~ + Q~ dQ~ + sum B~_{t+1} dB~_{t+1} (+ sum_n S_j dS_j at the block's end),
// the log-decay's gradient being its reverse cumulative sum over the block. The state dimension is walked in
// slices of 16 columns, so the block's matrices stay in shared memory. Pass 3 runs in fp32 on the CUDA cores.
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>

#include "dplr_internal.h"
#include "smem_gemm.cuh"

namespace dplr {
namespace {

using smem::mm;
using smem::mm_ksplit_out;
using smem::KOut;
using smem::KTerm;

constexpr int BT = 256;      // threads of the block-backward kernel
constexpr int BMX = 32;      // rows of A~ (R = cb r), K~ (P = cb p) and Q~ (cb) at most
constexpr int BNS = 16;      // state columns per slice
constexpr int BD = 128;      // dk, dv at most
// Row strides in shared memory, odd so that a warp reading a column (the transposed operand of a product) touches
// 32 different banks.
constexpr int LD = BD + 1;   // [*][dk] rows
constexpr int LM = BMX + 1;  // [*][R] rows
constexpr int LS = BNS + 1;  // [*][slice] rows
static_assert(2 * BD * LS >= BMX * LD, "the decay-gradient table fits the two slice buffers");

template <class T> __device__ __forceinline__ float ldg(const T* p, size_t i);
template <> __device__ __forceinline__ float ldg<float>(const float* p, size_t i) { return p[i]; }
template <> __device__ __forceinline__ float ldg<__nv_bfloat16>(const __nv_bfloat16* p, size_t i) {
    return __bfloat162float(p[i]);
}

struct BwdArgs {
    const void* q; const void* k; const void* v; const float* decay; const float* beta;
    const void* A; const void* Bm; const void* K; const void* V;
    const float* dO; const float* Sb; const float* dSb; const float* ST;
    float* dq; float* dk; float* dv; float* ddecay; float* dbeta; float* dA; float* dBm; float* dK; float* dV;
};

// Keeps C[m][n] where (token of column n) < (token of row m) (strict) or <= (inclusive); zero elsewhere.
__device__ __forceinline__ void mask(float* C, int ldc, int M, int N, int rdiv, int cdiv, bool strict) {
    for (int idx = threadIdx.x; idx < M * N; idx += blockDim.x) {
        const int m = idx / N, n = idx - m * N;
        const int tm = m / rdiv, tn = n / cdiv;
        if (strict ? !(tn < tm) : !(tn <= tm)) C[m * ldc + n] = 0.f;
    }
}

template <int MODE, class IT>
__global__ void __launch_bounds__(BT)
block_bwd_kernel(Plan pl, BwdArgs a) {
    extern __shared__ __align__(16) float sm[];
    float* At = sm;                 // [BMX][LD] scaled factors
    float* Bt = At + BMX * LD;
    float* Kt = Bt + BMX * LD;
    float* Qt = Kt + BMX * LD;
    float* dAt = Qt + BMX * LD;     // their gradients
    float* dBt = dAt + BMX * LD;
    float* dKt = dBt + BMX * LD;
    float* dQt = dKt + BMX * LD;
    float* Mm = dQt + BMX * LD;     // [BMX][LM] L, then M
    float* Gm = Mm + BMX * LM;
    float* QA = Gm + BMX * LM;
    float* QK = QA + BMX * LM;
    float* dL = QK + BMX * LM;
    float* dG = dL + BMX * LM;
    float* dQA = dG + BMX * LM;
    float* dQK = dQA + BMX * LM;
    float* S0s = dQK + BMX * LM;   // [BD][LS] slice of e^a S_{j-1}; with dSs also the dG_t / d decay table later
    float* dSs = S0s + BD * LS;    // [BD][LS] slice of e^a dS_j
    float* dOs = dSs + BD * LS;    // [BMX][LS]
    float* Vs = dOs + BMX * LS;
    float* Hs = Vs + BMX * LS;
    float* Es = Hs + BMX * LS;
    float* dEs = Es + BMX * LS;
    float* dHs = dEs + BMX * LS;
    float* Gc = dHs + BMX * LS;    // [BMX][LD] inclusive cumulative log-decay G_t
    float* va = Gc + BMX * LD;      // [BD] anchor a
    float* sd = va + BD;            // [BD] sum_n S_j dS_j per row
    float* ct = sd + BD;            // [BMX] HDLA: k^T Lambda k per token; GDN: e^{-g_t}
    float* ks = ct + BMX;           // [8][BMX][BNS] partial tiles of the slice's small products (K split 8 ways)
    float* dVt = ks + 8 * BMX * BNS; // [BMX][BNS] the slice of dV

    const int tid = threadIdx.x, nth = blockDim.x, warp = tid >> 5, lane = tid & 31;
    const int dk = pl.dk, dv = pl.dv, T = pl.T, nb = pl.nb, cb = pl.cw;
    const int r = MODE == DPLR_GENERIC ? pl.r : (MODE == DPLR_GDN ? 1 : 2);
    const int p = MODE == DPLR_GENERIC ? pl.p : 1;
    const int R = cb * r, P = cb * p;
    const int j = blockIdx.x % nb;
    const size_t bh = blockIdx.x / nb;
    const size_t tok0 = bh * (size_t)T + (size_t)j * cb;
    const int valid = min(cb, T - j * cb);
    const IT* q = static_cast<const IT*>(a.q);
    const IT* kin = static_cast<const IT*>(a.k);
    const IT* vin = static_cast<const IT*>(a.v);
    const IT* Ain = static_cast<const IT*>(a.A);
    const IT* Bin = static_cast<const IT*>(a.Bm);
    const IT* Kin = static_cast<const IT*>(a.K);
    const IT* Vin = static_cast<const IT*>(a.V);

    // The block's rows of every input, its dO rows and the three states it reads are contiguous: thread 0 asks
    // for them in L2 first, so that the loads below wait on L2 rather than on DRAM.
    const float* S0g = a.Sb + (bh * (size_t)nb + j) * (size_t)dk * dv;
    const float* dSg = a.dSb + (bh * (size_t)nb + j) * (size_t)dk * dv;
    const float* S1g = j + 1 < nb ? a.Sb + (bh * (size_t)nb + j + 1) * (size_t)dk * dv : a.ST + bh * (size_t)dk * dv;
    if (tid == 0) {
        auto pf = [&](const void* p, size_t bytes) {
            if (p != nullptr && bytes > 0 && bytes % 16 == 0)
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                             :: "l"(reinterpret_cast<uint64_t>(p)), "r"((uint32_t)bytes) : "memory");
        };
        const size_t nt = (size_t)valid;
        pf(q == nullptr ? nullptr : q + tok0 * dk, nt * dk * sizeof(IT));
        if (MODE == DPLR_GENERIC) {
            pf(Ain == nullptr ? nullptr : Ain + tok0 * r * dk, nt * r * dk * sizeof(IT));
            pf(Bin == nullptr ? nullptr : Bin + tok0 * r * dk, nt * r * dk * sizeof(IT));
            if (p > 0) {
                pf(Kin == nullptr ? nullptr : Kin + tok0 * p * dk, nt * p * dk * sizeof(IT));
                pf(Vin == nullptr ? nullptr : Vin + tok0 * p * dv, nt * p * dv * sizeof(IT));
            }
        } else {
            pf(kin + tok0 * dk, nt * dk * sizeof(IT));
            pf(vin + tok0 * dv, nt * dv * sizeof(IT));
        }
        if (MODE != DPLR_GDN) pf(a.decay + tok0 * dk, nt * dk * sizeof(float));
        pf(a.dO + tok0 * dv, nt * dv * sizeof(float));
        pf(S0g, (size_t)dk * dv * sizeof(float));
        pf(dSg, (size_t)dk * dv * sizeof(float));
        pf(S1g, (size_t)dk * dv * sizeof(float));
    }

    // ---- the block's log-decay (identity padding past the end), its inclusive prefix per channel, the anchor
    for (int i = tid; i < cb * dk; i += nth) {
        const int t = i / dk, c = i - t * dk;
        float d = 0.f;
        if (t < valid) d = MODE == DPLR_GDN ? a.decay[tok0 + t] : a.decay[(tok0 + t) * dk + c];
        Gc[t * LD + c] = d;
    }
    if (MODE == DPLR_HDLA)
        for (int t = tid; t < cb; t += nth) ct[t] = 0.f;
    __syncthreads();
    for (int c = tid; c < dk; c += nth) {
        float g = 0.f;
        for (int t = 0; t < cb; ++t) {
            g += Gc[t * LD + c];
            Gc[t * LD + c] = g;
        }
        va[c] = 0.5f * g;
    }
    if (MODE == DPLR_HDLA) {   // c_t = k_t^T Lambda_t k_t (warp per token)
        for (int t = warp; t < valid; t += nth / 32) {
            float s = 0.f;
            for (int c = lane; c < dk; c += 32) {
                const float kk = ldg(kin, (tok0 + t) * dk + c);
                s = fmaf(__expf(a.decay[(tok0 + t) * dk + c]) * kk, kk, s);
            }
            for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
            if (lane == 0) ct[t] = s;
        }
    }
    __syncthreads();

    // ---- the decay-scaled generic-form factors of the block's tokens
    for (int i = tid; i < cb * dk; i += nth) {
        const int t = i / dk, c = i - t * dk;
        const float G = Gc[t * LD + c], Gx = t > 0 ? Gc[(t - 1) * LD + c] : 0.f, an = va[c];
        const float er = __expf(an - G), ef = __expf(Gx - an), eq = __expf(G - an);
        const bool ok = t < valid;
        const size_t tg = tok0 + t;
        Qt[t * LD + c] = ok ? eq * ldg(q, tg * dk + c) : 0.f;
        if (MODE == DPLR_GENERIC) {
            for (int e = 0; e < r; ++e) {
                At[(t * r + e) * LD + c] = ok ? er * ldg(Ain, (tg * r + e) * dk + c) : 0.f;
                Bt[(t * r + e) * LD + c] = ok ? ef * ldg(Bin, (tg * r + e) * dk + c) : 0.f;
            }
            for (int e = 0; e < p; ++e) Kt[(t * p + e) * LD + c] = ok ? er * ldg(Kin, (tg * p + e) * dk + c) : 0.f;
        } else {
            const float kk = ok ? ldg(kin, tg * dk + c) : 0.f, b = ok ? a.beta[tg] : 0.f;
            if (MODE == DPLR_GDN) {
                const float eg = ok ? __expf(a.decay[tg]) : 1.f;
                At[t * LD + c] = er * eg * b * kk;
                Bt[t * LD + c] = ef * kk;
                if (c == 0) ct[t] = ok ? __expf(-a.decay[tg]) : 1.f;   // K~_t = e^{-g_t} A~_t
            } else {
                const float lam = ok ? __expf(a.decay[tg * dk + c]) : 1.f;
                At[(2 * t) * LD + c] = er * kk;
                At[(2 * t + 1) * LD + c] = er * lam * kk;
                Bt[(2 * t) * LD + c] = ef * (b * lam * kk - b * b * ct[t] * kk);
                Bt[(2 * t + 1) * LD + c] = ef * b * kk;
            }
            Kt[t * LD + c] = er * b * kk;
        }
    }
    __syncthreads();

    // ---- Gram blocks and the WY inverse M = (I + L)^{-1} (forward substitution, one column per thread)
    // (few tiles each, K = dk: split over every thread)
    {
        const KOut kl = {Mm, LM, R, R, 1.f, false, 1, {{Bt, LD, false, At, LD, true, dk}, {}, {}}};
        const KOut kq = {QA, LM, cb, R, 1.f, false, 1, {{Qt, LD, false, At, LD, true, dk}, {}, {}}};
        if (MODE == DPLR_GDN) {   // K~ = Diag(e^{-g}) A~: G = L Diag(e^{-g}) and QK = QA Diag(e^{-g})
            const KOut g1[2] = {kl, kq};
            mm_ksplit_out(g1, ks);
            __syncthreads();
            for (int i = tid; i < cb * cb; i += nth) {
                const int t = i / cb, s2 = i - t * cb;
                Gm[t * LM + s2] = Mm[t * LM + s2] * ct[s2];
                QK[t * LM + s2] = QA[t * LM + s2] * ct[s2];
            }
            __syncthreads();
        } else if (P > 0) {   // two at a time
            const KOut g1[2] = {kl, {Gm, LM, R, P, 1.f, false, 1, {{Bt, LD, false, Kt, LD, true, dk}, {}, {}}}};
            mm_ksplit_out(g1, ks);
            __syncthreads();
            const KOut g2[2] = {kq, {QK, LM, cb, P, 1.f, false, 1, {{Qt, LD, false, Kt, LD, true, dk}, {}, {}}}};
            mm_ksplit_out(g2, ks);
            __syncthreads();
        } else {
            const KOut g1[2] = {kl, kq};
            mm_ksplit_out(g1, ks);
            __syncthreads();
        }
    }
    mask(Mm, LM, R, R, r, r, true);
    mask(Gm, LM, R, P, r, p, true);
    mask(QA, LM, cb, R, 1, r, false);
    mask(QK, LM, cb, P, 1, p, false);
    __syncthreads();
    if (tid < R) {   // column tid of M into dL (scratch), then back over L
        const int col = tid;
        for (int i = 0; i < R; ++i) {
            float s = i == col ? 1.f : 0.f;
            for (int kx = 0; kx < i; ++kx) s = fmaf(-Mm[i * LM + kx], dL[kx * LM + col], s);
            dL[i * LM + col] = s;
        }
    }
    __syncthreads();
    for (int i = tid; i < R * LM; i += nth) Mm[i] = dL[i];
    for (int i = tid; i < BMX * LD; i += nth) dAt[i] = dBt[i] = dKt[i] = dQt[i] = 0.f;
    for (int i = tid; i < BMX * LM; i += nth) dL[i] = dG[i] = dQA[i] = dQK[i] = 0.f;
    for (int c = tid; c < dk; c += nth) sd[c] = 0.f;
    __syncthreads();
    if (MODE == DPLR_GDN) {   // W = QA M over QA: the slices' dH takes W^T dO for M^T QA^T dO
        mm(ks, LM, QA, LM, false, Mm, LM, false, cb, R, R, 1.f, false);
        __syncthreads();
        for (int i = tid; i < cb * LM; i += nth) QA[i] = ks[i];
        __syncthreads();
    }

    // ---- the state dimension in slices
    for (int n0 = 0; n0 < dv; n0 += BNS) {
        // (BNS = 16 and nth a multiple of 32: the 16 lanes of a half-warp take the 16 columns of one row c, so
        // the row's sum of S_j dS_j over the slice is a half-warp shuffle reduction, added by its first lane)
#pragma unroll 4
        for (int i = tid; i < dk * BNS; i += nth) {
            const int c = i / BNS, n = i - c * BNS;
            const float e = __expf(va[c]);
            S0s[c * LS + n] = e * S0g[(size_t)c * dv + n0 + n];
            const float ds = dSg[(size_t)c * dv + n0 + n];
            dSs[c * LS + n] = e * ds;
            float x = S1g[(size_t)c * dv + n0 + n] * ds;
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
            if (n == 0) sd[c] += x;
        }
#pragma unroll 4
        for (int i = tid; i < cb * BNS; i += nth) {
            const int t = i / BNS, n = i - t * BNS;
            dOs[t * LS + n] = t < valid ? a.dO[(tok0 + t) * dv + n0 + n] : 0.f;
        }
#pragma unroll 4
        for (int i = tid; i < P * BNS; i += nth) {
            const int u = i / BNS, n = i - u * BNS, t = u / p, e = u - t * p;
            float x = 0.f;
            if (t < valid) x = MODE == DPLR_GENERIC ? ldg(Vin, ((tok0 + t) * p + e) * dv + n0 + n) : ldg(vin, (tok0 + t) * dv + n0 + n);
            Vs[u * LS + n] = x;
        }
        __syncthreads();
        // the slice's R x 16 products have few tiles: their K is split over the threads, two outputs at a time
        if (MODE == DPLR_GDN) {
            // H = B~ S0 + G V, and X = A~ dS^ (over dE): dE = -(X + QA^T dO), so dH = M^T dE = -(M^T X + W^T dO), and
            // the dV term K~ dS^ is e^{-g} X (K~ = Diag(e^{-g}) A~)
            {
                const KOut ko[2] = {
                    {Hs, LS, R, BNS, 1.f, false, 2, {{Bt, LD, false, S0s, LS, false, dk}, {Gm, LM, false, Vs, LS, false, P}, {}}},
                    {dEs, LS, R, BNS, 1.f, false, 1, {{At, LD, false, dSs, LS, false, dk}, {}, {}}}};
                mm_ksplit_out(ko, ks);
            }
            __syncthreads();
            {
                const KOut ko[2] = {{Es, LS, R, BNS, 1.f, false, 1, {{Mm, LM, false, Hs, LS, false, R}, {}, {}}},
                                    {dHs, LS, R, BNS, -1.f, false, 2,
                                     {{Mm, LM, true, dEs, LS, false, R}, {QA, LM, true, dOs, LS, false, cb}, {}}}};
                mm_ksplit_out(ko, ks);
            }
            __syncthreads();
        } else {
            {   // H = B~ S0 + G V and dE = -(A~ dS^ + QA^T dO)
                const KOut ko[2] = {
                    {Hs, LS, R, BNS, 1.f, false, 2, {{Bt, LD, false, S0s, LS, false, dk}, {Gm, LM, false, Vs, LS, false, P}, {}}},
                    {dEs, LS, R, BNS, -1.f, false, 2, {{At, LD, false, dSs, LS, false, dk}, {QA, LM, true, dOs, LS, false, cb}, {}}}};
                mm_ksplit_out(ko, ks);
            }
            __syncthreads();
            {   // E = M H and dH = M^T dE
                const KOut ko[2] = {{Es, LS, R, BNS, 1.f, false, 1, {{Mm, LM, false, Hs, LS, false, R}, {}, {}}},
                                    {dHs, LS, R, BNS, 1.f, false, 1, {{Mm, LM, true, dEs, LS, false, R}, {}, {}}}};
                mm_ksplit_out(ko, ks);
            }
            __syncthreads();
        }
        if (R == cb && P == cb) {   // (rank 1) the four in one pass: dS^ and S0 columns loaded once for two each
            const int nt = dk >> 2;
            for (int tile = tid; tile < (cb >> 2) * nt; tile += nth) {
                const int m0 = (tile / nt) << 2, n0 = (tile % nt) << 2;
                float cA[4][4] = {}, cB[4][4] = {}, cK[4][4] = {}, cQ[4][4] = {};
#pragma unroll 4
                for (int kx = 0; kx < BNS; ++kx) {
                    float e[4], h[4], vv[4], oo[4], ds[4], s0[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        e[i] = Es[(m0 + i) * LS + kx];
                        h[i] = dHs[(m0 + i) * LS + kx];
                        vv[i] = Vs[(m0 + i) * LS + kx];
                        oo[i] = dOs[(m0 + i) * LS + kx];
                        ds[i] = dSs[(n0 + i) * LS + kx];
                        s0[i] = S0s[(n0 + i) * LS + kx];
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) {
                            cA[i][jj] = fmaf(e[i], ds[jj], cA[i][jj]);
                            cK[i][jj] = fmaf(vv[i], ds[jj], cK[i][jj]);
                            cB[i][jj] = fmaf(h[i], s0[jj], cB[i][jj]);
                            cQ[i][jj] = fmaf(oo[i], s0[jj], cQ[i][jj]);
                        }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const int ix = (m0 + i) * LD + n0 + jj;
                        dAt[ix] -= cA[i][jj];
                        dBt[ix] += cB[i][jj];
                        dKt[ix] += cK[i][jj];
                        dQt[ix] += cQ[i][jj];
                    }
            }
        } else {
            mm(dAt, LD, Es, LS, false, dSs, LS, true, R, dk, BNS, -1.f, true);
            mm(dBt, LD, dHs, LS, false, S0s, LS, true, R, dk, BNS, 1.f, true);
            mm(dKt, LD, Vs, LS, false, dSs, LS, true, P, dk, BNS, 1.f, true);
            mm(dQt, LD, dOs, LS, false, S0s, LS, true, cb, dk, BNS, 1.f, true);
        }
        // (four small products, at most 64 tiles each: a quarter of the threads each)
        const int q4 = nth / 4;
        mm(dL, LM, dHs, LS, false, Es, LS, true, R, R, BNS, -1.f, true, 0, q4);
        mm(dG, LM, dHs, LS, false, Vs, LS, true, R, P, BNS, 1.f, true, q4, q4);
        mm(dQA, LM, dOs, LS, false, Es, LS, true, cb, R, BNS, -1.f, true, 2 * q4, q4);
        mm(dQK, LM, dOs, LS, false, Vs, LS, true, cb, P, BNS, 1.f, true, 3 * q4, q4);
        __syncthreads();
        // dV = K~ dS^ + QK^T dO + G^T dH for this slice, then to the output (a generic mode may have no K, V)
        if (MODE == DPLR_GDN) {   // K~ dS^ = e^{-g} X, X over dE
            const KOut ko[1] = {{dVt, BNS, P, BNS, 1.f, false, 2,
                                 {{QK, LM, true, dOs, LS, false, cb}, {Gm, LM, true, dHs, LS, false, R}, {}}}};
            mm_ksplit_out(ko, ks);
            __syncthreads();
        } else if (P > 0) {
            const KOut ko[1] = {{dVt, BNS, P, BNS, 1.f, false, 3,
                                 {{Kt, LD, false, dSs, LS, false, dk}, {QK, LM, true, dOs, LS, false, cb},
                                  {Gm, LM, true, dHs, LS, false, R}}}};
            mm_ksplit_out(ko, ks);
            __syncthreads();
        }
        for (int idx = tid; idx < P * BNS; idx += nth) {
            const int u = idx / BNS, n = idx - u * BNS, t = u / p, e = u - t * p;
            if (t < valid) {
                if (MODE == DPLR_GENERIC) a.dV[((tok0 + t) * p + e) * dv + n0 + n] = dVt[idx];
                else if (MODE == DPLR_GDN) a.dv[(tok0 + t) * dv + n0 + n] = dVt[idx] + ct[t] * dEs[t * LS + n];
                else a.dv[(tok0 + t) * dv + n0 + n] = dVt[idx];
            }
        }
        __syncthreads();
    }

    // ---- the remaining terms of the factor gradients
    mask(dL, LM, R, R, r, r, true);
    mask(dG, LM, R, P, r, p, true);
    mask(dQA, LM, cb, R, 1, r, false);
    mask(dQK, LM, cb, P, 1, p, false);
    __syncthreads();
    if (R == cb && P == cb) {   // (rank 1) the eight in one pass over the block's tokens
        const int nt = dk >> 2;
        for (int tile = tid; tile < (cb >> 2) * nt; tile += nth) {
            const int m0 = (tile / nt) << 2, n0 = (tile % nt) << 2;
            float cA[4][4] = {}, cB[4][4] = {}, cK[4][4] = {}, cQ[4][4] = {};
#pragma unroll 2
            for (int kx = 0; kx < cb; ++kx) {
                float qv[4], kv[4], av[4], bv[4];
                float qaT[4], lT[4], qkT[4], gT[4], gR[4], lR[4], qaR[4], qkR[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    qv[i] = Qt[kx * LD + n0 + i];
                    kv[i] = Kt[kx * LD + n0 + i];
                    av[i] = At[kx * LD + n0 + i];
                    bv[i] = Bt[kx * LD + n0 + i];
                    qaT[i] = dQA[kx * LM + m0 + i];
                    lT[i] = dL[kx * LM + m0 + i];
                    qkT[i] = dQK[kx * LM + m0 + i];
                    gT[i] = dG[kx * LM + m0 + i];
                    gR[i] = dG[(m0 + i) * LM + kx];
                    lR[i] = dL[(m0 + i) * LM + kx];
                    qaR[i] = dQA[(m0 + i) * LM + kx];
                    qkR[i] = dQK[(m0 + i) * LM + kx];
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        cA[i][jj] = fmaf(qaT[i], qv[jj], fmaf(lT[i], bv[jj], cA[i][jj]));
                        cB[i][jj] = fmaf(gR[i], kv[jj], fmaf(lR[i], av[jj], cB[i][jj]));
                        cK[i][jj] = fmaf(qkT[i], qv[jj], fmaf(gT[i], bv[jj], cK[i][jj]));
                        cQ[i][jj] = fmaf(qaR[i], av[jj], fmaf(qkR[i], kv[jj], cQ[i][jj]));
                    }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int ix = (m0 + i) * LD + n0 + jj;
                    dAt[ix] += cA[i][jj];
                    dBt[ix] += cB[i][jj];
                    dKt[ix] += cK[i][jj];
                    dQt[ix] += cQ[i][jj];
                }
        }
    } else {
        mm(dAt, LD, dQA, LM, true, Qt, LD, false, R, dk, cb, 1.f, true);
        mm(dBt, LD, dG, LM, false, Kt, LD, false, R, dk, P, 1.f, true);
        mm(dKt, LD, dQK, LM, true, Qt, LD, false, P, dk, cb, 1.f, true);
        mm(dQt, LD, dQA, LM, false, At, LD, false, cb, dk, R, 1.f, true);
        __syncthreads();
        mm(dAt, LD, dL, LM, true, Bt, LD, false, R, dk, R, 1.f, true);
        mm(dBt, LD, dL, LM, false, At, LD, false, R, dk, R, 1.f, true);
        mm(dKt, LD, dG, LM, true, Bt, LD, false, P, dk, R, 1.f, true);
        mm(dQt, LD, dQK, LM, false, Kt, LD, false, cb, dk, P, 1.f, true);
    }
    __syncthreads();

    // ---- the cumulative log-decay's gradient dG_t (over S0s / dSs), then its reverse prefix: d decay
    float* dGt = S0s;   // [BMX][LD] (fits the two slices: 2 BD LS >= BMX LD)
    for (int i = tid; i < cb * dk; i += nth) {
        const int t = i / dk, c = i - t * dk;
        float s = Qt[t * LD + c] * dQt[t * LD + c];
        for (int e = 0; e < r; ++e) s -= At[(t * r + e) * LD + c] * dAt[(t * r + e) * LD + c];
        for (int e = 0; e < p; ++e) s -= Kt[(t * p + e) * LD + c] * dKt[(t * p + e) * LD + c];
        if (t + 1 < cb)
            for (int e = 0; e < r; ++e) s += Bt[((t + 1) * r + e) * LD + c] * dBt[((t + 1) * r + e) * LD + c];
        else
            s += sd[c];
        dGt[t * LD + c] = s;
    }
    __syncthreads();
    for (int c = tid; c < dk; c += nth) {
        float s = 0.f;
        for (int t = cb - 1; t >= 0; --t) {
            s += dGt[t * LD + c];
            dGt[t * LD + c] = s;
        }
    }
    __syncthreads();

    // ---- unscaled gradients and the mode's factor construction: warp per token, lanes over channels
    for (int t = warp; t < valid; t += nth / 32) {
        const size_t tg = tok0 + t;
        float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f;   // per-token sums over channels
        for (int c = lane; c < dk; c += 32) {
            const float G = Gc[t * LD + c], Gx = t > 0 ? Gc[(t - 1) * LD + c] : 0.f, an = va[c];
            const float er = __expf(an - G), ef = __expf(Gx - an), eq = __expf(G - an);
            const float dd = dGt[t * LD + c];
            a.dq[tg * dk + c] = eq * dQt[t * LD + c];
            if (MODE == DPLR_GENERIC) {
                a.ddecay[tg * dk + c] = dd;
                for (int e = 0; e < r; ++e) {
                    a.dA[(tg * r + e) * dk + c] = er * dAt[(t * r + e) * LD + c];
                    a.dBm[(tg * r + e) * dk + c] = ef * dBt[(t * r + e) * LD + c];
                }
                for (int e = 0; e < p; ++e) a.dK[(tg * p + e) * dk + c] = er * dKt[(t * p + e) * LD + c];
            } else if (MODE == DPLR_GDN) {
                const float kk = ldg(kin, tg * dk + c), b = a.beta[tg], eg = __expf(a.decay[tg]);
                const float dA = er * dAt[t * LD + c], dB = ef * dBt[t * LD + c], dK = er * dKt[t * LD + c];
                a.dk[tg * dk + c] = eg * b * dA + dB + b * dK;
                acc0 = fmaf(kk, dA, acc0);   // k . dA
                acc1 = fmaf(kk, dK, acc1);   // k . dK
                acc2 += dd;                  // sum of the channels' decay gradients
            } else {
                const float kk = ldg(kin, tg * dk + c);
                const float dB0 = ef * dBt[(2 * t) * LD + c];
                acc0 = fmaf(kk, dB0, acc0);  // k . dB0 (needed before dk below)
            }
        }
        for (int off = 16; off > 0; off >>= 1) {
            acc0 += __shfl_xor_sync(0xffffffffu, acc0, off);
            acc1 += __shfl_xor_sync(0xffffffffu, acc1, off);
            acc2 += __shfl_xor_sync(0xffffffffu, acc2, off);
        }
        if (MODE == DPLR_GDN) {
            if (lane == 0) {
                const float b = a.beta[tg], eg = __expf(a.decay[tg]);
                a.dbeta[tg] = eg * acc0 + acc1;
                a.ddecay[tg] = eg * b * acc0 + acc2;
            }
        } else if (MODE == DPLR_HDLA) {
            const float b = a.beta[tg], cc = ct[t], kb0 = acc0;
            float db = 0.f;
            for (int c = lane; c < dk; c += 32) {
                const float G = Gc[t * LD + c], Gx = t > 0 ? Gc[(t - 1) * LD + c] : 0.f, an = va[c];
                const float er = __expf(an - G), ef = __expf(Gx - an);
                const float kk = ldg(kin, tg * dk + c), lam = __expf(a.decay[tg * dk + c]);
                const float dA0 = er * dAt[(2 * t) * LD + c], dA1 = er * dAt[(2 * t + 1) * LD + c];
                const float dB0 = ef * dBt[(2 * t) * LD + c], dB1 = ef * dBt[(2 * t + 1) * LD + c];
                const float dK = er * dKt[t * LD + c];
                a.dk[tg * dk + c] = dA0 + lam * dA1 + (b * lam - b * b * cc) * dB0 - 2.f * b * b * lam * kk * kb0 +
                                    b * dB1 + b * dK;
                const float dlam = kk * dA1 + b * kk * dB0 - b * b * kk * kk * kb0;
                a.ddecay[tg * dk + c] = dGt[t * LD + c] + lam * dlam;
                db = fmaf(lam * kk, dB0, db);
                db = fmaf(kk, dB1 + dK, db);
            }
            for (int off = 16; off > 0; off >>= 1) db += __shfl_xor_sync(0xffffffffu, db, off);
            if (lane == 0) a.dbeta[tg] = db - 2.f * b * cc * kb0;
        }
    }
}

size_t bwd_smem_bytes() {
    return sizeof(float) * (size_t)(8 * BMX * LD + 8 * BMX * LM + 2 * BD * LS + 6 * BMX * LS + BMX * LD + 2 * BD + BMX +
                                    9 * BMX * BNS);
}

// ---- pass 2: the block-boundary state gradients, per (head, 16 state columns), blocks in reverse order
constexpr int CBV = 32;

// 256 threads: the 4 x 4 tiles of a 128 x 32 block of dS (fewer rows leave threads idle).
__global__ void __launch_bounds__(256)
chain_bwd_kernel(Plan pl, const float* Pm, const float* Qm, const float* dO, const float* dST, float* dSb,
                 float* dS0) {
    extern __shared__ __align__(16) float sm[];
    const int dk = pl.dk, dv = pl.dv, cw = pl.cw, nb = pl.nb, T = pl.T;
    const int ncb = dv / CBV;
    const size_t bh = blockIdx.x / ncb;
    const int n0 = (blockIdx.x % ncb) * CBV;
    const int tid = threadIdx.x, nth = blockDim.x;
    float* dS = sm;                     // [dk][CBV]
    float* Ps = dS + dk * CBV;          // [dk][dk + 1]
    float* Qs = Ps + dk * (dk + 1);     // [cw][dk]
    float* Os = Qs + cw * dk;           // [cw][CBV]
    for (int i = tid; i < dk * CBV; i += nth) {
        const int c = i / CBV, n = i - c * CBV;
        dS[i] = dST ? dST[(bh * dk + c) * dv + n0 + n] : 0.f;
    }
    auto prefetch = [&](int jj) {   // block jj's maps into L2 (contiguous in the workspace)
        const float* P = Pm + (bh * (size_t)nb + jj) * (size_t)dk * dk;
        const float* Q = Qm + (bh * (size_t)nb + jj) * (size_t)cw * dk;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(reinterpret_cast<uint64_t>(P)), "r"((uint32_t)(dk * dk * 4)) : "memory");
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(reinterpret_cast<uint64_t>(Q)), "r"((uint32_t)(cw * dk * 4)) : "memory");
    };
    if (tid == 0)
        for (int jj = nb - 1; jj >= 0 && jj >= nb - 4; --jj) prefetch(jj);
    for (int j = nb - 1; j >= 0; --j) {
        __syncthreads();   // dS complete
        if (tid == 0 && j - 4 >= 0) prefetch(j - 4);
        float* dst = dSb + (bh * (size_t)nb + j) * (size_t)dk * dv + n0;   // gradient of the state after block j
        for (int i = tid; i < dk * CBV; i += nth) dst[(size_t)(i / CBV) * dv + i % CBV] = dS[i];
        const float4* P4 = reinterpret_cast<const float4*>(Pm + (bh * (size_t)nb + j) * (size_t)dk * dk);
        const float4* Q4 = reinterpret_cast<const float4*>(Qm + (bh * (size_t)nb + j) * (size_t)cw * dk);
        for (int i = tid; i < dk * dk / 4; i += nth) {
            const float4 x = P4[i];
            const int row = (4 * i) / dk, col = (4 * i) % dk;
            float* d = Ps + row * (dk + 1) + col;
            d[0] = x.x; d[1] = x.y; d[2] = x.z; d[3] = x.w;
        }
        for (int i = tid; i < cw * dk / 4; i += nth) reinterpret_cast<float4*>(Qs)[i] = Q4[i];
        for (int i = tid; i < cw * CBV; i += nth) {
            const int t = i / CBV, n = i - t * CBV, tg = j * cw + t;
            Os[i] = tg < T ? dO[(bh * (size_t)T + tg) * dv + n0 + n] : 0.f;
        }
        __syncthreads();
        // dS_{j-1} = P_j^T dS_j + Q'_j^T dO_j: thread tid takes rows 4 (tid / 8) .., columns 4 (tid % 8) .. (4 x 4)
        const int i0 = 4 * (tid >> 3), c0 = 4 * (tid & 7);
        const bool act = i0 < dk;
        float acc[4][4] = {};
        if (act) {
            for (int c = 0; c < dk; ++c) {
                float x[4], y[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    x[e] = Ps[c * (dk + 1) + i0 + e];
                    y[e] = dS[c * CBV + c0 + e];
                }
#pragma unroll
                for (int e = 0; e < 4; ++e)
#pragma unroll
                    for (int f = 0; f < 4; ++f) acc[e][f] = fmaf(x[e], y[f], acc[e][f]);
            }
            for (int t = 0; t < cw; ++t) {
                float x[4], y[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    x[e] = Qs[t * dk + i0 + e];
                    y[e] = Os[t * CBV + c0 + e];
                }
#pragma unroll
                for (int e = 0; e < 4; ++e)
#pragma unroll
                    for (int f = 0; f < 4; ++f) acc[e][f] = fmaf(x[e], y[f], acc[e][f]);
            }
        }
        __syncthreads();
        if (act)
#pragma unroll
            for (int e = 0; e < 4; ++e)
#pragma unroll
                for (int f = 0; f < 4; ++f) dS[(i0 + e) * CBV + c0 + f] = acc[e][f];
    }
    __syncthreads();
    if (dS0)
        for (int i = tid; i < dk * CBV; i += nth) {
            const int c = i / CBV, n = i - c * CBV;
            dS0[(bh * dk + c) * dv + n0 + n] = dS[i];
        }
}

size_t chain_bwd_smem_bytes(const Plan& pl) {
    return sizeof(float) * (size_t)(pl.dk * CBV + pl.dk * (pl.dk + 1) + pl.cw * pl.dk + pl.cw * CBV);
}

constexpr size_t kBwdAlign = 256;
size_t bround(size_t x) { return (x + kBwdAlign - 1) / kBwdAlign * kBwdAlign; }

// The backward's plan: the fp32 two-stage layout at WY blocks of cb tokens, and its workspace after the forward's
// maps: scratch o, S_T, the checkpoints and the boundary gradients.
struct BwdPlan {
    Plan pl;
    size_t off_o, off_ST, off_Sb, off_dSb, total;
};

dplr_status make_bwd_plan(const dplr_desc* d, BwdPlan* bp) {
    Plan p;
    dplr_status st = make_plan(d, &p);
    if (st != DPLR_OK) return st;
    if (p.dk > BD || p.dv > BD || p.dv % CBV != 0) return DPLR_ERR_UNSUPPORTED;
    const int rg = p.mode == DPLR_GENERIC ? p.r : (p.mode == DPLR_GDN ? 1 : 2);
    const int pg = p.mode == DPLR_GENERIC ? p.p : 1;
    const int m = std::max(rg, std::max(pg, 1));
    if (m > BMX) return DPLR_ERR_UNSUPPORTED;
    p.fused = p.tc = p.gtc = 0;
    // a power of two: the fp32 chunk-map kernel reads float4 rows, so its block dimensions (cw, cw r, cw p) must be
    // multiples of 4, as the forward's WY blocks always are
    int cb = BMX;
    while (cb > 4 && cb * m > BMX) cb /= 2;
    if (cb * m > BMX) return DPLR_ERR_UNSUPPORTED;
    p.cw = cb;
    p.nb = (p.T + p.cw - 1) / p.cw;
    const size_t units = (size_t)p.BH * p.nb;
    size_t off = kBwdAlign;   // the first 256 bytes hold the device status word
    p.off_P = off; off = bround(off + units * (size_t)p.dk * p.dk * sizeof(float));
    p.off_c = off; off = bround(off + units * (size_t)p.dk * p.dv * sizeof(float));
    p.off_Q = off; off = bround(off + units * (size_t)p.cw * p.dk * sizeof(float));
    p.ws_stages = off;
    if (prep_smem_bytes(p) > 227 * 1024 || scan_smem_bytes(p) > 227 * 1024) return DPLR_ERR_UNSUPPORTED;
    bp->off_o = off; off = bround(off + (size_t)p.BH * p.T * p.dv * sizeof(float));
    bp->off_ST = off; off = bround(off + (size_t)p.BH * p.dk * p.dv * sizeof(float));
    bp->off_Sb = off; off = bround(off + units * (size_t)p.dk * p.dv * sizeof(float));
    bp->off_dSb = off; off = bround(off + units * (size_t)p.dk * p.dv * sizeof(float));
    bp->total = off;
    p.ws_bytes = off;
    bp->pl = p;
    return DPLR_OK;
}

std::atomic<uint64_t> g_bwd_smem[6] = {{0}, {0}, {0}, {0}, {0}, {0}};
std::atomic<uint64_t> g_chain_bwd_smem{0};

template <int MODE, class IT>
cudaError_t launch_block_bwd(const Plan& pl, const BwdArgs& a, cudaStream_t s, int slot) {
    const size_t smem = bwd_smem_bytes();
    cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(block_bwd_kernel<MODE, IT>), (int)smem, g_bwd_smem[slot]);
    if (e != cudaSuccess) return e;
    block_bwd_kernel<MODE, IT><<<(unsigned)((size_t)pl.BH * pl.nb), BT, smem, s>>>(pl, a);
    return cudaGetLastError();
}

}  // namespace
}  // namespace dplr

using namespace dplr;

extern "C" size_t dplr_la_backward_workspace_size(const dplr_desc* desc) {
    BwdPlan bp;
    if (make_bwd_plan(desc, &bp) != DPLR_OK) return 0;
    return bp.total;
}

extern "C" dplr_status dplr_la_backward(const dplr_desc* desc, const void* q, const void* k, const void* v,
                                        const float* decay, const float* beta, const void* A, const void* Bm,
                                        const void* K, const void* V, const float* S0, const float* dO,
                                        const float* dST, float* dq, float* dk, float* dv, float* ddecay,
                                        float* dbeta, float* dA, float* dBm, float* dK, float* dV, float* dS0,
                                        void* workspace, size_t ws_bytes, void* stream) {
    BwdPlan bp;
    dplr_status st = make_bwd_plan(desc, &bp);
    if (st != DPLR_OK) return st;
    const Plan& pl = bp.pl;
    auto al = [](const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!al(q) || !al(k) || !al(v) || !al(decay) || !al(beta) || !al(A) || !al(Bm) || !al(K) || !al(V) || !al(S0) ||
        !al(dO) || !al(dST) || !al(dq) || !al(dk) || !al(dv) || !al(ddecay) || !al(dbeta) || !al(dA) || !al(dBm) ||
        !al(dK) || !al(dV) || !al(dS0))
        return DPLR_ERR_INVALID_ARG;
    if (pl.T > 0) {
        if (!q || !decay || !dO || !dq || !ddecay) return DPLR_ERR_INVALID_ARG;
        if (pl.mode == DPLR_GENERIC) {
            if (!A || !Bm || !dA || !dBm) return DPLR_ERR_INVALID_ARG;
            if (pl.p > 0 && (!K || !V || !dK || !dV)) return DPLR_ERR_INVALID_ARG;
        } else if (!k || !v || !beta || !dk || !dv || !dbeta) {
            return DPLR_ERR_INVALID_ARG;
        }
    }
    if (!workspace || ws_bytes < bp.total || (reinterpret_cast<uintptr_t>(workspace) % kBwdAlign) != 0)
        return DPLR_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(workspace);
    float* o_scratch = reinterpret_cast<float*>(ws + bp.off_o);
    float* ST = reinterpret_cast<float*>(ws + bp.off_ST);
    float* Sb = reinterpret_cast<float*>(ws + bp.off_Sb);
    float* dSb = reinterpret_cast<float*>(ws + bp.off_dSb);
    if (pl.T == 0) {   // no tokens: the initial state's gradient is dS_T
        if (dS0) {
            const size_t bytes = (size_t)pl.BH * pl.dk * pl.dv * sizeof(float);
            if ((dST ? cudaMemcpyAsync(dS0, dST, bytes, cudaMemcpyDeviceToDevice, s) : cudaMemsetAsync(dS0, 0, bytes, s)) !=
                cudaSuccess)
                return DPLR_ERR_CUDA;
        }
        return DPLR_OK;
    }
    // pass 1: the forward at blocks of cb tokens, with the state before every block
    ChunkMapArgs ma;
    ma.q = q; ma.k = k; ma.v = v; ma.decay = decay; ma.beta = beta;
    ma.A = A; ma.Bm = Bm; ma.K = K; ma.V = V; ma.o = o_scratch;
    ma.Pm = reinterpret_cast<float*>(ws + pl.off_P);
    ma.Cm = reinterpret_cast<float*>(ws + pl.off_c);
    ma.Qm = reinterpret_cast<float*>(ws + pl.off_Q);
    if (launch_chunk_maps(pl, ma, s) != cudaSuccess) return DPLR_ERR_CUDA;
    ScanArgs sa;
    sa.S0 = S0; sa.o = o_scratch; sa.ST = ST;
    sa.Pm = ma.Pm; sa.Cm = ma.Cm; sa.Qm = ma.Qm; sa.Sb = Sb;
    if (launch_state_scan(pl, sa, s) != cudaSuccess) return DPLR_ERR_CUDA;
    // pass 2: the boundary state gradients
    {
        const size_t smem = chain_bwd_smem_bytes(pl);
        if (set_smem_limit_once(reinterpret_cast<const void*>(chain_bwd_kernel), 227 * 1024, g_chain_bwd_smem) != cudaSuccess)
            return DPLR_ERR_CUDA;
        chain_bwd_kernel<<<(unsigned)((size_t)pl.BH * (pl.dv / CBV)), 256, smem, s>>>(pl, ma.Pm, ma.Qm, dO, dST, dSb, dS0);
        if (cudaGetLastError() != cudaSuccess) return DPLR_ERR_CUDA;
    }
    // pass 3: every block's input gradients
    BwdArgs ba;
    ba.q = q; ba.k = k; ba.v = v; ba.decay = decay; ba.beta = beta; ba.A = A; ba.Bm = Bm; ba.K = K; ba.V = V;
    ba.dO = dO; ba.Sb = Sb; ba.dSb = dSb; ba.ST = ST;
    ba.dq = dq; ba.dk = dk; ba.dv = dv; ba.ddecay = ddecay; ba.dbeta = dbeta; ba.dA = dA; ba.dBm = dBm; ba.dK = dK; ba.dV = dV;
    cudaError_t e;
    if (pl.bf16) {
        e = pl.mode == DPLR_GDN    ? launch_block_bwd<DPLR_GDN, __nv_bfloat16>(pl, ba, s, 0)
            : pl.mode == DPLR_HDLA ? launch_block_bwd<DPLR_HDLA, __nv_bfloat16>(pl, ba, s, 1)
                                   : launch_block_bwd<DPLR_GENERIC, __nv_bfloat16>(pl, ba, s, 2);
    } else {
        e = pl.mode == DPLR_GDN    ? launch_block_bwd<DPLR_GDN, float>(pl, ba, s, 3)
            : pl.mode == DPLR_HDLA ? launch_block_bwd<DPLR_HDLA, float>(pl, ba, s, 4)
                                   : launch_block_bwd<DPLR_GENERIC, float>(pl, ba, s, 5);
    }
    return e == cudaSuccess ? DPLR_OK : DPLR_ERR_CUDA;
}
