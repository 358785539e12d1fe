// One recurrent step of the DPLR recurrence for every (batch, head): the decode-time form of the
// linear-attention state update, whose state has constant size (HDLA page, research background;
// HLA page, results: per-token decode cost).
//
//   S <- (D_t - A_t B_t^T) S + K_t V_t^T,     o_t = S^T q_t          (HDLA page, Key design 3)
//
// GDN applies e^{g}(S - b k (k^T S)) + b k v^T (HLA page, prerequisites), HDLA its three factors
// S <- S - b k (k^T S); S <- Diag(lambda) S; S <- S - b k (k^T S) + b k v^T (HDLA page, Key
// design 2), the generic mode the displayed update. Each CTA owns 32 columns of one head's state: the
// columns evolve independently because the decay acts from the left. Thread (warp w, lane l) holds
// rows w, w + 8, ... of column l in registers; the column sums k^T S, B^T S and S^T q reduce over the
// eight warps through shared memory. The step reads and writes the state once (2 dk dv 4 bytes per
// head) and is bound by that traffic.
#include <cuda_bf16.h>

#include "dplr_internal.h"

namespace dplr {
namespace {

constexpr int DNV = 32;          // state columns per CTA
constexpr int DTH = 256;         // threads: 8 warps x 32 columns
constexpr int DMAXR = 16;        // rows per thread at dk = 128
constexpr int DMAXRANK = 8;      // generic ranks

template <class T> __device__ __forceinline__ float ldx(const T* p, size_t i);
template <> __device__ __forceinline__ float ldx<float>(const float* p, size_t i) { return p[i]; }
template <> __device__ __forceinline__ float ldx<__nv_bfloat16>(const __nv_bfloat16* p, size_t i) {
    return __bfloat162float(p[i]);
}

struct DecodeArgs {
    const void* q; const void* k; const void* v;
    const float* decay; const float* beta;
    const void* A; const void* Bm; const void* K; const void* V;
    float* S; float* o;
};

// Sum over the eight warps of one value per (warp, lane); every thread gets its lane's total.
__device__ __forceinline__ float col_sum(float x, float* red, int w, int l) {
    red[w * DNV + l] = x;
    __syncthreads();
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < DTH / DNV; ++i) s += red[i * DNV + l];
    __syncthreads();
    return s;
}

template <int MODE, class IT>
__global__ void __launch_bounds__(DTH)
decode_step_kernel(Plan pl, DecodeArgs a) {
    __shared__ float vq[128], vk[128], vlam[128];
    __shared__ float vA[DMAXRANK][128], vB[DMAXRANK][128], vK[DMAXRANK][128], vV[DMAXRANK][DNV];
    __shared__ float vv[DNV];
    __shared__ float red[DTH];
    __shared__ float scal[2];
    const int dk = pl.dk, dv = pl.dv, R = (MODE == DPLR_GENERIC) ? pl.r : 0, P = (MODE == DPLR_GENERIC) ? pl.p : 0;
    const int nblk = dv / DNV;
    const size_t bh = blockIdx.x / nblk;
    const int n0 = (blockIdx.x % nblk) * DNV;
    const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;
    const int rows = dk / (DTH / DNV);   // rows per thread: 4, 8 or 16
    const IT* q = static_cast<const IT*>(a.q);

    // ---- the step's vectors into shared memory
    for (int i = tid; i < dk; i += DTH) {
        vq[i] = ldx(q, bh * dk + i);
        if (MODE != DPLR_GENERIC) vk[i] = ldx(static_cast<const IT*>(a.k), bh * dk + i);
        if (MODE != DPLR_GDN) vlam[i] = __expf(a.decay[bh * dk + i]);
    }
    if (MODE == DPLR_GENERIC) {
        const IT* A = static_cast<const IT*>(a.A);
        const IT* Bm = static_cast<const IT*>(a.Bm);
        for (int i = tid; i < R * dk; i += DTH) {
            vA[i / dk][i % dk] = ldx(A, bh * R * dk + i);
            vB[i / dk][i % dk] = ldx(Bm, bh * R * dk + i);
        }
        for (int i = tid; i < P * dk; i += DTH) vK[i / dk][i % dk] = ldx(static_cast<const IT*>(a.K), bh * P * dk + i);
        for (int i = tid; i < P * DNV; i += DTH)
            vV[i / DNV][i % DNV] = ldx(static_cast<const IT*>(a.V), (bh * P + i / DNV) * dv + n0 + i % DNV);
    } else {
        if (tid < DNV) vv[tid] = ldx(static_cast<const IT*>(a.v), bh * dv + n0 + tid);
        if (tid == 0) {
            scal[0] = a.beta[bh];
            scal[1] = (MODE == DPLR_GDN) ? __expf(a.decay[bh]) : 0.f;
        }
    }
    // ---- the state: rows w + 8 r of column n0 + l
    float s[DMAXR];
    float* Sp = a.S + bh * (size_t)dk * dv + n0 + l;
#pragma unroll
    for (int r = 0; r < DMAXR; ++r)
        if (r < rows) s[r] = Sp[(size_t)(w + 8 * r) * dv];
    __syncthreads();

    if (MODE == DPLR_GDN || MODE == DPLR_HDLA) {
        const float b = scal[0];
        // erase along k: S <- S - b k (k^T S)   (GDN: then the gate and the write)
        float p = 0.f;
#pragma unroll
        for (int r = 0; r < DMAXR; ++r)
            if (r < rows) p = fmaf(vk[w + 8 * r], s[r], p);
        float kS = col_sum(p, red, w, l);
        if (MODE == DPLR_GDN) {
            const float gate = scal[1], vn = vv[l];
#pragma unroll
            for (int r = 0; r < DMAXR; ++r)
                if (r < rows) {
                    const float ki = vk[w + 8 * r];
                    s[r] = gate * (s[r] - b * ki * kS) + b * ki * vn;
                }
        } else {
#pragma unroll
            for (int r = 0; r < DMAXR; ++r)
                if (r < rows) s[r] = vlam[w + 8 * r] * (s[r] - b * vk[w + 8 * r] * kS);   // erase, then Diag(lambda)
            p = 0.f;
#pragma unroll
            for (int r = 0; r < DMAXR; ++r)
                if (r < rows) p = fmaf(vk[w + 8 * r], s[r], p);
            kS = col_sum(p, red, w, l);
            const float vn = vv[l];
#pragma unroll
            for (int r = 0; r < DMAXR; ++r)
                if (r < rows) {
                    const float ki = vk[w + 8 * r];
                    s[r] = s[r] - b * ki * kS + b * ki * vn;   // erase again, then the write
                }
        }
    } else {
        // S <- D S - A (B^T S) + K V^T
        float wcol[DMAXRANK];
#pragma unroll
        for (int j = 0; j < DMAXRANK; ++j) {
            if (j < R) {
                float p = 0.f;
#pragma unroll
                for (int r = 0; r < DMAXR; ++r)
                    if (r < rows) p = fmaf(vB[j][w + 8 * r], s[r], p);
                wcol[j] = col_sum(p, red, w, l);
            }
        }
#pragma unroll
        for (int r = 0; r < DMAXR; ++r)
            if (r < rows) {
                const int i = w + 8 * r;
                float x = vlam[i] * s[r];
#pragma unroll
                for (int j = 0; j < DMAXRANK; ++j)
                    if (j < R) x = fmaf(-vA[j][i], wcol[j], x);
#pragma unroll
                for (int j = 0; j < DMAXRANK; ++j)
                    if (j < P) x = fmaf(vK[j][i], vV[j][l], x);
                s[r] = x;
            }
    }
    // ---- the readout o = S^T q and the new state
    float p = 0.f;
#pragma unroll
    for (int r = 0; r < DMAXR; ++r)
        if (r < rows) p = fmaf(vq[w + 8 * r], s[r], p);
    const float on = col_sum(p, red, w, l);
    if (w == 0) a.o[bh * dv + n0 + l] = on;
#pragma unroll
    for (int r = 0; r < DMAXR; ++r)
        if (r < rows) Sp[(size_t)(w + 8 * r) * dv] = s[r];
}

template <int MODE, class IT>
cudaError_t launch_decode_mode(const Plan& pl, const DecodeArgs& a, cudaStream_t s) {
    decode_step_kernel<MODE, IT><<<(unsigned)(pl.BH * (pl.dv / DNV)), DTH, 0, s>>>(pl, a);
    return cudaGetLastError();
}

}  // namespace
}  // namespace dplr

using namespace dplr;

extern "C" dplr_status dplr_la_decode_step(const dplr_desc* desc, const void* q, const void* k, const void* v,
                                           const float* decay, const float* beta, const void* A, const void* Bm,
                                           const void* K, const void* V, float* S, float* o, void* stream) {
    if (desc == nullptr) return DPLR_ERR_INVALID_ARG;
    if (desc->T != 1) return DPLR_ERR_INVALID_ARG;
    Plan pl;
    dplr_status st = make_plan(desc, &pl);
    if (st != DPLR_OK) return st;
    auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!q || !decay || !S || !o || !al(q) || !al(decay) || !al(S) || !al(o)) return DPLR_ERR_INVALID_ARG;
    if (pl.mode == DPLR_GENERIC) {
        if (pl.r > DMAXRANK || pl.p > DMAXRANK) return DPLR_ERR_UNSUPPORTED;
        if (!A || !Bm || !al(A) || !al(Bm)) return DPLR_ERR_INVALID_ARG;
        if (pl.p > 0 && (!K || !V || !al(K) || !al(V))) return DPLR_ERR_INVALID_ARG;
    } else if (!k || !v || !beta || !al(k) || !al(v) || !al(beta)) {
        return DPLR_ERR_INVALID_ARG;
    }
    DecodeArgs a{q, k, v, decay, beta, A, Bm, K, V, S, o};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (pl.bf16) {
        e = pl.mode == DPLR_GDN    ? launch_decode_mode<DPLR_GDN, __nv_bfloat16>(pl, a, s)
            : pl.mode == DPLR_HDLA ? launch_decode_mode<DPLR_HDLA, __nv_bfloat16>(pl, a, s)
                                   : launch_decode_mode<DPLR_GENERIC, __nv_bfloat16>(pl, a, s);
    } else {
        e = pl.mode == DPLR_GDN    ? launch_decode_mode<DPLR_GDN, float>(pl, a, s)
            : pl.mode == DPLR_HDLA ? launch_decode_mode<DPLR_HDLA, float>(pl, a, s)
                                   : launch_decode_mode<DPLR_GENERIC, float>(pl, a, s);
    }
    return e == cudaSuccess ? DPLR_OK : DPLR_ERR_CUDA;
}
