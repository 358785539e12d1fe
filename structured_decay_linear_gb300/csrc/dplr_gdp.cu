// Gated DeltaProduct-style stacked Householders ("Householder-Diagonalized Linear Attention", research background
// and the computation table: GDP with n_h = 2, 3 and r_ab = r_kv = n_h), through the generic mode.
//
// Per token the gate once, then n_h delta-rule steps, each an erase and a write with its own key, value and beta:
//   S <- e^{g_t} S;  for h = 1 .. n_h:  S <- (I - b_h k_h k_h^T) S + b_h k_h v_h^T.
// The token's update is exactly the generic DPLR form S <- D S - A (B^T S) + K V^T with D = e^{g_t} I and rank n_h:
//   A_h = e^{g_t} k_h,   B_1 = b_1 k_1,   B_h = b_h (k_h - sum_{h' < h} (k_h'^T k_h) B_h')
//   (so that the product (I - b_n k_n k_n^T) .. (I - b_1 k_1 k_1^T) = I - sum_h k_h B_h^T),
//   K_h = (I - b_n k_n k_n^T) .. (I - b_{h+1} k_{h+1} k_{h+1}^T) b_h k_h,   V_h = v_h
// (each write passes through the later steps' erases). One kernel builds these factors per token in fp32 (the
// inputs upcast exactly), then the generic-mode forward runs on them: its tensor-core path for dk = dv = 64 with
// n_h <= 2, its fp32 path otherwise.
#include <cuda_bf16.h>

#include "dplr_internal.h"

namespace dplr {
namespace {

constexpr int GMAXH = 8;   // n_h at most (the generic mode's rank limit)

template <class T> __device__ __forceinline__ float ldx(const T* p, size_t i);
template <> __device__ __forceinline__ float ldx<float>(const float* p, size_t i) { return p[i]; }
template <> __device__ __forceinline__ float ldx<__nv_bfloat16>(const __nv_bfloat16* p, size_t i) {
    return __bfloat162float(p[i]);
}

// One warp per token: lanes over the key channels (dk <= 128: four per lane).
template <class IT>
__global__ void __launch_bounds__(256)
gdp_factor_kernel(long long tokens, int dk, int dv, int nh, const IT* q, const IT* k, const IT* v, const float* g,
                  const float* beta, float* q32, float* decay, float* A, float* Bm, float* K, float* V32) {
    const long long tok = (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (tok >= tokens) return;
    const int per = dk / 32;   // channels per lane (1, 2 or 4)
    float kk[GMAXH][4], bb[GMAXH][4], x[4];
    const float gt = g[tok], eg = __expf(gt);
    for (int e = 0; e < per; ++e) {
        const int c = lane + 32 * e;
        q32[tok * dk + c] = ldx(q, (size_t)tok * dk + c);
        decay[tok * dk + c] = gt;
    }
    for (int h = 0; h < nh; ++h)
        for (int e = 0; e < per; ++e) kk[h][e] = ldx(k, ((size_t)tok * nh + h) * dk + lane + 32 * e);
    auto dot = [&](const float (&a)[4], const float (&b)[4]) {
        float s = 0.f;
        for (int e = 0; e < per; ++e) s = fmaf(a[e], b[e], s);
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        return s;
    };
    // B_h = b_h (k_h - sum_{h' < h} (k_h'^T k_h) B_h')
    for (int h = 0; h < nh; ++h) {
        const float bh = beta[tok * nh + h];
        for (int e = 0; e < per; ++e) x[e] = kk[h][e];
        for (int h2 = 0; h2 < h; ++h2) {
            const float s = dot(kk[h2], kk[h]);
            for (int e = 0; e < per; ++e) x[e] = fmaf(-s, bb[h2][e], x[e]);
        }
        for (int e = 0; e < per; ++e) {
            bb[h][e] = bh * x[e];
            const int c = lane + 32 * e;
            A[(tok * nh + h) * dk + c] = eg * kk[h][e];
            Bm[(tok * nh + h) * dk + c] = bb[h][e];
        }
    }
    // K_h = (I - b_n k_n k_n^T) .. (I - b_{h+1} k_{h+1} k_{h+1}^T) b_h k_h
    for (int h = 0; h < nh; ++h) {
        for (int e = 0; e < per; ++e) x[e] = beta[tok * nh + h] * kk[h][e];
        for (int h2 = h + 1; h2 < nh; ++h2) {
            const float s = beta[tok * nh + h2] * dot(kk[h2], x);
            for (int e = 0; e < per; ++e) x[e] = fmaf(-s, kk[h2][e], x[e]);
        }
        for (int e = 0; e < per; ++e) K[(tok * nh + h) * dk + lane + 32 * e] = x[e];
    }
    for (int h = 0; h < nh; ++h)
        for (int n = lane; n < dv; n += 32) V32[(tok * nh + h) * dv + n] = ldx(v, ((size_t)tok * nh + h) * dv + n);
}

constexpr size_t kGAlign = 256;
size_t ground(size_t x) { return (x + kGAlign - 1) / kGAlign * kGAlign; }

// The generic descriptor the factors run through (fp32 inputs), and the workspace: the factors, then the generic
// forward's workspace.
struct GdpPlan {
    dplr_desc gd;
    size_t off_q, off_d, off_A, off_B, off_K, off_V, off_fwd, fwd_bytes, total;
};

dplr_status make_gdp_plan(const dplr_desc* d, GdpPlan* gp) {
    if (!d || d->mode != DPLR_GENERIC || d->r_ab != d->r_kv || d->r_ab < 1 || d->r_ab > GMAXH) return DPLR_ERR_INVALID_ARG;
    if (d->dk % 32 != 0 || d->dk > 128) return DPLR_ERR_UNSUPPORTED;
    dplr_desc gd = *d;
    gd.in_dtype = DPLR_F32;
    const size_t fwd = dplr_la_workspace_size(&gd);
    if (fwd == 0) return DPLR_ERR_UNSUPPORTED;
    const size_t tokens = (size_t)d->B * d->H * d->T, nh = (size_t)d->r_ab;
    size_t off = 0;
    gp->off_q = off; off = ground(off + tokens * d->dk * 4);
    gp->off_d = off; off = ground(off + tokens * d->dk * 4);
    gp->off_A = off; off = ground(off + tokens * nh * d->dk * 4);
    gp->off_B = off; off = ground(off + tokens * nh * d->dk * 4);
    gp->off_K = off; off = ground(off + tokens * nh * d->dk * 4);
    gp->off_V = off; off = ground(off + tokens * nh * d->dv * 4);
    gp->off_fwd = off; off = ground(off + fwd);
    gp->fwd_bytes = fwd;
    gp->total = off;
    gp->gd = gd;
    return DPLR_OK;
}

}  // namespace
}  // namespace dplr

using namespace dplr;

extern "C" size_t dplr_gdp_workspace_size(const dplr_desc* desc) {
    GdpPlan gp;
    if (make_gdp_plan(desc, &gp) != DPLR_OK) return 0;
    return gp.total;
}

extern "C" dplr_status dplr_gdp_forward(const dplr_desc* desc, const void* q, const void* k, const void* v,
                                        const float* g, const float* beta, const float* S0, float* o, float* S_T,
                                        void* workspace, size_t ws_bytes, void* stream) {
    GdpPlan gp;
    dplr_status st = make_gdp_plan(desc, &gp);
    if (st != DPLR_OK) return st;
    const long long tokens = (long long)desc->B * desc->H * desc->T;
    auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (tokens > 0 && (!q || !k || !v || !g || !beta || !o || !al(q) || !al(k) || !al(v) || !al(g) || !al(beta) || !al(o)))
        return DPLR_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < gp.total || (reinterpret_cast<uintptr_t>(workspace) % kGAlign) != 0)
        return DPLR_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(workspace);
    float* q32 = reinterpret_cast<float*>(ws + gp.off_q);
    float* dec = reinterpret_cast<float*>(ws + gp.off_d);
    float* A = reinterpret_cast<float*>(ws + gp.off_A);
    float* Bm = reinterpret_cast<float*>(ws + gp.off_B);
    float* K = reinterpret_cast<float*>(ws + gp.off_K);
    float* V = reinterpret_cast<float*>(ws + gp.off_V);
    if (tokens > 0) {
        const unsigned grid = (unsigned)((tokens + 7) / 8);
        if (desc->in_dtype == DPLR_BF16)
            gdp_factor_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(tokens, desc->dk, desc->dv, desc->r_ab,
                static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v),
                g, beta, q32, dec, A, Bm, K, V);
        else
            gdp_factor_kernel<float><<<grid, 256, 0, s>>>(tokens, desc->dk, desc->dv, desc->r_ab, static_cast<const float*>(q),
                static_cast<const float*>(k), static_cast<const float*>(v), g, beta, q32, dec, A, Bm, K, V);
        if (cudaGetLastError() != cudaSuccess) return DPLR_ERR_CUDA;
    }
    return dplr_la_forward(&gp.gd, q32, nullptr, nullptr, dec, nullptr, A, Bm, K, V, S0, o, S_T, ws + gp.off_fwd,
                           gp.fwd_bytes, stream);
}

extern "C" const char* dplr_gdp_path(const dplr_desc* desc) {
    GdpPlan gp;
    if (make_gdp_plan(desc, &gp) != DPLR_OK) return "";
    return dplr_la_path(&gp.gd);
}
