// HLA: query-conditioned composition of exact chunk transitions ("HLA: Expressive Hybrid Linear Attention via
// Chunk-Wise Dynamic Mixing", Method steps 1, 2, 4 and 5) on the Gated DeltaNet update.
//
// The sequence is cut into chunks of L tokens (L = 64, 128 or 256). Chunk j has the exact affine summary
// S -> A_j S + B_j of its token updates (affine closure, the page's Prerequisites). For query token i in chunk c,
// with gates w_ij for the earlier chunks (those below a threshold set to zero),
//     S_i = 0;  S_i = ((1 - w_ij) I + w_ij A_j) S_i + w_ij B_j  for j = 0 .. c - 1,
//     then the current chunk's causal prefix;  o_i = S_i^T q_i.
// The prefix makes o_i = U_i S_{i,c-1} + O_i, with U_i = q_i^T A_{c,<=i} (the query's readout row through the
// prefix) and O_i its output from a zero state. Unrolling the composition from the newest chunk backwards:
//     o_i = O_i;  for j = c - 1 .. 0:  o_i += w_ij U_i B_j;  U_i <- (1 - w_ij) U_i + w_ij U_i A_j
// (the page's reverse-order history readout). Three passes:
//   1. the fp32 chunk-map kernel at WY blocks of 64 tokens: P_b, c_b, the readout rows Q'_t and O_t;
//   2. (L > 64) the L-chunk summaries composed from their blocks, A = P_{m-1} .. P_0, B likewise, and each
//      query's row U_t = Q'_t (the composition of its chunk's earlier blocks), its output O_t updated;
//   3. per 64 queries of one chunk, the history chunks newest first: two products per chunk, U A_j and U B_j,
//      with the gates applied per query; a chunk whose gates are all zero for the 64 queries is skipped.
// Passes 2 and 3 run in fp32 on the CUDA cores, with 4 x 4 register tiles.
#include <algorithm>
#include <cstring>

#include "dplr_internal.h"

namespace dplr {
namespace {

constexpr int HQ = 64;       // queries per CTA of pass 3, tokens per WY block
constexpr int HT = 256;      // threads

struct HlaPlan {
    Plan pl;          // the fp32 two-stage plan at WY blocks of 64 tokens (GDN)
    int L, m, N;      // chunk length, WY blocks per chunk, chunks per head
    size_t off_A, off_B, total;   // L-chunk summaries (L > 64; else the blocks' own maps)
};

__device__ __forceinline__ void l2_prefetch(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(reinterpret_cast<uint64_t>(p)), "r"(bytes) : "memory");
}

// ---- pass 2: per (head, L-chunk), its m blocks in order
__global__ void __launch_bounds__(HT, 1)
hla_compose_kernel(Plan pl, int m, int N, const float* Pm, const float* Cm, float* Qm, float* o, float* Aout,
                   float* Bout) {
    extern __shared__ __align__(16) float sm[];
    const int dk = pl.dk, dv = pl.dv, T = pl.T, nb = pl.nb;
    float* A = sm;                // [dk][dk] the composition of the chunk's blocks so far
    float* Bc = A + dk * dk;      // [dk][dv]
    float* P = Bc + dk * dv;      // [dk][dk] the block's transition
    float* Q = P + dk * dk;       // [64][dk] the block's readout rows
    const int tid = threadIdx.x, nth = blockDim.x;
    const int c = blockIdx.x % N;
    const size_t bh = blockIdx.x / N;
    const int b0 = c * m, nbc = min(m, nb - b0);   // the chunk's blocks
    auto unit = [&](int b) { return bh * (size_t)nb + b; };
    for (int i = tid; i < dk * dk; i += nth) A[i] = Pm[unit(b0) * dk * dk + i];
    for (int i = tid; i < dk * dv; i += nth) Bc[i] = Cm[unit(b0) * dk * dv + i];
    for (int k = 1; k < nbc; ++k) {
        const size_t u = unit(b0 + k);
        __syncthreads();
        for (int i = tid; i < HQ * dk; i += nth) Q[i] = Qm[u * HQ * dk + i];
        for (int i = tid; i < dk * dk; i += nth) P[i] = Pm[u * dk * dk + i];
        __syncthreads();
        // the block's queries: U_t = Q'_t A (over Q'_t in the workspace), O_t += Q'_t B (valid tokens)
        for (int tile = tid; tile < (HQ / 4) * (dk / 4); tile += nth) {
            const int r0 = 4 * (tile / (dk / 4)), n0 = 4 * (tile % (dk / 4));
            float acc[4][4] = {};
            for (int kx = 0; kx < dk; ++kx) {
                const float4 b = *reinterpret_cast<const float4*>(A + kx * dk + n0);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float a = Q[(r0 + i) * dk + kx];
                    acc[i][0] = fmaf(a, b.x, acc[i][0]); acc[i][1] = fmaf(a, b.y, acc[i][1]);
                    acc[i][2] = fmaf(a, b.z, acc[i][2]); acc[i][3] = fmaf(a, b.w, acc[i][3]);
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
                *reinterpret_cast<float4*>(Qm + u * HQ * dk + (size_t)(r0 + i) * dk + n0) =
                    make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        }
        for (int tile = tid; tile < (HQ / 4) * (dv / 4); tile += nth) {
            const int r0 = 4 * (tile / (dv / 4)), n0 = 4 * (tile % (dv / 4));
            float acc[4][4] = {};
            for (int kx = 0; kx < dk; ++kx) {
                const float4 b = *reinterpret_cast<const float4*>(Bc + kx * dv + n0);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float a = Q[(r0 + i) * dk + kx];
                    acc[i][0] = fmaf(a, b.x, acc[i][0]); acc[i][1] = fmaf(a, b.y, acc[i][1]);
                    acc[i][2] = fmaf(a, b.z, acc[i][2]); acc[i][3] = fmaf(a, b.w, acc[i][3]);
                }
            }
            const int t0 = (b0 + k) * HQ;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (t0 + r0 + i < T) {
                    float4* po = reinterpret_cast<float4*>(o + (bh * (size_t)T + t0 + r0 + i) * dv + n0);
                    float4 x = *po;
                    x.x += acc[i][0]; x.y += acc[i][1]; x.z += acc[i][2]; x.w += acc[i][3];
                    *po = x;
                }
        }
        __syncthreads();   // A and B read by every query tile
        // A <- P A and B <- P B + c_k: 4 x 4 tiles formed in registers from shared memory, written to this chunk's
        // slots of the output arrays, then read back once every tile is formed
        float* Ag = Aout + (bh * (size_t)N + c) * dk * dk;
        float* Bg = Bout + (bh * (size_t)N + c) * dk * dv;
        const float* cg = Cm + u * dk * dv;
        auto prod = [&](const float* Y, int ny, float* dst, const float* add) {
            for (int tile = tid; tile < (dk / 4) * (ny / 4); tile += nth) {
                const int r0 = 4 * (tile / (ny / 4)), n0 = 4 * (tile % (ny / 4));
                float acc[4][4] = {};
                for (int kx = 0; kx < dk; ++kx) {
                    const float4 b = *reinterpret_cast<const float4*>(Y + kx * ny + n0);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float a = P[(r0 + i) * dk + kx];
                        acc[i][0] = fmaf(a, b.x, acc[i][0]); acc[i][1] = fmaf(a, b.y, acc[i][1]);
                        acc[i][2] = fmaf(a, b.z, acc[i][2]); acc[i][3] = fmaf(a, b.w, acc[i][3]);
                    }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float4 x = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
                    if (add) {
                        const float4 y = *reinterpret_cast<const float4*>(add + (size_t)(r0 + i) * ny + n0);
                        x.x += y.x; x.y += y.y; x.z += y.z; x.w += y.w;
                    }
                    *reinterpret_cast<float4*>(dst + (size_t)(r0 + i) * ny + n0) = x;
                }
            }
        };
        prod(A, dk, Ag, nullptr);
        prod(Bc, dv, Bg, cg);
        __syncthreads();
        for (int i = tid; i < dk * dk; i += nth) A[i] = Ag[i];
        for (int i = tid; i < dk * dv; i += nth) Bc[i] = Bg[i];
    }
    __syncthreads();
    for (int i = tid; i < dk * dk; i += nth) Aout[(bh * (size_t)N + c) * dk * dk + i] = A[i];
    for (int i = tid; i < dk * dv; i += nth) Bout[(bh * (size_t)N + c) * dk * dv + i] = Bc[i];
}

// ---- pass 3: per (head, 64 queries), the history chunks newest first
__global__ void __launch_bounds__(HT, 1)
hla_gated_kernel(Plan pl, int L, int N, float theta, const float* Um, const float* Acs, const float* Bcs,
                 const float* W, float* o) {
    extern __shared__ __align__(16) float sm[];
    const int dk = pl.dk, dv = pl.dv, T = pl.T, nb = pl.nb;
    float* U = sm;                // [64][dk]
    float* A = U + HQ * dk;       // [dk][dk]
    float* B = A + dk * dk;       // [dk][dv]
    float* w = B + dk * dv;       // [64]
    const int tid = threadIdx.x, nth = blockDim.x;
    const int nqb = nb;           // query blocks per head (64 tokens each)
    const int qb = blockIdx.x % nqb;
    const size_t bh = blockIdx.x / nqb;
    const int t0 = qb * HQ, c = t0 / L;
    for (int i = tid; i < HQ * dk; i += nth) U[i] = Um[(bh * (size_t)nb + qb) * HQ * dk + i];
    const int ntx = dk / 4, nty = dv / 4;
    float oacc[2][4][4] = {};
    float xacc[2][4][4];
    if (tid == 0 && c > 0) {
        l2_prefetch(Acs + (bh * (size_t)N + (c - 1)) * dk * dk, (uint32_t)(dk * dk * 4));
        l2_prefetch(Bcs + (bh * (size_t)N + (c - 1)) * dk * dv, (uint32_t)(dk * dv * 4));
    }
    for (int l = c - 1; l >= 0; --l) {
        __syncthreads();   // the previous chunk's reads of A, B and w done; U updated
        bool any = false;
        if (tid < HQ) {
            const int t = t0 + tid;
            float x = t < T ? W[(bh * (size_t)T + t) * N + l] : 0.f;
            if (!(x >= theta)) x = 0.f;
            w[tid] = x;
            any = x != 0.f;
        }
        if (!__syncthreads_or(any)) continue;   // every query passes this chunk unchanged
        if (tid == 0 && l > 0) {
            l2_prefetch(Acs + (bh * (size_t)N + (l - 1)) * dk * dk, (uint32_t)(dk * dk * 4));
            l2_prefetch(Bcs + (bh * (size_t)N + (l - 1)) * dk * dv, (uint32_t)(dk * dv * 4));
        }
        const float4* A4 = reinterpret_cast<const float4*>(Acs + (bh * (size_t)N + l) * dk * dk);
        const float4* B4 = reinterpret_cast<const float4*>(Bcs + (bh * (size_t)N + l) * dk * dv);
        for (int i = tid; i < dk * dk / 4; i += nth) reinterpret_cast<float4*>(A)[i] = A4[i];
        for (int i = tid; i < dk * dv / 4; i += nth) reinterpret_cast<float4*>(B)[i] = B4[i];
        __syncthreads();
        // o += diag(w) U B_l  and  X = U A_l, from the current U
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int tile = tid + e * nth;
            if (tile < (HQ / 4) * nty) {
                const int r0 = 4 * (tile / nty), n0 = 4 * (tile % nty);
                float acc[4][4] = {};
                for (int kx = 0; kx < dk; ++kx) {
                    const float4 b = *reinterpret_cast<const float4*>(B + kx * dv + n0);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float a = U[(r0 + i) * dk + kx];
                        acc[i][0] = fmaf(a, b.x, acc[i][0]); acc[i][1] = fmaf(a, b.y, acc[i][1]);
                        acc[i][2] = fmaf(a, b.z, acc[i][2]); acc[i][3] = fmaf(a, b.w, acc[i][3]);
                    }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) oacc[e][i][jj] = fmaf(w[r0 + i], acc[i][jj], oacc[e][i][jj]);
            }
            if (tile < (HQ / 4) * ntx) {
                const int r0 = 4 * (tile / ntx), n0 = 4 * (tile % ntx);
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) xacc[e][i][jj] = 0.f;
                for (int kx = 0; kx < dk; ++kx) {
                    const float4 b = *reinterpret_cast<const float4*>(A + kx * dk + n0);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float a = U[(r0 + i) * dk + kx];
                        xacc[e][i][0] = fmaf(a, b.x, xacc[e][i][0]); xacc[e][i][1] = fmaf(a, b.y, xacc[e][i][1]);
                        xacc[e][i][2] = fmaf(a, b.z, xacc[e][i][2]); xacc[e][i][3] = fmaf(a, b.w, xacc[e][i][3]);
                    }
                }
            }
        }
        __syncthreads();   // every read of U done: U <- (1 - w) U + w X
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int tile = tid + e * nth;
            if (tile < (HQ / 4) * ntx) {
                const int r0 = 4 * (tile / ntx), n0 = 4 * (tile % ntx);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float wi = w[r0 + i];
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        float* u = U + (r0 + i) * dk + n0 + jj;
                        *u = (1.f - wi) * *u + wi * xacc[e][i][jj];
                    }
                }
            }
        }
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int tile = tid + e * nth;
        if (tile < (HQ / 4) * nty) {
            const int r0 = 4 * (tile / nty), n0 = 4 * (tile % nty);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (t0 + r0 + i < T) {
                    float4* po = reinterpret_cast<float4*>(o + (bh * (size_t)T + t0 + r0 + i) * dv + n0);
                    float4 x = *po;
                    x.x += oacc[e][i][0]; x.y += oacc[e][i][1]; x.z += oacc[e][i][2]; x.w += oacc[e][i][3];
                    *po = x;
                }
        }
    }
}

constexpr size_t kHAlign = 256;
size_t hround(size_t x) { return (x + kHAlign - 1) / kHAlign * kHAlign; }

dplr_status make_hla_plan(const dplr_desc* d, int L, HlaPlan* hp) {
    Plan p;
    dplr_status st = make_plan(d, &p);
    if (st != DPLR_OK) return st;
    if (p.mode != DPLR_GDN) return DPLR_ERR_INVALID_ARG;
    if (L != 64 && L != 128 && L != 256) return DPLR_ERR_UNSUPPORTED;
    if (p.dk > 128 || p.dv > 128) return DPLR_ERR_UNSUPPORTED;
    p.fused = p.tc = p.gtc = 0;
    p.cw = HQ;
    p.nb = (p.T + HQ - 1) / HQ;
    const size_t units = (size_t)p.BH * p.nb;
    size_t off = kHAlign;
    p.off_P = off; off = hround(off + units * (size_t)p.dk * p.dk * sizeof(float));
    p.off_c = off; off = hround(off + units * (size_t)p.dk * p.dv * sizeof(float));
    p.off_Q = off; off = hround(off + units * (size_t)HQ * p.dk * sizeof(float));
    p.ws_stages = off;
    if (prep_smem_bytes(p) > 227 * 1024) return DPLR_ERR_UNSUPPORTED;
    hp->L = L;
    hp->m = L / HQ;
    hp->N = (p.T + L - 1) / L;
    if (hp->m > 1) {
        const size_t chunks = (size_t)p.BH * hp->N;
        hp->off_A = off; off = hround(off + chunks * (size_t)p.dk * p.dk * sizeof(float));
        hp->off_B = off; off = hround(off + chunks * (size_t)p.dk * p.dv * sizeof(float));
    } else {
        hp->off_A = p.off_P;
        hp->off_B = p.off_c;
    }
    hp->total = off;
    p.ws_bytes = off;
    hp->pl = p;
    return DPLR_OK;
}

std::atomic<uint64_t> g_hla_smem[2] = {{0}, {0}};

}  // namespace
}  // namespace dplr

using namespace dplr;

extern "C" size_t dplr_hla_workspace_size(const dplr_desc* desc, int L) {
    HlaPlan hp;
    if (make_hla_plan(desc, L, &hp) != DPLR_OK) return 0;
    return hp.total;
}

extern "C" dplr_status dplr_hla_forward(const dplr_desc* desc, const void* q, const void* k, const void* v,
                                        const float* g, const float* beta, const float* W, float theta, int L,
                                        float* o, void* workspace, size_t ws_bytes, void* stream) {
    HlaPlan hp;
    dplr_status st = make_hla_plan(desc, L, &hp);
    if (st != DPLR_OK) return st;
    const Plan& pl = hp.pl;
    if (pl.T == 0) return DPLR_OK;
    auto al = [](const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!al(q) || !al(k) || !al(v) || !al(g) || !al(beta) || !al(W) || !al(o)) return DPLR_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < hp.total || (reinterpret_cast<uintptr_t>(workspace) % kHAlign) != 0)
        return DPLR_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(workspace);
    ChunkMapArgs ma;
    ma.q = q; ma.k = k; ma.v = v; ma.decay = g; ma.beta = beta;
    ma.A = nullptr; ma.Bm = nullptr; ma.K = nullptr; ma.V = nullptr; ma.o = o;
    ma.Pm = reinterpret_cast<float*>(ws + pl.off_P);
    ma.Cm = reinterpret_cast<float*>(ws + pl.off_c);
    ma.Qm = reinterpret_cast<float*>(ws + pl.off_Q);
    if (launch_chunk_maps(pl, ma, s) != cudaSuccess) return DPLR_ERR_CUDA;   // pass 1 (o <- O_t)
    float* Acs = reinterpret_cast<float*>(ws + hp.off_A);
    float* Bcs = reinterpret_cast<float*>(ws + hp.off_B);
    if (hp.m > 1) {   // pass 2
        const size_t smem = sizeof(float) * (size_t)(2 * pl.dk * pl.dk + pl.dk * pl.dv + HQ * pl.dk);
        if (set_smem_limit_once(reinterpret_cast<const void*>(hla_compose_kernel), 227 * 1024, g_hla_smem[0]) != cudaSuccess)
            return DPLR_ERR_CUDA;
        hla_compose_kernel<<<(unsigned)((size_t)pl.BH * hp.N), HT, smem, s>>>(pl, hp.m, hp.N, ma.Pm, ma.Cm, ma.Qm, o, Acs, Bcs);
        if (cudaGetLastError() != cudaSuccess) return DPLR_ERR_CUDA;
    }
    {   // pass 3
        const size_t smem = sizeof(float) * (size_t)(HQ * pl.dk + pl.dk * pl.dk + pl.dk * pl.dv + HQ);
        if (set_smem_limit_once(reinterpret_cast<const void*>(hla_gated_kernel), 227 * 1024, g_hla_smem[1]) != cudaSuccess)
            return DPLR_ERR_CUDA;
        hla_gated_kernel<<<(unsigned)((size_t)pl.BH * pl.nb), HT, smem, s>>>(pl, hp.L, hp.N, theta, ma.Qm, Acs, Bcs, W, o);
        if (cudaGetLastError() != cudaSuccess) return DPLR_ERR_CUDA;
    }
    return DPLR_OK;
}
