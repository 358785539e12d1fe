// Stage 2 of the chunkwise DPLR forward: the inter-chunk state scan.
//
// The chunk maps of stage 1 are exact (affine closure: the token updates of a
// chunk compose into one map S -> P_j S + c_j), so the state at every chunk
// boundary follows from one matrix product per chunk, in order:
//     S_j = P_j S_{j-1} + c_j,        o_t += Q'_t S_{j-1}   (t in chunk j)
// (HDLA page, Key design 3: "serially compute the chunk-state checkpoints",
// then the per-chunk outputs; HLA page, affine closure.) The columns of S
// evolve independently (the decay acts from the left), so each CTA owns a
// block of kScanCols state columns of one head and walks all chunks.
#include "dplr_internal.h"

namespace dplr {
namespace {

__global__ void __launch_bounds__(kScanThreads)
state_scan_kernel(Plan pl, ScanArgs args) {
    extern __shared__ float sm[];
    const int dk = pl.dk, dv = pl.dv, cw = pl.cw, T = pl.T;
    const int nv = dv < kScanCols ? dv : kScanCols;
    const int ncb = dv / nv;
    const size_t bh = blockIdx.x / ncb;
    const int n0 = (blockIdx.x % ncb) * nv;
    const int tid = threadIdx.x, nth = blockDim.x;
    float* S = sm;                 // [dk][nv]
    float* Pj = S + dk * nv;       // [dk][dk]
    float* Qj = Pj + dk * dk;      // [cw][dk]
    float* cj = Qj + cw * dk;      // [dk][nv]

    for (int i = tid; i < dk * nv; i += nth) {
        const int r = i / nv, n = i % nv;
        S[i] = args.S0 ? args.S0[(bh * dk + r) * dv + n0 + n] : 0.f;
    }
    // Each thread owns a fixed set of 4x4 output tiles of S_new (dk x nv) and O (cw x nv).
    const int tiles_s = (dk / 4) * (nv / 4);
    const int tiles_o = (cw / 4) * (nv / 4);
    const int tn = nv / 4;
    for (int j = 0; j < pl.nb; ++j) {
        const size_t unit = bh * (size_t)pl.nb + j;
        const float4* Pg = reinterpret_cast<const float4*>(args.Pm + unit * (size_t)dk * dk);
        const float4* Qg = reinterpret_cast<const float4*>(args.Qm + unit * (size_t)cw * dk);
        for (int i = tid; i < dk * dk / 4; i += nth) reinterpret_cast<float4*>(Pj)[i] = Pg[i];
        for (int i = tid; i < cw * dk / 4; i += nth) reinterpret_cast<float4*>(Qj)[i] = Qg[i];
        const float* Cg = args.Cm + unit * (size_t)dk * dv;
        for (int i = tid; i < dk * nv; i += nth) cj[i] = Cg[(i / nv) * dv + n0 + i % nv];
        __syncthreads();
        // o_t += Q'_t S_{j-1}
        const int t0 = j * cw;
        for (int tile = tid; tile < tiles_o; tile += nth) {
            const int m0 = (tile / tn) * 4, c0 = (tile % tn) * 4;
            float acc[4][4] = {};
            for (int k = 0; k < dk; ++k) {
                float a[4], b[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) a[i] = Qj[(m0 + i) * dk + k];
#pragma unroll
                for (int i = 0; i < 4; ++i) b[i] = S[k * nv + c0 + i];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int l = 0; l < 4; ++l) acc[i][l] = fmaf(a[i], b[l], acc[i][l]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (t0 + m0 + i >= T) continue;
                float* orow = args.o + (bh * (size_t)T + t0 + m0 + i) * dv + n0 + c0;
#pragma unroll
                for (int l = 0; l < 4; ++l) orow[l] += acc[i][l];
            }
        }
        // S_j = P_j S_{j-1} + c_j   (computed into registers, then written back)
        float snew[2][4][4];
        int ntile = 0;
        for (int tile = tid; tile < tiles_s && ntile < 2; tile += nth, ++ntile) {
            const int m0 = (tile / tn) * 4, c0 = (tile % tn) * 4;
            float acc[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int l = 0; l < 4; ++l) acc[i][l] = cj[(m0 + i) * nv + c0 + l];
            for (int k = 0; k < dk; ++k) {
                float a[4], b[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) a[i] = Pj[(m0 + i) * dk + k];
#pragma unroll
                for (int i = 0; i < 4; ++i) b[i] = S[k * nv + c0 + i];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int l = 0; l < 4; ++l) acc[i][l] = fmaf(a[i], b[l], acc[i][l]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int l = 0; l < 4; ++l) snew[ntile][i][l] = acc[i][l];
        }
        __syncthreads();
        ntile = 0;
        for (int tile = tid; tile < tiles_s && ntile < 2; tile += nth, ++ntile) {
            const int m0 = (tile / tn) * 4, c0 = (tile % tn) * 4;
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int l = 0; l < 4; ++l) S[(m0 + i) * nv + c0 + l] = snew[ntile][i][l];
        }
        __syncthreads();
    }
    if (args.ST)
        for (int i = tid; i < dk * nv; i += nth) {
            const int r = i / nv, n = i % nv;
            args.ST[(bh * dk + r) * dv + n0 + n] = S[i];
        }
}

}  // namespace

size_t scan_smem_bytes(const Plan& pl) {
    const int nv = pl.dv < kScanCols ? pl.dv : kScanCols;
    return sizeof(float) * ((size_t)pl.dk * nv * 2 + (size_t)pl.dk * pl.dk + (size_t)pl.cw * pl.dk);
}

cudaError_t launch_state_scan(const Plan& pl, const ScanArgs& a, cudaStream_t s) {
    const int nv = pl.dv < kScanCols ? pl.dv : kScanCols;
    const size_t smem = scan_smem_bytes(pl);
    cudaError_t e = cudaFuncSetAttribute(state_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const long long grid = (long long)pl.BH * (pl.dv / nv);
    state_scan_kernel<<<(unsigned)grid, kScanThreads, smem, s>>>(pl, a);
    return cudaGetLastError();
}

}  // namespace dplr
