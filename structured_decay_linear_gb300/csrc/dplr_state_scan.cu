// Stage 2 of the chunkwise DPLR forward: the inter-chunk state scan.
//
// The chunk maps of stage 1 are exact (affine closure: the token updates of a
// chunk compose into one map S -> P_j S + c_j), so the state at every chunk
// boundary follows from one matrix product per chunk, in order:
//     S_j = P_j S_{j-1} + c_j,        o_t += Q'_t S_{j-1}   (t in chunk j)
// (HDLA page, Key design 3: the chunk-boundary states are computed one after the
// other, then every chunk's output from its starting state; HLA page, affine
// closure.) The columns of S evolve independently (the decay acts from the left),
// so each CTA owns a block of kScanCols state columns of one head and walks all
// chunks. The next chunk's maps are copied in (cp.async) while the current one is
// applied.
#include <algorithm>

#include "dplr_internal.h"

namespace dplr {
namespace {

constexpr int kPad = 4;   // floats added to each row of the staged P and Q' (conflict-free float4 reads)

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                 :: "r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

// Shared-memory carve-up (floats): S [dk][nv], then two stages of {P [dk][dk+kPad],
// Q' [cw][dk+kPad], c [dk][nv]}.
struct ScanLayout {
    int nv, dkp, stage, p0, q0, c0, total;
    __host__ __device__ ScanLayout(int dk, int dv, int cw) {
        dkp = dk + kPad;
        // kScanCols state columns per CTA, fewer when the two stages would not fit
        for (nv = dv < kScanCols ? dv : kScanCols; nv > 4; nv /= 2)
            if (4 * (dk * nv + 2 * (dk * dkp + cw * dkp + dk * nv)) <= 227 * 1024) break;
        stage = dk * dkp + cw * dkp + dk * nv;
        p0 = dk * nv;             // S first
        q0 = p0 + dk * dkp;
        c0 = q0 + cw * dkp;
        total = dk * nv + 2 * stage;
    }
    __host__ __device__ int P(int b) const { return p0 + b * stage; }
    __host__ __device__ int Q(int b) const { return q0 + b * stage; }
    __host__ __device__ int C(int b) const { return c0 + b * stage; }
};

// acc (4 x 4) += A[m0..m0+3][0..K) * S[0..K)[c0..c0+3]; rows of A with stride lda, S with
// stride nv, all float4-aligned. K is a multiple of 4.
__device__ __forceinline__ void tile_4x4(const float* A, int lda, const float* S, int nv, int K, int m0, int c0,
                                         float (&acc)[4][4]) {
    for (int k = 0; k < K; k += 4) {
        float4 a[4], b[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = *reinterpret_cast<const float4*>(A + (m0 + i) * lda + k);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) b[kk] = *reinterpret_cast<const float4*>(S + (k + kk) * nv + c0);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const float av = kk == 0 ? a[i].x : (kk == 1 ? a[i].y : (kk == 2 ? a[i].z : a[i].w));
                acc[i][0] = fmaf(av, b[kk].x, acc[i][0]);
                acc[i][1] = fmaf(av, b[kk].y, acc[i][1]);
                acc[i][2] = fmaf(av, b[kk].z, acc[i][2]);
                acc[i][3] = fmaf(av, b[kk].w, acc[i][3]);
            }
        }
    }
}

__global__ void __launch_bounds__(2 * kScanThreads, 1)
state_scan_kernel(Plan pl, ScanArgs args) {
    extern __shared__ __align__(16) float sm[];
    const int dk = pl.dk, dv = pl.dv, cw = pl.cw, T = pl.T;
    const ScanLayout Ly(dk, dv, cw);
    const int nv = Ly.nv, dkp = Ly.dkp;
    const int ncb = dv / nv;
    const size_t bh = blockIdx.x / ncb;
    const int n0 = (blockIdx.x % ncb) * nv;
    const int tid = threadIdx.x, nth = blockDim.x;
    float* S = sm;

    // chunk jj's maps into stage b: P and Q' are contiguous rows, c a column block of its rows
    auto prefetch = [&](int jj, int b) {
        const size_t unit = bh * (size_t)pl.nb + jj;
        const float* Pg = args.Pm + unit * (size_t)dk * dk;
        const float* Qg = args.Qm + unit * (size_t)cw * dk;
        const float* Cg = args.Cm + unit * (size_t)dk * dv + n0;
        const int q4 = dk / 4, n4 = nv / 4;
        for (int i = tid; i < dk * q4; i += nth) cp_async16(sm + Ly.P(b) + (i / q4) * dkp + 4 * (i % q4), Pg + 4 * i);
        for (int i = tid; i < cw * q4; i += nth) cp_async16(sm + Ly.Q(b) + (i / q4) * dkp + 4 * (i % q4), Qg + 4 * i);
        for (int i = tid; i < dk * n4; i += nth) cp_async16(sm + Ly.C(b) + 4 * i, Cg + (size_t)(i / n4) * dv + 4 * (i % n4));
        cp_async_commit();
    };

    for (int i = tid; i < dk * nv; i += nth) {
        const int r = i / nv, n = i % nv;
        S[i] = args.S0 ? args.S0[(bh * dk + r) * dv + n0 + n] : 0.f;
    }
    if (pl.nb > 0) prefetch(0, 0);
    // Thread roles for a chunk: one 4x4 tile of S_j (tiles_s of them), then one 4x4 tile of
    // the readout Q'_j S_{j-1} (tiles_o), computed side by side from S_{j-1}.
    const int tn = nv / 4;
    const int tiles_s = (dk / 4) * tn, tiles_o = (cw / 4) * tn;
    for (int j = 0; j < pl.nb; ++j) {
        const int b = j & 1;
        if (j + 1 < pl.nb) {   // the other stage was last read by chunk j-1 (finished below)
            prefetch(j + 1, b ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();   // chunk j's maps (every thread's copies) and S_{j-1} in place
        if (args.Sb) {     // the state before chunk j, for the backward
            float* dst = args.Sb + (bh * (size_t)pl.nb + j) * (size_t)dk * dv + n0;
            for (int i = tid; i < dk * nv; i += nth) dst[(size_t)(i / nv) * dv + i % nv] = S[i];
        }
        const float* Pj = sm + Ly.P(b);
        const float* Qj = sm + Ly.Q(b);
        const float* cj = sm + Ly.C(b);
        float acc[4][4];
        int m0 = 0, c0 = 0;
        const bool upd = tid < tiles_s;
        for (int tile = tid; tile < tiles_s + tiles_o; tile += nth) {
            if (tile < tiles_s) {   // S_j = P_j S_{j-1} + c_j  (one tile per thread: tiles_s <= nth)
                m0 = (tile / tn) * 4; c0 = (tile % tn) * 4;
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int l = 0; l < 4; ++l) acc[i][l] = cj[(m0 + i) * nv + c0 + l];
                tile_4x4(Pj, dkp, S, nv, dk, m0, c0, acc);
            } else {                // o_t += Q'_t S_{j-1}
                const int tt = tile - tiles_s;
                const int r0 = (tt / tn) * 4, d0 = (tt % tn) * 4;
                const int t0 = j * cw;
                // stage 1's zero-state outputs, loaded first: their latency overlaps the product
                float4 v[4];
                float4* orow[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    orow[i] = reinterpret_cast<float4*>(args.o + (bh * (size_t)T + t0 + r0 + i) * dv + n0 + d0);
                    v[i] = (t0 + r0 + i < T) ? *orow[i] : make_float4(0.f, 0.f, 0.f, 0.f);
                }
                float ao[4][4] = {};
                tile_4x4(Qj, dkp, S, nv, dk, r0, d0, ao);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (t0 + r0 + i >= T) continue;
                    v[i].x += ao[i][0]; v[i].y += ao[i][1]; v[i].z += ao[i][2]; v[i].w += ao[i][3];
                    *orow[i] = v[i];
                }
            }
        }
        __syncthreads();   // every read of S_{j-1} done
        if (upd) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                *reinterpret_cast<float4*>(S + (m0 + i) * nv + c0) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        }
    }
    __syncthreads();
    if (args.ST)
        for (int i = tid; i < dk * nv; i += nth) {
            const int r = i / nv, n = i % nv;
            args.ST[(bh * dk + r) * dv + n0 + n] = S[i];
        }
}

}  // namespace

size_t scan_smem_bytes(const Plan& pl) { return sizeof(float) * (size_t)ScanLayout(pl.dk, pl.dv, pl.cw).total; }

cudaError_t launch_state_scan(const Plan& pl, const ScanArgs& a, cudaStream_t s) {
    const int nv = ScanLayout(pl.dk, pl.dv, pl.cw).nv;
    const size_t smem = scan_smem_bytes(pl);
    static std::atomic<uint64_t> done{0};   // raised to the largest footprint once per device
    cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(state_scan_kernel), 227 * 1024, done);
    if (e != cudaSuccess) return e;
    const long long grid = (long long)pl.BH * (pl.dv / nv);
    // one 4 x 4 tile per thread: the state update's and the readout's tiles side by side, not one after the other
    const int tiles = (pl.dk / 4) * (nv / 4) + (pl.cw / 4) * (nv / 4);
    const int nth = std::min(2 * kScanThreads, std::max(kScanThreads, (tiles + 31) / 32 * 32));
    state_scan_kernel<<<(unsigned)grid, nth, smem, s>>>(pl, a);
    return cudaGetLastError();
}

}  // namespace dplr
