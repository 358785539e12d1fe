// A block-wide fp32 product in shared memory (CUDA cores), shared by the backward and the HLA kernels.
#pragma once

namespace dplr {
namespace smem {

// C[m][n] (=, +=) alpha sum_k A(m, k) B(k, n) over the CTA's threads, with A(m, k) = A[m lda + k] (ta: A[k lda + m])
// and B(k, n) = B[k ldb + n] (tb: B[n ldb + k]); all in shared memory. M and N are multiples of 4: each thread takes
// 4 x 4 tiles of C (8 shared loads per 16 FMAs).
__device__ __forceinline__ void mm(float* C, int ldc, const float* A, int lda, bool ta, const float* B, int ldb,
                                   bool tb, int M, int N, int K, float alpha, bool acc) {
    const int nt = N >> 2, tiles = (M >> 2) * nt;
    const int as = ta ? 1 : lda, ak = ta ? lda : 1;   // A(m, k) = A[m as + k ak]
    const int bs = tb ? ldb : 1, bk = tb ? 1 : ldb;   // B(k, n) = B[k bk + n bs]
    for (int tile = threadIdx.x; tile < tiles; tile += blockDim.x) {
        const int m0 = (tile / nt) << 2, n0 = (tile % nt) << 2;
        float c[4][4] = {};
        const float* Ap = A + m0 * as;
        const float* Bp = B + n0 * bs;
        for (int k = 0; k < K; ++k) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                a[i] = Ap[i * as + k * ak];
                b[i] = Bp[i * bs + k * bk];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) c[i][jj] = fmaf(a[i], b[jj], c[i][jj]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                float* o = C + (m0 + i) * ldc + n0 + jj;
                *o = acc ? *o + alpha * c[i][jj] : alpha * c[i][jj];
            }
    }
}

}  // namespace smem
}  // namespace dplr
