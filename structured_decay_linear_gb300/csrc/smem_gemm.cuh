// Block-wide fp32 products in shared memory (CUDA cores): mm, and mm_ksplit_out for products with few tiles
// and a long K. Used by the backward kernels.
#pragma once

namespace dplr {
namespace smem {

// C[m][n] (=, +=) alpha sum_k A(m, k) B(k, n) over the CTA's threads (or over threads t0 .. t0 + nt_ - 1 only, so
// that independent small products can run side by side), with A(m, k) = A[m lda + k] (ta: A[k lda + m]) and
// B(k, n) = B[k ldb + n] (tb: B[n ldb + k]); all in shared memory. M and N are multiples of 4: each thread takes
// 4 x 4 tiles of C (8 shared loads per 16 FMAs).
__device__ __forceinline__ void mm(float* C, int ldc, const float* A, int lda, bool ta, const float* B, int ldb,
                                   bool tb, int M, int N, int K, float alpha, bool acc, int t0 = 0, int nt_ = 0) {
    const int nt = N >> 2, tiles = (M >> 2) * nt;
    const int as = ta ? 1 : lda, ak = ta ? lda : 1;   // A(m, k) = A[m as + k ak]
    const int bs = tb ? ldb : 1, bk = tb ? 1 : ldb;   // B(k, n) = B[k bk + n bs]
    const int step = nt_ > 0 ? nt_ : (int)blockDim.x, me = (int)threadIdx.x - t0;
    if (me < 0 || me >= step) return;
    for (int tile = me; tile < tiles; tile += step) {
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

// One term A B of a K-split product (operands as in mm) and its K.
struct KTerm {
    const float* A; int lda; bool ta;
    const float* B; int ldb; bool tb;
    int K;
};
// One output of mm_ksplit_out: C (=, +=) alpha (the sum of its nt <= 3 terms), C M x N (M, N multiples of 4).
struct KOut {
    float* C; int ldc; int M, N;
    float alpha; bool acc;
    int nt; KTerm t[3];
};

namespace detail {
// The partial tiles of output q (index o of NOUT) by the CTA's threads of that output.
template <int NOUT>
__device__ __forceinline__ void ksplit_partials(const KOut& q, int o, float* scratch) {
    const int per = blockDim.x / NOUT, lt = threadIdx.x - o * per;
    const int nt = q.N >> 2, tiles = (q.M >> 2) * nt, G = max(1, per / tiles);
    int Ktot = 0;
#pragma unroll
    for (int i = 0; i < 3; ++i) Ktot += i < q.nt ? q.t[i].K : 0;
    const int kc = (Ktot + G - 1) / G;
    float* part = scratch + (size_t)o * 16 * per;
    for (int w = lt; w < G * tiles; w += per) {
        const int g = w / tiles, tile = w - g * tiles;
        const int m0 = (tile / nt) << 2, n0 = (tile % nt) << 2;
        const int k0 = g * kc, k1 = min(Ktot, k0 + kc);
        float c[4][4] = {};
        int off = 0;
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            if (i >= q.nt) break;
            const KTerm& t = q.t[i];
            const int lo = max(k0, off) - off, hi = min(k1, off + t.K) - off;
            off += t.K;
            const int as = t.ta ? 1 : t.lda, ak = t.ta ? t.lda : 1;
            const int bs = t.tb ? t.ldb : 1, bk = t.tb ? 1 : t.ldb;
            const float* Ap = t.A + m0 * as;
            const float* Bp = t.B + n0 * bs;
            for (int k = lo; k < hi; ++k) {
                float a[4], b[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    a[e] = Ap[e * as + k * ak];
                    b[e] = Bp[e * bs + k * bk];
                }
#pragma unroll
                for (int e = 0; e < 4; ++e)
#pragma unroll
                    for (int f = 0; f < 4; ++f) c[e][f] = fmaf(a[e], b[f], c[e][f]);
            }
        }
        float* P = part + (size_t)g * q.M * q.N;
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
            for (int f = 0; f < 4; ++f) P[(m0 + e) * q.N + n0 + f] = c[e][f];
    }
}
}  // namespace detail

// NOUT (1 or 2) outputs, each a sum of products with few 4 x 4 tiles (at most as many as the output has
// threads) and a longer K, in two barriers. With two outputs each takes half of the CTA's threads. An output's threads split the concatenation of its terms' K
// ranges into G groups (G = its threads / its tiles); each thread forms tiles over its group's part, and the
// partial tiles go to scratch (16 floats per thread of the CTA); then every element of C sums its G partials in
// group order (a fixed order: the result does not depend on the timing). The caller's threads must all call it;
// it ends with the sums written (no barrier after).
template <int NOUT>
__device__ __forceinline__ void mm_ksplit_out(const KOut (&outs)[NOUT], float* scratch) {
    const int per = blockDim.x / NOUT, o = threadIdx.x / per;
#pragma unroll
    for (int oo = 0; oo < NOUT; ++oo)
        if (oo == o) detail::ksplit_partials<NOUT>(outs[oo], oo, scratch);
    __syncthreads();
#pragma unroll
    for (int oo = 0; oo < NOUT; ++oo) {
        const KOut& q = outs[oo];
        const int tiles = (q.M >> 2) * (q.N >> 2), G = max(1, per / tiles);
        const float* part = scratch + (size_t)oo * 16 * per;
        for (int idx = threadIdx.x; idx < q.M * q.N; idx += blockDim.x) {
            float sum = 0.f;
            for (int g = 0; g < G; ++g) sum += part[(size_t)g * q.M * q.N + idx];
            const int m = idx / q.N, n = idx - m * q.N;
            float* d = q.C + m * q.ldc + n;
            *d = q.acc ? *d + q.alpha * sum : q.alpha * sum;
        }
    }
}

}  // namespace smem
}  // namespace dplr
