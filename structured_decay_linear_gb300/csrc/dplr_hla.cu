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
// For dk = dv = 128, passes 2 and 3 run on the tensor cores (tcgen05, bf16 hi + lo operands, three partial
// products, fp32 accumulators in tensor memory: the products keep ~16 significant bits of each operand, against
// the 1e-3 of the output RMS this composition is held to); pass 3 after a small pass that splits each chunk's A_j
// and B_j into bf16 hi/lo operand tiles once. Otherwise both run in fp32 on the CUDA cores (4 x 4 register
// tiles).
#include <cuda_bf16.h>

#include <algorithm>
#include <type_traits>
#include <cstring>

#include "dplr_internal.h"
#include "sm100_ops.cuh"
#include "tc_common.cuh"

namespace dplr {
namespace {

constexpr int HQ = 64;       // queries per CTA of pass 3, tokens per WY block
constexpr int HT = 256;      // threads

struct HlaPlan {
    Plan pl;          // the fp32 two-stage plan at WY blocks of 64 tokens (GDN)
    int L, m, N;      // chunk length, WY blocks per chunk, chunks per head
    int tc;           // pass 3 on the tensor cores
    size_t off_A, off_B, off_T, total;   // L-chunk summaries (L > 64; else the blocks' own maps); operand tiles
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

// ---- pass 3 on the tensor cores (dk = dv = 128)
using namespace tc;

constexpr int HD2 = 128;                          // dk = dv
constexpr uint32_t kOpTile = HD2 * HD2 * 2;       // one bf16 [128][128] operand tile
constexpr int kGT = 192;                          // warps 0-3: U (thread = feature = tensor-memory lane); 4: MMAs; 5: copies
constexpr int kHlaMaxChunks = 256;                // history chunks per query block that fit the step list

// Each chunk's A_j and B_j (fp32 [128][128], row k = the contracted index) as bf16 hi and lo tiles in the
// 128-byte swizzled layout, row k and column n at sw_bf16(k, n, 128): the MN-major A operand of
// X^T = A_j^T U^T and of o^T += B_j^T (w U)^T. Tiles [A hi | A lo | B hi | B lo] per (head, chunk).
__global__ void __launch_bounds__(256)
hla_split_kernel(int N, const float* Acs, const float* Bcs, unsigned char* tiles) {
    const size_t unit = blockIdx.x;   // (head, chunk)
    unsigned char* dst = tiles + unit * 4 * kOpTile;
    for (int e = 0; e < 2; ++e) {
        const float* src = (e == 0 ? Acs : Bcs) + unit * HD2 * HD2;
        unsigned char* th = dst + (2 * e) * kOpTile;
        unsigned char* tl = th + kOpTile;
        for (int i = threadIdx.x; i < HD2 * HD2 / 8; i += blockDim.x) {   // 8 columns of one row per item
            const int k = i >> 4, n = (i & 15) * 8;
            const float4 a = *reinterpret_cast<const float4*>(src + (size_t)k * HD2 + n);
            const float4 b = *reinterpret_cast<const float4*>(src + (size_t)k * HD2 + n + 4);
            uint32_t h[4], l[4];
            split2(a.x, a.y, h[0], l[0]);
            split2(a.z, a.w, h[1], l[1]);
            split2(b.x, b.y, h[2], l[2]);
            split2(b.z, b.w, h[3], l[3]);
            const uint32_t off = sw_bf16(k, n, HD2);
            *reinterpret_cast<uint4*>(th + off) = make_uint4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<uint4*>(tl + off) = make_uint4(l[0], l[1], l[2], l[3]);
        }
    }
}

// ---- pass 2 on the tensor cores (dk = dv = 128): one CTA per (head, L-chunk) walks the chunk's blocks b = b0 + 1 ..
// with the composition of its earlier blocks, A (dk x dk) and B (dk x dv), held in tensor memory:
//     U^T = A^T Q'_b^T,  O^T = B^T Q'_b^T     (M = 128 features, N = 64 tokens, K = 128)
//     A <- P_b A,        B <- P_b B + c_b      (M = N = K = 128, c_b written into B's accumulator first)
// Every product takes three bf16 terms (hi hi + hi lo + lo hi) into fp32 accumulators (tensor-memory columns 0-127 A,
// 128-255 B, 256-319 U^T, 320-383 O^T). P_b and Q'_b are split from fp32 into K-major tiles, row r and column n at
// sw_bf16(r, n, rows); A and B into one pair of tiles at sw_bf16(k, n, 128) (row k the contracted index), which is
// the MN-major B operand of P_b A and the MN-major A operand of A^T Q'^T alike.
struct CSm {
    static constexpr int PH = 0, PL = PH + (int)kOpTile;                  // P_b hi, lo: bf16 [128][128]
    static constexpr int XH = PL + (int)kOpTile, XL = XH + (int)kOpTile;  // A or B: bf16 [128][128]
    static constexpr int QH = XL + (int)kOpTile, QL = QH + HQ * HD2 * 2;  // Q'_b hi, lo: bf16 [64][128]
    static constexpr int BAR = QL + HQ * HD2 * 2;
    static constexpr int TOTAL = BAR + 64;
};
static_assert(CSm::TOTAL <= 227 * 1024, "shared memory budget");
constexpr int kCT = 256;   // threads: warp w takes tensor-memory lanes 32 (w % 4) .. + 31 and column half w / 4

__global__ void __launch_bounds__(kCT, 1)
hla_compose_tc_kernel(Plan pl, int m, int N, const float* Pm, const float* Cm, float* Qm, float* o, float* Aout,
                      float* Bout, int* status) {
    using S = CSm;
    extern __shared__ __align__(1024) unsigned char smem[];
    const uint32_t sb = smem_addr(smem);
    if (sb & 1023u) {
        if (threadIdx.x == 0) atomicExch(status, (int)DPLR_ERR_CUDA);
        return;
    }
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::BAR);
    uint64_t* mb = bars + 0;
    uint64_t* drain = bars + 1;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int row = 32 * (warp & 3) + lane;   // tensor-memory lane: a row of A, B and P_b; a feature of U^T and O^T
    const int hf = warp >> 2;                 // column half
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const int T = pl.T, nb = pl.nb;
    const int c = blockIdx.x % N;
    const size_t bh = blockIdx.x / N;
    const int b0 = c * m, nbc = min(m, nb - b0);
    const long long wl = pl.wait_cycles;
    auto unit = [&](int b) { return bh * (size_t)nb + b; };
    float* Ag = Aout + (bh * (size_t)N + c) * HD2 * HD2;
    float* Bg = Bout + (bh * (size_t)N + c) * HD2 * HD2;
    if (nbc == 1) {   // a chunk of one block is that block
        const float4* P4 = reinterpret_cast<const float4*>(Pm + unit(b0) * HD2 * HD2);
        const float4* C4 = reinterpret_cast<const float4*>(Cm + unit(b0) * HD2 * HD2);
        for (int i = tid; i < HD2 * HD2 / 4; i += kCT) {
            reinterpret_cast<float4*>(Ag)[i] = P4[i];
            reinterpret_cast<float4*>(Bg)[i] = C4[i];
        }
        return;
    }
    constexpr uint32_t TA = 0, TB = 128, TU = 256, TO = 320;
    if (tid == 0) {
        mbar_init(mb, 1);
        mbar_init(drain, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(tmem_holder, 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_holder;

    // fp32 rows [ROWS][128] from global memory into bf16 hi / lo tiles, row r and column n at sw_bf16(r, n, ROWS):
    // every load of the thread is issued before the first store
    auto split_rows = [&](auto rows_tag, const float* src, uint32_t th, uint32_t tl) {
        constexpr int ROWS = decltype(rows_tag)::value, IT = ROWS * 16 / kCT;
        float4 a[IT], b[IT];
#pragma unroll
        for (int it = 0; it < IT; ++it) {
            const int i = tid + it * kCT, r = i >> 4, n = (i & 15) * 8;
            a[it] = *reinterpret_cast<const float4*>(src + (size_t)r * HD2 + n);
            b[it] = *reinterpret_cast<const float4*>(src + (size_t)r * HD2 + n + 4);
        }
#pragma unroll
        for (int it = 0; it < IT; ++it) {
            const int i = tid + it * kCT, r = i >> 4, n = (i & 15) * 8;
            uint32_t h[4], l[4];
            split2(a[it].x, a[it].y, h[0], l[0]);
            split2(a[it].z, a[it].w, h[1], l[1]);
            split2(b[it].x, b[it].y, h[2], l[2]);
            split2(b[it].z, b[it].w, h[3], l[3]);
            const uint32_t off = sw_bf16(r, n, ROWS);
            sts128(th + off, h[0], h[1], h[2], h[3]);
            sts128(tl + off, l[0], l[1], l[2], l[3]);
        }
    };
    using Rows64 = std::integral_constant<int, HQ>;
    using Rows128 = std::integral_constant<int, HD2>;
    // the maps of block b into L2, for the step that reads them next
    auto prefetch_block = [&](int b) {
        if (tid != 0 || b >= b0 + nbc) return;
        const size_t ub = unit(b);
        l2_prefetch(Pm + ub * HD2 * HD2, HD2 * HD2 * 4);
        l2_prefetch(Cm + ub * HD2 * HD2, HD2 * HD2 * 4);
        l2_prefetch(Qm + ub * HQ * HD2, HQ * HD2 * 4);
    };
    // this thread's row and column half of the accumulator at col0 into the A / B operand tiles
    auto tmem_to_x = [&](uint32_t col0) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            float x[32];
            tmem_ld32(tmem + lane_base + col0 + 64 * hf + 32 * q, x);
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t h[4], l[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) split2(x[8 * ch + 2 * e], x[8 * ch + 2 * e + 1], h[e], l[e]);
                const uint32_t off = sw_bf16(row, 64 * hf + 32 * q + 8 * ch, HD2);
                sts128(sb + S::XH + off, h[0], h[1], h[2], h[3]);
                sts128(sb + S::XL + off, l[0], l[1], l[2], l[3]);
            }
        }
    };
    // X^T Q'^T into columns dst, then P_b X into columns acc (onto its content when acc_in), issued by lane 0 of
    // warp 0 and committed to mb
    auto products = [&](uint32_t dst, uint32_t acc, uint32_t acc_in) {
        if (warp != 0) return;
        const uint32_t lead = lane == 0;
        const uint32_t idT = idesc_bf16(128, HQ, true, false), idP = idesc_bf16(128, 128, false, true);
        const uint64_t xh = smem_desc_sw128(sb + S::XH, 16384, 1024), xl = smem_desc_sw128(sb + S::XL, 16384, 1024);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {   // Q'_b: 64-column halves of 64 rows (8 KB)
            const uint32_t ko = (kk >> 2) * 8192 + (kk & 3) * 32;
            const uint64_t qh = smem_desc_sw128(sb + S::QH + ko, 16, 1024), ql = smem_desc_sw128(sb + S::QL + ko, 16, 1024);
            mma_ss_if(tmem + dst, dadd(xh, 2048 * kk), qh, idT, kk > 0 ? 1u : 0u, lead);
            mma_ss_if(tmem + dst, dadd(xh, 2048 * kk), ql, idT, 1u, lead);
            mma_ss_if(tmem + dst, dadd(xl, 2048 * kk), qh, idT, 1u, lead);
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {   // P_b: 64-column halves of 128 rows (16 KB)
            const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
            const uint64_t ph = smem_desc_sw128(sb + S::PH + ko, 16, 1024), pq = smem_desc_sw128(sb + S::PL + ko, 16, 1024);
            mma_ss_if(tmem + acc, ph, dadd(xh, 2048 * kk), idP, (acc_in || kk > 0) ? 1u : 0u, lead);
            mma_ss_if(tmem + acc, ph, dadd(xl, 2048 * kk), idP, 1u, lead);
            mma_ss_if(tmem + acc, pq, dadd(xh, 2048 * kk), idP, 1u, lead);
        }
        commit_if(mb, lead);
    };
    uint32_t phase = 0;
    bool failed = false;
    auto wait_products = [&]() -> bool {   // every thread polls; the CTA takes one decision
        const bool ok = mbar_wait(mb, phase & 1, wl);
        ++phase;
        const bool bad = __syncthreads_or(!ok);
        fence_after_sync();
        return !bad;
    };
    auto operands_ready = [&]() {
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
    };
    for (int k = 1; k < nbc; ++k) {
        const size_t u = unit(b0 + k);
        prefetch_block(b0 + k + 1);
        split_rows(Rows64{}, Qm + u * HQ * HD2, sb + S::QH, sb + S::QL);
        split_rows(Rows128{}, Pm + u * HD2 * HD2, sb + S::PH, sb + S::PL);
        if (k == 1) split_rows(Rows128{}, Pm + unit(b0) * HD2 * HD2, sb + S::XH, sb + S::XL);
        else tmem_to_x(TA);
        operands_ready();
        products(TU, TA, 0u);
        if (!wait_products()) { failed = true; break; }
        // X = B (its tiles free now), and c_b into B's accumulator, this thread's row and column half
        if (k == 1) split_rows(Rows128{}, Cm + unit(b0) * HD2 * HD2, sb + S::XH, sb + S::XL);
        else tmem_to_x(TB);
        {
            const float* cr = Cm + u * HD2 * HD2 + (size_t)row * HD2 + 64 * hf;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                uint32_t r[32];
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    const float4 v = *reinterpret_cast<const float4*>(cr + 32 * q + e);
                    r[e] = __float_as_uint(v.x); r[e + 1] = __float_as_uint(v.y);
                    r[e + 2] = __float_as_uint(v.z); r[e + 3] = __float_as_uint(v.w);
                }
                tmem_st32(tmem + lane_base + TB + 64 * hf + 32 * q, r);
            }
            tmem_wait_st();
        }
        operands_ready();
        products(TO, TB, 1u);
        if (!wait_products()) { failed = true; break; }
        // the block's query rows: U_t over Q'_t in the workspace, O_t added to o (tokens of the sequence)
        {
            const int t0 = (b0 + k) * HQ;
            float x[32];
            tmem_ld32(tmem + lane_base + TU + 32 * hf, x);
            float* qr = Qm + u * HQ * HD2 + row;
#pragma unroll
            for (int e = 0; e < 32; ++e) qr[(size_t)(32 * hf + e) * HD2] = x[e];
            tmem_ld32(tmem + lane_base + TO + 32 * hf, x);
            float* orow = o + (bh * (size_t)T + t0 + 32 * hf) * HD2 + row;
            const int nv = min(32, T - t0 - 32 * hf);   // tokens of the sequence in this half
            float ov[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = e < nv ? orow[(size_t)e * HD2] : 0.f;   // every load, then the stores
#pragma unroll
            for (int e = 0; e < 32; ++e)
                if (e < nv) orow[(size_t)e * HD2] = ov[e] + x[e];
        }
    }
    if (!failed) {   // the chunk's summary, A then B
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
            float* dst = (e2 ? Bg : Ag) + (size_t)row * HD2 + 64 * hf;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                float x[32];
                tmem_ld32(tmem + lane_base + (e2 ? TB : TA) + 64 * hf + 32 * q, x);
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                    *reinterpret_cast<float4*>(dst + 32 * q + e) = make_float4(x[e], x[e + 1], x[e + 2], x[e + 3]);
            }
        }
    } else if (tid == 0) {   // no product may outlive the tensor memory
        atomicExch(status, (int)DPLR_ERR_TIMEOUT);
        mma_commit(drain);
        mbar_wait(drain, 0, 400000000LL);
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

struct GSm {
    static constexpr int OPS = 0;                          // the step's A_j^T hi, lo, B_j^T hi, lo
    static constexpr int UTB = HD2 * HQ * 2;               // bf16 [128 k][64 q] MN-major B operand
    // U^T hi, lo, then (w U)^T hi, lo in two buffers by step parity: the o^T products of a step may still read
    // theirs while the next step's tiles are written (X^T's completion, which the state warps wait for, implies
    // that of the previous step's o^T products: one thread issues them all, in order)
    static constexpr int UT = OPS + 4 * (int)kOpTile;
    static constexpr int WB = UT + 6 * UTB;                // the step's gates [64]
    static constexpr int FLAGS = WB + HQ * 4;              // per history chunk, per query warp: some gate >= theta
    static constexpr int LIST = FLAGS + 2 * kHlaMaxChunks; // the history chunks that are composed, newest first
    static constexpr int BAR = LIST + kHlaMaxChunks * 4;
    static constexpr int TOTAL = BAR + 128;
};
static_assert(GSm::TOTAL <= 227 * 1024, "shared memory budget");

struct GatedArgs {
    const float* Um; const float* W; const unsigned char* tiles; float* o; int* status;
};

// One CTA per (head, 64 queries of one chunk c). The chunks j < c with some gate >= theta among the CTA's
// queries are walked newest first; per chunk (a step) the issuer runs X^T = A_j^T U^T and o^T += B_j^T (w U)^T,
// both M = 128 (the feature), N = 64 (the query), K = 128, in three terms (hi hi + lo hi + hi lo), while the
// state warps keep U^T in fp32 registers (thread = feature) and update it, U <- U + w (X - U), once X^T is done.
// o^T accumulates in tensor memory over the steps and is added to o (the chunk-local part of pass 1/2) at the end.
__global__ void __launch_bounds__(kGT, 1)
hla_gated_tc_kernel(Plan pl, int L, int N, float theta, GatedArgs args) {
    using S = GSm;
    extern __shared__ __align__(1024) unsigned char smem[];
    const uint32_t sb = smem_addr(smem);
    if (sb & 1023u) {
        if (threadIdx.x == 0) atomicExch(args.status, (int)DPLR_ERR_CUDA);
        return;
    }
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::BAR);
    uint64_t* full = bars + 0;     // the step's operand tiles landed
    uint64_t* freed = bars + 1;    // the step's products are done with the operand tiles
    uint64_t* ready = bars + 2;    // the step's U^T and (w U)^T tiles written (4 arrivals, one per state warp)
    uint64_t* mX = bars + 3;       // the step's X^T is complete
    uint64_t* drain = bars + 4;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 5);
    int* nsteps = reinterpret_cast<int*>(bars + 6);
    int* list = reinterpret_cast<int*>(smem + S::LIST);
    float* wb = reinterpret_cast<float*>(smem + S::WB);
    unsigned char* flags = smem + S::FLAGS;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = pl.T, nb = pl.nb;
    const int qb = blockIdx.x % nb;
    const size_t bh = blockIdx.x / nb;
    const int t0 = qb * HQ, c = t0 / L;
    const long long wl = pl.wait_cycles;
    auto gate = [&](int q, int l) -> float {   // w_ql, with gates below theta (and absent queries) as zero
        if (t0 + q >= T) return 0.f;
        const float x = args.W[(bh * (size_t)T + t0 + q) * N + l];
        return x >= theta ? x : 0.f;
    };

    // ---- the steps: history chunks, newest first, with some gate >= theta among the 64 queries
    if (warp < 2) {
        const int q = tid;
        for (int l = c - 1; l >= 0; --l) {
            const unsigned any = __ballot_sync(0xffffffffu, gate(q, l) != 0.f);
            if (lane == 0) flags[warp * kHlaMaxChunks + (c - 1 - l)] = any != 0u;
        }
    }
    __syncthreads();
    if (tid == 0) {
        int n = 0;
        for (int s = 0; s < c; ++s)
            if (flags[s] | flags[kHlaMaxChunks + s]) list[n++] = c - 1 - s;
        *nsteps = n;
        mbar_init(full, 1);
        mbar_init(freed, 1);
        mbar_init(ready, 4);
        mbar_init(mX, 1);
        mbar_init(drain, 1);
        mbar_fence_init();
    }
    __syncthreads();
    const int ns = *nsteps;
    if (ns == 0) return;   // every query's history is gated off: o keeps the chunk-local part
    if (warp == 0) tmem_alloc(tmem_holder, 128);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_holder;   // columns 0-63: X^T; 64-127: o^T
    bool failed = false;

    if (warp == 5) {
        // ---- copies of each step's operand tiles, once the previous step's products are done with them
        int last = -1;
        for (int st = 0; st < ns && lane == 0; ++st) {
            if (st >= 1 && !mbar_wait(freed, (st - 1) & 1, wl)) { failed = true; break; }
            const unsigned char* src = args.tiles + (bh * (size_t)N + list[st]) * 4 * kOpTile;
            mbar_expect_tx(full, 4 * kOpTile);
            for (int e = 0; e < 4; ++e) bulk_g2s(smem + S::OPS + e * kOpTile, src + e * kOpTile, kOpTile, full);
            if (st + 1 < ns) {
                const unsigned char* nx = args.tiles + (bh * (size_t)N + list[st + 1]) * 4 * kOpTile;
                for (int e = 0; e < 4; ++e)
                    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(reinterpret_cast<uint64_t>(nx + e * kOpTile)),
                                 "r"(kOpTile) : "memory");
            }
            last = st;
        }
        if (failed) {   // (lane 0) no copy may land after the CTA has exited
            atomicExch(args.status, (int)DPLR_ERR_TIMEOUT);
            if (last >= 0) mbar_wait(full, last & 1, 400000000LL);
        }
        __syncwarp();
    } else if (warp == 4) {
        // ---- the products of each step, issued by lane 0
        const uint32_t id = idesc_bf16(128, HQ, true, true);
        for (int st = 0; st < ns && lane == 0; ++st) {
            if (!mbar_wait(ready, st & 1, wl) || !mbar_wait(full, st & 1, wl)) { failed = true; break; }
            fence_after_sync();
            // (A operand: 64-column halves 16 KB apart, K = 16 rows per slice; B: one 64-query atom per row)
            const uint64_t aH = smem_desc_sw128(sb + S::OPS, 16384, 1024), aL = dadd(aH, kOpTile);
            const uint64_t bH = aH + ((uint64_t)(2 * kOpTile) >> 4), bL = dadd(bH, kOpTile);
            const uint64_t uH = smem_desc_sw128(sb + S::UT, 16384, 1024), uL = dadd(uH, S::UTB);
            const uint64_t wH = dadd(uH, (2 + 2 * (st & 1)) * S::UTB), wL = dadd(wH, S::UTB);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {   // X^T = A^T U^T
                const uint32_t o = kk * 2048;
                mma_bf16(tmem, dadd(aH, o), dadd(uH, o), id, kk > 0);
                mma_bf16(tmem, dadd(aL, o), dadd(uH, o), id, 1u);
                mma_bf16(tmem, dadd(aH, o), dadd(uL, o), id, 1u);
            }
            mma_commit(mX);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {   // o^T += B^T (w U)^T
                const uint32_t o = kk * 2048;
                mma_bf16(tmem + 64, dadd(bH, o), dadd(wH, o), id, (st > 0 || kk > 0) ? 1u : 0u);
                mma_bf16(tmem + 64, dadd(bL, o), dadd(wH, o), id, 1u);
                mma_bf16(tmem + 64, dadd(bH, o), dadd(wL, o), id, 1u);
            }
            mma_commit(freed);
        }
        if (failed) {   // (lane 0) no product may outlive the tensor memory
            atomicExch(args.status, (int)DPLR_ERR_TIMEOUT);
            mma_commit(drain);
            mbar_wait(drain, 0, 400000000LL);
        }
        __syncwarp();
    } else {
        // ---- U^T, row d = this thread (the feature), 64 queries, in fp32 registers
        const int d = tid;
        const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
        float u[HQ];
        const float* U0 = args.Um + (bh * (size_t)nb + qb) * HQ * HD2;
#pragma unroll
        for (int q = 0; q < HQ; ++q) u[q] = U0[(size_t)q * HD2 + d];
        // a wait of the four state warps: each warp's lane 0 polls, and the group takes one decision
        auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
            bool ok = true;
            if (lane == 0) ok = mbar_wait(bar, parity, wl);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            return !named_sync_or(1, 128, !ok);
        };
        for (int st = 0; st < ns; ++st) {
            // the step's gates, then the U^T and (w U)^T tiles: row d, query q at sw_bf16(d, q, 128)
            if (tid < HQ) wb[tid] = gate(tid, list[st]);
            named_sync(1, 128);
#pragma unroll
            for (int ch = 0; ch < HQ / 8; ++ch) {
                uint32_t h[4], l[4], wh[4], wlo[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int q = 8 * ch + 2 * e;
                    split2(u[q], u[q + 1], h[e], l[e]);
                    split2(wb[q] * u[q], wb[q + 1] * u[q + 1], wh[e], wlo[e]);
                }
                const uint32_t off = sw_bf16(d, 8 * ch, HD2), wbuf = sb + S::UT + (2 + 2 * (st & 1)) * S::UTB;
                sts128(sb + S::UT + off, h[0], h[1], h[2], h[3]);
                sts128(sb + S::UT + S::UTB + off, l[0], l[1], l[2], l[3]);
                sts128(wbuf + off, wh[0], wh[1], wh[2], wh[3]);
                sts128(wbuf + S::UTB + off, wlo[0], wlo[1], wlo[2], wlo[3]);
            }
            fence_async_smem();
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(ready);
            // X^T of this step, then U <- U + w (X - U)
            if (!wait_all(mX, st & 1)) { failed = true; break; }
            fence_after_sync();
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float x[32];
                tmem_ld32(tmem + lane_base + 32 * hf, x);
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int q = 32 * hf + e;
                    u[q] = fmaf(wb[q], x[e] - u[q], u[q]);
                }
            }
            fence_before_sync();
            named_sync(1, 128);   // every state warp has read the gates and X^T (the next step rewrites both)
        }
        // o += o^T once the last step's products are done
        if (!failed && !wait_all(freed, (ns - 1) & 1)) failed = true;
        if (!failed) {
            fence_after_sync();
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float x[32];
                tmem_ld32(tmem + lane_base + 64 + 32 * hf, x);
                float* orow = args.o + (bh * (size_t)T + t0 + 32 * hf) * HD2 + d;
                const int nv = min(32, T - t0 - 32 * hf);   // queries of the sequence in this half
                float ov[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) ov[e] = e < nv ? orow[(size_t)e * HD2] : 0.f;   // every load, then the stores
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    if (e < nv) orow[(size_t)e * HD2] = ov[e] + x[e];
            }
        }
        if (failed && lane == 0) atomicExch(args.status, (int)DPLR_ERR_TIMEOUT);
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
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
    hp->tc = (p.dk == HD2 && p.dv == HD2 && hp->N <= kHlaMaxChunks) ? 1 : 0;
    hp->off_T = off;
    if (hp->tc) off = hround(off + (size_t)p.BH * hp->N * 4 * kOpTile);
    hp->total = off;
    p.ws_bytes = off;
    hp->pl = p;
    return DPLR_OK;
}

std::atomic<uint64_t> g_hla_smem[4] = {{0}, {0}, {0}, {0}};

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
    if (cudaMemsetAsync(ws, 0, kHAlign, s) != cudaSuccess) return DPLR_ERR_CUDA;   // the status word
    ChunkMapArgs ma;
    ma.q = q; ma.k = k; ma.v = v; ma.decay = g; ma.beta = beta;
    ma.A = nullptr; ma.Bm = nullptr; ma.K = nullptr; ma.V = nullptr; ma.o = o;
    ma.Pm = reinterpret_cast<float*>(ws + pl.off_P);
    ma.Cm = reinterpret_cast<float*>(ws + pl.off_c);
    ma.Qm = reinterpret_cast<float*>(ws + pl.off_Q);
    if (launch_chunk_maps(pl, ma, s) != cudaSuccess) return DPLR_ERR_CUDA;   // pass 1 (o <- O_t)
    float* Acs = reinterpret_cast<float*>(ws + hp.off_A);
    float* Bcs = reinterpret_cast<float*>(ws + hp.off_B);
    if (hp.m > 1 && pl.dk == HD2 && pl.dv == HD2) {   // pass 2 on the tensor cores
        if (set_smem_limit_once(reinterpret_cast<const void*>(hla_compose_tc_kernel), CSm::TOTAL, g_hla_smem[3]) != cudaSuccess)
            return DPLR_ERR_CUDA;
        hla_compose_tc_kernel<<<(unsigned)((size_t)pl.BH * hp.N), kCT, CSm::TOTAL, s>>>(pl, hp.m, hp.N, ma.Pm, ma.Cm, ma.Qm, o,
                                                                                       Acs, Bcs, reinterpret_cast<int*>(ws));
        if (cudaGetLastError() != cudaSuccess) return DPLR_ERR_CUDA;
    } else if (hp.m > 1) {   // pass 2 on the CUDA cores
        const size_t smem = sizeof(float) * (size_t)(2 * pl.dk * pl.dk + pl.dk * pl.dv + HQ * pl.dk);
        if (set_smem_limit_once(reinterpret_cast<const void*>(hla_compose_kernel), 227 * 1024, g_hla_smem[0]) != cudaSuccess)
            return DPLR_ERR_CUDA;
        hla_compose_kernel<<<(unsigned)((size_t)pl.BH * hp.N), HT, smem, s>>>(pl, hp.m, hp.N, ma.Pm, ma.Cm, ma.Qm, o, Acs, Bcs);
        if (cudaGetLastError() != cudaSuccess) return DPLR_ERR_CUDA;
    }
    if (hp.tc) {   // pass 3 on the tensor cores: the chunks' operand tiles, then the gated composition
        unsigned char* tiles = reinterpret_cast<unsigned char*>(ws + hp.off_T);
        hla_split_kernel<<<(unsigned)((size_t)pl.BH * hp.N), 256, 0, s>>>(hp.N, Acs, Bcs, tiles);
        if (cudaGetLastError() != cudaSuccess) return DPLR_ERR_CUDA;
        if (set_smem_limit_once(reinterpret_cast<const void*>(hla_gated_tc_kernel), GSm::TOTAL, g_hla_smem[2]) != cudaSuccess)
            return DPLR_ERR_CUDA;
        GatedArgs ga;
        ga.Um = ma.Qm; ga.W = W; ga.tiles = tiles; ga.o = o; ga.status = reinterpret_cast<int*>(ws);
        hla_gated_tc_kernel<<<(unsigned)((size_t)pl.BH * pl.nb), kGT, GSm::TOTAL, s>>>(pl, hp.L, hp.N, theta, ga);
        if (cudaGetLastError() != cudaSuccess) return DPLR_ERR_CUDA;
    } else {   // pass 3 on the CUDA cores
        const size_t smem = sizeof(float) * (size_t)(HQ * pl.dk + pl.dk * pl.dk + pl.dk * pl.dv + HQ);
        if (set_smem_limit_once(reinterpret_cast<const void*>(hla_gated_kernel), 227 * 1024, g_hla_smem[1]) != cudaSuccess)
            return DPLR_ERR_CUDA;
        hla_gated_kernel<<<(unsigned)((size_t)pl.BH * pl.nb), HT, smem, s>>>(pl, hp.L, hp.N, theta, ma.Qm, Acs, Bcs, W, o);
        if (cudaGetLastError() != cudaSuccess) return DPLR_ERR_CUDA;
    }
    return DPLR_OK;
}

extern "C" const char* dplr_hla_path(const dplr_desc* desc, int L) {
    HlaPlan hp;
    if (make_hla_plan(desc, L, &hp) != DPLR_OK) return "";
    return hp.tc ? "hla_gated_tcgen05" : "hla_gated_fp32";
}
