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
//   1. the maps of the WY blocks of 64 tokens: P_b, c_b, the readout rows Q'_t and O_t;
//   2. (L > 64) the L-chunk summaries composed from their blocks, A = P_{m-1} .. P_0, B likewise, and each
//      query's row U_t = Q'_t (the composition of its chunk's earlier blocks), its output O_t updated;
//   3. per 64 queries of one chunk, the history chunks newest first: two products per chunk, U A_j and U B_j,
//      with the gates applied per query; a chunk whose gates are all zero for the 64 queries is skipped.
// For dk = dv = 128, passes 2 and 3 run on the tensor cores (tcgen05, bf16 hi + lo operands, three partial
// products, fp32 accumulators in tensor memory: the products keep ~16 significant bits of each operand, against
// the 1e-3 of the output RMS this composition is held to); pass 3 after a small pass that splits each chunk's A_j
// and B_j into bf16 hi/lo operand tiles once. Pass 1 runs there too when the inputs are bf16. Otherwise the
// passes run in fp32 on the CUDA cores (4 x 4 register tiles).
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

// ---- pass 1 on the tensor cores (Gated DeltaNet, bf16, dk = dv = 128): the exact maps of one 64-token block,
// the same quantities as the fp32 chunk-map kernel. With G_t the inclusive cumulative log-gate, a = G_C / 2,
// eb_t = e^{G_t - a}, w_t = e^{a - G_t} beta_t and D = [K; Q] K^T (raw bf16 k, q: exact):
//     L_ts = e^{G_t - G_s} beta_s (k_t . k_s)  (s < t),   QA_ts = e^{G_t - G_s} beta_s (q_t . k_s)  (s <= t)
//     M = (I + L)^{-1},  Y = M Diag(eb) K,  U = -M V
//     P = e^{G_C} (I - K^T Diag(w) Y),  c = -e^{G_C - a} K^T Diag(w) U
//     Q'_t = e^{G_t} q_t - e^{a} (QA Y)_t,  O = -QA U
// D on the tensor cores in one term; L and QA scaled in fp32; M by the blocked fp32 inverse (three-term tf32
// merges); then Y^T = K^T (M Diag(eb))^T and U^T = V^T (-M)^T, P and c as K^T [Diag(w) Y] and K^T [Diag(w) U],
// and (Q A Y)^T, (QA U)^T, each with the rounded operand in bf16 hi + lo (the raw k and v are exact in bf16).
// Tensor-memory columns: D, then (QA Y)^T (0-63); Y^T (64-127); U^T (128-191); P (192-319); c (320-447);
// (QA U)^T (448-511).
struct BSm {
    static constexpr int KQ = 0;                  // [k 0-63 | q 0-63 | k 64-127 | q 64-127] features, 64 tokens each
    static constexpr int VT = KQ + 32768;         // v: two halves of 64 features (8 KB each)
    static constexpr int X = VT + 16384;          // fp32 [64][kLdX]: L, then M
    static constexpr int QAF = X + 64 * kLdX * 4; // fp32 [64][kLdX]: QA
    static constexpr int MB = QAF + 64 * kLdX * 4;   // M Diag(eb): hi, lo [64][64] (8 KB each)
    static constexpr int MN = MB + 16384;         // -M: hi, lo
    static constexpr int QT = MN + 16384;         // QA: hi, lo [64 t][64 s]
    static constexpr int YW = QT + 16384;         // Diag(w) Y, then Y, as [128 k][64 t]: hi, lo (16 KB each)
    static constexpr int UW = YW + 32768;         // Diag(w) U, then -U, as [128 n][64 t]: hi, lo
    static constexpr int VEC = UW + 32768;        // G [64], eb [64], w [64], e^{G_C}, e^{G_C - a}, e^a
    static constexpr int BAR = VEC + 1024;
    static constexpr int TOTAL = BAR + 64;
};
static_assert(BSm::TOTAL <= 227 * 1024, "shared memory budget");
static_assert(BSm::MB % 1024 == 0 && BSm::YW % 1024 == 0 && BSm::UW % 1024 == 0 && BSm::QT % 1024 == 0,
              "swizzled tiles are 1024-byte aligned");
constexpr int kBT = 256;   // threads: warp w takes tensor-memory lanes 32 (w % 4) .. + 31 and column half w / 4

__global__ void __launch_bounds__(kBT, 1)
hla_block_maps_tc_kernel(Plan pl, const __nv_bfloat16* q, const __nv_bfloat16* k, const __nv_bfloat16* v,
                         const float* g, const float* beta, float* Pm, float* Cm, float* Qm, float* o, int* status) {
    using S = BSm;
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
    float* X = reinterpret_cast<float*>(smem + S::X);
    float* QAf = reinterpret_cast<float*>(smem + S::QAF);
    float* vG = reinterpret_cast<float*>(smem + S::VEC);
    float* veb = vG + 64;
    float* vw = vG + 128;
    float* vsc = vG + 192;   // e^{G_C}, e^{G_C - a}, e^a
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int row = 32 * (warp & 3) + lane, hf = warp >> 2;
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const int T = pl.T, nb = pl.nb;
    const long long total = (long long)pl.BH * nb;
    const long long wl = pl.wait_cycles;
    constexpr uint32_t TD = 0, TY = 64, TU = 128, TP = 192, TC = 320, TO = 448;

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
    uint32_t phase = 0;
    bool failed = false;
    auto wait_products = [&]() -> bool {
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
    const uint32_t lead = (warp == 0 && lane == 0) ? 1u : 0u;
    // Kt: K^T (or V^T) as the MN-major A operand over the tokens; halves of 64 features `half` bytes apart
    auto mn_desc = [&](uint32_t base, uint32_t half) { return smem_desc_sw128(sb + base, half, 1024); };

  // persistent: CTA b takes the blocks b, b + gridDim.x, ... (the next one's rows asked for in L2 first)
  for (long long ux = blockIdx.x; ux < total && !failed; ux += gridDim.x) {
    const int blk = static_cast<int>(ux % nb);
    const size_t bh = static_cast<size_t>(ux / nb);
    const int t0 = blk * HQ, valid = min(HQ, T - t0);
    const size_t tok0 = bh * (size_t)T + t0;
    const size_t unit = bh * (size_t)nb + blk;
    if (tid == 0 && ux + gridDim.x < total) {
        const long long nx = ux + gridDim.x;
        const int nt0 = static_cast<int>(nx % nb) * HQ, nvalid = min(HQ, T - nt0);
        const size_t ntok = (size_t)(nx / nb) * T + nt0;
        for (const __nv_bfloat16* src : {k, q, v})
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                         :: "l"(reinterpret_cast<uint64_t>(src + ntok * HD2)), "r"((uint32_t)(nvalid * HD2 * 2)) : "memory");
    }
    // ---- k, q, v of the block (zeros past the sequence), in the 128-byte swizzled layout
    for (int i = tid; i < HQ * 16; i += kBT) {
        const int t = i >> 4, cb = i & 15;
        uint4 zk = make_uint4(0, 0, 0, 0), zq = zk, zv = zk;
        if (t < valid) {
            const size_t gix = (tok0 + t) * HD2 + 8 * cb;
            zk = *reinterpret_cast<const uint4*>(k + gix);
            zq = *reinterpret_cast<const uint4*>(q + gix);
            zv = *reinterpret_cast<const uint4*>(v + gix);
        }
        const uint32_t off = swz(t, cb & 7);
        sts128(sb + S::KQ + (cb >> 3) * 16384 + off, zk.x, zk.y, zk.z, zk.w);
        sts128(sb + S::KQ + (cb >> 3) * 16384 + 8192 + off, zq.x, zq.y, zq.z, zq.w);
        sts128(sb + S::VT + (cb >> 3) * 8192 + off, zv.x, zv.y, zv.z, zv.w);
    }
    // ---- the gates (warp 0: tokens 2 lane, 2 lane + 1; identity past the sequence)
    if (warp == 0) {
        const int ta = 2 * lane, tb = ta + 1;
        const float g0 = ta < valid ? g[tok0 + ta] : 0.f, g1 = tb < valid ? g[tok0 + tb] : 0.f;
        const float b0 = ta < valid ? beta[tok0 + ta] : 0.f, b1 = tb < valid ? beta[tok0 + tb] : 0.f;
        float sum = g0 + g1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, sum, off);
            if (lane >= off) sum += y;
        }
        const float GC = __shfl_sync(0xffffffffu, sum, 31), G1 = sum, G0 = sum - g1, a = 0.5f * GC;
        vG[ta] = G0; vG[tb] = G1;
        veb[ta] = __expf(G0 - a); veb[tb] = __expf(G1 - a);
        vw[ta] = __expf(a - G0) * b0; vw[tb] = __expf(a - G1) * b1;
        if (lane == 0) {
            vsc[0] = __expf(GC);
            vsc[1] = __expf(GC - a);
            vsc[2] = __expf(a);
        }
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();

    // ---- D = [K; Q] K^T
    if (warp == 0) {
        const uint32_t id = idesc_bf16(128, 64, false, false);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
            const uint64_t ad = smem_desc_sw128(sb + S::KQ + ko, 16, 1024);
            mma_ss_if(tmem + TD, ad, ad, id, kk > 0 ? 1u : 0u, lead);   // B: the first 64 rows (k) of the same tile
        }
        commit_if(mb, lead);
    }
    if (!wait_products()) failed = true;

    if (!failed) {
        // ---- L (rows 0-63, lanes of k) and QA (rows 64-127, lanes of q), this thread's half of the columns s
        float x[32];
        tmem_ld32(tmem + lane_base + TD + 32 * hf, x);
        const int t = row & 63;
        const float Gt = vG[t];
        if (row < 64) {
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
                const int s0 = 32 * hf + e;
                float4 y;
                y.x = s0 + 0 < t ? __expf(Gt - vG[s0 + 0]) * vw[s0 + 0] * veb[s0 + 0] * x[e + 0] : 0.f;
                y.y = s0 + 1 < t ? __expf(Gt - vG[s0 + 1]) * vw[s0 + 1] * veb[s0 + 1] * x[e + 1] : 0.f;
                y.z = s0 + 2 < t ? __expf(Gt - vG[s0 + 2]) * vw[s0 + 2] * veb[s0 + 2] * x[e + 2] : 0.f;
                y.w = s0 + 3 < t ? __expf(Gt - vG[s0 + 3]) * vw[s0 + 3] * veb[s0 + 3] * x[e + 3] : 0.f;
                *reinterpret_cast<float4*>(X + t * kLdX + s0) = y;
            }
        } else {
            float qa[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int s0 = 32 * hf + e;
                qa[e] = s0 <= t ? __expf(Gt - vG[s0]) * vw[s0] * veb[s0] * x[e] : 0.f;
            }
#pragma unroll
            for (int e = 0; e < 32; e += 4)
                *reinterpret_cast<float4*>(QAf + t * kLdX + 32 * hf + e) = make_float4(qa[e], qa[e + 1], qa[e + 2], qa[e + 3]);
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {   // QA as the K-major B operand [t][s]: hi, lo
                uint32_t h[4], l[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) split2(qa[8 * c8 + 2 * e], qa[8 * c8 + 2 * e + 1], h[e], l[e]);
                const uint32_t off = swz(t, 4 * hf + c8);
                sts128(sb + S::QT + off, h[0], h[1], h[2], h[3]);
                sts128(sb + S::QT + 8192 + off, l[0], l[1], l[2], l[3]);
            }
        }
        __syncthreads();
        // ---- M = (I + L)^{-1} in place
        inv64_inplace<3>(X, tid, 1);
        __syncthreads();
        // ---- M Diag(eb) and -M as K-major B operands [s][u]: hi, lo
        for (int i = tid; i < 64 * 8; i += kBT) {
            const int r = i >> 3, c8 = i & 7;
            const float4 m0 = *reinterpret_cast<const float4*>(X + r * kLdX + 8 * c8);
            const float4 m1 = *reinterpret_cast<const float4*>(X + r * kLdX + 8 * c8 + 4);
            const float mv[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
            uint32_t bh_[4], bl_[4], nh[4], nl[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int u = 8 * c8 + 2 * e;
                split2(mv[2 * e] * veb[u], mv[2 * e + 1] * veb[u + 1], bh_[e], bl_[e]);
                split2(-mv[2 * e], -mv[2 * e + 1], nh[e], nl[e]);
            }
            const uint32_t off = swz(r, c8);
            sts128(sb + S::MB + off, bh_[0], bh_[1], bh_[2], bh_[3]);
            sts128(sb + S::MB + 8192 + off, bl_[0], bl_[1], bl_[2], bl_[3]);
            sts128(sb + S::MN + off, nh[0], nh[1], nh[2], nh[3]);
            sts128(sb + S::MN + 8192 + off, nl[0], nl[1], nl[2], nl[3]);
        }
        operands_ready();
        // ---- Y^T = K^T (M Diag(eb))^T and U^T = V^T (-M)^T
        if (warp == 0) {
            const uint32_t id = idesc_bf16(128, 64, true, false);
            const uint64_t ak = mn_desc(S::KQ, 16384), av = mn_desc(S::VT, 8192);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t bh_ = smem_desc_sw128(sb + S::MB + 32 * kk, 16, 1024), bl_ = dadd(bh_, 8192);
                const uint64_t nh = smem_desc_sw128(sb + S::MN + 32 * kk, 16, 1024), nl = dadd(nh, 8192);
                mma_ss_if(tmem + TY, dadd(ak, 2048 * kk), bh_, id, kk > 0 ? 1u : 0u, lead);
                mma_ss_if(tmem + TY, dadd(ak, 2048 * kk), bl_, id, 1u, lead);
                mma_ss_if(tmem + TU, dadd(av, 2048 * kk), nh, id, kk > 0 ? 1u : 0u, lead);
                mma_ss_if(tmem + TU, dadd(av, 2048 * kk), nl, id, 1u, lead);
            }
            commit_if(mb, lead);
        }
        if (!wait_products()) failed = true;
    }
    // this thread's row of Y^T (or U^T), tokens 32 hf .., times f_t, as bf16 hi / lo at row `row` of the tiles
    auto rows_out = [&](uint32_t col, uint32_t tile, const float* f, float sgn) {
        float x[32];
        tmem_ld32(tmem + lane_base + col + 32 * hf, x);
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {
            uint32_t h[4], l[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int t = 32 * hf + 8 * c8 + 2 * e;
                const float f0 = f ? f[t] : 1.f, f1 = f ? f[t + 1] : 1.f;
                split2(sgn * f0 * x[8 * c8 + 2 * e], sgn * f1 * x[8 * c8 + 2 * e + 1], h[e], l[e]);
            }
            const uint32_t off = swz(row, 4 * hf + c8);
            sts128(sb + tile + off, h[0], h[1], h[2], h[3]);
            sts128(sb + tile + 16384 + off, l[0], l[1], l[2], l[3]);
        }
    };
    if (!failed) {
        rows_out(TY, S::YW, vw, 1.f);   // Diag(w) Y, row k
        rows_out(TU, S::UW, vw, 1.f);   // Diag(w) U, row n
        operands_ready();
        // ---- K^T [Diag(w) Y] and K^T [Diag(w) U]
        if (warp == 0) {
            const uint32_t id = idesc_bf16(128, 128, true, false);
            const uint64_t ak = mn_desc(S::KQ, 16384);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t yh = smem_desc_sw128(sb + S::YW + 32 * kk, 16, 1024), yl = dadd(yh, 16384);
                const uint64_t uh = smem_desc_sw128(sb + S::UW + 32 * kk, 16, 1024), ul = dadd(uh, 16384);
                mma_ss_if(tmem + TP, dadd(ak, 2048 * kk), yh, id, kk > 0 ? 1u : 0u, lead);
                mma_ss_if(tmem + TP, dadd(ak, 2048 * kk), yl, id, 1u, lead);
                mma_ss_if(tmem + TC, dadd(ak, 2048 * kk), uh, id, kk > 0 ? 1u : 0u, lead);
                mma_ss_if(tmem + TC, dadd(ak, 2048 * kk), ul, id, 1u, lead);
            }
            commit_if(mb, lead);
        }
        if (!wait_products()) failed = true;
    }
    if (!failed) {
        rows_out(TY, S::YW, nullptr, 1.f);    // Y, row k (the A operand of (QA Y)^T)
        rows_out(TU, S::UW, nullptr, -1.f);   // -U, row n
        operands_ready();
        // ---- (QA Y)^T = Y^T QA^T and O^T = (-U)^T QA^T
        if (warp == 0) {
            const uint32_t id = idesc_bf16(128, 64, false, false);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t yh = smem_desc_sw128(sb + S::YW + 32 * kk, 16, 1024), yl = dadd(yh, 16384);
                const uint64_t uh = smem_desc_sw128(sb + S::UW + 32 * kk, 16, 1024), ul = dadd(uh, 16384);
                const uint64_t qh = smem_desc_sw128(sb + S::QT + 32 * kk, 16, 1024), ql = dadd(qh, 8192);
                mma_ss_if(tmem + TD, yh, qh, id, kk > 0 ? 1u : 0u, lead);
                mma_ss_if(tmem + TD, yh, ql, id, 1u, lead);
                mma_ss_if(tmem + TD, yl, qh, id, 1u, lead);
                mma_ss_if(tmem + TO, uh, qh, id, kk > 0 ? 1u : 0u, lead);
                mma_ss_if(tmem + TO, uh, ql, id, 1u, lead);
                mma_ss_if(tmem + TO, ul, qh, id, 1u, lead);
            }
            commit_if(mb, lead);
        }
        if (!wait_products()) failed = true;
    }
    if (!failed) {
        // ---- the maps: P and c rows (lane = row i, this thread's half of the columns), Q' and O columns
        const float eGC = vsc[0], eGCa = vsc[1], ea = vsc[2];
        float* Pr = Pm + unit * HD2 * HD2 + (size_t)row * HD2 + 64 * hf;
        float* Cr = Cm + unit * HD2 * HD2 + (size_t)row * HD2 + 64 * hf;
#pragma unroll
        for (int qq = 0; qq < 2; ++qq) {
            float x[32];
            tmem_ld32(tmem + lane_base + TP + 64 * hf + 32 * qq, x);
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
                const int c0 = 64 * hf + 32 * qq + e;
                float4 y;
                y.x = eGC * ((c0 + 0 == row ? 1.f : 0.f) - x[e + 0]);
                y.y = eGC * ((c0 + 1 == row ? 1.f : 0.f) - x[e + 1]);
                y.z = eGC * ((c0 + 2 == row ? 1.f : 0.f) - x[e + 2]);
                y.w = eGC * ((c0 + 3 == row ? 1.f : 0.f) - x[e + 3]);
                *reinterpret_cast<float4*>(Pr + 32 * qq + e) = y;
            }
            tmem_ld32(tmem + lane_base + TC + 64 * hf + 32 * qq, x);
#pragma unroll
            for (int e = 0; e < 32; e += 4)
                *reinterpret_cast<float4*>(Cr + 32 * qq + e) =
                    make_float4(-eGCa * x[e], -eGCa * x[e + 1], -eGCa * x[e + 2], -eGCa * x[e + 3]);
        }
        {   // Q'[t][k] = e^{G_t} q_t[k] - e^a (QA Y)[t][k] (lane = k), O[t][n] (lane = n): tokens 32 hf ..
            float x[32];
            tmem_ld32(tmem + lane_base + TD + 32 * hf, x);
            float* Qc = Qm + unit * HQ * HD2 + row;
            const uint32_t qrow = sb + S::KQ + (row >> 6) * 16384 + 8192 + ((row & 7) << 1);
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int t = 32 * hf + e;
                const float qt = lds_bf16(qrow + swz(t, (row & 63) >> 3));
                Qc[(size_t)t * HD2] = __expf(vG[t]) * qt - ea * x[e];
            }
            tmem_ld32(tmem + lane_base + TO + 32 * hf, x);
            float* oc = o + (tok0 + 32 * hf) * HD2 + row;
            const int nv = min(32, valid - 32 * hf);
#pragma unroll
            for (int e = 0; e < 32; ++e)
                if (e < nv) oc[(size_t)e * HD2] = x[e];
        }
    }
    fence_before_sync();
    __syncthreads();   // every read of this block's tiles and accumulators done before the next block's loads
    fence_after_sync();
  }   // blocks
    if (failed && tid == 0) {   // no product may outlive the tensor memory
        atomicExch(status, (int)DPLR_ERR_TIMEOUT);
        mma_commit(drain);
        mbar_wait(drain, 0, 400000000LL);
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
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
    uint64_t* full = bars + 0;     // the step's A_j tiles landed
    uint64_t* freed = bars + 1;    // the step's products are done (with the B_j tiles last)
    uint64_t* fullB = bars + 7;    // the step's B_j tiles landed
    uint64_t* freedA = bars + 8;   // the step's X^T is done with the A_j tiles (the next A_j may land)
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
        mbar_init(fullB, 1);
        mbar_init(freedA, 1);
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
        // ---- copies of each step's operand tiles: the A_j pair once the previous step's X^T is done with its own,
        // the B_j pair once the previous step's o^T products are
        int lastA = -1, lastB = -1;
        for (int st = 0; st < ns && lane == 0; ++st) {
            const unsigned char* src = args.tiles + (bh * (size_t)N + list[st]) * 4 * kOpTile;
            if (st >= 1 && !mbar_wait(freedA, (st - 1) & 1, wl)) { failed = true; break; }
            mbar_expect_tx(full, 2 * kOpTile);
            for (int e = 0; e < 2; ++e) bulk_g2s(smem + S::OPS + e * kOpTile, src + e * kOpTile, kOpTile, full);
            lastA = st;
            if (st >= 1 && !mbar_wait(freed, (st - 1) & 1, wl)) { failed = true; break; }
            mbar_expect_tx(fullB, 2 * kOpTile);
            for (int e = 2; e < 4; ++e) bulk_g2s(smem + S::OPS + e * kOpTile, src + e * kOpTile, kOpTile, fullB);
            lastB = st;
            if (st + 1 < ns) {
                const unsigned char* nx = args.tiles + (bh * (size_t)N + list[st + 1]) * 4 * kOpTile;
                for (int e = 0; e < 4; ++e)
                    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(reinterpret_cast<uint64_t>(nx + e * kOpTile)),
                                 "r"(kOpTile) : "memory");
            }
        }
        if (failed) {   // (lane 0) no copy may land after the CTA has exited
            atomicExch(args.status, (int)DPLR_ERR_TIMEOUT);
            if (lastA >= 0) mbar_wait(full, lastA & 1, 400000000LL);
            if (lastB >= 0) mbar_wait(fullB, lastB & 1, 400000000LL);
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
            mma_commit(freedA);
            if (!mbar_wait(fullB, st & 1, wl)) { failed = true; break; }
            fence_after_sync();
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

std::atomic<uint64_t> g_hla_smem[5] = {{0}, {0}, {0}, {0}, {0}};

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
    if (pl.bf16 && pl.dk == HD2 && pl.dv == HD2) {   // pass 1 on the tensor cores (o <- O_t)
        if (set_smem_limit_once(reinterpret_cast<const void*>(hla_block_maps_tc_kernel), BSm::TOTAL, g_hla_smem[4]) != cudaSuccess)
            return DPLR_ERR_CUDA;
        hla_block_maps_tc_kernel<<<(unsigned)std::min<long long>((long long)pl.BH * pl.nb, sm_count()), kBT, BSm::TOTAL, s>>>(
            pl, static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v),
            g, beta, ma.Pm, ma.Cm, ma.Qm, o, reinterpret_cast<int*>(ws));
        if (cudaGetLastError() != cudaSuccess) return DPLR_ERR_CUDA;
    } else if (launch_chunk_maps(pl, ma, s) != cudaSuccess) {   // pass 1 in fp32 (o <- O_t)
        return DPLR_ERR_CUDA;
    }
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
