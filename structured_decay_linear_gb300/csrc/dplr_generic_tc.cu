// The generic DPLR mode (S_t = D_t S_{t-1} - A_t (B_t^T S_{t-1}) + K_t V_t^T, o_t = S_t^T q_t, with
// D_t = Diag(e^{decay_t}), rank r_ab <= 4 and r_kv <= 2) at dk = dv = 64 on the tensor cores: the two-stage
// chunkwise algorithm of "Householder-Diagonalized Linear Attention" (Key design 3: the rank-generalised WY
// representation, every token's r x r block treated as one element).
//
// Stage 1, generic_chunk_kernel, takes one block of 32 tokens of one head per step. With G_t the inclusive
// cumulative log-decay inside the block (one value per key channel), anchor a = G_32 / 2 and the block's rows
// s = t r + i (factors) and u = t p + i (writes):
//
//   A~_s = e^{a - G_t} A_{t,i}     B~_s = e^{G_{t-1} - a} B_{t,i}     K~_u = e^{a - G_t} K_{t,i}
//   Q~_t = e^{G_t - a} q_t
//   L    = strict_block_tril(B~ A~^T)      G = strict_block_tril(B~ K~^T)      M = (I + L)^{-1}
//   Y    = M B~       U = M (G V)
//   P_j  = Diag(e^{G_32}) - Diag(e^a) (A~^T Y) Diag(e^a)         S_j = P_j S_{j-1} + c_j
//   c_j  = Diag(e^a) (K~^T V - A~^T U)
//   QA   = tril_incl(Q~ A~^T)   QK = tril_incl(Q~ K~^T)
//   Q'_j = (Q~ - QA Y) Diag(e^a)      O_j = QK V - QA U          o_t = Q'_t S_{j-1} + O_t
//
// With the write rows folded in as extra rows X = [A~; -K~] and coefficients Z = [[Y, U], [0, V]] (rows of X,
// columns [dk | dv]), the four results come from two products: Z^T X = [(A~^T Y)^T ; -(c_j e^{-a})^T] and
// Z^T [QA, -QK]^T = [(QA Y)^T ; -O_j^T]. The inverse is fp32: 16 x 16 diagonal blocks by substitution, merged
// 16 -> 32 -> 64 -> 128 with warp-level products in three tf32 terms.
//
// Stage 2, generic_chain_kernel, walks each head's blocks in order with one product per block,
// [P_j; Q'_j] S_{j-1}, the state kept in fp32 registers.
//
// Precision. The tolerance is that of fp32 inputs (max |err| <= 1e-4 of the RMS). Every product runs on tcgen05
// (kind::f16, fp32 accumulators in tensor memory) with both operands split into two fp16 terms after a
// power-of-two scale per operand, x s = hi + lo, and three partial products (hi hi + hi lo + lo hi), which keeps
// ~22 significant bits. A float64 emulation of these rounding points over the generic distributions gives
// 1e-6 to 5e-6 of the RMS; the same scheme with bf16 terms (16 bits, no scale needed) gives 4e-5 to 9e-5, too
// close to the tolerance, and one tf32 term for any operand, or a tf32 inverse, 3e-4 or more.
//
// Every wait is bounded by Plan::wait_cycles; a wait that gives up sets DPLR_ERR_TIMEOUT in the status word
// and the kernel drains its own copies and products before it frees tensor memory.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cstring>

#include "dplr_internal.h"
#include "sm100_ops.cuh"
#include "tc_common.cuh"

namespace dplr {
namespace {

using namespace sm100;
using namespace tc;

constexpr int GD = 64;      // dk = dv
constexpr int GCW = 32;     // tokens per WY block
constexpr int GT = 512;     // threads: four per tensor-memory lane
constexpr int GMAXR = 4;    // r_ab: at most 128 factor rows per block
constexpr int GMAXP = 2;    // r_kv: at most 64 write rows per block

// Shared memory (bytes from the 1024-aligned base). bf16 tiles are [rows][64] with 128-byte swizzled rows.
// -K~ follows A~ so that [A~; -K~] is one operand of 128 + Pp rows; a 128-row read of -K~ hi runs into A~ lo,
// one of -K~ lo into the zero tile.
struct GSmem {
    static constexpr int A_H = 0;              // A~ hi [128][64]
    static constexpr int K_H = 16384;          // -K~ hi [64][64]
    static constexpr int A_L = 24576;          // A~ lo
    static constexpr int K_L = 40960;          // -K~ lo
    static constexpr int ZERO = 49152;         // zeros [64][64]: the Y columns of Z's write rows
    static constexpr int B_H = 57344;          // B~ hi, then Y hi
    static constexpr int W_H = 73728;          // -(G V) hi, then U hi: the second 64-column block of [B~ | -(G V)]
    static constexpr int B_L = 90112;          // B~ lo, then Y lo
    static constexpr int W_L = 106496;         // -(G V) lo, then U lo
    static constexpr int V_H = 122880;         // V hi [64][64]
    static constexpr int V_L = 131072;         // V lo
    static constexpr int Q_H = 139264;         // Q~ hi [32][64]
    static constexpr int Q_L = 143360;         // Q~ lo
    static constexpr int X = 147456;           // fp32 blocks X11, X21, X22 of the inverse; then [QA, -QK]^T:
    static constexpr int QF_H = X;             //   QA^T hi [128][64] (row s, columns t < 32 used)
    static constexpr int QW_H = X + 16384;     //   -QK^T hi [64][64] (row u)
    static constexpr int QF_L = X + 24576;     //   QA^T lo
    static constexpr int QW_L = X + 40960;     //   -QK^T lo
    static constexpr int VEC = X + 3 * 64 * kLdX * 4;   // fp32 per channel: e^a, e^{G_32}; then the maxima slots
    static constexpr int BAR = VEC + 1024;
    static constexpr int TOTAL = BAR + 64;
    // [X | QX] as one MN-major operand: the QX block sits this far past the X rows (the same for hi and lo, and for
    // the factor and the write rows)
    static constexpr int LBO_XQ = QF_H - A_H;
};
static_assert(GSmem::TOTAL <= 227 * 1024, "shared memory budget");
static_assert(GSmem::QW_L + 8192 <= GSmem::VEC, "QX tiles fit the inverse's region");
static_assert(GSmem::QF_L - GSmem::A_L == GSmem::LBO_XQ && GSmem::QW_H - GSmem::K_H == GSmem::LBO_XQ &&
              GSmem::QW_L - GSmem::K_L == GSmem::LBO_XQ, "one leading-byte offset for every [X | QX] operand");
static_assert(GSmem::LBO_XQ < (1 << 18), "leading-byte offset field");

// Tensor-memory columns (512 allocated).
constexpr uint32_t TL = 0;      // L (and -G right after it), then [Y | -U]                    128
constexpr uint32_t TG = 128;    // -G (lane s, column u), then Z^T [X | QX]                    128 (with TW)
constexpr uint32_t TW = 192;    // -(G V)                                                       64
constexpr uint32_t TQA = 256;   // QA^T (lane s, column t)                                      32
constexpr uint32_t TQK = 288;   // -QK^T (lane u, column t)                                     32
constexpr uint32_t TMH = 320;   // M hi as a bf16 A operand                                     64
constexpr uint32_t TML = 384;   // M lo                                                         64
constexpr uint32_t TGH = 448;   // -G hi as a bf16 A operand                                    32
constexpr uint32_t TGL = 480;   // -G lo                                                        32

// Loads 8 consecutive values as fp32.
__device__ __forceinline__ void ld8(const float* p, float (&x)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
__device__ __forceinline__ void ld8(const __nv_bfloat16* p, float (&x)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// x (8 values) times sc, split into fp16 hi + lo and stored as one 16-byte chunk (columns 8 ch .. 8 ch + 7) of
// row `row` of the hi and lo tiles.
__device__ __forceinline__ void put8(uint32_t hi, uint32_t lo, int row, int ch, const float (&x)[8], float sc) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) splith2(x[2 * i], x[2 * i + 1], sc, h[i], l[i]);
    const uint32_t off = swz(row, ch);
    sts128(hi + off, h[0], h[1], h[2], h[3]);
    sts128(lo + off, l[0], l[1], l[2], l[3]);
}
__device__ __forceinline__ float absmax8(const float (&x)[8]) {
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(x[i]));
    return m;
}

// Per unit (head, 32-token block) the chunk kernel leaves the chain's operand [P_j; Q'_j] (rows 0-95 of a
// 128-row fp16 tile, hi then lo, 96 x 128 bytes each, P_j scaled by sP and Q'_j by sQ'), followed by 16 bytes:
// 1 / sP and 1 / sQ' (fp32), and c_j (fp32 [64][64]).
constexpr int kChainTile = 96 * 128;
constexpr int kChainA = 2 * kChainTile + 16;
constexpr int kChainStride = 2 * kChainTile + 256;   // bytes per unit of the operand array
constexpr int kChainC = GD * GD * 4;

struct GArgs {
    const void* q; const void* A; const void* Bm; const void* K; const void* V;
    const float* decay;
    float* o; void* Am; float* Cm; int* status;
};

__device__ __forceinline__ void prefetch_bulk_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(reinterpret_cast<uint64_t>(p)), "r"(bytes) : "memory");
}

// Slots of the operands' largest magnitudes (fp32 bit patterns) in shared memory.
enum { MX_X, MX_B, MX_V, MX_Q, MX_G, MX_M, MX_W, MX_QX, MX_Y, MX_U, MX_P, MX_QP, MX_N };

// Persistent: CTA b takes the units b, b + gridDim.x, ... (unit = head bh * nb + block j, so the CTAs running at
// once read neighbouring blocks). The next unit's inputs are prefetched into L2 while the current one is computed.
template <class IT>
__global__ void __launch_bounds__(GT, 1)
generic_chunk_kernel(Plan pl, GArgs args) {
    using S = GSmem;
    extern __shared__ __align__(1024) unsigned char smem[];
    const uint32_t sb = smem_addr(smem);
    if (sb & 1023u) {   // the swizzled tiles need 1024-byte alignment
        if (threadIdx.x == 0) atomicExch(args.status, (int)DPLR_ERR_CUDA);
        return;
    }
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::BAR);
    uint64_t* mb_mma = bars + 0;
    uint64_t* mb_drain = bars + 1;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2);
    float* ea = reinterpret_cast<float*>(smem + S::VEC);   // [64] e^{a}
    float* gam = ea + 64;                                  // [64] e^{G_32}
    unsigned int* mx = reinterpret_cast<unsigned int*>(smem + S::VEC + 512);   // [MX_N]
    float* Xf = reinterpret_cast<float*>(smem + S::X);
    auto mxf = [&](int k) { return __uint_as_float(*reinterpret_cast<volatile unsigned int*>(&mx[k])); };
    auto scl = [&](int k) { return scale_for(mxf(k)); };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = pl.r, p = pl.p, R = GCW * r, Pp = GCW * p;
    const int T = pl.T, nb = pl.nb;
    const long long total = (long long)pl.BH * nb;
    const long long wl = pl.wait_cycles;
    const IT* q = static_cast<const IT*>(args.q);
    const IT* Ag = static_cast<const IT*>(args.A);
    const IT* Bg = static_cast<const IT*>(args.Bm);
    const IT* Kg = static_cast<const IT*>(args.K);
    const IT* Vg = static_cast<const IT*>(args.V);

    if (tid == 0) {
        mbar_init(mb_mma, 1);
        mbar_init(mb_drain, 1);
        mbar_fence_init();
    }
    for (int i = tid; i < 8192 / 16; i += GT) sts128(sb + S::ZERO + 16 * i, 0u, 0u, 0u, 0u);
    if (warp == 0) tmem_alloc(tmem_holder, 512);
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_holder;
    uint32_t mma_phase = 0;
    bool failed = false;
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const int s = tid & 127;   // tensor-memory lane of this thread
    const int qd = tid >> 7;   // which quarter of the columns it takes

    auto wait_mma = [&]() {
        const bool ok = mbar_wait(mb_mma, mma_phase & 1, wl);
        ++mma_phase;
        if (__syncthreads_or(!ok)) failed = true;
        fence_after_sync();
    };

  for (long long uidx = blockIdx.x; uidx < total && !failed; uidx += gridDim.x) {
    const int j = static_cast<int>(uidx % nb);
    const size_t bh = static_cast<size_t>(uidx / nb);
    const int valid = min(GCW, T - j * GCW);
    const size_t tok0 = bh * (size_t)T + (size_t)j * GCW;   // first token row of the block
    if (tid == 0 && uidx + gridDim.x < total) {   // the next unit's inputs into L2 (whole blocks only)
        const long long nx = uidx + gridDim.x;
        const int jn = static_cast<int>(nx % nb);
        if (T - jn * GCW >= GCW) {
            const size_t t1 = (size_t)(nx / nb) * T + (size_t)jn * GCW;
            const uint32_t rowb = GD * sizeof(IT) * GCW;
            prefetch_bulk_l2(args.decay + t1 * GD, GD * 4 * GCW);
            prefetch_bulk_l2(q + t1 * GD, rowb);
            prefetch_bulk_l2(Ag + t1 * r * GD, rowb * r);
            prefetch_bulk_l2(Bg + t1 * r * GD, rowb * r);
            if (p > 0) {
                prefetch_bulk_l2(Kg + t1 * p * GD, rowb * p);
                prefetch_bulk_l2(Vg + t1 * p * GD, rowb * p);
            }
        }
    }
    if (tid < MX_N) mx[tid] = 0u;   // (the previous unit's last reads of the slots precede its final barrier)

    // ---- a1: this thread's pieces of the block's rows (8 channels each), loaded before any is used: A~ and B~ rows
    // row0 and row0 + 64, -K~ and V row row0 (Pp rows), Q~ row row0 (32 rows)
    const int ch = tid & 7, row0 = tid >> 3;
    float xa[2][8], xb[2][8], xk[8], xv[8], xq[8];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int row = row0 + 64 * h, t = row / r, i = row - t * r;
        if (row < R && t < valid) {
            ld8(Ag + ((tok0 + t) * r + i) * GD + 8 * ch, xa[h]);
            ld8(Bg + ((tok0 + t) * r + i) * GD + 8 * ch, xb[h]);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) xa[h][e] = xb[h][e] = 0.f;
        }
    }
    {
        const int t = p > 0 ? row0 / p : 0, i = row0 - t * p;
        if (row0 < Pp && t < valid) {
            ld8(Kg + ((tok0 + t) * p + i) * GD + 8 * ch, xk);
            ld8(Vg + ((tok0 + t) * p + i) * GD + 8 * ch, xv);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) xk[e] = xv[e] = 0.f;
        }
        if (row0 < GCW && row0 < valid) {
            ld8(q + (tok0 + row0) * GD + 8 * ch, xq);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) xq[e] = 0.f;
        }
    }

    // ---- a2: cumulative log-decay. Warp w takes channels 4 w .. 4 w + 3, lane t token t (identity padding past the
    // end: log-decay 0); an inclusive scan over the lanes gives G_t, a shift G_{t-1}. The decay tables
    // Er[t] = e^{a - G_t} and Ef[t] = e^{G_{t-1} - a} (Ef[32] = e^{G_31 - a}) go to the inverse's region.
    float* Er = Xf;              // [32][64]
    float* Ef = Xf + 32 * GD;    // [33][64]
    {
        const int c0 = 4 * warp, t = lane;
        float4 g = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t < valid) g = *reinterpret_cast<const float4*>(args.decay + (tok0 + t) * GD + c0);
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float x0 = __shfl_up_sync(0xffffffffu, g.x, off), x1 = __shfl_up_sync(0xffffffffu, g.y, off);
            const float x2 = __shfl_up_sync(0xffffffffu, g.z, off), x3 = __shfl_up_sync(0xffffffffu, g.w, off);
            if (lane >= off) { g.x += x0; g.y += x1; g.z += x2; g.w += x3; }
        }
        float4 gp;
        gp.x = __shfl_up_sync(0xffffffffu, g.x, 1); gp.y = __shfl_up_sync(0xffffffffu, g.y, 1);
        gp.z = __shfl_up_sync(0xffffffffu, g.z, 1); gp.w = __shfl_up_sync(0xffffffffu, g.w, 1);
        if (lane == 0) gp = make_float4(0.f, 0.f, 0.f, 0.f);
        const float a0 = 0.5f * __shfl_sync(0xffffffffu, g.x, 31), a1 = 0.5f * __shfl_sync(0xffffffffu, g.y, 31);
        const float a2 = 0.5f * __shfl_sync(0xffffffffu, g.z, 31), a3 = 0.5f * __shfl_sync(0xffffffffu, g.w, 31);
        *reinterpret_cast<float4*>(Er + t * GD + c0) =
            make_float4(__expf(a0 - g.x), __expf(a1 - g.y), __expf(a2 - g.z), __expf(a3 - g.w));
        *reinterpret_cast<float4*>(Ef + t * GD + c0) =
            make_float4(__expf(gp.x - a0), __expf(gp.y - a1), __expf(gp.z - a2), __expf(gp.w - a3));
        if (lane == 31) {
            *reinterpret_cast<float4*>(Ef + 32 * GD + c0) =
                make_float4(__expf(g.x - a0), __expf(g.y - a1), __expf(g.z - a2), __expf(g.w - a3));
            *reinterpret_cast<float4*>(ea + c0) = make_float4(__expf(a0), __expf(a1), __expf(a2), __expf(a3));
            *reinterpret_cast<float4*>(gam + c0) = make_float4(__expf(g.x), __expf(g.y), __expf(g.z), __expf(g.w));
        }
    }
    __syncthreads();

    // ---- a3: the decay-scaled factors (their largest magnitudes first), then the fp16 hi / lo tiles
    {
        float mX = 0.f, mB = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int t = min((row0 + 64 * h) / r, GCW - 1);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                xa[h][e] *= Er[t * GD + 8 * ch + e];
                xb[h][e] *= Ef[t * GD + 8 * ch + e];
            }
            mX = fmaxf(mX, absmax8(xa[h]));
            mB = fmaxf(mB, absmax8(xb[h]));
        }
        const int tk = p > 0 ? min(row0 / p, GCW - 1) : 0, tq = min(row0, GCW - 1);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            xk[e] *= -Er[tk * GD + 8 * ch + e];
            xq[e] *= Ef[(tq + 1) * GD + 8 * ch + e];
        }
        warp_max_to(&mx[MX_X], fmaxf(mX, absmax8(xk)));
        warp_max_to(&mx[MX_B], mB);
        warp_max_to(&mx[MX_V], absmax8(xv));
        warp_max_to(&mx[MX_Q], absmax8(xq));
    }
    if (tid == 0) bulk_wait_read();   // the previous unit's [P_j; Q'_j] has left the staging area over B~
    __syncthreads();
    {
    const float sX = scl(MX_X), sB = scl(MX_B), sV = scl(MX_V), sQ = scl(MX_Q);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        put8(sb + S::A_H, sb + S::A_L, row0 + 64 * h, ch, xa[h], sX);
        put8(sb + S::B_H, sb + S::B_L, row0 + 64 * h, ch, xb[h], sB);
    }
    put8(sb + S::K_H, sb + S::K_L, row0, ch, xk, sX);
    put8(sb + S::V_H, sb + S::V_L, row0, ch, xv, sV);
    if (row0 < GCW) put8(sb + S::Q_H, sb + S::Q_L, row0, ch, xq, sQ);
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();

    // ---- a4: [L | -G] = B~ [A~; -K~]^T, QA^T = A~ Q~^T, -QK^T = (-K~) Q~^T (three terms each)
    if (warp == 0) {
        const uint32_t lead = lane == 0;
        const uint32_t loA[3] = {0, 0, 1}, loB[3] = {0, 1, 0};   // terms (A, B): (hi, hi), (hi, lo), (lo, hi)
        const uint32_t idL = idesc_f16(128, 128 + Pp, false, false), idQ = idesc_f16(128, 32, false, false);
#pragma unroll
        for (int term = 0; term < 3; ++term) {
            const uint32_t bt = sb + (loA[term] ? S::B_L : S::B_H);
            const uint32_t ax = sb + (loB[term] ? S::A_L : S::A_H);   // [A~; -K~] as the B operand
            const uint32_t qt = sb + (loB[term] ? S::Q_L : S::Q_H);
            const uint32_t aa = sb + (loA[term] ? S::A_L : S::A_H);
            const uint32_t ka = sb + (loA[term] ? S::K_L : S::K_H);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint32_t acc = (term > 0 || kk > 0);
                mma_ss_if(tmem + TL, smem_desc_sw128(bt + 32 * kk, 16, 1024), smem_desc_sw128(ax + 32 * kk, 16, 1024),
                          idL, acc, lead);
                mma_ss_if(tmem + TQA, smem_desc_sw128(aa + 32 * kk, 16, 1024), smem_desc_sw128(qt + 32 * kk, 16, 1024),
                          idQ, acc, lead);
                if (p > 0)
                    mma_ss_if(tmem + TQK, smem_desc_sw128(ka + 32 * kk, 16, 1024), smem_desc_sw128(qt + 32 * kk, 16, 1024),
                              idQ, acc, lead);
            }
        }
        commit_if(mb_mma, lead);
    }
    wait_mma();
    if (failed) break;

    // ---- L into the inverse's fp32 blocks (strict lower part by token: column c < r * token of s); the largest
    // magnitudes of -G (strict: u < p * token of s) and of [QA, -QK] (inclusive: token of the row <= t); then -G as
    // an fp16 hi / lo tensor-memory operand, read again once its scale is known
    const bool has_g = p > 0 && qd < 2 && 32 * qd < Pp;
    const bool qa = qd == 2 && s < R, qk = qd == 3 && p > 0 && s < Pp;
    {
        const float uBX = 1.f / (scl(MX_B) * scl(MX_X));   // (powers of two: exact)
        const int ts = s / r, cl = ts * r;
        float x[32];
        tmem_ld32(tmem + lane_base + TL + 32 * qd, x);
        float* dst = nullptr;   // row s of X11 / X21 (columns 0-63), or of X22 (columns 64-127, shifted)
        if (qd < 2) dst = Xf + s * kLdX;
        else if (s >= 64) dst = Xf + (128 + (s - 64)) * kLdX - 64;
        if (dst) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                const int c = 32 * qd + i;
                *reinterpret_cast<float4*>(dst + c) =
                    make_float4(c < cl ? uBX * x[i] : 0.f, c + 1 < cl ? uBX * x[i + 1] : 0.f,
                                c + 2 < cl ? uBX * x[i + 2] : 0.f, c + 3 < cl ? uBX * x[i + 3] : 0.f);
            }
        }
        float mg = 0.f;
        if (has_g) {
            const int ul = ts * p;
            tmem_ld32(tmem + lane_base + TG + 32 * qd, x);
#pragma unroll
            for (int i = 0; i < 32; ++i) mg = fmaxf(mg, 32 * qd + i < ul ? fabsf(x[i]) : 0.f);
        }
        if (p > 0 && qd < 2) warp_max_to(&mx[MX_G], mg * uBX);
        float mq = 0.f;
        if (qa || qk) {
            tmem_ld32(tmem + lane_base + (qa ? TQA : TQK), x);
            const int tk = qa ? ts : s / max(p, 1);   // token of this lane's row
#pragma unroll
            for (int t = 0; t < GCW; ++t) mq = fmaxf(mq, tk <= t ? fabsf(x[t]) : 0.f);
        }
        if (qd >= 2) warp_max_to(&mx[MX_QX], mq / (scl(MX_X) * scl(MX_Q)));
    }
    __syncthreads();
    if (has_g) {
        const float sG = scl(MX_G), u = sG / (scl(MX_B) * scl(MX_X));
        const int ul = (s / r) * p;
        float x[32];
        tmem_ld32(tmem + lane_base + TG + 32 * qd, x);
        uint32_t h[16], l[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int u0 = 32 * qd + 2 * i;
            splith2(u0 < ul ? x[2 * i] * u : 0.f, u0 + 1 < ul ? x[2 * i + 1] * u : 0.f, 1.f, h[i], l[i]);
        }
        tmem_st16(tmem + lane_base + TGH + 16 * qd, h);
        tmem_st16(tmem + lane_base + TGL + 16 * qd, l);
    }
    tmem_wait_st();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();

    // ---- a5: -(G V) on the tensor cores while the CUDA cores invert I + L
    if (p > 0 && warp == 0) {
        const uint32_t lead = lane == 0;
        const uint32_t idW = idesc_f16(128, 64, false, true);
#pragma unroll
        for (int term = 0; term < 3; ++term) {
            const uint32_t ga = tmem + (term == 2 ? TGL : TGH);
            const uint64_t vb = smem_desc_sw128(sb + (term == 1 ? S::V_L : S::V_H), 8192, 1024);
            for (int kk = 0; kk < Pp / 16; ++kk)
                mma_ts_if(tmem + TW, ga + 8 * kk, dadd(vb, 2048 * kk), idW, (term > 0 || kk > 0), lead);
        }
        commit_if(mb_mma, lead);
    }
    {
        if (warp < 8) inv64_inplace<3>(Xf, tid, 1);                    // M11 in place of L11
        else inv64_inplace<3>(Xf + 128 * kLdX, tid - 256, 2);          // M22 in place of L22
        __syncthreads();
        // 64 -> 128: M21 = -M22 (L21 M11); warp w takes column block w % 8 and row blocks 2 (w / 8), 2 (w / 8) + 1
        float* X11 = Xf;
        float* X21 = Xf + 64 * kLdX;
        float* X22 = Xf + 128 * kLdX;
        const int cb = warp & 7, rb0 = 2 * (warp >> 3);
        float c[2][4];
        warp_mma_tf32_tiles<3, 2>(X21 + 16 * rb0 * kLdX, kLdX, X11 + 8 * cb, kLdX, 64, c);
        __syncthreads();
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) store_tile_16x8(X21 + 16 * (rb0 + rr) * kLdX + 8 * cb, kLdX, c[rr], 1.f);
        __syncthreads();
        warp_mma_tf32_tiles<3, 2>(X22 + 16 * rb0 * kLdX, kLdX, X21 + 8 * cb, kLdX, 64, c);
        __syncthreads();
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) store_tile_16x8(X21 + 16 * (rb0 + rr) * kLdX + 8 * cb, kLdX, c[rr], -1.f);
        __syncthreads();
    }
    // ---- the largest magnitude of M; then (after the barrier) M as fp16 hi / lo tensor-memory operands, read
    // again from the inverse's blocks (thread (s, qd): columns 32 qd .. 32 qd + 31 of row s)
    auto m_row = [&]() -> const float* {   // nullptr: zero (above the diagonal blocks)
        if (qd < 2) return Xf + s * kLdX + 32 * qd;
        if (s >= 64) return Xf + (128 + (s - 64)) * kLdX + 32 * (qd - 2);
        return nullptr;
    };
    {
        const float* row = m_row();
        float mm = 0.f;
        if (row) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                const float4 v = *reinterpret_cast<const float4*>(row + i);
                mm = fmaxf(mm, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
            }
        }
        warp_max_to(&mx[MX_M], mm);
    }
    if (p > 0) {
        wait_mma();   // -(G V) done; also the barrier after which M's maximum is known
        if (failed) break;
    } else {
        __syncthreads();
    }
    {
        const float* row = m_row();
        const float sM = scl(MX_M);
        uint32_t h[16], l[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) splith2(row ? row[2 * i] : 0.f, row ? row[2 * i + 1] : 0.f, sM, h[i], l[i]);
        tmem_st16(tmem + lane_base + TMH + 16 * qd, h);
        tmem_st16(tmem + lane_base + TML + 16 * qd, l);
    }
    {   // the largest magnitude of -(G V) (thread (s, qd): columns 16 qd ..)
        float mw = 0.f;
        if (p > 0) {
            float x[16];
            tmem_ld16(tmem + lane_base + TW + 16 * qd, x);
#pragma unroll
            for (int i = 0; i < 16; ++i) mw = fmaxf(mw, fabsf(x[i]));
        }
        warp_max_to(&mx[MX_W], mw / (scl(MX_G) * scl(MX_V)));
    }
    __syncthreads();   // (also: every row of M read, so the inverse's region is free)
    {   // -(G V) hi / lo into the second column block of [B~ | -(G V)] (zero when there is no write term)
        const float u = scl(MX_W) / (scl(MX_G) * scl(MX_V));
        float x[16];
        if (p > 0) {
            tmem_ld16(tmem + lane_base + TW + 16 * qd, x);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) x[i] = 0.f;
        }
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
            uint32_t h[4], l[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) splith2(x[8 * c2 + 2 * i], x[8 * c2 + 2 * i + 1], u, h[i], l[i]);
            const uint32_t off = swz(s, 2 * qd + c2);
            sts128(sb + S::W_H + off, h[0], h[1], h[2], h[3]);
            sts128(sb + S::W_L + off, l[0], l[1], l[2], l[3]);
        }
    }
    if (qa || qk) {   // [QA, -QK]^T hi / lo, MN-major [row][t] over the inverse's region: the QX block of [X | QX]
        const float u = scl(MX_QX) / (scl(MX_X) * scl(MX_Q));
        const int tk = qa ? s / r : s / max(p, 1);
        float x[32];
        tmem_ld32(tmem + lane_base + (qa ? TQA : TQK), x);
        const uint32_t th = sb + (qa ? S::QF_H : S::QW_H), tl = sb + (qa ? S::QF_L : S::QW_L);
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
            uint32_t h[4], l[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int t0 = 8 * c4 + 2 * i;
                splith2(tk <= t0 ? x[t0] : 0.f, tk <= t0 + 1 ? x[t0 + 1] : 0.f, u, h[i], l[i]);
            }
            const uint32_t off = swz(s, c4);
            sts128(th + off, h[0], h[1], h[2], h[3]);
            sts128(tl + off, l[0], l[1], l[2], l[3]);
        }
    }
    tmem_wait_st();
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();

    // ---- a5 (applications): [Y | -U] = M [B~ | -(G V)]
    if (warp == 0) {
        const uint32_t lead = lane == 0;
        const uint32_t idY = idesc_f16(128, 128, false, true);
#pragma unroll
        for (int term = 0; term < 3; ++term) {
            const uint32_t ma = tmem + (term == 2 ? TML : TMH);
            const uint64_t bb = smem_desc_sw128(sb + (term == 1 ? S::B_L : S::B_H), 16384, 1024);
            for (int kk = 0; kk < R / 16; ++kk)
                mma_ts_if(tmem + TL, ma + 8 * kk, dadd(bb, 2048 * kk), idY, (term > 0 || kk > 0), lead);
        }
        commit_if(mb_mma, lead);
    }
    wait_mma();
    if (failed) break;

    // ---- Z's factor rows [Y | U]: Y with its own scale, U with the scale it shares with V (the same products sum
    // them); V's tiles are rescaled to it (powers of two: exact). The largest magnitudes first, then the tiles from
    // a second read of the accumulator.
    {
        float x[32];
        tmem_ld32(tmem + lane_base + TL + 32 * qd, x);
        float m = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) m = fmaxf(m, fabsf(x[i]));
        warp_max_to(&mx[qd < 2 ? MX_Y : MX_U], m / (scl(MX_M) * (qd < 2 ? scl(MX_B) : scl(MX_W))));
    }
    __syncthreads();
    {
        const float sY = scl(MX_Y), sUV = scale_for(fmaxf(mxf(MX_U), mxf(MX_V))), sV = scl(MX_V);
        const float u = qd < 2 ? sY / (scl(MX_M) * scl(MX_B)) : -sUV / (scl(MX_M) * scl(MX_W));
        const uint32_t th = sb + (qd < 2 ? S::B_H : S::W_H), tl = sb + (qd < 2 ? S::B_L : S::W_L);
        float x[32];
        tmem_ld32(tmem + lane_base + TL + 32 * qd, x);
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
            uint32_t h[4], l[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) splith2(x[8 * c4 + 2 * i], x[8 * c4 + 2 * i + 1], u, h[i], l[i]);
            const uint32_t off = swz(s, 4 * (qd & 1) + c4);
            sts128(th + off, h[0], h[1], h[2], h[3]);
            sts128(tl + off, l[0], l[1], l[2], l[3]);
        }
        if (p > 0 && sUV != sV) {   // V hi and lo (Pp rows of 128 bytes each) times sUV / sV
            const float d = sUV / sV;
            for (int i = tid; i < 2 * Pp * 8; i += GT) {
                const uint32_t a = sb + (i < Pp * 8 ? S::V_H : S::V_L) + 16 * (i % (Pp * 8));
                uint32_t w[4];
                asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "r"(a));
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
                    const __half2 g = __floats2half2_rn(f.x * d, f.y * d);
                    w[e] = *reinterpret_cast<const uint32_t*>(&g);
                }
                sts128(a, w[0], w[1], w[2], w[3]);
            }
        }
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();

    // ---- a6/a7 (block part): Z^T [X | QX] over the factor rows, then the write rows (N = 128: columns 0-63
    // A~^T Y and c_j, 64-95 QA Y and O_j, 96-127 unused)
    if (warp == 0) {
        const uint32_t lead = lane == 0;
        const uint32_t idP = idesc_f16(128, 128, true, true);
        const int nk = (R + Pp) / 16;
#pragma unroll
        for (int term = 0; term < 3; ++term) {
            const bool zl = term == 2, xl = term == 1;
            for (int kk = 0; kk < nk; ++kk) {
                uint64_t za, xb;
                if (kk < R / 16) {
                    za = smem_desc_sw128(sb + (zl ? S::B_L : S::B_H) + 2048 * kk, 16384, 1024);
                    xb = smem_desc_sw128(sb + (xl ? S::A_L : S::A_H) + 2048 * kk, S::LBO_XQ, 1024);
                } else {
                    const int k2 = kk - R / 16;
                    za = smem_desc_sw128(sb + S::ZERO + 2048 * k2, zl ? (S::V_L - S::ZERO) : (S::V_H - S::ZERO), 1024);
                    xb = smem_desc_sw128(sb + (xl ? S::K_L : S::K_H) + 2048 * k2, S::LBO_XQ, 1024);
                }
                mma_ss_if(tmem + TG, za, xb, idP, (term > 0 || kk > 0), lead);
            }
        }
        commit_if(mb_mma, lead);
    }
    wait_mma();
    if (failed) break;

    // ---- epilogue: lane m < 64 holds column m of A~^T Y (columns 0-63) and of (QA Y)^T (64-95); lane 64 + n holds
    // -(c_j e^{-a})^T and -O_j^T for column n. Thread (m, qd) takes a quarter of the columns. c_j and O_j are stored
    // in fp32 at once; P_j and Q'_j become rows 0-63 and 64-95 of the chain's operand [P_j; Q'_j] (fp16 hi and lo
    // with one scale each, 128-byte swizzled rows of 64 columns) once their largest magnitudes are known, from a
    // second read of the accumulator.
    {
        const size_t unit = bh * (size_t)nb + j;
        // staged in shared memory over Z's tiles (read by the last products, which are done), then one bulk copy
        unsigned char* Ah = smem + S::B_H;
        unsigned char* Al = Ah + kChainTile;
        const int m = s;
        const float sz = m < GD ? scl(MX_Y) : scale_for(fmaxf(mxf(MX_U), mxf(MX_V)));
        const float uX = 1.f / (sz * scl(MX_X)), uQ = 1.f / (sz * scl(MX_QX)), uq = 1.f / scl(MX_Q);
        // P_j[i][m] = [i == m] e^{G_32,i} - e^{a_i} (A~^T Y)[i][m] e^{a_m}, i = 16 qd + e
        auto pval = [&](const float (&x)[16], int e) {
            const int i = 16 * qd + e;
            return (i == m ? gam[i] : 0.f) - ea[i] * (uX * x[e]) * ea[m];
        };
        // Q'_j[t][c] = e^{a_c} (Q~[t][c] - (QA Y)[t][c]), c = m, t = 16 qd + e; Q~ from its hi and lo tiles
        auto qval = [&](const float (&x)[16], int e) {
            const int t = 16 * qd + e;
            const uint32_t oq = swz(t, m >> 3) + ((m & 7) << 1);
            uint16_t qh, ql;
            asm volatile("ld.shared.b16 %0, [%1];" : "=h"(qh) : "r"(sb + S::Q_H + oq));
            asm volatile("ld.shared.b16 %0, [%1];" : "=h"(ql) : "r"(sb + S::Q_L + oq));
            return ea[m] * ((half_value(qh) + half_value(ql)) * uq - uQ * x[e]);
        };
        float mp = 0.f, mo = 0.f;
        {
            float x[16];
            tmem_ld16(tmem + lane_base + TG + 16 * qd, x);
            if (m < GD) {
#pragma unroll
                for (int e = 0; e < 16; ++e) mp = fmaxf(mp, fabsf(pval(x, e)));
            } else {        // c_j[i][n] = -e^{a_i} (Z^T X)[64 + n][i]
                float* Ccol = args.Cm + unit * (size_t)(GD * GD) + (m - GD);
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int i = 16 * qd + e;
                    Ccol[(size_t)i * GD] = -ea[i] * (uX * x[e]);
                }
            }
        }
        if (qd < 2) {
            float x[16];
            tmem_ld16(tmem + lane_base + TG + 64 + 16 * qd, x);
            if (m < GD) {
#pragma unroll
                for (int e = 0; e < 16; ++e) mo = fmaxf(mo, fabsf(qval(x, e)));
            } else {        // O_j[t][n] = -(Z^T QX)[64 + n][t]
                float* ocol = args.o + tok0 * GD + (m - GD);
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int t = 16 * qd + e;
                    if (t < valid) ocol[(size_t)t * GD] = -uQ * x[e];
                }
            }
        }
        warp_max_to(&mx[MX_P], mp);
        warp_max_to(&mx[MX_QP], mo);
        __syncthreads();
        const float sP = scl(MX_P), sQP = scl(MX_QP);
        if (m < GD) {
            const uint32_t cm = (uint32_t)((m & 7) << 1);
            float x[16];
            tmem_ld16(tmem + lane_base + TG + 16 * qd, x);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                uint16_t h, l;
                splith1(pval(x, e), sP, h, l);
                const uint32_t off = swz(16 * qd + e, m >> 3) + cm;
                *reinterpret_cast<uint16_t*>(Ah + off) = h;
                *reinterpret_cast<uint16_t*>(Al + off) = l;
            }
            if (qd < 2) {
                tmem_ld16(tmem + lane_base + TG + 64 + 16 * qd, x);
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    uint16_t h, l;
                    splith1(qval(x, e), sQP, h, l);
                    const uint32_t off = swz(GD + 16 * qd + e, m >> 3) + cm;
                    *reinterpret_cast<uint16_t*>(Ah + off) = h;
                    *reinterpret_cast<uint16_t*>(Al + off) = l;
                }
            }
        }
        if (tid == 0)
            *reinterpret_cast<float4*>(Ah + 2 * kChainTile) = make_float4(1.f / sP, 1.f / sQP, 0.f, 0.f);
        fence_async_smem();
        __syncthreads();
        if (tid == 0) {   // (the next unit waits for this copy's reads before its factor build rewrites B~)
            bulk_s2g(reinterpret_cast<unsigned char*>(args.Am) + unit * (size_t)kChainStride, sb + S::B_H, kChainA);
            bulk_commit();
        }
    }
    fence_before_sync();
    __syncthreads();   // every read of this unit's tiles and tensor memory done before the next unit rewrites them
    fence_after_sync();
  }   // units

    if (failed && tid == 0) {
        atomicExch(args.status, (int)DPLR_ERR_TIMEOUT);
        mma_commit(mb_drain);   // tracks every product issued by this thread: none may touch freed tensor memory
        mbar_wait(mb_drain, 0, 400000000LL);
    }
    if (tid == 0) {   // bulk stores still in flight read shared memory: wait before the CTA exits
        bulk_commit();
        bulk_wait_read();
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// ================================================================================================
// Stage 2: the chain over blocks, one CTA per head
// ================================================================================================
//
// S_j = P_j S_{j-1} + c_j and o_t = O_t + Q'_t S_{j-1} for the block's tokens come from one product per block,
// D = [P_j; Q'_j] S_{j-1} (M = 128: rows 0-63 the chain, 64-95 the readout), both operands as fp16 hi + lo with
// a scale each (three terms): the state is kept in fp32 registers and re-split after every block with a scale
// from its largest magnitude. Warp roles: warps 0, 1, 4, 5 hold the state (lane = row i, warps 0-1 columns 0-31,
// warps 4-5 columns 32-63), warps 2 and 6 write the outputs (lane = token), warp 3 copies each block's operand,
// c_j and O_j into a ring of stages (bulk copies and TMA, after an L2 prefetch a few blocks ahead), warp 7 issues
// the products as soon as S_{j-1} is in place.

constexpr int CT = 256;
constexpr int CS = 3;      // stages
constexpr int CPF = 4;     // blocks between the L2 prefetch of a block's maps and their copy

struct GCSmem {
    static constexpr int A_H = 0, A_L = 16384, C_ = 32768, O_ = 49152;   // per stage: [P; Q'] hi, lo (+ scales);
    static constexpr int STAGE = 57344;                                   // c_j, O_j (two fp32 32-column boxes each)
    static constexpr int SH = CS * STAGE;      // S_{j-1} hi: fp16 [64][64], 128-byte swizzled rows (MN-major operand)
    static constexpr int SL = SH + 8192;       // S_{j-1} lo
    static constexpr int RED = SL + 8192;      // the state warps' maxima [4], the state's inverse scales [4]
    static constexpr int BAR = RED + 64;
    static constexpr int TOTAL = BAR + 128;
};
static_assert(GCSmem::TOTAL <= 227 * 1024, "shared memory budget");

struct GCArgs {
    const float* S0; float* o; float* ST; const unsigned char* Am; int* status;
};

__global__ void __launch_bounds__(CT, 1)
generic_chain_kernel(Plan pl, GCArgs args, const __grid_constant__ CUtensorMap tm_C, const __grid_constant__ CUtensorMap tm_O) {
    using S = GCSmem;
    extern __shared__ __align__(1024) unsigned char smem[];
    const uint32_t sb = smem_addr(smem);
    if (sb & 1023u) {
        if (threadIdx.x == 0) atomicExch(args.status, (int)DPLR_ERR_CUDA);
        return;
    }
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::BAR);
    uint64_t* full = bars;               // [CS] a block's maps landed
    uint64_t* freed = bars + CS;         // [CS] the stage was read: the product's commit, 4 state and 2 output warps
    uint64_t* mD = bars + 2 * CS;        // [2] the product of the blocks using accumulator j % 2
    uint64_t* outd = bars + 2 * CS + 2;  // [2] the output warps are done with accumulator j % 2 (2 arrivals)
    uint64_t* ready = bars + 2 * CS + 4; // S_{j-1} tiles (and their scale) written (4 arrivals)
    uint64_t* drain = bars + 2 * CS + 5;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * CS + 6);
    float* wmax = reinterpret_cast<float*>(smem + S::RED);        // [4]
    float* sinv = reinterpret_cast<float*>(smem + S::RED + 16);   // [4] 1 / scale of S_{j-1}, slot j % 4

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = pl.T, nb = pl.nb;
    const size_t bh = blockIdx.x;
    const long long wl = pl.wait_cycles;

    if (tid == 0) {
        for (int u = 0; u < CS; ++u) {
            mbar_init(&full[u], 1);
            mbar_init(&freed[u], 7);
        }
        mbar_init(&mD[0], 1);
        mbar_init(&mD[1], 1);
        mbar_init(&outd[0], 2);
        mbar_init(&outd[1], 2);
        mbar_init(ready, 4);
        mbar_init(drain, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(tmem_holder, 128);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_holder;   // columns 64 (j % 2) ..: the product of block j
    bool failed = false;
    const unsigned char* Ahead = args.Am + bh * (size_t)nb * kChainStride;

    if (warp == 3) {
        // ---- copies of block j into stage j % CS once the stage's previous block is done with
        auto prefetch = [&](int jj) {
            const unsigned char* a = Ahead + (size_t)jj * kChainStride;
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(reinterpret_cast<uint64_t>(a)), "r"((uint32_t)kChainA) : "memory");
            const int yc = static_cast<int>((bh * (size_t)nb + jj) * GD);
            prefetch_l2_tile(&tm_C, 0, yc);
            prefetch_l2_tile(&tm_C, 32, yc);
        };
        int last = -1;
        if (lane == 0)
            for (int jj = 0; jj < CPF && jj < nb; ++jj) prefetch(jj);
        for (int j = 0; j < nb && lane == 0; ++j) {
            const int u = j % CS;
            if (j >= CS && !mbar_wait(&freed[u], ((j - CS) / CS) & 1, wl)) { failed = true; break; }
            if (j + CPF < nb) prefetch(j + CPF);
            unsigned char* st = smem + u * S::STAGE;
            mbar_expect_tx(&full[u], kChainA + kChainC + 2 * 4096);
            const unsigned char* a = Ahead + (size_t)j * kChainStride;
            bulk_g2s(st + S::A_H, a, kChainTile, &full[u]);
            bulk_g2s(st + S::A_L, a + kChainTile, kChainTile + 16, &full[u]);   // with the two scales after it
            const int yc = static_cast<int>((bh * (size_t)nb + j) * GD);
            tma_load_2d(st + S::C_, &tm_C, 0, yc, &full[u]);
            tma_load_2d(st + S::C_ + 8192, &tm_C, 32, yc, &full[u]);
            // rows past the end of the sequence read the next head's rows (or zeros past the tensor): unused
            const int yo = static_cast<int>(bh * (size_t)T + (size_t)j * GCW);
            tma_load_2d(st + S::O_, &tm_O, 0, yo, &full[u]);
            tma_load_2d(st + S::O_ + 4096, &tm_O, 32, yo, &full[u]);
            last = j;
        }
        if (failed) {   // (lane 0) wait for the copies in flight before leaving
            atomicExch(args.status, (int)DPLR_ERR_TIMEOUT);
            for (int jj = last - CS + 1; jj <= last; ++jj)
                if (jj >= 0) mbar_wait(&full[jj % CS], (jj / CS) & 1, 400000000LL);
        }
        __syncwarp();
    } else if (warp == 7) {
        // ---- the product of block j into accumulator j % 2, once S_{j-1} is in place, the maps have landed and the
        // outputs of block j - 2 have been read from that accumulator
        const uint32_t idD = idesc_f16(128, GD, false, true);
        for (int j = 0; j < nb && lane == 0; ++j) {
            const int u = j % CS, b = j & 1;
            if (!mbar_wait(ready, j & 1, wl) || !mbar_wait(&full[u], (j / CS) & 1, wl) ||
                (j >= 2 && !mbar_wait(&outd[b], ((j - 2) >> 1) & 1, wl))) {
                failed = true;
                break;
            }
            fence_after_sync();
            const uint32_t st = sb + u * S::STAGE;
            const uint32_t ao[3] = {st + S::A_H, st + S::A_H, st + S::A_L};
            const uint32_t bo[3] = {sb + S::SH, sb + S::SL, sb + S::SH};
#pragma unroll
            for (int term = 0; term < 3; ++term)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + 64 * b, smem_desc_sw128(ao[term] + 32 * kk, 16, 1024),
                             smem_desc_sw128(bo[term] + 2048 * kk, 8192, 1024), idD, (term > 0 || kk > 0));
            mma_commit(&mD[b]);
            mma_commit(&freed[u]);
        }
        if (failed) {   // (lane 0) no product may outlive the tensor memory
            atomicExch(args.status, (int)DPLR_ERR_TIMEOUT);
            mma_commit(drain);
            mbar_wait(drain, 0, 400000000LL);
        }
        __syncwarp();
    } else if (warp == 2 || warp == 6) {
        // ---- outputs: lane t = token t of the block, columns 32 h .. 32 h + 31
        const int h = warp == 6, t = lane;
        const uint32_t lane_base = static_cast<uint32_t>(64) << 16;
        for (int j = 0; j < nb; ++j) {
            const int u = j % CS, b = j & 1;
            bool ok = true;
            if (lane == 0)
                ok = mbar_wait(&mD[b], (j >> 1) & 1, wl) && mbar_wait(&full[u], (j / CS) & 1, wl) &&
                     mbar_wait(ready, j & 1, wl);
            if (__shfl_sync(0xffffffffu, ok ? 1 : 0, 0) == 0) { failed = true; break; }
            fence_after_sync();
            float x[32];
            tmem_ld32(tmem + lane_base + 64 * b + 32 * h, x);
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&outd[b]);
            const uint32_t stg = sb + u * S::STAGE;
            const float uo = lds_f32(stg + S::A_L + kChainTile + 4) * sinv[j & 3];   // 1 / (sQ' s_S)
            const int valid = min(GCW, T - j * GCW);
            if (t < valid) {
                const uint32_t ob = stg + S::O_ + h * 4096;
                float4* orow = reinterpret_cast<float4*>(args.o + (bh * (size_t)T + (size_t)j * GCW + t) * GD + 32 * h);
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4) {
                    float4 ol;
                    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(ol.x), "=f"(ol.y), "=f"(ol.z), "=f"(ol.w)
                                 : "r"(ob + swz(t, q4)));
                    orow[q4] = make_float4(ol.x + uo * x[4 * q4], ol.y + uo * x[4 * q4 + 1], ol.z + uo * x[4 * q4 + 2],
                                           ol.w + uo * x[4 * q4 + 3]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&freed[u]);
        }
        if (failed && lane == 0) atomicExch(args.status, (int)DPLR_ERR_TIMEOUT);
    } else {
        // ---- the state: warps 0, 1, 4, 5; lane i of warp w holds row i = 32 (w % 4) + lane, columns 32 h .. 32 h + 31
        const int h = warp >= 4, i = 32 * (warp & 3) + lane, sw = (warp & 3) + 2 * h;   // sw: this warp's slot
        const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
        float st[32];
#pragma unroll
        for (int n = 0; n < 32; ++n) st[n] = args.S0 ? args.S0[(bh * GD + i) * GD + 32 * h + n] : 0.f;
        // S into the hi / lo tiles with a scale from its largest magnitude over the four state warps (named barrier 1);
        // returns 1 / scale, also left in slot ph % 4 for the output warps
        auto write_state = [&](int ph) -> float {
            float m = 0.f;
#pragma unroll
            for (int n = 0; n < 32; ++n) m = fmaxf(m, fabsf(st[n]));
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
            if (lane == 0) wmax[sw] = m;
            named_sync(1, 128);
            const float sc = scale_for(fmaxf(fmaxf(wmax[0], wmax[1]), fmaxf(wmax[2], wmax[3])));
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                uint32_t hh[4], ll[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) splith2(st[8 * c4 + 2 * e], st[8 * c4 + 2 * e + 1], sc, hh[e], ll[e]);
                const uint32_t off = swz(i, 4 * h + c4);
                sts128(sb + S::SH + off, hh[0], hh[1], hh[2], hh[3]);
                sts128(sb + S::SL + off, ll[0], ll[1], ll[2], ll[3]);
            }
            if (tid == 0) sinv[ph & 3] = 1.f / sc;
            fence_async_smem();
            fence_before_sync();
            named_sync(1, 128);   // (also: every warp has read wmax before the next write_state rewrites it)
            if (lane == 0) mbar_arrive(ready);
            return 1.f / sc;
        };
        float us = write_state(0);
        for (int j = 0; j < nb; ++j) {
            const int u = j % CS, b = j & 1;
            bool ok = true;
            if (lane == 0) ok = mbar_wait(&mD[b], (j >> 1) & 1, wl) && mbar_wait(&full[u], (j / CS) & 1, wl);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (named_sync_or(1, 128, !ok)) { failed = true; break; }   // one decision for the four warps
            fence_after_sync();
            float x[32];
            tmem_ld32(tmem + lane_base + 64 * b + 32 * h, x);
            const uint32_t stg = sb + u * S::STAGE;
            const float ud = lds_f32(stg + S::A_L + kChainTile) * us;   // 1 / (sP s_S)
            const uint32_t cb = stg + S::C_ + h * 8192;
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {   // c_j row i, columns 32 h + 4 q4 .. (fp32 swizzled box)
                float4 c4;
                asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(c4.x), "=f"(c4.y), "=f"(c4.z), "=f"(c4.w)
                             : "r"(cb + swz(i, q4)));
                st[4 * q4 + 0] = ud * x[4 * q4 + 0] + c4.x;
                st[4 * q4 + 1] = ud * x[4 * q4 + 1] + c4.y;
                st[4 * q4 + 2] = ud * x[4 * q4 + 2] + c4.z;
                st[4 * q4 + 3] = ud * x[4 * q4 + 3] + c4.w;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&freed[u]);
            if (j + 1 < nb) us = write_state(j + 1);   // the product of block j has read S_{j-1}: overwrite it with S_j
        }
        if (!failed && args.ST) {
            float4* dst = reinterpret_cast<float4*>(args.ST + (bh * GD + i) * GD + 32 * h);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) dst[q4] = make_float4(st[4 * q4], st[4 * q4 + 1], st[4 * q4 + 2], st[4 * q4 + 3]);
        }
        if (failed && lane == 0) atomicExch(args.status, (int)DPLR_ERR_TIMEOUT);
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

std::atomic<uint64_t> g_gsmem_set[2] = {{0}, {0}};
std::atomic<uint64_t> g_gcsmem_set{0};

template <class IT>
cudaError_t launch_generic(const Plan& pl, const GArgs& a, cudaStream_t s, int which) {
    cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(generic_chunk_kernel<IT>), GSmem::TOTAL,
                                        g_gsmem_set[which]);
    if (e != cudaSuccess) return e;
    const long long units = (long long)pl.BH * pl.nb;
    const long long grid = std::min<long long>(units, (long long)sm_count());
    generic_chunk_kernel<IT><<<(unsigned)grid, GT, GSmem::TOTAL, s>>>(pl, a);
    return cudaGetLastError();
}

}  // namespace

bool generic_tc_supported(const Plan& pl) {
    return pl.mode == DPLR_GENERIC && pl.dk == GD && pl.dv == GD && pl.r >= 1 && pl.r <= GMAXR && pl.p >= 0 &&
           pl.p <= GMAXP;
}

int generic_tc_block() { return GCW; }

// Workspace: the status word (256 bytes), then per unit [P_j; Q'_j] hi/lo, then per unit c_j.
void generic_tc_offsets(const Plan& pl, size_t* off_A, size_t* off_c, size_t* total) {
    const size_t units = (size_t)pl.BH * pl.nb;
    *off_A = 256;
    *off_c = *off_A + units * (size_t)kChainStride;
    *total = *off_c + units * (size_t)kChainC;
}

cudaError_t launch_generic_chunks(const Plan& pl, const ChunkMapArgs& m, void* workspace, cudaStream_t s) {
    if (pl.T == 0 || pl.nb == 0) return cudaSuccess;
    size_t oA, oC, total;
    generic_tc_offsets(pl, &oA, &oC, &total);
    char* ws = static_cast<char*>(workspace);
    GArgs a;
    a.q = m.q; a.A = m.A; a.Bm = m.Bm; a.K = m.K; a.V = m.V; a.decay = m.decay;
    a.o = m.o; a.Am = ws + oA; a.Cm = reinterpret_cast<float*>(ws + oC);
    a.status = reinterpret_cast<int*>(ws);
    return pl.bf16 ? launch_generic<__nv_bfloat16>(pl, a, s, 1) : launch_generic<float>(pl, a, s, 0);
}

cudaError_t launch_generic_chain(const Plan& pl, const float* S0, float* o, float* ST, void* workspace, cudaStream_t s) {
    size_t oA, oC, total;
    generic_tc_offsets(pl, &oA, &oC, &total);
    char* ws = static_cast<char*>(workspace);
    GCArgs a;
    a.S0 = S0; a.o = o; a.ST = ST;
    a.Am = reinterpret_cast<const unsigned char*>(ws + oA);
    a.status = reinterpret_cast<int*>(ws);
    CUtensorMap mC, mO;
    std::memset(&mC, 0, sizeof(mC));
    std::memset(&mO, 0, sizeof(mO));
    if (pl.nb > 0) {
        const uint64_t units = (uint64_t)pl.BH * (uint64_t)pl.nb;
        if (!tensor_map_2d(&mC, ws + oC, false, units * GD, GD, GD, 32) ||
            !tensor_map_2d(&mO, o, false, (uint64_t)pl.BH * pl.T, GD, GCW, 32))
            return cudaErrorInvalidValue;
    }
    cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(generic_chain_kernel), GCSmem::TOTAL, g_gcsmem_set);
    if (e != cudaSuccess) return e;
    generic_chain_kernel<<<(unsigned)pl.BH, CT, GCSmem::TOTAL, s>>>(pl, a, mC, mO);
    return cudaGetLastError();
}

}  // namespace dplr
