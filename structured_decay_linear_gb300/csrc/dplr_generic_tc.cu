// The generic DPLR mode (S_t = D_t S_{t-1} - A_t (B_t^T S_{t-1}) + K_t V_t^T, o_t = S_t^T q_t, with
// D_t = Diag(e^{decay_t}), rank r_ab <= 4 and r_kv <= 2) at dk = dv = 64, its WY blocks on the tensor cores:
// stage 1 of the two-stage chunkwise algorithm of "Householder-Diagonalized Linear Attention" (Key design 3:
// the rank-generalised WY representation, every token's r x r block treated as one element).
//
// One CTA step takes a block of 32 tokens of one head. With G_t the inclusive cumulative log-decay inside the
// block (one value per key channel), anchor a = G_32 / 2 and the block's rows s = t r + i (factors) and
// u = t p + i (writes):
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
// Z^T [QA, -QK]^T = [(QA Y)^T ; -O_j^T]. Every product runs on tcgen05 (kind::f16, fp32 accumulators in
// tensor memory) with both operands split into two bf16 terms, x = hi + lo, and three partial products
// (hi hi + hi lo + lo hi): a float64 emulation of these rounding points on the benchmark's generic
// distributions gives max |err| / RMS ~4e-5 for o, inside the fp32 tolerance of 1e-4, where one tf32 term for
// any operand already costs 3e-4 or more. The inverse is fp32: 16 x 16 diagonal blocks by substitution, merged
// 16 -> 32 -> 64 -> 128 with warp-level products in three tf32 terms (one term would cost 3.4e-4).
//
// The maps are written in fp32 for the fp32 scan over blocks (stage 2); O_j goes into o.
//
// Every wait is bounded by Plan::wait_cycles; a wait that gives up sets DPLR_ERR_TIMEOUT in the status word
// and the kernel drains its own products before it frees tensor memory.
#include <cuda_bf16.h>

#include <algorithm>

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
struct GSmem {
    static constexpr int A_H = 0;              // A~ hi [128][64]
    static constexpr int A_L = 16384;          // A~ lo
    static constexpr int B_H = 32768;          // B~ hi, then Y hi
    static constexpr int W_H = 49152;          // (G V) hi, then U hi: the second 64-column block of [B~ | G V]
    static constexpr int B_L = 65536;          // B~ lo, then Y lo
    static constexpr int W_L = 81920;          // (G V) lo, then U lo
    static constexpr int K_H = 98304;          // -K~ hi [64][64]
    static constexpr int K_L = 106496;         // -K~ lo (a 128-row read of -K~ hi covers both)
    static constexpr int ZERO = 114688;        // zeros [64][64] (the Y columns of Z's write rows; ends a 128-row read of -K~ lo)
    static constexpr int V_H = 122880;         // V hi [64][64]
    static constexpr int V_L = 131072;         // V lo
    static constexpr int Q_H = 139264;         // Q~ hi [32][64]
    static constexpr int Q_L = 143360;         // Q~ lo
    static constexpr int QX_H = 147456;        // [QA, -QK] hi: K-major [32][R + Pp], blocks of 64 columns (4 KB each)
    static constexpr int QX_L = 159744;        // lo
    static constexpr int X = 172032;           // fp32: the decay tables, then the inverse's blocks X11, X21, X22
    static constexpr int VEC = X + 3 * 64 * kLdX * 4;   // fp32 per channel: e^a, e^{G_32}
    static constexpr int BAR = VEC + 512;
    static constexpr int TOTAL = BAR + 64;
};
static_assert(GSmem::TOTAL <= 227 * 1024, "shared memory budget");
static_assert(GSmem::QX_L + 3 * 4096 <= GSmem::X, "QX tiles");
static_assert((33 + 32 + 33) * 64 * 4 <= 3 * 64 * kLdX * 4, "decay tables fit the inverse's region");

// Tensor-memory columns (512 allocated).
constexpr uint32_t TL = 0;      // L, then [Y | -U]                                            128
constexpr uint32_t TG = 128;    // -G (lane s, column u), then Z^T X                            64
constexpr uint32_t TW = 192;    // -(G V), then Z^T [QA, -QK]^T                                 64
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

// x (8 values) scaled by s (8 values, may be null: 1) and sign, split hi + lo, stored as one 16-byte chunk of
// row `row`, columns 8 ch .. 8 ch + 7, of the hi and lo tiles.
__device__ __forceinline__ void put8(uint32_t hi, uint32_t lo, int row, int ch, const float (&x)[8], const float* s,
                                     float sign) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float a = sign * x[2 * i] * (s ? s[2 * i] : 1.f), b = sign * x[2 * i + 1] * (s ? s[2 * i + 1] : 1.f);
        split2(a, b, h[i], l[i]);
    }
    const uint32_t off = swz(row, ch);
    sts128(hi + off, h[0], h[1], h[2], h[3]);
    sts128(lo + off, l[0], l[1], l[2], l[3]);
}

struct GArgs {
    const void* q; const void* A; const void* Bm; const void* K; const void* V;
    const float* decay;
    float* o; float* Pm; float* Cm; float* Qm; int* status;
};

__device__ __forceinline__ void prefetch_bulk_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(reinterpret_cast<uint64_t>(p)), "r"(bytes) : "memory");
}

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
    float* Xf = reinterpret_cast<float*>(smem + S::X);
    float* Gs = Xf;                 // [33][64] G_{t-1}: row t holds the prefix before token t (row 0 = 0)
    float* Er = Xf + 33 * 64;       // [32][64] e^{a - G_t}
    float* Ef = Xf + 65 * 64;       // [33][64] e^{G_{t-1} - a} (row 32: e^{G_31 - a})

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

    // ---- a2: cumulative log-decay per channel (identity padding past the end: log-decay 0), anchor, tables
    if (tid < GD) {
        const int c = tid;
        float ll[GCW];
#pragma unroll
        for (int t = 0; t < GCW; ++t) ll[t] = t < valid ? args.decay[(tok0 + t) * GD + c] : 0.f;
        float G = 0.f;
        Gs[c] = 0.f;
#pragma unroll
        for (int t = 0; t < GCW; ++t) {
            G += ll[t];
            Gs[(t + 1) * GD + c] = G;
        }
        ea[c] = __expf(0.5f * G);
        gam[c] = __expf(G);
    }
    __syncthreads();
    for (int i = tid; i < 33 * GD; i += GT) {
        const int c = i & (GD - 1);
        const float a = 0.5f * Gs[32 * GD + c];
        Ef[i] = __expf(Gs[i] - a);
        if (i >= GD) Er[i - GD] = __expf(a - Gs[i]);
    }
    __syncthreads();

    // ---- a1/a3: the decay-scaled factor tiles, hi + lo, from 32-byte row pieces (8 channels per item)
    for (int it = tid; it < 128 * 8 + 64 * 8 + 32 * 8; it += GT) {
        const int ch = it & 7;
        float x[8];
        if (it < 1024) {   // A~ and B~ rows s (zero past R or past the end)
            const int row = it >> 3, t = row / r, i = row - t * r;
            if (row < R && t < valid) {
                ld8(Ag + ((tok0 + t) * r + i) * GD + 8 * ch, x);
                put8(sb + S::A_H, sb + S::A_L, row, ch, x, Er + t * GD + 8 * ch, 1.f);
                ld8(Bg + ((tok0 + t) * r + i) * GD + 8 * ch, x);
                put8(sb + S::B_H, sb + S::B_L, row, ch, x, Ef + t * GD + 8 * ch, 1.f);
            } else {
                const uint32_t off = swz(row, ch);
                sts128(sb + S::A_H + off, 0u, 0u, 0u, 0u); sts128(sb + S::A_L + off, 0u, 0u, 0u, 0u);
                sts128(sb + S::B_H + off, 0u, 0u, 0u, 0u); sts128(sb + S::B_L + off, 0u, 0u, 0u, 0u);
            }
        } else if (it < 1536) {   // -K~ and V rows u
            const int row = (it - 1024) >> 3, t = p > 0 ? row / p : 0, i = row - t * p;
            if (row < Pp && t < valid) {
                ld8(Kg + ((tok0 + t) * p + i) * GD + 8 * ch, x);
                put8(sb + S::K_H, sb + S::K_L, row, ch, x, Er + t * GD + 8 * ch, -1.f);
                ld8(Vg + ((tok0 + t) * p + i) * GD + 8 * ch, x);
                put8(sb + S::V_H, sb + S::V_L, row, ch, x, nullptr, 1.f);
            } else {
                const uint32_t off = swz(row, ch);
                sts128(sb + S::K_H + off, 0u, 0u, 0u, 0u); sts128(sb + S::K_L + off, 0u, 0u, 0u, 0u);
                sts128(sb + S::V_H + off, 0u, 0u, 0u, 0u); sts128(sb + S::V_L + off, 0u, 0u, 0u, 0u);
            }
        } else {   // Q~ rows t
            const int t = (it - 1536) >> 3;
            if (t < valid) {
                ld8(q + (tok0 + t) * GD + 8 * ch, x);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = 0.f;
            }
            put8(sb + S::Q_H, sb + S::Q_L, t, ch, x, Ef + (t + 1) * GD + 8 * ch, 1.f);
        }
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();

    // ---- a4: L = B~ A~^T, -G = B~ (-K~)^T, QA^T = A~ Q~^T, -QK^T = (-K~) Q~^T (three terms each)
    if (warp == 0) {
        const uint32_t lead = lane == 0;
        const uint32_t loA[3] = {0, 0, 1}, loB[3] = {0, 1, 0};   // terms (A, B): (hi, hi), (hi, lo), (lo, hi)
#pragma unroll
        for (int term = 0; term < 3; ++term) {
            const uint32_t bt = sb + (loA[term] ? S::B_L : S::B_H);
            const uint32_t at = sb + (loB[term] ? S::A_L : S::A_H);
            const uint32_t kt = sb + (loB[term] ? S::K_L : S::K_H);
            const uint32_t qt = sb + (loB[term] ? S::Q_L : S::Q_H);
            const uint32_t ka = sb + (loA[term] ? S::K_L : S::K_H);
            const uint32_t aa = sb + (loA[term] ? S::A_L : S::A_H);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint32_t acc = (term > 0 || kk > 0);
                mma_ss_if(tmem + TL, smem_desc_sw128(bt + 32 * kk, 16, 1024), smem_desc_sw128(at + 32 * kk, 16, 1024),
                          idesc_bf16(128, 128, false, false), acc, lead);
                mma_ss_if(tmem + TQA, smem_desc_sw128(aa + 32 * kk, 16, 1024), smem_desc_sw128(qt + 32 * kk, 16, 1024),
                          idesc_bf16(128, 32, false, false), acc, lead);
                if (p > 0) {
                    mma_ss_if(tmem + TG, smem_desc_sw128(bt + 32 * kk, 16, 1024), smem_desc_sw128(kt + 32 * kk, 16, 1024),
                              idesc_bf16(128, Pp, false, false), acc, lead);
                    mma_ss_if(tmem + TQK, smem_desc_sw128(ka + 32 * kk, 16, 1024), smem_desc_sw128(qt + 32 * kk, 16, 1024),
                              idesc_bf16(128, 32, false, false), acc, lead);
                }
            }
        }
        commit_if(mb_mma, lead);
    }
    wait_mma();
    if (failed) break;

    // ---- L into the inverse's fp32 blocks (strict lower part by token); -G as a bf16 hi/lo tensor-memory operand
    // (strict: token of u before token of s); QA and -QK (inclusive) into the K-major [QA, -QK] tiles
    {
        const int ts = s / r;
        float x[32];
        tmem_ld32(tmem + lane_base + TL + 32 * qd, x);
        float* dst = nullptr;   // row s of X11 / X21 (columns 0-63), or of X22 (columns 64-127, shifted)
        if (qd < 2) dst = Xf + s * kLdX;
        else if (s >= 64) dst = Xf + (128 + (s - 64)) * kLdX - 64;
        if (dst) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                const int c = 32 * qd + i;
                float4 y;
                y.x = (c + 0) / r < ts ? x[i + 0] : 0.f;
                y.y = (c + 1) / r < ts ? x[i + 1] : 0.f;
                y.z = (c + 2) / r < ts ? x[i + 2] : 0.f;
                y.w = (c + 3) / r < ts ? x[i + 3] : 0.f;
                *reinterpret_cast<float4*>(dst + c) = y;
            }
        }
        if (p > 0 && qd < 2 && 32 * qd < Pp) {
            tmem_ld32(tmem + lane_base + TG + 32 * qd, x);
            uint32_t h[16], l[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int u = 32 * qd + 2 * i;
                split2(u / p < ts ? x[2 * i] : 0.f, (u + 1) / p < ts ? x[2 * i + 1] : 0.f, h[i], l[i]);
            }
            tmem_st16(tmem + lane_base + TGH + 16 * qd, h);
            tmem_st16(tmem + lane_base + TGL + 16 * qd, l);
        }
        const bool qa = qd == 2 && s < R, qk = qd == 3 && p > 0 && s < Pp;
        if (qa || qk) {
            tmem_ld32(tmem + lane_base + (qa ? TQA : TQK), x);
            const int k = qa ? s : R + s;             // row of Z this lane's values meet
            const int tk = qa ? ts : s / max(p, 1);  // its token
            const uint32_t col = (uint32_t)((k >> 6) * 4096 + ((k & 7) << 1));
            const int kc = (k & 63) >> 3;
#pragma unroll
            for (int t = 0; t < GCW; ++t) {
                uint16_t h, l;
                split1(tk <= t ? x[t] : 0.f, h, l);
                const uint32_t off = col + (uint32_t)(t * 128 + ((kc ^ (t & 7)) << 4));
                *reinterpret_cast<uint16_t*>(smem + S::QX_H + off) = h;
                *reinterpret_cast<uint16_t*>(smem + S::QX_L + off) = l;
            }
        }
    }
    tmem_wait_st();
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();

    // ---- a5: -(G V) on the tensor cores while the CUDA cores invert I + L
    if (p > 0 && warp == 0) {
        const uint32_t lead = lane == 0;
        const uint32_t idW = idesc_bf16(128, 64, false, true);
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
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) warp_mma_tf32_x<3>(X21 + 16 * (rb0 + rr) * kLdX, kLdX, X11 + 8 * cb, kLdX, 64, c[rr]);
        __syncthreads();
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) store_tile_16x8(X21 + 16 * (rb0 + rr) * kLdX + 8 * cb, kLdX, c[rr], 1.f);
        __syncthreads();
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) warp_mma_tf32_x<3>(X22 + 16 * (rb0 + rr) * kLdX, kLdX, X21 + 8 * cb, kLdX, 64, c[rr]);
        __syncthreads();
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) store_tile_16x8(X21 + 16 * (rb0 + rr) * kLdX + 8 * cb, kLdX, c[rr], -1.f);
        __syncthreads();
    }
    {   // M as bf16 hi / lo tensor-memory operands: thread (s, qd) takes columns 32 qd .. 32 qd + 31 of row s
        const float* row = nullptr;   // nullptr: zero (above the diagonal blocks)
        if (qd < 2) row = Xf + s * kLdX + 32 * qd;
        else if (s >= 64) row = Xf + (128 + (s - 64)) * kLdX + 32 * (qd - 2);
        uint32_t h[16], l[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float m0 = row ? row[2 * i] : 0.f, m1 = row ? row[2 * i + 1] : 0.f;
            split2(m0, m1, h[i], l[i]);
        }
        tmem_st16(tmem + lane_base + TMH + 16 * qd, h);
        tmem_st16(tmem + lane_base + TML + 16 * qd, l);
    }
    if (p > 0) {
        wait_mma();
        if (failed) break;
    }
    {   // -(G V) hi / lo into the second column block of [B~ | G V] (zero when there is no write term)
        float x[16];
        if (p > 0) {
            tmem_ld16(tmem + lane_base + TW + 16 * qd, x);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) x[i] = 0.f;
        }
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
            uint32_t h[4], l[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) split2(x[8 * ch + 2 * i], x[8 * ch + 2 * i + 1], h[i], l[i]);
            const uint32_t off = swz(s, 2 * qd + ch);
            sts128(sb + S::W_H + off, h[0], h[1], h[2], h[3]);
            sts128(sb + S::W_L + off, l[0], l[1], l[2], l[3]);
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
        const uint32_t idY = idesc_bf16(128, 128, false, true);
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

    {   // Z's factor rows [Y | U] hi / lo over [B~ | G V] (no longer read): thread (s, qd) takes 32 columns
        float x[32];
        tmem_ld32(tmem + lane_base + TL + 32 * qd, x);
        const float sg = qd < 2 ? 1.f : -1.f;
        const uint32_t th = sb + (qd < 2 ? S::B_H : S::W_H), tl = sb + (qd < 2 ? S::B_L : S::W_L);
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
            uint32_t h[4], l[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) split2(sg * x[8 * ch + 2 * i], sg * x[8 * ch + 2 * i + 1], h[i], l[i]);
            const uint32_t off = swz(s, 4 * (qd & 1) + ch);
            sts128(th + off, h[0], h[1], h[2], h[3]);
            sts128(tl + off, l[0], l[1], l[2], l[3]);
        }
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();

    // ---- a6/a7 (block part): Z^T X and Z^T [QA, -QK]^T over the factor rows, then the write rows
    if (warp == 0) {
        const uint32_t lead = lane == 0;
        const uint32_t idP = idesc_bf16(128, 64, true, true), idO = idesc_bf16(128, 32, true, false);
        const int nk = (R + Pp) / 16;
#pragma unroll
        for (int term = 0; term < 3; ++term) {
            const bool zl = term == 2, xl = term == 1;
            for (int kk = 0; kk < nk; ++kk) {
                uint64_t za, xb;
                if (kk < R / 16) {
                    za = smem_desc_sw128(sb + (zl ? S::B_L : S::B_H) + 2048 * kk, 16384, 1024);
                    xb = smem_desc_sw128(sb + (xl ? S::A_L : S::A_H) + 2048 * kk, 8192, 1024);
                } else {
                    const int k2 = kk - R / 16;
                    za = smem_desc_sw128(sb + S::ZERO + 2048 * k2, zl ? (S::V_L - S::ZERO) : (S::V_H - S::ZERO), 1024);
                    xb = smem_desc_sw128(sb + (xl ? S::K_L : S::K_H) + 2048 * k2, 8192, 1024);
                }
                const uint64_t qb = smem_desc_sw128(sb + (xl ? S::QX_L : S::QX_H) + (kk >> 2) * 4096 + (kk & 3) * 32, 16, 1024);
                const uint32_t acc = (term > 0 || kk > 0);
                mma_ss_if(tmem + TG, za, xb, idP, acc, lead);
                mma_ss_if(tmem + TW, za, qb, idO, acc, lead);
            }
        }
        commit_if(mb_mma, lead);
    }
    wait_mma();
    if (failed) break;

    // ---- epilogue: lane m < 64 holds column m of A~^T Y and of (QA Y)^T; lane 64 + n holds -(c_j e^{-a})^T and
    // -O_j^T for column n. Thread (m, qd) takes a quarter of the columns.
    {
        const size_t unit = bh * (size_t)nb + j;
        const int m = s;
        float x[16];
        tmem_ld16(tmem + lane_base + TG + 16 * qd, x);
        if (m < GD) {   // P_j[i][m] = [i == m] e^{G_32,i} - e^{a_i} (A~^T Y)[i][m] e^{a_m}
            float* Pcol = args.Pm + unit * (size_t)(GD * GD) + m;
            const float em = ea[m];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int i = 16 * qd + e;
                Pcol[(size_t)i * GD] = (i == m ? gam[i] : 0.f) - ea[i] * x[e] * em;
            }
        } else {        // c_j[i][n] = -e^{a_i} (Z^T X)[64 + n][i]
            const int n = m - GD;
            float* Ccol = args.Cm + unit * (size_t)(GD * GD) + n;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int i = 16 * qd + e;
                Ccol[(size_t)i * GD] = -ea[i] * x[e];
            }
        }
        if (qd < 2) {
            tmem_ld16(tmem + lane_base + TW + 16 * qd, x);
            if (m < GD) {   // Q'_j[t][c] = e^{a_c} (Q~[t][c] - (QA Y)[t][c]), c = m; Q~ from its hi and lo tiles
                const int c = m;
                const float ec = ea[c];
                float* Qcol = args.Qm + unit * (size_t)(GCW * GD) + c;
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int t = 16 * qd + e;
                    const uint32_t oq = swz(t, c >> 3) + ((c & 7) << 1);
                    const float qt = lds_bf16(sb + S::Q_H + oq) + lds_bf16(sb + S::Q_L + oq);
                    Qcol[(size_t)t * GD] = ec * (qt - x[e]);
                }
            } else {        // O_j[t][n] = -(Z^T [QA, -QK]^T)[64 + n][t]
                const int n = m - GD;
                float* ocol = args.o + tok0 * GD + n;
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int t = 16 * qd + e;
                    if (t < valid) ocol[(size_t)t * GD] = -x[e];
                }
            }
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
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

std::atomic<uint64_t> g_gsmem_set[2] = {{0}, {0}};

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

cudaError_t launch_generic_chunks(const Plan& pl, const ChunkMapArgs& m, void* workspace, cudaStream_t s) {
    if (pl.T == 0 || pl.nb == 0) return cudaSuccess;
    GArgs a;
    a.q = m.q; a.A = m.A; a.Bm = m.Bm; a.K = m.K; a.V = m.V; a.decay = m.decay;
    a.o = m.o; a.Pm = m.Pm; a.Cm = m.Cm; a.Qm = m.Qm;
    a.status = static_cast<int*>(workspace);
    return pl.bf16 ? launch_generic<__nv_bfloat16>(pl, a, s, 1) : launch_generic<float>(pl, a, s, 0);
}

}  // namespace dplr
