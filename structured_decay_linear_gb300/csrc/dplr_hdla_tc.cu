// HDLA (rank-2 decay P_t = (I - b k k^T) Diag(lambda_t) (I - b k k^T), write b k v^T) with bf16
// inputs and dk = dv = 128, on the tensor cores: the two-stage chunkwise algorithm of
// "Householder-Diagonalized Linear Attention" (Key design 3) with both stages on tcgen05.
//
// Stage 1, hdla_chunk_kernel: one CTA per (head, chunk of C = 64 tokens), all chunks in parallel.
// With G_t the inclusive cumulative log-decay of the chunk (one value per key channel), anchor
// a = G_C / 2, F_t = e^{G_t - a}, R_t = e^{a - G_t} (elementwise over channels) and the rank-2
// factors A_t = [k, Lambda k], B_t = [b Lambda k - b^2 (k^T Lambda k) k, b k] (Key design 2, written
// as D - A B^T), the chunk's rows s = 2t + i are
//
//   A~_{2t} = R_t k_t,  A~_{2t+1} = R_{t-1} k_t            (e^{-(G_t - a)} A_t; R_t lambda_t = R_{t-1})
//   B~_{2t} = b F_t k_t - b^2 c_t F_{t-1} k_t,  B~_{2t+1} = b F_{t-1} k_t   (e^{G_{t-1} - a} B_t)
//   Q~_t = F_t q_t,   c_t = k_t^T Lambda_t k_t
//
// and the chunk's exact maps follow from the UT/WY transform with the block operator that treats
// every token's 2 x 2 block as one element:
//
//   L   = strict_block_tril(B~ A~^T)            M = (I + L)^{-1}
//   Y   = M B~,  MW = M W  (W_{2t} = b_t v_t, W_{2t+1} = 0)
//   P_j = Diag(e^{G_C}) - Diag(e^a) (A~^T Y) Diag(e^a)      S_j = P_j S_{j-1} + c_j
//   c_j = Diag(e^a) A~^T MW
//   QA  = tril_incl(Q~ A~^T)   Q'_j = (Q~ - QA Y) Diag(e^a)   O_j = QA MW      o_t = Q'_t S_{j-1} + O_t
//
// The products run on tcgen05 (kind::f16, fp32 accumulators in tensor memory). Operands whose
// bf16 rounding alone would cost more than the output tolerance are split into two bf16 terms
// x = hi + lo (A~ and Q~ in QA and c, M in MW, MW and QA in O): a float64 emulation of these
// rounding points over the benchmark's distributions gives max |err| / RMS = 4.2e-3 for o, while a
// single bf16 term everywhere gives 4.2e-2. L, Y, P_j and QA Y tolerate one term. The inverse is
// fp32: 16 x 16 diagonal blocks by substitution, merged 16 -> 32 -> 64 -> 128 with warp-level tf32
// products. Stage 1 writes P_j (bf16), c_j (fp32) and Q'_j (bf16 hi and lo) to the workspace and
// O_j into o.
//
// Stage 2, hdla_chain_kernel: one CTA per (head, 32 state columns). It walks the chunks in order,
// S_j = P_j S_{j-1} + c_j with P_j as one bf16 term and S_{j-1} as bf16 hi + lo (the decay makes
// P_j contracting, so its rounding does not accumulate from chunk to chunk), and o_t += Q'_t S_{j-1}
// with both operands split into bf16 hi + lo. The kernel's warps take roles: two copy warps stage each chunk's
// maps by TMA (P_j and c_j, and Q'_j and O_j, after an L2 prefetch four chunks earlier), an issuing warp starts
// the chain's product of chunk j as soon as S_{j-1} is in place and then the output product of chunk j - 1, and
// four warps update the state and, a chunk behind, write the outputs while the tensor cores work. The state
// stays in registers in fp32; the maps arrive by TMA up to two chunks ahead.
//
// Every wait is bounded by Plan::wait_cycles; a wait that gives up sets DPLR_ERR_TIMEOUT in the
// status word and the kernel drains its own copies and products before it frees tensor memory.
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>

#include "dplr_internal.h"
#include "sm100_ops.cuh"
#include "tc_common.cuh"

namespace dplr {
namespace {

using namespace sm100;
using namespace tc;

constexpr int HD = 128;    // dk = dv
constexpr int HCK = 64;    // tokens per chunk
constexpr int K1T = 512;   // threads of the chunk kernel: four per tensor-memory lane

// ================================================================================================
// Stage 1: chunk maps
// ================================================================================================

// Shared memory (bytes from the 1024-aligned base).
struct K1Smem {
    static constexpr int A_HI = 0;                // A~ hi: bf16 [128][128], swizzled
    static constexpr int A_LO = A_HI + 32768;     // A~ lo
    static constexpr int BT = A_LO + 32768;       // B~ (bf16); later Y
    static constexpr int Q_HI = BT + 32768;       // Q~ hi: bf16 [64][128]
    static constexpr int Q_LO = Q_HI + 16384;     // Q~ lo
    static constexpr int V = Q_LO + 16384;        // v: bf16 [64][128] (TMA); later QA hi [128][64]
    static constexpr int R0 = V + 16384;          // 64 KB shared by, in turn:
    static constexpr int K_ = R0;                 //   k [64][128] bf16 (TMA)
    static constexpr int Q_ = R0 + 16384;         //   q [64][128] bf16 (TMA)
    static constexpr int LAM = R0 + 32768;        //   log lambda [64][128] fp32 (TMA)
    static constexpr int X22 = R0 + 128 * kLdX * 4;  //   the inverse's fp32 blocks X11, X21, X22 (64 x kLdX each)
    static constexpr int MB_HI = R0;              //   M Diag(beta) restricted to the even columns, hi / lo:
    static constexpr int MB_LO = R0 + 16384;      //   bf16 [128][64]
    static constexpr int QA_LO = R0 + 32768;      //   QA^T lo: bf16 [128][64]
    static constexpr int VEC = R0 + 65536;        // fp32 vectors (see below)
    static constexpr int BAR = VEC + 6144;        // mbarriers and the tensor-memory address (vectors: 1408 floats)
    static constexpr int TOTAL = BAR + 64;
};
static_assert(K1Smem::X22 + 64 * kLdX * 4 <= K1Smem::R0 + 65536, "inverse blocks fit the shared region");
static_assert(K1Smem::TOTAL <= 227 * 1024, "shared memory budget");

// Tensor-memory columns of the chunk kernel (512 allocated).
constexpr uint32_t TL = 0;       // L, then Y, then the product A~^T Y                 128
constexpr uint32_t TQA = 128;    // QA^T (lane s, column t), then O^T = (QA MW)^T          64
constexpr uint32_t TM = 192;     // M as a bf16 A operand, then Zq = (QA Y)^T             64
constexpr uint32_t TMW = 256;    // MW^T (lane n, column s), then c^T                      128
constexpr uint32_t TMWH = 384;   // MW^T hi (bf16 A operand)                               64
constexpr uint32_t TMWL = 448;   // MW^T lo                                                 64

struct K1Args {
    const __nv_bfloat16* q; const __nv_bfloat16* k; const __nv_bfloat16* v;
    const float* decay; const float* beta;
    float* o; __nv_bfloat16* P; float* Cm; __nv_bfloat16* Qm; int* status;
};

// Persistent: CTA b takes the units b, b + gridDim.x, ... in head-major order (chunk j of head bh is unit
// bh * NC + j), so the CTAs running at once read neighbouring chunks. The next unit's inputs are prefetched
// into L2 while the current one is computed.
__global__ void __launch_bounds__(K1T, 1)
hdla_chunk_kernel(Plan pl, K1Args args, const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_l,
                  const __grid_constant__ CUtensorMap tm_P, const __grid_constant__ CUtensorMap tm_Q) {
    using S = K1Smem;
    extern __shared__ __align__(1024) unsigned char smem[];
    const uint32_t sb = smem_addr(smem);
    if (sb & 1023u) {   // the swizzled tiles need 1024-byte alignment
        if (threadIdx.x == 0) atomicExch(args.status, (int)DPLR_ERR_CUDA);
        return;
    }
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::BAR);
    uint64_t* mb_tma = bars + 0;
    uint64_t* mb_mma = bars + 1;
    uint64_t* mb_drain = bars + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 3);
    float* vec = reinterpret_cast<float*>(smem + S::VEC);
    float* cdot = vec;          // [64]  k_t^T Lambda_t k_t
    float* betav = vec + 64;    // [64]
    float* ea = vec + 128;      // [128] e^{a}
    float* gam = vec + 256;     // [128] e^{G_C}
    float* gq = vec + 384;      // [7][128] G after tokens 7, 15, ..., 55 (the start of token eighths 1-7)
    float* av = vec + 1280;     // [128] a = G_C / 2

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int NC = (pl.T + HCK - 1) / HCK;
    const long long total = (long long)pl.BH * NC;
    const long long wl = pl.wait_cycles;

    if (tid == 0) {
        mbar_init(mb_tma, 1);
        mbar_init(mb_mma, 1);
        mbar_init(mb_drain, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(tmem_holder, 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_holder;
    uint32_t mma_phase = 0;   // phases of mb_mma completed so far
    uint32_t tma_phase = 0;   // phases of mb_tma completed so far
    bool failed = false;
    bool tma_pending = false;
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const int s = tid & 127;   // tensor-memory lane of this thread (row of the chunk's 128-row tiles)
    const int qd = tid >> 7;   // which quarter of the columns this thread takes in the lane-mapped phases

    // the TMA copies of unit ux's k, q, v (into R0 and V) and log-decay (thread 0)
    auto stage_in = [&](long long ux) {
        if (tid != 0) return;
        const int jx = static_cast<int>(ux % NC);
        const int y = static_cast<int>((ux / NC) * pl.T + (long long)jx * HCK);
        mbar_expect_tx(mb_tma, 3 * 16384 + 32768);
        for (int h = 0; h < 2; ++h) {
            tma_load_2d(smem + S::K_ + h * 8192, &tm_k, 64 * h, y, mb_tma);
            tma_load_2d(smem + S::Q_ + h * 8192, &tm_q, 64 * h, y, mb_tma);
            tma_load_2d(smem + S::V + h * 8192, &tm_v, 64 * h, y, mb_tma);
        }
        for (int b = 0; b < 4; ++b) tma_load_2d(smem + S::LAM + b * 8192, &tm_l, 32 * b, y, mb_tma);
    };
    bool staged = false;   // this unit's copies were issued during the previous unit
  for (long long uidx = blockIdx.x; uidx < total && !failed; uidx += gridDim.x) {
    const int j = static_cast<int>(uidx % NC);
    const size_t bh = static_cast<size_t>(uidx / NC);
    const int valid = min(HCK, pl.T - j * HCK);
    const size_t tok0 = bh * (size_t)pl.T + (size_t)j * HCK;
    const size_t unit = (size_t)j * pl.BH + bh;   // maps are stored chunk-major: a chunk's heads side by side
    const bool full = valid == HCK;
    if (tid == 0 && uidx + gridDim.x < total) {   // the next unit's inputs into L2
        const long long nx = uidx + gridDim.x;
        const int jn = static_cast<int>(nx % NC);
        if (pl.T - jn * HCK >= HCK) {
            const int y = static_cast<int>((nx / NC) * pl.T + (long long)jn * HCK);
            for (int h = 0; h < 2; ++h) {
                prefetch_l2_tile(&tm_k, 64 * h, y);
                prefetch_l2_tile(&tm_q, 64 * h, y);
                prefetch_l2_tile(&tm_v, 64 * h, y);
            }
            for (int b = 0; b < 4; ++b) prefetch_l2_tile(&tm_l, 32 * b, y);
        }
    }

    // ---- a1: stage k, q, v and the log-decay of the chunk (TMA, issued during the previous unit's epilogue when
    // there was one; plain loads for a ragged chunk)
    if (full) {
        if (!staged) stage_in(uidx);
    } else {   // identity padding past the end: k = q = v = 0, log-decay 0, beta 0
        for (int i = tid; i < HCK * 16; i += K1T) {
            const int t = i >> 4, cb = i & 15;
            uint4 zk = make_uint4(0, 0, 0, 0), zq = zk, zv = zk;
            if (t < valid) {
                const size_t g = (tok0 + t) * HD + 8 * cb;
                zk = *reinterpret_cast<const uint4*>(args.k + g);
                zq = *reinterpret_cast<const uint4*>(args.q + g);
                zv = *reinterpret_cast<const uint4*>(args.v + g);
            }
            const uint32_t off = (uint32_t)((cb >> 3) * 8192) + swz(t, cb & 7);
            sts128(sb + S::K_ + off, zk.x, zk.y, zk.z, zk.w);
            sts128(sb + S::Q_ + off, zq.x, zq.y, zq.z, zq.w);
            sts128(sb + S::V + off, zv.x, zv.y, zv.z, zv.w);
        }
        for (int i = tid; i < HCK * 32; i += K1T) {
            const int t = i >> 5, cb = i & 31;
            float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
            if (t < valid) z = *reinterpret_cast<const float4*>(args.decay + (tok0 + t) * HD + 4 * cb);
            const uint32_t off = (uint32_t)((cb >> 3) * 8192) + swz(t, cb & 7);
            sts128(sb + S::LAM + off, __float_as_uint(z.x), __float_as_uint(z.y), __float_as_uint(z.z), __float_as_uint(z.w));
        }
        fence_async_smem();   // v is read by the tensor cores
    }
    if (tid < HCK) betav[tid] = tid < valid ? args.beta[tok0 + tid] : 0.f;
    if (full) {
        tma_pending = true;
        const bool ok = mbar_wait(mb_tma, tma_phase & 1, wl);
        if (__syncthreads_or(!ok)) failed = true;
        else { tma_pending = false; ++tma_phase; }
    } else {
        __syncthreads();
    }

    if (!failed) {
        // ---- a2: per-channel prefixes of the log-decay at every eighth of the chunk and at its end (warps 0-3),
        // and c_t = k_t^T Lambda_t k_t per token (warps 4-11, eight tokens each)
        if (warp < 4) {
            const int c = tid;
            float G = 0.f;
#pragma unroll
            for (int e8 = 0; e8 < 8; ++e8) {
#pragma unroll
                for (int t = 8 * e8; t < 8 * e8 + 8; ++t) G += lds_f32(sb + S::LAM + sw_f32(t, c, HCK));
                if (e8 < 7) gq[128 * e8 + c] = G;
            }
            const float a = 0.5f * G;
            av[c] = a;
            ea[c] = __expf(a);
            gam[c] = __expf(G);
        } else if (warp < 12) {
            for (int tt = 0; tt < 8; ++tt) {
                const int t = 8 * (warp - 4) + tt;
                float acc = 0.f;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int c = lane + 32 * i;
                    const float kk = lds_bf16(sb + S::K_ + sw_bf16(t, c, HCK));
                    acc = fmaf(__expf(lds_f32(sb + S::LAM + sw_f32(t, c, HCK))) * kk, kk, acc);
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
                if (lane == 0) cdot[t] = acc;
            }
        }
        if (tid == 0) bulk_wait_read();   // the previous unit's P_j and Q'_j have left A~ hi / lo
        __syncthreads();

        // ---- a3: the decay-scaled factor tiles. Warp w takes key channels 64 (w % 2) .. + 63 (two per lane,
        // stored as bf16 pairs) and tokens 8 (w / 2) .. + 7, starting from that eighth's prefix of G.
        {
            const int c0 = 64 * (warp & 1) + 2 * lane, e8 = warp >> 1;
            const float a0 = av[c0], a1 = av[c0 + 1];
            float G0 = e8 ? gq[128 * (e8 - 1) + c0] : 0.f, G1 = e8 ? gq[128 * (e8 - 1) + c0 + 1] : 0.f;
            float Fp0 = __expf(G0 - a0), Fp1 = __expf(G1 - a1), Rp0 = __expf(a0 - G0), Rp1 = __expf(a1 - G1);
            // byte offsets of channel c0 inside a swizzled row, for each row residue mod 8
            const uint32_t col_f32 = (uint32_t)((c0 >> 5) * (HCK * 128) + ((c0 & 3) << 2));
            const int chunk16 = (c0 & 63) >> 3, chunk32 = (c0 & 31) >> 2;
#pragma unroll
            for (int tt = 0; tt < 8; ++tt) {
                const int t = 8 * e8 + tt;   // t % 8 == tt
                const uint32_t rowl = (uint32_t)(t * 128) + (uint32_t)(((chunk32 ^ tt)) << 4) + col_f32;
                const uint32_t rowb = (uint32_t)((c0 >> 6) * (HCK * 128) + t * 128 + ((chunk16 ^ tt) << 4) + ((c0 & 7) << 1));
                const float2 ll = *reinterpret_cast<const float2*>(smem + S::LAM + rowl);
                const uint32_t kb = *reinterpret_cast<const uint32_t*>(smem + S::K_ + rowb);
                const uint32_t qb = *reinterpret_cast<const uint32_t*>(smem + S::Q_ + rowb);
                const float k0 = __uint_as_float(kb << 16), k1 = __uint_as_float(kb & 0xFFFF0000u);
                const float q0 = __uint_as_float(qb << 16), q1 = __uint_as_float(qb & 0xFFFF0000u);
                G0 += ll.x;
                G1 += ll.y;
                const float F0 = __expf(G0 - a0), F1 = __expf(G1 - a1), R0 = __expf(a0 - G0), R1 = __expf(a1 - G1);
                const float b = betav[t], bcd = b * cdot[t];
                const float bt10 = b * Fp0 * k0, bt11 = b * Fp1 * k1;
                uint32_t h, l;
                // rows 2t and 2t + 1 of the 128-row tiles (2t % 8 = (2 tt) % 8), row t of the 64-row tile
                const uint32_t o0 = (uint32_t)((c0 >> 6) * 16384 + (2 * t) * 128 + ((chunk16 ^ ((2 * tt) & 7)) << 4) + ((c0 & 7) << 1));
                const uint32_t o1 = (uint32_t)((c0 >> 6) * 16384 + (2 * t + 1) * 128 + ((chunk16 ^ ((2 * tt + 1) & 7)) << 4) + ((c0 & 7) << 1));
                split2(R0 * k0, R1 * k1, h, l);            // A~ row 2t
                *reinterpret_cast<uint32_t*>(smem + S::A_HI + o0) = h;
                *reinterpret_cast<uint32_t*>(smem + S::A_LO + o0) = l;
                split2(Rp0 * k0, Rp1 * k1, h, l);          // A~ row 2t + 1
                *reinterpret_cast<uint32_t*>(smem + S::A_HI + o1) = h;
                *reinterpret_cast<uint32_t*>(smem + S::A_LO + o1) = l;
                *reinterpret_cast<uint32_t*>(smem + S::BT + o0) = pack_bf16(b * F0 * k0 - bcd * bt10, b * F1 * k1 - bcd * bt11);
                *reinterpret_cast<uint32_t*>(smem + S::BT + o1) = pack_bf16(bt10, bt11);
                split2(F0 * q0, F1 * q1, h, l);            // Q~ row t
                *reinterpret_cast<uint32_t*>(smem + S::Q_HI + rowb) = h;
                *reinterpret_cast<uint32_t*>(smem + S::Q_LO + rowb) = l;
                Fp0 = F0; Fp1 = F1; Rp0 = R0; Rp1 = R1;
            }
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();

        // ---- a4: L = B~ A~^T and QA^T = A~ Q~^T (three terms) on the tensor cores
        if (warp == 0) {
            const uint32_t lead = lane == 0;
            const uint32_t idL = idesc_bf16(128, 128, false, false);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                mma_ss_if(tmem + TL, smem_desc_sw128(sb + S::BT + off, 16, 1024), smem_desc_sw128(sb + S::A_HI + off, 16, 1024),
                          idL, kk > 0, lead);
            }
            const uint32_t idQ = idesc_bf16(128, 64, false, false);
            const uint32_t aop[3] = {sb + S::A_HI, sb + S::A_LO, sb + S::A_HI};
            const uint32_t bop[3] = {sb + S::Q_HI, sb + S::Q_HI, sb + S::Q_LO};
#pragma unroll
            for (int term = 0; term < 3; ++term)
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ss_if(tmem + TQA, smem_desc_sw128(aop[term] + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                              smem_desc_sw128(bop[term] + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024), idQ,
                              (term > 0 || kk > 0), lead);
            commit_if(mb_mma, lead);
        }
        {
            const bool ok = mbar_wait(mb_mma, mma_phase & 1, wl);
            ++mma_phase;
            if (__syncthreads_or(!ok)) failed = true;
            fence_after_sync();
        }
    }

    if (!failed) {
        // ---- a5: L into the inverse's fp32 blocks (strict lower part by token), then M = (I + L)^{-1}
        {
            float* X = reinterpret_cast<float*>(smem + S::R0);
            float x[32];
            tmem_ld32(tmem + lane_base + TL + 32 * qd, x);
            const int c0 = 32 * qd;
            float* dst = nullptr;   // row s of X11 / X21 (columns 0-63), or of X22 (columns 64-127, shifted)
            if (qd < 2) dst = X + s * kLdX;
            else if (s >= 64) dst = X + (128 + (s - 64)) * kLdX - 64;
            if (dst) {
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    const int c = c0 + i;
                    float4 y;
                    y.x = ((c + 0) >> 1) < (s >> 1) ? x[i + 0] : 0.f;
                    y.y = ((c + 1) >> 1) < (s >> 1) ? x[i + 1] : 0.f;
                    y.z = ((c + 2) >> 1) < (s >> 1) ? x[i + 2] : 0.f;
                    y.w = ((c + 3) >> 1) < (s >> 1) ? x[i + 3] : 0.f;
                    *reinterpret_cast<float4*>(dst + c) = y;
                }
            }
        }
        __syncthreads();
        {
            float* X = reinterpret_cast<float*>(smem + S::R0);
            if (warp < 8) inv64_inplace(X, tid, 1);                  // M11 in place of L11
            else inv64_inplace(X + 128 * kLdX, tid - 256, 2);        // M22 in place of L22
            __syncthreads();
            // 64 -> 128: M21 = -M22 (L21 M11), 32 tiles of 16 x 8 per product: warp w takes column block
            // w % 8 and row blocks 2 (w / 8), 2 (w / 8) + 1
            float* X11 = X;
            float* X21 = X + 64 * kLdX;
            float* X22 = X + 128 * kLdX;
            const int cb = warp & 7, rb0 = 2 * (warp >> 3);
            float c[2][4];
#pragma unroll
            for (int r = 0; r < 2; ++r) warp_mma_tf32_rn(X21 + 16 * (rb0 + r) * kLdX, kLdX, X11 + 8 * cb, kLdX, 64, c[r]);
            __syncthreads();
#pragma unroll
            for (int r = 0; r < 2; ++r) store_tile_16x8(X21 + 16 * (rb0 + r) * kLdX + 8 * cb, kLdX, c[r], 1.f);
            __syncthreads();
#pragma unroll
            for (int r = 0; r < 2; ++r) warp_mma_tf32_rn(X22 + 16 * (rb0 + r) * kLdX, kLdX, X21 + 8 * cb, kLdX, 64, c[r]);
            __syncthreads();
#pragma unroll
            for (int r = 0; r < 2; ++r) store_tile_16x8(X21 + 16 * (rb0 + r) * kLdX + 8 * cb, kLdX, c[r], -1.f);
            __syncthreads();
        }

        // ---- M as the bf16 A operand of Y (tensor memory), and M Diag(beta) on the even columns (the columns
        // that meet W) as hi + lo tiles for MW. Thread (s, qd) takes columns 32 qd .. 32 qd + 31 of row s of M.
        {
            const float* X = reinterpret_cast<const float*>(smem + S::R0);
            const float* row = nullptr;   // nullptr: zero (above the diagonal blocks)
            if (qd < 2) row = X + s * kLdX + 32 * qd;                       // X11 row s or X21 row s - 64
            else if (s >= 64) row = X + (128 + (s - 64)) * kLdX + 32 * (qd - 2);   // X22 row s - 64
            uint32_t pk[16];
            uint32_t mbh[8], mbl[8];
#pragma unroll
            for (int i = 0; i < 16; ++i) pk[i] = row ? pack_bf16(row[2 * i], row[2 * i + 1]) : 0u;
            // M Diag(beta) on columns 2t of M, t = 16 qd + 2 i2, 16 qd + 2 i2 + 1 (pairs of t)
#pragma unroll
            for (int i2 = 0; i2 < 8; ++i2) {
                const float m0 = row ? row[4 * i2] : 0.f, m1 = row ? row[4 * i2 + 2] : 0.f;
                split2(m0 * betav[16 * qd + 2 * i2], m1 * betav[16 * qd + 2 * i2 + 1], mbh[i2], mbl[i2]);
            }
            tmem_st16(tmem + lane_base + TM + 16 * qd, pk);
            tmem_wait_st();
            __syncthreads();   // every row of M read: its region takes the M Diag(beta) tiles
#pragma unroll
            for (int ch = 0; ch < 2; ++ch) {
                const uint32_t off = swz(s, 2 * qd + ch);   // columns t = 16 qd + 8 ch ..
                sts128(sb + S::MB_HI + off, mbh[4 * ch], mbh[4 * ch + 1], mbh[4 * ch + 2], mbh[4 * ch + 3]);
                sts128(sb + S::MB_LO + off, mbl[4 * ch], mbl[4 * ch + 1], mbl[4 * ch + 2], mbl[4 * ch + 3]);
            }
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();

        // ---- a5 (applications): Y = M B~ and MW^T = V^T (M Diag(beta))^T on the tensor cores
        if (warp == 0) {
            const uint32_t lead = lane == 0;
            const uint32_t idY = idesc_bf16(128, 128, false, true);
            const uint64_t bY = smem_desc_sw128(sb + S::BT, 16384, 1024);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) mma_ts_if(tmem + TL, tmem + TM + 8 * kk, dadd(bY, 2048 * kk), idY, kk > 0, lead);
            const uint32_t idW = idesc_bf16(128, 128, true, false);
            const uint64_t aW = smem_desc_sw128(sb + S::V, 8192, 1024);
#pragma unroll
            for (int term = 0; term < 2; ++term) {
                const uint64_t bW = smem_desc_sw128(sb + (term ? S::MB_LO : S::MB_HI), 16, 1024);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ss_if(tmem + TMW, dadd(aW, 2048 * kk), dadd(bW, 32 * kk), idW, (term > 0 || kk > 0), lead);
            }
            commit_if(mb_mma, lead);
        }
        {
            const bool ok = mbar_wait(mb_mma, mma_phase & 1, wl);
            ++mma_phase;
            if (__syncthreads_or(!ok)) failed = true;
            fence_after_sync();
        }
    }

    if (!failed) {
        // ---- operand tiles for the last products: Y (bf16, over B~), MW^T hi/lo (tensor memory),
        // QA^T hi/lo (masked t >= token of s); thread (s, qd) takes a quarter of the columns
        {
            float x[32];
            tmem_ld32(tmem + lane_base + TL + 32 * qd, x);
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                const int c = 32 * qd + 8 * ch;
                sts128(sb + S::BT + sw_bf16(s, c, 128), pack_bf16(x[8 * ch + 0], x[8 * ch + 1]),
                       pack_bf16(x[8 * ch + 2], x[8 * ch + 3]), pack_bf16(x[8 * ch + 4], x[8 * ch + 5]),
                       pack_bf16(x[8 * ch + 6], x[8 * ch + 7]));
            }
            tmem_ld32(tmem + lane_base + TMW + 32 * qd, x);
            uint32_t h[16], l[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) split2(x[2 * i], x[2 * i + 1], h[i], l[i]);
            tmem_st16(tmem + lane_base + TMWH + 16 * qd, h);
            tmem_st16(tmem + lane_base + TMWL + 16 * qd, l);
        }
        {
            float x[16];
            tmem_ld16(tmem + lane_base + TQA + 16 * qd, x);
            const int tok_s = s >> 1;
#pragma unroll
            for (int ch = 0; ch < 2; ++ch) {
                uint32_t h[4], l[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int t0 = 16 * qd + 8 * ch + 2 * i;
                    split2(t0 >= tok_s ? x[8 * ch + 2 * i] : 0.f, t0 + 1 >= tok_s ? x[8 * ch + 2 * i + 1] : 0.f, h[i], l[i]);
                }
                const uint32_t off = swz(s, 2 * qd + ch);
                sts128(sb + S::V + off, h[0], h[1], h[2], h[3]);       // QA hi over v
                sts128(sb + S::QA_LO + off, l[0], l[1], l[2], l[3]);
            }
        }
        tmem_wait_st();
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();

        // ---- a6/a7 (chunk part): A~^T Y, c^T = MW^T A~ (3 terms), Zq = Y^T QA^T, O^T = MW^T QA^T (3 terms)
        if (warp == 0) {
            const uint32_t lead = lane == 0;
            const uint32_t idP = idesc_bf16(128, 128, true, true);
            const uint64_t aP = smem_desc_sw128(sb + S::A_HI, 16384, 1024), bP = smem_desc_sw128(sb + S::BT, 16384, 1024);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) mma_ss_if(tmem + TL, dadd(aP, 2048 * kk), dadd(bP, 2048 * kk), idP, kk > 0, lead);
            const uint32_t idC = idesc_bf16(128, 128, false, true);
            const uint32_t ta[3] = {tmem + TMWH, tmem + TMWL, tmem + TMWH};
            const uint32_t sbB[3] = {sb + S::A_HI, sb + S::A_HI, sb + S::A_LO};
#pragma unroll
            for (int term = 0; term < 3; ++term) {
                const uint64_t b = smem_desc_sw128(sbB[term], 16384, 1024);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ts_if(tmem + TMW, ta[term] + 8 * kk, dadd(b, 2048 * kk), idC, (term > 0 || kk > 0), lead);
            }
            const uint32_t idZ = idesc_bf16(128, 64, true, true);
            const uint64_t aZ = smem_desc_sw128(sb + S::BT, 16384, 1024), bZ = smem_desc_sw128(sb + S::V, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) mma_ss_if(tmem + TM, dadd(aZ, 2048 * kk), dadd(bZ, 2048 * kk), idZ, kk > 0, lead);
            const uint32_t idO = idesc_bf16(128, 64, false, true);
            const uint32_t sbQ[3] = {sb + S::V, sb + S::V, sb + S::QA_LO};
#pragma unroll
            for (int term = 0; term < 3; ++term) {
                const uint64_t b = smem_desc_sw128(sbQ[term], 16, 1024);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ts_if(tmem + TQA, ta[term] + 8 * kk, dadd(b, 2048 * kk), idO, (term > 0 || kk > 0), lead);
            }
            commit_if(mb_mma, lead);
        }
        {
            const bool ok = mbar_wait(mb_mma, mma_phase & 1, wl);
            ++mma_phase;
            if (__syncthreads_or(!ok)) failed = true;
            fence_after_sync();
        }
    }
    // the last products have read R0 and V: the next unit's copies can land there during the epilogue
    staged = false;
    if (!failed && uidx + gridDim.x < total) {
        const long long nx = uidx + gridDim.x;
        if (pl.T - static_cast<int>(nx % NC) * HCK >= HCK) {
            stage_in(nx);
            staged = true;
            tma_pending = true;
        }
    }

    if (!failed) {
        // ---- epilogues: thread (s, qd) takes a quarter of the columns of each result. P_j and Q'_j go to
        // shared staging tiles over A~ hi and A~ lo (no longer read by then) and leave by TMA bulk stores;
        // c_j and O_j are stored directly, a column per thread.
        {   // P_j row i = s: bf16 [128][128]
            const int i = s;
            const float ei = ea[i], gi = gam[i];
            float x[32];
            tmem_ld32(tmem + lane_base + TL + 32 * qd, x);
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int k0 = 32 * qd + 8 * ch + 2 * e;
                    const float p0 = (k0 == i ? gi : 0.f) - ei * x[8 * ch + 2 * e] * ea[k0];
                    const float p1 = (k0 + 1 == i ? gi : 0.f) - ei * x[8 * ch + 2 * e + 1] * ea[k0 + 1];
                    w[e] = pack_bf16(p0, p1);
                }
                sts128(sb + S::A_HI + sw_bf16(i, 32 * qd + 8 * ch, 128), w[0], w[1], w[2], w[3]);
            }
        }
        {   // c_j column n = s: c[i][n] = e^{a_i} (MW^T A~)[n][i] (each warp store writes 128 contiguous bytes)
            const int n = s;
            float* Ccol = args.Cm + unit * (size_t)(HD * HD) + n;
            float x[32];
            tmem_ld32(tmem + lane_base + TMW + 32 * qd, x);
#pragma unroll
            for (int i2 = 0; i2 < 32; ++i2) Ccol[(size_t)(32 * qd + i2) * HD] = ea[32 * qd + i2] * x[i2];
        }
        {   // Q'[t][c] = e^{a_c} (Q~[t][c] - Zq[c][t]), c = s, t = 16 qd ..; Q~ from its hi and lo tiles. Q'_j is
            // a bf16 [128][128] block whose rows 32 g .. 32 g + 15 hold the hi parts of tokens 16 g .. 16 g + 15
            // and rows 32 g + 16 .. 32 g + 31 their lo parts: one product of the block with S_{j-1} then puts a
            // token's two partial outputs in lanes l and l + 16 of the same warp.
            const int c = s;
            const float ec = ea[c];
            float x[16];
            tmem_ld16(tmem + lane_base + TM + 16 * qd, x);
#pragma unroll
            for (int i2 = 0; i2 < 16; ++i2) {
                const int t = 16 * qd + i2;
                const uint32_t oq = sw_bf16(t, c, HCK);
                const float qt = lds_bf16(sb + S::Q_HI + oq) + lds_bf16(sb + S::Q_LO + oq);
                uint16_t h, l;
                split1(ec * (qt - x[i2]), h, l);
                *reinterpret_cast<uint16_t*>(smem + S::A_LO + sw_bf16(32 * qd + i2, c, 128)) = h;   // g = t / 16 = qd
                *reinterpret_cast<uint16_t*>(smem + S::A_LO + sw_bf16(32 * qd + 16 + i2, c, 128)) = l;
            }
        }
        {   // O_j column n = s, tokens t = 16 qd ..
            const int n = s;
            float x[16];
            tmem_ld16(tmem + lane_base + TQA + 16 * qd, x);
            float* ocol = args.o + tok0 * HD + n;
#pragma unroll
            for (int i2 = 0; i2 < 16; ++i2)
                if (16 * qd + i2 < valid) ocol[(size_t)(16 * qd + i2) * HD] = x[i2];
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        if (tid == 0) {   // (the next unit waits for these reads before its factor build rewrites A~)
            const int yu = static_cast<int>(unit * HD);
            for (int h = 0; h < 2; ++h) {
                tma_store_2d(&tm_P, 64 * h, yu, sb + S::A_HI + h * 16384);
                tma_store_2d(&tm_Q, 64 * h, yu, sb + S::A_LO + h * 16384);
            }
            bulk_commit();
        }
    }
  }   // units

    if (failed) {
        if (tid == 0) {
            atomicExch(args.status, (int)DPLR_ERR_TIMEOUT);
            // no copy may land after the CTA exits, and no product may touch freed tensor memory
            if (tma_pending) mbar_wait(mb_tma, tma_phase & 1, 400000000LL);
            mma_commit(mb_drain);   // tracks every product issued by this thread
            mbar_wait(mb_drain, 0, 400000000LL);
        }
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
// Stage 2: the chain over chunks, per (head, block of state columns)
// ================================================================================================

constexpr int NV = 32;       // state columns per chain CTA
constexpr int K2T = 224;     // warps 0-3: the state (thread = key channel = tensor-memory lane); 4: issuer;
                             // 5: copies of P_j and c_j; 6: copies of Q'_j and O_j
constexpr int K2PF = 4;      // chunks between the L2 prefetch of a chunk's maps and their copy into shared memory
constexpr int K2SB = 3;      // state tile buffers: S_{j-1} is read by P(j) and by Q'(j), which runs after P(j+1)

// Shared memory of the chain kernel, all TMA tiles in the 128-byte swizzled layout:
// - two stages of the chain's maps: P_j (bf16 [128][128]) and this CTA's columns of c_j (fp32 [128][32]);
// - two stages of the output maps: Q'_j (bf16 [128][128], hi/lo rows interleaved by 16) and this CTA's
//   columns of the chunk-local outputs O_j (fp32 [64][32]);
// - three buffers of S_{j-1} as one bf16 core-matrix tile [128][64]: hi in columns 0-31, lo in 32-63, so that one
//   MMA of N = 64 forms the product with both parts.
struct K2Smem {
    static constexpr int PC = 32768 + 16384, P_ = 0, C_ = 32768;   // a chain stage
    static constexpr int QO = 32768 + 8192, Q_ = 0, O_ = 32768;    // an output stage
    static constexpr int PCS = 0;
    static constexpr int QOS = PCS + 2 * PC;
    static constexpr int SB = QOS + 2 * QO;       // S_{j-1} [hi | lo]: bf16 [128][2 NV] core-matrix tiles, K2SB buffers
    static constexpr int SBB = 128 * 2 * NV * 2;
    static constexpr int BAR = SB + K2SB * SBB;
    static constexpr int TOTAL = BAR + 128;
};
static_assert(K2Smem::TOTAL <= 227 * 1024, "shared memory budget");
static_assert(K2Smem::QOS % 1024 == 0 && K2Smem::PC % 1024 == 0 && K2Smem::QO % 1024 == 0, "swizzled tiles");

struct K2Args {
    const float* S0; float* o; float* ST; int* status;
};

__global__ void __launch_bounds__(K2T, 1)
hdla_chain_kernel(Plan pl, K2Args args, const __grid_constant__ CUtensorMap tm_P, const __grid_constant__ CUtensorMap tm_Q,
                  const __grid_constant__ CUtensorMap tm_C, const __grid_constant__ CUtensorMap tm_O) {
    using S = K2Smem;
    extern __shared__ __align__(1024) unsigned char smem[];
    const uint32_t sb = smem_addr(smem);
    if (sb & 1023u) {
        if (threadIdx.x == 0) atomicExch(args.status, (int)DPLR_ERR_CUDA);
        return;
    }
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::BAR);
    uint64_t* fullPC = bars + 0;    // [2] chunk j's P_j and c_j landed in stage j % 2
    uint64_t* freedPC = bars + 2;   // [2] P(j) done (issuer) and c_j read (each state warp): 5 arrivals
    uint64_t* fullQO = bars + 4;    // [2] chunk j's Q'_j and O_j landed in stage j % 2
    uint64_t* freedQO = bars + 6;   // [2] Q'(j) done (issuer) and O_j read (each state warp): 5 arrivals
    uint64_t* mS = bars + 8;        // P(j), the chain product of chunk j (issuer -> state warps)
    uint64_t* mO = bars + 9;        // [2] Q'(j), the output product of the chunks using accumulator j % 2
    uint64_t* ready = bars + 11;    // S_{j-1} tiles written (4 arrivals, one per state warp; -> issuer)
    uint64_t* drain = bars + 12;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 13);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = pl.T;
    const int NC = (T + HCK - 1) / HCK;
    constexpr int kSlices = HD / NV;
    const int slice = blockIdx.x % kSlices;
    const size_t bh = blockIdx.x / kSlices;
    const int n0 = slice * NV;
    const long long wl = pl.wait_cycles;

    if (tid == 0) {
        for (int u = 0; u < 2; ++u) {
            mbar_init(&fullPC[u], 1);
            mbar_init(&freedPC[u], 5);
            mbar_init(&fullQO[u], 1);
            mbar_init(&freedQO[u], 5);
        }
        mbar_init(mS, 1);
        mbar_init(&mO[0], 1);
        mbar_init(&mO[1], 1);
        mbar_init(ready, 4);
        mbar_init(drain, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(tmem_holder, 256);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    // columns 0-63: P_j [S_hi | S_lo]; 64-191: two output accumulators [Q'_hi; Q'_lo] [S_hi | S_lo]
    const uint32_t tmem = *tmem_holder;
    bool failed = false;
    auto unit_row = [&](int jj) { return static_cast<int>(((size_t)jj * pl.BH + bh) * HD); };

    if (warp == 5 || warp == 6) {
        // ---- copies: warp 5 the chain's maps (P_j, c_j), warp 6 the output maps (Q'_j, O_j). Chunk j goes to
        // stage j % 2 once chunk j - 2 is done with it; chunk j + K2PF is prefetched into L2 at the same time.
        const bool chain = warp == 5;
        uint64_t* full = chain ? fullPC : fullQO;
        uint64_t* freed = chain ? freedPC : freedQO;
        auto prefetch = [&](int jj) {
            const int y = unit_row(jj);
            if (chain) {
                prefetch_l2_tile(&tm_P, 0, y);
                prefetch_l2_tile(&tm_P, 64, y);
                prefetch_l2_tile(&tm_C, n0, y);
            } else {
                prefetch_l2_tile(&tm_Q, 0, y);
                prefetch_l2_tile(&tm_Q, 64, y);
                prefetch_l2_tile(&tm_O, n0, static_cast<int>(bh * T + (size_t)jj * HCK));
            }
        };
        int last = -1;
        if (lane == 0)
            for (int jj = 0; jj < K2PF && jj < NC; ++jj) prefetch(jj);
        for (int j = 0; j < NC && lane == 0; ++j) {
            const int u = j & 1;
            if (j >= 2 && !mbar_wait(&freed[u], ((j - 2) >> 1) & 1, wl)) { failed = true; break; }
            if (j + K2PF < NC) prefetch(j + K2PF);
            const int y = unit_row(j);
            if (chain) {
                unsigned char* st = smem + S::PCS + u * S::PC;
                mbar_expect_tx(&full[u], S::PC);
                tma_load_2d(st + S::P_, &tm_P, 0, y, &full[u]);
                tma_load_2d(st + S::P_ + 16384, &tm_P, 64, y, &full[u]);
                tma_load_2d(st + S::C_, &tm_C, n0, y, &full[u]);
            } else {
                unsigned char* st = smem + S::QOS + u * S::QO;
                mbar_expect_tx(&full[u], S::QO);
                tma_load_2d(st + S::Q_, &tm_Q, 0, y, &full[u]);
                tma_load_2d(st + S::Q_ + 16384, &tm_Q, 64, y, &full[u]);
                // rows past the end of the sequence read the next head's rows (or zeros past the tensor): unused
                tma_load_2d(st + S::O_, &tm_O, n0, static_cast<int>(bh * T + (size_t)j * HCK), &full[u]);
            }
            last = j;
        }
        if (failed) {   // (lane 0) wait for the copies in flight before leaving
            atomicExch(args.status, (int)DPLR_ERR_TIMEOUT);
            for (int jj = last - 1; jj <= last; ++jj)
                if (jj >= 0) mbar_wait(&full[jj & 1], (jj >> 1) & 1, 400000000LL);
        }
        __syncwarp();
    } else if (warp == 4) {
        // ---- the products, issued by lane 0: P(j) = P_j [S_hi | S_lo] into columns 0-63 as soon as S_{j-1} is in
        // place, then Q'(j-1) = [Q'_hi; Q'_lo] [S_hi | S_lo] of the previous chunk into accumulator (j - 1) % 2. The
        // chain's product never waits behind the output product of its own chunk. (A second issuing warp for the
        // output products, so that P(j+1) need not wait for the issue of Q'(j), was slower: the two share the
        // tensor pipe.)
        const uint32_t idS = idesc_bf16(128, 2 * NV, false, true);
        auto products = [&](uint32_t d, uint64_t a, int buf) {   // 8 MMAs, M = 128, N = 64, K = 16 each
            const uint64_t b = smem_desc(sb + S::SB + buf * S::SBB, (2 * NV / 8) * 128, 128);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t ao = (kk >> 2) * 16384 + (kk & 3) * 32, bo = kk * 2 * (2 * NV / 8) * 128;
                mma_bf16(d, dadd(a, ao), dadd(b, bo), idS, kk > 0);
            }
        };
        auto output_product = [&](int jj) -> bool {   // Q'(jj), from S_{jj-1} in buffer jj % 3
            const int u = jj & 1;
            if (!mbar_wait(&fullQO[u], (jj >> 1) & 1, wl)) return false;
            fence_after_sync();
            products(tmem + 64 + 64 * u, smem_desc_sw128(sb + S::QOS + u * S::QO + S::Q_, 16, 1024), jj % K2SB);
            mma_commit(&mO[u]);
            mma_commit(&freedQO[u]);
            return true;
        };
        for (int j = 0; j < NC && lane == 0; ++j) {
            const int u = j & 1;
            if (!mbar_wait_spin(ready, j & 1, wl) || !mbar_wait(&fullPC[u], (j >> 1) & 1, wl)) { failed = true; break; }
            fence_after_sync();
            products(tmem, smem_desc_sw128(sb + S::PCS + u * S::PC + S::P_, 16, 1024), j % K2SB);
            mma_commit(mS);
            mma_commit(&freedPC[u]);
            if (j >= 1 && !output_product(j - 1)) { failed = true; break; }
        }
        if (lane == 0 && !failed && NC > 0 && !output_product(NC - 1)) failed = true;
        if (failed) {   // (lane 0) no product may outlive the tensor memory
            atomicExch(args.status, (int)DPLR_ERR_TIMEOUT);
            mma_commit(drain);
            mbar_wait(drain, 0, 400000000LL);
        }
        __syncwarp();
    } else {
        // ---- the state: thread i holds row i of S (NV columns) in fp32
        const int i = tid;
        const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
        float st[NV];
#pragma unroll
        for (int n = 0; n < NV; ++n) st[n] = args.S0 ? args.S0[(bh * HD + i) * HD + n0 + n] : 0.f;
        // S_{j-1} into buffer b as bf16 [hi | lo], core-matrix layout (MN-major operand: K = row i, N = 64)
        auto write_state = [&](int b) {
            const uint32_t r0 = (i >> 3) * (2 * NV / 8) * 128 + (i & 7) * 16;
#pragma unroll
            for (int ch = 0; ch < NV / 8; ++ch) {
                uint32_t h[4], l[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) split2(st[8 * ch + 2 * e], st[8 * ch + 2 * e + 1], h[e], l[e]);
                sts128(sb + S::SB + b * S::SBB + r0 + ch * 128, h[0], h[1], h[2], h[3]);
                sts128(sb + S::SB + b * S::SBB + r0 + (ch + NV / 8) * 128, l[0], l[1], l[2], l[3]);
            }
        };
        // a wait of the four state warps: each warp's lane 0 polls, and the group takes one decision (a warp
        // must not leave the loop while the others go on to the group barrier)
        auto wait_all = [&](uint64_t* bar, uint32_t parity, uint64_t* bar2, uint32_t parity2) -> bool {
            bool ok = true;
            if (lane == 0) ok = mbar_wait_spin(bar, parity, wl) && (bar2 == nullptr || mbar_wait(bar2, parity2, wl));
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            return !named_sync_or(1, 128, !ok);
        };
        // o_t = O_t + Q'_t S_{jj-1} for chunk jj: a token's hi and lo partial outputs sit in lanes l and l + 16;
        // warp g, lane l holds token t = 16 g + (l % 16) and writes columns 16 (l / 16) .. + 15
        const int tok = 16 * warp + (lane & 15), cseg = 16 * (lane >> 4);
        auto outputs = [&](int jj) -> bool {
            const int u = jj & 1;
            if (!wait_all(&mO[u], (jj >> 1) & 1, &fullQO[u], (jj >> 1) & 1)) return false;
            fence_after_sync();
            const uint32_t stg = sb + S::QOS + u * S::QO;
            float x[32], y[32];
            tmem_ld32(tmem + lane_base + 64 + 64 * u, x);        // x S_hi
            tmem_ld32(tmem + lane_base + 64 + 64 * u + 32, y);   // x S_lo
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                x[e] += y[e];
                x[e] += __shfl_xor_sync(0xffffffffu, x[e], 16);
            }
            const int valid = min(HCK, T - jj * HCK);
            if (tok < valid) {
                const bool upper = lane >= 16;   // (selects keep x in registers)
                float4* orow = reinterpret_cast<float4*>(args.o + (bh * (size_t)T + (size_t)jj * HCK + tok) * HD + n0 + cseg);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    float4 ol;
                    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(ol.x), "=f"(ol.y), "=f"(ol.z), "=f"(ol.w)
                                 : "r"(stg + S::O_ + swz(tok, 4 * (lane >> 4) + q4)));
                    orow[q4] = make_float4(ol.x + (upper ? x[16 + 4 * q4] : x[4 * q4]),
                                           ol.y + (upper ? x[17 + 4 * q4] : x[4 * q4 + 1]),
                                           ol.z + (upper ? x[18 + 4 * q4] : x[4 * q4 + 2]),
                                           ol.w + (upper ? x[19 + 4 * q4] : x[4 * q4 + 3]));
                }
            }
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&freedQO[u]);   // this warp is done with O_jj and the accumulator
            return true;
        };
        write_state(0);
        fence_async_smem();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(ready);
        for (int j = 0; j < NC; ++j) {
            const int u = j & 1;
            // S_j = P_j S_{j-1} + c_j
            if (!wait_all(mS, j & 1, &fullPC[u], (j >> 1) & 1)) { failed = true; break; }
            fence_after_sync();
            {
                const uint32_t stg = sb + S::PCS + u * S::PC;
                float x[32], y[32];
                tmem_ld32(tmem + lane_base, x);        // P_j S_hi
                tmem_ld32(tmem + lane_base + 32, y);   // P_j S_lo
#pragma unroll
                for (int ch = 0; ch < NV / 4; ++ch) {   // c_j row i, columns 4 ch .. 4 ch + 3 (fp32 swizzled box)
                    float4 c4;
                    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(c4.x), "=f"(c4.y), "=f"(c4.z), "=f"(c4.w)
                                 : "r"(stg + S::C_ + swz(i, ch)));
                    st[4 * ch + 0] = (x[4 * ch + 0] + y[4 * ch + 0]) + c4.x;
                    st[4 * ch + 1] = (x[4 * ch + 1] + y[4 * ch + 1]) + c4.y;
                    st[4 * ch + 2] = (x[4 * ch + 2] + y[4 * ch + 2]) + c4.z;
                    st[4 * ch + 3] = (x[4 * ch + 3] + y[4 * ch + 3]) + c4.w;
                }
            }
            // buffer (j + 1) % 3 was last read by Q'(j - 2), which the issuer queued before P(j) (and which
            // outputs(j - 2) saw complete)
            if (j + 1 < NC) {
                write_state((j + 1) % K2SB);
                fence_async_smem();
            }
            fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                if (j + 1 < NC) mbar_arrive(ready);
                mbar_arrive(&freedPC[u]);   // this warp is done with c_j and with the chain accumulator
            }
            // the outputs of the previous chunk, whose product the issuer queued after P(j)
            if (j >= 1 && !outputs(j - 1)) { failed = true; break; }
        }
        if (!failed && NC > 0 && !outputs(NC - 1)) failed = true;
        if (!failed && args.ST) {
            float* dst = args.ST + (bh * HD + i) * HD + n0;
#pragma unroll
            for (int q4 = 0; q4 < NV / 4; ++q4)
                reinterpret_cast<float4*>(dst)[q4] = make_float4(st[4 * q4], st[4 * q4 + 1], st[4 * q4 + 2], st[4 * q4 + 3]);
        }
        if (failed && lane == 0) atomicExch(args.status, (int)DPLR_ERR_TIMEOUT);
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

std::atomic<uint64_t> g_k1_smem_set{0}, g_k2_smem_set{0};


}  // namespace

bool hdla_tc_supported(const Plan& pl) {
    return pl.mode == DPLR_HDLA && pl.bf16 && pl.dk == HD && pl.dv == HD;
}

// Workspace of the tensor-core HDLA path after the 256-byte status word: per (chunk, head) unit, chunk-major
// (the chain reads one chunk of every head at a time),
// P_j bf16 [128][128], then c_j fp32 [128][128], then Q'_j bf16 [2][64][128] (hi rows, then lo rows).
void hdla_tc_offsets(const Plan& pl, size_t* off_P, size_t* off_c, size_t* off_Q, size_t* total) {
    const size_t units = (size_t)pl.BH * (size_t)((pl.T + HCK - 1) / HCK);
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    size_t off = 256;
    *off_P = off; off = up(off + units * HD * HD * 2);
    *off_c = off; off = up(off + units * HD * HD * 4);
    *off_Q = off; off = up(off + units * 2 * HCK * HD * 2);
    *total = off;
}

cudaError_t launch_hdla_chunks(const Plan& pl, const void* q, const void* k, const void* v, const float* decay,
                               const float* beta, float* o, void* workspace, cudaStream_t s) {
    if (pl.T == 0) return cudaSuccess;
    size_t oP, oC, oQ, total;
    hdla_tc_offsets(pl, &oP, &oC, &oQ, &total);
    char* ws = static_cast<char*>(workspace);
    K1Args a;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.k = static_cast<const __nv_bfloat16*>(k);
    a.v = static_cast<const __nv_bfloat16*>(v);
    a.decay = decay; a.beta = beta; a.o = o;
    a.P = reinterpret_cast<__nv_bfloat16*>(ws + oP);
    a.Cm = reinterpret_cast<float*>(ws + oC);
    a.Qm = reinterpret_cast<__nv_bfloat16*>(ws + oQ);
    a.status = reinterpret_cast<int*>(ws);
    CUtensorMap mq, mk, mv, ml, mP, mQ;
    std::memset(&mq, 0, sizeof(mq)); std::memset(&mk, 0, sizeof(mk));
    std::memset(&mv, 0, sizeof(mv)); std::memset(&ml, 0, sizeof(ml));
    const uint64_t units = (uint64_t)pl.BH * (uint64_t)((pl.T + HCK - 1) / HCK);
    if (pl.T >= HCK) {   // only full chunks are loaded and their outputs stored by TMA
        const uint64_t rows = (uint64_t)pl.BH * (uint64_t)pl.T;
        if (!tensor_map_2d(&mq, q, true, rows, HD, HCK, 64) || !tensor_map_2d(&mk, k, true, rows, HD, HCK, 64) ||
            !tensor_map_2d(&mv, v, true, rows, HD, HCK, 64) || !tensor_map_2d(&ml, decay, false, rows, HD, HCK, 32))
            return cudaErrorInvalidValue;
    }
    if (!tensor_map_2d(&mP, ws + oP, true, units * HD, HD, HD, 64) || !tensor_map_2d(&mQ, ws + oQ, true, units * HD, HD, HD, 64))
        return cudaErrorInvalidValue;
    cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(hdla_chunk_kernel), K1Smem::TOTAL, g_k1_smem_set);
    if (e != cudaSuccess) return e;
    const long long grid = std::min<long long>((long long)units, (long long)sm_count());
    hdla_chunk_kernel<<<(unsigned)grid, K1T, K1Smem::TOTAL, s>>>(pl, a, mq, mk, mv, ml, mP, mQ);
    return cudaGetLastError();
}

cudaError_t launch_hdla_chain(const Plan& pl, const float* S0, float* o, float* ST, void* workspace, cudaStream_t s) {
    size_t oP, oC, oQ, total;
    hdla_tc_offsets(pl, &oP, &oC, &oQ, &total);
    char* ws = static_cast<char*>(workspace);
    K2Args a;
    a.S0 = S0; a.o = o; a.ST = ST;
    a.status = reinterpret_cast<int*>(ws);
    CUtensorMap mP, mQ, mC, mO;
    std::memset(&mP, 0, sizeof(mP)); std::memset(&mQ, 0, sizeof(mQ));
    std::memset(&mC, 0, sizeof(mC)); std::memset(&mO, 0, sizeof(mO));
    const int NC = (pl.T + HCK - 1) / HCK;
    if (NC > 0) {
        const uint64_t units = (uint64_t)pl.BH * (uint64_t)NC;
        if (!tensor_map_2d(&mP, ws + oP, true, units * HD, HD, HD, 64) ||
            !tensor_map_2d(&mQ, ws + oQ, true, units * HD, HD, HD, 64) ||
            !tensor_map_2d(&mC, ws + oC, false, units * HD, HD, HD, 32) ||
            !tensor_map_2d(&mO, o, false, (uint64_t)pl.BH * pl.T, HD, HCK, 32))
            return cudaErrorInvalidValue;
    }
    cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(hdla_chain_kernel), K2Smem::TOTAL, g_k2_smem_set);
    if (e != cudaSuccess) return e;
    hdla_chain_kernel<<<(unsigned)(pl.BH * (HD / NV)), K2T, K2Smem::TOTAL, s>>>(pl, a, mP, mQ, mC, mO);
    return cudaGetLastError();
}

}  // namespace dplr
