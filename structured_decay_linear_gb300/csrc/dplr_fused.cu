// Fused per-head forward for Gated DeltaNet with bf16 inputs and dk = dv = 128: one
// CTA owns one (batch, head), walks its chunks of C = 64 tokens in order and keeps
// everything of a chunk on chip -- the Gram blocks, the UT/WY triangular inverse, the
// state-dependent products and the fp32 state itself -- so HBM sees the inputs once and
// the outputs once.
//
// GDN's decay is one scalar per token, so every decay factor of the chunkwise form
// ("Householder-Diagonalized Linear Attention", Key design 3; GDN as the rank-1 case,
// HLA page, Prerequisites) can be moved out of the contractions into row/column
// scalings applied in fp32. With G_t the inclusive cumulative log-gate inside the chunk,
// anchor a = G_C / 2, ef_t = e^{G_t - a}, eb_t = e^{-(G_t - a)} and the folded factors
// A = beta k, B = e^{g} k, W = v, the tensor cores only ever see the raw bf16 q, k, v
// (exact) and a few rounded intermediates:
//
//   D     = [K ; Q] K^T                          (tcgen05 M=128 N=64  K=dk)
//   L_ts  = ef_t D_ts beta_s eb_s  (s < t)       (fp32 epilogue)
//   QK~   = tril_incl(Q K^T) / c,  c = e^{G_C-a} (bf16 hi + lo)
//   M     = (I + L)^{-1}                         (CUDA cores, fp32, blocked 16/32/64)
//   Y^T   = K^T (M Diag(ef))^T                   (tcgen05 M=128 N=64  K=C)
//   E^T   = S'^T Y^T - V^T M^T,  S' = e^{a} S    (tcgen05 M=128 N=64  K=dk+C)
//   Es~   = -c Diag(beta eb) E                   (bf16 hi + lo, in tensor memory)
//   S_j   = e^{G_C} S_{j-1} + K^T Es~            (fp32 accumulator in tensor memory)
//   O'^T  = S'^T Q^T + Es~^T QK~^T, o_t = ef_t O'_t (tcgen05 M=128 N=64 K=dk+C)
//
// E_t = e^{g_t} k_t^T S_{t-1} - v_t is the delta-rule prediction error. Computing the
// transposes E^T, Y^T and O'^T keeps every MMA at M = 128 (full tensor-core rate). The
// rounding of E, QK and of S' in the output product is compensated with a second bf16
// term (x = hi + lo), which keeps the result within ~2e-3 of the float64 recurrence
// (relative to the output RMS) where plain bf16 operands reach ~4e-2.
//
// Work split. Only the chain S_{j-1} -> S' -> E -> Es~ -> S_j is sequential; the WY build
// of a chunk (D, L, M, Y) and its output epilogue are not. Three groups of four warps (one
// thread per tensor-memory lane) and one issuing warp run them concurrently:
//   A  state chain: S' (hi, lo) and e^{G_C} S into tensor memory, then Es~ in place of E;
//   B  WY build: L and QK~ from D, the triangular inverse, the M tiles;
//   C  the chunk outputs o_t, then the Y^T tile of the next chunk.
// Group A issues E(j) and X(j) itself; the issuer queues O(j), D(j+2), O~(j), Y(j+1) and
// Z(j+1) = V^T (-M)^T, so the tensor cores run the chain's products as soon as their operands
// exist and fill the CUDA-core phases of the chain (Es~ while O runs, S' while the rest runs)
// with the others. O~(j) goes before Y(j+1): Y(j+1) waits for the WY build of chunk j+1, and
// the QK~ buffer that build writes is free only once O~(j-1) has run. The state S^T (lane n,
// column c) stays in tensor memory as the accumulator of X for the whole sequence.
//
// Operand tiles. q, k and v arrive by TMA tensor copies of 64 tokens x 64 features
// (128-byte rows) in the 128-byte swizzled layout: token t of a half-tile at t*128, its
// 16-byte chunk c at chunk position c ^ (t % 8). One such tile feeds an MMA K-major
// (contracting over features) or MN-major (contracting over tokens) by the descriptor
// alone. Tiles written from registers use the unswizzled core-matrix layout
//   RBM (row-block major, C columns): (r, c) -> (r/8)*C*16 + (c/8)*128 + (r%8)*16 + (c%8)*2
// (8x8 core matrices of 16-byte rows), whose 16-byte rows of a warp land in distinct bank
// groups; it too serves either major order through LBO/SBO, so no tile is ever transposed.
#include <cstring>

#include "dplr_internal.h"
#include "sm100_ops.cuh"

namespace dplr {
namespace {

using namespace sm100;

constexpr int FD = 128;    // dk = dv
constexpr int FC = 64;     // tokens per chunk
constexpr int kGrp = 128;  // threads of each CUDA-core group (one per TMEM lane)
// Warps 0-3: state chain (group A). Warps 4-7: WY build (group B). Warps 8-11: Y^T tiles and
// outputs (group C). Warp 12: copies of k, q, v into shared memory. Warp 13: MMA issuer
// (on another scheduler than the copy warp).
constexpr int FNT = 3 * kGrp + 64;
constexpr uint32_t kBarA = 1, kBarB = 2, kBarC = 3;   // named barriers of the groups
constexpr uint32_t kTmemCols = 512;
constexpr int kLdL = 68;   // padded row stride (floats) of the fp32 L and M buffers (16-byte rows)
constexpr int kKQBuf = 3;  // k/q buffers: chunk j's are read until X(j); chunk j+2's are needed for D(j+2)

// Tile geometry. A swizzled half-tile is 64 tokens x 128 bytes = 8 KB; a k/q buffer holds
// [k features 0-63][q features 0-63][k features 64-127][q features 64-127].
constexpr uint32_t SWH = FC * 128;     // bytes of one swizzled half-tile
constexpr uint32_t KQ_H = 2 * SWH;     // k/q buffer: stride between the two feature halves
constexpr uint32_t KQ_BYTES = 2 * KQ_H;
constexpr uint32_t N64_RB = 64 * 16;   // RBM tiles with 64 columns

struct GdnLayout {
    static constexpr int T_KQ = 0;                          // k, q of a chunk (4 swizzled half-tiles), 3 buffers
    static constexpr int T_V = T_KQ + kKQBuf * KQ_BYTES;    // v of a chunk (2 swizzled half-tiles)
    static constexpr int T_MN = T_V + FC * FD * 2;          // [64 rho][64 sigma] RBM  -M
    static constexpr int T_MY = T_MN + FC * FC * 2;         // [64][64] RBM  M Diag(ef)
    static constexpr int T_YT = T_MY + FC * FC * 2;         // [128 c][64 rho] RBM  Y^T
    static constexpr int T_QK = T_YT + FD * FC * 2;         // 2 buffers x {hi, lo} [64 t][64 sigma] RBM  QK / c
    static constexpr int F_L = T_QK + 4 * FC * FC * 2;      // fp32 [64][68]
    static constexpr int F_M = F_L + FC * kLdL * 4;         // fp32 [64][68]
    static constexpr int SCR = F_M + FC * kLdL * 4;         // fp32 scratch of the inverse (32 x 36)
    static constexpr int VEC = SCR + 32 * 36 * 4;          // per group, 2 buffers of 256 floats
    static constexpr int kVec = 1024;
    static constexpr int BAR = VEC + 6 * kVec;              // mbarriers, TMEM address, counter
    static constexpr int TOTAL = BAR + 176;   // 19 mbarriers, TMEM address, two counters
};
static_assert(GdnLayout::TOTAL <= 227 * 1024, "shared memory budget");
static_assert(GdnLayout::T_V % 1024 == 0 && KQ_BYTES % 1024 == 0, "swizzled tiles are 1024-byte aligned");

// TMEM columns (512 allocated)
constexpr uint32_t TM_S = 0;      // S^T fp32 (lane n, column c)            128 lanes x 128
constexpr uint32_t TM_SH = 128;   // S'^T hi (A operand, bf16 pairs)         128 x 64
constexpr uint32_t TM_SL = 192;   // S'^T lo
constexpr uint32_t TM_E = 256;    // E^T fp32, then Es~^T hi/lo in place     128 x 64
constexpr uint32_t TM_O = 320;    // O'^T                                    128 x 64
constexpr uint32_t TM_D = 384;    // [K;Q] K^T                               128 x 64
constexpr uint32_t TM_Y = 448;    // Y^T                                     128 x 64

struct FusedArgs {
    const __nv_bfloat16* q; const __nv_bfloat16* k; const __nv_bfloat16* v;
    const float* decay; const float* beta; const float* S0;
    float* o; float* ST; int* status;
};

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" :: "r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ uint32_t rbm_off(int r, int c, int cols) {
    return static_cast<uint32_t>((r >> 3) * (cols * 16) + (c >> 3) * 128 + (r & 7) * 16 + (c & 7) * 2);
}

// 8 consecutive fp32 values (cols c..c+7, c % 8 == 0) of row r into an RBM bf16 tile.
__device__ __forceinline__ void rbm_store8(uint32_t tile, int cols, int r, int c, const float* x) {
    st_shared_v4(tile + rbm_off(r, c, cols), pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]),
                 pack_bf16(x[6], x[7]));
}

// Forms predicated by `issue`: a warp issues MMAs from one lane without diverging, so that it
// does not have to re-converge afterwards (which costs hundreds of cycles after MMAs).
__device__ __forceinline__ void mma_tmem_a_if(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc,
                                              uint32_t issue) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %4, 0;\n\tsetp.ne.b32 q, %5, 0;\n\t"
        "@q tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        :: "r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc), "r"(issue));
}
__device__ __forceinline__ void mma_commit_if(uint64_t* mbar, uint32_t issue) {
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %1, 0;\n\t"
        "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}"
        :: "r"(smem_addr(mbar)), "r"(issue) : "memory");
}
__device__ __forceinline__ void mbar_arrive_if(uint64_t* mbar, uint32_t issue) {
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %1, 0;\n\t@q mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}"
                 :: "r"(smem_addr(mbar)), "r"(issue) : "memory");
}

// x = hi + lo with both parts bf16: packed pairs (element 2i in the low half).
__device__ __forceinline__ void split_pair(float x0, float x1, uint32_t& h, uint32_t& l) {
    h = pack_bf16(x0, x1);
    const float2 r = __fadd2_rn(make_float2(x0, x1), make_float2(-__uint_as_float(h << 16), -__uint_as_float(h & 0xFFFF0000u)));
    l = pack_bf16(r.x, r.y);
}
__device__ __forceinline__ void split_pair(float2 x, uint32_t& h, uint32_t& l) { split_pair(x.x, x.y, h, l); }

__device__ __forceinline__ void rbm_store8_split(uint32_t th, uint32_t tl, int cols, int r, int c, const float* x) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) split_pair(x[2 * i], x[2 * i + 1], h[i], l[i]);
    const uint32_t off = rbm_off(r, c, cols);
    st_shared_v4(th + off, h[0], h[1], h[2], h[3]);
    st_shared_v4(tl + off, l[0], l[1], l[2], l[3]);
}

__device__ __forceinline__ float4 lds4(const float* p) { return *reinterpret_cast<const float4*>(p); }

constexpr int kLds = 36;   // row stride (floats) of the merge scratch (32 rows)

// (I + L)^{-1} for a 64x64 strictly lower-triangular fp32 L (row stride kLdL = 68 floats, so
// rows are 16-byte aligned), by the 128 threads of group B (t = 0..127, named barrier kBarB).
// The four 16x16 diagonal blocks are solved row by row (left-looking, one column per thread,
// rows of L read as 16-byte broadcasts); the blocks are merged 16 -> 32 -> 64 with
// [[A,0],[C,B]]^{-1} = [[A^{-1},0],[-B^{-1} C A^{-1}, B^{-1}]], the merge products on the tensor
// cores in tf32 (their ~1e-3 relative error is below the bf16 rounding the result gets next).
// Writes -M and M Diag(ef) as bf16 RBM tiles.
__device__ __forceinline__ void unit_lower_inverse64(const float* L, float* Mf, float* scr, uint32_t t_mn,
                                                     uint32_t t_my, const float* ef, int t) {
    if (t < 64) {   // diagonal 16x16 blocks: M[i][j] = delta_ij - sum_{k<i} L[i][k] M[k][j]
        const int b = t >> 4, j = t & 15, o = 16 * b;
        float m[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float* Lr = L + (o + i) * kLdL + o;
            float acc0 = (i == j) ? 1.f : 0.f, acc1 = 0.f;
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
                if (4 * k4 < i) {
                    const float4 l = lds4(Lr + 4 * k4);
                    if (4 * k4 + 0 < i) acc0 = fmaf(-l.x, m[4 * k4 + 0], acc0);
                    if (4 * k4 + 1 < i) acc1 = fmaf(-l.y, m[4 * k4 + 1], acc1);
                    if (4 * k4 + 2 < i) acc0 = fmaf(-l.z, m[4 * k4 + 2], acc0);
                    if (4 * k4 + 3 < i) acc1 = fmaf(-l.w, m[4 * k4 + 3], acc1);
                }
            }
            m[i] = acc0 + acc1;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) Mf[(o + i) * kLdL + o + j] = m[i];
    } else {        // zero the 16x16 blocks above the diagonal inside each 32x32 diagonal block
        const int e = t - 64;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int f = e + 64 * h, r = f >> 2, cc = 4 * (f & 3), pp = r >> 4, rr = r & 15;
            *reinterpret_cast<float4*>(Mf + (32 * pp + rr) * kLdL + 32 * pp + 16 + cc) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    named_sync(kBarB, kGrp);
    // merges on the tensor cores (mma.sync tf32, fp32 accumulate)
    const int warp = t >> 5;
    {   // 16 -> 32 for the pairs of diagonal blocks (0,1) and (2,3): one 16x8 tile per warp
        const int p = warp >> 1, ct = warp & 1, o = 32 * p;
        float c[4];
        warp_mma_tf32(L + (o + 16) * kLdL + o, kLdL, Mf + o * kLdL + o + 8 * ct, kLdL, 16, c);   // T = C A^{-1}
        store_tile_16x8(scr + p * 16 * kLds + 8 * ct, kLds, c, 1.f);
        named_sync(kBarB, kGrp);
        warp_mma_tf32(Mf + (o + 16) * kLdL + o + 16, kLdL, scr + p * 16 * kLds + 8 * ct, kLds, 16, c);  // B^{-1} T
        store_tile_16x8(Mf + (o + 16) * kLdL + o + 8 * ct, kLdL, c, -1.f);
        named_sync(kBarB, kGrp);
    }
    {   // 32 -> 64: M[32:64, 0:32] = -B^{-1} (C A^{-1}); eight 16x8 tiles, two per warp
        float c0[4], c1[4];
        warp_mma_tf32(L + 32 * kLdL, kLdL, Mf + 8 * warp, kLdL, 32, c0);
        warp_mma_tf32(L + 48 * kLdL, kLdL, Mf + 8 * warp, kLdL, 32, c1);
        store_tile_16x8(scr + 8 * warp, kLds, c0, 1.f);
        store_tile_16x8(scr + 16 * kLds + 8 * warp, kLds, c1, 1.f);
        named_sync(kBarB, kGrp);
        warp_mma_tf32(Mf + 32 * kLdL + 32, kLdL, scr + 8 * warp, kLds, 32, c0);
        warp_mma_tf32(Mf + 48 * kLdL + 32, kLdL, scr + 8 * warp, kLds, 32, c1);
        store_tile_16x8(Mf + 32 * kLdL + 8 * warp, kLdL, c0, -1.f);
        store_tile_16x8(Mf + 48 * kLdL + 8 * warp, kLdL, c1, -1.f);
        named_sync(kBarB, kGrp);
    }
    // bf16 tiles -M and M Diag(ef); the 32x32 block above the diagonal is zero
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        const int item = t + kGrp * h, r = item & 63, c = (item >> 6) * 8;
        float x[8], y[8];
        if ((c >> 5) > (r >> 5)) {
#pragma unroll
            for (int i = 0; i < 8; ++i) { x[i] = 0.f; y[i] = 0.f; }
        } else {
            const float4 m0 = lds4(Mf + r * kLdL + c), m1 = lds4(Mf + r * kLdL + c + 4);
            const float m[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) { x[i] = -m[i]; y[i] = m[i] * ef[c + i]; }
        }
        rbm_store8(t_mn, FC, r, c, x);
        rbm_store8(t_my, FC, r, c, y);
    }
}

// Inclusive scan of a chunk's log-gates by one warp (lane holds tokens 2*lane, 2*lane+1).
struct ChunkGates {
    float G0, G1, GC;   // G at tokens 2*lane, 2*lane+1; G at the chunk end
};
__device__ __forceinline__ ChunkGates scan_gates(float g0, float g1) {
    const int lane = threadIdx.x & 31;
    float s = g0 + g1;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, s, off);
        if (lane >= off) s += y;
    }
    ChunkGates r;
    r.GC = __shfl_sync(0xffffffffu, s, 31);
    r.G1 = s;
    r.G0 = s - g1;
    return r;
}

__global__ void __launch_bounds__(FNT, 1)
gdn_fused_head_kernel(Plan pl, FusedArgs args, const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
    using Ly = GdnLayout;
    extern __shared__ __align__(1024) unsigned char smem[];
    const uint32_t sbase = smem_addr(smem);
    if (sbase & 1023u) {   // the swizzled tiles need 1024-byte alignment
        if (threadIdx.x == 0) atomicExch(args.status, (int)DPLR_ERR_CUDA);
        return;
    }
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Ly::BAR);
    // MMA completions (issuer -> groups)
    uint64_t* mbar_D = bars + 0;     // D(j)                              -> B
    uint64_t* mbar_Y = bars + 1;     // Y(j)                              -> C
    uint64_t* mbar_Z = bars + 2;     // Z(j) (and the issuer's MMAs before) -> A, B, copy warp
    uint64_t* mbar_E = bars + 3;     // E(j), issued by A                 -> A, C
    uint64_t* mbar_X = bars + 4;     // E(j), X(j), issued by A           -> A, issuer
    uint64_t* mbar_O = bars + 5;     // O~(j), the issuer's last product of chunk j -> C
    // bulk copies
    uint64_t* mbar_kq = bars + 6;    // [kKQBuf]
    uint64_t* mbar_v = bars + 9;
    // groups -> issuer
    uint64_t* rdy_S = bars + 10;     // A: S'(j) in TMEM (for O(j))
    uint64_t* rdy_E = bars + 11;     // A: Es~(j) in TMEM (for O~(j))
    uint64_t* rdy_M = bars + 12;     // B: M(j) tiles
    uint64_t* rdy_Yt = bars + 13;    // C: Y^T(j) tile (and Y(j) consumed)
    uint64_t* o_free = bars + 14;    // C: O(j) consumed
    uint64_t* drain = bars + 15;     // [2]: the issuer's and group A's MMAs
    uint64_t* mbar_O1 = bars + 17;   // O(j) = S'^T Q^T, issued by the issuer -> A
    uint64_t* d_free = bars + 18;    // B: D(j) read (its accumulator may take D(j+1))
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 19);
    int* o_seen = reinterpret_cast<int*>(bars + 20);    // C: chunks whose O~ has completed
    int* x_seen = reinterpret_cast<int*>(bars + 20) + 1;   // A: chunks whose X has completed
    float* scr = reinterpret_cast<float*>(smem + Ly::SCR);
    float* F_L = reinterpret_cast<float*>(smem + Ly::F_L);
    float* F_M = reinterpret_cast<float*>(smem + Ly::F_M);
    auto vec = [&](int grp, int buf) { return reinterpret_cast<float*>(smem + Ly::VEC + (2 * grp + buf) * Ly::kVec); };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int grp = warp >> 2;                  // 0 = A, 1 = B, 2 = C, 3 = issuer
    const int gt = tid & (kGrp - 1);            // thread within its group = TMEM lane
    const size_t bh = blockIdx.x;
    const int T = pl.T;
    const int nchunk = (T + FC - 1) / FC;
    const int nfull = T / FC;                   // chunks loaded by TMA (only the last may be ragged)
    const size_t tok_base = bh * (size_t)T;
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;

    if (tid == 0) {
        for (int i = 0; i < 19; ++i) mbar_init(bars + i, 1);
        *o_seen = 0;
        *x_seen = 0;
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(tmem_holder, kTmemCols);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_holder;
    auto tKQ_of = [&](int jj) -> uint32_t { return sbase + Ly::T_KQ + (jj % kKQBuf) * KQ_BYTES; };
    auto tQK_of = [&](int jj, int lo) -> uint32_t { return sbase + Ly::T_QK + ((jj & 1) * 2 + lo) * FC * FC * 2; };
    // raw gates of chunk jj for one warp: tokens 2*lane, 2*lane+1 (zero past the end)
    auto load_gates = [&](int jj, float (&r)[4]) {
        const int t0 = jj * FC + 2 * lane;
        r[0] = (t0 < T) ? args.decay[tok_base + t0] : 0.f;
        r[1] = (t0 + 1 < T) ? args.decay[tok_base + t0 + 1] : 0.f;
        r[2] = (t0 < T) ? args.beta[tok_base + t0] : 0.f;
        r[3] = (t0 + 1 < T) ? args.beta[tok_base + t0 + 1] : 0.f;
    };
    const long long wl = pl.wait_cycles;   // limit of every wait on another role (drains excepted)
    // bounded wait of a whole group on an mbarrier phase; false (for every thread) if it gave up.
    // One thread polls; the others sleep on the group's hardware barrier, so the polling does
    // not take issue slots from the warps that work (the issuer above all).
    auto group_wait = [&](uint64_t* bar, uint32_t parity, uint32_t barid) -> bool {
        bool got = true;
        if (gt < 32) got = mbar_wait(bar, parity, wl);   // the group's first warp, converged
        const bool bad = named_sync_or(barid, kGrp, !got);
        fence_after_sync();
        return !bad;
    };
    bool failed = false;

    if (warp == 12) {
        // ======================= copy warp: TMA (lane 0) and the ragged last chunk (all lanes) ==========
        // the last chunk copied into each k/q buffer and into the v buffer (-1: none): the phase of
        // that copy is the one a drain waits for
        int last_kq[kKQBuf], last_v = -1;
        for (int b = 0; b < kKQBuf; ++b) last_kq[b] = -1;
        auto ragged_rows = [&](int jj, const __nv_bfloat16* src, uint32_t dst, uint32_t half_stride) {
            const int valid = T - jj * FC;
            const size_t g0 = tok_base + (size_t)jj * FC;
#pragma unroll 1
            for (int i = lane; i < FC * (FD / 8); i += 32) {
                const int cb = i & 15, t = i >> 4;   // 16-byte chunk cb of token t, in the swizzled layout
                uint4 z = make_uint4(0, 0, 0, 0);
                if (t < valid) z = *reinterpret_cast<const uint4*>(src + (g0 + t) * FD + 8 * cb);
                st_shared_v4(dst + (cb >> 3) * half_stride + t * 128 + (((cb & 7) ^ (t & 7)) << 4), z.x, z.y, z.z, z.w);
            }
        };
        auto load_kq = [&](int jj) {
            const int b = jj % kKQBuf;
            if (jj < nfull) {
                const int y = static_cast<int>(tok_base + (size_t)jj * FC);
                unsigned char* dst = smem + Ly::T_KQ + b * KQ_BYTES;
                if (lane == 0) {
                    mbar_expect_tx(&mbar_kq[b], KQ_BYTES);
                    for (int x = 0; x < 4; ++x)   // x = 2 * half + (q ? 1 : 0)
                        tma_load_2d(dst + x * SWH, (x & 1) ? &tm_q : &tm_k, 64 * (x >> 1), y, &mbar_kq[b]);
                }
            } else {   // ragged last chunk: plain loads, zero rows past the end; then a plain arrival
                ragged_rows(jj, args.k, tKQ_of(jj), KQ_H);
                ragged_rows(jj, args.q, tKQ_of(jj) + SWH, KQ_H);
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&mbar_kq[b]);
            }
            last_kq[b] = jj;
            __syncwarp();
        };
        auto load_v = [&](int jj) {
            if (jj < nfull) {
                const int y = static_cast<int>(tok_base + (size_t)jj * FC);
                if (lane == 0) {
                    mbar_expect_tx(mbar_v, FC * FD * 2);
                    for (int x = 0; x < 2; ++x) tma_load_2d(smem + Ly::T_V + x * SWH, &tm_v, 64 * x, y, mbar_v);
                }
            } else {
                ragged_rows(jj, args.v, sbase + Ly::T_V, SWH);
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(mbar_v);
            }
            last_v = jj;
            __syncwarp();
        };
        if (nchunk > 0) {
            load_kq(0);
            if (nchunk > 1) load_kq(1);
            load_v(0);
        }
        for (int j = 0; j < nchunk && !failed; ++j) {
            // k/q of chunk j+2 into the buffer of chunk j-1 once the products that read it, O~(j-1)
            // (issuer) and X(j-1) (group A), are done
            if (j + 2 < nchunk) {
                bool ok = true;
                if (lane == 0) {
                    const long long t0 = clock64();
                    while (ld_acquire_shared(o_seen) < j || ld_acquire_shared(x_seen) < j) {
                        if (clock64() - t0 > wl) { ok = false; break; }
                        __nanosleep(100);
                    }
                }
                if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) { failed = true; break; }
                load_kq(j + 2);
            }
            // v of chunk j+1 once Z(j) has read v(j)
            if (j + 1 < nchunk) {
                bool ok = true;
                if (lane == 0) ok = mbar_wait(mbar_Z, j & 1, wl);
                if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) { failed = true; break; }
                load_v(j + 1);
            }
        }
        if (failed) {
            if (lane == 0) {
                atomicExch(args.status, (int)DPLR_ERR_TIMEOUT);
                // no copy may land in shared memory after the CTA has exited: wait for the phase of
                // the last copy into each buffer (copy n into k/q buffer b completes phase n / kKQBuf)
                for (int b = 0; b < kKQBuf; ++b)
                    if (last_kq[b] >= 0) mbar_wait(&mbar_kq[b], (last_kq[b] / kKQBuf) & 1, 400000000LL);
                if (last_v >= 0) mbar_wait(mbar_v, last_v & 1, 400000000LL);
            }
            __syncwarp();
        }
    } else if (warp == 13) {
        // ======================= issuer warp: the MMAs =======================
        // Lane 0 runs the whole loop alone; lanes 1-31 wait at the warp barrier after it. (A warp
        // that re-converges right after one lane has issued MMAs loses hundreds of cycles there.)
        auto wait1 = [&](uint64_t* bar, uint32_t parity) -> bool {
            const bool ok = mbar_wait(bar, parity, wl);
            fence_after_sync();
            return ok;
        };
        auto wait_kq = [&](int jj) -> bool {   // (the ragged last chunk completes the phase by a plain arrival)
            return wait1(&mbar_kq[jj % kKQBuf], (jj / kKQBuf) & 1);
        };
        const uint32_t idN64 = idesc_bf16(128, FC, false, false);
        // ---- the MMA groups
        auto mma_D = [&](int jj) {   // D = [K;Q] K^T: rows 0-63 k, 64-127 q of each feature half
            const uint32_t tk = tKQ_of(jj);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint64_t d = smem_desc_sw128(tk + h * KQ_H, 16, 1024);
                mma_chain(tmem + TM_D, d, 32, d, 32, idN64, 64, h > 0);
            }
            mma_commit(mbar_D);
        };
        auto mma_Y = [&](int jj) {   // Y^T = K^T (M Diag(ef))^T
            mma_chain(tmem + TM_Y, smem_desc_sw128(tKQ_of(jj), KQ_H, 1024), 2048,
                      smem_desc(sbase + Ly::T_MY, 128, N64_RB), 256, idesc_bf16(128, FC, true, false), FC, false);
            mma_commit(mbar_Y);
        };
        auto mma_Z = [&]() {         // E^T := V^T (-M)^T
            mma_chain(tmem + TM_E, smem_desc_sw128(sbase + Ly::T_V, SWH, 1024), 2048,
                      smem_desc(sbase + Ly::T_MN, 128, N64_RB), 256, idesc_bf16(128, FC, true, false), FC, false);
            mma_commit(mbar_Z);
        };
        auto mma_O = [&](int j) {    // O'^T = S'^T Q^T with S' = hi + lo (q rows, K-major)
            const uint32_t tq = tKQ_of(j) + SWH;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {   // c = 2 * half + (lo ? 1 : 0)
                const int h = c >> 1;
                const uint64_t dQ = smem_desc_sw128(tq + h * KQ_H, 16, 1024);
                mma_chain_tmem_a(tmem + TM_O, tmem + ((c & 1) ? TM_SL : TM_SH) + 32 * h, dQ, 32, idN64, 64, c > 0);
            }
            mma_commit(mbar_O1);
        };
        auto mma_Oes = [&](int j) {  // O'^T += Es~^T QK~^T: hi*hi + lo*hi + hi*lo
            const uint64_t bh0 = smem_desc(tQK_of(j, 0), 128, N64_RB), bl0 = smem_desc(tQK_of(j, 1), 128, N64_RB);
#pragma unroll
            for (int sl = 0; sl < 4; ++sl) {
                const uint32_t ah = tmem + TM_E + 32 * (sl >> 1) + 8 * (sl & 1);
                const uint64_t bh_ = bh0 + static_cast<uint64_t>(16 * sl), bl_ = bl0 + static_cast<uint64_t>(16 * sl);
                mma_bf16_tmem_a(tmem + TM_O, ah, bh_, idN64, 1u);
                mma_bf16_tmem_a(tmem + TM_O, ah + 16, bh_, idN64, 1u);
                mma_bf16_tmem_a(tmem + TM_O, ah, bl_, idN64, 1u);
            }
            mma_commit(mbar_O);
        };

        // j = -2, -1: the WY build of chunks 0 and 1 only. E(j) and X(j) are issued by group A.
        for (int j = -2; lane == 0 && j < nchunk && !failed; ++j) {
            const bool next = j + 1 < nchunk;
            if (j >= 0) {
                // O(j) once S'(j) is in place and the outputs of chunk j-1 have been read
                if (!wait1(rdy_S, j & 1)) { failed = true; break; }
                if (j >= 1 && !wait1(o_free, (j - 1) & 1)) { failed = true; break; }
                mma_O(j);
            }
            // D(j+2) as soon as group B has read D(j+1) out of the accumulator
            if (j + 2 < nchunk) {
                if ((j >= -1 && !wait1(d_free, (j + 1) & 1)) || !wait_kq(j + 2)) { failed = true; break; }
                mma_D(j + 2);
            }
            // O~(j) once Es~(j) is in place (after O(j), in this thread's order)
            if (j >= 0) {
                if (!wait1(rdy_E, j & 1)) { failed = true; break; }
                mma_Oes(j);
            }
            // Y(j+1), whose Y^T tile gates E(j+1), once its M tiles exist and group C has read Y(j)
            if (j >= -1 && next) {
                if (!wait1(rdy_M, (j + 1) & 1) || (j >= 0 && !wait1(rdy_Yt, j & 1))) { failed = true; break; }
                mma_Y(j + 1);
            }
            // Z(j+1) reuses the E accumulator: after O~(j) (this thread) and X(j) (group A)
            if (j >= -1 && next) {
                if ((j >= 0 && !wait1(mbar_X, j & 1)) || !wait1(mbar_v, (j + 1) & 1)) { failed = true; break; }
                mma_Z();
            }
        }
        if (failed) {   // (lane 0 only)
            atomicExch(args.status, (int)DPLR_ERR_TIMEOUT);
            mma_commit(drain);   // tracks every MMA this thread issued
            mbar_wait(drain, 0, 400000000LL);
        }
        __syncwarp();
    } else if (grp == 0) {
        // ======================= group A: the state chain =======================
        float graw[4];
        if (warp == 0 && nchunk > 0) load_gates(0, graw);
        auto gates = [&](int jj) {   // warp 0: e^{a}, gamma = e^{G_C}, nc_bs = -beta e^{G_C - G}
            if (warp != 0) return;
            float* vf = vec(0, jj & 1);
            const ChunkGates g = scan_gates(graw[0], graw[1]);
            vf[64 + 2 * lane] = -graw[2] * __expf(g.GC - g.G0);
            vf[64 + 2 * lane + 1] = -graw[3] * __expf(g.GC - g.G1);
            if (lane == 0) {
                vf[0] = __expf(0.5f * g.GC);
                vf[1] = __expf(g.GC);
            }
            if (jj + 1 < nchunk) load_gates(jj + 1, graw);
        };
        if (nchunk > 0) {
            gates(0);
#pragma unroll 1
            for (int p = 0; p < 4; ++p) {   // S0^T into the accumulator
                uint32_t x[32];
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    x[i] = __float_as_uint(args.S0 ? args.S0[(bh * FD + 32 * p + i) * FD + gt] : 0.f);
                tmem_st32(tmem + TM_S + lane_off + 32 * p, x);
            }
            tmem_wait_st();
        }
        named_sync(kBarA, kGrp);
        // The leader thread issues this group's own MMAs, E(j) and X(j), straight after the group
        // barrier that publishes their tensor-memory operand: no hand-off to another warp on the chain.
        const uint32_t idE = idesc_bf16(128, FC, false, true), idX = idesc_bf16(128, FD, false, true);
        const uint64_t dYt = smem_desc(sbase + Ly::T_YT, N64_RB, 128);
        for (int j = 0; j < nchunk && !failed; ++j) {
            const float* vf = vec(0, j & 1);
            if (j > 0) {   // S_{j-1} complete (X(j-1)); S'(j-1) read by E(j-1) and O(j-1)
                if (!group_wait(mbar_X, (j - 1) & 1, kBarA) || !group_wait(mbar_O1, (j - 1) & 1, kBarA)) {
                    failed = true;
                    break;
                }
                if (gt == 0) st_release_shared(x_seen, j);
            }
            {   // ---- S'^T (hi, lo) and gamma S^T
                const float ea = vf[0], gam = vf[1];
#pragma unroll 1
                for (int p = 0; p < 4; ++p) {
                    float x[32];
                    tmem_ld32(tmem + TM_S + lane_off + 32 * p, x);
                    uint32_t hi[16], lo[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        split_pair(__fmul2_rn(make_float2(ea, ea), make_float2(x[2 * i], x[2 * i + 1])), hi[i], lo[i]);
                    tmem_st16(tmem + TM_SH + lane_off + 16 * p, hi);
                    tmem_st16(tmem + TM_SL + lane_off + 16 * p, lo);
                    uint32_t g[32];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float2 y = __fmul2_rn(make_float2(gam, gam), make_float2(x[2 * i], x[2 * i + 1]));
                        g[2 * i] = __float_as_uint(y.x);
                        g[2 * i + 1] = __float_as_uint(y.y);
                    }
                    tmem_st32(tmem + TM_S + lane_off + 32 * p, g);
                }
                tmem_wait_st();
            }
            fence_before_sync();
            named_sync(kBarA, kGrp);
            if (warp == 0) {   // converged; lane 0 issues through a predicate
                const uint32_t lead = lane == 0;
                mbar_arrive_if(rdy_S, lead);
                // E(j) += S'^T Y^T onto Z(j) (issuer), once Z(j) is done and Y^T(j) is in place
                if (mbar_wait(mbar_Z, j & 1, wl) && mbar_wait(rdy_Yt, j & 1, wl)) {
                    fence_after_sync();
#pragma unroll
                    for (int ks = 0; ks < FD / 16; ++ks)
                        mma_tmem_a_if(tmem + TM_E, tmem + TM_SH + 8 * ks, dYt + static_cast<uint64_t>(ks * (2 * N64_RB / 16)),
                                      idE, 1u, lead);
                    mma_commit_if(mbar_E, lead);
                }
            }
            // ---- Es~^T of chunk j, in place of E^T
            if (!group_wait(mbar_E, j & 1, kBarA)) { failed = true; break; }
#pragma unroll 1
            for (int p = 0; p < 2; ++p) {
                float x[32];
                tmem_ld32(tmem + TM_E + lane_off + 32 * p, x);
                uint32_t hi[16], lo[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    split_pair(__fmul2_rn(*reinterpret_cast<const float2*>(vf + 64 + 32 * p + 2 * i), make_float2(x[2 * i], x[2 * i + 1])),
                               hi[i], lo[i]);
                tmem_st16(tmem + TM_E + lane_off + 32 * p, hi);
                tmem_st16(tmem + TM_E + lane_off + 32 * p + 16, lo);
            }
            tmem_wait_st();
            fence_before_sync();
            named_sync(kBarA, kGrp);
            if (warp == 0) {   // converged; lane 0 issues through a predicate
                const uint32_t lead = lane == 0;
                // X(j): S^T += Es~^T K (hi + lo); Es~ hi at 32*(s/2) + 8*(s%2), lo 16 columns further
                fence_after_sync();
                const uint64_t dK = smem_desc_sw128(tKQ_of(j), KQ_H, 1024);   // k rows, MN-major B (K = rho)
#pragma unroll
                for (int sl = 0; sl < 4; ++sl) {
                    const uint32_t ah = tmem + TM_E + 32 * (sl >> 1) + 8 * (sl & 1);
                    const uint64_t b = dK + static_cast<uint64_t>((2048u * sl) >> 4);
                    mma_tmem_a_if(tmem + TM_S, ah, b, idX, 1u, lead);
                    mma_tmem_a_if(tmem + TM_S, ah + 16, b, idX, 1u, lead);
                }
                mma_commit_if(mbar_X, lead);
                mbar_arrive_if(rdy_E, lead);
            }
            if (j + 1 < nchunk) gates(j + 1);
            named_sync(kBarA, kGrp);   // gates of chunk j + 1 visible to the group
        }
        if (!failed) {   // final state
            if (nchunk > 0 && !group_wait(mbar_X, (nchunk - 1) & 1, kBarA)) failed = true;
            if (!failed && args.ST) {
#pragma unroll 1
                for (int p = 0; p < 4; ++p) {
                    float x[32];
                    if (nchunk == 0) {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            x[i] = args.S0 ? args.S0[(bh * FD + 32 * p + i) * FD + gt] : 0.f;
                    } else {
                        tmem_ld32(tmem + TM_S + lane_off + 32 * p, x);
                    }
#pragma unroll
                    for (int i = 0; i < 32; ++i) args.ST[(bh * FD + 32 * p + i) * FD + gt] = x[i];
                }
            }
        }
        if (failed && gt == 0) {
            atomicExch(args.status, (int)DPLR_ERR_TIMEOUT);
            mma_commit(drain + 1);   // tracks every MMA this thread issued
            mbar_wait(drain + 1, 0, 400000000LL);
        }
    } else if (grp == 1) {
        // ======================= group B: the WY build of each chunk =======================
        float graw[4];
        if (warp == 4 && nchunk > 0) load_gates(0, graw);
        for (int jj = 0; jj < nchunk && !failed; ++jj) {
            float* vf = vec(1, jj & 1);
            if (warp == 4) {   // ef = e^{G - a}, bs = beta e^{a - G}, 1/c = e^{a - G_C}
                const ChunkGates g = scan_gates(graw[0], graw[1]);
                const float a = 0.5f * g.GC;
                vf[2 * lane] = __expf(g.G0 - a);
                vf[2 * lane + 1] = __expf(g.G1 - a);
                vf[64 + 2 * lane] = graw[2] * __expf(a - g.G0);
                vf[64 + 2 * lane + 1] = graw[3] * __expf(a - g.G1);
                if (lane == 0) vf[128] = __expf(a - g.GC);
                if (jj + 1 < nchunk) load_gates(jj + 1, graw);
            }
            if (!group_wait(mbar_D, jj & 1, kBarB)) { failed = true; break; }   // also orders the gates
            if (jj >= 2) {   // QK~ tiles of buffer jj & 1 were read by the last product of chunk jj - 2
                bool ok = true;
                if (gt == 0) {
                    const long long t0 = clock64();
                    while (ld_acquire_shared(o_seen) < jj - 1) {
                        if (clock64() - t0 > wl) { ok = false; break; }
                        __nanosleep(100);
                    }
                }
                if (named_sync_or(kBarB, kGrp, !ok)) { failed = true; break; }
            }
            {   // ---- L (rows 0-63 of D) and QK~ (rows 64-127), one TMEM lane per thread
                const float inv_c = vf[128];
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {
                    float x[32];
                    tmem_ld32(tmem + TM_D + lane_off + 32 * hh, x);
                    if (gt < FC) {
                        const int t = gt;
                        const float eft = vf[t];
                        const float2 ef2 = make_float2(eft, eft);
#pragma unroll
                        for (int i = 0; i < 32; i += 4) {
                            const float4 bs = *reinterpret_cast<const float4*>(vf + 64 + 32 * hh + i);
                            const float2 y01 = __fmul2_rn(__fmul2_rn(ef2, make_float2(x[i], x[i + 1])), make_float2(bs.x, bs.y));
                            const float2 y23 = __fmul2_rn(__fmul2_rn(ef2, make_float2(x[i + 2], x[i + 3])), make_float2(bs.z, bs.w));
                            const int sg = 32 * hh + i;
                            *reinterpret_cast<float4*>(F_L + t * kLdL + sg) =
                                make_float4(sg < t ? y01.x : 0.f, sg + 1 < t ? y01.y : 0.f, sg + 2 < t ? y23.x : 0.f, sg + 3 < t ? y23.y : 0.f);
                        }
                    } else {
                        const int t = gt - FC;
                        const float2 ic2 = make_float2(inv_c, inv_c);
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            const float2 y = __fmul2_rn(ic2, make_float2(x[i], x[i + 1]));
                            x[i] = (32 * hh + i <= t) ? y.x : 0.f;
                            x[i + 1] = (32 * hh + i + 1 <= t) ? y.y : 0.f;
                        }
#pragma unroll
                        for (int i = 0; i < 32; i += 8)
                            rbm_store8_split(tQK_of(jj, 0), tQK_of(jj, 1), FC, t, 32 * hh + i, x + i);
                    }
                }
            }
            fence_before_sync();
            named_sync(kBarB, kGrp);
            if (gt == 0) mbar_arrive(d_free);   // every thread's tcgen05.ld of D(jj) has completed
            if (jj >= 1 && !group_wait(mbar_Z, (jj - 1) & 1, kBarB)) { failed = true; break; }   // M tiles free
            unit_lower_inverse64(F_L, F_M, scr, sbase + Ly::T_MN, sbase + Ly::T_MY, vf, gt);
            fence_async_smem();
            fence_before_sync();
            named_sync(kBarB, kGrp);
            if (gt == 0) mbar_arrive(rdy_M);
        }
        if (failed && gt == 0) atomicExch(args.status, (int)DPLR_ERR_TIMEOUT);
    } else {
        // ======================= group C: the chunk outputs, then the next Y^T tile =======================
        float graw[4];
        if (warp == 8 && nchunk > 0) load_gates(0, graw);
        auto epi_Y = [&]() {
#pragma unroll 1
            for (int hh = 0; hh < 2; ++hh) {
                float x[32];
                tmem_ld32(tmem + TM_Y + lane_off + 32 * hh, x);
#pragma unroll
                for (int i = 0; i < 32; i += 8) rbm_store8(sbase + Ly::T_YT, FC, gt, 32 * hh + i, x + i);
            }
            fence_async_smem();
            fence_before_sync();
            named_sync(kBarC, kGrp);
            if (gt == 0) mbar_arrive(rdy_Yt);
        };
        if (nchunk > 0) {
            if (!group_wait(mbar_Y, 0, kBarC)) failed = true;
            else epi_Y();
        }
        for (int j = 0; j < nchunk && !failed; ++j) {
            float* vf = vec(2, j & 1);
            if (warp == 8) {   // ef of chunk j
                const ChunkGates g = scan_gates(graw[0], graw[1]);
                const float a = 0.5f * g.GC;
                vf[2 * lane] = __expf(g.G0 - a);
                vf[2 * lane + 1] = __expf(g.G1 - a);
                if (j + 1 < nchunk) load_gates(j + 1, graw);
            }
            if (!group_wait(mbar_O, j & 1, kBarC)) { failed = true; break; }   // also orders ef
            if (gt == 0) st_release_shared(o_seen, j + 1);
            {   // ---- o_t = ef_t O'_t
                const int valid = min(FC, T - j * FC);
                float* ocol = args.o + (tok_base + (size_t)j * FC) * FD + gt;
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {
                    float x[32];
                    tmem_ld32(tmem + TM_O + lane_off + 32 * hh, x);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int t = 32 * hh + i;
                        if (t < valid) ocol[(size_t)t * FD] = vf[t] * x[i];
                    }
                }
            }
            fence_before_sync();
            named_sync(kBarC, kGrp);
            if (gt == 0) mbar_arrive(o_free);
            if (j + 1 < nchunk) {   // Y^T of chunk j + 1 (its tile was read by E(j)); Y(j + 2) waits for it
                if (!group_wait(mbar_Y, (j + 1) & 1, kBarC) || !group_wait(mbar_E, j & 1, kBarC)) {
                    failed = true;
                    break;
                }
                epi_Y();
            }
        }
        if (failed && gt == 0) atomicExch(args.status, (int)DPLR_ERR_TIMEOUT);
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// [rows][128] bf16 row-major, boxes of 64 columns x 64 rows, 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, uint64_t rows) {
    return tensor_map_2d(map, base, true, rows, FD, FC, 64);
}

std::atomic<uint64_t> g_fused_smem_set{0};

}  // namespace

bool fused_supported(const Plan& pl) {
    return pl.mode == DPLR_GDN && pl.bf16 && pl.dk == FD && pl.dv == FD;
}

cudaError_t launch_fused(const Plan& pl, const void* q, const void* k, const void* v, const float* decay,
                         const float* beta, const float* S0, float* o, float* ST, int* status, cudaStream_t s) {
    FusedArgs a;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.k = static_cast<const __nv_bfloat16*>(k);
    a.v = static_cast<const __nv_bfloat16*>(v);
    a.decay = decay; a.beta = beta; a.S0 = S0; a.o = o; a.ST = ST; a.status = status;
    CUtensorMap mq, mk, mv;
    std::memset(&mq, 0, sizeof(mq));
    std::memset(&mk, 0, sizeof(mk));
    std::memset(&mv, 0, sizeof(mv));
    if (pl.T >= FC) {   // only full chunks are loaded by TMA
        const uint64_t rows = (uint64_t)pl.BH * (uint64_t)pl.T;
        if (!make_map(&mq, q, rows) || !make_map(&mk, k, rows) || !make_map(&mv, v, rows))
            return cudaErrorInvalidValue;
    }
    cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(gdn_fused_head_kernel), GdnLayout::TOTAL,
                                        g_fused_smem_set);
    if (e != cudaSuccess) return e;
    gdn_fused_head_kernel<<<(unsigned)pl.BH, FNT, GdnLayout::TOTAL, s>>>(pl, a, mq, mk, mv);
    return cudaGetLastError();
}

size_t fused_smem_bytes(int) { return (size_t)GdnLayout::TOTAL; }

}  // namespace dplr
