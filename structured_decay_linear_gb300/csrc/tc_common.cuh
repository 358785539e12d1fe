// Helpers shared by the tensor-core chunk kernels: 128-byte-swizzled tile addressing, bf16 hi/lo
// splits, single-lane tcgen05 issue, tensor-memory loads, warp-level tf32 products, the blocked
// unit-lower-triangular inverse, and bulk stores. Device code only; written against the PTX ISA.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sm100_ops.cuh"

namespace dplr {
namespace tc {

using namespace sm100;

constexpr int kLdX = 68;   // row stride (floats) of the inverse's fp32 blocks (16-byte rows, 4 banks apart)

// ---- 128-byte-swizzled tiles (the layout the TMA writes with SWIZZLE_128B): rows of 128 bytes whose
// 16-byte chunks are permuted by XOR with the row index mod 8. A bf16 [R][128] tile is two half-tiles
// (columns 0-63, 64-127) of R rows; an fp32 [R][128] tile is four column boxes of 32.
__device__ __forceinline__ uint32_t swz(int r, int chunk) { return (uint32_t)(r * 128 + (((chunk) ^ (r & 7)) << 4)); }
__device__ __forceinline__ uint32_t sw_bf16(int r, int c, int R) {
    return (uint32_t)((c >> 6) * (R * 128)) + swz(r, (c & 63) >> 3) + (uint32_t)((c & 7) << 1);
}
__device__ __forceinline__ uint32_t sw_f32(int r, int c, int R) {
    return (uint32_t)((c >> 5) * (R * 128)) + swz(r, (c & 31) >> 2) + (uint32_t)((c & 3) << 2);
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" :: "r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ float lds_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ float lds_bf16(uint32_t addr) {
    uint16_t v;
    asm volatile("ld.shared.b16 %0, [%1];" : "=h"(v) : "r"(addr));
    return __uint_as_float(static_cast<uint32_t>(v) << 16);
}
__device__ __forceinline__ uint16_t bf16_bits(float x) {
    __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t*>(&h);
}
__device__ __forceinline__ float bf16_value(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }
__device__ __forceinline__ float tf32_rn(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// x = hi + lo with both parts bf16 (scalar): the pair of bit patterns.
__device__ __forceinline__ void split1(float x, uint16_t& h, uint16_t& l) {
    h = bf16_bits(x);
    l = bf16_bits(x - bf16_value(h));
}
// x = hi + lo for a pair of values, packed (element 0 in the low half).
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& h, uint32_t& l) {
    h = pack_bf16(x0, x1);
    l = pack_bf16(x0 - __uint_as_float(h << 16), x1 - __uint_as_float(h & 0xFFFF0000u));
}

// ---- fp16 hi + lo with a power-of-two scale. y = x * sc is split as hi = rn_fp16(y), lo = rn_fp16(y - hi);
// with the scale chosen so that the largest magnitude of the operand lands in [2^14, 2^15) (fp16 overflows at
// 65504), hi + lo carries ~22 significant bits for every value within 2^11 of the largest, and smaller values
// keep an absolute error below 2^-25 of the scaled range.
__device__ __forceinline__ void splith2(float x0, float x1, float sc, uint32_t& h, uint32_t& l) {
    const float y0 = x0 * sc, y1 = x1 * sc;
    const __half2 hh = __floats2half2_rn(y0, y1);
    const float2 hf = __half22float2(hh);
    const __half2 ll = __floats2half2_rn(y0 - hf.x, y1 - hf.y);
    h = *reinterpret_cast<const uint32_t*>(&hh);
    l = *reinterpret_cast<const uint32_t*>(&ll);
}
__device__ __forceinline__ void splith1(float x, float sc, uint16_t& h, uint16_t& l) {
    const float y = x * sc;
    const __half hh = __float2half_rn(y);
    const __half ll = __float2half_rn(y - __half2float(hh));
    h = *reinterpret_cast<const uint16_t*>(&hh);
    l = *reinterpret_cast<const uint16_t*>(&ll);
}
__device__ __forceinline__ float half_value(uint16_t b) {
    return __half2float(*reinterpret_cast<const __half*>(&b));
}
// The scale 2^(14 - floor(log2 m)) for a largest magnitude m (1 when m is zero, tiny or not finite), from the
// exponent field.
__device__ __forceinline__ float scale_for(float m) {
    const int e = static_cast<int>((__float_as_uint(m) >> 23) & 255u) - 127;   // floor(log2 m) for normal m
    if (!(m > 0.f) || e < -110 || e > 120) return 1.f;
    return __uint_as_float(static_cast<uint32_t>(14 - e + 127) << 23);
}
// Maximum of v over the warp, folded into a shared slot (non-negative floats order like their bit patterns).
// Every lane of the warp must call it.
__device__ __forceinline__ void warp_max_to(unsigned int* slot, float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    if ((threadIdx.x & 31) == 0) atomicMax(slot, __float_as_uint(v));
}
// Instruction descriptor for kind::f16 with fp16 A and B, fp32 accumulation.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4) | (static_cast<uint32_t>(a_mn) << 15) | (static_cast<uint32_t>(b_mn) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// MMAs issued by lane 0 of a converged warp through a predicate (no divergence, so no costly
// re-convergence after the issue).
__device__ __forceinline__ void mma_ss_if(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc, uint32_t issue) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %4, 0;\n\tsetp.ne.b32 q, %5, 0;\n\t"
        "@q tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(issue));
}
__device__ __forceinline__ void mma_ts_if(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc,
                                          uint32_t issue) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %4, 0;\n\tsetp.ne.b32 q, %5, 0;\n\t"
        "@q tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        :: "r"(d), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc), "r"(issue));
}
__device__ __forceinline__ void commit_if(uint64_t* mbar, uint32_t issue) {
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %1, 0;\n\t"
        "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}"
        :: "r"(smem_addr(mbar)), "r"(issue) : "memory");
}
__device__ __forceinline__ uint64_t dadd(uint64_t desc, uint32_t bytes) { return desc + static_cast<uint64_t>(bytes >> 4); }

// 16 consecutive fp32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// One mma.sync m16n8k8 tf32 (fp32 accumulate) on fragments in registers. Not volatile: independent products
// may be interleaved by the compiler.
__device__ __forceinline__ void mma_tf32_frag(float (&c)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Warp-level products C_i[16x8] = A_i[16xK] B[Kx8], i < NT, for NT row tiles A_i = A + 16 i lda sharing the
// columns of B (mma.sync m16n8k8 tf32, fp32 accumulate); A, B row-major fp32 in shared memory, fragments as in
// the PTX ISA. TERMS = 1: the operands rounded to tf32 (cvt.rna). TERMS = 3: each operand split as x = hi + lo
// with both parts tf32, and hi*hi, hi*lo, lo*hi accumulated separately and added at the end (the dropped lo*lo
// is ~2^-22 of the product), which keeps the product close to fp32 accuracy.
template <int TERMS, int NT>
__device__ __forceinline__ void warp_mma_tf32_tiles(const float* A, int lda, const float* B, int ldb, int K,
                                                    float (&c)[NT][4]) {
    const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    float acc[NT][TERMS][4];
#pragma unroll
    for (int i = 0; i < NT; ++i)
#pragma unroll
        for (int t = 0; t < TERMS; ++t) acc[i][t][0] = acc[i][t][1] = acc[i][t][2] = acc[i][t][3] = 0.f;
#pragma unroll
    for (int k0 = 0; k0 < K; k0 += 8) {
        uint32_t bh[2], bl[2];
        {
            const float bf[2] = {B[(k0 + q) * ldb + g], B[(k0 + q + 4) * ldb + g]};
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float h = tf32_rn(bf[e]);
                bh[e] = __float_as_uint(h);
                bl[e] = __float_as_uint(tf32_rn(bf[e] - h));
            }
        }
#pragma unroll
        for (int i = 0; i < NT; ++i) {
            const float* Ai = A + 16 * i * lda;
            const float af[4] = {Ai[g * lda + k0 + q], Ai[(g + 8) * lda + k0 + q], Ai[g * lda + k0 + q + 4],
                                 Ai[(g + 8) * lda + k0 + q + 4]};
            uint32_t ah[4], al[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float h = tf32_rn(af[e]);
                ah[e] = __float_as_uint(h);
                al[e] = __float_as_uint(tf32_rn(af[e] - h));
            }
            mma_tf32_frag(acc[i][0], ah, bh);
            if (TERMS == 3) {
                mma_tf32_frag(acc[i][1], ah, bl);
                mma_tf32_frag(acc[i][2], al, bh);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < NT; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float v = acc[i][0][e];
            if (TERMS == 3) v += acc[i][1][e] + acc[i][2][e];
            c[i][e] = v;
        }
}
template <int TERMS>
__device__ __forceinline__ void warp_mma_tf32_x(const float* A, int lda, const float* B, int ldb, int K, float (&c)[4]) {
    float t[1][4];
    warp_mma_tf32_tiles<TERMS, 1>(A, lda, B, ldb, K, t);
    c[0] = t[0][0]; c[1] = t[0][1]; c[2] = t[0][2]; c[3] = t[0][3];
}
__device__ __forceinline__ void warp_mma_tf32_rn(const float* A, int lda, const float* B, int ldb, int K, float (&c)[4]) {
    warp_mma_tf32_x<1>(A, lda, B, ldb, K, c);
}

// In place, for the 256 threads t of one group (named barrier `bar`): X (64 x 64, row stride kLdX)
// holds a strictly lower-triangular L on entry (zeros on and above the diagonal) and
// M = (I + L)^{-1} on exit. Diagonal 16 x 16 blocks by substitution (one column per thread), then
// the block merges [[A,0],[C,B]]^{-1} = [[A^{-1},0],[-B^{-1} C A^{-1}, B^{-1}]] for 16 -> 32 -> 64,
// each product formed in registers and written over C once every warp has read C.
template <int TERMS = 1>
__device__ __forceinline__ void inv64_inplace(float* X, int t, uint32_t bar) {
    const int w = t >> 5;
    if (t < 64) {
        const int b = t >> 4, jj = t & 15, o = 16 * b;
        float m[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float* Lr = X + (o + i) * kLdX + o;
            float acc0 = (i == jj) ? 1.f : 0.f, acc1 = 0.f;
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
                if (4 * k4 < i) {
                    const float4 l = *reinterpret_cast<const float4*>(Lr + 4 * k4);
                    if (4 * k4 + 0 < i) acc0 = fmaf(-l.x, m[4 * k4 + 0], acc0);
                    if (4 * k4 + 1 < i) acc1 = fmaf(-l.y, m[4 * k4 + 1], acc1);
                    if (4 * k4 + 2 < i) acc0 = fmaf(-l.z, m[4 * k4 + 2], acc0);
                    if (4 * k4 + 3 < i) acc1 = fmaf(-l.w, m[4 * k4 + 3], acc1);
                }
            }
            m[i] = acc0 + acc1;
        }
        named_sync(bar, 256);   // every row of the diagonal blocks read
#pragma unroll
        for (int i = 0; i < 16; ++i) X[(o + i) * kLdX + o + jj] = m[i];
    } else {
        named_sync(bar, 256);
    }
    named_sync(bar, 256);
    {   // 16 -> 32 for the pairs of diagonal blocks (0,1) and (2,3): one 16 x 8 tile for each of warps 0-3
        const int p = (w >> 1) & 1, ct = w & 1, o = 32 * p;
        float c[4];
        if (w < 4) warp_mma_tf32_x<TERMS>(X + (o + 16) * kLdX + o, kLdX, X + o * kLdX + o + 8 * ct, kLdX, 16, c);   // C A^{-1}
        named_sync(bar, 256);
        if (w < 4) store_tile_16x8(X + (o + 16) * kLdX + o + 8 * ct, kLdX, c, 1.f);
        named_sync(bar, 256);
        if (w < 4) warp_mma_tf32_x<TERMS>(X + (o + 16) * kLdX + o + 16, kLdX, X + (o + 16) * kLdX + o + 8 * ct, kLdX, 16, c);
        named_sync(bar, 256);
        if (w < 4) store_tile_16x8(X + (o + 16) * kLdX + o + 8 * ct, kLdX, c, -1.f);
        named_sync(bar, 256);
    }
    {   // 32 -> 64: rows 32-63, columns 0-31; one 16 x 8 tile per warp (row block 16 (w / 4), column block 8 (w % 4))
        const int rb = w >> 2, cb = w & 3;
        float c[4];
        warp_mma_tf32_x<TERMS>(X + (32 + 16 * rb) * kLdX, kLdX, X + 8 * cb, kLdX, 32, c);
        named_sync(bar, 256);
        store_tile_16x8(X + (32 + 16 * rb) * kLdX + 8 * cb, kLdX, c, 1.f);
        named_sync(bar, 256);
        warp_mma_tf32_x<TERMS>(X + (32 + 16 * rb) * kLdX + 32, kLdX, X + 32 * kLdX + 8 * cb, kLdX, 32, c);
        named_sync(bar, 256);
        store_tile_16x8(X + (32 + 16 * rb) * kLdX + 8 * cb, kLdX, c, -1.f);
        named_sync(bar, 256);
    }
}

// A bounded wait that polls (mbarrier.test_wait) instead of suspending: for the chain's hand-offs, where the
// waiting warps have nothing else to do and the wake-up of a suspended wait is on the critical path.
__device__ __forceinline__ bool mbar_wait_spin(uint64_t* mbar, uint32_t parity, long long max_cycles) {
    const uint32_t a = smem_addr(mbar);
    const long long t0 = clock64();
    for (;;) {
        uint32_t done;
        asm volatile("{\n\t.reg .pred q;\n\tmbarrier.test_wait.parity.shared::cta.b64 q, [%1], %2;\n\tselp.u32 %0, 1, 0, q;\n\t}"
                     : "=r"(done) : "r"(a), "r"(parity) : "memory");
        if (done) return true;
        if (clock64() - t0 > max_cycles) return false;
    }
}

// Bulk stores (shared -> global) by tensor map, and their completion.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, uint32_t src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];"
                 :: "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(src) : "memory");
}
// Shared -> global bulk copy (16-byte aligned addresses, size a multiple of 16) in the current bulk group.
__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 :: "l"(reinterpret_cast<uint64_t>(dst)), "r"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void prefetch_l2_tile(const CUtensorMap* map, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
                 :: "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y) : "memory");
}

}  // namespace tc
}  // namespace dplr
