// Inline-PTX helpers for sm_100-family tensor cores (tcgen05), TMEM, mbarriers and
// bulk copies, written against the PTX ISA. Every wait is bounded.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

namespace dplr {
namespace sm100 {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// Core-matrix tiled bf16 operand layout (no swizzle).
// A matrix X[rows][cols] is stored as 8x8 core matrices of 128 bytes: element (r, c)
// lives at (r/8)*RS + (c/8)*128 + (r%8)*16 + (c%8)*2 with row-block stride RS = cols*16.
// The same buffer serves as
//   * a K-major operand contracting over cols (rows = M or N):  LBO = 128, SBO = RS
//   * an MN-major operand contracting over rows (cols = M or N): LBO = RS,  SBO = 128
// (LBO is the byte distance between core matrices adjacent along K, SBO along M/N).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t tile_off(int r, int c, int cols) {
    return static_cast<uint32_t>((r >> 3) * (cols * 16) + (c >> 3) * 128 + (r & 7) * 16 + (c & 7) * 2);
}

// Shared-memory matrix descriptor: start address, LBO, SBO (bytes), no swizzle,
// fixed 0b001 at bits 46-48 (sm_100 descriptor version).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    return d;
}

// The same for a tile in the 128-byte swizzled layout (rows of 128 bytes whose 16-byte chunks
// are permuted by XOR with the row index mod 8, as the TMA writes them with SWIZZLE_128B).
// K-major: SBO = stride of 8-row groups (LBO unused). MN-major: LBO = stride between
// 64-element blocks along MN, SBO = stride of 8-row groups along K. Base 1024-byte aligned.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return smem_desc(saddr, lbo, sbo) | (static_cast<uint64_t>(2) << 61);
}

// Descriptor of tile (base, cols) used K-major (contract over cols) or MN-major (contract over rows).
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t base, int cols) { return smem_desc(base, 128, cols * 16); }
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t base, int cols) { return smem_desc(base, cols * 16, 128); }

// Instruction descriptor for kind::f16 with bf16 A/B, f32 accumulate.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
           (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A * B for one K=16 slice, issued by a single thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

// D[tmem] (+)= A * B with the A operand in tensor memory (lane = row, column j holding the
// bf16 pair (2j, 2j+1) of the row, low half = even element), B from shared memory.
__device__ __forceinline__ void mma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                                uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        :: "r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}

// Chain of K/16 MMAs with A in tensor memory (8 columns per K=16 slice).
__device__ __forceinline__ void mma_chain_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t b_step,
                                                 uint32_t idesc, int K, bool accumulate) {
#pragma unroll
    for (int ks = 0; ks < K / 16; ++ks)
        mma_bf16_tmem_a(d_tmem, a_tmem + 8 * ks, b + static_cast<uint64_t>((b_step * ks) >> 4), idesc,
                        (accumulate || ks > 0) ? 1u : 0u);
}

// Stores 32 consecutive 32-bit columns of this thread's TMEM lane (then waits for completion).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
        :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
           "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
           "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
           "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Stores 16 consecutive 32-bit columns of this thread's TMEM lane (completion: tmem_wait_st).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
           "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
// Waits until this thread's earlier tcgen05.st have completed.
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Named barrier `id` over the first `n` threads (a multiple of 32) of the CTA.
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t n) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(n) : "memory");
}

// Named barrier that also ORs a predicate over the participating threads.
__device__ __forceinline__ bool named_sync_or(uint32_t id, uint32_t n, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %3, 0;\n\tbar.red.or.pred q, %1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r) : "r"(id), "r"(n), "r"(static_cast<uint32_t>(v)) : "memory");
    return r != 0;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* mbar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_addr(mbar)) : "memory");
}

// Chain of K/16 MMAs; a_step/b_step: byte advance of each operand per K=16 slice.
__device__ __forceinline__ void mma_chain(uint32_t d_tmem, uint64_t a, uint32_t a_step, uint64_t b, uint32_t b_step,
                                          uint32_t idesc, int K, bool accumulate) {
#pragma unroll
    for (int ks = 0; ks < K / 16; ++ks) {
        mma_bf16(d_tmem, a + static_cast<uint64_t>((a_step * ks) >> 4), b + static_cast<uint64_t>((b_step * ks) >> 4),
                 idesc, (accumulate || ks > 0) ? 1u : 0u);
    }
}

__device__ __forceinline__ void mma_commit(uint64_t* mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(smem_addr(mbar)) : "memory");
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Makes generic-proxy shared-memory writes visible to the tensor core / bulk-copy (async) proxy.
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// TMEM allocation (whole warp).
__device__ __forceinline__ void tmem_alloc(uint32_t* holder, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_addr(holder)), "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// ---------------------------------------------------------------------------
// mbarriers and bulk copies.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* mbar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_addr(mbar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

__device__ __forceinline__ void mbar_expect_tx(uint64_t* mbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(smem_addr(mbar)), "r"(bytes) : "memory");
}

// Shared-memory counters with acquire / release ordering (CTA scope).
__device__ __forceinline__ int ld_acquire_shared(const int* p) {
    int v;
    asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_shared(int* p, int v) {
    asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" :: "r"(smem_addr(p)), "r"(v) : "memory");
}

// Bounded wait for the phase with the given parity. Returns false if it gave up
// (after roughly `max_cycles` SM cycles). Each try_wait may suspend the thread until the
// phase completes (at most ~0.1 ms per attempt), so a waiting thread takes no issue slots
// from the warps that share its scheduler.
__device__ __forceinline__ bool mbar_wait(uint64_t* mbar, uint32_t parity, long long max_cycles = 4000000000LL) {
    const uint32_t a = smem_addr(mbar);
    const long long t0 = clock64();
    for (;;) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred q;\n\tmbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, q;\n\t}"
            : "=r"(done) : "r"(a), "r"(parity), "r"(100000u) : "memory");
        if (done) return true;
        if (clock64() - t0 > max_cycles) return false;
    }
}

// Global -> shared bulk copy (16-byte aligned addresses, size a multiple of 16), completing
// `bytes` on the mbarrier's transaction count.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* mbar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        :: "r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(mbar)) : "memory");
}

// 2-D tiled tensor copy global -> shared (box defined by the tensor map), completing its
// bytes on the mbarrier. x is the innermost coordinate (elements; x * elem_size must be a
// multiple of 16 bytes), y the row.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* mbar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        :: "r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(mbar))
        : "memory");
}

// Warp-level C[16x8] = A[16xK] * B[Kx8] with fp32 operands read as tf32 (mma.sync m16n8k8, fp32
// accumulate); A and B row-major in shared memory with row strides lda / ldb. Fragment layout of
// the PTX ISA: g = lane / 4, q = lane % 4; A (g, q), (g+8, q), (g, q+4), (g+8, q+4); B (q, g),
// (q+4, g); C (g, 2q), (g, 2q+1), (g+8, 2q), (g+8, 2q+1).
__device__ __forceinline__ void warp_mma_tf32(const float* A, int lda, const float* B, int ldb, int K, float (&c)[4]) {
    const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    c[0] = c[1] = c[2] = c[3] = 0.f;
    for (int k0 = 0; k0 < K; k0 += 8) {
        const uint32_t a0 = __float_as_uint(A[g * lda + k0 + q]), a1 = __float_as_uint(A[(g + 8) * lda + k0 + q]);
        const uint32_t a2 = __float_as_uint(A[g * lda + k0 + q + 4]), a3 = __float_as_uint(A[(g + 8) * lda + k0 + q + 4]);
        const uint32_t b0 = __float_as_uint(B[(k0 + q) * ldb + g]), b1 = __float_as_uint(B[(k0 + q + 4) * ldb + g]);
        asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                     "{%0,%1,%2,%3};"
                     : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                     : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
}

__device__ __forceinline__ void store_tile_16x8(float* C, int ldc, const float (&c)[4], float scale) {
    const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    C[g * ldc + 2 * q] = scale * c[0];
    C[g * ldc + 2 * q + 1] = scale * c[1];
    C[(g + 8) * ldc + 2 * q] = scale * c[2];
    C[(g + 8) * ldc + 2 * q + 1] = scale * c[3];
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

}  // namespace sm100
}  // namespace dplr
