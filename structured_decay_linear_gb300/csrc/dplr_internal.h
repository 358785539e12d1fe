// Internal declarations shared by the libdplr translation units (not part of the ABI).
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/dplr.h"

namespace dplr {

// Largest stacked rank-row count C_w * max(r_ab, r_kv) a WY block may hold. The
// chunk given in the descriptor is split into WY blocks of C_w tokens so that
// the Gram / triangular-solve tiles stay within shared memory.
constexpr int kMaxStackedRows = 64;
constexpr int kPrepThreads = 256;
constexpr int kScanThreads = 256;
constexpr int kScanCols = 32;  // state columns per scan CTA (dv split)

// Everything the launches need, derived from a validated descriptor.
struct Plan {
    int mode, bf16;
    int BH, T, dk, dv, r, p;   // p = 0 in the structured modes (write term folded into A)
    int cw;                    // WY block length in tokens (two-stage path)
    int nb;                    // WY blocks per head = ceil(T / cw)
    int fused;                 // dplr_la_forward runs the fused per-head kernel (GDN)
    int tc;                    // the stages run the tensor-core HDLA kernels
    int gtc;                   // stage 1 runs the tensor-core generic-mode kernel (32-token WY blocks)
    long long wait_cycles;     // limit (SM cycles) of a kernel's bounded waits on other roles
    size_t off_P, off_c, off_Q;
    size_t ws_stages;          // workspace of the two-stage entry points
    size_t ws_bytes;           // workspace of dplr_la_forward
};

// Per-launch arguments of the chunk-map kernel.
struct ChunkMapArgs {
    const void* q; const void* k; const void* v;
    const float* decay; const float* beta;
    const void* A; const void* Bm; const void* K; const void* V;
    float* o;
    float* Pm;  // [BH, nb, dk, dk]   chunk transition P_j
    float* Cm;  // [BH, nb, dk, dv]   chunk offset c_j
    float* Qm;  // [BH, nb, cw, dk]   chunk readout Q'_j
};

struct ScanArgs {
    const float* S0; float* o; float* ST;
    const float* Pm; const float* Cm; const float* Qm;
    float* Sb = nullptr;   // optional [BH, nb, dk, dv]: the state before each WY block (the backward's checkpoints)
};

dplr_status make_plan(const dplr_desc* d, Plan* plan);

constexpr long long kDefaultWaitCycles = 4000000000LL;   // ~2 s at 2 GHz

// Raises a kernel's dynamic shared-memory limit to `bytes` once per device: the attribute
// belongs to the device's copy of the function, so later launches skip the driver call.
// `done` holds one bit per device ordinal (64 devices at most).
inline cudaError_t set_smem_limit_once(const void* func, int bytes, std::atomic<uint64_t>& done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const uint64_t bit = uint64_t(1) << dev;
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}
int sm_count();   // SMs of the current device
size_t prep_smem_bytes(const Plan& pl);
size_t scan_smem_bytes(const Plan& pl);
cudaError_t launch_chunk_maps(const Plan& pl, const ChunkMapArgs& a, cudaStream_t s);
cudaError_t launch_state_scan(const Plan& pl, const ScanArgs& a, cudaStream_t s);

// A 2-D tensor map of a row-major [rows][cols] matrix (fp32 or bf16) read in 128-byte-swizzled
// boxes of box_rows x box_cols elements (box_cols * element size = 128 bytes). Encoded once and
// then served from a small per-thread cache keyed on (base, rows, cols, box, type).
bool tensor_map_2d(CUtensorMap* map, const void* base, bool bf16, uint64_t rows, uint64_t cols, uint32_t box_rows,
                   uint32_t box_cols);

// Tensor-core HDLA path (bf16 inputs, dk = dv = 128): chunk maps, then the chain over chunks.
bool hdla_tc_supported(const Plan& pl);
void hdla_tc_offsets(const Plan& pl, size_t* off_P, size_t* off_c, size_t* off_Q, size_t* total);
cudaError_t launch_hdla_chunks(const Plan& pl, const void* q, const void* k, const void* v, const float* decay,
                               const float* beta, float* o, void* workspace, cudaStream_t s);
cudaError_t launch_hdla_chain(const Plan& pl, const float* S0, float* o, float* ST, void* workspace, cudaStream_t s);

// Tensor-core stages of the generic mode (dk = dv = 64, r_ab <= 4, r_kv <= 2): maps of 32-token WY blocks, then
// the chain over blocks.
bool generic_tc_supported(const Plan& pl);
int generic_tc_block();
void generic_tc_offsets(const Plan& pl, size_t* off_A, size_t* off_c, size_t* total);
cudaError_t launch_generic_chunks(const Plan& pl, const ChunkMapArgs& a, void* workspace, cudaStream_t s);
cudaError_t launch_generic_chain(const Plan& pl, const float* S0, float* o, float* ST, void* workspace, cudaStream_t s);

// Fused per-head kernel (structured modes, bf16 inputs, dk = dv = 128).
bool fused_supported(const Plan& pl);
size_t fused_smem_bytes(int mode);
cudaError_t launch_fused(const Plan& pl, const void* q, const void* k, const void* v, const float* decay,
                         const float* beta, const float* S0, float* o, float* ST, int* status, cudaStream_t s);

}  // namespace dplr
