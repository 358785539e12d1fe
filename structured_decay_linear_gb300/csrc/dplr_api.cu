// Host side of the libdplr C ABI: descriptor validation, workspace plan, launches.
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "dplr_internal.h"

namespace dplr {
namespace {

constexpr size_t kAlign = 256;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool valid_dim(int d) { return d == 32 || d == 64 || d == 128; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

std::atomic<long long> g_wait_cycles{kDefaultWaitCycles};

// Largest power-of-two WY block (<= chunk) whose stacked rank rows fit.
int wy_block(int chunk, int r, int p) {
    const int m = r > p ? r : p;
    int cw = chunk;
    while (cw > 8 && cw * m > kMaxStackedRows) cw /= 2;
    return cw;
}

// cuTensorMapEncodeTiled from the driver (looked up once).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool encode_map_2d(CUtensorMap* map, const void* base, bool bf16, uint64_t rows, uint64_t cols, uint32_t box_rows,
                   uint32_t box_cols) {
    auto fn = encode_fn();
    if (!fn) return false;
    const uint64_t esize = bf16 ? 2 : 4;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * esize};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base),
              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Number of SMs of the current device (looked up once per device).
int sm_count() {
    static std::atomic<int> cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cached[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

bool tensor_map_2d(CUtensorMap* map, const void* base, bool bf16, uint64_t rows, uint64_t cols, uint32_t box_rows,
                   uint32_t box_cols) {
    struct Entry { const void* base; uint64_t rows, cols; uint32_t br, bc; bool bf16; CUtensorMap map; };
    constexpr int kEntries = 32;
    thread_local Entry cache[kEntries] = {};
    thread_local int next = 0;
    for (int i = 0; i < kEntries; ++i) {
        const Entry& e = cache[i];
        if (e.base == base && e.rows == rows && e.cols == cols && e.br == box_rows && e.bc == box_cols &&
            e.bf16 == bf16) {
            *map = e.map;
            return true;
        }
    }
    if (!encode_map_2d(map, base, bf16, rows, cols, box_rows, box_cols)) return false;
    cache[next] = Entry{base, rows, cols, box_rows, box_cols, bf16, *map};
    next = (next + 1) % kEntries;
    return true;
}

dplr_status make_plan(const dplr_desc* d, Plan* pl) {
    if (!d) return DPLR_ERR_INVALID_ARG;
    if (d->mode != DPLR_GDN && d->mode != DPLR_HDLA && d->mode != DPLR_GENERIC) return DPLR_ERR_INVALID_ARG;
    if (d->in_dtype != DPLR_F32 && d->in_dtype != DPLR_BF16) return DPLR_ERR_INVALID_ARG;
    if (d->B < 1 || d->H < 1 || d->T < 0 || d->dk < 1 || d->dv < 1 || d->chunk < 1) return DPLR_ERR_INVALID_ARG;
    if (d->r_ab < 0 || d->r_kv < 0) return DPLR_ERR_INVALID_ARG;
    if (d->mode == DPLR_GDN && (d->r_ab != 1 || d->r_kv != 1)) return DPLR_ERR_INVALID_ARG;
    if (d->mode == DPLR_HDLA && (d->r_ab != 2 || d->r_kv != 1)) return DPLR_ERR_INVALID_ARG;
    if (!valid_dim(d->dk) || !valid_dim(d->dv)) return DPLR_ERR_UNSUPPORTED;
    if (d->chunk != 64) return DPLR_ERR_UNSUPPORTED;
    if (d->mode == DPLR_GENERIC && (d->r_ab < 1 || d->r_ab > 8 || d->r_kv > 8)) return DPLR_ERR_UNSUPPORTED;
    const long long bh = (long long)d->B * d->H;
    if (bh * (long long)d->T >= (1LL << 31) || bh >= (1LL << 24)) return DPLR_ERR_UNSUPPORTED;

    Plan p{};
    p.mode = d->mode;
    p.bf16 = d->in_dtype == DPLR_BF16;
    p.BH = (int)bh;
    p.T = d->T;
    p.dk = d->dk;
    p.dv = d->dv;
    p.r = d->mode == DPLR_GDN ? 1 : (d->mode == DPLR_HDLA ? 2 : d->r_ab);
    p.p = d->mode == DPLR_GENERIC ? d->r_kv : 0;
    p.cw = wy_block(d->chunk, p.r, p.p);
    p.nb = (d->T + p.cw - 1) / p.cw;
    p.fused = fused_supported(p) ? 1 : 0;
    p.tc = (!p.fused && hdla_tc_supported(p)) ? 1 : 0;
    p.gtc = (!p.fused && !p.tc && generic_tc_supported(p)) ? 1 : 0;
    p.wait_cycles = g_wait_cycles.load(std::memory_order_relaxed);
    if (p.gtc) {
        p.cw = generic_tc_block();
        p.nb = (d->T + p.cw - 1) / p.cw;
        const long long rows = bh * (long long)p.nb * 64;   // c_j rows, addressed as int by the copies
        if (rows >= (1LL << 31)) return DPLR_ERR_UNSUPPORTED;
        size_t total = 0, off_A = 0;
        generic_tc_offsets(p, &off_A, &p.off_c, &total);
        p.off_P = off_A;
        p.off_Q = 0;
        p.ws_stages = total;
        p.ws_bytes = total;
        *pl = p;
        return DPLR_OK;
    }
    if (p.tc) {
        // one unit per (head, 64-token chunk): P_j has 128 rows, addressed as int by the copies
        const long long rows = bh * (long long)((d->T + 63) / 64) * 128;
        if (rows >= (1LL << 31)) return DPLR_ERR_UNSUPPORTED;
        p.cw = 64;
        p.nb = (d->T + 63) / 64;
        size_t total = 0;
        hdla_tc_offsets(p, &p.off_P, &p.off_c, &p.off_Q, &total);
        p.ws_stages = total;
        p.ws_bytes = total;
    } else {
        // fp32 stages: a shorter WY block when the block's tiles would not fit one CTA's shared memory
        while (!p.fused && p.cw > 8 && prep_smem_bytes(p) > 227 * 1024) {
            p.cw /= 2;
            p.nb = (d->T + p.cw - 1) / p.cw;
        }
        const size_t units = (size_t)p.BH * p.nb;
        size_t off = kAlign;   // the first 256 bytes hold the device status word
        p.off_P = off; off = round_up(off + units * (size_t)p.dk * p.dk * sizeof(float));
        p.off_c = off; off = round_up(off + units * (size_t)p.dk * p.dv * sizeof(float));
        p.off_Q = off; off = round_up(off + units * (size_t)p.cw * p.dk * sizeof(float));
        p.ws_stages = off;
        p.ws_bytes = p.fused ? kAlign : p.ws_stages;   // fused: the status word alone
        if ((!p.gtc && prep_smem_bytes(p) > 227 * 1024) || scan_smem_bytes(p) > 227 * 1024) return DPLR_ERR_UNSUPPORTED;
    }
    *pl = p;
    return DPLR_OK;
}

namespace {

dplr_status check_inputs(const Plan& pl, const void* q, const void* k, const void* v, const float* decay,
                         const float* beta, const void* A, const void* Bm, const void* K, const void* V,
                         const float* o) {
    if (pl.T == 0) return DPLR_OK;
    if (!q || !decay || !o) return DPLR_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(decay) || !aligned16(o)) return DPLR_ERR_INVALID_ARG;
    if (pl.mode == DPLR_GENERIC) {
        if (!A || !Bm || !aligned16(A) || !aligned16(Bm)) return DPLR_ERR_INVALID_ARG;
        if (pl.p > 0 && (!K || !V || !aligned16(K) || !aligned16(V))) return DPLR_ERR_INVALID_ARG;
    } else {
        if (!k || !v || !beta) return DPLR_ERR_INVALID_ARG;
        if (!aligned16(k) || !aligned16(v) || !aligned16(beta)) return DPLR_ERR_INVALID_ARG;
    }
    return DPLR_OK;
}

dplr_status check_workspace(size_t need, const void* ws, size_t ws_bytes) {
    if (need == 0) return DPLR_OK;
    if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0) return DPLR_ERR_WORKSPACE;
    return DPLR_OK;
}

ChunkMapArgs map_args(const Plan& pl, const void* q, const void* k, const void* v, const float* decay,
                      const float* beta, const void* A, const void* Bm, const void* K, const void* V,
                      float* o, void* ws) {
    char* base = static_cast<char*>(ws);
    ChunkMapArgs a;
    a.q = q; a.k = k; a.v = v; a.decay = decay; a.beta = beta;
    a.A = A; a.Bm = Bm; a.K = K; a.V = V; a.o = o;
    a.Pm = reinterpret_cast<float*>(base + pl.off_P);
    a.Cm = reinterpret_cast<float*>(base + pl.off_c);
    a.Qm = reinterpret_cast<float*>(base + pl.off_Q);
    return a;
}

ScanArgs scan_args(const Plan& pl, const float* S0, float* o, float* ST, void* ws) {
    char* base = static_cast<char*>(ws);
    ScanArgs a;
    a.S0 = S0; a.o = o; a.ST = ST;
    a.Pm = reinterpret_cast<const float*>(base + pl.off_P);
    a.Cm = reinterpret_cast<const float*>(base + pl.off_c);
    a.Qm = reinterpret_cast<const float*>(base + pl.off_Q);
    return a;
}

}  // namespace
}  // namespace dplr

using namespace dplr;

extern "C" {

dplr_status dplr_la_check(const dplr_desc* desc) {
    Plan pl;
    return make_plan(desc, &pl);
}

size_t dplr_la_workspace_size(const dplr_desc* desc) {
    Plan pl;
    if (make_plan(desc, &pl) != DPLR_OK) return 0;
    return pl.ws_bytes;
}

size_t dplr_la_stage_workspace_size(const dplr_desc* desc) {
    Plan pl;
    if (make_plan(desc, &pl) != DPLR_OK) return 0;
    return pl.ws_stages;
}

int dplr_la_kernel_count(const dplr_desc* desc) {
    Plan pl;
    if (make_plan(desc, &pl) != DPLR_OK) return 0;
    if (pl.fused) return 1;
    return pl.T > 0 ? 2 : 1;
}

dplr_status dplr_la_chunk_maps(const dplr_desc* desc, const void* q, const void* k, const void* v,
                               const float* decay, const float* beta, const void* A, const void* Bm,
                               const void* K, const void* V, float* o, void* workspace, size_t ws_bytes,
                               void* stream) {
    Plan pl;
    dplr_status st = make_plan(desc, &pl);
    if (st != DPLR_OK) return st;
    if ((st = check_inputs(pl, q, k, v, decay, beta, A, Bm, K, V, o)) != DPLR_OK) return st;
    if ((st = check_workspace(pl.ws_stages, workspace, ws_bytes)) != DPLR_OK) return st;
    if (pl.tc) {
        if (launch_hdla_chunks(pl, q, k, v, decay, beta, o, workspace, static_cast<cudaStream_t>(stream)) != cudaSuccess)
            return DPLR_ERR_CUDA;
        return DPLR_OK;
    }
    const ChunkMapArgs a = map_args(pl, q, k, v, decay, beta, A, Bm, K, V, o, workspace);
    const cudaError_t e = pl.gtc ? launch_generic_chunks(pl, a, workspace, static_cast<cudaStream_t>(stream))
                                 : launch_chunk_maps(pl, a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return DPLR_ERR_CUDA;
    return DPLR_OK;
}

dplr_status dplr_la_state_scan(const dplr_desc* desc, const float* S0, float* o, float* S_T, void* workspace,
                               size_t ws_bytes, void* stream) {
    Plan pl;
    dplr_status st = make_plan(desc, &pl);
    if (st != DPLR_OK) return st;
    if ((S0 && !aligned16(S0)) || (S_T && !aligned16(S_T))) return DPLR_ERR_INVALID_ARG;
    if (pl.T > 0 && (!o || !aligned16(o))) return DPLR_ERR_INVALID_ARG;
    if ((st = check_workspace(pl.ws_stages, workspace, ws_bytes)) != DPLR_OK) return st;
    if (pl.tc) {
        if (launch_hdla_chain(pl, S0, o, S_T, workspace, static_cast<cudaStream_t>(stream)) != cudaSuccess)
            return DPLR_ERR_CUDA;
        return DPLR_OK;
    }
    if (pl.gtc) {
        if (launch_generic_chain(pl, S0, o, S_T, workspace, static_cast<cudaStream_t>(stream)) != cudaSuccess)
            return DPLR_ERR_CUDA;
        return DPLR_OK;
    }
    const ScanArgs a = scan_args(pl, S0, o, S_T, workspace);
    if (launch_state_scan(pl, a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return DPLR_ERR_CUDA;
    return DPLR_OK;
}

dplr_status dplr_la_forward(const dplr_desc* desc, const void* q, const void* k, const void* v,
                            const float* decay, const float* beta, const void* A, const void* Bm, const void* K,
                            const void* V, const float* S0, float* o, float* S_T, void* workspace,
                            size_t ws_bytes, void* stream) {
    Plan pl;
    dplr_status st = make_plan(desc, &pl);
    if (st != DPLR_OK) return st;
    if ((st = check_inputs(pl, q, k, v, decay, beta, A, Bm, K, V, o)) != DPLR_OK) return st;
    if ((S0 && !aligned16(S0)) || (S_T && !aligned16(S_T))) return DPLR_ERR_INVALID_ARG;
    if ((st = check_workspace(pl.ws_bytes, workspace, ws_bytes)) != DPLR_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (pl.fused) {
        if (launch_fused(pl, q, k, v, decay, beta, S0, o, S_T, static_cast<int*>(workspace), s) != cudaSuccess)
            return DPLR_ERR_CUDA;
        return DPLR_OK;
    }
    if (pl.tc) {
        if (launch_hdla_chunks(pl, q, k, v, decay, beta, o, workspace, s) != cudaSuccess) return DPLR_ERR_CUDA;
        if (launch_hdla_chain(pl, S0, o, S_T, workspace, s) != cudaSuccess) return DPLR_ERR_CUDA;
        return DPLR_OK;
    }
    const ChunkMapArgs a = map_args(pl, q, k, v, decay, beta, A, Bm, K, V, o, workspace);
    if (pl.gtc) {
        if (launch_generic_chunks(pl, a, workspace, s) != cudaSuccess) return DPLR_ERR_CUDA;
        if (launch_generic_chain(pl, S0, o, S_T, workspace, s) != cudaSuccess) return DPLR_ERR_CUDA;
        return DPLR_OK;
    }
    if (launch_chunk_maps(pl, a, s) != cudaSuccess) return DPLR_ERR_CUDA;
    if (launch_state_scan(pl, scan_args(pl, S0, o, S_T, workspace), s) != cudaSuccess) return DPLR_ERR_CUDA;
    return DPLR_OK;
}

const char* dplr_la_path(const dplr_desc* desc) {
    Plan pl;
    if (make_plan(desc, &pl) != DPLR_OK) return "";
    if (pl.fused) return "gdn_fused_tcgen05";
    if (pl.tc) return "hdla_tcgen05";
    if (pl.gtc) return "generic_tcgen05";
    return "two_stage_fp32";
}

void dplr_la_set_wait_limit(long long cycles) {
    g_wait_cycles.store(cycles > 0 ? cycles : kDefaultWaitCycles, std::memory_order_relaxed);
}

dplr_status dplr_la_read_status(const void* workspace, size_t ws_bytes, int clear, int* status, void* stream) {
    if (status == nullptr) return DPLR_ERR_INVALID_ARG;
    if (workspace == nullptr || ws_bytes < sizeof(int)) return DPLR_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int word = 0;
    if (cudaMemcpyAsync(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return DPLR_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return DPLR_ERR_CUDA;
    *status = word;
    if (clear && cudaMemsetAsync(const_cast<void*>(workspace), 0, sizeof(int), s) != cudaSuccess) return DPLR_ERR_CUDA;
    return DPLR_OK;
}

const char* dplr_status_string(dplr_status s) {
    switch (s) {
        case DPLR_OK: return "DPLR_OK";
        case DPLR_ERR_INVALID_ARG: return "DPLR_ERR_INVALID_ARG: null or misaligned pointer, or malformed descriptor";
        case DPLR_ERR_UNSUPPORTED: return "DPLR_ERR_UNSUPPORTED: shape outside the supported sizes";
        case DPLR_ERR_WORKSPACE: return "DPLR_ERR_WORKSPACE: workspace missing, misaligned or too small";
        case DPLR_ERR_CUDA: return "DPLR_ERR_CUDA: a CUDA call or kernel launch failed";
        case DPLR_ERR_TIMEOUT: return "DPLR_ERR_TIMEOUT: a bounded device-side wait gave up";
    }
    return "unknown dplr_status";
}

}  // extern "C"
