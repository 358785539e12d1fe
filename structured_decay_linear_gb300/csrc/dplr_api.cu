// Host side of the libdplr C ABI: descriptor validation, workspace plan, launches.
#include <cstring>

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

}  // namespace

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
    const size_t units = (size_t)p.BH * p.nb;
    size_t off = kAlign;   // the first 256 bytes hold the device status word
    p.off_P = off; off = round_up(off + units * (size_t)p.dk * p.dk * sizeof(float));
    p.off_c = off; off = round_up(off + units * (size_t)p.dk * p.dv * sizeof(float));
    p.off_Q = off; off = round_up(off + units * (size_t)p.cw * p.dk * sizeof(float));
    p.ws_stages = off;
    p.fused = fused_supported(p) ? 1 : 0;
    p.wait_cycles = g_wait_cycles.load(std::memory_order_relaxed);
    p.ws_bytes = p.fused ? kAlign : p.ws_stages;   // fused: the status word alone
    if (prep_smem_bytes(p) > 227 * 1024 || scan_smem_bytes(p) > 227 * 1024) return DPLR_ERR_UNSUPPORTED;
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
    const ChunkMapArgs a = map_args(pl, q, k, v, decay, beta, A, Bm, K, V, o, workspace);
    if (launch_chunk_maps(pl, a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return DPLR_ERR_CUDA;
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
    if (launch_chunk_maps(pl, map_args(pl, q, k, v, decay, beta, A, Bm, K, V, o, workspace), s) != cudaSuccess)
        return DPLR_ERR_CUDA;
    if (launch_state_scan(pl, scan_args(pl, S0, o, S_T, workspace), s) != cudaSuccess) return DPLR_ERR_CUDA;
    return DPLR_OK;
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
