// dplr_la_forward_host: the forward from host buffers, with the transfers overlapped.
//
// The heads (B*H) are split into `groups` equal groups. Each group's inputs are copied
// to a device staging slot, its forward runs there (dplr_la_forward on a sub-descriptor
// with B = 1, H = B*H/groups), and its outputs are copied back; `slots` staging slots are
// used in turn. Copies into the device run on one internal stream, copies back on a
// second, and each slot's forward on its own compute stream, with events between them:
// while group g computes, group g+1 is being copied in and group g-1 copied out, and
// forwards of different groups run side by side on different SMs.
//
// dplr_la_forward_host_seq splits the sequence instead: segment g holds tokens [g Ts, (g+1) Ts) of every head
// (Ts a multiple of the 64-token chunk). Its inputs arrive by one 2-D copy per tensor (a row per head), its
// forward starts from the state the previous segment's forward left in one of two device state buffers,
// and its outputs go back by 2-D copies. The forwards run one after another on one stream, each a short
// one (Ts tokens), so the last copy out follows the last copy in by one short forward.
//
// The internal streams and events are created once per device (on the first call made
// while that device is current) and reused; calls on one device are serialised by a lock
// while they enqueue, and their GPU work runs in call order. Nothing here allocates device
// memory: the staging area is the caller's.
#include <cstdint>
#include <cstring>
#include <mutex>

#include "dplr_internal.h"

namespace dplr {
namespace {

constexpr int kMaxSlots = 8;
constexpr int kMaxDevices = 64;
constexpr size_t kAlign = 256;

struct HostPipe {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr, comp[kMaxSlots] = {};
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t ev_in[kMaxSlots] = {}, ev_comp[kMaxSlots] = {}, ev_free[kMaxSlots] = {};
};

std::mutex g_pipe_mu;
HostPipe g_pipe[kMaxDevices];

cudaError_t make_pipe(HostPipe& p) {
    const unsigned sf = cudaStreamNonBlocking, ef = cudaEventDisableTiming;
    cudaError_t e = cudaStreamCreateWithFlags(&p.in, sf);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p.out, sf);
    for (int i = 0; i < kMaxSlots && e == cudaSuccess; ++i) e = cudaStreamCreateWithFlags(&p.comp[i], sf);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.start, ef);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.done, ef);
    for (int i = 0; i < kMaxSlots && e == cudaSuccess; ++i) {
        e = cudaEventCreateWithFlags(&p.ev_in[i], ef);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.ev_comp[i], ef);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.ev_free[i], ef);
    }
    p.ready = (e == cudaSuccess);
    return e;
}

size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Byte sizes of one group's tensors (0 where the mode does not use a tensor).
struct GroupBytes {
    size_t q, k, v, decay, beta, A, Bm, K, V, S, o, ws, slot;
};

bool group_bytes(const dplr_desc& sub, bool with_s0, bool with_st, GroupBytes* g) {
    const size_t H = (size_t)sub.H, T = (size_t)sub.T, dk = (size_t)sub.dk, dv = (size_t)sub.dv;
    const size_t e = sub.in_dtype == DPLR_BF16 ? 2 : 4;
    const size_t r = (size_t)sub.r_ab, p = (size_t)sub.r_kv;
    std::memset(g, 0, sizeof(*g));
    g->q = H * T * dk * e;
    if (sub.mode == DPLR_GENERIC) {
        g->decay = H * T * dk * 4;
        g->A = g->Bm = H * T * r * dk * e;
        g->K = H * T * p * dk * e;
        g->V = H * T * p * dv * e;
    } else {
        g->k = H * T * dk * e;
        g->v = H * T * dv * e;
        g->decay = H * T * (sub.mode == DPLR_GDN ? 1 : dk) * 4;
        g->beta = H * T * 4;
    }
    g->S = H * dk * dv * 4;
    g->o = H * T * dv * 4;
    g->ws = dplr_la_workspace_size(&sub);
    if (g->ws == 0) return false;
    g->slot = up(g->q) + up(g->k) + up(g->v) + up(g->decay) + up(g->beta) + up(g->A) + up(g->Bm) + up(g->K) +
              up(g->V) + (with_s0 ? up(g->S) : 0) + up(g->o) + (with_st ? up(g->S) : 0) + up(g->ws);
    return true;
}

bool sub_desc(const dplr_desc* desc, int groups, dplr_desc* sub) {
    if (desc == nullptr || groups < 1) return false;
    const long long bh = (long long)desc->B * (long long)desc->H;
    if (bh <= 0 || bh % groups != 0) return false;
    *sub = *desc;
    sub->B = 1;
    sub->H = (int)(bh / groups);
    return dplr_la_check(sub) == DPLR_OK;
}

// Per-token row bytes of each host tensor, for the 2-D copies of sequence segments.
struct RowBytes {
    size_t q, k, v, decay, beta, A, Bm, K, V, o;
};

RowBytes row_bytes(const dplr_desc& d) {
    const size_t e = d.in_dtype == DPLR_BF16 ? 2 : 4, dk = (size_t)d.dk, dv = (size_t)d.dv;
    RowBytes r;
    std::memset(&r, 0, sizeof(r));
    r.q = dk * e;
    r.o = dv * 4;
    if (d.mode == DPLR_GENERIC) {
        r.decay = dk * 4;
        r.A = r.Bm = (size_t)d.r_ab * dk * e;
        r.K = (size_t)d.r_kv * dk * e;
        r.V = (size_t)d.r_kv * dv * e;
    } else {
        r.k = dk * e;
        r.v = dv * e;
        r.decay = d.mode == DPLR_GDN ? 4 : dk * 4;
        r.beta = 4;
    }
    return r;
}

// Segment length (a multiple of the chunk) and count for `segments` requested segments.
bool seq_split(const dplr_desc* desc, int segments, int* ts, int* nseg) {
    if (desc == nullptr || segments < 1) return false;
    const int C = 64;
    const int T = desc->T;
    const int per = (T + segments - 1) / segments;
    *ts = T == 0 ? C : (per + C - 1) / C * C;
    *nseg = T == 0 ? 1 : (T + *ts - 1) / *ts;
    return true;
}

// Staging bytes of one segment slot (inputs, o and the workspace for ts tokens) and of the two state buffers.
bool seq_bytes(const dplr_desc* desc, int ts, size_t* slot, size_t* state) {
    dplr_desc sub = *desc;
    sub.T = ts;
    if (dplr_la_check(&sub) != DPLR_OK) return false;
    const size_t ws = dplr_la_workspace_size(&sub);
    if (ws == 0) return false;
    const RowBytes r = row_bytes(*desc);
    const size_t n = (size_t)desc->B * (size_t)desc->H * (size_t)ts;
    *slot = up(n * r.q) + up(n * r.k) + up(n * r.v) + up(n * r.decay) + up(n * r.beta) + up(n * r.A) + up(n * r.Bm) +
            up(n * r.K) + up(n * r.V) + up(n * r.o) + up(ws);
    *state = up((size_t)desc->B * (size_t)desc->H * (size_t)desc->dk * (size_t)desc->dv * 4);
    return true;
}

}  // namespace
}  // namespace dplr

extern "C" size_t dplr_la_host_workspace_size(const dplr_desc* desc, int groups, int slots) {
    using namespace dplr;
    dplr_desc sub;
    if (slots < 1 || slots > kMaxSlots || !sub_desc(desc, groups, &sub)) return 0;
    GroupBytes g;
    if (!group_bytes(sub, true, true, &g)) return 0;
    return g.slot * (size_t)(slots < groups ? slots : groups);
}

extern "C" dplr_status dplr_la_forward_host(const dplr_desc* desc, const void* q, const void* k, const void* v,
                                            const float* decay, const float* beta, const void* A, const void* Bm,
                                            const void* K, const void* V, const float* S0, float* o, float* S_T,
                                            void* staging, size_t staging_bytes, int groups, int slots,
                                            void* stream) {
    using namespace dplr;
    dplr_status st = dplr_la_check(desc);
    if (st != DPLR_OK) return st;
    dplr_desc sub;
    if (slots < 1 || slots > kMaxSlots || !sub_desc(desc, groups, &sub)) return DPLR_ERR_INVALID_ARG;
    const bool generic = desc->mode == DPLR_GENERIC;
    if (q == nullptr || decay == nullptr || o == nullptr) return DPLR_ERR_INVALID_ARG;
    if (generic ? (A == nullptr || Bm == nullptr || (desc->r_kv > 0 && (K == nullptr || V == nullptr)))
                : (k == nullptr || v == nullptr || beta == nullptr))
        return DPLR_ERR_INVALID_ARG;
    GroupBytes g;
    if (!group_bytes(sub, S0 != nullptr, S_T != nullptr, &g)) return DPLR_ERR_INVALID_ARG;
    const int nslot = slots < groups ? slots : groups;
    if (staging == nullptr || (reinterpret_cast<uintptr_t>(staging) % kAlign) != 0 ||
        staging_bytes < g.slot * (size_t)nslot)
        return DPLR_ERR_WORKSPACE;
    if (desc->T == 0 && S_T == nullptr) return DPLR_OK;

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DPLR_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_pipe_mu);
    HostPipe& p = g_pipe[dev];
    if (!p.ready && make_pipe(p) != cudaSuccess) return DPLR_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

#define DPLR_CK(x) do { if ((x) != cudaSuccess) return DPLR_ERR_CUDA; } while (0)
    // everything starts after the work already queued on the caller's stream
    DPLR_CK(cudaEventRecord(p.start, s));
    DPLR_CK(cudaStreamWaitEvent(p.in, p.start, 0));
    DPLR_CK(cudaStreamWaitEvent(p.out, p.start, 0));
    for (int i = 0; i < nslot; ++i) DPLR_CK(cudaStreamWaitEvent(p.comp[i], p.start, 0));

    const auto H2D = cudaMemcpyHostToDevice, D2H = cudaMemcpyDeviceToHost;
    for (int gi = 0; gi < groups; ++gi) {
        const int si = gi % nslot;
        unsigned char* base = static_cast<unsigned char*>(staging) + (size_t)si * g.slot;
        // carve the slot: inputs, then outputs, then the workspace
        size_t off = 0;
        auto carve = [&](size_t bytes) -> unsigned char* {   // (a valid address even for 0 bytes)
            unsigned char* r = base + off;
            off += up(bytes);
            return r;
        };
        unsigned char *dq = carve(g.q), *dk_ = carve(g.k), *dv_ = carve(g.v), *dd = carve(g.decay),
                      *db = carve(g.beta), *dA = carve(g.A), *dB = carve(g.Bm), *dK = carve(g.K), *dV = carve(g.V);
        if (generic) dk_ = dv_ = db = nullptr;
        else dA = dB = dK = dV = nullptr;
        unsigned char* dS0 = S0 ? carve(g.S) : nullptr;
        unsigned char* dO = carve(g.o);
        unsigned char* dST = S_T ? carve(g.S) : nullptr;
        unsigned char* dws = carve(g.ws);
        const size_t gg = (size_t)gi;
        auto in_copy = [&](unsigned char* dst, const void* src, size_t bytes) -> bool {
            if (!bytes || src == nullptr) return true;
            return cudaMemcpyAsync(dst, static_cast<const unsigned char*>(src) + gg * bytes, bytes, H2D, p.in) ==
                   cudaSuccess;
        };
        // the slot's previous group has been copied out (and so computed)
        if (gi >= nslot) DPLR_CK(cudaStreamWaitEvent(p.in, p.ev_free[si], 0));
        if (!in_copy(dq, q, g.q) || !in_copy(dk_, k, g.k) || !in_copy(dv_, v, g.v) || !in_copy(dd, decay, g.decay) ||
            !in_copy(db, beta, g.beta) || !in_copy(dA, A, g.A) || !in_copy(dB, Bm, g.Bm) || !in_copy(dK, K, g.K) ||
            !in_copy(dV, V, g.V) || !in_copy(dS0, S0, S0 ? g.S : 0))
            return DPLR_ERR_CUDA;
        if (g.ws) DPLR_CK(cudaMemsetAsync(dws, 0, g.ws < kAlign ? g.ws : kAlign, p.in));   // status word
        DPLR_CK(cudaEventRecord(p.ev_in[si], p.in));
        DPLR_CK(cudaStreamWaitEvent(p.comp[si], p.ev_in[si], 0));
        st = dplr_la_forward(&sub, dq, dk_, dv_, reinterpret_cast<const float*>(dd), reinterpret_cast<const float*>(db),
                             dA, dB, dK, dV, reinterpret_cast<const float*>(dS0), reinterpret_cast<float*>(dO),
                             reinterpret_cast<float*>(dST), dws, g.ws, p.comp[si]);
        if (st != DPLR_OK) return st;
        DPLR_CK(cudaEventRecord(p.ev_comp[si], p.comp[si]));
        DPLR_CK(cudaStreamWaitEvent(p.out, p.ev_comp[si], 0));
        DPLR_CK(cudaMemcpyAsync(reinterpret_cast<unsigned char*>(o) + gg * g.o, dO, g.o, D2H, p.out));
        if (S_T) DPLR_CK(cudaMemcpyAsync(reinterpret_cast<unsigned char*>(S_T) + gg * g.S, dST, g.S, D2H, p.out));
        DPLR_CK(cudaEventRecord(p.ev_free[si], p.out));
    }
    // the caller's stream resumes once the last copy back is done (it follows every forward)
    DPLR_CK(cudaEventRecord(p.done, p.out));
    DPLR_CK(cudaStreamWaitEvent(s, p.done, 0));
#undef DPLR_CK
    return DPLR_OK;
}

extern "C" size_t dplr_la_host_seq_workspace_size(const dplr_desc* desc, int segments, int slots) {
    using namespace dplr;
    int ts = 0, nseg = 0;
    if (slots < 1 || slots > kMaxSlots || dplr_la_check(desc) != DPLR_OK || !seq_split(desc, segments, &ts, &nseg))
        return 0;
    size_t slot = 0, state = 0;
    if (!seq_bytes(desc, ts, &slot, &state)) return 0;
    return 2 * state + slot * (size_t)(slots < nseg ? slots : nseg);
}

extern "C" dplr_status dplr_la_forward_host_seq(const dplr_desc* desc, const void* q, const void* k, const void* v,
                                                const float* decay, const float* beta, const void* A, const void* Bm,
                                                const void* K, const void* V, const float* S0, float* o, float* S_T,
                                                void* staging, size_t staging_bytes, int segments, int slots,
                                                void* stream) {
    using namespace dplr;
    dplr_status st = dplr_la_check(desc);
    if (st != DPLR_OK) return st;
    int ts = 0, nseg = 0;
    if (slots < 1 || slots > kMaxSlots || !seq_split(desc, segments, &ts, &nseg)) return DPLR_ERR_INVALID_ARG;
    const bool generic = desc->mode == DPLR_GENERIC;
    if (desc->T > 0) {   // (an empty sequence has no token tensors: only S0 -> S_T)
        if (q == nullptr || decay == nullptr || o == nullptr) return DPLR_ERR_INVALID_ARG;
        if (generic ? (A == nullptr || Bm == nullptr || (desc->r_kv > 0 && (K == nullptr || V == nullptr)))
                    : (k == nullptr || v == nullptr || beta == nullptr))
            return DPLR_ERR_INVALID_ARG;
    }
    size_t slot = 0, state = 0;
    if (!seq_bytes(desc, ts, &slot, &state)) return DPLR_ERR_INVALID_ARG;
    const int nslot = slots < nseg ? slots : nseg;
    if (staging == nullptr || (reinterpret_cast<uintptr_t>(staging) % kAlign) != 0 ||
        staging_bytes < 2 * state + slot * (size_t)nslot)
        return DPLR_ERR_WORKSPACE;

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DPLR_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_pipe_mu);
    HostPipe& p = g_pipe[dev];
    if (!p.ready && make_pipe(p) != cudaSuccess) return DPLR_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaStream_t comp = p.comp[0];   // the forwards, one after another (each starts from the last one's state)

#define DPLR_CK(x) do { if ((x) != cudaSuccess) return DPLR_ERR_CUDA; } while (0)
    DPLR_CK(cudaEventRecord(p.start, s));
    DPLR_CK(cudaStreamWaitEvent(p.in, p.start, 0));
    DPLR_CK(cudaStreamWaitEvent(p.out, p.start, 0));
    DPLR_CK(cudaStreamWaitEvent(comp, p.start, 0));

    const RowBytes rb = row_bytes(*desc);
    const size_t bh = (size_t)desc->B * (size_t)desc->H, T = (size_t)desc->T;
    unsigned char* st_buf[2] = {static_cast<unsigned char*>(staging), static_cast<unsigned char*>(staging) + state};
    const auto H2D = cudaMemcpyHostToDevice, D2H = cudaMemcpyDeviceToHost;
    // state before segment 0: S0 (or none)
    if (S0) DPLR_CK(cudaMemcpyAsync(st_buf[0], S0, bh * desc->dk * desc->dv * 4, H2D, p.in));
    for (int gi = 0; gi < nseg; ++gi) {
        const int si = gi % nslot;
        const size_t t0 = (size_t)gi * (size_t)ts;
        const size_t tg = T == 0 ? 0 : (t0 + (size_t)ts <= T ? (size_t)ts : T - t0);
        dplr_desc sub = *desc;
        sub.T = (int)tg;
        unsigned char* base = st_buf[1] + state + (size_t)si * slot;
        size_t off = 0;
        const size_t nmax = bh * (size_t)ts;
        auto carve = [&](size_t row) -> unsigned char* {
            unsigned char* r = base + off;
            off += up(nmax * row);
            return r;
        };
        unsigned char *dq = carve(rb.q), *dk_ = carve(rb.k), *dv_ = carve(rb.v), *dd = carve(rb.decay),
                      *db = carve(rb.beta), *dA = carve(rb.A), *dB = carve(rb.Bm), *dK = carve(rb.K), *dV = carve(rb.V),
                      *dO = carve(rb.o);
        unsigned char* dws = base + off;
        const size_t ws = dplr_la_workspace_size(&sub);   // (at most the full segment's, which the slot holds)
        if (ws > slot - off) return DPLR_ERR_WORKSPACE;
        if (generic) dk_ = dv_ = db = nullptr;
        else dA = dB = dK = dV = nullptr;
        // tokens [t0, t0 + tg) of every head: one row of tg * row bytes per head
        auto in_copy = [&](unsigned char* dst, const void* src, size_t row) -> bool {
            if (!row || src == nullptr || tg == 0) return true;
            return cudaMemcpy2DAsync(dst, tg * row, static_cast<const unsigned char*>(src) + t0 * row, T * row,
                                     tg * row, bh, H2D, p.in) == cudaSuccess;
        };
        if (gi >= nslot) DPLR_CK(cudaStreamWaitEvent(p.in, p.ev_free[si], 0));   // the slot's outputs are out
        if (!in_copy(dq, q, rb.q) || !in_copy(dk_, k, rb.k) || !in_copy(dv_, v, rb.v) || !in_copy(dd, decay, rb.decay) ||
            !in_copy(db, beta, rb.beta) || !in_copy(dA, A, rb.A) || !in_copy(dB, Bm, rb.Bm) || !in_copy(dK, K, rb.K) ||
            !in_copy(dV, V, rb.V))
            return DPLR_ERR_CUDA;
        if (ws) DPLR_CK(cudaMemsetAsync(dws, 0, ws < kAlign ? ws : kAlign, p.in));   // status word
        DPLR_CK(cudaEventRecord(p.ev_in[si], p.in));
        DPLR_CK(cudaStreamWaitEvent(comp, p.ev_in[si], 0));
        const float* s_in = (gi == 0 && S0 == nullptr) ? nullptr : reinterpret_cast<const float*>(st_buf[gi & 1]);
        float* s_out = reinterpret_cast<float*>(st_buf[(gi + 1) & 1]);
        st = dplr_la_forward(&sub, dq, dk_, dv_, reinterpret_cast<const float*>(dd), reinterpret_cast<const float*>(db),
                             dA, dB, dK, dV, s_in, reinterpret_cast<float*>(dO), s_out, dws, ws, comp);
        if (st != DPLR_OK) return st;
        DPLR_CK(cudaEventRecord(p.ev_comp[si], comp));
        DPLR_CK(cudaStreamWaitEvent(p.out, p.ev_comp[si], 0));
        if (tg) DPLR_CK(cudaMemcpy2DAsync(reinterpret_cast<unsigned char*>(o) + t0 * rb.o, T * rb.o, dO, tg * rb.o,
                                          tg * rb.o, bh, D2H, p.out));
        DPLR_CK(cudaEventRecord(p.ev_free[si], p.out));
    }
    if (S_T) DPLR_CK(cudaMemcpyAsync(S_T, st_buf[nseg & 1], bh * desc->dk * desc->dv * 4, D2H, p.out));
    DPLR_CK(cudaEventRecord(p.done, p.out));
    DPLR_CK(cudaStreamWaitEvent(s, p.done, 0));
#undef DPLR_CK
    return DPLR_OK;
}
