/*
 * dplr.h -- C ABI of libdplr: the chunkwise-parallel forward of linear attention
 * with a diagonal-plus-low-rank (DPLR) decay, for NVIDIA GB300 (sm_103a).
 *
 * The operation (per batch b and head h, state S in R^{dk x dv}, tokens t = 1..T):
 *
 *     S_t = (D_t - A_t B_t^T) S_{t-1} + K_t V_t^T,        o_t = S_t^T q_t
 *
 * is the general recurrence of "Householder-Diagonalized Linear Attention"
 * (HDLA page, Key design 3, displayed equation), with A_t, B_t in R^{dk x r_ab},
 * K_t in R^{dk x r_kv}, V_t in R^{dv x r_kv}, D_t diagonal. Two structured cases
 * build the factors from (k, v, decay, beta) on the device:
 *
 *   DPLR_GDN   Gated DeltaNet, P_t = exp(g_t)(I - beta_t k_t k_t^T), write
 *              beta_t k_t v_t^T (HLA page, Prerequisites and Method step 1).
 *   DPLR_HDLA  P_t = (I - beta_t k_t k_t^T) Diag(lambda_t) (I - beta_t k_t k_t^T),
 *              write beta_t k_t v_t^T (HDLA page, Key design 2).
 *   DPLR_GENERIC  A, B, K, V and log(diag D) given directly (Key design 3).
 *
 * The readout uses the state after token t's update (o_t = S_t^T q_t); there is
 * no 1/sqrt(dk) factor (pre-scale q if wanted). The state enters as S0 and
 * leaves as S_T, so a sequence can be continued across calls.
 *
 * The method is the two-stage chunkwise algorithm of the HDLA page (Key design
 * 3): stage 1 computes, for every chunk independently, its exact affine map
 * S -> P_j S + c_j and its readout map (the rank-generalised WY/UT transform);
 * stage 2 scans the chunk maps in order and reads out o.
 *
 * Layouts: every tensor is contiguous, row-major, on the device of `stream`.
 *   q      [B,H,T,dk]   in_dtype
 *   k      [B,H,T,dk]   in_dtype   (GDN, HDLA)
 *   v      [B,H,T,dv]   in_dtype   (GDN, HDLA)
 *   decay  fp32, log-space: GDN [B,H,T] (log gate g <= 0);
 *          HDLA and GENERIC [B,H,T,dk] (log lambda; D_t = Diag(exp(decay_t)))
 *   beta   [B,H,T]      fp32       (GDN, HDLA; ignored for GENERIC)
 *   A, Bm  [B,H,T,r_ab,dk] in_dtype (GENERIC; row i is column i of A_t / B_t)
 *   K      [B,H,T,r_kv,dk] in_dtype (GENERIC)
 *   V      [B,H,T,r_kv,dv] in_dtype (GENERIC)
 *   S0     [B,H,dk,dv]  fp32, may be NULL (zero initial state)
 *   o      [B,H,T,dv]   fp32 (written)
 *   S_T    [B,H,dk,dv]  fp32, may be NULL (final state not returned)
 *
 * Ownership: the caller allocates every buffer, including the workspace
 * (size from dplr_la_workspace_size). The library allocates no device memory
 * and keeps no state between calls, apart from per-device kernel attributes
 * set once. All calls are asynchronous on `stream` (a cudaStream_t; NULL is
 * the legacy default stream). Calls that share a workspace must not overlap.
 *
 * Errors: argument, shape and alignment problems return a status code before
 * anything is launched (nothing is written). A failed launch returns
 * DPLR_ERR_CUDA. Every pointer must be 16-byte aligned.
 *
 * Supported sizes: dk, dv in {32, 64, 128}; chunk = 64; B, H >= 1; T >= 0 with
 * B*H*T < 2^31; GDN has r_ab = r_kv = 1, HDLA r_ab = 2, r_kv = 1; GENERIC
 * 1 <= r_ab <= 8 and 0 <= r_kv <= 8.
 */
#ifndef DPLR_H
#define DPLR_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DPLR_API __attribute__((visibility("default")))
#else
#define DPLR_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DPLR_OK = 0,
    DPLR_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad shape or enum value */
    DPLR_ERR_UNSUPPORTED = 2,   /* well-formed but outside the supported sizes */
    DPLR_ERR_WORKSPACE = 3,     /* workspace pointer null or smaller than required */
    DPLR_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed */
    DPLR_ERR_TIMEOUT = 5        /* a bounded device-side wait gave up (device status word) */
} dplr_status;

typedef enum { DPLR_GDN = 1, DPLR_HDLA = 2, DPLR_GENERIC = 3 } dplr_mode;
typedef enum { DPLR_F32 = 0, DPLR_BF16 = 1 } dplr_dtype;

/* Problem descriptor. r_ab / r_kv are fixed by the structured modes (GDN 1/1,
 * HDLA 2/1) and must be given with those values. */
typedef struct {
    int32_t mode;      /* dplr_mode */
    int32_t in_dtype;  /* dplr_dtype of q, k, v, A, Bm, K, V */
    int32_t B, H, T;   /* batch, heads, sequence length */
    int32_t dk, dv;    /* key / value head dimensions */
    int32_t r_ab;      /* rank of the low-rank decay term A_t B_t^T */
    int32_t r_kv;      /* rank of the write term K_t V_t^T */
    int32_t chunk;     /* chunk length C of the chunkwise algorithm (64) */
} dplr_desc;

/* Bytes of device workspace dplr_la_forward needs for `desc`; 0 if `desc` is
 * invalid or unsupported (call dplr_la_check for the reason). The first 256 bytes
 * of every workspace hold the device status word (its first int32): a kernel whose
 * bounded wait gives up sets it to DPLR_ERR_TIMEOUT (DPLR_ERR_CUDA if its shared
 * memory is not 1024-byte aligned, in which case it computes nothing). Kernels
 * never clear it: zero it once after allocating the workspace, and read it with
 * dplr_la_read_status. The rest holds the per-chunk maps of the paths that keep
 * them between kernels. */
DPLR_API size_t dplr_la_workspace_size(const dplr_desc* desc);

/* Bytes of device workspace dplr_la_chunk_maps and dplr_la_state_scan need for
 * `desc` (the chunk maps of every chunk); 0 if `desc` is invalid. */
DPLR_API size_t dplr_la_stage_workspace_size(const dplr_desc* desc);

/* Validates `desc` alone (no pointers). DPLR_OK if the shape is supported. */
DPLR_API dplr_status dplr_la_check(const dplr_desc* desc);

/* The whole forward: o and (optionally) S_T from the inputs and S0.
 * Structured modes read q, k, v, decay, beta and ignore A, Bm, K, V;
 * GENERIC reads q, decay, A, Bm, K (if r_kv > 0), V (if r_kv > 0) and ignores
 * k, v, beta. */
DPLR_API dplr_status dplr_la_forward(const dplr_desc* desc,
                            const void* q, const void* k, const void* v,
                            const float* decay, const float* beta,
                            const void* A, const void* Bm, const void* K, const void* V,
                            const float* S0, float* o, float* S_T,
                            void* workspace, size_t ws_bytes, void* stream);

/* Stage 1 alone (HDLA page, Key design 3, stage "compute each chunk's
 * quantities in parallel"): per chunk, the cumulative decay, the factor build,
 * the Gram blocks, the UT/WY triangular solve, and from them the chunk's affine
 * map (P_j, c_j) and readout map (Q'_j, local output). Writes the maps to the
 * workspace (dplr_la_stage_workspace_size bytes) and each chunk's
 * zero-initial-state output into o. Other arguments as for dplr_la_forward. */
DPLR_API dplr_status dplr_la_chunk_maps(const dplr_desc* desc,
                               const void* q, const void* k, const void* v,
                               const float* decay, const float* beta,
                               const void* A, const void* Bm, const void* K, const void* V,
                               float* o, void* workspace, size_t ws_bytes, void* stream);

/* Stage 2 alone (HDLA page, Key design 3, "serially compute the chunk-state
 * checkpoints"): scans the chunk maps written by dplr_la_chunk_maps in chunk
 * order, S_j = P_j S_{j-1} + c_j from S0, adds each chunk's state readout
 * Q'_j S_{j-1} into o and writes S_T. Must follow dplr_la_chunk_maps with the
 * same descriptor and workspace on the same stream. */
DPLR_API dplr_status dplr_la_state_scan(const dplr_desc* desc, const float* S0, float* o, float* S_T,
                               void* workspace, size_t ws_bytes, void* stream);

/* Synchronous check of the device status word (no counterpart in the paper). Waits
 * for the work queued on `stream`, then copies the first int32 of `workspace` (a
 * dplr_la_forward / stage workspace of `ws_bytes` bytes) into *status: DPLR_OK, or
 * the code a kernel left there (DPLR_ERR_TIMEOUT after a bounded device-side wait
 * gave up). With `clear` nonzero the word is zeroed afterwards on `stream`. Returns
 * DPLR_ERR_WORKSPACE for a null or undersized workspace, DPLR_ERR_INVALID_ARG for a
 * null `status`, DPLR_ERR_CUDA if a CUDA call fails (including an earlier
 * asynchronous failure of the stream's work). Blocks the calling thread. */
DPLR_API dplr_status dplr_la_read_status(const void* workspace, size_t ws_bytes, int clear, int* status,
                                         void* stream);

/* Sets the limit, in SM clock cycles, of every bounded device-side wait that a kernel
 * makes on another part of the same launch (no counterpart in the paper). It applies
 * to the launches of later calls in the process; `cycles` <= 0 restores the default
 * (4e9 cycles, about 2 s). A wait that reaches the limit gives up: the kernel sets the
 * status word to DPLR_ERR_TIMEOUT, waits for its own copies and tensor-core work
 * already in flight, and returns with its outputs incomplete. Meant for tests of that
 * path; a small limit makes correct launches give up too. */
DPLR_API void dplr_la_set_wait_limit(long long cycles);

/* One recurrent step for every (batch, head): the decode-time form of the recurrence, whose
 * state has constant size (HDLA page, research background; HLA page, results: per-token decode
 * cost). S <- (D_t - A_t B_t^T) S + K_t V_t^T in place, then o = S^T q_t, exactly as one token
 * of dplr_la_forward (GDN and HDLA build the factors from k, v, decay, beta as there).
 * desc->T must be 1: the inputs are the layouts above with T = 1 (q [B,H,1,dk], ...).
 * S: [B,H,dk,dv] fp32, read and written in place (device, 16-byte aligned). o: [B,H,1,dv]
 * fp32. All arithmetic is fp32. Needs no workspace and allocates nothing; asynchronous on
 * `stream`. Errors: as dplr_la_forward; DPLR_ERR_INVALID_ARG when desc->T != 1. */
DPLR_API dplr_status dplr_la_decode_step(const dplr_desc* desc,
                                const void* q, const void* k, const void* v,
                                const float* decay, const float* beta,
                                const void* A, const void* Bm, const void* K, const void* V,
                                float* S, float* o, void* stream);

/* Backward of dplr_la_forward: the gradients of a scalar loss L with respect to every input,
 * given dO = dL/do [B,H,T,dv] and dST = dL/dS_T [B,H,dk,dv] (nullable: zero), for the same
 * descriptor and inputs as the forward. The chunkwise algorithm exists for chunk-parallel
 * training (HDLA page, Key design 3); its backward reuses the WY factors of every block:
 * the forward again at blocks of cb tokens keeping the state before each block (cb = 32 for
 * GDN, 16 for HDLA, the largest power of two with cb max(r_ab, r_kv) <= 32 in the generic mode,
 * so ranks up to 8), the blocks' state gradients
 * backwards through the transposed block maps, then every block's input gradients in parallel.
 * Outputs, all fp32 whatever the input type, same layouts as the inputs:
 *   dq [B,H,T,dk]; ddecay (GDN [B,H,T], HDLA/generic [B,H,T,dk]); dS0 [B,H,dk,dv] (nullable);
 *   GDN, HDLA: dk [B,H,T,dk], dv [B,H,T,dv], dbeta [B,H,T];
 *   generic:   dA, dBm [B,H,T,r_ab,dk], dK [B,H,T,r_kv,dk], dV [B,H,T,r_kv,dv].
 * Unused outputs of a mode may be null. The arithmetic is fp32 on the CUDA cores. Workspace:
 * dplr_la_backward_workspace_size(desc) bytes (the maps, states and state gradients of every
 * block), 256-byte aligned, owned by the caller. Asynchronous on `stream`; allocates nothing.
 * Errors: as dplr_la_forward; DPLR_ERR_UNSUPPORTED for dk or dv above 128. */
DPLR_API size_t dplr_la_backward_workspace_size(const dplr_desc* desc);
DPLR_API dplr_status dplr_la_backward(const dplr_desc* desc,
                             const void* q, const void* k, const void* v,
                             const float* decay, const float* beta,
                             const void* A, const void* Bm, const void* K, const void* V,
                             const float* S0, const float* dO, const float* dST,
                             float* dq, float* dk, float* dv, float* ddecay, float* dbeta,
                             float* dA, float* dBm, float* dK, float* dV, float* dS0,
                             void* workspace, size_t ws_bytes, void* stream);

/* HLA's query-conditioned composition of chunk transitions ("HLA: Expressive Hybrid Linear Attention via
 * Chunk-Wise Dynamic Mixing", Method steps 1, 2, 4, 5) on the Gated DeltaNet update of `desc` (mode DPLR_GDN,
 * dk, dv <= 128): the sequence is cut into chunks of L tokens (64, 128 or 256), chunk j summarised exactly as
 * S -> A_j S + B_j; query token i of chunk c starts from a zero state, composes the earlier chunks in order as
 * S <- ((1 - w_ij) I + w_ij A_j) S + w_ij B_j, runs its own chunk's causal prefix, and reads o_i = S^T q_i.
 * W [B,H,T,N] fp32, N = ceil(T / L): the gates (only w_ij with j < c are used); gates below `theta` count as
 * zero. q, k, v, g, beta as for dplr_la_forward (no initial state). o [B,H,T,dv] fp32. Workspace:
 * dplr_hla_workspace_size(desc, L) bytes, 256-byte aligned; its first 256 bytes are a status word, zeroed by the
 * call, into which a bounded wait of the tensor-core pass that gives up writes DPLR_ERR_TIMEOUT (read it with
 * dplr_la_read_status). For dk = dv = 128 the maps of 64-token blocks (bf16 inputs), the L-chunk summaries
 * composed from them, and the gated composition (at most 256 chunks; dplr_hla_path) run on the tensor cores (bf16
 * hi + lo operands, fp32 accumulation); in fp32 on the CUDA cores otherwise. Asynchronous on `stream`; allocates
 * nothing. Errors: DPLR_ERR_INVALID_ARG for another
 * mode or a null / misaligned pointer, DPLR_ERR_UNSUPPORTED for another L or dk, dv > 128, DPLR_ERR_WORKSPACE,
 * DPLR_ERR_CUDA. */
DPLR_API size_t dplr_hla_workspace_size(const dplr_desc* desc, int L);
DPLR_API dplr_status dplr_hla_forward(const dplr_desc* desc, const void* q, const void* k, const void* v,
                             const float* g, const float* beta, const float* W, float theta, int L,
                             float* o, void* workspace, size_t ws_bytes, void* stream);

/* The kernel path dplr_hla_forward takes for `desc` and `L`: "hla_gated_tcgen05" (the gated composition on
 * the tensor cores, dk = dv = 128 and at most 256 chunks of L tokens), "hla_gated_fp32" (on the CUDA cores),
 * or "" if the arguments are invalid. */
DPLR_API const char* dplr_hla_path(const dplr_desc* desc, int L);

/* Gated DeltaProduct-style stacked Householders (HDLA page: research background and the computation table,
 * GDP with n_h = r_ab = r_kv): per token the gate once, then n_h delta-rule steps with their own key, value and
 * beta, S <- e^{g_t} S; S <- (I - b_h k_h k_h^T) S + b_h k_h v_h^T (h = 1 .. n_h); o_t = S^T q_t. `desc`: mode
 * DPLR_GENERIC with r_ab = r_kv = n_h (1 .. 8), dk in {32, 64, 128}. Layouts: q [B,H,T,dk]; k [B,H,T,n_h,dk];
 * v [B,H,T,n_h,dv] (in_dtype); g [B,H,T] and beta [B,H,T,n_h] fp32; S0 (nullable), S_T (nullable), o as for
 * dplr_la_forward. The token's exact rank-n_h factors are built in fp32, then the generic-mode forward runs
 * (dplr_gdp_path names its kernels). Workspace: dplr_gdp_workspace_size(desc) bytes, 256-byte aligned.
 * Asynchronous on `stream`; allocates nothing. Errors as dplr_la_forward; DPLR_ERR_INVALID_ARG for another mode
 * or r_ab != r_kv. */
DPLR_API size_t dplr_gdp_workspace_size(const dplr_desc* desc);
DPLR_API dplr_status dplr_gdp_forward(const dplr_desc* desc, const void* q, const void* k, const void* v,
                             const float* g, const float* beta, const float* S0, float* o, float* S_T,
                             void* workspace, size_t ws_bytes, void* stream);
DPLR_API const char* dplr_gdp_path(const dplr_desc* desc);

/* Name of the kernel path that dplr_la_forward runs for `desc` (no counterpart in the
 * paper; static storage): "gdn_fused_tcgen05" (GDN, bf16, dk = dv = 128: one fused
 * per-head kernel on the tensor cores), "hdla_tcgen05" (HDLA, bf16, dk = dv = 128: the
 * chunk-map and chain kernels on the tensor cores), "generic_tcgen05" (generic mode,
 * dk = dv = 64, r_ab <= 4, r_kv <= 2: the generic chunk and chain kernels on the tensor
 * cores), "two_stage_fp32" (every other case: the chunk-map and state-scan kernels in fp32
 * on the CUDA cores), or "" if `desc` is invalid or unsupported. */
DPLR_API const char* dplr_la_path(const dplr_desc* desc);

/* Human-readable name of a status code (static storage). */
DPLR_API const char* dplr_status_string(dplr_status status);

/* Number of CUDA kernels one dplr_la_forward launches for `desc` (0 if the
 * descriptor is invalid): 1 for the fused per-head kernel, else 2 (one per
 * stage). dplr_la_chunk_maps and dplr_la_state_scan each launch one. */
DPLR_API int dplr_la_kernel_count(const dplr_desc* desc);

/* The whole forward without a workspace argument (no counterpart in the paper:
 * an addition for callers that cannot allocate device memory at call time, such
 * as an inference engine that reserved the device up front or a plugin whose
 * host framework owns the allocator). Scratch comes from a 64 MiB array compiled
 * into the library; descriptors whose dplr_la_workspace_size exceeds 64 MiB return
 * DPLR_ERR_UNSUPPORTED before anything is launched. Allocates nothing. Runs on the
 * current device (make the stream's device current).
 * Memory: the array is part of the library's device code. Under CUDA's default
 * lazy module loading a device reserves it when the first call on that device
 * looks up its address; from then on the device holds it until the process exits.
 * Make that first call (or a warm-up call) before reserving the rest of the
 * device's memory, and before any stream capture. A device reset (for instance
 * cudaDeviceReset) invalidates the looked-up address: do not call this entry point
 * on a device after resetting it.
 * Sharing: every call shares the array, so calls whose GPU work overlaps race and
 * must be serialised. Each call first zeroes the array's status word on `stream`;
 * dplr_la_noalloc_status reads it after the call. Other arguments and errors as
 * for dplr_la_forward. */
DPLR_API dplr_status dplr_la_forward_noalloc(const dplr_desc* desc,
                                    const void* q, const void* k, const void* v,
                                    const float* decay, const float* beta,
                                    const void* A, const void* Bm, const void* K, const void* V,
                                    const float* S0, float* o, float* S_T, void* stream);

/* Synchronous status check for dplr_la_forward_noalloc (no counterpart in the paper):
 * waits for the work queued on `stream`, then copies the status word of the
 * library's scratch array on the current device into *status (DPLR_OK, or the code
 * a kernel of the last call left there, such as DPLR_ERR_TIMEOUT). Allocates
 * nothing. DPLR_ERR_INVALID_ARG for a null `status`; DPLR_ERR_CUDA if a CUDA call
 * fails or no dplr_la_forward_noalloc call has run on the current device yet. */
DPLR_API dplr_status dplr_la_noalloc_status(int* status, void* stream);

/* Bytes of device staging area dplr_la_forward_host needs for `desc` split into
 * `groups` groups of heads with `slots` staging slots (1 <= slots <= 8); 0 if the
 * descriptor is invalid, B*H is not a multiple of `groups` or `slots` is out of range. */
DPLR_API size_t dplr_la_host_workspace_size(const dplr_desc* desc, int groups, int slots);

/* The whole forward with HOST inputs and outputs (no counterpart in the paper: the
 * transfers a caller would otherwise make around dplr_la_forward, overlapped with it).
 * q .. S0 are host pointers in the layouts above (S0 may be NULL), o and S_T host
 * outputs (S_T may be NULL); pinned host memory gives full transfer bandwidth, other host
 * memory works but the copies then do not overlap. The B*H heads are split into `groups`
 * equal groups (B*H must be a multiple of it); each group is copied into one of `slots`
 * staging slots in `staging` (device memory, 256-byte aligned, at least
 * dplr_la_host_workspace_size bytes, owned by the caller), computed there with
 * dplr_la_forward, and copied back, so copies in, forwards and copies out of different
 * groups overlap. The work starts after the work already queued on `stream` and `stream`
 * waits for all of it (synchronise `stream` before reading o and S_T); the host buffers
 * must stay valid until then. The library keeps, per device, two copy streams, 8 compute
 * streams and their events, created on the first call made while that device is current;
 * calls on one device run in call order when they are made on one stream; calls on
 * different streams that share a staging area must be serialised by the caller (wait for
 * the earlier call's stream before making the next call). Allocates no device memory. Errors: as
 * dplr_la_forward, plus DPLR_ERR_INVALID_ARG for a bad group or slot count and
 * DPLR_ERR_WORKSPACE for a missing, misaligned or small staging area; a CUDA error after
 * some groups were queued returns DPLR_ERR_CUDA, and the groups already queued may still be
 * running: synchronise the device before freeing `staging` or the host buffers. A
 * device-side timeout (DPLR_ERR_TIMEOUT in dplr_la_forward) is written to the status word of
 * the group's staging slot, which the next group in that slot clears; callers that need to
 * read it use dplr_la_forward. */
DPLR_API dplr_status dplr_la_forward_host(const dplr_desc* desc,
                                 const void* q, const void* k, const void* v,
                                 const float* decay, const float* beta,
                                 const void* A, const void* Bm, const void* K, const void* V,
                                 const float* S0, float* o, float* S_T,
                                 void* staging, size_t staging_bytes, int groups, int slots,
                                 void* stream);

/* Bytes of device staging area dplr_la_forward_host_seq needs for `desc` split into
 * `segments` sequence segments with `slots` staging slots (1 <= slots <= 8); 0 if the
 * descriptor or the counts are invalid. */
DPLR_API size_t dplr_la_host_seq_workspace_size(const dplr_desc* desc, int segments, int slots);

/* The whole forward with HOST inputs and outputs, as dplr_la_forward_host, but split along the
 * sequence instead of over the heads (no counterpart in the paper; the state carry it relies on
 * is the chunkwise recurrence's own, "Householder-Diagonalized Linear Attention", Key design 3).
 * Segment g holds tokens [g Ts, (g + 1) Ts) of every head, with Ts = `segments`-th of T rounded up
 * to a multiple of the 64-token chunk (so there are ceil(T / Ts) <= `segments` of them). Each
 * segment's inputs are copied into one of `slots` staging slots by one 2-D copy per tensor (a row
 * per head); its dplr_la_forward starts from the state the previous segment's forward left on the
 * device (S0 for the first) and its outputs are copied back the same way; the final state goes to
 * S_T. Segments are computed one after another (the state carries), each a short forward, while
 * the copies of the others run; the result equals dplr_la_forward's up to the rounding of the
 * chunk maps of the two-stage paths (the fused path gives the same bits). Pointers, staging
 * (256-byte aligned, at least dplr_la_host_seq_workspace_size bytes), streams, ordering and
 * errors as dplr_la_forward_host, with `segments` (>= 1) in place of `groups`. */
DPLR_API dplr_status dplr_la_forward_host_seq(const dplr_desc* desc,
                                 const void* q, const void* k, const void* v,
                                 const float* decay, const float* beta,
                                 const void* A, const void* Bm, const void* K, const void* V,
                                 const float* S0, float* o, float* S_T,
                                 void* staging, size_t staging_bytes, int segments, int slots,
                                 void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DPLR_H */
