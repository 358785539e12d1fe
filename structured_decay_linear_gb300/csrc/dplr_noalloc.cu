// dplr_la_forward_noalloc: the whole forward without a caller-provided workspace.
//
// Some callers cannot allocate device memory when they call the forward: an
// inference engine that reserved the whole device up front and forbids later
// cudaMalloc calls, or a plugin running inside a host framework that owns the
// device allocator and hands it only the inputs and outputs. For them this entry
// point takes its scratch (the per-chunk maps written by stage 1 and read by
// stage 2) from a fixed array compiled into the library instead of a workspace
// argument. Nothing here calls cudaMalloc, cudaFree or any allocating routine.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds kNoallocScratchBytes of device memory until the process exits.
// Host code cannot use the array's name as a device pointer (on the host it is a
// stand-in symbol); its device address is looked up with cudaGetSymbolAddress
// once per device, with that device current, on the first call made while the
// device is current. Make that first call before any stream capture. The library
// is built without relocatable device code, so this file is a module of its own:
// under CUDA's lazy module loading the array is reserved on a device only when that
// first lookup loads the module. Callers that reserve a device's memory up front
// therefore make one call (or a warm-up call) first. The address stays valid until
// the device is reset; a reset (cudaDeviceReset) reloads the module elsewhere, and
// this entry point must not be used on that device afterwards.
//
// Every call shares the one array and the array keeps the previous call's
// contents. Its first 256 bytes are the device status word, which each call zeroes
// on its stream before launching (a kernel sets it when a bounded wait gives up);
// dplr_la_noalloc_status reads it. Nothing else needs zeroing: the kernels write
// every map before they read it. Calls whose work overlaps on the GPU (two streams,
// or two threads on one device) race on the array; serialise them.
#include <mutex>

#include "dplr_internal.h"

namespace dplr {
namespace {

constexpr size_t kNoallocScratchBytes = size_t(64) << 20;   // 64 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
cudaError_t scratch_address(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace dplr

extern "C" dplr_status dplr_la_forward_noalloc(const dplr_desc* desc, const void* q, const void* k,
                                               const void* v, const float* decay, const float* beta,
                                               const void* A, const void* Bm, const void* K, const void* V,
                                               const float* S0, float* o, float* S_T, void* stream) {
    using namespace dplr;
    Plan pl;
    dplr_status st = make_plan(desc, &pl);
    if (st != DPLR_OK) return st;
    if (pl.ws_bytes > kNoallocScratchBytes) return DPLR_ERR_UNSUPPORTED;   // problem too large for the array
    void* ws = nullptr;
    if (scratch_address(&ws) != cudaSuccess) return DPLR_ERR_CUDA;
    // a fresh status word for this call (a memset allocates nothing)
    if (cudaMemsetAsync(ws, 0, 256, static_cast<cudaStream_t>(stream)) != cudaSuccess) return DPLR_ERR_CUDA;
    return dplr_la_forward(desc, q, k, v, decay, beta, A, Bm, K, V, S0, o, S_T, ws, kNoallocScratchBytes, stream);
}

extern "C" dplr_status dplr_la_noalloc_status(int* status, void* stream) {
    using namespace dplr;
    if (status == nullptr) return DPLR_ERR_INVALID_ARG;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DPLR_ERR_CUDA;
    void* ws = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        ws = g_scratch_addr[dev];
    }
    if (ws == nullptr) return DPLR_ERR_CUDA;   // no call has looked the array up on this device
    return dplr_la_read_status(ws, kNoallocScratchBytes, 0, status, stream);
}
