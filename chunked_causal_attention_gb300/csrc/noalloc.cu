// Forward entry point for callers that cannot allocate device memory.
//
// Some callers have no way to obtain a device buffer for the workspace: code
// running inside a runtime that owns all device memory and exposes no
// allocator, callers that must not allocate after start-up, or plain C hosts
// without access to the caching allocator of a framework. attn_fwd_noalloc
// serves them with a scratch area that lives inside this library: a
// file-scope __device__ array of ATTN_NOALLOC_SCRATCH_BYTES, which every GPU
// that loads the library holds until the process exits. The caller still
// passes the inputs and outputs.
//
// In host code the array's name is only a host-side stand-in, so its device
// address is looked up with cudaGetSymbolAddress, once per device, with that
// device current, the first time the entry point runs there; that first call
// should therefore come before any stream capture. All calls share the one
// array and it keeps whatever the last call left in it: the forward clears its
// status header and rewrites its work list and partials on every call, and
// calls whose work overlaps on the GPU (different streams, or threads racing
// on the same device) race on the array.
#include <mutex>

#include "attn_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_scratch[ATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_dev[kMaxDevices] = {};

// Device address of g_scratch on the current device (looked up once per device).
int scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_E_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return ATTN_E_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_dev[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return ATTN_E_CUDA;
        g_scratch_dev[dev] = p;
    }
    *out = g_scratch_dev[dev];
    return ATTN_OK;
}

}  // namespace

extern "C" int attn_fwd_noalloc(const void* q, const void* k, const void* v, const attn_chunk* chunks, int32_t n,
                                const attn_shape* shape, void* o, float* lse, void* stream) {
    size_t need = 0;
    int st = attn_workspace_size(shape, chunks, n, 0, &need);
    if (st) return st;
    if (need > (size_t)ATTN_NOALLOC_SCRATCH_BYTES) return ATTN_E_WORKSPACE;
    void* ws = nullptr;
    if ((st = scratch_address(&ws))) return st;
    return attn_fwd(q, k, v, chunks, n, shape, o, lse, ws, (size_t)ATTN_NOALLOC_SCRATCH_BYTES, stream);
}
