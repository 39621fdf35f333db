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
// address is looked up with cudaGetSymbolAddress in the context that is
// current when the call runs. The lookup is made on every call and nothing is
// cached: an address kept from an earlier call would be stale after a device
// reset or under another context of the same device. The first call in a
// context loads this library's kernels there, so make it before any stream
// capture. All calls share the one array and it keeps whatever the last call
// left in it: the forward clears its status header and rewrites its work list
// and partials on every call, and calls whose work overlaps on the GPU
// (different streams, or threads racing on the same device) race on the array.
#include "attn_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_scratch[ATTN_NOALLOC_SCRATCH_BYTES];

// Device address of g_scratch in the current context.
int scratch_address(void** out) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return ATTN_E_CUDA;
    *out = p;
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

extern "C" int attn_noalloc_status(void* stream) {
    void* ws = nullptr;
    int st = scratch_address(&ws);
    if (st) return st;
    return attn_status(ws, stream);
}
