// Work lists, merge segments and row segments reach the workspace as kernel
// parameters: each launch of upload_kernel carries up to kUploadBytes of them
// by value and writes them to device memory. Launch parameters are copied when
// the launch is enqueued, so the host arrays may be released as soon as the
// call returns, and no copy from pageable host memory waits in a stream behind
// the kernels before it (such copies also held up unrelated copies that other
// streams had queued at the same time).
#include <algorithm>
#include <cstring>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr uint32_t kUploadBytes = 31744;   // under the 32 KB limit of a launch's parameters, a multiple of 16

struct UploadBlock {
    uint4 v[kUploadBytes / 16];
};

// Each thread copies 16-byte words of the parameter block to dst (16-byte aligned).
__global__ void __launch_bounds__(256) upload_kernel(uint4* dst, const __grid_constant__ UploadBlock blk,
                                                     uint32_t words) {
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < words; i += gridDim.x * blockDim.x)
        dst[i] = blk.v[i];
}

}  // namespace

cudaError_t launch_upload(void* dst, const void* src, size_t bytes, cudaStream_t s) {
    if ((reinterpret_cast<uintptr_t>(dst) & 15u) != 0) return cudaErrorInvalidValue;
    UploadBlock blk;
    const uint8_t* p = static_cast<const uint8_t*>(src);
    uint8_t* d = static_cast<uint8_t*>(dst);
    for (size_t off = 0; off < bytes; off += kUploadBytes) {
        const size_t n = std::min<size_t>(kUploadBytes, bytes - off);
        std::memcpy(&blk, p + off, n);
        if (n % 16) std::memset(reinterpret_cast<uint8_t*>(&blk) + n, 0, 16 - n % 16);
        const uint32_t words = (uint32_t)((n + 15) / 16);
        upload_kernel<<<std::max<uint32_t>(1, (words + 255) / 256), 256, 0, s>>>(reinterpret_cast<uint4*>(d + off),
                                                                                   blk, words);
        const cudaError_t e = counted(cudaGetLastError());
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace attn
