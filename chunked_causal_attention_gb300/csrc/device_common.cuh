// Device helpers shared by the libattn kernels: bf16 packing, shared-memory
// addressing, fast exp2/log2 (the PTX ex2.approx / lg2.approx instructions),
// the error word and the work-index decoding.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "attn_internal.h"

namespace attn {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// two floats -> bf16x2 (round to nearest even); `lo` lands in the low half
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void set_error(uint32_t* status, uint32_t code) {
    if (status) atomicCAS(status, 0u, code);
}

// Decode a work index into (item, batch*head) so that consecutive work
// indices walk `group` items of one head before the next head: CTAs that run
// together then share a head's K/V in L2, and items stay in cost order.
__device__ __forceinline__ void decode_work(int64_t w, int32_t n_items, int32_t BH, int32_t group,
                                            int32_t& item, int32_t& bh) {
    int64_t per = (int64_t)group * BH;
    int64_t g = w / per;
    int64_t rem = w - g * per;
    int32_t gsize = (int32_t)min((int64_t)group, (int64_t)n_items - g * group);
    bh = (int32_t)(rem / gsize);
    item = (int32_t)(g * group + rem % gsize);
}

}  // namespace attn
