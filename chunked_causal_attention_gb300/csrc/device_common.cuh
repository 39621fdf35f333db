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

// Index checks of the work descriptors a kernel reads from the workspace,
// made before any address is formed from them. The host lays the
// descriptors out from a validated chunk table, so a failure means the
// workspace was overwritten between the call's copy and the kernel, or a
// layout bug: the kernel records ATTN_E_BOUNDS and does not touch memory for
// that descriptor.
//
// Forward item: at most 128 query rows inside [0, T); keys [kv_lo, kv_hi)
// with kv_hi <= r1 (no key after the last row); a partial block (part_off >= 0)
// holds the rows and lies inside the partial region of part_floats floats
// (BH*R rows of Dv floats, then BH*R LSEs).
__device__ __forceinline__ bool fwd_item_ok(const FwdItem& it, int32_t T, int64_t BH, int32_t Dv,
                                            int64_t part_floats) {
    if (!(0 <= it.r0 && it.r0 < it.r1 && it.r1 - it.r0 <= 128 && it.r1 <= T)) return false;
    if (!(0 <= it.kv_lo && it.kv_lo < it.kv_hi && it.kv_hi <= it.r1)) return false;
    if (it.part_off < 0) return true;
    return it.part_R > 0 && it.part_row0 <= it.r0 && (int64_t)it.r1 <= (int64_t)it.part_row0 + it.part_R &&
           it.part_off + BH * it.part_R * (Dv + 1) <= part_floats;
}

// Backward item: keys [j0, j1), at most 128, inside [0, T); queries
// [q_lo, q_end) with j0 <= q_lo < q_end <= T and j1 <= q_end; their workspace
// rows q + row_off inside [0, rows).
__device__ __forceinline__ bool bwd_item_ok(const BwdItem& it, int32_t T, int32_t rows) {
    return 0 <= it.j0 && it.j0 < it.j1 && it.j1 - it.j0 <= 128 && it.j1 <= it.q_end && it.j0 <= it.q_lo &&
           it.q_lo < it.q_end && it.q_end <= T && (int64_t)it.q_lo + it.row_off >= 0 &&
           (int64_t)it.q_end + it.row_off <= rows;
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
