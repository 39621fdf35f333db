// Row-wise kernels around the backward key-tile kernel (HBM-bound).
//   prep: D_t = sum_d dO_td * O_td in fp32 (the row term of dS = P o (dP - D)),
//         and zeroing of the fp32 dQ accumulator.
//   dq:   dQ = bf16(fp32 accumulator), written with the caller's strides.
// One warp per (batch*head, workspace row); the rows are the tokens of one or
// more segments (all tokens for the whole backward, the chunks' rows for the
// chunk-streamed backward). A row whose segment maps it outside the tokens is
// reported as ATTN_E_BOUNDS and not touched.
#include "device_common.cuh"

namespace attn {
namespace {

// Two bf16 (low half first) to floats: a bf16 is the upper 16 bits of its float.
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t x) {
    return make_float2(__uint_as_float(x << 16), __uint_as_float(x & 0xffff0000u));
}

// Token of workspace row r: the segment with the largest ws_row0 <= r.
__device__ __forceinline__ int token_of_row(const RowSeg* segs, int n, int r) {
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (segs[mid].ws_row0 <= r) lo = mid; else hi = mid - 1;
    }
    return segs[lo].t0 + (r - segs[lo].ws_row0);
}

// One warp per (batch*head, token): delta = dO . O; zero the dQ accumulator row.
// Lane l takes the four elements from d = 4l and, for D above 128, those from
// d = 4l + 128 (D is a multiple of 8, at most 256).
__global__ void __launch_bounds__(256) prep_kernel(PrepArgs a) {
    const int64_t w = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int64_t total = (int64_t)a.g.B * a.g.H * a.rows;
    if (w >= total) return;
    const int D = a.g.D;
    const int bh = (int)(w / a.rows), t = token_of_row(a.segs, a.n_segs, (int)(w % a.rows));
    if (t < 0 || t >= a.g.T) {                 // a row segment outside the tokens
        if (lane == 0) set_error(a.status, ATTN_E_BOUNDS);
        return;
    }
    const int b = bh / a.g.H, h = bh % a.g.H;
    const int64_t off = (int64_t)b * a.g.sb + (int64_t)h * a.g.sh + (int64_t)t * a.g.st;
    float acc = 0.f;
#pragma unroll
    for (int d = 4 * lane; d < 256; d += 128) {
        if (d < D) {
            const uint2 xo = *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(a.o) + off + d);
            const uint2 xd =
                *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(a.dout) + off + d);
            const float2 o0 = bf16x2_to_float2(xo.x), o1 = bf16x2_to_float2(xo.y);
            const float2 g0 = bf16x2_to_float2(xd.x), g1 = bf16x2_to_float2(xd.y);
            acc += fmaf(o0.x, g0.x, fmaf(o0.y, g0.y, fmaf(o1.x, g1.x, o1.y * g1.y)));
            *reinterpret_cast<float4*>(a.dq_acc + w * D + d) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    if (lane == 0) a.delta[w] = acc;
}

// One warp per (batch*head, token): dq = bf16(accumulator); lane l takes the
// four elements from d = 4l (and from d = 4l + 128 for D above 128).
__global__ void __launch_bounds__(256) dq_kernel(DqArgs a) {
    const int64_t w = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int64_t total = (int64_t)a.g.B * a.g.H * a.rows;
    if (w >= total) return;
    const int D = a.g.D;
    const int bh = (int)(w / a.rows), t = token_of_row(a.segs, a.n_segs, (int)(w % a.rows));
    if (t < 0 || t >= a.g.T) {                 // a row segment outside the tokens
        if (lane == 0) set_error(a.status, ATTN_E_BOUNDS);
        return;
    }
    const int b = bh / a.g.H, h = bh % a.g.H;
    __nv_bfloat16* row = reinterpret_cast<__nv_bfloat16*>(a.dq) + (int64_t)b * a.g.sb + (int64_t)h * a.g.sh +
                         (int64_t)t * a.g.st;
#pragma unroll
    for (int d = 4 * lane; d < 256; d += 128) {
        if (d < D) {
            const float4 v = *reinterpret_cast<const float4*>(a.dq_acc + w * D + d);
            *reinterpret_cast<uint2*>(row + d) = make_uint2(pack_bf16(v.x, v.y), pack_bf16(v.z, v.w));
        }
    }
}

}  // namespace

cudaError_t launch_bwd_prep(const PrepArgs& a, cudaStream_t s) {
    const int64_t blocks = ((int64_t)a.g.B * a.g.H * a.rows + 7) / 8;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > INT32_MAX) return cudaErrorInvalidValue;
    prep_kernel<<<(unsigned)blocks, 256, 0, s>>>(a);
    return counted(cudaGetLastError());
}

cudaError_t launch_bwd_dq(const DqArgs& a, cudaStream_t s) {
    const int64_t blocks = ((int64_t)a.g.B * a.g.H * a.rows + 7) / 8;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > INT32_MAX) return cudaErrorInvalidValue;
    dq_kernel<<<(unsigned)blocks, 256, 0, s>>>(a);
    return counted(cudaGetLastError());
}

}  // namespace attn
