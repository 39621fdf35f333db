// Row-wise kernels around the backward key-tile kernel (HBM-bound).
//   prep: D_t = sum_d dO_td * O_td in fp32 (the row term of dS = P o (dP - D)),
//         and zeroing of the fp32 dQ accumulator.
//   dq:   dQ = bf16(fp32 accumulator), written with the caller's strides.
// One warp per (batch*head, workspace row); the rows are the tokens of one or
// more segments (all tokens for the whole backward, the chunks' rows for the
// chunk-streamed backward).
#include "device_common.cuh"

namespace attn {
namespace {

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
template <int D>
__global__ void __launch_bounds__(256) prep_kernel(PrepArgs a) {
    constexpr int PER = D / 32;
    const int64_t w = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int64_t total = (int64_t)a.g.B * a.g.H * a.rows;
    if (w >= total) return;
    const int bh = (int)(w / a.rows), t = token_of_row(a.segs, a.n_segs, (int)(w % a.rows));
    const int b = bh / a.g.H, h = bh % a.g.H;
    const int64_t off = (int64_t)b * a.g.sb + (int64_t)h * a.g.sh + (int64_t)t * a.g.st + lane * PER;
    const __nv_bfloat16* O = reinterpret_cast<const __nv_bfloat16*>(a.o) + off;
    const __nv_bfloat16* dO = reinterpret_cast<const __nv_bfloat16*>(a.dout) + off;
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < PER; e += 2) {
        __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(O + e);
        __nv_bfloat162 y = *reinterpret_cast<const __nv_bfloat162*>(dO + e);
        float2 fx = __bfloat1622float2(x), fy = __bfloat1622float2(y);
        acc = fmaf(fx.x, fy.x, acc);
        acc = fmaf(fx.y, fy.y, acc);
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    if (lane == 0) a.delta[w] = acc;
    float* q = a.dq_acc + w * D + lane * PER;
#pragma unroll
    for (int e = 0; e < PER; ++e) q[e] = 0.f;
}

// One warp per (batch*head, token): dq = bf16(accumulator).
template <int D>
__global__ void __launch_bounds__(256) dq_kernel(DqArgs a) {
    constexpr int PER = D / 32;
    const int64_t w = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int64_t total = (int64_t)a.g.B * a.g.H * a.rows;
    if (w >= total) return;
    const int bh = (int)(w / a.rows), t = token_of_row(a.segs, a.n_segs, (int)(w % a.rows));
    const int b = bh / a.g.H, h = bh % a.g.H;
    const float* src = a.dq_acc + w * D + lane * PER;
    __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(a.dq) + (int64_t)b * a.g.sb + (int64_t)h * a.g.sh +
                         (int64_t)t * a.g.st + lane * PER;
#pragma unroll
    for (int e = 0; e < PER; e += 2) *reinterpret_cast<uint32_t*>(dst + e) = pack_bf16(src[e], src[e + 1]);
}

}  // namespace

cudaError_t launch_bwd_prep(const PrepArgs& a, cudaStream_t s) {
    const int64_t blocks = ((int64_t)a.g.B * a.g.H * a.rows + 7) / 8;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > INT32_MAX) return cudaErrorInvalidValue;
    if (a.g.D == 128)
        prep_kernel<128><<<(unsigned)blocks, 256, 0, s>>>(a);
    else
        prep_kernel<64><<<(unsigned)blocks, 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_bwd_dq(const DqArgs& a, cudaStream_t s) {
    const int64_t blocks = ((int64_t)a.g.B * a.g.H * a.rows + 7) / 8;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > INT32_MAX) return cudaErrorInvalidValue;
    if (a.g.D == 128)
        dq_kernel<128><<<(unsigned)blocks, 256, 0, s>>>(a);
    else
        dq_kernel<64><<<(unsigned)blocks, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace attn
