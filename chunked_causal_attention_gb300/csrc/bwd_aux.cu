// Row-wise kernels around the backward key-tile kernel (HBM-bound).
//   prep: D_t = sum_d dO_td * O_td in fp32 (the row term of dS = P o (dP - D)),
//         and zeroing of the fp32 dQ accumulator.
//   dq:   dQ = bf16(fp32 accumulator), written with the caller's strides.
// Two rows per warp (batch*head, workspace row); the rows are the tokens of one or
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

// Rows per 256-thread block of the row kernels: each warp takes two rows, one
// per 16-lane half, and lane l of a half takes the eight elements from d = 8l
// (and from d = 8l + 128 for D above 128; D is a multiple of 8, at most 256).
constexpr int kRowsPerBlock = 16;

// (batch*head, workspace row) of row index w < B*H*rows, in 32-bit arithmetic
// when the count fits.
__device__ __forceinline__ void split_row(int64_t w, int64_t total, int32_t rows, int& bh, int& r) {
    if (total <= INT32_MAX) {
        bh = (int)((uint32_t)w / (uint32_t)rows);
        r = (int)((uint32_t)w - (uint32_t)bh * (uint32_t)rows);
    } else {
        bh = (int)(w / rows);
        r = (int)(w % rows);
    }
}

// delta = dO . O per (batch*head, token), and the dQ accumulator row zeroed.
__global__ void __launch_bounds__(256) prep_kernel(PrepArgs a) {
    const int lane = threadIdx.x & 31, sub = lane & 15;
    const int64_t w = ((int64_t)blockIdx.x * 8 + (threadIdx.x >> 5)) * 2 + (lane >> 4);
    const int64_t total = (int64_t)a.g.B * a.g.H * a.rows;
    const int D = a.g.D;
    bool ok = w < total;                        // the same in the 16 lanes of a row
    float acc = 0.f;
    if (ok) {
        int bh, r;
        split_row(w, total, a.rows, bh, r);
        const int t = token_of_row(a.segs, a.n_segs, r);
        if (t < 0 || t >= a.g.T) {             // a row segment outside the tokens
            if (sub == 0) set_error(a.status, ATTN_E_BOUNDS);
            ok = false;
        } else {
            const int b = bh / a.g.H, h = bh % a.g.H;
            const int64_t off = (int64_t)b * a.g.sb + (int64_t)h * a.g.sh + (int64_t)t * a.g.st;
            const __nv_bfloat16* o = reinterpret_cast<const __nv_bfloat16*>(a.o) + off;
            const __nv_bfloat16* g = reinterpret_cast<const __nv_bfloat16*>(a.dout) + off;
#pragma unroll
            for (int d = 8 * sub; d < 256; d += 128) {
                if (d < D) {
                    const uint4 xo = *reinterpret_cast<const uint4*>(o + d);
                    const uint4 xd = *reinterpret_cast<const uint4*>(g + d);
                    const uint32_t ow[4] = {xo.x, xo.y, xo.z, xo.w}, gw[4] = {xd.x, xd.y, xd.z, xd.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float2 ov = bf16x2_to_float2(ow[u]), gv = bf16x2_to_float2(gw[u]);
                        acc = fmaf(ov.x, gv.x, fmaf(ov.y, gv.y, acc));
                    }
                    float4* z = reinterpret_cast<float4*>(a.dq_acc + w * D + d);
                    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
                    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
        }
    }
    // sum over the 16 lanes of the row (the shuffles stay inside each half)
#pragma unroll
    for (int m = 8; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    if (ok && sub == 0) a.delta[w] = acc;
}

// dq = bf16(accumulator) per (batch*head, token), written with the caller's strides.
__global__ void __launch_bounds__(256) dq_kernel(DqArgs a) {
    const int lane = threadIdx.x & 31, sub = lane & 15;
    const int64_t w = ((int64_t)blockIdx.x * 8 + (threadIdx.x >> 5)) * 2 + (lane >> 4);
    const int64_t total = (int64_t)a.g.B * a.g.H * a.rows;
    if (w >= total) return;                     // no shuffles follow
    const int D = a.g.D;
    int bh, r;
    split_row(w, total, a.rows, bh, r);
    const int t = token_of_row(a.segs, a.n_segs, r);
    if (t < 0 || t >= a.g.T) {                 // a row segment outside the tokens
        if (sub == 0) set_error(a.status, ATTN_E_BOUNDS);
        return;
    }
    const int b = bh / a.g.H, h = bh % a.g.H;
    __nv_bfloat16* row = reinterpret_cast<__nv_bfloat16*>(a.dq) + (int64_t)b * a.g.sb + (int64_t)h * a.g.sh +
                         (int64_t)t * a.g.st;
#pragma unroll
    for (int d = 8 * sub; d < 256; d += 128) {
        if (d < D) {
            const float4* src = reinterpret_cast<const float4*>(a.dq_acc + w * D + d);
            const float4 v0 = src[0], v1 = src[1];
            *reinterpret_cast<uint4*>(row + d) = make_uint4(pack_bf16(v0.x, v0.y), pack_bf16(v0.z, v0.w),
                                                            pack_bf16(v1.x, v1.y), pack_bf16(v1.z, v1.w));
        }
    }
}

}  // namespace

cudaError_t launch_bwd_prep(const PrepArgs& a, cudaStream_t s) {
    const int64_t blocks = ((int64_t)a.g.B * a.g.H * a.rows + kRowsPerBlock - 1) / kRowsPerBlock;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > INT32_MAX) return cudaErrorInvalidValue;
    prep_kernel<<<(unsigned)blocks, 256, 0, s>>>(a);
    return counted(cudaGetLastError());
}

cudaError_t launch_bwd_dq(const DqArgs& a, cudaStream_t s) {
    const int64_t blocks = ((int64_t)a.g.B * a.g.H * a.rows + kRowsPerBlock - 1) / kRowsPerBlock;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > INT32_MAX) return cudaErrorInvalidValue;
    dq_kernel<<<(unsigned)blocks, 256, 0, s>>>(a);
    return counted(cudaGetLastError());
}

}  // namespace attn
