// Log-sum-exp merge of the two key-range partials of re-split chunks.
//
// SPPO §4 re-splits the subsequences next to the pipeline bubbles into two
// sub-subsequences whose results are combined afterwards; the Ring
// Self-Attention accumulation O = sum_i S_i V_i over key/value blocks is made
// exact across blocks by the log-sum-exp rule:
//     LSE = ln(e^{LSE_A} + e^{LSE_B}),  O = e^{LSE_A - LSE} O_A + e^{LSE_B - LSE} O_B,
// where a part with no visible key (LSE = -inf) has weight 0.
// One warp per (segment row, batch*head); fp32 partials in, bf16 O and fp32 LSE out.
#include "device_common.cuh"

namespace attn {
namespace {

// One warp per (segment row, batch*head): merge the two partials.
template <int D>
__global__ void __launch_bounds__(256) merge_kernel(MergeArgs a) {
    constexpr int PER = D / 32;   // floats per lane
    const int64_t w = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (w >= a.total_work) return;
    int si = 0;
    while (si + 1 < a.n_segs && a.segs[si + 1].work0 <= w) ++si;
    const MergeSeg sg = a.segs[si];
    const int BH = a.g.B * a.g.H;
    const int64_t local = w - sg.work0;
    const int bh = (int)(local / sg.R);
    const int i = (int)(local % sg.R);
    const int t = sg.row0 + i;
    const int64_t R = sg.R;
    const float* A = a.ws_f + sg.off_a;
    const float* Bp = a.ws_f + sg.off_b;
    const float la = A[(int64_t)BH * R * D + (int64_t)bh * R + i];
    const float lb = Bp[(int64_t)BH * R * D + (int64_t)bh * R + i];
    const float mx = fmaxf(la, lb);
    float wa = 0.f, wb = 0.f, lse = -INFINITY;
    if (mx != -INFINITY) {
        float ea = la == -INFINITY ? 0.f : __expf(la - mx);
        float eb = lb == -INFINITY ? 0.f : __expf(lb - mx);
        float tot = ea + eb;
        lse = mx + __logf(tot);
        wa = ea / tot;
        wb = eb / tot;
    }
    const float* oa = A + ((int64_t)bh * R + i) * D + lane * PER;
    const float* ob = Bp + ((int64_t)bh * R + i) * D + lane * PER;
    float r[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) r[e] = wa * oa[e] + wb * ob[e];
    const int b = bh / a.g.H, h = bh % a.g.H;
    __nv_bfloat16* O = reinterpret_cast<__nv_bfloat16*>(a.o) + (int64_t)b * a.g.sb + (int64_t)h * a.g.sh +
                       (int64_t)t * a.g.st + lane * PER;
#pragma unroll
    for (int e = 0; e < PER; e += 2) *reinterpret_cast<uint32_t*>(O + e) = pack_bf16(r[e], r[e + 1]);
    if (lane == 0) a.lse[(int64_t)bh * a.g.T + t] = lse;
}

}  // namespace

cudaError_t launch_fwd_merge(const MergeArgs& a, cudaStream_t s) {
    if (a.total_work <= 0) return cudaSuccess;
    const int64_t blocks = (a.total_work + 7) / 8;
    if (blocks > INT32_MAX) return cudaErrorInvalidValue;
    if (a.g.D == 128)
        merge_kernel<128><<<(unsigned)blocks, 256, 0, s>>>(a);
    else
        merge_kernel<64><<<(unsigned)blocks, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace attn
