// Log-sum-exp merge of the key-range partials of re-split chunks.
//
// SPPO §4 re-splits the subsequences next to the pipeline bubbles into
// sub-subsequences whose results are combined afterwards (Table 3: as many as
// there are idle devices); the Ring Self-Attention accumulation
// O = sum_i S_i V_i over key/value blocks is made exact across blocks by the
// log-sum-exp rule:
//     LSE = ln sum_p e^{LSE_p},  O = sum_p e^{LSE_p - LSE} O_p,
// where a part with no visible key (LSE = -inf, or a part that starts after
// the row) has weight 0.
// One warp per (segment row, batch*head); fp32 partials in, bf16 O and fp32 LSE out.
#include "device_common.cuh"

namespace attn {
namespace {

// One warp per (segment row, batch*head): merge the row's partials. Lane l
// takes the four elements from d = 4l (D is a multiple of 8, at most 128).
__global__ void __launch_bounds__(256) merge_kernel(MergeArgs a) {
    const int64_t w = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (w >= a.total_work) return;
    const int D = a.g.D;
    int si = 0;
    while (si + 1 < a.n_segs && a.segs[si + 1].work0 <= w) ++si;
    const MergeSeg sg = a.segs[si];
    const int BH = a.g.B * a.g.H;
    const int64_t local = w - sg.work0;
    const int bh = (int)(local / sg.R);
    const int i = (int)(local % sg.R);
    const int t = sg.row0 + i;
    const int64_t R = sg.R;
    const int32_t* kb = a.kbounds + sg.kb;
    // parts whose key range starts at or before this row
    int np = 0;
    while (np < sg.P && kb[np] <= t) ++np;
    float mx = -INFINITY;
    for (int p = 0; p < np; ++p) mx = fmaxf(mx, a.ws_f[sg.off0 + p * sg.blk + (int64_t)BH * R * D + (int64_t)bh * R + i]);
    const int d = 4 * lane;
    float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
    float lse = -INFINITY;
    if (mx != -INFINITY) {
        float tot = 0.f;
        for (int p = 0; p < np; ++p) {
            const float* base = a.ws_f + sg.off0 + p * sg.blk;
            const float lp = base[(int64_t)BH * R * D + (int64_t)bh * R + i];
            if (lp == -INFINITY) continue;
            const float ep = __expf(lp - mx);
            tot += ep;
            if (d < D) {
                const float4 v = *reinterpret_cast<const float4*>(base + ((int64_t)bh * R + i) * D + d);
                r.x = fmaf(ep, v.x, r.x);
                r.y = fmaf(ep, v.y, r.y);
                r.z = fmaf(ep, v.z, r.z);
                r.w = fmaf(ep, v.w, r.w);
            }
        }
        lse = mx + __logf(tot);
        const float inv = 1.f / tot;
        r.x *= inv;
        r.y *= inv;
        r.z *= inv;
        r.w *= inv;
    }
    const int b = bh / a.g.H, h = bh % a.g.H;
    __nv_bfloat16* O = reinterpret_cast<__nv_bfloat16*>(a.o) + (int64_t)b * a.g.sb + (int64_t)h * a.g.sh +
                       (int64_t)t * a.g.st;
    if (d < D) *reinterpret_cast<uint2*>(O + d) = make_uint2(pack_bf16(r.x, r.y), pack_bf16(r.z, r.w));
    if (lane == 0) a.lse[(int64_t)bh * a.g.T + t] = lse;
}

}  // namespace

cudaError_t launch_fwd_merge(const MergeArgs& a, cudaStream_t s) {
    if (a.total_work <= 0) return cudaSuccess;
    const int64_t blocks = (a.total_work + 7) / 8;
    if (blocks > INT32_MAX) return cudaErrorInvalidValue;
    merge_kernel<<<(unsigned)blocks, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace attn
