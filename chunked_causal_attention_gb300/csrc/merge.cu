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

// One warp per (segment row, batch*head): merge the row's partials.
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
    const int32_t* kb = a.kbounds + sg.kb;
    // parts whose key range starts at or before this row
    int np = 0;
    while (np < sg.P && kb[np] <= t) ++np;
    float mx = -INFINITY;
    for (int p = 0; p < np; ++p) mx = fmaxf(mx, a.ws_f[sg.off0 + p * sg.blk + (int64_t)BH * R * D + (int64_t)bh * R + i]);
    float r[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) r[e] = 0.f;
    float lse = -INFINITY;
    if (mx != -INFINITY) {
        float tot = 0.f;
        for (int p = 0; p < np; ++p) {
            const float* base = a.ws_f + sg.off0 + p * sg.blk;
            const float lp = base[(int64_t)BH * R * D + (int64_t)bh * R + i];
            if (lp == -INFINITY) continue;
            const float ep = __expf(lp - mx);
            tot += ep;
            const float* op = base + ((int64_t)bh * R + i) * D + lane * PER;
#pragma unroll
            for (int e = 0; e < PER; ++e) r[e] = fmaf(ep, op[e], r[e]);
        }
        lse = mx + __logf(tot);
        const float inv = 1.f / tot;
#pragma unroll
        for (int e = 0; e < PER; ++e) r[e] *= inv;
    }
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
