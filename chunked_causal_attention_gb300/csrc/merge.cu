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
// A segment that does not fit the geometry or the workspace is reported as
// ATTN_E_BOUNDS and not read.
#include "device_common.cuh"

namespace attn {
namespace {

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, m));
    return x;
}

__device__ __forceinline__ float4 fma4(float e, float4 v, float4 r) {
    return make_float4(fmaf(e, v.x, r.x), fmaf(e, v.y, r.y), fmaf(e, v.z, r.z), fmaf(e, v.w, r.w));
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
    return x;
}

// One warp per (segment row, batch*head): merge the row's partials. Lane l
// takes the four elements from d = 4l, and for NH = 2 (head dims above 128)
// also the four from d = 4l + 128 (D is a multiple of 8, at most 128 * NH).
// The row's loads go out in few dependent rounds: the parts it sees (a
// prefix of the segment's increasing key boundaries) are counted by one
// ballot; then lane p reads part p's LSE while every lane reads its slice of
// the first two parts' O; the weights reach all lanes by shuffles.
template <int NH>
__global__ void __launch_bounds__(256, NH == 1 ? 5 : 3) merge_kernel(MergeArgs a) {
    const int64_t w = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (w >= a.total_work) return;   // the same w for every lane of a warp
    const int D = a.g.D;
    int si = 0;
    while (si + 1 < a.n_segs && a.segs[si + 1].work0 <= w) ++si;
    const MergeSeg sg = a.segs[si];
    const int BH = a.g.B * a.g.H;
    const int64_t local = w - sg.work0;
    // index checks of the segment before any address is formed from it
    if (!(sg.R > 0 && sg.row0 >= 0 && (int64_t)sg.row0 + sg.R <= a.g.T && sg.P >= 1 && sg.P <= 64 && sg.kb >= 0 &&
          sg.kb + sg.P + 1 <= a.n_kbounds && local >= 0 && local < (int64_t)sg.R * BH && sg.off0 >= 0 &&
          sg.blk >= (int64_t)BH * sg.R * (D + 1) && sg.off0 + sg.P * sg.blk <= a.part_floats)) {
        if (lane == 0) set_error(a.status, ATTN_E_BOUNDS);
        return;
    }
    int bh, i;
    if (local <= INT32_MAX) {
        const uint32_t l = (uint32_t)local, r = (uint32_t)sg.R;
        bh = (int)(l / r);
        i = (int)(l - (uint32_t)bh * r);
    } else {
        bh = (int)(local / sg.R);
        i = (int)(local % sg.R);
    }
    const int t = sg.row0 + i;
    const int64_t R = sg.R;
    const int64_t blk = sg.blk;
    const int32_t* kb = a.kbounds + sg.kb;
    // parts whose key range starts at or before this row (at least part 0,
    // which starts at the document start). A split at one point needs no count:
    // the forward writes both partials of every row of the segment (part 1 with
    // LSE = -inf where the row sees none of its keys, which gives it weight 0).
    int np = 2;
    if (sg.P != 2) {
        np = 0;
        for (int p0 = 0; p0 < sg.P; p0 += 32) {
            const int p = p0 + lane;
            np += __popc(__ballot_sync(0xffffffffu, p < sg.P && kb[p] <= t));
        }
    }
    // part p's LSE is at lse_row[p * blk], its O row at o_row[p * blk]
    const float* lse_row = a.ws_f + sg.off0 + (int64_t)BH * R * D + (int64_t)bh * R + i;
    const float* o_row = a.ws_f + sg.off0 + ((int64_t)bh * R + i) * D;
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 v0[NH], v1[NH], r[NH];
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) {
        const int d = 4 * lane + 128 * hh;
        v0[hh] = v1[hh] = r[hh] = zero;
        if (d < D) {
            v0[hh] = *reinterpret_cast<const float4*>(o_row + d);
            if (np > 1) v1[hh] = *reinterpret_cast<const float4*>(o_row + blk + d);
        }
    }
    float tot = 0.f, mx;
    if (np <= 2) {
        // two parts at most (every split of one point): lanes 0 and 1 read the LSEs
        const float l = lane < np ? lse_row[lane * blk] : -INFINITY;
        const float l0 = __shfl_sync(0xffffffffu, l, 0), l1 = __shfl_sync(0xffffffffu, l, 1);
        mx = fmaxf(l0, l1);
        if (mx != -INFINITY) {
            if (l0 != -INFINITY) {
                const float e = __expf(l0 - mx);
                tot += e;
#pragma unroll
                for (int hh = 0; hh < NH; ++hh) r[hh] = fma4(e, v0[hh], r[hh]);
            }
            if (l1 != -INFINITY) {
                const float e = __expf(l1 - mx);
                tot += e;
#pragma unroll
                for (int hh = 0; hh < NH; ++hh) r[hh] = fma4(e, v1[hh], r[hh]);
            }
        }
    } else {
        // P-part splits: lane p reads part p's LSE, 32 parts at a time
        mx = -INFINITY;
        for (int p0 = 0; p0 < np; p0 += 32) {
            const int p = p0 + lane;
            if (p < np) mx = fmaxf(mx, lse_row[p * blk]);
        }
        mx = warp_max(mx);
        for (int p0 = 0; p0 < np && mx != -INFINITY; p0 += 32) {
            const int p = p0 + lane;
            float e = 0.f;
            if (p < np) {
                const float lp = lse_row[p * blk];
                if (lp != -INFINITY) e = __expf(lp - mx);
            }
            tot += warp_sum(e);
            const int cnt = min(32, np - p0);
            for (int j = 0; j < cnt; ++j) {
                const float ej = __shfl_sync(0xffffffffu, e, j);
                const int pj = p0 + j;
#pragma unroll
                for (int hh = 0; hh < NH; ++hh) {
                    const int d = 4 * lane + 128 * hh;
                    float4 v = pj == 0 ? v0[hh] : v1[hh];
                    if (pj > 1 && d < D) v = *reinterpret_cast<const float4*>(o_row + pj * blk + d);
                    if (ej != 0.f) r[hh] = fma4(ej, v, r[hh]);
                }
            }
        }
    }
    float lse = -INFINITY;
    if (mx != -INFINITY) {
        lse = mx + __logf(tot);
        const float inv = 1.f / tot;
#pragma unroll
        for (int hh = 0; hh < NH; ++hh) {
            r[hh].x *= inv;
            r[hh].y *= inv;
            r[hh].z *= inv;
            r[hh].w *= inv;
        }
    }
    const int b = bh / a.g.H, h = bh % a.g.H;
    __nv_bfloat16* O = reinterpret_cast<__nv_bfloat16*>(a.o) + (int64_t)b * a.g.sb + (int64_t)h * a.g.sh +
                       (int64_t)t * a.g.st;
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) {
        const int d = 4 * lane + 128 * hh;
        if (d < D)
            *reinterpret_cast<uint2*>(O + d) = make_uint2(pack_bf16(r[hh].x, r[hh].y), pack_bf16(r[hh].z, r[hh].w));
    }
    if (lane == 0) a.lse[(int64_t)bh * a.g.T + t] = lse;
}

}  // namespace

cudaError_t launch_fwd_merge(const MergeArgs& a, cudaStream_t s) {
    if (a.total_work <= 0) return cudaSuccess;
    const int64_t blocks = (a.total_work + 7) / 8;
    if (blocks > INT32_MAX) return cudaErrorInvalidValue;
    if (a.g.D > 128)
        merge_kernel<2><<<(unsigned)blocks, 256, 0, s>>>(a);
    else
        merge_kernel<1><<<(unsigned)blocks, 256, 0, s>>>(a);
    return counted(cudaGetLastError());
}

}  // namespace attn
