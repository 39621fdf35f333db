// Forward tile kernel (warp-level bf16 mma) and the log-sum-exp merge kernel.
//
// One CTA = one work item x one (batch, head): 128 query rows against the
// item's key range, in blocks of 64 keys, with the online softmax that turns
// the per-block products S_i V_i of Ring Self-Attention ("Sequence
// Parallelism: Long Sequence Training from System Perspective", Deep Dive) into
// the exact softmax: m = running row max, l = running row sum, O rescaled by
// 2^(m_old - m_new) whenever the max grows. Scores are kept in base 2
// (scale * log2 e folded into the exponent); LSE is written in natural log.
#include "device_common.cuh"

namespace attn {
namespace {

constexpr int FM = 128;   // query rows per CTA
constexpr int FN = 64;    // keys per block
constexpr int FWARPS = 8;
constexpr int FTHREADS = FWARPS * 32;

template <int D>
struct FwdSmem {
    static constexpr int DCH = D / 8;
    static constexpr int Q = FM * D;        // elements
    static constexpr int KV = FN * D;
    static constexpr size_t bytes = (size_t)(Q + 4 * KV) * 2;
};

template <int D>
__device__ __forceinline__ void load_rows(__nv_bfloat16* dst, const __nv_bfloat16* src, int64_t st, int row0,
                                          int nrows, int valid_end, int tid) {
    constexpr int DCH = D / 8;
    for (int i = tid; i < nrows * DCH; i += FTHREADS) {
        int r = i / DCH, ch = i % DCH;
        int t = row0 + r;
        bool ok = t < valid_end;
        const __nv_bfloat16* s = src + (int64_t)(ok ? t : row0) * st + ch * 8;
        cp_async16(smem_u32(dst + swz<DCH>(r, ch)), s, ok);
    }
}

template <int D>
__global__ void __launch_bounds__(FTHREADS, 1) fwd_mma_kernel(FwdArgs a) {
    constexpr int DCH = D / 8;
    constexpr int KS = D / 16;      // k-steps over the head dim
    constexpr int NT = FN / 8;      // n-tiles of S per warp
    constexpr int OT = D / 8;       // n-tiles of O per warp
    extern __shared__ __align__(128) uint8_t smem_raw[];
    __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(smem_raw);
    __nv_bfloat16* sK = sQ + FwdSmem<D>::Q;
    __nv_bfloat16* sV = sK + 2 * FwdSmem<D>::KV;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g4 = lane >> 2, c4 = lane & 3;
    const int BH = a.g.B * a.g.H;
    int32_t it, bh;
    decode_work(blockIdx.x, a.n_items, BH, a.group, it, bh);
    const FwdItem item = a.items[it];
    const int b = bh / a.g.H, h = bh % a.g.H;
    const int64_t base = (int64_t)b * a.g.sb + (int64_t)h * a.g.sh;
    const __nv_bfloat16* Qg = reinterpret_cast<const __nv_bfloat16*>(a.q) + base;
    const __nv_bfloat16* Kg = reinterpret_cast<const __nv_bfloat16*>(a.k) + base;
    const __nv_bfloat16* Vg = reinterpret_cast<const __nv_bfloat16*>(a.v) + base;
    const int r0 = item.r0, r1 = item.r1, lo = item.kv_lo, hi = item.kv_hi;
    const float sl2 = a.g.scale * kLog2e;

    load_rows<D>(sQ, Qg, a.g.st, r0, FM, r1, tid);
    cp_async_commit();
    const int nblk = hi > lo ? (hi - lo + FN - 1) / FN : 0;
    if (nblk > 0) {
        load_rows<D>(sK, Kg, a.g.st, lo, FN, hi, tid);
        load_rows<D>(sV, Vg, a.g.st, lo, FN, hi, tid);
    }
    cp_async_commit();

    float o[OT][4];
#pragma unroll
    for (int i = 0; i < OT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
    uint32_t qf[KS][4];
    const int row_a = r0 + warp * 16 + g4, row_b = row_a + 8;

    cp_async_wait<1>();
    __syncthreads();
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
        int r = warp * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
        int ch = 2 * ks + (lane >> 4);
        ldsm_x4(smem_u32(sQ + swz<DCH>(r, ch)), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
    }

    for (int blk = 0; blk < nblk; ++blk) {
        const int buf = blk & 1;
        if (blk + 1 < nblk) {
            int j1 = lo + (blk + 1) * FN;
            load_rows<D>(sK + (buf ^ 1) * FwdSmem<D>::KV, Kg, a.g.st, j1, FN, hi, tid);
            load_rows<D>(sV + (buf ^ 1) * FwdSmem<D>::KV, Vg, a.g.st, j1, FN, hi, tid);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const __nv_bfloat16* cK = sK + buf * FwdSmem<D>::KV;
        const __nv_bfloat16* cV = sV + buf * FwdSmem<D>::KV;
        const int j0 = lo + blk * FN;

        float s[NT][4];
#pragma unroll
        for (int i = 0; i < NT; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
            for (int np = 0; np < NT / 2; ++np) {
                int key = np * 16 + (lane & 7) + 8 * (lane >> 4);
                int ch = 2 * ks + ((lane >> 3) & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(smem_u32(cK + swz<DCH>(key, ch)), b0, b1, b2, b3);
                mma16816(s[2 * np], qf[ks], b0, b1);
                mma16816(s[2 * np + 1], qf[ks], b2, b3);
            }
        }
        // scale to base 2, mask, new running max
        const bool need_mask = (j0 + FN - 1 > r0) || (j0 + FN > hi);
        float mx_a = m_a, mx_b = m_b;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float xa = s[nt][e] * sl2, xb = s[nt][2 + e] * sl2;
                if (need_mask) {
                    int j = j0 + nt * 8 + 2 * c4 + e;
                    if (j > row_a || j >= hi) xa = -INFINITY;
                    if (j > row_b || j >= hi) xb = -INFINITY;
                }
                s[nt][e] = xa;
                s[nt][2 + e] = xb;
                mx_a = fmaxf(mx_a, xa);
                mx_b = fmaxf(mx_b, xb);
            }
        }
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
        const float base_a = mx_a == -INFINITY ? 0.f : mx_a;
        const float base_b = mx_b == -INFINITY ? 0.f : mx_b;
        const float alpha_a = ex2(m_a - base_a), alpha_b = ex2(m_b - base_b);
        m_a = mx_a;
        m_b = mx_b;
        l_a *= alpha_a;
        l_b *= alpha_b;
#pragma unroll
        for (int i = 0; i < OT; ++i) {
            o[i][0] *= alpha_a; o[i][1] *= alpha_a;
            o[i][2] *= alpha_b; o[i][3] *= alpha_b;
        }
        uint32_t pf[FN / 16][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            float p0 = ex2(s[nt][0] - base_a), p1 = ex2(s[nt][1] - base_a);
            float p2 = ex2(s[nt][2] - base_b), p3 = ex2(s[nt][3] - base_b);
            l_a += p0 + p1;
            l_b += p2 + p3;
            pf[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16(p0, p1);
            pf[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16(p2, p3);
        }
        // O += P V
#pragma unroll
        for (int kk = 0; kk < FN / 16; ++kk) {
#pragma unroll
            for (int dp = 0; dp < OT / 2; ++dp) {
                int key = kk * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
                int ch = 2 * dp + (lane >> 4);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(smem_u32(cV + swz<DCH>(key, ch)), b0, b1, b2, b3);
                mma16816(o[2 * dp], pf[kk], b0, b1);
                mma16816(o[2 * dp + 1], pf[kk], b2, b3);
            }
        }
        __syncthreads();
    }

    l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
    const float inv_a = l_a > 0.f ? 1.f / l_a : 0.f;
    const float inv_b = l_b > 0.f ? 1.f / l_b : 0.f;
    const float lse_a = l_a > 0.f ? (m_a + lg2(l_a)) * kLn2 : -INFINITY;
    const float lse_b = l_b > 0.f ? (m_b + lg2(l_b)) * kLn2 : -INFINITY;

    if (item.part_off < 0) {
        __nv_bfloat16* Og = reinterpret_cast<__nv_bfloat16*>(a.o) + base;
        float* L = a.lse + (int64_t)bh * a.g.T;
#pragma unroll
        for (int i = 0; i < OT; ++i) {
            int d = i * 8 + 2 * c4;
            if (row_a < r1)
                *reinterpret_cast<uint32_t*>(Og + (int64_t)row_a * a.g.st + d) = pack_bf16(o[i][0] * inv_a, o[i][1] * inv_a);
            if (row_b < r1)
                *reinterpret_cast<uint32_t*>(Og + (int64_t)row_b * a.g.st + d) = pack_bf16(o[i][2] * inv_b, o[i][3] * inv_b);
        }
        if (c4 == 0) {
            if (row_a < r1) L[row_a] = lse_a;
            if (row_b < r1) L[row_b] = lse_b;
        }
    } else {
        const int64_t R = item.part_R;
        float* P = a.ws_f + item.part_off;
        float* PL = P + (int64_t)BH * R * D + (int64_t)bh * R;
        const int ia = row_a - item.part_row0, ib = row_b - item.part_row0;
#pragma unroll
        for (int i = 0; i < OT; ++i) {
            int d = i * 8 + 2 * c4;
            if (row_a < r1)
                *reinterpret_cast<float2*>(P + ((int64_t)bh * R + ia) * D + d) = make_float2(o[i][0] * inv_a, o[i][1] * inv_a);
            if (row_b < r1)
                *reinterpret_cast<float2*>(P + ((int64_t)bh * R + ib) * D + d) = make_float2(o[i][2] * inv_b, o[i][3] * inv_b);
        }
        if (c4 == 0) {
            if (row_a < r1) PL[ia] = lse_a;
            if (row_b < r1) PL[ib] = lse_b;
        }
    }
}

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

cudaError_t launch_fwd_tiles(const FwdArgs& a, cudaStream_t s) {
    const int64_t work = (int64_t)a.n_items * a.g.B * a.g.H;
    if (work <= 0) return cudaSuccess;
    if (work > INT32_MAX) return cudaErrorInvalidValue;
    if (a.g.D == 128) {
        size_t sm = FwdSmem<128>::bytes;
        cudaError_t e = cudaFuncSetAttribute(fwd_mma_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        if (e != cudaSuccess) return e;
        fwd_mma_kernel<128><<<(unsigned)work, FTHREADS, sm, s>>>(a);
    } else {
        size_t sm = FwdSmem<64>::bytes;
        cudaError_t e = cudaFuncSetAttribute(fwd_mma_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        if (e != cudaSuccess) return e;
        fwd_mma_kernel<64><<<(unsigned)work, FTHREADS, sm, s>>>(a);
    }
    return cudaGetLastError();
}

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
