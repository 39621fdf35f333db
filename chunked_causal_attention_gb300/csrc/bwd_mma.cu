// Backward kernels (warp-level bf16 mma): preprocess, key-tile gradients, dQ
// finalize.
//
// The key-tile kernel owns 128 keys of one (batch, head) and walks every
// query block that can see them (queries t >= j up to the document end): a
// key's dK/dV gather contributions from all later tokens of its sequence
// (InfiniPipe §II-A "Pipeline Parallelism": the backward of a slice needs the
// slices after it). Per query block of 64 rows, with S^T and dP^T kept with
// keys as rows so that P^T and dS^T feed the dV and dK products straight
// from registers:
//     S^T = K Q^T,  P^T = 2^(S^T * scale*log2 e - LSE_t*log2 e)
//     dP^T = V dO^T, dS^T = P^T o (dP^T - D_t)
//     dV += P^T dO,  dK += dS^T Q,  dQ += dS K  (fp32 atomics into the workspace)
// dK is scaled by the softmax scale at the end; dQ's scale is applied before
// the atomics.
#include "device_common.cuh"

namespace attn {
namespace {

constexpr int BN = 128;   // keys per CTA
constexpr int BM = 64;    // queries per step
constexpr int BWARPS = 8;
constexpr int BTHREADS = BWARPS * 32;

template <int D>
struct BwdSmem {
    static constexpr int KV = BN * D;
    static constexpr int QB = BM * D;
    static constexpr int DS = BN * BM;
    static constexpr size_t bytes = (size_t)(2 * KV + 4 * QB + DS) * 2 + 4 * BM * 4;
};

template <int D>
__device__ __forceinline__ void load_rows_b(__nv_bfloat16* dst, const __nv_bfloat16* src, int64_t st, int row0,
                                            int nrows, int valid_end, int tid) {
    constexpr int DCH = D / 8;
    for (int i = tid; i < nrows * DCH; i += BTHREADS) {
        int r = i / DCH, ch = i % DCH;
        int t = row0 + r;
        bool ok = t < valid_end;
        const __nv_bfloat16* s = src + (int64_t)(ok ? t : row0) * st + ch * 8;
        cp_async16(smem_u32(dst + swz<DCH>(r, ch)), s, ok);
    }
}

template <int D>
__global__ void __launch_bounds__(BTHREADS, 1) bwd_mma_kernel(BwdArgs a) {
    constexpr int DCH = D / 8;
    constexpr int KS = D / 16;     // k-steps over the head dim
    constexpr int QT = BM / 8;     // n-tiles over the query block
    constexpr int DT = D / 8;      // n-tiles over the head dim
    constexpr int DQT = D / 16;    // dQ n-tiles per warp (half the head dim)
    extern __shared__ __align__(128) uint8_t smem_raw[];
    __nv_bfloat16* sK = reinterpret_cast<__nv_bfloat16*>(smem_raw);
    __nv_bfloat16* sV = sK + BwdSmem<D>::KV;
    __nv_bfloat16* sQ = sV + BwdSmem<D>::KV;         // 2 buffers
    __nv_bfloat16* sO = sQ + 2 * BwdSmem<D>::QB;     // dO, 2 buffers
    __nv_bfloat16* sS = sO + 2 * BwdSmem<D>::QB;     // dS^T [BN][BM]
    float* sL = reinterpret_cast<float*>(sS + BwdSmem<D>::DS);   // 2 x BM (LSE * log2 e)
    float* sDl = sL + 2 * BM;                                      // 2 x BM (delta)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g4 = lane >> 2, c4 = lane & 3;
    const int BH = a.g.B * a.g.H;
    int32_t it, bh;
    decode_work(blockIdx.x, a.n_items, BH, a.group, it, bh);
    const BwdItem item = a.items[it];
    const int b = bh / a.g.H, h = bh % a.g.H;
    const int64_t base = (int64_t)b * a.g.sb + (int64_t)h * a.g.sh;
    const __nv_bfloat16* Qg = reinterpret_cast<const __nv_bfloat16*>(a.q) + base;
    const __nv_bfloat16* Kg = reinterpret_cast<const __nv_bfloat16*>(a.k) + base;
    const __nv_bfloat16* Vg = reinterpret_cast<const __nv_bfloat16*>(a.v) + base;
    const __nv_bfloat16* dOg = reinterpret_cast<const __nv_bfloat16*>(a.dout) + base;
    const float* Lg = a.lse + (int64_t)bh * a.g.T;
    const float* Dg = a.delta + (int64_t)bh * a.g.T;
    float* dQg = a.dq_acc + (int64_t)bh * a.g.T * D;
    const int j0 = item.j0, j1 = item.j1, qend = item.q_end;
    const float sl2 = a.g.scale * kLog2e;
    const int nq = (qend - j0 + BM - 1) / BM;

    load_rows_b<D>(sK, Kg, a.g.st, j0, BN, j1, tid);
    load_rows_b<D>(sV, Vg, a.g.st, j0, BN, j1, tid);
    load_rows_b<D>(sQ, Qg, a.g.st, j0, BM, qend, tid);
    load_rows_b<D>(sO, dOg, a.g.st, j0, BM, qend, tid);
    cp_async_commit();
    if (tid < BM) {
        int t = j0 + tid;
        sL[tid] = t < qend ? Lg[t] * kLog2e : 0.f;
    } else if (tid < 2 * BM) {
        int t = j0 + tid - BM;
        sDl[tid - BM] = t < qend ? Dg[t] : 0.f;
    }

    float dk[DT][4], dv[DT][4];
#pragma unroll
    for (int i = 0; i < DT; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) dk[i][e] = dv[i][e] = 0.f;

    const int key_a = j0 + warp * 16 + g4, key_b = key_a + 8;

    for (int qi = 0; qi < nq; ++qi) {
        const int buf = qi & 1;
        const int i0 = j0 + qi * BM;
        cp_async_wait<0>();
        __syncthreads();
        if (qi + 1 < nq) {
            const int i1 = i0 + BM;
            load_rows_b<D>(sQ + (buf ^ 1) * BwdSmem<D>::QB, Qg, a.g.st, i1, BM, qend, tid);
            load_rows_b<D>(sO + (buf ^ 1) * BwdSmem<D>::QB, dOg, a.g.st, i1, BM, qend, tid);
            cp_async_commit();
            if (tid < BM) {
                int t = i1 + tid;
                sL[(buf ^ 1) * BM + tid] = t < qend ? Lg[t] * kLog2e : 0.f;
            } else if (tid < 2 * BM) {
                int t = i1 + tid - BM;
                sDl[(buf ^ 1) * BM + tid - BM] = t < qend ? Dg[t] : 0.f;
            }
        }
        const __nv_bfloat16* cQ = sQ + buf * BwdSmem<D>::QB;
        const __nv_bfloat16* cO = sO + buf * BwdSmem<D>::QB;
        const float* cL = sL + buf * BM;
        const float* cD = sDl + buf * BM;

        // S^T = K Q^T and dP^T = V dO^T for this warp's 16 keys x 64 queries
        float s[QT][4], dp[QT][4];
#pragma unroll
        for (int i = 0; i < QT; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[i][e] = dp[i][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            uint32_t ka[4], va[4];
            {
                int r = warp * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
                int ch = 2 * ks + (lane >> 4);
                ldsm_x4(smem_u32(sK + swz<DCH>(r, ch)), ka[0], ka[1], ka[2], ka[3]);
                ldsm_x4(smem_u32(sV + swz<DCH>(r, ch)), va[0], va[1], va[2], va[3]);
            }
#pragma unroll
            for (int np = 0; np < QT / 2; ++np) {
                int qr = np * 16 + (lane & 7) + 8 * (lane >> 4);
                int ch = 2 * ks + ((lane >> 3) & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(smem_u32(cQ + swz<DCH>(qr, ch)), b0, b1, b2, b3);
                mma16816(s[2 * np], ka, b0, b1);
                mma16816(s[2 * np + 1], ka, b2, b3);
                ldsm_x4(smem_u32(cO + swz<DCH>(qr, ch)), b0, b1, b2, b3);
                mma16816(dp[2 * np], va, b0, b1);
                mma16816(dp[2 * np + 1], va, b2, b3);
            }
        }
        // P^T and dS^T; dS^T also to shared memory for the dQ product
        uint32_t pa[BM / 16][4], da[BM / 16][4];
#pragma unroll
        for (int nt = 0; nt < QT; ++nt) {
            float pv[4], dsv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                int ql = nt * 8 + 2 * c4 + (e & 1);
                int qg = i0 + ql;
                int key = e < 2 ? key_a : key_b;
                bool vis = key <= qg && qg < qend && key < j1;
                float p = vis ? ex2(s[nt][e] * sl2 - cL[ql]) : 0.f;
                pv[e] = p;
                dsv[e] = p * (dp[nt][e] - cD[ql]);
            }
            pa[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16(pv[0], pv[1]);
            pa[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16(pv[2], pv[3]);
            uint32_t d01 = pack_bf16(dsv[0], dsv[1]);
            uint32_t d23 = pack_bf16(dsv[2], dsv[3]);
            da[nt >> 1][(nt & 1) * 2 + 0] = d01;
            da[nt >> 1][(nt & 1) * 2 + 1] = d23;
            int ra = warp * 16 + g4, rb = ra + 8;
            *reinterpret_cast<uint32_t*>(sS + ra * BM + ((nt ^ (ra & 7)) << 3) + 2 * c4) = d01;
            *reinterpret_cast<uint32_t*>(sS + rb * BM + ((nt ^ (rb & 7)) << 3) + 2 * c4) = d23;
        }
        // dV += P^T dO, dK += dS^T Q
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk) {
#pragma unroll
            for (int dp2 = 0; dp2 < DT / 2; ++dp2) {
                int qr = kk * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
                int ch = 2 * dp2 + (lane >> 4);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(smem_u32(cO + swz<DCH>(qr, ch)), b0, b1, b2, b3);
                mma16816(dv[2 * dp2], pa[kk], b0, b1);
                mma16816(dv[2 * dp2 + 1], pa[kk], b2, b3);
                ldsm_x4_t(smem_u32(cQ + swz<DCH>(qr, ch)), b0, b1, b2, b3);
                mma16816(dk[2 * dp2], da[kk], b0, b1);
                mma16816(dk[2 * dp2 + 1], da[kk], b2, b3);
            }
        }
        __syncthreads();
        // dQ (64 x D) += dS K: warp -> 16 query rows x D/2 columns
        {
            const int qr0 = 16 * (warp & 3);
            const int dc0 = (D / 2) * (warp >> 2);
            float dq[DQT][4];
#pragma unroll
            for (int i = 0; i < DQT; ++i) dq[i][0] = dq[i][1] = dq[i][2] = dq[i][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk) {
                uint32_t af[4];
                {
                    int kr = kk * 16 + (lane & 7) + 8 * (lane >> 4);
                    int qc = (qr0 >> 3) + ((lane >> 3) & 1);
                    ldsm_x4_t(smem_u32(sS + kr * BM + ((qc ^ (kr & 7)) << 3)), af[0], af[1], af[2], af[3]);
                }
#pragma unroll
                for (int dp2 = 0; dp2 < DQT / 2; ++dp2) {
                    int kr = kk * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
                    int ch = (dc0 >> 3) + 2 * dp2 + (lane >> 4);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(smem_u32(sK + swz<DCH>(kr, ch)), b0, b1, b2, b3);
                    mma16816(dq[2 * dp2], af, b0, b1);
                    mma16816(dq[2 * dp2 + 1], af, b2, b3);
                }
            }
            const int qa = i0 + qr0 + g4, qb = qa + 8;
            const float sc = a.g.scale;
#pragma unroll
            for (int nt = 0; nt < DQT; ++nt) {
                int d = dc0 + nt * 8 + 2 * c4;
                if (qa < qend)
                    atomicAdd(reinterpret_cast<float2*>(dQg + (int64_t)qa * D + d), make_float2(dq[nt][0] * sc, dq[nt][1] * sc));
                if (qb < qend)
                    atomicAdd(reinterpret_cast<float2*>(dQg + (int64_t)qb * D + d), make_float2(dq[nt][2] * sc, dq[nt][3] * sc));
            }
        }
    }

    // write dK (scaled) and dV for keys < j1
    __nv_bfloat16* dKg = reinterpret_cast<__nv_bfloat16*>(a.dk) + base;
    __nv_bfloat16* dVg = reinterpret_cast<__nv_bfloat16*>(a.dv) + base;
    const float sc = a.g.scale;
#pragma unroll
    for (int nt = 0; nt < DT; ++nt) {
        int d = nt * 8 + 2 * c4;
        if (key_a < j1) {
            *reinterpret_cast<uint32_t*>(dKg + (int64_t)key_a * a.g.st + d) = pack_bf16(dk[nt][0] * sc, dk[nt][1] * sc);
            *reinterpret_cast<uint32_t*>(dVg + (int64_t)key_a * a.g.st + d) = pack_bf16(dv[nt][0], dv[nt][1]);
        }
        if (key_b < j1) {
            *reinterpret_cast<uint32_t*>(dKg + (int64_t)key_b * a.g.st + d) = pack_bf16(dk[nt][2] * sc, dk[nt][3] * sc);
            *reinterpret_cast<uint32_t*>(dVg + (int64_t)key_b * a.g.st + d) = pack_bf16(dv[nt][2], dv[nt][3]);
        }
    }
}

// One warp per (batch*head, token): delta = dO . O; zero the dQ accumulator row.
template <int D>
__global__ void __launch_bounds__(256) prep_kernel(PrepArgs a) {
    constexpr int PER = D / 32;
    const int64_t w = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int64_t total = (int64_t)a.g.B * a.g.H * a.g.T;
    if (w >= total) return;
    const int bh = (int)(w / a.g.T), t = (int)(w % a.g.T);
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
    const int64_t total = (int64_t)a.g.B * a.g.H * a.g.T;
    if (w >= total) return;
    const int bh = (int)(w / a.g.T), t = (int)(w % a.g.T);
    const int b = bh / a.g.H, h = bh % a.g.H;
    const float* src = a.dq_acc + w * D + lane * PER;
    __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(a.dq) + (int64_t)b * a.g.sb + (int64_t)h * a.g.sh +
                         (int64_t)t * a.g.st + lane * PER;
#pragma unroll
    for (int e = 0; e < PER; e += 2) *reinterpret_cast<uint32_t*>(dst + e) = pack_bf16(src[e], src[e + 1]);
}

}  // namespace

cudaError_t launch_bwd_prep(const PrepArgs& a, cudaStream_t s) {
    const int64_t blocks = ((int64_t)a.g.B * a.g.H * a.g.T + 7) / 8;
    if (blocks > INT32_MAX) return cudaErrorInvalidValue;
    if (a.g.D == 128)
        prep_kernel<128><<<(unsigned)blocks, 256, 0, s>>>(a);
    else
        prep_kernel<64><<<(unsigned)blocks, 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_bwd_dq(const DqArgs& a, cudaStream_t s) {
    const int64_t blocks = ((int64_t)a.g.B * a.g.H * a.g.T + 7) / 8;
    if (blocks > INT32_MAX) return cudaErrorInvalidValue;
    if (a.g.D == 128)
        dq_kernel<128><<<(unsigned)blocks, 256, 0, s>>>(a);
    else
        dq_kernel<64><<<(unsigned)blocks, 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_bwd_tiles(const BwdArgs& a, cudaStream_t s) {
    const int64_t work = (int64_t)a.n_items * a.g.B * a.g.H;
    if (work <= 0) return cudaSuccess;
    if (work > INT32_MAX) return cudaErrorInvalidValue;
    if (a.g.D == 128) {
        size_t sm = BwdSmem<128>::bytes;
        cudaError_t e = cudaFuncSetAttribute(bwd_mma_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        if (e != cudaSuccess) return e;
        bwd_mma_kernel<128><<<(unsigned)work, BTHREADS, sm, s>>>(a);
    } else {
        size_t sm = BwdSmem<64>::bytes;
        cudaError_t e = cudaFuncSetAttribute(bwd_mma_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        if (e != cudaSuccess) return e;
        bwd_mma_kernel<64><<<(unsigned)work, BTHREADS, sm, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace attn
