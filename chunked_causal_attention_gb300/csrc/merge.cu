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
// A block merges RB consecutive (batch*head, segment row) rows of one segment.
// Their partials are contiguous in the workspace, so for a split at one point
// (P = 2, every re-split edge) one thread copies both parts' RB rows into
// shared memory with two bulk copies, and the warps merge the rows from there:
// several blocks per SM keep their copies in flight at once. Segments of P > 2
// parts take one warp per row with loads from global memory. fp32 partials
// in, bf16 O and fp32 LSE out. A segment that does not fit the geometry or the
// workspace is reported as ATTN_E_BOUNDS and not read.
#include "tc_common.cuh"

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

// Rows per block: 32 rows of up to 128 dims, 16 of up to 256 (32 KB of fp32
// partials for two parts either way).
template <int NH>
constexpr int rows_per_block() { return NH == 1 ? 32 : 16; }
static_assert(kBulkParts == 4, "the merge's shared-memory budget assumes at most four parts per bulk copy");

// 1-D bulk copy global -> shared memory, completing on an mbarrier.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
                 : "memory");
}

// Normalise and store one merged row: r holds sum_p e^{LSE_p - mx} O_p with
// tot = sum_p e^{LSE_p - mx}; mx = -inf means no part saw a key.
template <int NH>
__device__ __forceinline__ void store_row(const MergeArgs& a, int bh, int t, int lane, float4 (&r)[NH], float mx,
                                          float tot) {
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
        if (d < a.g.D)
            *reinterpret_cast<uint2*>(O + d) = make_uint2(pack_bf16(r[hh].x, r[hh].y), pack_bf16(r[hh].z, r[hh].w));
    }
    if (lane == 0) a.lse[(int64_t)bh * a.g.T + t] = lse;
}

// Two parts (LSEs l0, l1; O slices v0, v1): the weights in a fixed order, so
// every path gives the same bits.
template <int NH>
__device__ __forceinline__ void merge_two(const float4 (&v0)[NH], const float4 (&v1)[NH], float l0, float l1,
                                          float4 (&r)[NH], float& mx, float& tot) {
    tot = 0.f;
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
}

// Segment row `local` (= bh * R + i) of a segment of any P, one warp, loads
// from global memory: the parts the row sees (a prefix of the segment's
// increasing key boundaries) are counted by one ballot; lane p reads part p's
// LSE; the weights reach all lanes by shuffles.
template <int NH>
__device__ __noinline__ void merge_row_general(const MergeArgs& a, const MergeSeg& sg, int64_t local, int lane) {
    const int D = a.g.D;
    const int BH = a.g.B * a.g.H;
    const int bh = (int)(local / sg.R), i = (int)(local % sg.R);
    const int t = sg.row0 + i;
    const int64_t R = sg.R, blk = sg.blk;
    const int32_t* kb = a.kbounds + sg.kb;
    int np = 0;
    for (int p0 = 0; p0 < sg.P; p0 += 32) {
        const int p = p0 + lane;
        np += __popc(__ballot_sync(0xffffffffu, p < sg.P && kb[p] <= t));
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
        const float l = lane < np ? lse_row[lane * blk] : -INFINITY;
        merge_two<NH>(v0, v1, __shfl_sync(0xffffffffu, l, 0), __shfl_sync(0xffffffffu, l, 1), r, mx, tot);
    } else {
        // lane p reads part p's LSE, 32 parts at a time
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
    store_row<NH>(a, bh, t, lane, r, mx, tot);
}

// Block b merges rows [local0, local0 + RB) of the segment whose block range
// holds b. The rows' partials are contiguous in the workspace, so for a
// segment of up to kBulkParts parts one thread copies every part's rows into
// shared memory with one bulk copy per part, while thread r works out row r's
// weights (the parts the row sees: all of them for a split at one point, whose
// part 1 is written for every row, with LSE = -inf where the row sees none of
// its keys; otherwise those whose key range starts at or before the row), its
// LSE and its O row; then the warps merge the rows from shared memory. A part
// the row does not see is never read, whatever its buffer holds. Segments of
// more parts take one warp per row with loads from global memory. Lane l of a
// warp takes the four elements from d = 4l, and for NH = 2 (head dims above
// 128) also those from d = 4l + 128 (D is a multiple of 8, at most 128 * NH).
// The segment table comes from the kernel parameters when it is short (no
// dependent load before the copies).
template <int NH, int NP>
__global__ void __launch_bounds__(256) merge_kernel(const __grid_constant__ MergeArgs a) {
    constexpr int RB = rows_per_block<NH>();
    extern __shared__ __align__(128) float s_part[];    // [P][RB][D] fp32
    __shared__ float s_e[NP + 1][RB];                    // per row: e^{LSE_p - mx}, then 1 / sum
    __shared__ int s_use[RB];                            // per row: bit p = part p has weight
    __shared__ int64_t s_off[RB];                        // per row: element offset of its O row
    __shared__ __align__(8) uint64_t s_bar;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int D = a.g.D;
    const int BH = a.g.B * a.g.H;
    const MergeSeg* segs = a.n_segs <= kMergeSegsInline ? a.segs_inline : a.segs;
    // the segment: the last one whose first block is at or before this block
    int lo = 0, hi = a.n_segs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (segs[mid].work0 <= (int64_t)blockIdx.x) lo = mid; else hi = mid - 1;
    }
    const MergeSeg sg = segs[lo];
    const int64_t rows = (int64_t)sg.R * BH;
    const int64_t local0 = ((int64_t)blockIdx.x - sg.work0) * RB;
    // index checks of the segment before any address is formed from it (the
    // same answer in every thread of the block)
    if (!(sg.R > 0 && sg.row0 >= 0 && (int64_t)sg.row0 + sg.R <= a.g.T && sg.P >= 1 && sg.P <= 64 && sg.kb >= 0 &&
          sg.kb + sg.P + 1 <= a.n_kbounds && local0 >= 0 && local0 < rows && sg.off0 >= 0 &&
          sg.blk >= (int64_t)BH * sg.R * (D + 1) && sg.off0 + sg.P * sg.blk <= a.part_floats)) {
        if (threadIdx.x == 0) set_error(a.status, ATTN_E_BOUNDS);
        return;
    }
    const int nrow = (int)(rows - local0 < RB ? rows - local0 : RB);
    const int P = sg.P;
    if (P > NP) {
        for (int r = warp; r < nrow; r += 8) merge_row_general<NH>(a, sg, local0 + r, lane);
        return;
    }
    const float* part0 = a.ws_f + sg.off0 + local0 * D;          // part p's rows at part0 + p * blk
    const float* lse0 = a.ws_f + sg.off0 + rows * D + local0;     // part p's LSEs at lse0[p * blk]
    const uint32_t bar = smem_u32(&s_bar);
    const uint32_t bytes = (uint32_t)nrow * D * 4;
    if (threadIdx.x == 0) {
        tc::mbar_init(bar, 1);
        tc::fence_barrier_init();
        tc::mbar_expect_tx(bar, (uint32_t)P * bytes);
        for (int p = 0; p < P; ++p) bulk_load(smem_u32(s_part + p * RB * D), part0 + p * sg.blk, bytes, bar);
    }
    // while the copies are in flight, thread r < nrow works out row r's weights
    // (added in part order, as merge_row_general adds the O rows), writes its LSE
    // and finds its O row
    if (threadIdx.x < nrow) {
        const int r = threadIdx.x;
        const int64_t local = local0 + r;
        int bh, i;
        if (local <= INT32_MAX) {
            const uint32_t l = (uint32_t)local, R = (uint32_t)sg.R;
            bh = (int)(l / R);
            i = (int)(l - (uint32_t)bh * R);
        } else {
            bh = (int)(local / sg.R);
            i = (int)(local % sg.R);
        }
        const int t = sg.row0 + i;
        int np = P;
        if (P != 2) {
            const int32_t* kb = a.kbounds + sg.kb;
            np = 0;
            for (int p = 0; p < P; ++p) np += kb[p] <= t;
        }
        float l[NP];
        float mx = -INFINITY;
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            l[p] = p < np ? lse0[p * sg.blk + r] : -INFINITY;
            mx = fmaxf(mx, l[p]);
        }
        float tot = 0.f, inv = 1.f, lse = -INFINITY;
        int use = 0;
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            float e = 0.f;
            if (mx != -INFINITY && l[p] != -INFINITY) {
                e = __expf(l[p] - mx);
                tot += e;
                use |= 1 << p;
            }
            s_e[p][r] = e;
        }
        if (mx != -INFINITY) {
            lse = mx + __logf(tot);
            inv = 1.f / tot;
        }
        s_e[NP][r] = inv;
        s_use[r] = use;
        const int b = bh / a.g.H, h = bh % a.g.H;
        s_off[r] = (int64_t)b * a.g.sb + (int64_t)h * a.g.sh + (int64_t)t * a.g.st;
        a.lse[(int64_t)bh * a.g.T + t] = lse;
    }
    // One thread waits for the copies (the others wait at the barrier without
    // taking issue slots). They always complete; the wait is bounded all the
    // same, and a block that gives up records ATTN_E_TIMEOUT and waits once more
    // before leaving.
    bool ok = true;
    if (threadIdx.x == 0) {
        ok = tc::mbar_try_wait(bar, 0);
        const uint64_t t0 = tc::globaltimer();
        while (!ok && tc::globaltimer() - t0 < 1000000000ull) ok = tc::mbar_try_wait(bar, 0);
        if (!ok) {
            set_error(a.status, ATTN_E_TIMEOUT);
            const uint64_t t1 = tc::globaltimer();
            while (!tc::mbar_try_wait(bar, 0) && tc::globaltimer() - t1 < 1000000000ull) {
            }
        }
    }
    if (!__syncthreads_and(ok)) return;
    __nv_bfloat16* O = reinterpret_cast<__nv_bfloat16*>(a.o);
    for (int r = warp; r < nrow; r += 8) {
        const int use = s_use[r];
        const float inv = s_e[NP][r];
        __nv_bfloat16* orow = O + s_off[r];
#pragma unroll
        for (int hh = 0; hh < NH; ++hh) {
            const int d = 4 * lane + 128 * hh;
            if (d < D) {
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int p = 0; p < NP; ++p)
                    if (use & (1 << p))
                        acc = fma4(s_e[p][r], *reinterpret_cast<const float4*>(s_part + (p * RB + r) * D + d), acc);
                if (use) {
                    acc.x *= inv;
                    acc.y *= inv;
                    acc.z *= inv;
                    acc.w *= inv;
                }
                *reinterpret_cast<uint2*>(orow + d) = make_uint2(pack_bf16(acc.x, acc.y), pack_bf16(acc.z, acc.w));
            }
        }
    }
}

}  // namespace

int merge_rows_per_block(int D) { return D > 128 ? rows_per_block<2>() : rows_per_block<1>(); }

cudaError_t launch_fwd_merge(const MergeArgs& a, cudaStream_t s) {
    if (a.total_work <= 0) return cudaSuccess;
    if (a.total_work > INT32_MAX) return cudaErrorInvalidValue;
    const int RB = merge_rows_per_block(a.g.D);
    if (a.bulk_parts < 2 || a.bulk_parts > kBulkParts) return cudaErrorInvalidValue;
    // splits at one point only (every re-split edge): the two-part instantiation
    const int np = a.bulk_parts == 2 ? 2 : kBulkParts;
    const size_t smem = (size_t)a.bulk_parts * RB * a.g.D * sizeof(float);   // up to 64 KB
    auto kern = a.g.D > 128 ? (np == 2 ? merge_kernel<2, 2> : merge_kernel<2, kBulkParts>)
                            : (np == 2 ? merge_kernel<1, 2> : merge_kernel<1, kBulkParts>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)a.total_work, 256, smem, s>>>(a);
    return counted(cudaGetLastError());
}

}  // namespace attn
