// Backward key-tile kernel on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// One work item = 128 keys [j0, j1) of one (batch, head); the item walks the
// query blocks of 128 rows that can see those keys (queries t >= j0 up to the
// document end) from the last block down to the diagonal one, so the CTAs
// working on one head meet the same Q/dO tiles and dQ rows at about the same
// time and both stay in L2: a key's dK/dV collect the contributions of every later
// token of its sequence (InfiniPipe §II-A: K/V gradients of a token depend on
// all subsequent tokens). Persistent CTAs take items from the cost-sorted list.
//
// Warp roles:
//   warp 0      TMA producer: K, V once per item; Q and dO per query block
//               through a two-stage ring.
//   warp 1      MMA issuer (one thread) and TMEM owner. Per query block:
//                 S^T  = K Q^T     -> TMEM [0,128)      (SS, both K-major)
//                 dP^T = V dO^T    -> TMEM [128,256)    (SS, both K-major)
//                 dV  += P^T dO    -> TMEM dV           (A = P^T in TMEM, B = dO MN-major)
//                 dK  += dS^T Q    -> TMEM dK           (A = dS^T in TMEM, B = Q MN-major)
//                 dQ   = dS K      -> TMEM [128,128+D)  (A = dS MN-major in shared memory,
//                                                        B = K MN-major)
//   warps 4-7   softmax gradient, one key row per thread (TMEM lane = key):
//                 P^T  = 2^(S^T * scale*log2 e - LSE_t*log2 e)   (zero where t < key or t >= end)
//                 dS^T = P^T o (dP^T - D_t)
//               P^T and dS^T go back to TMEM as bf16 (A operands of dV, dK), dS
//               also to shared memory for dQ; at the end of the item these
//               warps write dK * scale and dV as bf16.
//   warps 8-11  dQ drain, one query row per thread: dQ * scale from TMEM,
//               added into the fp32 workspace accumulator with vector atomics.
// Every mbarrier wait is bounded (ATTN_E_TIMEOUT in the status word).
#include "tc_common.cuh"

namespace attn {
namespace {

using namespace tc;

constexpr int BT_THREADS = 384;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;
constexpr uint32_t kColDP = 128;
constexpr uint32_t kColDV = 256;
constexpr uint64_t kWaitNs = 4000000000ull;

template <int D>
struct BwdTcLayout {
    static constexpr int TILE = 128 * D * 2;
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = K_OFF + TILE;
    static constexpr int Q_OFF = V_OFF + TILE;            // 2 stages
    static constexpr int DO_OFF = Q_OFF + 2 * TILE;       // 2 stages
    static constexpr int DS_OFF = DO_OFF + 2 * TILE;      // 128 keys x 128 queries bf16, MN-major
    static constexpr int LSE_OFF = DS_OFF + 32768;        // 128 floats (LSE * log2 e)
    static constexpr int DLT_OFF = LSE_OFF + 512;         // 128 floats (D_t)
    static constexpr int BAR_OFF = DLT_OFF + 512;
    static constexpr int B_KVFULL = 0, B_KVEMPTY = 1;
    static constexpr int B_QFULL = 2, B_QEMPTY = 4;       // 2 each
    static constexpr int B_SDP = 6, B_PCH = 7;            // B_PCH + c: P^T/dS^T of query chunk c ready
    static constexpr int B_DQFULL = 11, B_DQFREE = 12;
    static constexpr int B_DKDVFULL = 13, B_DKDVFREE = 14, B_DRAIN = 15;
    static constexpr int NBAR = 16;
    static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
    static constexpr int BYTES = MISC_OFF + 16;
    static constexpr size_t ALLOC = (size_t)BYTES + 1024;
};

__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory");
}

template <int D>
__device__ __forceinline__ void load_tile_b(uint32_t dst, const CUtensorMap* map, uint32_t bar, const TcMaps& mp,
                                            int row, int h, int b) {
    int c[4];
    c[0] = 0;
    c[mp.pos_t] = row;
    c[mp.pos_h] = h;
    c[mp.pos_b] = b;
#pragma unroll
    for (int a = 0; a < D / 64; ++a) tma_load_4d(dst + a * 16384, map, bar, a * 64, c[1], c[2], c[3]);
}

template <int D>
__global__ void __launch_bounds__(BT_THREADS, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo, const BwdArgs a,
                  const TcMaps mp, const int32_t n_work) {
    using LY = BwdTcLayout<D>;
    constexpr uint32_t kColDK = kColDV + D;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);
    const uint32_t bar0 = sbase + LY::BAR_OFF;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + LY::MISC_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + LY::MISC_OFF + 4);
    float* s_lse = reinterpret_cast<float*>(sm + LY::LSE_OFF);
    float* s_dlt = reinterpret_cast<float*>(sm + LY::DLT_OFF);

    const int tid = threadIdx.x, warp = tid >> 5;
    const int BH = a.g.B * a.g.H;

    if (tid == 0) {
        mbar_init(bar(LY::B_KVFULL), 1);
        mbar_init(bar(LY::B_KVEMPTY), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(LY::B_QFULL + s), 1);
            mbar_init(bar(LY::B_QEMPTY + s), 1);
        }
        mbar_init(bar(LY::B_SDP), 1);
        for (int c = 0; c < 4; ++c) mbar_init(bar(LY::B_PCH + c), 128);
        mbar_init(bar(LY::B_DQFULL), 1);
        mbar_init(bar(LY::B_DQFREE), 128);
        mbar_init(bar(LY::B_DKDVFULL), 1);
        mbar_init(bar(LY::B_DKDVFREE), 128);
        mbar_init(bar(LY::B_DRAIN), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (elect_one()) {
            tma_prefetch_desc(&tmq);
            tma_prefetch_desc(&tmk);
            tma_prefetch_desc(&tmv);
            tma_prefetch_desc(&tmdo);
            uint32_t qc = 0, ic = 0;
            bool ok = true;
            for (int w = blockIdx.x; w < n_work && ok && !*abort_flag; w += gridDim.x, ++ic) {
                int32_t it, bh;
                decode_work(w, a.n_items, BH, a.group, it, bh);
                const BwdItem item = a.items[it];
                const int b = bh / a.g.H, h = bh % a.g.H;
                ok = mbar_wait(bar(LY::B_KVEMPTY), (ic & 1) ^ 1, abort_flag, a.status, kWaitNs);
                if (!ok) break;
                mbar_expect_tx(bar(LY::B_KVFULL), 2 * LY::TILE);
                load_tile_b<D>(sbase + LY::K_OFF, &tmk, bar(LY::B_KVFULL), mp, item.j0, h, b);
                load_tile_b<D>(sbase + LY::V_OFF, &tmv, bar(LY::B_KVFULL), mp, item.j0, h, b);
                const int nq = (item.q_end - item.j0 + 127) / 128;
                for (int i = 0; i < nq; ++i, ++qc) {
                    const uint32_t s = qc & 1;
                    ok = mbar_wait(bar(LY::B_QEMPTY + s), ((qc >> 1) & 1) ^ 1, abort_flag, a.status, kWaitNs);
                    if (!ok) break;
                    mbar_expect_tx(bar(LY::B_QFULL + s), 2 * LY::TILE);
                    const int row = item.j0 + (nq - 1 - i) * 128;
                    load_tile_b<D>(sbase + LY::Q_OFF + s * LY::TILE, &tmq, bar(LY::B_QFULL + s), mp, row, h, b);
                    load_tile_b<D>(sbase + LY::DO_OFF + s * LY::TILE, &tmdo, bar(LY::B_QFULL + s), mp, row, h, b);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (elect_one()) {
            constexpr uint32_t id_s = idesc_bf16(128, 128, 0, 0);
            constexpr uint32_t id_g = idesc_bf16(128, D, 0, 1);    // dV, dK: A from TMEM, B MN-major
            constexpr uint32_t id_q = idesc_bf16(128, D, 1, 1);    // dQ: A, B MN-major
            const uint32_t k0 = sbase + LY::K_OFF, v0 = sbase + LY::V_OFF, ds0 = sbase + LY::DS_OFF;
            uint32_t qc = 0, ic = 0, gb = 0;
            bool ok = true;
            for (int w = blockIdx.x; w < n_work && ok && !*abort_flag; w += gridDim.x, ++ic) {
                int32_t it, bh;
                decode_work(w, a.n_items, BH, a.group, it, bh);
                const BwdItem item = a.items[it];
                const int nq = (item.q_end - item.j0 + 127) / 128;
                ok = mbar_wait(bar(LY::B_KVFULL), ic & 1, abort_flag, a.status, kWaitNs);
                if (!ok) break;
                tc_fence_after();
                for (int i = 0; i < nq; ++i, ++qc, ++gb) {
                    const uint32_t s = qc & 1;
                    ok = mbar_wait(bar(LY::B_QFULL + s), (qc >> 1) & 1, abort_flag, a.status, kWaitNs);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t q0 = sbase + LY::Q_OFF + s * LY::TILE;
                    const uint32_t o0 = sbase + LY::DO_OFF + s * LY::TILE;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                        mma_ss(tmem + kColS, sdesc_sw128(k0 + off, 16, 1024), sdesc_sw128(q0 + off, 16, 1024), id_s,
                               kk > 0);
                    }
                    if (gb > 0) {
                        ok = mbar_wait(bar(LY::B_DQFREE), (gb - 1) & 1, abort_flag, a.status, kWaitNs);
                        if (!ok) break;
                        tc_fence_after();
                    }
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                        mma_ss(tmem + kColDP, sdesc_sw128(v0 + off, 16, 1024), sdesc_sw128(o0 + off, 16, 1024), id_s,
                               kk > 0);
                    }
                    mma_commit(bar(LY::B_SDP));
                    if (i == 0) {
                        ok = mbar_wait(bar(LY::B_DKDVFREE), (ic & 1) ^ 1, abort_flag, a.status, kWaitNs);
                        if (!ok) break;
                    }
                    // dV += P^T dO and dK += dS^T Q, 32 queries (two k-steps) at a time as the
                    // softmax-gradient warps finish each chunk
                    for (int c = 0; c < 4 && ok; ++c) {
                        ok = mbar_wait(bar(LY::B_PCH + c), gb & 1, abort_flag, a.status, kWaitNs);
                        if (!ok) break;
                        tc_fence_after();
#pragma unroll
                        for (int kk = 2 * c; kk < 2 * c + 2; ++kk) {
                            mma_ts(tmem + kColDV, tmem + kColS + kk * 8, sdesc_sw128(o0 + kk * 2048, 16384, 1024), id_g,
                                   (i > 0 || kk > 0) ? 1u : 0u);
                            mma_ts(tmem + kColDK, tmem + kColDP + kk * 8, sdesc_sw128(q0 + kk * 2048, 16384, 1024),
                                   id_g, (i > 0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    if (!ok) break;
                    mma_commit(bar(LY::B_QEMPTY + s));
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ss(tmem + kColDP, sdesc_sw128(ds0 + kk * 2048, 16384, 1024),
                               sdesc_sw128(k0 + kk * 2048, 16384, 1024), id_q, kk > 0);
                    mma_commit(bar(LY::B_DQFULL));
                }
                if (!ok) break;
                mma_commit(bar(LY::B_KVEMPTY));
                mma_commit(bar(LY::B_DKDVFULL));
            }
        }
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ softmax gradient + dK/dV epilogue
        const int krow = tid - 128;
        const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
        const float sl2 = a.g.scale * kLog2e;
        const float* Lg = a.lse + 0;
        uint32_t gb = 0, ic = 0;
        bool ok = true;
        uint8_t* ds_row = sm + LY::DS_OFF + krow * 128;
        for (int w = blockIdx.x; w < n_work && ok && !*abort_flag; w += gridDim.x, ++ic) {
            int32_t it, bh;
            decode_work(w, a.n_items, BH, a.group, it, bh);
            const BwdItem item = a.items[it];
            const int nq = (item.q_end - item.j0 + 127) / 128;
            const int key = item.j0 + krow;
            const float* L = Lg + (int64_t)bh * a.g.T;
            const float* Dl = a.delta + (int64_t)bh * a.g.T;
            // LSE and D_t of the next query block are fetched one block ahead into
            // registers, so the global-load latency stays off the critical path
            float next_l = 0.f, next_d = 0.f;
            {
                const int q = item.j0 + (nq - 1) * 128 + krow;
                if (q < item.q_end) {
                    next_l = L[q] * kLog2e;
                    next_d = Dl[q];
                }
            }
            for (int i = 0; i < nq; ++i, ++gb) {
                const int i0 = item.j0 + (nq - 1 - i) * 128;   // query blocks walked from the last one down
                named_sync(1, 128);
                s_lse[krow] = next_l;
                s_dlt[krow] = next_d;
                named_sync(1, 128);
                if (i + 1 < nq) {
                    const int q = i0 - 128 + krow;             // next block (always inside the document)
                    next_l = L[q] * kLog2e;
                    next_d = Dl[q];
                }
                ok = mbar_wait(bar(LY::B_SDP), gb & 1, abort_flag, a.status, kWaitNs);
                if (!ok) break;
                if (gb > 0) {
                    // dS in shared memory is free once dQ of the previous block has completed
                    ok = mbar_wait(bar(LY::B_DQFULL), (gb - 1) & 1, abort_flag, a.status, kWaitNs);
                    if (!ok) break;
                }
                tc_fence_after();
                const bool edge = (i0 == item.j0) || (i0 + 128 > item.q_end) || (item.j1 - item.j0 < 128);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t sr[32], dr[32];
                    tmem_ld32(tmem + lane_addr + kColS + c * 32, sr);
                    tmem_ld32(tmem + lane_addr + kColDP + c * 32, dr);
                    tmem_ld_wait();
                    uint32_t pp[16], dd[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        float pv[2], dv[2];
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int ql = c * 32 + e + u;
                            float p = ex2(fmaf(__uint_as_float(sr[e + u]), sl2, -s_lse[ql]));
                            if (edge) {
                                const int q = i0 + ql;
                                const bool vis = key <= q && q < item.q_end && key < item.j1;
                                p = vis ? p : 0.f;
                            }
                            pv[u] = p;
                            dv[u] = p * (__uint_as_float(dr[e + u]) - s_dlt[ql]);
                        }
                        pp[e >> 1] = pack_bf16(pv[0], pv[1]);
                        dd[e >> 1] = pack_bf16(dv[0], dv[1]);
                    }
                    tmem_st16(tmem + lane_addr + kColS + c * 16, pp);
                    tmem_st16(tmem + lane_addr + kColDP + c * 16, dd);
                    // dS row (this key) for queries [32c, 32c+32): 4 chunks of 16 bytes, 128-byte swizzle
                    uint8_t* atom = ds_row + (c >> 1) * 16384;
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int chunk = (c & 1) * 4 + u;
                        uint4 v = make_uint4(dd[4 * u], dd[4 * u + 1], dd[4 * u + 2], dd[4 * u + 3]);
                        *reinterpret_cast<uint4*>(atom + ((chunk ^ (krow & 7)) << 4)) = v;
                    }
                    tmem_st_wait();
                    fence_proxy_async_smem();
                    tc_fence_before();
                    mbar_arrive(bar(LY::B_PCH + c));
                }
            }
            if (!ok) break;
            // epilogue: dK * scale, dV as bf16
            ok = mbar_wait(bar(LY::B_DKDVFULL), ic & 1, abort_flag, a.status, kWaitNs);
            if (!ok) break;
            tc_fence_after();
            const int b_ = bh / a.g.H, h_ = bh % a.g.H;
            const int64_t roff = (int64_t)b_ * a.g.sb + (int64_t)h_ * a.g.sh + (int64_t)key * a.g.st;
            const bool live = key < item.j1;
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                const uint32_t col = which == 0 ? kColDK : kColDV;
                const float mul = which == 0 ? a.g.scale : 1.f;
                __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(which == 0 ? a.dk : a.dv) + roff;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lane_addr + col + c * 32, r);
                    tmem_ld_wait();
                    if (live) {
                        uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            uint4 v;
                            v.x = pack_bf16(__uint_as_float(r[8 * u + 0]) * mul, __uint_as_float(r[8 * u + 1]) * mul);
                            v.y = pack_bf16(__uint_as_float(r[8 * u + 2]) * mul, __uint_as_float(r[8 * u + 3]) * mul);
                            v.z = pack_bf16(__uint_as_float(r[8 * u + 4]) * mul, __uint_as_float(r[8 * u + 5]) * mul);
                            v.w = pack_bf16(__uint_as_float(r[8 * u + 6]) * mul, __uint_as_float(r[8 * u + 7]) * mul);
                            d4[u] = v;
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(bar(LY::B_DKDVFREE));
        }
    } else if (warp >= 8) {
        // ------------------------------------------------------------ dQ drain
        const int qrow = tid - 256;
        const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
        uint32_t gb = 0;
        bool ok = true;
        for (int w = blockIdx.x; w < n_work && ok && !*abort_flag; w += gridDim.x) {
            int32_t it, bh;
            decode_work(w, a.n_items, BH, a.group, it, bh);
            const BwdItem item = a.items[it];
            const int nq = (item.q_end - item.j0 + 127) / 128;
            float* dQg = a.dq_acc + (int64_t)bh * a.g.T * D;
            for (int i = 0; i < nq; ++i, ++gb) {
                ok = mbar_wait(bar(LY::B_DQFULL), gb & 1, abort_flag, a.status, kWaitNs);
                if (!ok) break;
                tc_fence_after();
                const int q = item.j0 + (nq - 1 - i) * 128 + qrow;
                const bool live = q < item.q_end;
                float* dst = dQg + (int64_t)q * D;
                // copy the dQ row out of TMEM, release the columns at once, then
                // send the reductions: the next block's dP^T can start while the
                // fp32 adds drain through L2
                uint32_t r[D / 32][32];
#pragma unroll
                for (int c = 0; c < D / 32; ++c) tmem_ld32(tmem + lane_addr + kColDP + c * 32, r[c]);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(bar(LY::B_DQFREE));
                if (live) {
#pragma unroll
                    for (int c = 0; c < D / 32; ++c)
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            float4 v = make_float4(__uint_as_float(r[c][4 * u]) * a.g.scale,
                                                   __uint_as_float(r[c][4 * u + 1]) * a.g.scale,
                                                   __uint_as_float(r[c][4 * u + 2]) * a.g.scale,
                                                   __uint_as_float(r[c][4 * u + 3]) * a.g.scale);
                            atomicAdd(reinterpret_cast<float4*>(dst + c * 32 + 4 * u), v);
                        }
                }
            }
        }
    }
    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        if (*abort_flag) {
            if (elect_one()) {
                mma_commit(bar(LY::B_DRAIN));
                const uint64_t t0 = globaltimer();
                while (!mbar_try_wait(bar(LY::B_DRAIN), 0) && globaltimer() - t0 < kWaitNs) {
                }
            }
            __syncwarp();
        }
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D>
cudaError_t launch_d(const BwdArgs& a, cudaStream_t s) {
    CUtensorMap mq, mk, mv, mdo;
    TcMaps mp{1, 2, 3};
    if (!make_tile_map(&mq, a.q, a.g, mp) || !make_tile_map(&mk, a.k, a.g, mp) || !make_tile_map(&mv, a.v, a.g, mp) ||
        !make_tile_map(&mdo, a.dout, a.g, mp))
        return cudaErrorInvalidValue;
    const int64_t work = (int64_t)a.n_items * a.g.B * a.g.H;
    if (work <= 0) return cudaSuccess;
    if (work > INT32_MAX) return cudaErrorInvalidValue;
    const size_t smem = BwdTcLayout<D>::ALLOC;
    cudaError_t e = cudaFuncSetAttribute(bwd_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int grid = (int)std::min<int64_t>(work, device_sm_count());
    bwd_tc_kernel<D><<<grid, BT_THREADS, smem, s>>>(mq, mk, mv, mdo, a, mp, (int32_t)work);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_tiles_tc(const BwdArgs& a, cudaStream_t s) {
    return a.g.D == 128 ? launch_d<128>(a, s) : launch_d<64>(a, s);
}

}  // namespace attn
