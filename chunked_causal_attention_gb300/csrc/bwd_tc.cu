// Backward key-tile kernel on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// One work item = 128 keys [j0, j1) of one (batch, head); the item walks the
// query blocks of 128 rows [q_lo, q_end) that can see those keys from the last
// block down to the first: a key's dK/dV collect the contributions of every
// later token of its sequence (InfiniPipe §II-A: K/V gradients of a token
// depend on all subsequent tokens). For the whole backward q_lo = j0 and q_end
// is the document end; for the backward of one chunk the queries are that
// chunk's rows, and dK/dV are added into fp32 accumulators that the chunks of a
// document share when run in reverse order. Persistent CTAs take items
// head-major (all CTAs on one head at a time), so the head's Q/dO tiles and
// dQ accumulator rows are reused from L2. With grouped key/value heads (GQA/MQA)
// an item is a key tile of one key/value head and walks the query blocks of
// each of its H / Hkv query heads in turn, so dK/dV collect the group's sum.
// The tiles are D = 64 or 128 dims wide; a head dim below D loads its
// remaining dims as zeros and only its own dims are written (PAD).
//
// Warp roles (16 warps):
//   warp 0       TMA producer: K, V once per item; Q and dO of a query block into
//                one 2-tile stage of a two-stage ring.
//   warp 1       MMA issuer (one thread) and TMEM owner. Per query block:
//                  S^T  = K Q^T     -> TMEM [0,128)      (SS, both K-major)
//                  dP^T = V dO^T    -> TMEM [128,256)    (SS, both K-major)
//                  dV  += P^T dO    -> TMEM [256,256+D)  (A = P^T in TMEM, B = dO MN-major)
//                  dK  += dS^T Q    -> TMEM dK           (A = dS^T in TMEM, B = Q MN-major)
//                  dQ   = dS K      -> TMEM [128,128+D)  (A = dS MN-major in shared memory,
//                                                         B = K MN-major)
//   warps 4-7    softmax gradient for query columns [0,64), one key row per thread
//   warps 8-11   softmax gradient for query columns [64,128):
//                  P^T  = 2^(S^T * scale*log2 e - LSE_t*log2 e)   (zero where t < key or t >= end)
//                  dS^T = P^T o (dP^T - D_t)
//                P^T and dS^T of a 32-column chunk go back into that chunk's own
//                TMEM columns as bf16 (A operands of dV, dK); dS also goes to
//                shared memory for dQ. The MMA thread consumes chunks as they
//                are released. At the end of the item warps 4-7 write dK*scale
//                and warps 8-11 write dV; in the chunk-streamed backward a tile
//                whose keys are all context adds them into the fp32 accumulators
//                by TMA reduce-adds staged through the dS buffer.
//   warps 12-15  dQ drain, one query row per thread: dQ*scale from TMEM into the
//                block's Q/dO stage (free once the block's MMAs are done; the
//                fp32 tile is exactly its size), then one thread issues TMA
//                reduce-adds into the fp32 accumulator and hands the stage back
//                to the producer once the TMA engine has read it.
// Every mbarrier wait is bounded (ATTN_E_TIMEOUT in the status word). The
// warps of a group that meets at named barriers leave their loop only
// together, by a vote taken at one of those barriers (bar.red), so a wait
// that gives up in one warp cannot leave the others waiting for it. Every
// role checks each work item against the geometry before using it
// (ATTN_E_BOUNDS; all roles read the same item and decide alike).
#include "tc_common.cuh"

namespace attn {
namespace {

using namespace tc;

constexpr int BT_THREADS = 512;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;
constexpr uint32_t kColDP = 128;
constexpr uint32_t kColDV = 256;

template <int D>
struct BwdTcLayout {
    static constexpr int TILE = 128 * D * 2;           // one 128-row bf16 tile
    static constexpr int STAGE = 2 * TILE;             // Q + dO of a block; also the fp32 dQ staging
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = K_OFF + TILE;
    static constexpr int QDO_OFF = V_OFF + TILE;       // 2 stages
    static constexpr int DS_OFF = QDO_OFF + 2 * STAGE; // 128 keys x 128 queries bf16, MN-major
    static constexpr int NL_OFF = DS_OFF + 32768;      // 128 floats: -LSE_t * log2 e
    static constexpr int ND_OFF = NL_OFF + 512;        // 128 floats: -D_t
    static constexpr int BAR_OFF = ND_OFF + 512;
    static constexpr int B_KVFULL = 0, B_KVEMPTY = 1;
    static constexpr int B_QFULL = 2, B_QEMPTY = 4;    // 2 each
    static constexpr int B_SDP = 6, B_PCH = 7;         // B_PCH + c: P^T/dS^T of query chunk c ready
    static constexpr int B_DQFULL = 11, B_DQFREE = 12;
    static constexpr int B_DKDVFULL = 13, B_DKDVFREE = 14, B_DRAIN = 15;
    static constexpr int B_RFULL = 16, B_REMPTY = 18;  // work ring: 2 slots each
    static constexpr int NBAR = 20;
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
    // coordinates of map axes 1..3 (token, head, batch in stride order), by selects
    const int c1 = mp.pos_t == 1 ? row : (mp.pos_h == 1 ? h : b);
    const int c2 = mp.pos_t == 2 ? row : (mp.pos_h == 2 ? h : b);
    const int c3 = mp.pos_t == 3 ? row : (mp.pos_h == 3 ? h : b);
#pragma unroll
    for (int a = 0; a < D / 64; ++a) tma_load_4d(dst + a * 16384, map, bar, a * 64, c1, c2, c3);
}

// Softmax gradient of one query block for one warpgroup (query columns
// [64*grp, 64*grp+64)) as four half-chunks of 16 columns; the TMEM loads of the
// next half-chunk are in flight while the current one is computed. EDGE adds
// the causal/document/ragged-tile mask (diagonal block, partial last block,
// last key tile of a document); interior blocks skip it.
template <bool EDGE>
__device__ __forceinline__ void sg_block(uint32_t tm, int grp, int krow, int key, int i0, const BwdItem& item,
                                         const float* s_nl, const float* s_nd, uint8_t* ds_row, float2 sl2x2,
                                         uint32_t bar_pch) {
    uint32_t sr[2][16], dr[2][16];
    tmem_ld16(tm + kColS + grp * 64, sr[0]);
    tmem_ld16(tm + kColDP + grp * 64, dr[0]);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int h = k >> 1, hf = k & 1;
        const int c = 2 * grp + h;
        const int col = c * 32 + hf * 16;
        const int b = k & 1;
        tmem_ld_wait();
        if (k + 1 < 4) {
            const int ncol = (2 * grp + ((k + 1) >> 1)) * 32 + ((k + 1) & 1) * 16;
            tmem_ld16(tm + kColS + ncol, sr[b ^ 1]);
            tmem_ld16(tm + kColDP + ncol, dr[b ^ 1]);
        }
        // this half-chunk's 16 values of -LSE*log2e (lanes 0-15) and of -D (lanes
        // 16-31), one per lane from one load per warp, then to every lane by shuffles
        const int ln = threadIdx.x & 31;
        const float mine = ln < 16 ? s_nl[col + ln] : s_nd[col + ln - 16];
        uint32_t pp[8], dd[8];
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4) {
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int e = 4 * e4 + 2 * u;
                const float2 nl = make_float2(__shfl_sync(0xffffffffu, mine, e), __shfl_sync(0xffffffffu, mine, e + 1));
                const float2 nd = make_float2(__shfl_sync(0xffffffffu, mine, 16 + e),
                                              __shfl_sync(0xffffffffu, mine, 17 + e));
                const float2 x = ffma2(make_float2(__uint_as_float(sr[b][e]), __uint_as_float(sr[b][e + 1])), sl2x2, nl);
                float p0 = ex2(x.x), p1 = ex2(x.y);
                if (EDGE) {
                    const int q = i0 + col + e;
                    const bool key_ok = key < item.j1;
                    p0 = (key_ok && key <= q && q < item.q_end) ? p0 : 0.f;
                    p1 = (key_ok && key <= q + 1 && q + 1 < item.q_end) ? p1 : 0.f;
                }
                const float2 dpv = fadd2(make_float2(__uint_as_float(dr[b][e]), __uint_as_float(dr[b][e + 1])), nd);
                const float2 ds = fmul2(make_float2(p0, p1), dpv);
                pp[e >> 1] = pack_bf16(p0, p1);
                dd[e >> 1] = pack_bf16(ds.x, ds.y);
            }
        }
        // P^T and dS^T (8 columns per half) into the first 16 columns of this
        // chunk's own S^T / dP^T columns
        tmem_st8(tm + kColS + c * 32 + hf * 8, pp);
        tmem_st8(tm + kColDP + c * 32 + hf * 8, dd);
        // dS row (this key) for these 16 queries: 2 chunks of 16 bytes, 128-byte swizzle
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int chunk = h * 4 + hf * 2 + u;
            uint4 v = make_uint4(dd[4 * u], dd[4 * u + 1], dd[4 * u + 2], dd[4 * u + 3]);
            *reinterpret_cast<uint4*>(ds_row + ((chunk ^ (krow & 7)) << 4)) = v;
        }
        if (hf == 1) {
            tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar_pch + 8u * (uint32_t)c);
        }
    }
}

// TMA maps of the fp32 dK/dV accumulators, a kernel parameter only in the
// chunk-streamed instantiations.
template <bool ACC>
struct AccMaps {};
template <>
struct AccMaps<true> {
    CUtensorMap dk, dv;
};

// GROUPED: key/value heads shared by several query heads. The ungrouped
// instantiation has G = 1 at compile time, which keeps the per-block walk of
// the softmax-gradient warps as light as it was before grouping existed.
// PAD: the head dim is below the tile width D (its dims past it load as zeros
// and are not written); the unpadded instantiations keep every write bound at
// compile time. ACC: the chunk-streamed backward (fp32 dK/dV accumulators); the
// whole backward is compiled without its epilogue paths.
template <int D, bool GROUPED, bool PAD, bool ACC>
__global__ void __launch_bounds__(BT_THREADS, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo,
                  const __grid_constant__ CUtensorMap tmdq, const __grid_constant__ AccMaps<ACC> am,
                  const BwdArgs a, const TcMaps mp, const TcMaps mpkv, const int32_t n_work) {
    using LY = BwdTcLayout<D>;
    // every item comes from the work queue (see WorkRing); its consumers are the
    // MMA thread, the 8 softmax-gradient warps and the 4 drain warps
    constexpr uint32_t kColDK = kColDV + D;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);
    const uint32_t bar0 = sbase + LY::BAR_OFF;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + LY::MISC_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + LY::MISC_OFF + 4);
    float* s_nl = reinterpret_cast<float*>(sm + LY::NL_OFF);
    float* s_nd = reinterpret_cast<float*>(sm + LY::ND_OFF);
    const WorkRing ring{reinterpret_cast<volatile int32_t*>(sm + LY::MISC_OFF + 8), bar(LY::B_RFULL),
                        bar(LY::B_REMPTY)};

    const int tid = threadIdx.x, warp = tid >> 5;
    const int BHKV = a.g.B * a.g.Hkv;            // work items run over (key tile, batch, key/value head)
    const int G = GROUPED ? a.g.H / a.g.Hkv : 1;  // query heads per key/value head

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
        mbar_init(bar(LY::B_DKDVFREE), 256);
        mbar_init(bar(LY::B_DRAIN), 1);
        for (int r = 0; r < 2; ++r) {
            mbar_init(bar(LY::B_RFULL + r), 1);
            mbar_init(bar(LY::B_REMPTY + r), 13);      // MMA thread, 8 + 4 consumer warps
        }
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
            int32_t w = a.stall ? n_work : (int32_t)atomicAdd(a.counter, 1u);
            for (; !a.stall && ok; ++ic) {
                // publish the item (or the end of the work) to the consumers
                ok = ring_put(ring, ic, w < n_work ? w : -1, abort_flag, a.status, a.wait_ns);
                if (!ok || w >= n_work || *abort_flag) break;
                int32_t it, bkv;
                decode_work(w, a.n_items, BHKV, a.group, it, bkv);
                const BwdItem item = a.items[it];
                if (!bwd_item_ok(item, a.g.T, a.rows)) {
                    set_error(a.status, ATTN_E_BOUNDS);
                    *abort_flag = 1;
                    break;
                }
                int32_t w_next = n_work;
                const int b = bkv / a.g.Hkv, hk = bkv % a.g.Hkv;
                ok = mbar_wait(bar(LY::B_KVEMPTY), (ic & 1) ^ 1, abort_flag, a.status, a.wait_ns);
                if (!ok) break;
                mbar_expect_tx(bar(LY::B_KVFULL), 2 * LY::TILE);
                load_tile_b<D>(sbase + LY::K_OFF, &tmk, bar(LY::B_KVFULL), mpkv, item.j0, hk, b);
                load_tile_b<D>(sbase + LY::V_OFF, &tmv, bar(LY::B_KVFULL), mpkv, item.j0, hk, b);
                const int nq = (item.q_end - item.q_lo + 127) / 128;
                for (int blk = 0; blk < G * nq; ++blk, ++qc) {
                    const int g = blk / nq, i = blk - g * nq;
                    const uint32_t s = qc & 1;
                    ok = mbar_wait(bar(LY::B_QEMPTY + s), ((qc >> 1) & 1) ^ 1, abort_flag, a.status, a.wait_ns);
                    if (!ok) break;
                    mbar_expect_tx(bar(LY::B_QFULL + s), LY::STAGE);
                    const int row = item.q_lo + (nq - 1 - i) * 128;
                    const uint32_t st = sbase + LY::QDO_OFF + s * LY::STAGE;
                    load_tile_b<D>(st, &tmq, bar(LY::B_QFULL + s), mp, row, hk * G + g, b);
                    load_tile_b<D>(st + LY::TILE, &tmdo, bar(LY::B_QFULL + s), mp, row, hk * G + g, b);
                    // the item's last loads are out: claim the next item now, about two
                    // blocks before this CTA is free for it
                    if (blk == G * nq - 1) w_next = (int32_t)atomicAdd(a.counter, 1u);
                }
                w = w_next;
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
            for (; ok; ++ic) {
                int32_t w = -1;
                ok = ring_get(ring, ic, w, abort_flag, a.status, a.wait_ns);
                if (!ok || w < 0 || *abort_flag) break;
                int32_t it, bkv;
                decode_work(w, a.n_items, BHKV, a.group, it, bkv);
                const BwdItem item = a.items[it];
                if (!bwd_item_ok(item, a.g.T, a.rows)) {
                    set_error(a.status, ATTN_E_BOUNDS);
                    *abort_flag = 1;
                    break;
                }
                const int nq = (item.q_end - item.q_lo + 127) / 128;
                ok = mbar_wait(bar(LY::B_KVFULL), ic & 1, abort_flag, a.status, a.wait_ns);
                if (!ok) break;
                tc_fence_after();
                for (int blk = 0; blk < G * nq; ++blk, ++qc, ++gb) {
                    const uint32_t s = qc & 1;
                    ok = mbar_wait(bar(LY::B_QFULL + s), (qc >> 1) & 1, abort_flag, a.status, a.wait_ns);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t q0 = sbase + LY::QDO_OFF + s * LY::STAGE;
                    const uint32_t o0 = q0 + LY::TILE;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                        mma_ss(tmem + kColS, sdesc_sw128(k0 + off, 16, 1024), sdesc_sw128(q0 + off, 16, 1024), id_s,
                               kk > 0);
                    }
                    if (gb > 0) {
                        ok = mbar_wait(bar(LY::B_DQFREE), (gb - 1) & 1, abort_flag, a.status, a.wait_ns);
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
                    if (blk == 0) {
                        ok = mbar_wait(bar(LY::B_DKDVFREE), (ic & 1) ^ 1, abort_flag, a.status, a.wait_ns);
                        if (!ok) break;
                    }
                    // dV += P^T dO and dK += dS^T Q one 32-query chunk (two k-steps) at a
                    // time, in the order the two softmax-gradient groups release them
                    for (int n = 0; n < 4 && ok; ++n) {
                        const int c = (n & 1) * 2 + (n >> 1);     // 0, 2, 1, 3
                        ok = mbar_wait(bar(LY::B_PCH + c), gb & 1, abort_flag, a.status, a.wait_ns);
                        if (!ok) break;
                        tc_fence_after();
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int kk = 2 * c + h;
                            const uint32_t acc = (blk > 0 || n > 0 || h > 0) ? 1u : 0u;
                            mma_ts(tmem + kColDV, tmem + kColS + 32 * c + 8 * h,
                                   sdesc_sw128(o0 + kk * 2048, 16384, 1024), id_g, acc);
                            mma_ts(tmem + kColDK, tmem + kColDP + 32 * c + 8 * h,
                                   sdesc_sw128(q0 + kk * 2048, 16384, 1024), id_g, acc);
                        }
                    }
                    if (!ok) break;
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
    } else if (warp >= 4 && warp < 12) {
        // ------------------------------------------------------------ softmax gradient + dK/dV epilogue
        const int grp = (warp - 4) >> 2;                 // 0: query columns [0,64), 1: [64,128)
        const int krow = tid - 128 - 128 * grp;          // TMEM lane == key row
        const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
        const float sl2 = a.g.scale * kLog2e;
        const float2 sl2x2 = make_float2(sl2, sl2);
        uint32_t gb = 0, ic = 0;
        bool ok = true;
        uint8_t* ds_row = sm + LY::DS_OFF + grp * 16384 + krow * 128;
        // this thread stages one value per block: -LSE*log2e (krow < 64) or -D_t of
        // query 64*grp + (krow & 63), fetched one block ahead
        const bool stage_l = krow < 64;
        float* stage_dst = (stage_l ? s_nl : s_nd) + 64 * grp + (krow & 63);
        // The two groups synchronise on named barriers, so a thread never leaves
        // the loop on its own: `ok` changes only through a group vote
        // (named_sync_all), which every thread of the group reaches, and the item
        // check gives the same answer in every thread.
        for (; ok; ++ic) {
            // the next item: every warp reads it, and the group goes on only if all did
            int32_t w = -1;
            const bool got = ring_get_warp(ring, ic, w, abort_flag, a.status, a.wait_ns);
            if (!named_sync_all(1 + grp, 128, got && !*abort_flag)) {
                ok = false;
                break;
            }
            if (w < 0) break;                            // no more work (the same w in every thread)
            int32_t it, bkv;
            decode_work(w, a.n_items, BHKV, a.group, it, bkv);
            const BwdItem item = a.items[it];
            if (!bwd_item_ok(item, a.g.T, a.rows)) {
                set_error(a.status, ATTN_E_BOUNDS);
                *abort_flag = 1;
                break;
            }
            const int b = bkv / a.g.Hkv, hk = bkv % a.g.Hkv;
            const int nq = (item.q_end - item.q_lo + 127) / 128;
            const int key = item.j0 + krow;
            // src[t] for a token t of query head hk*G + g: LSE (all tokens) or delta
            // (workspace row t + row_off)
            auto src_of = [&](int g) -> const float* {
                const int64_t bhq = (int64_t)b * a.g.H + hk * G + g;
                return stage_l ? a.lse + bhq * a.g.T : a.delta + bhq * a.rows + item.row_off;
            };
            const float* src = src_of(0);
            const int qoff = 64 * grp + (krow & 63);      // the block row this thread stages
            const float mul = stage_l ? -kLog2e : -1.f;
            // raw value of the next block, scaled only when it is staged, so the
            // load's latency is not waited for until then
            float next = 0.f;
            {
                const int q = item.q_lo + (nq - 1) * 128 + qoff;
                if (q < item.q_end) next = src[q];
            }
            int i = 0, g = 0;                              // the block: query head hk*G + g, i-th from the top
            for (int blk = 0; blk < G * nq; ++blk, ++gb) {
                const int i0 = item.q_lo + (nq - 1 - i) * 128;  // query blocks walked from the last one down
                // the first of the block's two barriers carries the group's vote: go on
                // only if every wait of the previous block succeeded in every thread and
                // no thread has seen the abort flag
                if (!named_sync_all(1 + grp, 128, ok && !*abort_flag)) {
                    ok = false;
                    break;
                }
                *stage_dst = next * mul;
                named_sync(1 + grp, 128);
                if (i + 1 < nq) {
                    next = src[i0 - 128 + qoff];           // the next block down, same query head
                } else if (g + 1 < G) {
                    src = src_of(g + 1);                   // the top block of the group's next query head
                    const int q = item.q_lo + (nq - 1) * 128 + qoff;
                    next = q < item.q_end ? src[q] : 0.f;
                }
                // a failed wait skips the block's work (the warp-collective TMEM loads
                // and stores run in all lanes of a warp or in none); the group leaves at
                // the next vote
                ok = mbar_wait_warp(bar(LY::B_SDP), gb & 1, abort_flag, a.status, a.wait_ns);
                // dS in shared memory is free once dQ of the previous block has completed
                if (ok && gb > 0) ok = mbar_wait_warp(bar(LY::B_DQFULL), (gb - 1) & 1, abort_flag, a.status, a.wait_ns);
                if (ok) {
                    tc_fence_after();
                    // masks are needed where some key of the tile lies after some query of
                    // the block, where the block runs past the document or chunk end, and
                    // on a partial key tile
                    const bool edge = (i0 < item.j1 - 1) || (i0 + 128 > item.q_end) || (item.j1 - item.j0 < 128);
                    if (edge)
                        sg_block<true>(tmem + lane_addr, grp, krow, key, i0, item, s_nl, s_nd, ds_row, sl2x2,
                                       bar(LY::B_PCH));
                    else
                        sg_block<false>(tmem + lane_addr, grp, krow, key, i0, item, s_nl, s_nd, ds_row, sl2x2,
                                        bar(LY::B_PCH));
                }
                if (++i == nq) {
                    i = 0;
                    ++g;
                }
            }
            // epilogue: warps 4-7 write dK * scale, warps 8-11 write dV (bf16); the
            // group enters it only together (the streamed epilogue has barriers)
            if (ok) ok = mbar_wait_warp(bar(LY::B_DKDVFULL), ic & 1, abort_flag, a.status, a.wait_ns);
            if (!named_sync_all(1 + grp, 128, ok && !*abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int64_t roff = (int64_t)b * a.g.sb_kv + (int64_t)hk * a.g.sh_kv + (int64_t)key * a.g.st_kv;
            const bool live = key < item.j1;
            const uint32_t col = grp == 0 ? kColDK : kColDV;
            const float gmul = grp == 0 ? a.g.scale : 1.f;
            __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(grp == 0 ? a.dk : a.dv) + roff;
            // chunk-streamed backward: add into the fp32 accumulator row, and write
            // bf16 only for the chunk's own keys (complete once their chunk has run)
            float* acc = ACC ? (grp == 0 ? a.dk_acc : a.dv_acc) + roff : nullptr;
            const bool emit = acc == nullptr || key >= item.emit_from;
            const int Dv = PAD ? a.g.D : D;        // dims written (the tile's dims past the head dim are zero)
            if (ACC && item.emit_from >= item.j1) {
                // Every key of this tile is context of the call's rows, so only the fp32
                // accumulators change: stage 32 columns at a time in this group's half of
                // the dS buffer (free until this group's next softmax gradient) and add
                // them with a TMA reduce-add; the TMA unit does the read-modify-write in
                // L2. Rows past the tile's last key hold zeros (their P and dS are zero).
                uint8_t* stg_row = sm + LY::DS_OFF + grp * 16384 + krow * 128;
                const uint32_t stg = sbase + LY::DS_OFF + grp * 16384;
                const CUtensorMap* amap = nullptr;
                if constexpr (ACC) amap = grp == 0 ? &am.dk : &am.dv;
                const int c1 = mpkv.pos_t == 1 ? item.j0 : (mpkv.pos_h == 1 ? hk : b);
                const int c2 = mpkv.pos_t == 2 ? item.j0 : (mpkv.pos_h == 2 ? hk : b);
                const int c3 = mpkv.pos_t == 3 ? item.j0 : (mpkv.pos_h == 3 ? hk : b);
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    if (PAD && c * 32 >= Dv) break;    // the same for every thread of the group
                    uint32_t r[32];
                    tmem_ld32(tmem + lane_addr + col + c * 32, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const float4 v = live ? make_float4(__uint_as_float(r[4 * u]) * gmul,
                                                            __uint_as_float(r[4 * u + 1]) * gmul,
                                                            __uint_as_float(r[4 * u + 2]) * gmul,
                                                            __uint_as_float(r[4 * u + 3]) * gmul)
                                              : make_float4(0.f, 0.f, 0.f, 0.f);
                        *reinterpret_cast<float4*>(stg_row + ((u ^ (krow & 7)) << 4)) = v;
                    }
                    fence_proxy_async_smem();
                    named_sync(1 + grp, 128);
                    if (krow == 0) {
                        tma_reduce_add_4d(amap, stg, c * 32, c1, c2, c3);
                        bulk_commit();
                        bulk_wait_read_all();
                    }
                    named_sync(1 + grp, 128);          // the staging may be rewritten
                }
                tc_fence_before();
                mbar_arrive(bar(LY::B_DKDVFREE));
                continue;
            }
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_addr + col + c * 32, r);
                tmem_ld_wait();
                if (live) {
                    float f[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(r[e]) * gmul;
                    if (acc) {
                        float4* a4 = reinterpret_cast<float4*>(acc + c * 32);
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            if (c * 32 + u * 4 >= Dv) break;
                            float4 x = a4[u];
                            x.x += f[4 * u]; x.y += f[4 * u + 1]; x.z += f[4 * u + 2]; x.w += f[4 * u + 3];
                            a4[u] = x;
                            f[4 * u] = x.x; f[4 * u + 1] = x.y; f[4 * u + 2] = x.z; f[4 * u + 3] = x.w;
                        }
                    }
                    if (emit) {
                        uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            if (c * 32 + u * 8 >= Dv) break;
                            uint4 v;
                            v.x = pack_bf16(f[8 * u + 0], f[8 * u + 1]);
                            v.y = pack_bf16(f[8 * u + 2], f[8 * u + 3]);
                            v.z = pack_bf16(f[8 * u + 4], f[8 * u + 5]);
                            v.w = pack_bf16(f[8 * u + 6], f[8 * u + 7]);
                            d4[u] = v;
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(bar(LY::B_DKDVFREE));
        }
        if (ACC && krow == 0) bulk_wait_all();          // accumulator reduce-adds complete
    } else if (warp >= 12) {
        // ------------------------------------------------------------ dQ drain
        const int qrow = tid - 384;
        const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
        const float sc = a.g.scale;
        uint32_t gb = 0;
        bool ok = true;
        // as in the softmax-gradient groups, the four warps leave only together,
        // by the vote at their barrier (`ok` is the same in every thread)
        for (uint32_t ic = 0; ok; ++ic) {
            // the next item: every warp reads it, and the group goes on only if all did
            int32_t w = -1;
            const bool got = ring_get_warp(ring, ic, w, abort_flag, a.status, a.wait_ns);
            if (!named_sync_all(3, 128, got && !*abort_flag)) {
                ok = false;
                break;
            }
            if (w < 0) break;                            // no more work (the same w in every thread)
            int32_t it, bkv;
            decode_work(w, a.n_items, BHKV, a.group, it, bkv);
            const BwdItem item = a.items[it];
            if (!bwd_item_ok(item, a.g.T, a.rows)) {
                set_error(a.status, ATTN_E_BOUNDS);
                *abort_flag = 1;
                break;
            }
            const int b = bkv / a.g.Hkv, hk = bkv % a.g.Hkv;
            const int nq = (item.q_end - item.q_lo + 127) / 128;
            int i = 0, bhq = b * a.g.H + hk * G;             // the block's index and query head (dQ rows)
            for (int blk = 0; blk < G * nq; ++blk, ++gb) {
                const int i0 = item.q_lo + (nq - 1 - i) * 128;
                const uint32_t s = gb & 1;                   // the stage this block's Q/dO used
                uint8_t* stage = sm + LY::QDO_OFF + s * LY::STAGE;
                ok = mbar_wait_warp(bar(LY::B_DQFULL), gb & 1, abort_flag, a.status, a.wait_ns);
                if (ok) {
                    tc_fence_after();
                    // TMEM -> registers -> staging (fp32, 128-byte swizzled sub-tiles of 32
                    // columns), one sub-tile at a time; the TMEM columns are released after
                    // the last load
#pragma unroll
                    for (int cc = 0; cc < D / 32; ++cc) {
                        uint32_t r[32];
                        tmem_ld32(tmem + lane_addr + kColDP + cc * 32, r);
                        tmem_ld_wait();
                        if (cc == D / 32 - 1) {
                            tc_fence_before();
                            mbar_arrive(bar(LY::B_DQFREE));      // TMEM columns free for the next dP^T
                        }
                        uint8_t* sub = stage + cc * 16384 + qrow * 128;
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            float4 v = make_float4(__uint_as_float(r[4 * u]) * sc, __uint_as_float(r[4 * u + 1]) * sc,
                                                   __uint_as_float(r[4 * u + 2]) * sc, __uint_as_float(r[4 * u + 3]) * sc);
                            *reinterpret_cast<float4*>(sub + ((u ^ (qrow & 7)) << 4)) = v;
                        }
                    }
                    fence_proxy_async_smem();
                }
                if (!named_sync_all(3, 128, ok && !*abort_flag)) {
                    ok = false;
                    break;
                }
                if (qrow == 0) {
                    const uint32_t st = sbase + LY::QDO_OFF + s * LY::STAGE;
                    // 32-column boxes that start past the head dim hold only the zero
                    // dims of the tile; a box that runs past it is clipped by the TMA unit
#pragma unroll
                    for (int cc = 0; cc < D / 32; ++cc)
                        if (!PAD || cc * 32 < a.g.D)
                            tma_reduce_add_3d(&tmdq, st + cc * 16384, cc * 32, i0 + item.row_off, bhq);
                    bulk_commit();
                    bulk_wait_read_all();
                    mbar_arrive(bar(LY::B_QEMPTY + s));      // the producer may refill this stage
                }
                if (++i == nq) {
                    i = 0;
                    ++bhq;
                }
            }
        }
        if (qrow == 0) bulk_wait_all();
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
                while (!mbar_try_wait(bar(LY::B_DRAIN), 0) && globaltimer() - t0 < a.wait_ns) {
                }
            }
            __syncwarp();
        }
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D, bool GROUPED, bool PAD, bool ACC>
cudaError_t launch_d(const BwdArgs& a, cudaStream_t s) {
    CUtensorMap mq, mk, mv, mdo, mdq;
    TcMaps mp{1, 2, 3}, mpkv{1, 2, 3};
    const Geom gkv = a.g.kv();
    if (!make_tile_map(&mq, a.q, a.g, mp) || !make_tile_map(&mk, a.k, gkv, mpkv) ||
        !make_tile_map(&mv, a.v, gkv, mpkv) || !make_tile_map(&mdo, a.dout, a.g, mp) ||
        !make_dq_acc_map(&mdq, a.dq_acc, a.g, a.rows))
        return cudaErrorInvalidValue;
    // fp32 dK/dV accumulators of the chunk-streamed backward (unused otherwise);
    // they have the key/value strides, so their axis order is that of mpkv
    AccMaps<ACC> am;
    if constexpr (ACC) {
        TcMaps mpa{1, 2, 3};
        if (!make_kv_acc_map(&am.dk, a.dk_acc, gkv, mpa) || !make_kv_acc_map(&am.dv, a.dv_acc, gkv, mpa) ||
            mpa.pos_t != mpkv.pos_t || mpa.pos_h != mpkv.pos_h)
            return cudaErrorInvalidValue;
    }
    const int64_t work = (int64_t)a.n_items * a.g.B * a.g.Hkv;
    if (work <= 0) return cudaSuccess;
    if (work > INT32_MAX) return cudaErrorInvalidValue;
    const size_t smem = BwdTcLayout<D>::ALLOC;
    cudaError_t e =
        cudaFuncSetAttribute(bwd_tc_kernel<D, GROUPED, PAD, ACC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    const int grid = (int)std::min<int64_t>(work, device_sm_count());
    bwd_tc_kernel<D, GROUPED, PAD, ACC><<<grid, BT_THREADS, smem, s>>>(mq, mk, mv, mdo, mdq, am, a, mp, mpkv,
                                                                        (int32_t)work);
    return counted(cudaGetLastError());
}

// Head dims up to 64 run on 64-wide tiles, the others on 128-wide tiles.
template <bool ACC>
cudaError_t launch_variant(const BwdArgs& a, cudaStream_t s) {
    const bool grouped = a.g.Hkv != a.g.H;
    if (a.g.D == 128) return grouped ? launch_d<128, true, false, ACC>(a, s) : launch_d<128, false, false, ACC>(a, s);
    if (a.g.D == 64) return grouped ? launch_d<64, true, false, ACC>(a, s) : launch_d<64, false, false, ACC>(a, s);
    if (a.g.D > 64) return grouped ? launch_d<128, true, true, ACC>(a, s) : launch_d<128, false, true, ACC>(a, s);
    return grouped ? launch_d<64, true, true, ACC>(a, s) : launch_d<64, false, true, ACC>(a, s);
}

}  // namespace

cudaError_t launch_bwd_tiles_tc(const BwdArgs& a, cudaStream_t s) {
    return a.dk_acc != nullptr ? launch_variant<true>(a, s) : launch_variant<false>(a, s);
}

}  // namespace attn
