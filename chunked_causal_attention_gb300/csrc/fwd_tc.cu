// Forward tile kernel on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Persistent CTAs walk the cost-sorted work list (128 query rows x one key
// range x one (batch, head)). The tiles are D = 64, 128 or 256 dims wide; a
// head dim below D loads its remaining dims as zeros (the TMA maps carry the
// true head dim) and only its own dims are written. Warp roles:
//   warp 0      TMA producer: Q tile once per item; K and V tiles of 128 keys
//               (64 at D = 256) through two- or three-stage rings (128-byte
//               swizzled, 64-column boxes),
//               from the key/value head of the item's query head (grouped
//               heads: h / (H / Hkv)).
//   warp 1      MMA issuer (one thread) and TMEM owner:
//                 S_j   = Q K_j^T        (both operands K-major in shared memory)
//                 O    += P_j V_j        (P_j from TMEM, V_j MN-major in shared memory)
//               S_{j+1} is issued before P_j V_j so the tensor core computes the
//               next scores while the softmax warps work on the current ones.
//   warps 4-7   softmax: one query row per thread (TMEM lane = row). Reads S_j
//               from TMEM, applies the causal/range mask on edge tiles, keeps
//               the running max m and sum l in base 2, writes P_j as bf16 into
//               the first half of S_j's columns, and writes O/l and LSE at the
//               end of the item.
// Online softmax (the exact form of the blockwise accumulation O = sum_i S_i V_i
// of Ring Self-Attention): the running max is only moved when a tile's max
// exceeds it by more than 2^8; then O and l are rescaled by 2^(m_old - m_new).
// Keeping a stale max below that threshold leaves every P <= 2^8, so fp32 and
// bf16 hold it, and the final O/l is unchanged.
//
// TMEM columns: S buffers at [0,128) and [128,256), O at [256, 256+D).
// Every mbarrier wait is bounded; a wait that gives up sets ATTN_E_TIMEOUT in
// the workspace status word and all roles leave their loops. The softmax
// warps take each wait's result for the whole warp (its TMEM loads and stores
// are warp-collective) and meet no named barrier, so each warp leaves on its
// own. Every role checks each work item against the geometry and the partial
// region before using it (ATTN_E_BOUNDS).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "tc_common.cuh"

namespace attn {
namespace {

using namespace tc;

constexpr int TC_THREADS = 256;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 256;
constexpr float kRescaleThreshold = 8.0f;      // log2 units

// Keys per K/V tile: 128, or 64 for the 256-wide head dims, whose Q tile (64 KB)
// and two-stage K and V rings (4 x 32 KB) then fit in shared memory (a Q tile
// and three-stage rings of 128-key tiles take 224 KB at D = 128), and whose
// two S buffers (2 x 64 columns) and O (256 columns) fit in TMEM.
template <int D>
constexpr int kBlockN = D > 128 ? 64 : 128;

// KVS: stages of the K and V rings: three for tiles up to 128 dims (the deeper
// ring hides more of the latency of K/V tiles from L2 or DRAM), two for the
// 256-wide tiles, whose shared memory holds no third stage.
template <int D, int KVS>
struct FwdTcLayout {
    static constexpr int BN = kBlockN<D>;
    static constexpr int KV_STAGES = KVS;
    static constexpr int TILE_Q = 128 * D * 2;          // bytes of the 128-row bf16 Q tile
    static constexpr int TILE_KV = BN * D * 2;          // bytes of one BN-row bf16 K or V tile
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = Q_OFF + TILE_Q;
    static constexpr int V_OFF = K_OFF + KV_STAGES * TILE_KV;
    static constexpr int BAR_OFF = V_OFF + KV_STAGES * TILE_KV;
    // barrier indices
    static constexpr int B_QFULL = 0, B_QEMPTY = 1;
    static constexpr int B_KFULL = 2, B_KEMPTY = B_KFULL + KV_STAGES;
    static constexpr int B_VFULL = B_KEMPTY + KV_STAGES, B_VEMPTY = B_VFULL + KV_STAGES;
    static constexpr int B_SFULL = B_VEMPTY + KV_STAGES;       // 2
    static constexpr int B_PFULL = B_SFULL + 2;                // 2
    static constexpr int B_ODONE = B_PFULL + 2;
    static constexpr int B_OFREE = B_ODONE + 1;
    static constexpr int B_OFULL = B_OFREE + 1;                // last PV of an item complete
    static constexpr int B_DRAIN = B_OFULL + 1;
    static constexpr int B_RFULL = B_DRAIN + 1, B_REMPTY = B_RFULL + 2;   // work ring: 2 slots each
    static constexpr int NBAR = B_REMPTY + 2;
    static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;        // tmem base (u32), abort flag (int), work ring (2 x i32)
    static constexpr int BYTES = MISC_OFF + 16;
    static constexpr size_t ALLOC = (size_t)BYTES + 1024;      // slack for 1024-byte alignment
};

// One tile of ROWS rows x D dims: D / 64 boxes of 64 dims (128 bytes, 128-byte
// swizzle) x ROWS rows, box a at dst + a * ROWS * 128.
template <int D, int ROWS>
__device__ __forceinline__ void load_tile(uint32_t dst, const CUtensorMap* map, uint32_t bar, const TcMaps& mp,
                                          int row, int h, int b) {
    // coordinates of map axes 1..3 (token, head, batch in stride order), by selects
    const int c1 = mp.pos_t == 1 ? row : (mp.pos_h == 1 ? h : b);
    const int c2 = mp.pos_t == 2 ? row : (mp.pos_h == 2 ? h : b);
    const int c3 = mp.pos_t == 3 ? row : (mp.pos_h == 3 ? h : b);
#pragma unroll
    for (int a = 0; a < D / 64; ++a) tma_load_4d(dst + a * ROWS * 128, map, bar, a * 64, c1, c2, c3);
}

template <int D, int KVS>
__global__ void __launch_bounds__(TC_THREADS, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv, const FwdArgs a, const TcMaps mp, const TcMaps mpkv,
                  const int32_t n_work) {
    using LY = FwdTcLayout<D, KVS>;
    constexpr int KV_STAGES = KVS;
    constexpr int BN = LY::BN;                  // keys per K/V tile and columns per S buffer
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);
    const uint32_t bar0 = sbase + LY::BAR_OFF;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + LY::MISC_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + LY::MISC_OFF + 4);
    // every item comes from the work queue (see WorkRing); its consumers are the
    // MMA thread and the 4 softmax warps
    const WorkRing ring{reinterpret_cast<volatile int32_t*>(sm + LY::MISC_OFF + 8), bar(LY::B_RFULL),
                        bar(LY::B_REMPTY)};

    const int tid = threadIdx.x, warp = tid >> 5;
    const int BH = a.g.B * a.g.H;

    if (tid == 0) {
        mbar_init(bar(LY::B_QFULL), 1);
        mbar_init(bar(LY::B_QEMPTY), 1);
        for (int s = 0; s < KV_STAGES; ++s) {
            mbar_init(bar(LY::B_KFULL + s), 1);
            mbar_init(bar(LY::B_KEMPTY + s), 1);
            mbar_init(bar(LY::B_VFULL + s), 1);
            mbar_init(bar(LY::B_VEMPTY + s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(LY::B_SFULL + s), 1);
            mbar_init(bar(LY::B_PFULL + s), 128);
        }
        mbar_init(bar(LY::B_ODONE), 1);
        mbar_init(bar(LY::B_OFREE), 128);
        mbar_init(bar(LY::B_OFULL), 1);
        mbar_init(bar(LY::B_DRAIN), 1);
        for (int r = 0; r < 2; ++r) {
            mbar_init(bar(LY::B_RFULL + r), 1);
            mbar_init(bar(LY::B_REMPTY + r), 5);       // MMA thread, 4 softmax warps
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
            uint32_t kc = 0, vc = 0, ic = 0;
            int32_t w = a.stall ? n_work : (int32_t)atomicAdd(a.counter, 1u);
            for (; !a.stall; ++ic) {
                // publish the item (or the end of the work) to the consumers
                if (!ring_put(ring, ic, w < n_work ? w : -1, abort_flag, a.status, a.wait_ns)) break;
                if (w >= n_work || *abort_flag) break;
                int32_t it, bh;
                decode_work(w, a.n_items, BH, a.group, it, bh);
                const FwdItem item = a.items[it];
                if (!fwd_item_ok(item, a.g.T, BH, a.g.D, a.part_floats)) {
                    set_error(a.status, ATTN_E_BOUNDS);
                    *abort_flag = 1;
                    break;
                }
                const int b = bh / a.g.H, h = bh % a.g.H;
                const int hk = h / (a.g.H / a.g.Hkv);
                if (!mbar_wait(bar(LY::B_QEMPTY), (ic & 1) ^ 1, abort_flag, a.status, a.wait_ns)) break;
                mbar_expect_tx(bar(LY::B_QFULL), LY::TILE_Q);
                load_tile<D, 128>(sbase + LY::Q_OFF, &tmq, bar(LY::B_QFULL), mp, item.r0, h, b);
                const int nblk = (item.kv_hi - item.kv_lo + BN - 1) / BN;
                bool ok = true;
                int32_t w_next = n_work;
                for (int j = 0; j < nblk && ok; ++j) {
                    const int row = item.kv_lo + j * BN;
                    const uint32_t ks = kc % KV_STAGES, vs = vc % KV_STAGES;
                    ok = mbar_wait(bar(LY::B_KEMPTY + ks), ((kc / KV_STAGES) & 1) ^ 1, abort_flag, a.status, a.wait_ns);
                    if (!ok) break;
                    mbar_expect_tx(bar(LY::B_KFULL + ks), LY::TILE_KV);
                    load_tile<D, BN>(sbase + LY::K_OFF + ks * LY::TILE_KV, &tmk, bar(LY::B_KFULL + ks), mpkv, row, hk, b);
                    ++kc;
                    ok = mbar_wait(bar(LY::B_VEMPTY + vs), ((vc / KV_STAGES) & 1) ^ 1, abort_flag, a.status, a.wait_ns);
                    if (!ok) break;
                    mbar_expect_tx(bar(LY::B_VFULL + vs), LY::TILE_KV);
                    load_tile<D, BN>(sbase + LY::V_OFF + vs * LY::TILE_KV, &tmv, bar(LY::B_VFULL + vs), mpkv, row, hk, b);
                    ++vc;
                    // the item's last loads are out: claim the next item now, a block or
                    // two before this CTA is free for it
                    if (j == nblk - 1) w_next = (int32_t)atomicAdd(a.counter, 1u);
                }
                if (!ok) break;
                w = w_next;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (elect_one()) {
            constexpr uint32_t id_s = idesc_bf16(128, BN, 0, 0);
            constexpr uint32_t id_o = idesc_bf16(128, D, 0, 1);
            uint32_t kc = 0, vc = 0, ic = 0, gt = 0;   // gt: global tile counter (S buffer, P, PV index)
            bool ok = true;
            for (; ok; ++ic) {
                int32_t w = -1;
                ok = ring_get(ring, ic, w, abort_flag, a.status, a.wait_ns);
                if (!ok || w < 0 || *abort_flag) break;
                int32_t it, bh;
                decode_work(w, a.n_items, BH, a.group, it, bh);
                const FwdItem item = a.items[it];
                if (!fwd_item_ok(item, a.g.T, BH, a.g.D, a.part_floats)) {
                    set_error(a.status, ATTN_E_BOUNDS);
                    *abort_flag = 1;
                    break;
                }
                const int nblk = (item.kv_hi - item.kv_lo + BN - 1) / BN;
                ok = mbar_wait(bar(LY::B_QFULL), ic & 1, abort_flag, a.status, a.wait_ns);
                if (!ok) break;
                tc_fence_after();
                const uint32_t q0 = sbase + LY::Q_OFF;
                uint32_t pv_vc = vc;                 // V stage of the pending PV
                for (int j = 0; j <= nblk && ok; ++j) {
                    if (j < nblk) {
                        // S_j = Q K_j^T into S buffer (gt + j) & 1
                        const uint32_t ks = kc % KV_STAGES;
                        ok = mbar_wait(bar(LY::B_KFULL + ks), (kc / KV_STAGES) & 1, abort_flag, a.status, a.wait_ns);
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t k0 = sbase + LY::K_OFF + ks * LY::TILE_KV;
                        const uint32_t sb = tmem + kColS + ((gt + j) & 1) * BN;
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            // k-step kk: box kk / 4 (64 dims), 32 bytes further per 16 dims
                            const uint32_t qoff = (kk >> 2) * (128 * 128) + (kk & 3) * 32;
                            const uint32_t koff = (kk >> 2) * (BN * 128) + (kk & 3) * 32;
                            mma_ss(sb, sdesc_sw128(q0 + qoff, 16, 1024), sdesc_sw128(k0 + koff, 16, 1024), id_s, kk > 0);
                        }
                        mma_commit(bar(LY::B_KEMPTY + ks));
                        mma_commit(bar(LY::B_SFULL + ((gt + j) & 1)));
                        ++kc;
                        if (j == nblk - 1) mma_commit(bar(LY::B_QEMPTY));
                    }
                    if (j >= 1) {
                        // O += P_{j-1} V_{j-1}
                        const uint32_t t = gt + j - 1;
                        const uint32_t pb = t & 1;
                        if (j == 1) {
                            ok = mbar_wait(bar(LY::B_OFREE), (ic & 1) ^ 1, abort_flag, a.status, a.wait_ns);
                            if (!ok) break;
                        }
                        ok = mbar_wait(bar(LY::B_PFULL + pb), (t >> 1) & 1, abort_flag, a.status, a.wait_ns);
                        if (!ok) break;
                        const uint32_t vs = pv_vc % KV_STAGES;
                        ok = mbar_wait(bar(LY::B_VFULL + vs), (pv_vc / KV_STAGES) & 1, abort_flag, a.status, a.wait_ns);
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t v0 = sbase + LY::V_OFF + vs * LY::TILE_KV;
                        const uint32_t pa = tmem + kColS + pb * BN;
#pragma unroll
                        for (int kk = 0; kk < BN / 16; ++kk)
                            mma_ts(tmem + kColO, pa + kk * 8, sdesc_sw128(v0 + kk * 2048, BN * 128, 1024), id_o,
                                   (j - 1 > 0 || kk > 0) ? 1u : 0u);
                        mma_commit(bar(LY::B_VEMPTY + vs));
                        mma_commit(bar(LY::B_ODONE));
                        if (j == nblk) mma_commit(bar(LY::B_OFULL));
                        ++pv_vc;
                    }
                }
                vc = pv_vc;
                gt += nblk;
            }
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax / epilogue
        const int row = tid - 128;                       // TMEM lane == tile row
        const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
        const float sl2 = a.g.scale * kLog2e;
        uint32_t gt = 0, ic = 0;
        bool ok = true;
        for (; ok; ++ic) {
            // each softmax warp reads the next item on its own (they meet no named barrier)
            int32_t w = -1;
            ok = ring_get_warp(ring, ic, w, abort_flag, a.status, a.wait_ns);
            if (!ok || w < 0 || *abort_flag) break;
            int32_t it, bh;
            decode_work(w, a.n_items, BH, a.group, it, bh);
            const FwdItem item = a.items[it];
            if (!fwd_item_ok(item, a.g.T, BH, a.g.D, a.part_floats)) {
                set_error(a.status, ATTN_E_BOUNDS);
                *abort_flag = 1;
                break;
            }
            const int nblk = (item.kv_hi - item.kv_lo + BN - 1) / BN;
            const int t_row = item.r0 + row;
            float m_run = -INFINITY, l_run = 0.f;
            for (int j = 0; j < nblk && ok; ++j) {
                const uint32_t t = gt + j, b = t & 1;
                ok = mbar_wait_warp(bar(LY::B_SFULL + b), (t >> 1) & 1, abort_flag, a.status, a.wait_ns);
                if (!ok) break;
                tc_fence_after();
                constexpr int NC = BN / 32;                // 32-column chunks of an S tile
                const uint32_t sa = tmem + lane_addr + kColS + b * BN;
                uint32_t r[NC][32];
#pragma unroll
                for (int c = 0; c < NC; ++c) tmem_ld32(sa + c * 32, r[c]);
                tmem_ld_wait();
                const int j0 = item.kv_lo + j * BN;
                const bool edge = (j0 + BN - 1 > item.r0) || (j0 + BN > item.kv_hi);
                float mt = -INFINITY;
                if (edge) {
                    const int lim = min(t_row + 1, item.kv_hi) - j0;   // visible columns: c < lim
#pragma unroll
                    for (int c = 0; c < NC; ++c)
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            float x = __uint_as_float(r[c][i]);
                            x = (c * 32 + i < lim) ? x : -INFINITY;
                            r[c][i] = __float_as_uint(x);
                            mt = fmaxf(mt, x);
                        }
                } else {
                    // four independent chains of three-input maxima
                    float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int c = 0; c < NC; ++c)
#pragma unroll
                        for (int i = 0; i < 32; i += 2)
                            m4[(c * 2 + (i >> 4)) & 3] =
                                fmax3(m4[(c * 2 + (i >> 4)) & 3], __uint_as_float(r[c][i]), __uint_as_float(r[c][i + 1]));
                    mt = fmax3(fmaxf(m4[0], m4[1]), m4[2], m4[3]);
                }
                mt *= sl2;
                bool rescale = false;
                float alpha = 1.f;
                if (mt > m_run + kRescaleThreshold) {
                    if (m_run != -INFINITY) {
                        rescale = true;
                        alpha = ex2(m_run - mt);
                    }
                    m_run = mt;
                }
                const float base = m_run == -INFINITY ? 0.f : m_run;
                // exponents two at a time (f32x2 FMA), row sum in two paired accumulators
                const float2 sl2x2 = make_float2(sl2, sl2), nbase = make_float2(-base, -base);
                float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                uint32_t p[NC / 2][32];
#pragma unroll
                for (int c = 0; c < NC; ++c)
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const float2 x =
                            ffma2(make_float2(__uint_as_float(r[c][i]), __uint_as_float(r[c][i + 1])), sl2x2, nbase);
                        const float p0 = ex2(x.x), p1 = ex2(x.y);
                        acc[(i >> 1) & 1] = fadd2(acc[(i >> 1) & 1], make_float2(p0, p1));
                        p[c >> 1][(c & 1) * 16 + (i >> 1)] = pack_bf16(p0, p1);
                    }
                const float lsum = (acc[0].x + acc[0].y) + (acc[1].x + acc[1].y);
                l_run = rescale ? fmaf(l_run, alpha, lsum) : l_run + lsum;
#pragma unroll
                for (int c2 = 0; c2 < NC / 2; ++c2) tmem_st32(sa + 32 * c2, p[c2]);
                // tcgen05.ld/st are warp-collective: rescale O if any row of the warp needs it
                if (__any_sync(0xffffffffu, rescale) && j > 0) {
                    // O holds the sum over tiles < j once PV_{j-1} has completed
                    ok = mbar_wait_warp(bar(LY::B_ODONE), (t - 1) & 1, abort_flag, a.status, a.wait_ns);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t oa = tmem + lane_addr + kColO;
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(oa + c * 32, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(oa + c * 32, o);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar(LY::B_PFULL + b));
            }
            if (!ok) break;
            // epilogue: wait for the last PV of the item, then O / l. This uses the
            // once-per-item barrier: when the softmax warps get here up to two PVs
            // may still be in flight, more than a per-PV parity wait can tell apart.
            ok = mbar_wait_warp(bar(LY::B_OFULL), ic & 1, abort_flag, a.status, a.wait_ns);
            if (!ok) break;
            tc_fence_after();
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            const float lse = l_run > 0.f ? (m_run + lg2(l_run)) * kLn2 : -INFINITY;
            const uint32_t oa = tmem + lane_addr + kColO;
            const int b_ = bh / a.g.H, h_ = bh % a.g.H;
            const bool live = t_row < item.r1;
            const int Dv = a.g.D;                      // dims written: D (the tile's dims past it are zero)
            if (item.part_off < 0) {
                __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(a.o) + (int64_t)b_ * a.g.sb +
                                     (int64_t)h_ * a.g.sh + (int64_t)t_row * a.g.st;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(oa + c * 32, o);
                    tmem_ld_wait();
                    if (live) {
                        uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            if (c * 32 + i * 8 >= Dv) break;
                            uint4 v;
                            v.x = pack_bf16(__uint_as_float(o[8 * i + 0]) * inv, __uint_as_float(o[8 * i + 1]) * inv);
                            v.y = pack_bf16(__uint_as_float(o[8 * i + 2]) * inv, __uint_as_float(o[8 * i + 3]) * inv);
                            v.z = pack_bf16(__uint_as_float(o[8 * i + 4]) * inv, __uint_as_float(o[8 * i + 5]) * inv);
                            v.w = pack_bf16(__uint_as_float(o[8 * i + 6]) * inv, __uint_as_float(o[8 * i + 7]) * inv);
                            d4[i] = v;
                        }
                    }
                }
                if (live) a.lse[(int64_t)bh * a.g.T + t_row] = lse;
            } else {
                const int64_t R = item.part_R;
                const int i_row = t_row - item.part_row0;
                float* dst = a.ws_f + item.part_off + ((int64_t)bh * R + i_row) * Dv;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(oa + c * 32, o);
                    tmem_ld_wait();
                    if (live) {
                        float4* d4 = reinterpret_cast<float4*>(dst + c * 32);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            if (c * 32 + i * 4 < Dv)
                                d4[i] = make_float4(__uint_as_float(o[4 * i]) * inv, __uint_as_float(o[4 * i + 1]) * inv,
                                                    __uint_as_float(o[4 * i + 2]) * inv,
                                                    __uint_as_float(o[4 * i + 3]) * inv);
                    }
                }
                if (live) a.ws_f[item.part_off + (int64_t)BH * R * Dv + (int64_t)bh * R + i_row] = lse;
            }
            tc_fence_before();
            mbar_arrive(bar(LY::B_OFREE));
            gt += nblk;
        }
    }
    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        if (*abort_flag) {
            // a wait gave up: let the MMAs already issued drain (bounded) before TMEM is released
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

template <int D, int KVS>
cudaError_t launch_d(const FwdArgs& a, cudaStream_t s) {
    CUtensorMap mq, mk, mv;
    TcMaps mp{1, 2, 3}, mpkv{1, 2, 3};
    const Geom gkv = a.g.kv();
    if (!make_tile_map(&mq, a.q, a.g, mp) || !make_tile_map(&mk, a.k, gkv, mpkv, kBlockN<D>) ||
        !make_tile_map(&mv, a.v, gkv, mpkv, kBlockN<D>))
        return cudaErrorInvalidValue;
    const int64_t work = (int64_t)a.n_items * a.g.B * a.g.H;
    if (work <= 0) return cudaSuccess;
    if (work > INT32_MAX) return cudaErrorInvalidValue;
    const size_t smem = FwdTcLayout<D, KVS>::ALLOC;
    static_assert(FwdTcLayout<D, KVS>::ALLOC <= 232448, "shared memory of the forward tile kernel");
    cudaError_t e =
        cudaFuncSetAttribute(fwd_tc_kernel<D, KVS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int grid = (int)std::min<int64_t>(work, device_sm_count());
    fwd_tc_kernel<D, KVS><<<grid, TC_THREADS, smem, s>>>(mq, mk, mv, a, mp, mpkv, (int32_t)work);
    return counted(cudaGetLastError());
}

}  // namespace

cudaError_t launch_fwd_tiles_tc(const FwdArgs& a, cudaStream_t s) {
    // head dims up to 64 run on 64-wide tiles, up to 128 on 128-wide tiles, the
    // others (up to 256) on 256-wide tiles with 64-key K/V tiles
    if (a.g.D > 128) return launch_d<256, 2>(a, s);
    return a.g.D > 64 ? launch_d<128, 3>(a, s) : launch_d<64, 3>(a, s);
}

}  // namespace attn
