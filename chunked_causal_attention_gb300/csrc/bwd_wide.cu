// Backward key-tile kernel for head dims 129..256 on the tcgen05 tensor cores.
//
// The key/value gradients of a token collect contributions from every later
// token of its sequence (InfiniPipe §II-A), computed per 128-key tile as in the
// kernel for narrower heads: S^T = K Q^T, P^T = exp(S^T - LSE), dP^T = V dO^T,
// dS^T = P^T o (dP^T - D_t), dV += P^T dO, dK += dS^T Q, dQ += dS K. At 256
// dims the three D-wide accumulators (dV, dK, dQ) of a 128-key tile do not fit
// the 512 TMEM columns next to S^T and dP^T, so each tile is split into two
// work items by output dims: item half h produces dims [128h, 128h + 128) of
// dV, dK and dQ and recomputes S^T and dP^T (which contract over all dims) for
// itself. The two halves of a tile are adjacent in the work order, so they run
// at the same time and read the same K/V/Q/dO tiles from L2.
//
// Shared memory (1 CTA per SM): K and V of the tile (128 x 256 bf16 each,
// resident for the item), Q and dO of one 64-query block (64 x 256 each), and
// dS^T (128 keys x 64 queries bf16). TMEM columns: S^T [0,64), dP^T [64,128),
// P^T as bf16 [128,160), dQ^T [160,224), dV [256,384), dK [384,512).
//
// Per query block, all 8 warps step together: one leader thread (warp 1,
// lane 0) issues the TMA loads and the MMAs; every warp computes 32 queries x
// 32 keys of the softmax gradient (TMEM lanes = keys) and drains 32 queries x
// 32 dims of dQ^T (TMEM lanes = dims) into the fp32 dQ accumulator by
// reductions in L2 while the next block's Q and dO load.
//   S^T  = K Q^T          M=128 keys, N=64 queries, K=256 dims   (SS, K-major)
//   dP^T = V dO^T         as S^T
//   dV_h += P^T dO_h      M=128 keys, N=128 dims,  K=64 queries  (A = P^T in TMEM, B MN-major)
//   dK_h += dS^T Q_h      M=128 keys, N=128 dims,  K=64 queries  (A = dS^T K-major, B MN-major)
//   dQ_h^T = K_h^T dS^T   M=128 dims, N=64 queries, K=128 keys   (A, B MN-major)
// Every mbarrier wait is bounded; the warps decide to go on or to leave by a
// vote at the block's CTA barriers (__syncthreads_and), so they leave together.
// Each work item is checked against the geometry before it is used.
#include "tc_common.cuh"

namespace attn {
namespace {

using namespace tc;

constexpr int BW_THREADS = 256;
constexpr int kQB = 64;                      // query rows per block
constexpr uint32_t kWCols = 512;
constexpr uint32_t cS = 0, cDP = 64, cP = 128, cDQ = 160, cDV = 256, cDK = 384;

struct WideLayout {
    static constexpr int KV_TILE = 128 * 256 * 2;   // 4 boxes of 128 rows x 64 dims (16 KB each)
    static constexpr int QB_TILE = kQB * 256 * 2;   // 4 boxes of 64 rows x 64 dims (8 KB each)
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = K_OFF + KV_TILE;
    static constexpr int Q_OFF = V_OFF + KV_TILE;
    static constexpr int DO_OFF = Q_OFF + QB_TILE;
    static constexpr int DS_OFF = DO_OFF + QB_TILE; // dS^T: 128 keys x 64 queries bf16, 128-byte swizzle
    static constexpr int NL_OFF = DS_OFF + 16384;   // 64 floats: -LSE_t * log2 e
    static constexpr int ND_OFF = NL_OFF + 256;     // 64 floats: -D_t
    static constexpr int BAR_OFF = ND_OFF + 256;
    static constexpr int B_KV = 0, B_Q = 1, B_DO = 2, B_SDP = 3, B_G = 4, B_DRAIN = 5;
    static constexpr int NBAR = 6;
    static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;   // TMEM address, abort flag, next work index
    static constexpr int BYTES = MISC_OFF + 16;
    static constexpr size_t ALLOC = (size_t)BYTES + 1024;
};
static_assert(WideLayout::ALLOC <= 232448, "shared memory of the wide backward");

// Coordinates of map axes 1..3 (token, head, batch in stride order).
__device__ __forceinline__ void axes(const TcMaps& mp, int row, int h, int b, int& c1, int& c2, int& c3) {
    c1 = mp.pos_t == 1 ? row : (mp.pos_h == 1 ? h : b);
    c2 = mp.pos_t == 2 ? row : (mp.pos_h == 2 ? h : b);
    c3 = mp.pos_t == 3 ? row : (mp.pos_h == 3 ? h : b);
}

// One tile of 256 dims as 4 boxes of 64 dims (box_bytes apart); dims past the
// head dim read as zeros.
__device__ __forceinline__ void load_wide(uint32_t dst, const CUtensorMap* map, uint32_t bar, const TcMaps& mp,
                                          int row, int h, int b, int box_bytes) {
    int c1, c2, c3;
    axes(mp, row, h, b, c1, c2, c3);
#pragma unroll
    for (int a = 0; a < 4; ++a) tma_load_4d(dst + a * box_bytes, map, bar, a * 64, c1, c2, c3);
}

// ACC: the chunk-streamed backward (fp32 dK/dV accumulators, bf16 written for
// keys at or after the item's emit_from); otherwise bf16 dK/dV are written.
template <bool ACC>
__global__ void __launch_bounds__(BW_THREADS, 1)
    bwd_wide_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo,
                    const BwdArgs a, const TcMaps mp, const TcMaps mpkv,
                    const int32_t n_work) {
    using LY = WideLayout;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);
    const uint32_t bar0 = sbase + LY::BAR_OFF;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + LY::MISC_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + LY::MISC_OFF + 4);
    volatile int32_t* s_work = reinterpret_cast<volatile int32_t*>(sm + LY::MISC_OFF + 8);
    float* s_nl = reinterpret_cast<float*>(sm + LY::NL_OFF);
    float* s_nd = reinterpret_cast<float*>(sm + LY::ND_OFF);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool leader = tid == 32;                  // TMA, MMA and work claims
    const int BHKV = a.g.B * a.g.Hkv;
    const int G = a.g.H / a.g.Hkv;
    const int Dh = a.g.D;                           // the head dim (the tiles are 256 wide)
    const float sl2 = a.g.scale * kLog2e;

    if (tid == 0) {
        for (int i = 0; i < LY::NBAR; ++i) mbar_init(bar(i), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kWCols);
        tmem_relinquish();
    }
    if (leader) *s_work = (int32_t)atomicAdd(a.counter, 1u);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
    const int ch = warp >> 2;                       // column half: queries [32ch, 32ch + 32)

    constexpr uint32_t id_s = idesc_bf16(128, kQB, 0, 0);
    constexpr uint32_t id_g = idesc_bf16(128, 128, 0, 1);
    constexpr uint32_t id_q = idesc_bf16(128, kQB, 1, 1);
    uint32_t ph_sdp = 0, ph_g = 0;                  // MMA commits waited for (every thread)
    // the leader's TMA loads issued and waited for, per barrier (a load still in
    // flight when the CTA leaves early is waited for at the end)
    uint32_t iss_kv = 0, got_kv = 0, iss_q = 0, got_q = 0, iss_do = 0, got_do = 0;
    bool ok = true;

    while (ok) {
        const int32_t w = *s_work;
        if (w >= n_work) break;                     // the same in every thread
        const int half = w & 1;
        int32_t it, bkv;
        decode_work(w >> 1, a.n_items, BHKV, a.group, it, bkv);
        const BwdItem item = a.items[it];
        if (!bwd_item_ok(item, a.g.T, a.rows)) {    // every thread reads the same item
            if (leader) set_error(a.status, ATTN_E_BOUNDS);
            break;
        }
        const int b = bkv / a.g.Hkv, hk = bkv % a.g.Hkv;
        const int nq = (item.q_end - item.q_lo + kQB - 1) / kQB;
        const int nblk = G * nq;
        // block n: query head hk*G + n / nq, rows from the last block of the range down
        auto blk_row = [&](int n) { return item.q_lo + (nq - 1 - n % nq) * kQB; };
        auto blk_head = [&](int n) { return hk * G + n / nq; };
        if (leader && !a.stall) {                   // (a stalled producer issues nothing: every wait runs out)
            mbar_expect_tx(bar(LY::B_KV), 2 * LY::KV_TILE);
            load_wide(sbase + LY::K_OFF, &tmk, bar(LY::B_KV), mpkv, item.j0, hk, b, 16384);
            load_wide(sbase + LY::V_OFF, &tmv, bar(LY::B_KV), mpkv, item.j0, hk, b, 16384);
            ++iss_kv;
            mbar_expect_tx(bar(LY::B_Q), LY::QB_TILE);
            load_wide(sbase + LY::Q_OFF, &tmq, bar(LY::B_Q), mp, blk_row(0), blk_head(0), b, 8192);
            ++iss_q;
            mbar_expect_tx(bar(LY::B_DO), LY::QB_TILE);
            load_wide(sbase + LY::DO_OFF, &tmdo, bar(LY::B_DO), mp, blk_row(0), blk_head(0), b, 8192);
            ++iss_do;
        }
        const int key = item.j0 + 32 * (warp & 3) + lane;   // this thread's key row (TMEM lane)
        const int krow = key - item.j0;
        for (int n = 0; n < nblk; ++n) {
            const int i0 = blk_row(n);
            const int64_t bhq = (int64_t)b * a.g.H + blk_head(n);
            // stage -LSE*log2e and -D_t of the block's queries (0 past the range)
            if (tid < 2 * kQB) {
                const int q = i0 + (tid & (kQB - 1));
                float x = 0.f;
                if (q < item.q_end)
                    x = tid < kQB ? -kLog2e * a.lse[bhq * a.g.T + q] : -a.delta[bhq * a.rows + item.row_off + q];
                (tid < kQB ? s_nl : s_nd)[tid & (kQB - 1)] = x;
            }
            // S^T and dP^T of the block
            if (leader) {
                if (n == 0) {
                    ok = mbar_wait(bar(LY::B_KV), got_kv & 1, abort_flag, a.status, a.wait_ns);
                    got_kv += ok;
                }
                if (ok) {
                    ok = mbar_wait(bar(LY::B_Q), got_q & 1, abort_flag, a.status, a.wait_ns);
                    got_q += ok;
                }
                if (ok) {
                    // S^T as soon as Q is in, dP^T once dO is
                    tc_fence_after();
                    const uint32_t k0 = sbase + LY::K_OFF, v0 = sbase + LY::V_OFF;
                    const uint32_t q0 = sbase + LY::Q_OFF, o0 = sbase + LY::DO_OFF;
#pragma unroll
                    for (int kk = 0; kk < 16; ++kk) {
                        const uint32_t ok_ = (kk >> 2) * 16384 + (kk & 3) * 32;
                        const uint32_t oq = (kk >> 2) * 8192 + (kk & 3) * 32;
                        mma_ss(tmem + cS, sdesc_sw128(k0 + ok_, 16, 1024), sdesc_sw128(q0 + oq, 16, 1024), id_s,
                               kk > 0);
                    }
                    ok = mbar_wait(bar(LY::B_DO), got_do & 1, abort_flag, a.status, a.wait_ns);
                    got_do += ok;
                    if (ok) {
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < 16; ++kk) {
                            const uint32_t ok_ = (kk >> 2) * 16384 + (kk & 3) * 32;
                            const uint32_t oq = (kk >> 2) * 8192 + (kk & 3) * 32;
                            mma_ss(tmem + cDP, sdesc_sw128(v0 + ok_, 16, 1024), sdesc_sw128(o0 + oq, 16, 1024),
                                   id_s, kk > 0);
                        }
                        mma_commit(bar(LY::B_SDP));
                    }
                }
            }
            tc_fence_before();
            if (!__syncthreads_and(ok && !*abort_flag)) {
                ok = false;
                break;
            }
            // softmax gradient: 32 keys x 32 queries per warp
            ok = mbar_wait_warp(bar(LY::B_SDP), ph_sdp & 1, abort_flag, a.status, a.wait_ns);
            ++ph_sdp;
            if (ok) {
                tc_fence_after();
                uint32_t sr[32], dr[32];
                tmem_ld32(tmem + lane_addr + cS + 32 * ch, sr);
                tmem_ld32(tmem + lane_addr + cDP + 32 * ch, dr);
                tmem_ld_wait();
                uint32_t pp[16], dd[16];
                const float4* nl4 = reinterpret_cast<const float4*>(s_nl + 32 * ch);
                const float4* nd4 = reinterpret_cast<const float4*>(s_nd + 32 * ch);
#pragma unroll
                for (int e4 = 0; e4 < 8; ++e4) {
                    const float4 nl = nl4[e4], nd = nd4[e4];
                    const float nla[4] = {nl.x, nl.y, nl.z, nl.w}, nda[4] = {nd.x, nd.y, nd.z, nd.w};
                    float p[4], ds[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int e = 4 * e4 + u;
                        const int q = i0 + 32 * ch + e;
                        const bool vis = key < item.j1 && key <= q && q < item.q_end;
                        const float pv = ex2(fmaf(__uint_as_float(sr[e]), sl2, nla[u]));
                        p[u] = vis ? pv : 0.f;
                        ds[u] = vis ? pv * (__uint_as_float(dr[e]) + nda[u]) : 0.f;
                    }
                    pp[2 * e4] = pack_bf16(p[0], p[1]);
                    pp[2 * e4 + 1] = pack_bf16(p[2], p[3]);
                    dd[2 * e4] = pack_bf16(ds[0], ds[1]);
                    dd[2 * e4 + 1] = pack_bf16(ds[2], ds[3]);
                }
                // P^T (bf16 pairs) into TMEM: queries 32ch.. at columns cP + 16ch..
                tmem_st8(tmem + lane_addr + cP + 16 * ch, *reinterpret_cast<const uint32_t(*)[8]>(&pp[0]));
                tmem_st8(tmem + lane_addr + cP + 16 * ch + 8, *reinterpret_cast<const uint32_t(*)[8]>(&pp[8]));
                // dS^T row of this key: 64 bytes at 16-byte chunks 4ch.., 128-byte swizzle
                uint8_t* ds_row = sm + LY::DS_OFF + krow * 128;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int chunk = 4 * ch + u;
                    *reinterpret_cast<uint4*>(ds_row + ((chunk ^ (krow & 7)) << 4)) =
                        make_uint4(dd[4 * u], dd[4 * u + 1], dd[4 * u + 2], dd[4 * u + 3]);
                }
                tmem_st_wait();
                fence_proxy_async_smem();
            }
            tc_fence_before();
            if (!__syncthreads_and(ok && !*abort_flag)) {
                ok = false;
                break;
            }
            // dV_h, dK_h and dQ_h^T
            if (leader) {
                tc_fence_after();
                const uint32_t q0 = sbase + LY::Q_OFF, o0 = sbase + LY::DO_OFF, ds0 = sbase + LY::DS_OFF;
                const uint32_t k0 = sbase + LY::K_OFF;
#pragma unroll
                for (int kk = 0; kk < kQB / 16; ++kk) {
                    const uint32_t acc = (n > 0 || kk > 0) ? 1u : 0u;
                    mma_ts(tmem + cDV, tmem + cP + 8 * kk, sdesc_sw128(o0 + 2 * half * 8192 + kk * 2048, 8192, 1024),
                           id_g, acc);
                    mma_ss(tmem + cDK, sdesc_sw128(ds0 + kk * 32, 16, 1024),
                           sdesc_sw128(q0 + 2 * half * 8192 + kk * 2048, 8192, 1024), id_g, acc);
                }
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ss(tmem + cDQ, sdesc_sw128(k0 + 2 * half * 16384 + kk * 2048, 16384, 1024),
                           sdesc_sw128(ds0 + kk * 2048, 16384, 1024), id_q, kk > 0);
                mma_commit(bar(LY::B_G));
            }
            ok = mbar_wait_warp(bar(LY::B_G), ph_g & 1, abort_flag, a.status, a.wait_ns);
            ++ph_g;
            // Q, dO and dS are free: the next block's Q and dO go out now
            if (leader && ok && !a.stall && n + 1 < nblk) {
                mbar_expect_tx(bar(LY::B_Q), LY::QB_TILE);
                load_wide(sbase + LY::Q_OFF, &tmq, bar(LY::B_Q), mp, blk_row(n + 1), blk_head(n + 1), b, 8192);
                ++iss_q;
                mbar_expect_tx(bar(LY::B_DO), LY::QB_TILE);
                load_wide(sbase + LY::DO_OFF, &tmdo, bar(LY::B_DO), mp, blk_row(n + 1), blk_head(n + 1), b, 8192);
                ++iss_do;
            }
            // dQ^T: TMEM lane = dim 32*(warp&3) + lane of this half, columns = queries;
            // added into the fp32 accumulator by reductions in L2, one 128-byte row
            // segment (32 dims of one query) per warp instruction
            if (ok) {
                tc_fence_after();
                uint32_t r[32];
                tmem_ld32(tmem + lane_addr + cDQ + 32 * ch, r);
                tmem_ld_wait();
                const int d = 128 * half + 32 * (warp & 3) + lane;
                if (d < Dh) {
                    float* dst = a.dq_acc + (bhq * a.rows + item.row_off + i0 + 32 * ch) * (int64_t)Dh + d;
                    const int nrow = min(32, item.q_end - (i0 + 32 * ch));   // rows past the range add nothing
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (e < nrow) atomicAdd(dst + (int64_t)e * Dh, __uint_as_float(r[e]) * a.g.scale);
                }
            }
        }
        // a wait of the last block may have given up in some warps only: the CTA
        // decides together whether to write the epilogue or to leave
        tc_fence_before();
        if (!__syncthreads_and(ok && !*abort_flag)) break;
        // epilogue: warps 0-3 write dK_h * scale, warps 4-7 dV_h, one key row per thread
        {
            const int64_t roff = (int64_t)b * a.g.sb_kv + (int64_t)hk * a.g.sh_kv + (int64_t)key * a.g.st_kv;
            const bool live = key < item.j1;
            const uint32_t col = ch == 0 ? cDK : cDV;
            const float gmul = ch == 0 ? a.g.scale : 1.f;
            __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(ch == 0 ? a.dk : a.dv) + roff;
            float* acc = ACC ? (ch == 0 ? a.dk_acc : a.dv_acc) + roff : nullptr;
            const bool emit = !ACC || key >= item.emit_from;
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                const int d0 = 128 * half + 32 * c;
                uint32_t r[32];
                tmem_ld32(tmem + lane_addr + col + 32 * c, r);
                tmem_ld_wait();
                if (!live || d0 >= Dh) continue;
                float f[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(r[e]) * gmul;
                if (ACC) {
                    float4* a4 = reinterpret_cast<float4*>(acc + d0);
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        if (d0 + 4 * u >= Dh) break;
                        float4 x = a4[u];
                        x.x += f[4 * u]; x.y += f[4 * u + 1]; x.z += f[4 * u + 2]; x.w += f[4 * u + 3];
                        a4[u] = x;
                        f[4 * u] = x.x; f[4 * u + 1] = x.y; f[4 * u + 2] = x.z; f[4 * u + 3] = x.w;
                    }
                }
                if (emit) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + d0);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        if (d0 + 8 * u >= Dh) break;
                        d4[u] = make_uint4(pack_bf16(f[8 * u], f[8 * u + 1]), pack_bf16(f[8 * u + 2], f[8 * u + 3]),
                                           pack_bf16(f[8 * u + 4], f[8 * u + 5]), pack_bf16(f[8 * u + 6], f[8 * u + 7]));
                    }
                }
            }
        }
        // the next item (the TMEM loads above are complete before the next dV/dK MMAs,
        // which the leader issues only after two more CTA barriers)
        if (leader) *s_work = (int32_t)atomicAdd(a.counter, 1u);
        tc_fence_before();
        if (!__syncthreads_and(!*abort_flag)) break;
    }
    // ---------------------------------------------------------------- teardown
    if (leader) {
        // loads that a wait which gave up left in flight land before the CTA leaves
        // (bounded)
        const uint64_t t0 = globaltimer();
        while (iss_kv > got_kv && !mbar_try_wait(bar(LY::B_KV), got_kv & 1) && globaltimer() - t0 < a.wait_ns) {
        }
        while (iss_q > got_q && !mbar_try_wait(bar(LY::B_Q), got_q & 1) && globaltimer() - t0 < a.wait_ns) {
        }
        while (iss_do > got_do && !mbar_try_wait(bar(LY::B_DO), got_do & 1) && globaltimer() - t0 < a.wait_ns) {
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        if (*abort_flag) {
            // MMAs the leader issued may still be in flight: wait (bounded) for them
            if (lane == 0) {
                mma_commit(bar(LY::B_DRAIN));
                const uint64_t t0 = globaltimer();
                while (!mbar_try_wait(bar(LY::B_DRAIN), 0) && globaltimer() - t0 < a.wait_ns) {
                }
            }
            __syncwarp();
        }
        tmem_dealloc(tmem, kWCols);
    }
}

template <bool ACC>
cudaError_t launch_wide(const BwdArgs& a, cudaStream_t s) {
    CUtensorMap mq, mk, mv, mdo;
    TcMaps mp{1, 2, 3}, mpkv{1, 2, 3};
    const Geom gkv = a.g.kv();
    if (!make_tile_map(&mq, a.q, a.g, mp, kQB) || !make_tile_map(&mk, a.k, gkv, mpkv) ||
        !make_tile_map(&mv, a.v, gkv, mpkv) || !make_tile_map(&mdo, a.dout, a.g, mp, kQB))
        return cudaErrorInvalidValue;
    const int64_t work = 2 * (int64_t)a.n_items * a.g.B * a.g.Hkv;   // two output halves per key tile
    if (work <= 0) return cudaSuccess;
    if (work > INT32_MAX) return cudaErrorInvalidValue;
    const size_t smem = WideLayout::ALLOC;
    cudaError_t e = cudaFuncSetAttribute(bwd_wide_kernel<ACC>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int grid = (int)std::min<int64_t>(work, device_sm_count());
    bwd_wide_kernel<ACC><<<grid, BW_THREADS, smem, s>>>(mq, mk, mv, mdo, a, mp, mpkv, (int32_t)work);
    return counted(cudaGetLastError());
}

}  // namespace

cudaError_t launch_bwd_tiles_wide(const BwdArgs& a, cudaStream_t s) {
    return a.dk_acc != nullptr ? launch_wide<true>(a, s) : launch_wide<false>(a, s);
}

}  // namespace attn
