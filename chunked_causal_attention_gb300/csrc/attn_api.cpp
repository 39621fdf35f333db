// C-ABI layer of libattn: argument validation, workspace layout, work lists,
// kernel launches and status read-back. No device memory is allocated here.
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "attn_internal.h"

using namespace attn;

namespace {

constexpr size_t kAlign = 256;

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Head dims: any multiple of 8 up to 256, forward and backward (the backward
// above 128 dims splits each key tile's outputs over two work items).
constexpr int64_t kMaxDimFwd = 256;
constexpr int64_t kMaxDimBwd = 256;

int check_shape(const attn_shape* s, Geom* g) {
    if (!s) return ATTN_E_INVAL;
    if (s->B <= 0 || s->H <= 0 || s->T <= 0 || s->D <= 0) return ATTN_E_INVAL;
    if (s->T > INT32_MAX || s->B > INT32_MAX || s->H > INT32_MAX) return ATTN_E_INVAL;
    if ((int64_t)s->B * s->H > (1ll << 24)) return ATTN_E_INVAL;
    if (s->D < 8 || s->D > kMaxDimFwd || (s->D % 8)) return ATTN_E_UNSUPPORTED;
    if (s->sb <= 0 || s->st <= 0 || s->sh <= 0) return ATTN_E_INVAL;
    if (!std::isfinite(s->scale)) return ATTN_E_INVAL;
    if ((s->sb % 8) || (s->st % 8) || (s->sh % 8)) return ATTN_E_ALIGN;
    g->B = (int32_t)s->B; g->H = (int32_t)s->H; g->T = (int32_t)s->T; g->D = (int32_t)s->D;
    g->sb = s->sb; g->st = s->st; g->sh = s->sh; g->scale = s->scale;
    if (s->Hkv < 0 || s->Hkv > s->H) return ATTN_E_INVAL;
    if (s->Hkv == 0) {
        g->Hkv = g->H;
        g->sb_kv = g->sb; g->st_kv = g->st; g->sh_kv = g->sh;
    } else {
        if (s->H % s->Hkv) return ATTN_E_INVAL;
        if (s->sb_kv <= 0 || s->st_kv <= 0 || s->sh_kv <= 0) return ATTN_E_INVAL;
        if ((s->sb_kv % 8) || (s->st_kv % 8) || (s->sh_kv % 8)) return ATTN_E_ALIGN;
        g->Hkv = (int32_t)s->Hkv;
        g->sb_kv = s->sb_kv; g->st_kv = s->st_kv; g->sh_kv = s->sh_kv;
    }
    return ATTN_OK;
}

// Key-range boundaries of a chunk: [ctx, qe] unsplit, [ctx, m, qe] for a
// split point m > 0, the P-part equal-pair boundaries for kv_split = -P.
// False if the split is not valid for the chunk.
bool key_bounds(const attn_chunk& x, std::vector<int32_t>& k) {
    if (x.kv_split == 0) {
        k = {x.ctx_begin, x.q_end};
        return true;
    }
    if (x.kv_split > 0) {
        k = {x.ctx_begin, x.kv_split, x.q_end};
        return x.ctx_begin < x.kv_split && x.kv_split < x.q_end;
    }
    return x.kv_split >= -64 && resplit_bounds(x.q_begin, x.q_end, x.ctx_begin, -x.kv_split, k);
}

// Forward chunk rules: sorted by q_begin, disjoint, 0 <= ctx <= qb < qe <= T,
// kv_split == 0, ctx < m < qe, or -P (2 <= P <= 64) with valid boundaries.
int check_chunks_fwd(const attn_chunk* c, int32_t n, int32_t T) {
    if (n < 0 || (n > 0 && !c)) return ATTN_E_INVAL;
    std::vector<int32_t> k;
    for (int32_t i = 0; i < n; ++i) {
        const attn_chunk& x = c[i];
        if (!(0 <= x.ctx_begin && x.ctx_begin <= x.q_begin && x.q_begin < x.q_end && x.q_end <= T))
            return ATTN_E_INVAL;
        if (!key_bounds(x, k)) return ATTN_E_INVAL;
        if (i > 0 && c[i - 1].q_end > x.q_begin) return ATTN_E_INVAL;
    }
    return ATTN_OK;
}

// Backward additionally needs a partition of [0, T) into documents: chunks
// contiguous from 0 to T; a chunk either continues the previous chunk's
// document (same ctx_begin) or starts a new one (ctx_begin == q_begin).
int check_chunks_bwd(const attn_chunk* c, int32_t n, int32_t T) {
    int st = check_chunks_fwd(c, n, T);
    if (st) return st;
    if (n <= 0) return ATTN_E_INVAL;
    if (c[0].q_begin != 0 || c[n - 1].q_end != T) return ATTN_E_INVAL;
    for (int32_t i = 0; i < n; ++i) {
        if (i > 0 && c[i - 1].q_end != c[i].q_begin) return ATTN_E_INVAL;
        bool cont = i > 0 && c[i].ctx_begin == c[i - 1].ctx_begin;
        if (!cont && c[i].ctx_begin != c[i].q_begin) return ATTN_E_INVAL;
    }
    return ATTN_OK;
}

// ---------------------------------------------------------------- forward layout
struct FwdLayout {
    std::vector<FwdItem> items;
    std::vector<MergeSeg> segs;
    std::vector<int32_t> kbounds;   // key-range boundaries of the segments
    size_t off_items, off_segs, off_kb, off_parts, bytes;
    int64_t merge_work;
    int64_t part_floats;            // floats of the partial region
};

void fwd_layout(const Geom& g, const attn_chunk* c, int32_t n, FwdLayout& L) {
    const int64_t BH = (int64_t)g.B * g.H;
    L.items.clear();
    L.segs.clear();
    L.kbounds.clear();
    int64_t part_floats = 0;   // running float offset inside the partial region
    L.merge_work = 0;
    std::vector<int32_t> k;
    for (int32_t ci = 0; ci < n; ++ci) {
        const attn_chunk& x = c[ci];
        const int32_t qb = x.q_begin, qe = x.q_end, cb = x.ctx_begin;
        key_bounds(x, k);                       // validated by check_chunks_fwd
        const int32_t P = (int32_t)k.size() - 1;
        // rows before k_1 see only the first key range: whole 128-row tiles of
        // them get their final result directly; partials start at the tile of k_1
        const int32_t pr0 = P > 1 ? (k[1] > qb ? qb + kTile * ((k[1] - qb) / kTile) : qb) : qe;
        const int32_t R = qe - pr0;
        int64_t off0 = -1, blk = 0;
        if (P > 1) {
            blk = (int64_t)round_up((size_t)(BH * R * g.D + BH * R), 64);
            off0 = part_floats;
            part_floats += P * blk;
            MergeSeg s;
            s.row0 = pr0; s.R = R; s.P = P; s.kb = (int32_t)L.kbounds.size();
            s.off0 = off0; s.blk = blk; s.work0 = L.merge_work;
            const int64_t rb = merge_rows_per_block(g.D);
            L.merge_work += ((int64_t)R * BH + rb - 1) / rb;
            L.segs.push_back(s);
            L.kbounds.insert(L.kbounds.end(), k.begin(), k.end());
        }
        for (int32_t r0 = qb; r0 < qe; r0 += kTile) {
            int32_t r1 = std::min(r0 + kTile, qe);
            if (P == 1 || r0 < pr0) {
                L.items.push_back(FwdItem{r0, r1, cb, r1, -1, 0, 0});
            } else {
                // one partial per key range that some row of the tile can see
                for (int32_t p = 0; p < P && k[p] < r1; ++p)
                    L.items.push_back(FwdItem{r0, r1, k[p], std::min(k[p + 1], r1), off0 + p * blk, pr0, R});
            }
        }
    }
    // heaviest first (longest key range), stable for determinism
    std::stable_sort(L.items.begin(), L.items.end(), [](const FwdItem& a, const FwdItem& b) {
        return (a.kv_hi - a.kv_lo) > (b.kv_hi - b.kv_lo);
    });
    L.off_items = kHeaderBytes;
    L.off_segs = L.off_items + round_up(L.items.size() * sizeof(FwdItem), kAlign);
    L.off_kb = L.off_segs + round_up(L.segs.size() * sizeof(MergeSeg), kAlign);
    L.off_parts = L.off_kb + round_up(L.kbounds.size() * sizeof(int32_t), kAlign);
    L.bytes = L.off_parts + round_up((size_t)part_floats * sizeof(float), kAlign);
    L.part_floats = part_floats;
}

// --------------------------------------------------------------- backward layout
struct BwdLayout {
    std::vector<BwdItem> items;
    std::vector<RowSeg> segs;   // workspace rows <-> tokens
    int32_t rows;               // workspace rows of delta and the dQ accumulator per (batch, head)
    size_t off_items, off_segs, off_delta, off_dq, bytes;
};

void bwd_finish_layout(const Geom& g, BwdLayout& L) {
    const int64_t BH = (int64_t)g.B * g.H;
    // heaviest first: most query blocks
    std::stable_sort(L.items.begin(), L.items.end(), [](const BwdItem& a, const BwdItem& b) {
        return (a.q_end - a.q_lo) > (b.q_end - b.q_lo);
    });
    L.off_items = kHeaderBytes;
    L.off_segs = L.off_items + round_up(L.items.size() * sizeof(BwdItem), kAlign);
    L.off_delta = L.off_segs + round_up(L.segs.size() * sizeof(RowSeg), kAlign);
    L.off_dq = L.off_delta + round_up((size_t)BH * L.rows * sizeof(float), kAlign);
    L.bytes = L.off_dq + round_up((size_t)BH * L.rows * g.D * sizeof(float), kAlign);
}

// Whole backward: one item per key tile of every document; the tile's
// queries run from its first key to the document end.
void bwd_layout(const Geom& g, const attn_chunk* c, int32_t n, BwdLayout& L) {
    L.items.clear();
    int32_t i = 0;
    while (i < n) {
        int32_t s = c[i].ctx_begin, e = c[i].q_end;
        int32_t j = i + 1;
        while (j < n && c[j].ctx_begin == s) { e = c[j].q_end; ++j; }
        for (int32_t j0 = s; j0 < e; j0 += kTile)
            L.items.push_back(BwdItem{j0, std::min(j0 + kTile, e), e, j0, 0, 0, {0, 0}});
        i = j;
    }
    L.segs.assign(1, RowSeg{0, 0, g.T});
    L.rows = g.T;
    bwd_finish_layout(g, L);
}

// Backward of a set of chunks: one item per key tile of each chunk's context
// [ctx_begin, q_end); a tile's queries are the chunk's rows at or after its
// first key. delta and dQ hold the chunks' rows, one segment after another.
void bwd_chunk_layout(const Geom& g, const attn_chunk* c, int32_t n, BwdLayout& L) {
    L.items.clear();
    L.segs.clear();
    int32_t base = 0;
    for (int32_t i = 0; i < n; ++i) {
        const attn_chunk& x = c[i];
        const int32_t off = base - x.q_begin;
        for (int32_t j0 = x.ctx_begin; j0 < x.q_end; j0 += kTile)
            L.items.push_back(BwdItem{j0, std::min(j0 + kTile, x.q_end), x.q_end, std::max(j0, x.q_begin), off,
                                      x.q_begin, {0, 0}});
        L.segs.push_back(RowSeg{base, x.q_begin, x.q_end - x.q_begin});
        base += x.q_end - x.q_begin;
    }
    L.rows = base;
    bwd_finish_layout(g, L);
}

// Chunk-streamed backward: forward rules, plus disjoint key ranges: no chunk's
// context reaches into an earlier chunk of the same call.
int check_chunks_stream(const attn_chunk* c, int32_t n, int32_t T) {
    int st = check_chunks_fwd(c, n, T);
    if (st) return st;
    if (n <= 0) return ATTN_E_INVAL;
    for (int32_t i = 1; i < n; ++i)
        if (c[i].ctx_begin < c[i - 1].q_end) return ATTN_E_INVAL;
    return ATTN_OK;
}

}  // namespace

std::atomic<uint64_t> attn::g_kernel_launches{0};

void attn::wait_settings(uint64_t* wait_ns, int32_t* stall) {
    *wait_ns = 4000000000ull;
    *stall = 0;
    if (const char* e = std::getenv("ATTN_WAIT_LIMIT_MS")) {
        long v = std::strtol(e, nullptr, 10);
        if (v > 0 && v <= 600000) *wait_ns = (uint64_t)v * 1000000ull;
    }
    if (const char* e = std::getenv("ATTN_TEST_STALL_PRODUCER")) *stall = std::atoi(e) != 0;
}

bool attn::test_inconsistent_item() {
    const char* e = std::getenv("ATTN_TEST_INCONSISTENT_ITEM");
    return e && std::atoi(e) != 0;
}

namespace {

// Host arrays (work lists, segments) to the workspace, as kernel parameters
// (launch_upload): nothing refers to host memory once the call returns.
int upload(void* dst, const void* src, size_t bytes, cudaStream_t s) {
    if (!bytes) return ATTN_OK;
    return launch_upload(dst, src, bytes, s) == cudaSuccess ? ATTN_OK : ATTN_E_CUDA;
}

int reset_header(void* ws, cudaStream_t s) {
    return cudaMemsetAsync(ws, 0, kHeaderBytes, s) == cudaSuccess ? ATTN_OK : ATTN_E_CUDA;
}

int launched(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_E_CUDA; }

int check_ws(void* ws, size_t have, size_t need) {
    if (!ws || have < need) return ATTN_E_WORKSPACE;
    if (((uintptr_t)ws & (kAlign - 1)) != 0) return ATTN_E_ALIGN;
    return ATTN_OK;
}

// Items per head group in the work order (see decode_work). Both tile kernels
// run head-major (one group = all items of a head, heaviest first within the
// head). The forward's items of one head read the same K/V tiles, so with all
// CTAs on one head those tiles are reused from L2 (groups of 32 items, about
// five heads at a time, were 4-5% slower at 128K and 1M tokens). In the
// backward every dQ row of a head receives one fp32 reduction per key tile,
// and with all CTAs on the same head those reductions and the shared Q/dO
// tiles stay in L2.
constexpr int32_t kGroupFwd = 1 << 30;
constexpr int32_t kGroupBwd = 1 << 30;

int fwd_common(const void* q, const void* k, const void* v, const attn_chunk* chunks, int32_t n,
               const attn_shape* shape, void* o, float* lse, void* ws, size_t ws_bytes,
               cudaStream_t s, bool do_tiles, bool do_merge) {
    Geom g;
    int st = check_shape(shape, &g);
    if (st) return st;
    if ((st = check_chunks_fwd(chunks, n, g.T))) return st;
    if (!o || !lse || (do_tiles && (!q || !k || !v))) return ATTN_E_INVAL;
    if ((do_tiles && (!aligned16(q) || !aligned16(k) || !aligned16(v))) || !aligned16(o) ||
        !aligned16(lse))
        return ATTN_E_ALIGN;
    FwdLayout L;
    fwd_layout(g, chunks, n, L);
    if ((st = check_ws(ws, ws_bytes, L.bytes))) return st;
    uint8_t* w = (uint8_t*)ws;
    float* ws_f = (float*)(w + L.off_parts);
    if (do_tiles) {
        if ((st = reset_header(ws, s))) return st;
        if (!L.items.empty()) {
            // index-check test only: an empty row range, which addresses nothing
            if (test_inconsistent_item()) L.items[0].r1 = L.items[0].r0;
            if ((st = upload(w + L.off_items, L.items.data(), L.items.size() * sizeof(FwdItem), s))) return st;
            FwdArgs a;
            a.q = q; a.k = k; a.v = v; a.o = o; a.lse = lse; a.ws_f = ws_f;
            a.part_floats = L.part_floats;
            a.status = (uint32_t*)ws;
            a.counter = &((WsHeader*)ws)->counter[0];   // zeroed with the header above
            a.items = (const FwdItem*)(w + L.off_items);
            a.n_items = (int32_t)L.items.size();
            a.group = kGroupFwd;
            wait_settings(&a.wait_ns, &a.stall);
            a.g = g;
            if ((st = launched(launch_fwd_tiles_tc(a, s)))) return st;
        }
    }
    if (do_merge && !L.segs.empty()) {
        if ((st = upload(w + L.off_segs, L.segs.data(), L.segs.size() * sizeof(MergeSeg), s))) return st;
        if ((st = upload(w + L.off_kb, L.kbounds.data(), L.kbounds.size() * sizeof(int32_t), s))) return st;
        MergeArgs a;
        a.o = o; a.lse = lse; a.ws_f = ws_f;
        a.part_floats = L.part_floats;
        a.segs = (const MergeSeg*)(w + L.off_segs);
        a.kbounds = (const int32_t*)(w + L.off_kb);
        a.n_kbounds = (int32_t)L.kbounds.size();
        a.status = (uint32_t*)ws;
        a.n_segs = (int32_t)L.segs.size();
        a.total_work = L.merge_work;
        for (int32_t i = 0; i < (int32_t)L.segs.size() && i < kMergeSegsInline; ++i) a.segs_inline[i] = L.segs[i];
        a.bulk_parts = 2;
        for (const MergeSeg& sg : L.segs)
            if (sg.P <= kBulkParts) a.bulk_parts = std::max(a.bulk_parts, sg.P);
        a.g = g;
        if ((st = launched(launch_fwd_merge(a, s)))) return st;
    }
    return ATTN_OK;
}

enum BwdStage { kPrep = 1, kTiles = 2, kDq = 4 };

// Enqueue the stages of a backward laid out in L. dk_acc/dv_acc non-null:
// chunk-streamed epilogue (fp32 accumulation, bf16 from each item's emit_from on).
int bwd_launch(const Geom& g, const BwdLayout& L, const void* q, const void* k, const void* v, const void* o,
               const float* lse, const void* dout, void* dq, void* dk, void* dv, float* dk_acc, float* dv_acc,
               void* ws, cudaStream_t s, int stages) {
    int st;
    uint8_t* w = (uint8_t*)ws;
    float* delta = (float*)(w + L.off_delta);
    float* dq_acc = (float*)(w + L.off_dq);
    const RowSeg* segs = (const RowSeg*)(w + L.off_segs);
    const int32_t n_segs = (int32_t)L.segs.size();
    if (stages & (kPrep | kDq)) {
        if ((st = upload(w + L.off_segs, L.segs.data(), L.segs.size() * sizeof(RowSeg), s))) return st;
    }
    if (stages & kPrep) {
        if ((st = reset_header(ws, s))) return st;
        PrepArgs a{o, dout, delta, dq_acc, segs, n_segs, L.rows, (uint32_t*)ws, g};
        if ((st = launched(launch_bwd_prep(a, s)))) return st;
    }
    if (stages & kTiles) {
        if (test_inconsistent_item() && !L.items.empty()) {
            // index-check test only: an empty query range, which addresses nothing
            std::vector<BwdItem> items = L.items;
            items[0].q_end = items[0].q_lo;
            if ((st = upload(w + L.off_items, items.data(), items.size() * sizeof(BwdItem), s))) return st;
        } else if ((st = upload(w + L.off_items, L.items.data(), L.items.size() * sizeof(BwdItem), s))) {
            return st;
        }
        // the tile kernel's work queue starts at zero (the status word is kept: an
        // earlier stage of the same backward may have recorded an error)
        uint32_t* counter = &((WsHeader*)ws)->counter[1];
        if (cudaMemsetAsync(counter, 0, sizeof(uint32_t), s) != cudaSuccess) return ATTN_E_CUDA;
        BwdArgs a;
        a.q = q; a.k = k; a.v = v; a.dout = dout; a.lse = lse; a.delta = delta;
        a.counter = counter;
        a.dk = dk; a.dv = dv; a.dq_acc = dq_acc;
        a.rows = L.rows;
        a.dk_acc = dk_acc; a.dv_acc = dv_acc;
        a.status = (uint32_t*)ws;
        a.items = (const BwdItem*)(w + L.off_items);
        a.n_items = (int32_t)L.items.size();
        a.group = kGroupBwd;
        wait_settings(&a.wait_ns, &a.stall);
        a.g = g;
        if ((st = launched(g.D > 128 ? launch_bwd_tiles_wide(a, s) : launch_bwd_tiles_tc(a, s)))) return st;
    }
    if (stages & kDq) {
        DqArgs a{dq_acc, dq, segs, n_segs, L.rows, (uint32_t*)ws, g};
        if ((st = launched(launch_bwd_dq(a, s)))) return st;
    }
    return ATTN_OK;
}

int bwd_common(const void* q, const void* k, const void* v, const void* o, const float* lse,
               const void* dout, const attn_chunk* chunks, int32_t n, const attn_shape* shape,
               void* dq, void* dk, void* dv, void* ws, size_t ws_bytes, cudaStream_t s, int stages) {
    Geom g;
    int st = check_shape(shape, &g);
    if (st) return st;
    if (g.D > kMaxDimBwd) return ATTN_E_UNSUPPORTED;
    if ((st = check_chunks_bwd(chunks, n, g.T))) return st;
    if ((stages & kPrep) && (!o || !dout)) return ATTN_E_INVAL;
    if ((stages & kTiles) && (!q || !k || !v || !lse || !dout || !dk || !dv)) return ATTN_E_INVAL;
    if ((stages & kDq) && !dq) return ATTN_E_INVAL;
    const void* ptrs[] = {q, k, v, o, lse, dout, dq, dk, dv};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return ATTN_E_ALIGN;
    BwdLayout L;
    bwd_layout(g, chunks, n, L);
    if ((st = check_ws(ws, ws_bytes, L.bytes))) return st;
    return bwd_launch(g, L, q, k, v, o, lse, dout, dq, dk, dv, nullptr, nullptr, ws, s, stages);
}

}  // namespace

extern "C" {

int attn_workspace_size(const attn_shape* shape, const attn_chunk* chunks, int32_t n, int32_t pass,
                        size_t* bytes) {
    if (!bytes) return ATTN_E_INVAL;
    Geom g;
    int st = check_shape(shape, &g);
    if (st) return st;
    if (pass == 0) {
        if ((st = check_chunks_fwd(chunks, n, g.T))) return st;
        FwdLayout L;
        fwd_layout(g, chunks, n, L);
        *bytes = L.bytes;
    } else if (pass == 1) {
        if (g.D > kMaxDimBwd) return ATTN_E_UNSUPPORTED;
        if ((st = check_chunks_bwd(chunks, n, g.T))) return st;
        BwdLayout L;
        bwd_layout(g, chunks, n, L);
        *bytes = L.bytes;
    } else if (pass == 2) {
        if (g.D > kMaxDimBwd) return ATTN_E_UNSUPPORTED;
        if ((st = check_chunks_stream(chunks, n, g.T))) return st;
        BwdLayout L;
        bwd_chunk_layout(g, chunks, n, L);
        *bytes = L.bytes;
    } else {
        return ATTN_E_INVAL;
    }
    return ATTN_OK;
}

int attn_fwd(const void* q, const void* k, const void* v, const attn_chunk* chunks, int32_t n,
             const attn_shape* shape, void* o, float* lse, void* ws, size_t ws_bytes, void* stream) {
    return fwd_common(q, k, v, chunks, n, shape, o, lse, ws, ws_bytes, (cudaStream_t)stream, true, true);
}

int attn_fwd_tiles(const void* q, const void* k, const void* v, const attn_chunk* chunks, int32_t n,
                   const attn_shape* shape, void* o, float* lse, void* ws, size_t ws_bytes,
                   void* stream) {
    return fwd_common(q, k, v, chunks, n, shape, o, lse, ws, ws_bytes, (cudaStream_t)stream, true, false);
}

int attn_fwd_merge(const attn_chunk* chunks, int32_t n, const attn_shape* shape, void* o, float* lse,
                   void* ws, size_t ws_bytes, void* stream) {
    return fwd_common(nullptr, nullptr, nullptr, chunks, n, shape, o, lse, ws, ws_bytes,
                      (cudaStream_t)stream, false, true);
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dout, const attn_chunk* chunks, int32_t n, const attn_shape* shape, void* dq,
             void* dk, void* dv, void* ws, size_t ws_bytes, void* stream) {
    return bwd_common(q, k, v, o, lse, dout, chunks, n, shape, dq, dk, dv, ws, ws_bytes,
                      (cudaStream_t)stream, kPrep | kTiles | kDq);
}

int attn_bwd_prep(const void* o, const void* dout, const attn_chunk* chunks, int32_t n,
                  const attn_shape* shape, void* ws, size_t ws_bytes, void* stream) {
    return bwd_common(nullptr, nullptr, nullptr, o, nullptr, dout, chunks, n, shape, nullptr, nullptr,
                      nullptr, ws, ws_bytes, (cudaStream_t)stream, kPrep);
}

int attn_bwd_tiles(const void* q, const void* k, const void* v, const float* lse, const void* dout,
                   const attn_chunk* chunks, int32_t n, const attn_shape* shape, void* dk, void* dv,
                   void* ws, size_t ws_bytes, void* stream) {
    return bwd_common(q, k, v, nullptr, lse, dout, chunks, n, shape, nullptr, dk, dv, ws, ws_bytes,
                      (cudaStream_t)stream, kTiles);
}

int attn_bwd_dq(const attn_chunk* chunks, int32_t n, const attn_shape* shape, void* dq, void* ws,
                size_t ws_bytes, void* stream) {
    return bwd_common(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, chunks, n, shape, dq, nullptr,
                      nullptr, ws, ws_bytes, (cudaStream_t)stream, kDq);
}

int attn_bwd_chunk(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   const void* dout, const attn_chunk* chunks, int32_t n, const attn_shape* shape, void* dq,
                   void* dk, void* dv, float* dk_acc, float* dv_acc, void* ws, size_t ws_bytes, void* stream) {
    Geom g;
    int st = check_shape(shape, &g);
    if (st) return st;
    if (g.D > kMaxDimBwd) return ATTN_E_UNSUPPORTED;
    if ((st = check_chunks_stream(chunks, n, g.T))) return st;
    const void* ptrs[] = {q, k, v, o, lse, dout, dq, dk, dv, dk_acc, dv_acc};
    for (const void* p : ptrs)
        if (!p) return ATTN_E_INVAL;
    for (const void* p : ptrs)
        if (!aligned16(p)) return ATTN_E_ALIGN;
    BwdLayout L;
    bwd_chunk_layout(g, chunks, n, L);
    if ((st = check_ws(ws, ws_bytes, L.bytes))) return st;
    return bwd_launch(g, L, q, k, v, o, lse, dout, dq, dk, dv, dk_acc, dv_acc, ws, (cudaStream_t)stream,
                      kPrep | kTiles | kDq);
}

int attn_status(void* ws, void* stream) {
    if (!ws) return ATTN_E_INVAL;
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t word = 0;
    if (cudaMemcpyAsync(&word, ws, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess) return ATTN_E_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return ATTN_E_CUDA;
    if (word) {
        if (cudaMemsetAsync(ws, 0, sizeof(word), s) != cudaSuccess) return ATTN_E_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return ATTN_E_CUDA;
    }
    return (int)word;
}

const char* attn_strerror(int st) {
    switch (st) {
        case ATTN_OK: return "ok";
        case ATTN_E_INVAL: return "invalid argument (shape, chunk table, mode or pointer)";
        case ATTN_E_ALIGN: return "pointer or stride not 16-byte aligned";
        case ATTN_E_UNSUPPORTED: return "unsupported head dimension or device";
        case ATTN_E_WORKSPACE: return "workspace missing or too small";
        case ATTN_E_CUDA: return "CUDA runtime call or kernel launch failed";
        case ATTN_E_TIMEOUT: return "device wait gave up (bounded wait timed out)";
        case ATTN_E_BOUNDS: return "device index check failed";
        case ATTN_E_CAPACITY: return "plan output array too small";
        default: return "unknown status";
    }
}

const char* attn_version(void) { return "libattn 0.1 sm_103a"; }

uint64_t attn_kernel_launches(void) { return attn::g_kernel_launches.load(std::memory_order_relaxed); }

}  // extern "C"
