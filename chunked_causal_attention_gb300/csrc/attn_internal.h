// Internal declarations shared by the C-ABI layer and the kernels of libattn.
#pragma once

#include <cstddef>
#include <atomic>
#include <cstdint>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "attn.h"

namespace attn {

constexpr int kTile = 128;            // query rows per forward work item, keys per backward item
constexpr size_t kHeaderBytes = 256;  // workspace header: status word, counters

// Workspace header (first 256 bytes of every workspace).
struct WsHeader {
    uint32_t status;      // first device-side error code (ATTN_E_*), 0 if none
    uint32_t counter[3];  // work queues of the persistent kernels: [0] forward tiles, [1] backward tiles
};

// One forward work item: query rows [r0, r1) against keys [kv_lo, kv_hi)
// under the causal rule j <= t. part_off < 0: the rows' final O/LSE go to the
// output tensors; otherwise fp32 O goes to ws_f[part_off + (bh*R + i)*D + d]
// and LSE to ws_f[part_off + BH*R*D + bh*R + i], i = t - part_row0, R = part_R.
struct FwdItem {
    int32_t r0, r1;
    int32_t kv_lo, kv_hi;
    int64_t part_off;
    int32_t part_row0, part_R;
};
static_assert(sizeof(FwdItem) == 32, "FwdItem layout");

// Merge segment of one re-split chunk: rows [row0, row0 + R), P partial
// blocks, part p at float offset off0 + p * blk (layout as FwdItem); the
// part's key range starts at kbounds[kb + p], and row t merges the parts
// that start at or before t.
struct MergeSeg {
    int32_t row0, R;
    int32_t P, kb;
    int64_t off0, blk;
    int64_t work0;        // first merge block of this segment (blocks of merge_rows_per_block rows)
};
static_assert(sizeof(MergeSeg) == 40, "MergeSeg layout");

// One backward work item: keys [j0, j1) (j1 - j0 <= 128) of a document;
// the queries [q_lo, q_end) are walked in blocks of 128 rows starting at
// q_lo. Whole backward: q_lo = j0 and q_end = the document end. Backward of
// a chunk [q_begin, q_end): q_lo = max(j0, q_begin). Token t's row in delta
// and in the dQ accumulator is t + row_off. Chunk-streamed epilogue: keys >=
// emit_from (the chunk's q_begin) are written as bf16.
struct BwdItem {
    int32_t j0, j1;
    int32_t q_end;
    int32_t q_lo;
    int32_t row_off;
    int32_t emit_from;
    int32_t pad[2];
};
static_assert(sizeof(BwdItem) == 32, "BwdItem layout");

// Workspace rows [ws_row0, ws_row0 + R) of delta and the dQ accumulator hold
// tokens [t0, t0 + R) (one segment per chunk; one for the whole backward).
struct RowSeg {
    int32_t ws_row0, t0, R;
};

// Shape of q/o/dout/dq (B, H, T, D with strides sb, st, sh) and of the
// key/value tensors k/v/dk/dv (Hkv heads, strides sb_kv, st_kv, sh_kv); query
// head h reads key/value head h / (H / Hkv).
struct Geom {
    int32_t B, H, T, D;
    int64_t sb, st, sh;
    float scale;
    int32_t Hkv;
    int64_t sb_kv, st_kv, sh_kv;
    int32_t group() const { return H / Hkv; }
    // the key/value tensors' geometry in the query fields (for tensor maps)
    Geom kv() const {
        Geom k = *this;
        k.H = Hkv;
        k.sb = sb_kv; k.st = st_kv; k.sh = sh_kv;
        return k;
    }
};

struct FwdArgs {
    const void* q; const void* k; const void* v;
    void* o; float* lse;
    float* ws_f;
    int64_t part_floats;  // floats of the partial region at ws_f (index checks)
    uint32_t* status;
    uint32_t* counter;    // work queue: next work index to hand out (zero at launch)
    const FwdItem* items;
    int32_t n_items;
    int32_t group;        // items per head group in the work order
    uint64_t wait_ns;     // limit of every mbarrier wait
    int32_t stall;        // test only: the TMA producer issues nothing
    Geom g;
};

// Segment tables up to this length travel in the merge kernel's parameters.
constexpr int kMergeSegsInline = 8;
// Segments of up to this many parts are merged from bulk copies in shared memory.
constexpr int kBulkParts = 4;

struct MergeArgs {
    void* o; float* lse;
    const float* ws_f;
    int64_t part_floats;      // floats of the partial region at ws_f (index checks)
    const MergeSeg* segs;
    const int32_t* kbounds;   // key-range boundaries of all segments
    int32_t n_kbounds;
    uint32_t* status;
    int32_t n_segs;
    int64_t total_work;   // merge blocks: sum over segments of ceil(R * B * H / merge_rows_per_block)
    Geom g;
    MergeSeg segs_inline[kMergeSegsInline];   // a copy of segs when n_segs <= kMergeSegsInline
    int32_t bulk_parts;   // segments of 2..bulk_parts parts take the bulk path (the largest such P, at least 2)
};
// Rows (of B*H*R per segment) that one block of the merge kernel takes.
int merge_rows_per_block(int D);

// delta and the dQ accumulator hold `rows` workspace rows per (batch, head):
// delta[bh*rows + r], dq_acc[(bh*rows + r)*D + d]; segs map rows to tokens.
struct PrepArgs {
    const void* o; const void* dout;
    float* delta; float* dq_acc;
    const RowSeg* segs; int32_t n_segs;
    int32_t rows;
    uint32_t* status;
    Geom g;
};

struct BwdArgs {
    const void* q; const void* k; const void* v; const void* dout;
    const float* lse; const float* delta;
    void* dk; void* dv;
    float* dq_acc;
    int32_t rows;         // workspace rows of delta and dq_acc per (batch, head)
    // Chunk-streamed backward: fp32 dK/dV accumulators (element offsets of the
    // bf16 tensors); the epilogue adds into them and writes bf16 dk/dv only for
    // keys >= the item's emit_from. Null for the whole backward (bf16 written).
    float* dk_acc; float* dv_acc;
    uint32_t* status;
    uint32_t* counter;    // work queue: next work index to hand out (zero at launch)
    const BwdItem* items;
    int32_t n_items;
    int32_t group;
    uint64_t wait_ns;     // limit of every mbarrier wait
    int32_t stall;        // test only: the TMA producer issues nothing
    Geom g;
};

// Wait limit and producer stall for the tile kernels, from the environment:
// ATTN_WAIT_LIMIT_MS (default 4000) and ATTN_TEST_STALL_PRODUCER (default 0,
// used by the failure-detection test to make every wait run out).
void wait_settings(uint64_t* wait_ns, int32_t* stall);
// ATTN_TEST_INCONSISTENT_ITEM (default 0): used by the index-check test. The
// first work item of each tile kernel is made inconsistent before it is copied
// to the workspace, in a way that addresses nothing outside the buffers (an
// empty query range), so that the kernels' descriptor checks must report it.
bool test_inconsistent_item();

struct DqArgs {
    const float* dq_acc;  // rows as PrepArgs
    void* dq;
    const RowSeg* segs; int32_t n_segs;
    int32_t rows;
    uint32_t* status;
    Geom g;
};

// Coordinate slots (1..3) of the token, head and batch axes in a tile map.
struct TcMaps {
    int pos_t, pos_h, pos_b;
};

// Rank-4 TMA map of a bf16 [B, T, H, D]-strided tensor: axis 0 is the head
// dim, axes 1..3 are token/head/batch sorted by stride; box = 64 elements
// (128 bytes, 128-byte swizzle) x box_rows tokens. Fills `mp`. False on failure.
bool make_tile_map(CUtensorMap* m, const void* base, const Geom& g, TcMaps& mp, int box_rows = 128);
// Rank-3 TMA map of the fp32 dQ accumulator [B*H][rows][D]: box of 32 floats
// (128 bytes, 128-byte swizzle) x 128 tokens, used for reduce-adds.
bool make_dq_acc_map(CUtensorMap* m, float* dq_acc, const Geom& g, int32_t rows);
// Rank-4 TMA map of an fp32 dK or dV accumulator with the key/value strides of
// gkv (element offsets of dk/dv): box of 32 floats (128 bytes, 128-byte
// swizzle) x 128 tokens, used for reduce-adds. Fills `mp` (same axis order as
// the bf16 key/value maps).
bool make_kv_acc_map(CUtensorMap* m, float* acc, const Geom& gkv, TcMaps& mp);
int device_sm_count();

// Key-range boundaries cb = k_0 < ... < k_P = qe of a chunk re-split into P
// parts of equal visible-pair count (kv_split = -P). False if they collapse.
bool resplit_bounds(int32_t qb, int32_t qe, int32_t cb, int32_t P, std::vector<int32_t>& k);

// Kernels this library has enqueued since it was loaded (attn_kernel_launches);
// every launcher passes its launch error through counted().
extern std::atomic<uint64_t> g_kernel_launches;
inline cudaError_t counted(cudaError_t e) {
    if (e == cudaSuccess) g_kernel_launches.fetch_add(1, std::memory_order_relaxed);
    return e;
}

// Copy `bytes` of host data to device memory at dst (16-byte aligned), stream
// ordered, as the parameters of one small kernel per 31 KB (upload.cu).
cudaError_t launch_upload(void* dst, const void* src, size_t bytes, cudaStream_t s);

// Kernel launchers (return the launch error).
cudaError_t launch_fwd_tiles_tc(const FwdArgs& a, cudaStream_t s);   // fwd_tc.cu
cudaError_t launch_fwd_merge(const MergeArgs& a, cudaStream_t s);     // merge.cu
cudaError_t launch_bwd_prep(const PrepArgs& a, cudaStream_t s);       // bwd_aux.cu
cudaError_t launch_bwd_tiles_tc(const BwdArgs& a, cudaStream_t s);   // bwd_tc.cu (head dims up to 128)
cudaError_t launch_bwd_tiles_wide(const BwdArgs& a, cudaStream_t s); // bwd_wide.cu (129..256)
cudaError_t launch_bwd_dq(const DqArgs& a, cudaStream_t s);           // bwd_aux.cu

}  // namespace attn
