/*
 * attn.h - C ABI of libattn: chunked causal self-attention on GB300 (sm_103a).
 *
 * The operation: causal softmax attention computed subsequence by subsequence.
 * The query rows of chunk i attend to the resident keys/values of everything
 * before them (the chunk's context) and to themselves.
 *   - SPPO, "Efficient Long-sequence LLM Training via Adaptive Sequence Pipeline
 *     Parallel Offloading": §3.2 (FLOPs-based vs length-based partition), §4
 *     (multiplexing sequence partition: edge subsequences re-split, results
 *     combined), §5.1 (attention of subsequence i reads all K/V so far, which
 *     stay resident on the GPU).
 *   - InfiniPipe, "Elastic Pipeline Parallelism for Efficient Variable-Length
 *     Long-Context LLM Training": §II-A (a slice's queries see only preceding
 *     keys; K/V gradients depend on later slices), §II-B (packed [sum(S), D]
 *     layout), §III-A1 (chunk = {context C, slice lengths S}).
 *   - "Sequence Parallelism: Long Sequence Training from System Perspective"
 *     (blog summary), Deep Dive "Ring Self-Attention": a chunk's output is the
 *     accumulation of one partial per key/value block.
 *
 * Definition computed (one batch row b, head h; scale given by the caller):
 *   key j is visible to query t  iff  chunk(t).ctx_begin <= j <= t
 *   LSE_t = ln sum_{j visible} exp(scale * q_t . k_j)
 *   O_t   = sum_{j visible} exp(scale * q_t . k_j - LSE_t) v_j
 * and its gradient dQ, dK, dV for an upstream dO.
 *
 * Conventions shared by every entry point
 *   - Device pointers are CUDA device memory owned by the caller. The library
 *     never allocates, frees or retains device memory; the caller passes a
 *     workspace sized by attn_workspace_size().
 *   - q, k, v, o, dout, dq, dk, dv: bf16 (IEEE bfloat16), element (b, t, h, d)
 *     at  b*sb + t*st + h*sh + d  (strides in elements, d contiguous), the same
 *     strides for all eight tensors. Dense [B, H, L, D]: sb = H*L*D, sh = L*D,
 *     st = D. Packed [T, H, D] (B = 1): st = H*D, sh = D.
 *     Base pointers must be 16-byte aligned and sb, st, sh multiples of 8.
 *   - Head dim D: any multiple of 8 from 8 to 256 (InfiniPipe §III-A2 Eq. (3)
 *     carries D and D_kv as model dimensions). The tile kernels work on 64
 *     (D <= 64), 128 (D <= 128) or 256 dims; the dims past D are loaded as
 *     zeros, which leaves every score, output and gradient unchanged, and are
 *     never written. Throughput in FLOP of the true D is therefore D/64,
 *     D/128 or D/256 of that at the tile width. Above 128 dims the backward
 *     splits each 128-key tile into two work items, one per 128 output dims,
 *     which both compute the tile's scores and score gradients: it does 7/5
 *     of the backward's tensor work.
 *   - Grouped key/value heads (GQA/MQA): with Hkv > 0 in the shape, k, v, dk,
 *     dv (and the fp32 accumulators of attn_bwd_chunk) have Hkv heads and
 *     their own strides sb_kv, st_kv, sh_kv; query head h reads key/value head
 *     h / (H / Hkv), and the gradient of a key/value head is the sum over its
 *     H / Hkv query heads. Hkv = 0 means Hkv = H with the query strides.
 *   - lse: fp32, [B][H][T] contiguous, natural log.
 *   - stream: a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Compute calls only enqueue work and return before it completes.
 *   - chunks: a HOST array read during the call only. Each compute call lays
 *     out its work list on the host and writes it into the workspace with
 *     small copy kernels on `stream` that carry it in their launch
 *     parameters (up to 31 KB per launch), so nothing on the device refers to
 *     host memory after the call returns.
 *   - Every call returns an attn status code. Argument errors are detected on
 *     the host before anything is enqueued. Device-side errors are recorded in
 *     the workspace and read with attn_status(): ATTN_E_TIMEOUT (a bounded
 *     wait gave up) and ATTN_E_BOUNDS (a work descriptor in the workspace did
 *     not fit the shape or the workspace; every kernel checks each descriptor
 *     before it forms an address from it, and skips it). No entry point traps
 *     or aborts.
 */
#ifndef ATTN_H_
#define ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define ATTN_OK             0
#define ATTN_E_INVAL        1  /* bad shape, chunk table, mode or pointer      */
#define ATTN_E_ALIGN        2  /* pointer or stride not 16-byte aligned        */
#define ATTN_E_UNSUPPORTED  3  /* head dim not a multiple of 8 in [8, 256] */
#define ATTN_E_WORKSPACE    4  /* workspace NULL or smaller than required      */
#define ATTN_E_CUDA         5  /* a CUDA runtime call or kernel launch failed  */
#define ATTN_E_TIMEOUT      6  /* device: a bounded wait gave up               */
#define ATTN_E_BOUNDS       7  /* device: an index check failed                */
#define ATTN_E_CAPACITY     8  /* output array of attn_plan* too small          */

/* ---- plan modes (SPPO §3.2, §4) ---------------------------------------- */
#define ATTN_PLAN_UNIFORM              0  /* length-based: equal 128-multiples  */
#define ATTN_PLAN_FLOPS                1  /* FLOPs-based: b_k ~ L*sqrt(k/N)     */
#define ATTN_PLAN_FLOPS_RESPLIT_EDGES  2  /* FLOPS + first/last chunk re-split  */

/* One chunk (InfiniPipe §III-A1 split chunk {C, s}): query rows
 * [q_begin, q_end) with context C = q_begin - ctx_begin. ctx_begin is the
 * first visible key (the document start). kv_split = 0: no re-split; m with
 * ctx_begin < m < q_end: the chunk's key range is cut into [ctx_begin, m) and
 * [m, q_end); -P (2 <= P <= 64): the key range is cut into P parts carrying
 * equal numbers of visible (query, key) pairs of the chunk's queries, at the
 * multiples of 128 from ctx_begin nearest to the equal-pair points (ties up;
 * an error if they collapse). Each part is computed as a partial and the
 * parts are merged by log-sum-exp (SPPO §4 multiplexing, read as a key/value
 * split). */
typedef struct {
    int32_t q_begin, q_end;
    int32_t ctx_begin;
    int32_t kv_split;
} attn_chunk;

typedef struct {
    int64_t B, H, T, D;   /* batch rows, heads, tokens per row, head dim
                             (a multiple of 8, 8 <= D <= 256)               */
    int64_t sb, st, sh;   /* element strides of batch, token, head           */
    float   scale;        /* softmax scale; usually 1/sqrt(D)                */
    int64_t Hkv;          /* key/value heads (H % Hkv == 0); 0: Hkv = H     */
    int64_t sb_kv, st_kv, sh_kv;   /* strides of k, v, dk, dv when Hkv > 0  */
} attn_shape;

/* ---- planning (host only, integer-exact; never touches the GPU) -------- */

/* Chunk boundaries of one causal sequence of L tokens in N chunks.
 * UNIFORM: b_k = 128*floor(k*L/(128*N)). FLOPS: b_k = the multiple of 128
 * nearest to L*sqrt(k/N) (ties up), which equalises the quadratic attention
 * cost of InfiniPipe Eq. (1) (SPPO §3.2 FLOPs-based partition: long chunks
 * first, short later). b_0 = 0, b_N = L. RESPLIT_EDGES also sets kv_split of
 * the first and last chunk to q_begin + 128*floor((q_end-q_begin)/256 + 1/2)
 * when that falls strictly inside the chunk (SPPO §4).
 * out: host array of cap entries; *n_out = N on success.
 * Errors: ATTN_E_INVAL (L <= 0, N <= 0, unknown mode, boundaries not strictly
 * increasing), ATTN_E_CAPACITY (cap < N). */
int attn_plan(int64_t L, int32_t N, int32_t mode,
              attn_chunk* out, int32_t cap, int32_t* n_out);

/* FLOPS chunks of one sequence (as attn_plan) with the edge chunks re-split
 * as in SPPO's multiplexed sequence partition (§4, Table 3) for PP pipeline
 * stages: the SP range of an edge subsequence shrinks by one device per
 * subsequence away from each pipeline end, so chunk i and chunk N-1-i get
 * kv_split = -P with P the largest count from 2 up to PP - i that the chunk
 * can hold (none when PP - i < 2). Errors as attn_plan (PP <= 0 is
 * ATTN_E_INVAL). */
int attn_plan_multiplex(int64_t L, int32_t N, int32_t PP,
                        attn_chunk* out, int32_t cap, int32_t* n_out);

/* Chunks of a packed batch (InfiniPipe §II-B, §III-A1). cu_seqlens: host
 * array of ndocs+1 non-decreasing offsets, cu_seqlens[0] = 0. A document of
 * L_d tokens becomes ceil(L_d / max_chunk_tokens) chunks by the mode's rule
 * measured from the document start, all with ctx_begin = document start;
 * empty documents give no chunk. RESPLIT_EDGES re-splits the first and last
 * chunk of the whole plan. Errors as attn_plan. */
int attn_plan_varlen(const int64_t* cu_seqlens, int32_t ndocs, int32_t max_chunk_tokens,
                     int32_t mode, attn_chunk* out, int32_t cap, int32_t* n_out);

/* InfiniPipe's workload-balanced sequence chunking (Algorithm 1, §III-B),
 * on one GPU. Inputs: nseq sequence lengths (packed back to back in this
 * order, so sequence i starts at seq_lens[0] + ... + seq_lens[i-1]); K, the
 * number of slices of the longest sequence; token_cap, the most tokens one
 * chunk may hold (T_m); the cost model of Eq. (1) with N = d_p = 1: a chunk
 * {C, S} costs beta1 + alpha1((C+s0)^2 - C^2) + alpha2 s0 + the sum over its
 * other slices of alpha1 s^2 + alpha2 s.
 * Steps: the longest sequence is cut into K slices of equal cost (the mesh;
 * boundaries at the multiple of 128 nearest to each equal-cost point, ties
 * up); each sequence takes mesh slices in order while it is longer than the
 * next one (split chunks, one call each) and keeps the rest as its tail
 * slice; sequences no longer than the first mesh slice are short. Every tail
 * seeds a bucket (a hybrid chunk); short sequences, most expensive first, go
 * into the first bucket in order of increasing time per token whose time
 * stays within T_t (initially the costliest mesh slice) and whose tokens stay
 * within token_cap; a sequence that even the emptiest bucket cannot hold
 * opens a new bucket (a batched chunk); when no bucket fits, T_t is raised to
 * the least time among buckets with token room plus the sequence's time.
 * Output: the chunks of every call (chunk {C, S}), call after call, in out
 * (ctx_begin = the sequence start, kv_split = 0, sorted by q_begin within a
 * call); call c holds out[call_off[c] .. call_off[c+1]); *n_out chunks and
 * *n_calls calls. The order can be run one call at a time: forward with
 * attn_fwd in call order, backward with attn_bwd_chunk in reverse order.
 * Errors: ATTN_E_INVAL (no sequence, a negative length, more than INT32_MAX
 * tokens, K <= 0, costs negative or not finite or alpha1 = alpha2 = 0, a
 * mesh whose boundaries are not strictly increasing, token_cap below the
 * first mesh slice), ATTN_E_CAPACITY (cap < *n_out or call_cap < *n_calls + 1;
 * both counts are then set to what is needed). Host only. */
int attn_plan_infinipipe(const int64_t* seq_lens, int32_t nseq, int32_t K, int64_t token_cap,
                         double alpha1, double alpha2, double beta1,
                         attn_chunk* out, int32_t cap, int32_t* n_out,
                         int32_t* call_off, int32_t call_cap, int32_t* n_calls);

/* Workspace bytes for pass 0 (forward: attn_fwd and its stages), pass 1
 * (backward: attn_bwd and its stages) or pass 2 (attn_bwd_chunk on exactly
 * these chunks) of this shape and chunk table.
 * Validates like the compute calls. */
int attn_workspace_size(const attn_shape* shape, const attn_chunk* chunks, int32_t n,
                        int32_t pass, size_t* bytes);

/* ---- forward ----------------------------------------------------------- */

/* Forward of every chunk: o (bf16) and lse (fp32) for all rows of the
 * chunks. Chunks must be sorted by q_begin with disjoint query ranges and
 * 0 <= ctx_begin <= q_begin < q_end <= T. Rows outside every chunk are not
 * written. Equivalent to attn_fwd_tiles followed by attn_fwd_merge. */
int attn_fwd(const void* q, const void* k, const void* v,
             const attn_chunk* chunks, int32_t n, const attn_shape* shape,
             void* o, float* lse, void* ws, size_t ws_bytes, void* stream);

/* Stage 1 of the forward: the tile kernel. Rows of unsplit chunks (and rows
 * of split chunks whose tile lies wholly before the first split point) get
 * their final o and lse; the key-range partials of the remaining rows (two
 * for a split at one point, P for kv_split = -P) go to the workspace as
 * fp32. */
int attn_fwd_tiles(const void* q, const void* k, const void* v,
                   const attn_chunk* chunks, int32_t n, const attn_shape* shape,
                   void* o, float* lse, void* ws, size_t ws_bytes, void* stream);

/* Stage 2 of the forward: log-sum-exp merge of the partials of re-split
 * chunks (RSA accumulation over key/value blocks, made exact with LSE):
 * LSE = ln sum_p e^{LSE_p}; O = sum_p e^{LSE_p-LSE} O_p over the parts whose
 * key range starts at or before the row; a partial with LSE = -inf has
 * weight 0. A no-op when no chunk is split. */
int attn_fwd_merge(const attn_chunk* chunks, int32_t n, const attn_shape* shape,
                   void* o, float* lse, void* ws, size_t ws_bytes, void* stream);

/* ---- backward ---------------------------------------------------------- */

/* Gradients of the forward for upstream dout, given the forward's o and lse.
 * The chunk table must partition [0, T) (sorted, contiguous) with every
 * chunk of one document sharing ctx_begin = the document start; the result
 * depends on the documents only, not on where chunks are cut (InfiniPipe
 * §II-A: dK/dV of a token gather contributions of all later tokens).
 * dq, dk, dv are bf16 with the shared strides. Equivalent to
 * attn_bwd_prep, attn_bwd_tiles, attn_bwd_dq in that order. */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dout, const attn_chunk* chunks, int32_t n, const attn_shape* shape,
             void* dq, void* dk, void* dv, void* ws, size_t ws_bytes, void* stream);

/* Stage 1: D_t = sum_d dO_td * O_td (fp32) into the workspace, and zero the
 * fp32 dQ accumulator. */
int attn_bwd_prep(const void* o, const void* dout, const attn_chunk* chunks, int32_t n,
                  const attn_shape* shape, void* ws, size_t ws_bytes, void* stream);

/* Stage 2: one key tile per work item: recompute P = exp(S - LSE), then
 * dV += P^T dO, dS = P o (dO V^T - D), dK += scale dS^T Q (owned, written as
 * bf16) and dQ += scale dS K (fp32 reduction into the workspace). */
int attn_bwd_tiles(const void* q, const void* k, const void* v, const float* lse,
                   const void* dout, const attn_chunk* chunks, int32_t n,
                   const attn_shape* shape, void* dk, void* dv,
                   void* ws, size_t ws_bytes, void* stream);

/* Stage 3: dq = bf16(fp32 dQ accumulator). */
int attn_bwd_dq(const attn_chunk* chunks, int32_t n, const attn_shape* shape,
                void* dq, void* ws, size_t ws_bytes, void* stream);

/* ---- chunk-streamed backward ------------------------------------------- */

/* Backward of the query rows of a set of chunks against their resident
 * contexts, for a caller that runs chunks one call at a time: the forward in
 * chunk order (attn_fwd on the same chunks: their rows attend to the keys
 * [ctx_begin, q_end) already in k, v; SPPO §5.1, the K/V of earlier
 * subsequences stay resident), the backward in reverse order (InfiniPipe
 * §II-A: the K/V gradients of a token gather contributions from every later
 * token, so a chunk's keys are complete once the chunks after it and the
 * chunk itself have run). One call may hold the slices of several documents,
 * such as an InfiniPipe batched or hybrid chunk {C, S} (§III-A1).
 * For each chunk, with query rows t in [q_begin, q_end) (kv_split ignored):
 *   dq rows [q_begin, q_end)                 = their gradient (bf16; complete:
 *                                              every key they see is in the
 *                                              context);
 *   dk_acc, dv_acc rows [ctx_begin, q_end)  += the rows' contributions (fp32,
 *                                              dK including the scale);
 *   dk, dv rows [q_begin, q_end)             = bf16 of the updated accumulators.
 * Other rows of dq, dk, dv, dk_acc, dv_acc are not touched. Chunks: sorted by
 * q_begin, 0 <= ctx_begin <= q_begin < q_end <= T, and key ranges disjoint
 * (each ctx_begin >= the previous chunk's q_end), so that no accumulator row
 * is updated twice by one call. Zero dk_acc and dv_acc over a document before
 * the call holding its last chunk; after the calls holding all of its chunks,
 * in reverse chunk order, dq, dk, dv equal attn_bwd's result for the document.
 * o, lse are the forward's; o and dout are read for the chunks' rows.
 * dk_acc, dv_acc: fp32 device arrays indexed like the bf16 tensors, element
 * (b, t, h, d) at b*sb + t*st + h*sh + d, 16-byte aligned. The workspace comes
 * from attn_workspace_size(pass 2) for the same chunks; calls that share
 * dk_acc/dv_acc rows must run one after another (one stream).
 * Errors: ATTN_E_INVAL (bad shape or chunks, overlapping key ranges, a NULL
 * pointer), ATTN_E_ALIGN, ATTN_E_UNSUPPORTED, ATTN_E_WORKSPACE, ATTN_E_CUDA;
 * device errors through attn_status(ws). */
int attn_bwd_chunk(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   const void* dout, const attn_chunk* chunks, int32_t n, const attn_shape* shape,
                   void* dq, void* dk, void* dv, float* dk_acc, float* dv_acc,
                   void* ws, size_t ws_bytes, void* stream);

/* ---- forward without a caller-provided workspace ----------------------- */

/* Bytes of the scratch area inside the library used by attn_fwd_noalloc. */
#define ATTN_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/* The forward (as attn_fwd) for callers that cannot allocate device memory,
 * e.g. code hosted by a runtime that owns all device memory and offers no
 * allocator, or code that must not allocate once it is running. The pages
 * have no counterpart: this is a convenience of this library.
 * Instead of a workspace argument it uses a scratch area of
 * ATTN_NOALLOC_SCRATCH_BYTES that lives in the library and that every GPU
 * which loads the library holds until the process exits. The caller still
 * passes q, k, v, o and lse; arguments, layouts and errors are as attn_fwd.
 * Returns ATTN_E_WORKSPACE when this shape and chunk table need more forward
 * workspace than ATTN_NOALLOC_SCRATCH_BYTES (attn_workspace_size, pass 0);
 * re-split chunks need fp32 partials, so they reach the limit first.
 * Every call looks up the scratch address in the context current on the
 * calling thread (nothing is cached, so a device reset or another context on
 * the device gets its own address); the first call in a context loads the
 * library's kernels there, so make it before any stream capture. It
 * allocates nothing. All calls share the one scratch area and it keeps the
 * last call's contents (every call rewrites what it reads): calls that
 * overlap on the GPU race with each other, so issue them on one stream, or
 * otherwise one after the other. Device-side errors of this path are read
 * with attn_noalloc_status(). */
int attn_fwd_noalloc(const void* q, const void* k, const void* v,
                     const attn_chunk* chunks, int32_t n, const attn_shape* shape,
                     void* o, float* lse, void* stream);

/* Device error word of attn_fwd_noalloc (its status header lives in the
 * library's scratch area): synchronises `stream`, then reads and clears it,
 * like attn_status() does for a caller workspace. Returns ATTN_OK,
 * ATTN_E_TIMEOUT or ATTN_E_BOUNDS (ATTN_E_CUDA if the read fails). The word
 * is cleared by every attn_fwd_noalloc call when it starts, and is shared by
 * all of them, like the rest of the scratch area. No counterpart on the
 * pages. */
int attn_noalloc_status(void* stream);

/* ---- status ------------------------------------------------------------ */

/* Synchronises `stream`, then reads and clears the device error word in the
 * workspace header: ATTN_OK, ATTN_E_TIMEOUT or ATTN_E_BOUNDS (or ATTN_E_CUDA
 * if the read itself fails). The word lives in the first 256 bytes of the
 * workspace; attn_fwd / attn_fwd_tiles / attn_bwd / attn_bwd_prep / attn_bwd_chunk clear it
 * when they start, and a workspace no such call has used must be zeroed by
 * the caller before its status is read. */
int attn_status(void* ws, void* stream);

/* Static English text for a status code. */
const char* attn_strerror(int status);

/* Library version string, e.g. "libattn 0.1 sm_103a". */
const char* attn_version(void);

/* Number of kernels this library has enqueued, on any stream and device,
 * since it was loaded (a relaxed atomic counter; thread-safe). A compute
 * call enqueues its tile kernels plus one small copy kernel per 31 KB of
 * work list it writes into the workspace. No counterpart on the pages. */
uint64_t attn_kernel_launches(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H_ */
