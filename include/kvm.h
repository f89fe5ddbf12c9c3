/*
 * kvm.h -- C ABI of the per-step working-set recall library (libkvm.so).
 *
 * Sources (page titles, with the section / equation / figure each call follows):
 *   [KVMem] "KVMem: Virtualizing Million-Token Agent Workspaces on a Consumer GPU"
 *   [InfS]  "InferScale: GPU-Native KV Injection for Personalized LLM Serving"
 *
 * One process, one GPU (sm_103a).  Every buffer is allocated by the caller and
 * must outlive the calls that use it; the library never allocates or frees
 * device memory and never frees caller memory.  A buffer that a call's kernels
 * read or write may be device memory or pinned (page-locked) host memory; the
 * kernels then access pinned host memory directly over the host link, moving
 * only the bytes they touch.  Pageable host memory is rejected
 * (KVM_ERR_INVALID_ARG).  The one exception is the Mean-K index read by
 * kvm_score_select: with index_location KVM_DEVICE it must be device memory
 * (TMA streams it), and with KVM_HOST_PINNED it is pinned host memory staged
 * in tiles.  All work is enqueued on the caller's stream;
 * functions return after enqueueing unless stated otherwise.  No C++
 * exception crosses this boundary: every function returns a kvm_status.
 * Argument errors are detected on the host before anything is enqueued and
 * leave the context unchanged.  Device-side range checks (block ids, page ids)
 * skip the offending access and raise a sticky device error flag that
 * kvm_sync() reports as KVM_ERR_DEVICE and clears.
 * One context's calls share its workspace (scoring scratch, step descriptors,
 * page table) and its host bookkeeping: issue them on one stream, or order
 * the streams yourself (an event per call).  Two calls of one context that
 * run at the same time on unordered streams race.  Different contexts are
 * independent and may run concurrently on different streams and threads.
 *
 * Layouts (row-major, innermost last; B = block_tokens = 32, d = head_dim):
 *   K pages, V pages, raw K, V      [block or page][layer][kv_head][B][d]
 *   Mean-K index                     [layer][kv_head][max_blocks][d]
 *   RoPE-free queries                [layer][query][q_head][d]
 *   block relevance (scores)         [n_blocks] float32
 * Block b of the history holds tokens 32b .. 32b+31 (its original range);
 * view slot j holds compact positions 32j .. 32j+31.
 * RoPE pairs coordinate i with i + d/2 (rotate-half); the angle of pair i
 * at position p is p * theta^(-2i/d), evaluated in double precision and
 * rounded once to a float32 cos/sin table.
 */
#ifndef KVM_H_
#define KVM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t.  NULL means the legacy default stream. */
typedef struct CUstream_st *kvm_stream;

typedef enum {
    KVM_OK = 0,
    KVM_ERR_INVALID_ARG = -1,          /* bad pointer, size, dtype or config field     */
    KVM_ERR_WORKSPACE_TOO_SMALL = -2,  /* workspace smaller than kvm_workspace_bytes() */
    KVM_ERR_CAPACITY = -3,             /* n_blocks / queries / pages beyond the config */
    KVM_ERR_CUDA = -4,                 /* a CUDA runtime call failed (see kvm_last_error) */
    KVM_ERR_TIMEOUT = -5,              /* a bounded device wait gave up               */
    KVM_ERR_NOT_BOUND = -6,            /* kvm_step before kvm_bind                    */
    KVM_ERR_INJECTED = -7,             /* failure raised by kvm_debug_inject          */
    KVM_ERR_DEVICE = -8                /* a device-side range check fired             */
} kvm_status;

/* Element types.  KVM_E4M3 is 8-bit floating point (1 sign, 4 exponent bits
 * with bias 7, 3 mantissa bits; no infinity, S.1111.111 is NaN; largest
 * finite value 448), the FP8 KV cache of the [KVMem] §6.1 platforms.  It is
 * for kv_dtype only, stored at unit scale; values written by the library are
 * rounded to nearest even and saturate to +-448. */
enum { KVM_F32 = 0, KVM_BF16 = 1, KVM_E4M3 = 2 };
enum { KVM_DEVICE = 0, KVM_HOST_PINNED = 1 };    /* where a buffer lives     */

/* Shapes and budgets of one workspace.  All fields are required. */
typedef struct {
    int32_t n_layers;        /* L: scored attention layers                     */
    int32_t n_kv_heads;      /* G                                              */
    int32_t n_q_heads;       /* H, a multiple of G (grouped-query attention)   */
    int32_t head_dim;        /* d: 64 or 128                                   */
    int32_t block_tokens;    /* must be 32 ([KVMem] §4.3 default block size)   */
    double  rope_theta;      /* RoPE base                                      */
    int32_t kv_dtype;        /* K pages, raw K, V: KVM_F32, KVM_BF16, KVM_E4M3 */
    int32_t index_dtype;     /* Mean-K entries                                 */
    int32_t q_dtype;         /* queries                                        */
    int32_t sink_blocks;     /* S: always-kept leading blocks                  */
    int32_t recent_blocks;   /* W: always-kept trailing blocks                 */
    int32_t view_blocks;     /* V_b: execution-view budget, >= S + W + 1       */
    int32_t max_queries;     /* largest M_q accepted                           */
    int64_t max_blocks;      /* index capacity and largest history N           */
    int64_t max_positions;   /* RoPE table rows: > every token position used   */
    int32_t tile_blocks;     /* index tile for host-resident scoring ([KVMem] §5) */
    int32_t pool_pages;      /* pages of the kvm_step page pool (>= view_blocks) */
    int32_t index_location;  /* KVM_DEVICE or KVM_HOST_PINNED (kvm_step, kvm_score_select) */
    int32_t repo_location;   /* where kvm_step finds raw K / V of the history  */
    int32_t h2d_batch_blocks;/* missed blocks per pipelined H2D batch (kvm_step) */
    int32_t h2d_mode;        /* kvm_step with a host-resident repository:
                                0: copy engine -- coalesced cudaMemcpyAsync of each run of
                                   missed blocks into its pages, batch by batch;
                                1: the GPU reads the missed blocks from the pinned host
                                   repository itself (one fused kernel: raw K, re-RoPE'd K
                                   and V into the page); needs the repository pinned and
                                   device-mapped */
    int32_t score_variant;   /* 0: tcgen05 tensor cores for bf16 q/index (d 64 or 128,
                                <= 256 query rows per KV head), CUDA cores otherwise;
                                1: CUDA cores always;
                                2: as 0, with both softmax passes over a device index
                                in one persistent launch (<= 192 query rows per KV
                                head; the second pass reads each (layer, kv head)
                                slice again from L2) */
    int32_t delta_rerope_limit; /* kvm_step, hits whose slot moved ([KVMem] §4.4 bounded
                                delta re-RoPE): 0 = rebuild K from raw K every time;
                                n > 0 = rotate the page's K in place by the position
                                change, at most n times in a row, then rebuild from raw K.
                                Each delta adds at most one rounding of the pair's
                                magnitude, so n bounds the error growth. */
    int32_t candidate_mode;  /* the candidate set C of Eq. (10) ([KVMem] §4.3):
                                0 = every indexed block (the softmax of each query
                                row covers all N blocks; sink and recent blocks are
                                only kept out of the top-k fill);
                                1 = only the blocks the selector may still choose,
                                [sink_blocks, N - recent_blocks): the softmax covers
                                those, and sink / recent blocks score 0. */
    int64_t host_tier_blocks;/* 0 = off; else kvm_step keeps a host-tier policy
                                (see kvm_tier_step) over at most this many
                                blocks, >= view_blocks, fed with every step's
                                selection, and reports its hits / misses */
    double  host_tier_lambda;/* the policy's decay, in [0, 1]              */
    int32_t index_spill;     /* host-resident index ([KVMem] §5 tiled retrieval):
                                0 = both scoring passes stream the index tiles over the
                                    host link, through two tile-sized device buffers;
                                1 = pass 1 keeps every staged tile in device memory
                                    (the workspace then holds a copy of the whole
                                    index) and pass 2 reads it there, so each step
                                    moves the index over the link once. */
    int32_t spill_tiles;     /* with index_spill = 1: 0 = keep every tile; m > 0 =
                                keep at most m tiles (the last m of pass 1), which
                                pass 2 scores first while the other tiles cross the
                                link again through the two streaming buffers.  The
                                workspace then holds m + 2 tiles, and a step moves
                                (2T - min(m, T)) / T index reads over the link for T
                                tiles.  Results do not depend on m. */
} kvm_config;

typedef struct kvm_ctx kvm_ctx;

/* Device workspace bytes a context needs for `cfg` (RoPE table, scoring
 * scratch including that of the one-launch variant, a copy of the queries for
 * a device index when they are passed in host memory, index staging tiles --
 * two, one per index tile with index_spill, or spill_tiles + 2 -- step
 * descriptors and the
 * device-side residency of the page pool).  0 if cfg is invalid. */
size_t kvm_workspace_bytes(const kvm_config *cfg);

/* Create a context.  `workspace` is caller-owned device memory of at least
 * kvm_workspace_bytes(cfg) bytes, 256-byte aligned, used exclusively by this
 * context until kvm_destroy.  Fills the RoPE cos/sin table on `stream`
 * ([KVMem] §4.4: precomputed sine/cosine tables).  *out receives the context. */
kvm_status kvm_create(const kvm_config *cfg, void *workspace, size_t workspace_bytes,
                      kvm_stream stream, kvm_ctx **out);

kvm_status kvm_destroy(kvm_ctx *ctx);

/*
 * (a) Mean-K index build -- [KVMem] §4.3 (Mean-K block representation) and §5
 * (incremental indexing while K is still resident on the GPU).
 *
 * For blocks b = first_block .. first_block + n_blocks - 1:
 *   raw K of token p = R_{-p} K_pages[b - first_block][l][g][t]   (p = 32b + t)
 *   index[l][g][b]   = (1/32) * sum_t raw K                      (float32 sums)
 * k_pages  device, [n_blocks][L][G][32][d], kv_dtype, K rotated at original positions.
 * index    device, [L][G][max_blocks][d], index_dtype; entries [first_block,
 *          first_block + n_blocks) are written, others untouched.
 * raw_k_out nullable device, [n_blocks][L][G][32][d], kv_dtype: the
 *          position-independent raw K (float32 rotation, rounded once).
 * Errors: KVM_ERR_CAPACITY if first_block + n_blocks > max_blocks or the
 * positions exceed max_positions; KVM_ERR_INVALID_ARG on NULL inputs.
 */
kvm_status kvm_build_index(kvm_ctx *ctx, const void *k_pages, int64_t first_block,
                           int64_t n_blocks, void *index, void *raw_k_out, kvm_stream stream);

/*
 * (b) Query-conditioned block scoring, Eq. (10) of [KVMem] §4.3, and the
 * default selector (sink + recent + top-k, chronological order).
 *
 *   s[l,m,h,b] = q[l,m,h] . index[l, g(h), b] / sqrt(d),  g(h) = h / (H/G)
 *   R_b = 1/(L*H) * sum_{l,h} sum_m softmax_b(s[l,m,h,:])[b]
 * over all n_blocks indexed blocks (the softmax is global over blocks, also
 * when the index is scored tile by tile from host memory, [KVMem] §5).
 * Selection: blocks [0,S) and [N-W,N) always; the other V_b-S-W slots go to
 * the largest R_b (ties: lower block id; NaN last); output ascending.  If
 * N <= V_b every block is selected.
 *
 * q         device, [L][n_queries][H][d], q_dtype (RoPE-free queries); with
 *           score_variant 2 and a device index, queries in pinned host memory
 *           are first copied into the workspace (the one-launch kernel reads
 *           them by TMA from device memory).
 * index     [L][G][max_blocks][d], index_dtype; device memory when
 *           cfg.index_location == KVM_DEVICE, pinned host memory when
 *           KVM_HOST_PINNED (then scored in tiles of tile_blocks staged on the GPU).
 * scores_out   device, [n_blocks] float32: R_b.
 * sel_ids_out  device, [view_blocks] int32: selected ids, ascending; the
 *              first min(N, V_b) entries are written.
 * n_sel_out    nullable HOST int32: receives min(N, V_b).
 * Errors: KVM_ERR_CAPACITY if n_blocks > max_blocks or n_queries > max_queries;
 * KVM_ERR_INVALID_ARG if n_blocks < 1 or n_queries < 1.
 */
kvm_status kvm_score_select(kvm_ctx *ctx, const void *q, int32_t n_queries, const void *index,
                            int64_t n_blocks, float *scores_out, int32_t *sel_ids_out,
                            int32_t *n_sel_out, kvm_stream stream);

/*
 * (c) Chronological execution-view assembly -- [KVMem] §4.4 (view
 * separation: RoPE applied to raw K at the block's compact position, V copied
 * unchanged) and [InfS] Theorem 6 (re-rotation at a new position).
 *
 * For slot j < n_sel, with b = sel_ids[j] and page p = page_ids ? page_ids[j] : j:
 *   k_pages[p][l][g][t] = R_{32j+t} raw_k_repo[b][l][g][t]   (float32, rounded once)
 *   v_pages[p]          = v_repo[b]                           (byte copy)
 * sel_ids, page_ids   device int32 [n_sel] (page_ids nullable).
 * raw_k_repo, v_repo  device, [>= max id + 1][L][G][32][d], kv_dtype.
 * k_pages, v_pages    device, [>= max page + 1][L][G][32][d]; v_repo and
 *                     v_pages may both be NULL to skip the V copy.
 * Ids >= max_blocks or pages < 0 are skipped and raise the device error flag.
 */
kvm_status kvm_assemble_view(kvm_ctx *ctx, const int32_t *sel_ids, const int32_t *page_ids,
                             int32_t n_sel, const void *raw_k_repo, const void *v_repo,
                             void *k_pages, void *v_pages, kvm_stream stream);

/* Buffers used by kvm_step (bound once with kvm_bind). */
typedef struct {
    const void *index;   /* [L][G][max_blocks][d]; device or pinned host (index_location) */
    const void *raw_k;   /* history raw K [max_blocks][L][G][32][d]; device or pinned host (repo_location) */
    const void *v;       /* history V, same layout and location as raw_k */
    void *pool_k;        /* device [pool_pages][L][G][32][d]: K at compact positions */
    void *pool_v;        /* device [pool_pages][L][G][32][d]                         */
    void *pool_raw_k;    /* device [pool_pages][L][G][32][d]: each page's raw K;
                            required when repo_location == KVM_HOST_PINNED, else NULL */
    int32_t *page_table; /* device [view_blocks]: page of each view slot             */
    float *scores;       /* device [max_blocks]: R_b of the last step                */
    int32_t *sel_ids;    /* device [view_blocks]: selected ids of the last step      */
} kvm_buffers;

kvm_status kvm_bind(kvm_ctx *ctx, const kvm_buffers *bufs);

/*
 * Proactive stage-out -- [KVMem] §4.4: once a prefill chunk completes, the KV
 * of its completed blocks is copied to host memory asynchronously while the GPU
 * processes the next chunk, so that outgoing blocks already have host copies
 * when the working set changes (and §5: incremental indexing of the same
 * blocks with kvm_build_index while their K is still on the GPU).
 *
 * Copies raw K and V of blocks first_block .. first_block + n_blocks - 1 from
 * the device buffers raw_k and v (each [n_blocks][L][G][32][d], kv_dtype; raw_k
 * is typically kvm_build_index's raw_k_out) into the bound host repository
 * (kvm_bind's raw_k / v; requires repo_location == KVM_HOST_PINNED).  The
 * copies run on the context's copy stream after everything already enqueued
 * on `stream`, so work enqueued on `stream` afterwards overlaps them.  raw_k
 * and v must stay unchanged until the copies are done: kvm_sync waits for
 * them, and every later kvm_step orders its reads of the repository after them.
 * Errors: KVM_ERR_NOT_BOUND, KVM_ERR_INVALID_ARG (no host repository, NULL
 * buffers, or `stream` being captured into a CUDA graph), KVM_ERR_CAPACITY
 * (blocks beyond max_blocks).
 */
kvm_status kvm_stage_out(kvm_ctx *ctx, const void *raw_k, const void *v, int64_t first_block,
                         int64_t n_blocks, kvm_stream stream);

/* Forget which blocks the page pool holds (every page empty). */
kvm_status kvm_reset_pool(kvm_ctx *ctx);

typedef struct {
    int64_t n_blocks;     /* history blocks scored                     */
    int32_t n_sel;        /* view slots filled                         */
    int32_t hits;         /* selected blocks already held by a page    */
    int32_t misses;       /* selected blocks brought in (L_t^physical) */
    int32_t reroped;      /* slots whose K was (re)written             */
    int32_t evicted;      /* pages whose block left the pool           */
    int32_t h2d_copies;   /* host-to-device copies issued              */
    int64_t h2d_bytes;    /* bytes moved host to device               */
    int32_t delta_reroped;/* hits rotated in place by their position change */
    int32_t host_hits;    /* with host_tier_blocks: selected blocks in the host tier */
    int32_t host_misses;  /* ... and not in it (reads from the next tier)           */
    int32_t host_demoted; /* ... blocks the host tier demoted in this step          */
} kvm_step_stats;

/*
 * (d) One working-set update: score + select (b), then the delta working set
 * of [KVMem] §4.4: hits keep their page, misses (L_t^physical) take free pages
 * in ascending order, the page table maps view slots to pages.  Misses are
 * fetched from the repository: device-to-device inside the assembly kernel
 * when repo_location == KVM_DEVICE; with coalesced host-to-device copies of
 * raw K and V in batches of h2d_batch_blocks on an internal copy stream,
 * each batch re-RoPE'd by the GPU after its copy event (the three-stage
 * pipeline of [KVMem] §4.4, Figure 3) when KVM_HOST_PINNED.  Hits whose slot
 * changed are re-RoPE'd from raw K (the page's raw-K copy when pool_raw_k is
 * bound, else the repository), or rotated in place by the position change
 * under delta_rerope_limit.  pool_raw_k may be NULL unless the repository is
 * host-resident with h2d_mode 0.
 * Where the GPU reads the repository itself (repo_location == KVM_DEVICE, or
 * KVM_HOST_PINNED with h2d_mode 1) and no host-tier policy runs, the residency
 * diff (hits, misses, free pages, the page table, the assembly descriptors) is
 * a kernel over residency kept in the workspace: the step waits for nothing and
 * returns with all of its work enqueued on `stream`, and `stats` (nullable,
 * host) is filled by the next kvm_sync, so it must stay valid until then.
 * Otherwise (copy-engine transfers, which the host issues per run of missed
 * blocks, or a host-tier policy fed with the selection) the step synchronises
 * with `stream` once to read the selected ids, diffs on the host, returns with
 * the rest enqueued and fills `stats` before returning.  Both diffs give the
 * same pages.  kvm_bind and kvm_reset_pool empty the pool; they must not be
 * called while another thread enqueues a step on the same context.
 * CUDA graphs: a step with the residency diff on the device and the index in
 * device memory may be enqueued while `stream` is being captured; each launch
 * of the graph then runs one step on the query buffer `q` as it holds at
 * launch time, against the residency as the steps before it left it.  Such a
 * step takes stats = NULL (kvm_graph_step_stats reads the counters of the
 * last one that ran), waits at every
 * launch for the latest kvm_reset_pool and kvm_stage_out, and a later
 * kvm_reset_pool orders its clearing after the launches already enqueued.
 * Steps, eager or launched from graphs, must follow one another on one stream.
 * A graph keeps the buffers bound at capture time: after kvm_bind, capture
 * again.
 * Errors under capture: KVM_ERR_INVALID_ARG when the diff runs on the host,
 * the index is host-resident, or stats is not NULL; nothing is enqueued then.
 */
kvm_status kvm_step(kvm_ctx *ctx, const void *q, int32_t n_queries, int64_t n_blocks,
                    kvm_step_stats *stats, kvm_stream stream);

/*
 * Host-tier admission and eviction of repository blocks ([KVMem] §4.4,
 * retrieval-aware hierarchical reuse).  Host memory keeps at most
 * capacity_blocks blocks.  Admission and eviction weigh both recent and
 * cumulative retrieval.  The pages give no formula; the policy is LRFU (Lee et
 * al., IEEE Transactions on Computers 50(12), 2001):
 *
 *     CRF_t(b) = sum over b's references t_i of 2^(-lambda * (t - t_i))
 *
 * with lambda in [0, 1] (0 = reference counts, 1 = most recent use).
 *
 * Each kvm_tier_step is one agent step:
 * - first, blocks [previous n_blocks, n_blocks) are created: their K / V reach
 *   host memory by stage-out, so they become resident with one reference;
 * - then the `ids` (distinct, the step's selected blocks) count one reference
 *   each; a selected block that is not resident is a host miss (in a full
 *   system, a read from the next tier) and becomes resident;
 * - while more than capacity_blocks blocks are resident, the resident
 *   unselected block with the smallest CRF_t is demoted (ties: the lower id
 *   first).
 *
 * demoted_out (nullable, host, room for n_blocks ids) receives the demoted ids
 * in demotion order.  Host-only bookkeeping: no device memory, no stream.  The
 * next tier itself (NVMe) is not part of this library.
 * Errors: KVM_ERR_INVALID_ARG for a bad capacity or lambda, ids out of range or
 * repeated, or a shrinking history.  On error the tier is unchanged.
 */
typedef struct kvm_tier kvm_tier;
typedef struct {
    int32_t hits;       /* selected blocks already host-resident         */
    int32_t misses;     /* selected blocks that were not                 */
    int32_t demoted;    /* blocks demoted in this step                   */
    int64_t resident;   /* host-resident blocks after the step           */
} kvm_tier_stats;
kvm_status kvm_tier_create(int64_t capacity_blocks, double lambda, kvm_tier **out);
kvm_status kvm_tier_step(kvm_tier *tier, const int32_t *ids, int32_t n_ids, int64_t n_blocks,
                         int32_t *demoted_out, kvm_tier_stats *stats);
/* flags[b] = 1 if block b is host-resident, for b < n (host buffer). */
kvm_status kvm_tier_resident(const kvm_tier *tier, uint8_t *flags, int64_t n);
kvm_status kvm_tier_destroy(kvm_tier *tier);

/*
 * kvm_score_select without any device allocation: KVMem has no
 * counterpart; this is a deployment convenience.
 *
 * Computes what kvm_score_select computes for a device-resident index, with
 * the same kernels and the same chunking, so scores and selection are bit
 * for bit those of kvm_score_select on the same inputs.  It needs no context
 * and no workspace: its scratch is a fixed 32 MiB array in the library's own
 * device memory.  It is meant for callers that cannot allocate device memory
 * -- for example a plugin inside an inference engine whose memory planner
 * already owns the whole device, or a latency-critical caller that cannot
 * afford cudaMalloc/cudaFree, which may synchronise the device.  The call
 * allocates nothing (no cudaMalloc, no cudaFree, no allocating library
 * routine).
 *
 * cfg      host; the shape fields, dtypes, sink/recent/view budget,
 *          candidate_mode, score_variant and max_blocks (the index row
 *          stride) are used; index_location must be KVM_DEVICE.
 * index    device memory (checked: KVM_ERR_INVALID_ARG otherwise).
 * q, scores_out, sel_ids_out
 *          device memory or pinned host memory (checked as for
 *          kvm_score_select; pageable memory gives KVM_ERR_INVALID_ARG).
 *          n_sel_out is a host pointer, as for kvm_score_select.
 * Limit:   the scratch needs about 4 * L * G * n_blocks bytes (plus a little
 *          per query row); calls needing more than 32 MiB return
 *          KVM_ERR_CAPACITY with a message, before any work is enqueued.
 * Set-up:  the first call in each CUDA context (normally: on each device)
 *          looks up the array's device address (cudaGetSymbolAddress) with
 *          that context current; make that first call before any stream
 *          capture.  The address is kept for the life of the process, so do
 *          not call this entry point on a device after cudaDeviceReset of it.
 * Errors on the device: a bounded wait that gave up inside a tensor-core pass
 *          raises a flag in the array's error word; the call itself has
 *          already returned KVM_OK by then.  The word collects the flags of
 *          every call until kvm_score_select_static_status reads and clears
 *          it.  A call whose flag was raised left meaningless scores and
 *          selection (ids stay in range).
 * Sharing: every call on a device uses the same array.  Calls that overlap on
 *          the GPU (unordered streams or threads) race on it; order them.
 *          The array keeps the last call's contents; a call never reads
 *          them: the part that must start at zero (the histograms of the
 *          selection over 16384 or more blocks) is cleared on the call's
 *          stream first, and the rest is overwritten before it is read.
 * The array stays allocated on every GPU that loaded the library until the
 * process exits.
 */
kvm_status kvm_score_select_static(const kvm_config *cfg, const void *q, int32_t n_queries,
                                   const void *index, int64_t n_blocks, float *scores_out,
                                   int32_t *sel_ids_out, int32_t *n_sel_out, kvm_stream stream);

/*
 * The device errors of kvm_score_select_static calls in the current CUDA
 * context: waits for `stream` (the stream of those calls), reads the error
 * word of the fixed array, and clears it.  Returns KVM_OK when no flag was
 * raised since the last read, KVM_ERR_TIMEOUT when a bounded wait gave up,
 * KVM_ERR_DEVICE for any other flag, KVM_ERR_CUDA when the word cannot be
 * read.  Allocates nothing.  Synchronises with `stream`.
 */
kvm_status kvm_score_select_static_status(kvm_stream stream);

/* Wait for all work of the context (its internal streams and `stream`) and
 * report a raised device error flag (KVM_ERR_DEVICE), clearing it. */
kvm_status kvm_sync(kvm_ctx *ctx, kvm_stream stream);

/*
 * The counters of the last kvm_step launched from a CUDA graph on this context
 * (steps captured under stream capture report none through kvm_step; every
 * captured step of the context writes the same slot, so this is the step that
 * ran last).  Waits for `stream` (the stream the graph was launched on), then
 * fills *stats (host) as kvm_sync fills an eager step's, with n_blocks and
 * n_sel as given at capture time.  Errors: KVM_ERR_INVALID_ARG (NULL
 * arguments, or no step of this context was captured), KVM_ERR_CUDA.
 */
kvm_status kvm_graph_step_stats(kvm_ctx *ctx, kvm_step_stats *stats, kvm_stream stream);

const char *kvm_status_string(kvm_status s);

/* Detail of the last error raised on the calling thread ("" if none). */
const char *kvm_last_error(void);

/* Kernels this library has launched in the process so far, over every
 * context and entry point (a running total, for benchmarks and tests: the
 * difference across a region is the number of kernels it launched).  Copies
 * and memsets are not kernels and are not counted. */
int64_t kvm_launch_count(void);

/*
 * Page-locked host memory of exactly `bytes` bytes, for the buffers a caller
 * hands the library in host memory (the raw K / V repository, a host-resident
 * index).  A convenience for callers: the library itself never allocates.  The
 * memory is portable (usable from every context) and mapped (kernels address
 * it through its device alias), and the CUDA driver allocates it.  Measured on
 * GB300 with a 148 GB repository, the GPU reads scattered blocks of it over
 * the host link at the full pinned-copy rate; from ordinary host memory
 * registered after allocation it read at 0.48-0.93 of that rate, depending on
 * how the pages happened to be laid out.
 * out      host; receives the pointer (NULL on failure).
 * Errors:  KVM_ERR_INVALID_ARG for bytes == 0 or out == NULL; KVM_ERR_CUDA if
 *          the driver cannot allocate (kvm_last_error has its message).
 * Free with kvm_host_free once no copy or kernel uses the memory.
 */
kvm_status kvm_host_alloc(size_t bytes, void **out);
kvm_status kvm_host_free(void *ptr);

/* Fault injection for tests.  what = 1 / 2: make the n-th (1-based) next host
 * copy submission / kernel launch of kvm_step fail with KVM_ERR_INJECTED.
 * what = 3: the n-th next tensor-core scoring pass (kvm_score_select or
 * kvm_step; passes 1 and 2 both count) runs with its TMA producer idle, so
 * its bounded device waits run out after about a second each; the call
 * itself returns KVM_OK and the next kvm_sync returns KVM_ERR_TIMEOUT.  Its
 * scores and selection are then meaningless (ids stay in range).  what = 0
 * clears.  The context stays usable in every case. */
kvm_status kvm_debug_inject(kvm_ctx *ctx, int32_t what, int64_t nth);

#ifdef __cplusplus
}
#endif

#endif /* KVM_H_ */
