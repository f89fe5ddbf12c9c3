// Internal declarations shared by the kernels and the host runtime of libkvm.
// Layouts and semantics are those of include/kvm.h.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

namespace kvm {

// Sets the message kvm_last_error() returns on the calling thread.
void set_last_error(const std::string &msg);

// Counts one kernel launch of this library (read by kvm_launch_count).
void note_launch();

// The address a kernel uses for a caller buffer: device (or managed) memory as
// is, pinned host memory through its device alias; NULL stays NULL.  Pageable
// host memory and addresses the GPU cannot use are rejected.  Returns a
// kvm_status value (KVM_OK, KVM_ERR_INVALID_ARG or KVM_ERR_CUDA) and sets the
// last-error message.  Defined in kvm_api.cpp.
int resolve_kernel_ptr(const void *p, const void **out, const char *what);

constexpr int kBlockTokens = 32;
constexpr int kMaxHalfDim = 64;       // head_dim <= 128
constexpr int kMaxRows = 256;         // query rows per KV head (M_q * H/G)
constexpr int kMaxChunks = 64;        // block chunks per (layer, kv head) in scoring
constexpr int kFusedMaxRows = 192;    // query rows per KV head the one-launch scoring takes
constexpr int kFusedMaxCtas = 256;    // CTAs of one one-launch scoring grid, at most

enum DType { F32 = 0, BF16 = 1, E4M3 = 2 };

struct Omega {
    double w[kMaxHalfDim];            // theta^(-2i/d), double precision
};

// One view slot to (re)materialise: K = RoPE(src_k, pos0 + t) into dst_k, and
// optionally V copied from src_v to dst_v.  Pointers address one whole block
// ([L][G][32][d]).
struct SlotDesc {
    const void *src_k;
    const void *src_v;
    void *dst_k;
    void *dst_v;
    void *dst_raw;      // nullable: also store the raw K as read (a page's raw-K copy)
    int64_t pos0;       // first position; with kSlotDelta: the position change delta
    int32_t flags;      // kSlotDelta: rotate the K in place by pos0 (same angle per token)
};
constexpr int32_t kSlotDelta = 1;

struct ScoreShape {
    int L, G, H, d, n_queries;
    int gqa;            // H / G
    int rows;           // n_queries * gqa: query rows that read one KV head
    int64_t index_cap;  // row stride (in blocks) of the index buffer being read
    int chunk_cap;      // chunk stride of the (max, sum) scratch per (layer, kv head)
    int variant;        // 0: tensor cores where supported, 1: CUDA cores
    int idle_producer;  // 1: a tensor-core pass's TMA producer issues nothing, so
                        // that its bounded waits run out (failure-detection tests)
};

// ---- rope_table.cu
cudaError_t launch_rope_table(float2 *table, int64_t n_pos, int half_d, const Omega &om,
                              cudaStream_t s);

// ---- meank.cu
cudaError_t launch_meank(int kv_dtype, int index_dtype, int d, const void *k_pages,
                         void *raw_out, void *index, int64_t index_cap, int64_t first_block,
                         int64_t n_blocks, int LG, const float2 *table, int *err,
                         cudaStream_t s);

// ---- assemble.cu
// Slots given by (sel_ids, page_ids) against repository / page base pointers.
cudaError_t launch_assemble_ids(int kv_dtype, int d, const int32_t *sel_ids,
                                const int32_t *page_ids, int n_sel, int64_t max_blocks,
                                const void *raw_k_repo, const void *v_repo, void *k_pages,
                                void *v_pages, int LG, const float2 *table, int64_t max_pos,
                                int *err, cudaStream_t s);
// Slots given by explicit descriptors (device array).
cudaError_t launch_assemble_desc(int kv_dtype, int d, const SlotDesc *desc, int n_desc, int LG,
                                 const float2 *table, int64_t max_pos, int *err,
                                 cudaStream_t s);
// The same with the descriptor count in device memory (*n_dev <= n_max).
cudaError_t launch_assemble_desc_dev(int kv_dtype, int d, const SlotDesc *desc, int n_max,
                                     const int32_t *n_dev, int LG, const float2 *table,
                                     int64_t max_pos, int *err, cudaStream_t s);

// ---- residency.cu
// One kvm_step's residency diff on the device (the delta working set): reads
// the selection, writes the page table, the assembly descriptors (count in
// counts[0]) and the new residency; counts[1..4] = hits, misses, delta
// rotations, evicted blocks.  Residency arrays are int32, -1 = none.
struct ResidencyArgs {
    const int32_t *sel;        // [n_sel] selected block ids
    int n_sel;
    int32_t *page_of_block;    // [max_blocks]
    int32_t *block_of_page;    // [P]
    int32_t *baked_pos;        // [P] first token position of the K in the page
    int32_t *delta_count;      // [P] delta rotations since the page's K was rebuilt
    int32_t *stamp;            // [max_blocks] epoch of the last step that selected it
    int32_t *epoch;            // the last step's epoch; the kernel counts it up
    int P;
    int64_t max_blocks;
    int delta_limit;
    int32_t *page_table;       // [n_sel] out
    SlotDesc *desc;            // [n_sel] out
    int32_t *counts;           // [8] out
    int32_t *slot_page;        // [n_sel] scratch
    int32_t *free_list;        // [P] scratch
    char *pool_k, *pool_v, *pool_raw;    // pool_raw may be NULL
    const char *repo_k, *repo_v;         // repository as the GPU addresses it
    size_t blk;                // bytes of one block ([L][G][32][d])
    int pull;                  // host repository read by the GPU (keep raw K in the page)
    int *err;
};
cudaError_t launch_residency_diff(const ResidencyArgs &a, cudaStream_t s);

// ---- score.cu
// Scratch for one scoring call (device pointers inside the workspace).
struct ScoreScratch {
    float *part_m;     // [LG][chunk_cap][rows]  running max (log2 units)
    float *part_z;     // [LG][chunk_cap][rows]  partition sum at part_m
    float *row_m;      // [LG][rows]
    float *row_invz;   // [LG][rows]
    float *partial;    // [LG][max_blocks]   per-(layer, kv head) relevance
    int *err;          // device error flag (bit 4: a bounded wait gave up)
    // one-launch scoring, two slices deep: per-CTA row statistics, per-group
    // row offsets o = M + log2 Z, and two arrival counters per CTA group
    // (cleared by the launcher)
    float2 *fpart;     // [kFusedMaxCtas][2][rows]  (max, sum) of a CTA's share
    float *fo;         // [kFusedMaxCtas][2][rows]
    int *fcnt;         // [2][kFusedMaxCtas]
};

// Bytes of the one-launch scoring scratch (fpart, fo, then fcnt) for up to
// `rows` query rows per KV head; fused_scratch_carve sets the three pointers.
inline size_t fused_scratch_bytes(int rows) {
    return (size_t)kFusedMaxCtas * 2 * rows * (sizeof(float2) + sizeof(float)) +
           (size_t)2 * kFusedMaxCtas * sizeof(int);
}
inline void fused_scratch_carve(ScoreScratch *s, void *base, int rows) {
    char *b = static_cast<char *>(base);
    s->fpart = reinterpret_cast<float2 *>(b);
    b += (size_t)kFusedMaxCtas * 2 * rows * sizeof(float2);
    s->fo = reinterpret_cast<float *>(b);
    b += (size_t)kFusedMaxCtas * 2 * rows * sizeof(float);
    s->fcnt = reinterpret_cast<int *>(b);
}

// Pass 1 over blocks [b_begin, b_end) of the index (rows of `index` addressed
// relative to b_index0), writing chunks [chunk0, chunk0 + n_chunks).
// True where the passes of a call run on the tensor-core kernels.
bool score_uses_tc(int q_dtype, int index_dtype, const ScoreShape &sh);
cudaError_t launch_score_pass1(int q_dtype, int index_dtype, const ScoreShape &sh,
                               const void *q, const void *index, int64_t b_index0,
                               int64_t b_begin, int64_t b_end, int chunk0, int n_chunks,
                               const ScoreScratch &scr, cudaStream_t s);
cudaError_t launch_score_combine(const ScoreShape &sh, int n_chunks_total,
                                 const ScoreScratch &scr, cudaStream_t s);
cudaError_t launch_score_pass2(int q_dtype, int index_dtype, const ScoreShape &sh,
                               const void *q, const void *index, int64_t b_index0,
                               int64_t b_begin, int64_t b_end, int n_chunks,
                               const ScoreScratch &scr, int64_t partial_stride,
                               cudaStream_t s);
// Scores of [0, n_blocks): the partial sums over (l, g) for [c0, c1), 0 elsewhere.
cudaError_t launch_score_reduce(const ScoreShape &sh, int64_t n_blocks, int64_t c0, int64_t c1,
                                const ScoreScratch &scr, int64_t partial_stride,
                                float *scores_out, cudaStream_t s);
// Number of chunks used for a range of n blocks.
int score_chunks(const ScoreShape &sh, int64_t n_blocks, int max_chunks);

// One-launch tensor-core scoring (score_fused.cu): both passes over a
// device-resident bf16 index in one persistent cooperative launch, for the
// candidate blocks [c0, c1); writes scr.partial like pass 2.  Supported for
// bf16 queries and index, d = 64 or 128 and at most kFusedMaxRows query rows
// per KV head, with the queries in device memory (fused_q_ok: TMA reads them).
// sh.idle_producer: bit 0 / bit 1 keep the TMA producer from loading pass-1 /
// pass-2 tiles (failure-detection tests).
bool score_fused_supported(int q_dtype, int index_dtype, const ScoreShape &sh);
bool fused_q_ok(const void *q);
cudaError_t launch_score_fused(const ScoreShape &sh, const void *q, const void *index,
                               int64_t c0, int64_t c1, const ScoreScratch &scr,
                               int64_t partial_stride, cudaStream_t s);

// ---- select.cu
// Device scratch of one selection (histograms and segment counts); fixed size.
size_t select_scratch_bytes();
// sel_ids <- the selection over scores [0, n_blocks); `scratch` is device
// memory of select_scratch_bytes(), used by long histories only.
cudaError_t launch_select(const float *scores, int64_t n_blocks, int sink, int recent,
                          int view_blocks, int32_t *sel_ids, int *scratch, cudaStream_t s);

// Multiprocessors of the current device (152 where it cannot be read).
int sm_count();

}  // namespace kvm
