// Host runtime of libkvm: the C ABI of include/kvm.h.
//
// Owns only host metadata (config, residency of the page pool, baked
// positions), one internal copy stream and a few events.  Device memory is the
// caller's: one workspace carved into the RoPE table and scoring scratch, plus
// the buffers passed to each call or bound with kvm_bind.
//
// Residency and page reuse follow KVMem (Virtualizing Million-Token Agent
// Workspaces on a Consumer GPU), §4.4 (delta working set: hits keep their
// pages, only L_t^physical is staged in; packed, pipelined rematerialization
// with CUDA events, Figure 3) and §5 (block record: chronological id, tier,
// baked position).
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "kvm.h"
#include "kvm_internal.cuh"

namespace {

thread_local std::string g_last_error;

kvm_status fail(kvm_status s, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

kvm_status cuda_fail(cudaError_t e, const char *what) {
    return fail(KVM_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define KVM_CUDA(call)                                             \
    do {                                                           \
        cudaError_t e_ = (call);                                   \
        if (e_ != cudaSuccess) return cuda_fail(e_, #call);        \
    } while (0)

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

size_t elt_bytes(int dt) { return dt == KVM_E4M3 ? 1 : dt == KVM_BF16 ? 2 : 4; }

constexpr int kStatSlots = 64;   // steps whose counters can wait for kvm_sync

struct Layout {
    size_t table, part_m, part_z, row_m, row_invz, partial, fused, qstage, stage0, stage1, keep,
        desc, sel, resid, err, total;
    size_t qstage_bytes;
    size_t stage_bytes;
    int64_t keep_tiles;   // index tiles pass 1 keeps in device memory for pass 2
    int rows_max, chunk_cap;
};

bool config_ok(const kvm_config *c, std::string *why) {
    auto bad = [&](const char *m) { *why = m; return false; };
    if (!c) return bad("config is NULL");
    if (c->n_layers < 1 || c->n_kv_heads < 1 || c->n_q_heads < 1) return bad("L, G, H must be >= 1");
    if (c->n_q_heads % c->n_kv_heads) return bad("n_q_heads must be a multiple of n_kv_heads");
    if (c->head_dim != 64 && c->head_dim != 128) return bad("head_dim must be 64 or 128");
    if (c->block_tokens != 32) return bad("block_tokens must be 32");
    if (!(c->rope_theta > 1.0)) return bad("rope_theta must be > 1");
    if (c->kv_dtype != KVM_F32 && c->kv_dtype != KVM_BF16 && c->kv_dtype != KVM_E4M3)
        return bad("kv_dtype must be KVM_F32, KVM_BF16 or KVM_E4M3");
    for (int dt : {c->index_dtype, c->q_dtype})
        if (dt != KVM_F32 && dt != KVM_BF16)
            return bad("index_dtype and q_dtype must be KVM_F32 or KVM_BF16");
    if (c->sink_blocks < 0 || c->recent_blocks < 0) return bad("sink/recent must be >= 0");
    if (c->view_blocks < c->sink_blocks + c->recent_blocks + 1)
        return bad("view_blocks must be >= sink + recent + 1");
    if (c->max_queries < 1) return bad("max_queries must be >= 1");
    if ((int64_t)c->max_queries * (c->n_q_heads / c->n_kv_heads) > kvm::kMaxRows)
        return bad("max_queries * (H/G) must be <= 256");
    if (c->max_blocks < 1 || c->max_blocks > (int64_t)1 << 30) return bad("max_blocks out of range");
    if (c->max_positions < 32 * (int64_t)c->view_blocks)
        return bad("max_positions must cover the view (32 * view_blocks)");
    if (c->index_location != KVM_DEVICE && c->index_location != KVM_HOST_PINNED)
        return bad("index_location must be KVM_DEVICE or KVM_HOST_PINNED");
    if (c->repo_location != KVM_DEVICE && c->repo_location != KVM_HOST_PINNED)
        return bad("repo_location must be KVM_DEVICE or KVM_HOST_PINNED");
    if (c->index_location == KVM_HOST_PINNED && c->tile_blocks < 1)
        return bad("tile_blocks must be >= 1 for a host-resident index");
    if (c->pool_pages < c->view_blocks) return bad("pool_pages must be >= view_blocks");
    if (c->h2d_batch_blocks < 1) return bad("h2d_batch_blocks must be >= 1");
    if (c->score_variant < 0 || c->score_variant > 2) return bad("score_variant must be 0, 1 or 2");
    if (c->h2d_mode != 0 && c->h2d_mode != 1) return bad("h2d_mode must be 0 or 1");
    if (c->delta_rerope_limit < 0) return bad("delta_rerope_limit must be >= 0");
    if (c->candidate_mode != 0 && c->candidate_mode != 1) return bad("candidate_mode must be 0 or 1");
    if (c->host_tier_blocks < 0 || (c->host_tier_blocks > 0 && c->host_tier_blocks < c->view_blocks))
        return bad("host_tier_blocks must be 0 or >= view_blocks");
    if (c->host_tier_blocks > 0 && !(c->host_tier_lambda >= 0.0 && c->host_tier_lambda <= 1.0))
        return bad("host_tier_lambda must be in [0, 1]");
    if (c->index_spill != 0 && c->index_spill != 1) return bad("index_spill must be 0 or 1");
    if (c->spill_tiles < 0) return bad("spill_tiles must be >= 0");
    if (c->spill_tiles > 0 && !c->index_spill) return bad("spill_tiles needs index_spill = 1");
    return true;
}

Layout layout_of(const kvm_config *c) {
    Layout lo{};
    const size_t LG = (size_t)c->n_layers * c->n_kv_heads;
    lo.rows_max = c->max_queries * (c->n_q_heads / c->n_kv_heads);
    lo.chunk_cap = kvm::kMaxChunks;
    if (c->index_location == KVM_HOST_PINNED) {
        const int64_t tiles = (c->max_blocks + c->tile_blocks - 1) / c->tile_blocks;
        lo.chunk_cap = (int)std::max<int64_t>(kvm::kMaxChunks, tiles);
    }
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 256); return o; };
    lo.table = take((size_t)c->max_positions * (c->head_dim / 2) * sizeof(float2));
    lo.part_m = take(LG * lo.chunk_cap * lo.rows_max * sizeof(float));
    lo.part_z = take(LG * lo.chunk_cap * lo.rows_max * sizeof(float));
    lo.row_m = take(LG * lo.rows_max * sizeof(float));
    lo.row_invz = take(LG * lo.rows_max * sizeof(float));
    lo.partial = take(LG * (size_t)c->max_blocks * sizeof(float));
    lo.fused = take(kvm::fused_scratch_bytes(lo.rows_max));
    // queries in host memory are copied here for the one-launch scoring,
    // whose TMA reads them from device memory
    lo.qstage_bytes = c->index_location == KVM_DEVICE
                          ? (size_t)c->n_layers * c->max_queries * c->n_q_heads * c->head_dim *
                                elt_bytes(c->q_dtype)
                          : 0;
    lo.qstage = take(lo.qstage_bytes);
    lo.stage_bytes = 0;
    if (c->index_location == KVM_HOST_PINNED)
        lo.stage_bytes = LG * (size_t)c->tile_blocks * c->head_dim * elt_bytes(c->index_dtype);
    lo.keep_tiles = 0;
    const int64_t tiles = (c->max_blocks + c->tile_blocks - 1) / c->tile_blocks;
    if (c->index_location == KVM_HOST_PINNED && c->index_spill &&
        (c->spill_tiles == 0 || c->spill_tiles >= tiles)) {
        // one staging tile per index tile: pass 2 reads what pass 1 staged
        lo.keep_tiles = tiles;
        lo.keep = lo.stage0 = lo.stage1 = take(lo.stage_bytes * (size_t)tiles);
    } else {
        // two streaming tiles, and with a spill budget the tiles pass 1 keeps
        lo.stage0 = take(lo.stage_bytes);
        lo.stage1 = take(lo.stage_bytes);
        if (c->index_location == KVM_HOST_PINNED && c->index_spill) {
            lo.keep_tiles = c->spill_tiles;
            lo.keep = take(lo.stage_bytes * (size_t)lo.keep_tiles);
        }
    }
    lo.desc = take((size_t)(c->pool_pages + c->view_blocks) * sizeof(kvm::SlotDesc));
    lo.sel = take(kvm::select_scratch_bytes());
    // the device-side residency of kvm_step (int32 each): page_of_block and
    // stamp per block; block_of_page, baked_pos, delta_count and a free list
    // per page; a page per slot; kStatSlots steps of counters and one slot
    // for steps captured into a CUDA graph
    lo.resid = take(((size_t)2 * c->max_blocks + (size_t)4 * c->pool_pages + c->view_blocks +
                     (size_t)(kStatSlots + 1) * 8 + 1) *
                    sizeof(int32_t));
    lo.err = take(256);
    lo.total = off;
    return lo;
}

}  // namespace

void kvm::set_last_error(const std::string &msg) { g_last_error = msg; }

namespace {
std::atomic<int64_t> g_launches{0};
}
void kvm::note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

struct kvm_ctx {
    kvm_config cfg{};
    Layout lo{};
    char *ws = nullptr;
    float2 *table = nullptr;
    kvm::ScoreScratch scr{};
    void *stage[2] = {nullptr, nullptr};
    kvm::SlotDesc *desc_dev = nullptr;
    int *sel_scratch = nullptr;        // selection histograms and segment counts
    int *err_dev = nullptr;
    cudaStream_t copy_stream = nullptr;
    cudaEvent_t ev_ready[2] = {nullptr, nullptr};
    cudaEvent_t ev_free[2] = {nullptr, nullptr};
    cudaEvent_t ev_main = nullptr;
    cudaEvent_t ev_stage = nullptr;      // the last stage-out copies are done
    bool staged = false;
    std::vector<cudaEvent_t> ev_batch;
    bool bound = false;
    kvm_buffers bufs{};
    const void *repo_k_dev = nullptr;   // repository as the GPU addresses it
    const void *repo_v_dev = nullptr;
    // residency of the page pool
    std::vector<int64_t> block_of_page;
    std::vector<int64_t> baked_pos;
    std::vector<int32_t> delta_count;    // delta rotations since the page's K was rebuilt
    std::vector<int32_t> page_of_block;
    std::vector<uint8_t> mark;
    // residency diff on the device (repository read by the GPU, no host tier):
    // the state lives in the workspace and kvm_step never waits for the GPU
    bool device_diff = false;
    int32_t *d_page_of_block = nullptr, *d_stamp = nullptr, *d_block_of_page = nullptr,
            *d_baked_pos = nullptr, *d_delta_count = nullptr, *d_free_list = nullptr,
            *d_slot_page = nullptr, *d_counts = nullptr, *d_epoch = nullptr;
    int64_t n_dev_steps = 0;
    bool graph_steps = false;            // a step was captured into a CUDA graph
    int64_t graph_n_blocks = 0;          // ... its history and view sizes
    int32_t graph_n_sel = 0;
    struct Pending {
        kvm_step_stats *out;
        int64_t step;                    // its step number: ring slot step % kStatSlots
        int64_t n_blocks;
        int32_t n_sel;
    };
    std::vector<Pending> pending;        // steps whose counters kvm_sync copies out
    cudaEvent_t ev_reset = nullptr;      // the device residency was cleared on the copy stream
    cudaEvent_t ev_step = nullptr;       // the last device-diff step's work is enqueued
                                         // (eagerly, or by a graph launch)
    bool reset_pending = false;
    kvm_tier *tier = nullptr;            // host-tier policy (host_tier_blocks > 0)
    // fault injection
    int inject_what = 0;
    int64_t inject_nth = 0, inject_seen = 0;
    int device = 0;
};

namespace {

bool injected(kvm_ctx *c, int what) {
    if (c->inject_what != what) return false;
    if (++c->inject_seen == c->inject_nth) {
        c->inject_what = 0;
        return true;
    }
    return false;
}

kvm::ScoreShape shape_of(const kvm_ctx *c, int n_queries, int64_t index_cap) {
    kvm::ScoreShape sh{};
    sh.L = c->cfg.n_layers;
    sh.G = c->cfg.n_kv_heads;
    sh.H = c->cfg.n_q_heads;
    sh.d = c->cfg.head_dim;
    sh.n_queries = n_queries;
    sh.gqa = sh.H / sh.G;
    sh.rows = n_queries * sh.gqa;
    sh.index_cap = index_cap;
    sh.chunk_cap = c->lo.chunk_cap;
    sh.variant = c->cfg.score_variant;
    return sh;
}

size_t block_bytes(const kvm_config &c) {
    return (size_t)c.n_layers * c.n_kv_heads * 32 * c.head_dim * elt_bytes(c.kv_dtype);
}

// Clears the device-side residency on the copy stream, after the work already
// on `after` when `has_after` (a stream handle may be 0, the legacy default
// stream), else after the last step enqueued; the next step waits for it.
cudaError_t reset_device(kvm_ctx *c, cudaStream_t after, bool has_after) {
    if (!c->device_diff || !c->copy_stream) return cudaSuccess;
    cudaError_t e;
    if (has_after) {
        if ((e = cudaEventRecord(c->ev_main, after)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(c->copy_stream, c->ev_main, 0)) != cudaSuccess)
            return e;
    } else if ((c->n_dev_steps > 0 || c->graph_steps) &&
               (e = cudaStreamWaitEvent(c->copy_stream, c->ev_step, 0)) != cudaSuccess) {
        return e;   // after the last step enqueued
    }
    const size_t nb = (size_t)c->cfg.max_blocks, np = (size_t)c->cfg.pool_pages;
    if ((e = cudaMemsetAsync(c->d_page_of_block, 0xFF, nb * 4, c->copy_stream)) != cudaSuccess ||
        (e = cudaMemsetAsync(c->d_block_of_page, 0xFF, np * 4, c->copy_stream)) != cudaSuccess ||
        (e = cudaMemsetAsync(c->d_baked_pos, 0xFF, np * 4, c->copy_stream)) != cudaSuccess ||
        (e = cudaMemsetAsync(c->d_delta_count, 0, np * 4, c->copy_stream)) != cudaSuccess ||
        (e = cudaEventRecord(c->ev_reset, c->copy_stream)) != cudaSuccess)
        return e;
    c->reset_pending = true;
    return cudaSuccess;
}

void reset_pool(kvm_ctx *c, cudaStream_t after = nullptr, bool has_after = false) {
    if (reset_device(c, after, has_after) != cudaSuccess)
        kvm::set_last_error("device residency reset failed");
    for (int64_t b : c->block_of_page)
        if (b >= 0 && b < (int64_t)c->page_of_block.size()) c->page_of_block[b] = -1;
    std::fill(c->block_of_page.begin(), c->block_of_page.end(), -1);
    std::fill(c->baked_pos.begin(), c->baked_pos.end(), -1);
    std::fill(c->delta_count.begin(), c->delta_count.end(), 0);
}

}  // namespace

// Whether `s` is being captured into a CUDA graph.
static kvm_status stream_capturing(cudaStream_t s, bool *capturing) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    const cudaError_t e = cudaStreamIsCapturing(s, &cs);
    if (e != cudaSuccess) return cuda_fail(e, "stream capture status");
    *capturing = cs == cudaStreamCaptureStatusActive;
    return KVM_OK;
}

// The address a kernel uses for a caller buffer: device (or managed) memory as
// is; pinned host memory through its device alias, so that kernels read or
// write it over the host link without a staging copy.  Pageable host memory is
// rejected.  NULL stays NULL.
static kvm_status kernel_ptr(const void *p, const void **out, const char *what) {
    *out = nullptr;
    if (!p) return KVM_OK;
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return fail(KVM_ERR_INVALID_ARG, "%s: not an address the GPU can use", what);
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
        *out = p;
        return KVM_OK;
    }
    if (a.type == cudaMemoryTypeHost) {
        void *d = nullptr;
        const cudaError_t e = cudaHostGetDevicePointer(&d, const_cast<void *>(p), 0);
        if (e != cudaSuccess) return cuda_fail(e, what);
        *out = d;
        return KVM_OK;
    }
    return fail(KVM_ERR_INVALID_ARG,
                "%s: pageable host memory; use device memory or pinned host memory", what);
}

int kvm::resolve_kernel_ptr(const void *p, const void **out, const char *what) {
    return kernel_ptr(p, out, what);
}

template <typename T>
static kvm_status kernel_ptr(T *p, T **out, const char *what) {
    const void *q = nullptr;
    const kvm_status st = kernel_ptr(static_cast<const void *>(p), &q, what);
    *out = static_cast<T *>(const_cast<void *>(q));
    return st;
}

extern "C" {

size_t kvm_workspace_bytes(const kvm_config *cfg) {
    std::string why;
    if (!config_ok(cfg, &why)) return 0;
    return layout_of(cfg).total;
}

kvm_status kvm_create(const kvm_config *cfg, void *workspace, size_t workspace_bytes,
                      kvm_stream stream, kvm_ctx **out) {
    std::string why;
    if (!out) return fail(KVM_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (!config_ok(cfg, &why)) return fail(KVM_ERR_INVALID_ARG, "config: %s", why.c_str());
    Layout lo = layout_of(cfg);
    if (!workspace) return fail(KVM_ERR_INVALID_ARG, "workspace is NULL");
    if (((uintptr_t)workspace & 255) != 0) return fail(KVM_ERR_INVALID_ARG, "workspace not 256-byte aligned");
    if (workspace_bytes < lo.total)
        return fail(KVM_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu bytes", workspace_bytes, lo.total);
    auto *c = new (std::nothrow) kvm_ctx();
    if (!c) return fail(KVM_ERR_CAPACITY, "out of host memory");
    c->cfg = *cfg;
    c->lo = lo;
    c->ws = static_cast<char *>(workspace);
    c->table = reinterpret_cast<float2 *>(c->ws + lo.table);
    c->scr.part_m = reinterpret_cast<float *>(c->ws + lo.part_m);
    c->scr.part_z = reinterpret_cast<float *>(c->ws + lo.part_z);
    c->scr.row_m = reinterpret_cast<float *>(c->ws + lo.row_m);
    c->scr.row_invz = reinterpret_cast<float *>(c->ws + lo.row_invz);
    c->scr.partial = reinterpret_cast<float *>(c->ws + lo.partial);
    kvm::fused_scratch_carve(&c->scr, c->ws + lo.fused, lo.rows_max);
    c->stage[0] = c->ws + lo.stage0;
    c->stage[1] = c->ws + lo.stage1;
    c->desc_dev = reinterpret_cast<kvm::SlotDesc *>(c->ws + lo.desc);
    c->sel_scratch = reinterpret_cast<int *>(c->ws + lo.sel);
    c->err_dev = reinterpret_cast<int *>(c->ws + lo.err);
    c->scr.err = c->err_dev;
    {
        int32_t *r = reinterpret_cast<int32_t *>(c->ws + lo.resid);
        c->d_page_of_block = r;
        c->d_stamp = r + cfg->max_blocks;
        c->d_block_of_page = c->d_stamp + cfg->max_blocks;
        c->d_baked_pos = c->d_block_of_page + cfg->pool_pages;
        c->d_delta_count = c->d_baked_pos + cfg->pool_pages;
        c->d_free_list = c->d_delta_count + cfg->pool_pages;
        c->d_slot_page = c->d_free_list + cfg->pool_pages;
        c->d_counts = c->d_slot_page + cfg->view_blocks;
        c->d_epoch = c->d_counts + (kStatSlots + 1) * 8;
    }
    // the diff runs on the device when the kernels read the repository
    // themselves; copy-engine transfers and the host-tier policy need the
    // selected ids on the host
    c->device_diff = (cfg->repo_location == KVM_DEVICE || cfg->h2d_mode == 1) &&
                     cfg->host_tier_blocks == 0;
    try {   // no exception crosses the C ABI
        c->block_of_page.assign(cfg->pool_pages, -1);
        c->baked_pos.assign(cfg->pool_pages, -1);
        c->delta_count.assign(cfg->pool_pages, 0);
        c->page_of_block.assign((size_t)cfg->max_blocks, -1);
        c->mark.assign((size_t)cfg->max_blocks, 0);
        c->ev_batch.assign((cfg->pool_pages + cfg->h2d_batch_blocks - 1) / cfg->h2d_batch_blocks + 1,
                           nullptr);
    } catch (...) {
        delete c;
        return fail(KVM_ERR_CAPACITY, "out of host memory");
    }

    auto cleanup = [&](kvm_status s) { kvm_destroy(c); return s; };
    cudaError_t e = cudaGetDevice(&c->device);
    if (e != cudaSuccess) return cleanup(cuda_fail(e, "cudaGetDevice"));
    e = cudaStreamCreateWithFlags(&c->copy_stream, cudaStreamNonBlocking);
    if (e != cudaSuccess) return cleanup(cuda_fail(e, "cudaStreamCreateWithFlags"));
    for (int i = 0; i < 2; ++i) {
        if ((e = cudaEventCreateWithFlags(&c->ev_ready[i], cudaEventDisableTiming)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&c->ev_free[i], cudaEventDisableTiming)) != cudaSuccess)
            return cleanup(cuda_fail(e, "cudaEventCreate"));
    }
    if ((e = cudaEventCreateWithFlags(&c->ev_main, cudaEventDisableTiming)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&c->ev_stage, cudaEventDisableTiming)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&c->ev_reset, cudaEventDisableTiming)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&c->ev_step, cudaEventDisableTiming)) != cudaSuccess)
        return cleanup(cuda_fail(e, "cudaEventCreate"));
    for (auto &ev : c->ev_batch)
        if ((e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming)) != cudaSuccess)
            return cleanup(cuda_fail(e, "cudaEventCreate"));
    if (cfg->host_tier_blocks > 0) {
        const kvm_status ts = kvm_tier_create(cfg->host_tier_blocks, cfg->host_tier_lambda, &c->tier);
        if (ts != KVM_OK) return cleanup(ts);
    }

    kvm::Omega om{};
    const int hd = cfg->head_dim / 2;
    for (int i = 0; i < hd; ++i) om.w[i] = std::pow(cfg->rope_theta, -2.0 * i / cfg->head_dim);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if ((e = kvm::launch_rope_table(c->table, cfg->max_positions, hd, om, s)) != cudaSuccess)
        return cleanup(cuda_fail(e, "rope table"));
    if ((e = cudaMemsetAsync(c->err_dev, 0, sizeof(int), s)) != cudaSuccess)
        return cleanup(cuda_fail(e, "cudaMemsetAsync"));
    if (c->device_diff) {
        // an empty pool; no block has been selected yet (stamp 0 < every epoch)
        if ((e = cudaMemsetAsync(c->d_stamp, 0, (size_t)cfg->max_blocks * 4, s)) != cudaSuccess ||
            (e = cudaMemsetAsync(c->d_epoch, 0, sizeof(int32_t), s)) != cudaSuccess ||
            (e = reset_device(c, s, true)) != cudaSuccess)
            return cleanup(cuda_fail(e, "residency init"));
    }
    *out = c;
    return KVM_OK;
}

kvm_status kvm_destroy(kvm_ctx *c) {
    if (!c) return KVM_OK;
    if (c->copy_stream) cudaStreamSynchronize(c->copy_stream);
    for (auto ev : {c->ev_ready[0], c->ev_ready[1], c->ev_free[0], c->ev_free[1], c->ev_main,
                    c->ev_stage, c->ev_reset, c->ev_step})
        if (ev) cudaEventDestroy(ev);
    for (auto ev : c->ev_batch)
        if (ev) cudaEventDestroy(ev);
    if (c->copy_stream) cudaStreamDestroy(c->copy_stream);
    if (c->tier) kvm_tier_destroy(c->tier);
    delete c;
    return KVM_OK;
}

kvm_status kvm_build_index(kvm_ctx *c, const void *k_pages, int64_t first_block,
                           int64_t n_blocks, void *index, void *raw_k_out, kvm_stream stream) {
    if (!c) return fail(KVM_ERR_INVALID_ARG, "ctx is NULL");
    if (!k_pages || !index) return fail(KVM_ERR_INVALID_ARG, "k_pages and index are required");
    if (first_block < 0 || n_blocks < 0) return fail(KVM_ERR_INVALID_ARG, "negative block range");
    if (first_block + n_blocks > c->cfg.max_blocks)
        return fail(KVM_ERR_CAPACITY, "blocks [%lld, %lld) beyond max_blocks %lld",
                    (long long)first_block, (long long)(first_block + n_blocks),
                    (long long)c->cfg.max_blocks);
    if ((first_block + n_blocks) * 32 > c->cfg.max_positions)
        return fail(KVM_ERR_CAPACITY, "positions up to %lld beyond max_positions %lld",
                    (long long)((first_block + n_blocks) * 32), (long long)c->cfg.max_positions);
    if (n_blocks == 0) return KVM_OK;
    kvm_status st;
    if ((st = kernel_ptr(k_pages, &k_pages, "k_pages")) != KVM_OK ||
        (st = kernel_ptr(index, &index, "index")) != KVM_OK ||
        (st = kernel_ptr(raw_k_out, &raw_k_out, "raw_k_out")) != KVM_OK)
        return st;
    const cudaError_t e = kvm::launch_meank(
        c->cfg.kv_dtype, c->cfg.index_dtype, c->cfg.head_dim, k_pages, raw_k_out, index,
        c->cfg.max_blocks, first_block, n_blocks, c->cfg.n_layers * c->cfg.n_kv_heads,
        c->table, c->err_dev, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "meank launch");
    return KVM_OK;
}

// The shape for one scoring pass launch: a pending injection of kind 3 makes
// the n-th tensor-core pass run with an idle TMA producer.
static kvm::ScoreShape pass_shape(kvm_ctx *c, kvm::ScoreShape sh) {
    if (kvm::score_uses_tc(c->cfg.q_dtype, c->cfg.index_dtype, sh))
        sh.idle_producer = injected(c, 3) ? 1 : 0;
    return sh;
}

// Blocks [c0, c1) are scored (the candidate set); the rest of [0, N) get 0.
static kvm_status score_device(kvm_ctx *c, const kvm::ScoreShape &sh, const void *q,
                               const void *index, int64_t N, int64_t c0, int64_t c1,
                               float *scores, cudaStream_t s) {
    cudaError_t e;
    if (c1 > c0 && kvm::score_fused_supported(c->cfg.q_dtype, c->cfg.index_dtype, sh)) {
        // both passes in one launch; an injection of kind 3 counts it as two
        // passes (pass 1, then pass 2)
        if (!kvm::fused_q_ok(q)) {
            void *qs = c->ws + c->lo.qstage;
            KVM_CUDA(cudaMemcpyAsync(qs, q,
                                     (size_t)sh.L * sh.n_queries * sh.H * sh.d *
                                         elt_bytes(c->cfg.q_dtype),
                                     cudaMemcpyDefault, s));
            q = qs;
        }
        kvm::ScoreShape fs = sh;
        fs.idle_producer = injected(c, 3) ? 1 : 0;
        fs.idle_producer |= injected(c, 3) ? 2 : 0;
        if ((e = kvm::launch_score_fused(fs, q, index, c0, c1, c->scr, c->cfg.max_blocks, s)) !=
            cudaSuccess)
            return cuda_fail(e, "score (one launch)");
    } else if (c1 > c0) {
        const int nch = kvm::score_chunks(sh, c1 - c0, kvm::kMaxChunks);
        if ((e = kvm::launch_score_pass1(c->cfg.q_dtype, c->cfg.index_dtype, pass_shape(c, sh),
                                         q, index, 0, c0, c1, 0, nch, c->scr, s)) != cudaSuccess)
            return cuda_fail(e, "score pass 1");
        if ((e = kvm::launch_score_combine(sh, nch, c->scr, s)) != cudaSuccess)
            return cuda_fail(e, "score combine");
        if ((e = kvm::launch_score_pass2(c->cfg.q_dtype, c->cfg.index_dtype, pass_shape(c, sh),
                                         q, index, 0, c0, c1, nch, c->scr, c->cfg.max_blocks,
                                         s)) != cudaSuccess)
            return cuda_fail(e, "score pass 2");
    }
    if ((e = kvm::launch_score_reduce(sh, N, c0, c1, c->scr, c->cfg.max_blocks, scores, s)) !=
        cudaSuccess)
        return cuda_fail(e, "score reduce");
    return KVM_OK;
}

// Index in pinned host memory: tiles of tile_blocks staged through two device
// buffers on the copy stream; the softmax stays global because pass 1 only
// records per-chunk (max, sum) and the combine folds every tile's chunks
// before pass 2 re-streams the tiles (KVMem §5, tiled retrieval).  With
// index_spill the last m tiles of pass 1 (every tile, or at most spill_tiles)
// stay in buffers of their own: pass 2 scores them first, with no copy, while
// the copy stream re-streams the other tiles through the two buffers.  A
// block's pass-2 sum depends only on its own tile, so the order of pass 2
// does not change any result.
static kvm_status score_host_tiled(kvm_ctx *c, kvm::ScoreShape sh, const void *q,
                                   const void *index, int64_t N, int64_t c0, int64_t c1,
                                   float *scores, cudaStream_t s) {
    const int64_t tile = c->cfg.tile_blocks;
    const int64_t T = (N + tile - 1) / tile;
    const int cpt = std::max(1, std::min(kvm::score_chunks(sh, tile, kvm::kMaxChunks),
                                         (int)(c->lo.chunk_cap / T)));
    const size_t eb = elt_bytes(c->cfg.index_dtype);
    const size_t row = (size_t)c->cfg.head_dim * eb;
    const size_t LG = (size_t)c->cfg.n_layers * c->cfg.n_kv_heads;
    cudaError_t e;
    KVM_CUDA(cudaEventRecord(c->ev_main, s));
    KVM_CUDA(cudaStreamWaitEvent(c->copy_stream, c->ev_main, 0));
    kvm::ScoreShape tsh = sh;
    tsh.index_cap = tile;
    // tiles first_kept .. T-1 keep their pass-1 copy
    const int64_t m = std::min<int64_t>(c->lo.keep_tiles, T), first_kept = T - m;
    for (int pass = 1; pass <= 2 && c1 > c0; ++pass) {
        for (int64_t i = 0; i < T; ++i) {
            // pass 2 takes the kept tiles first
            const int64_t t = pass == 1 ? i : (i < m ? first_kept + i : i - m);
            const bool kept = t >= first_kept;
            const int buf = (int)(t & 1);
            const int64_t b0 = t * tile, nb = std::min(tile, N - b0);
            // the tile's part of the candidate range; an empty part still runs
            // pass 1 so that its chunks hold (-inf, 0) for the combine
            const int64_t lo = std::min(std::max(b0, c0), b0 + nb);
            const int64_t hi = std::max(std::min(b0 + nb, c1), lo);
            void *tile_buf = kept ? c->ws + c->lo.keep + (size_t)(t - first_kept) * c->lo.stage_bytes
                                  : c->stage[buf];
            if (!kept || pass == 1) {
                // a kept tile's buffer is not reused within the call; the copy
                // stream joined the caller's stream at the start, after the
                // previous call's pass 2
                if (!kept) KVM_CUDA(cudaStreamWaitEvent(c->copy_stream, c->ev_free[buf], 0));
                KVM_CUDA(cudaMemcpy2DAsync(tile_buf, tile * row,
                                           static_cast<const char *>(index) + b0 * row,
                                           (size_t)c->cfg.max_blocks * row, nb * row, LG,
                                           cudaMemcpyHostToDevice, c->copy_stream));
                KVM_CUDA(cudaEventRecord(c->ev_ready[buf], c->copy_stream));
                KVM_CUDA(cudaStreamWaitEvent(s, c->ev_ready[buf], 0));
            }
            if (pass == 1)
                e = kvm::launch_score_pass1(c->cfg.q_dtype, c->cfg.index_dtype,
                                            pass_shape(c, tsh), q,
                                            tile_buf, b0, lo, hi, (int)(t * cpt), cpt,
                                            c->scr, s);
            else
                e = kvm::launch_score_pass2(c->cfg.q_dtype, c->cfg.index_dtype,
                                            pass_shape(c, tsh), q,
                                            tile_buf, b0, lo, hi, cpt, c->scr,
                                            c->cfg.max_blocks, s);
            if (e != cudaSuccess) return cuda_fail(e, "tiled score pass");
            if (!kept) KVM_CUDA(cudaEventRecord(c->ev_free[buf], s));
        }
        if (pass == 1 && (e = kvm::launch_score_combine(sh, (int)(T * cpt), c->scr, s)) != cudaSuccess)
            return cuda_fail(e, "score combine");
    }
    if ((e = kvm::launch_score_reduce(sh, N, c0, c1, c->scr, c->cfg.max_blocks, scores, s)) !=
        cudaSuccess)
        return cuda_fail(e, "score reduce");
    return KVM_OK;
}

kvm_status kvm_score_select(kvm_ctx *c, const void *q, int32_t n_queries, const void *index,
                            int64_t n_blocks, float *scores_out, int32_t *sel_ids_out,
                            int32_t *n_sel_out, kvm_stream stream) {
    if (!c) return fail(KVM_ERR_INVALID_ARG, "ctx is NULL");
    if (!q || !index || !scores_out || !sel_ids_out)
        return fail(KVM_ERR_INVALID_ARG, "q, index, scores_out and sel_ids_out are required");
    if (n_queries < 1 || n_blocks < 1) return fail(KVM_ERR_INVALID_ARG, "n_queries and n_blocks must be >= 1");
    if (n_queries > c->cfg.max_queries)
        return fail(KVM_ERR_CAPACITY, "n_queries %d > max_queries %d", n_queries, c->cfg.max_queries);
    if (n_blocks > c->cfg.max_blocks)
        return fail(KVM_ERR_CAPACITY, "n_blocks %lld > max_blocks %lld", (long long)n_blocks,
                    (long long)c->cfg.max_blocks);
    kvm_status st;
    if ((st = kernel_ptr(q, &q, "q")) != KVM_OK ||
        (st = kernel_ptr(scores_out, &scores_out, "scores_out")) != KVM_OK ||
        (st = kernel_ptr(sel_ids_out, &sel_ids_out, "sel_ids_out")) != KVM_OK)
        return st;
    if (c->cfg.index_location == KVM_DEVICE) {
        // the scoring kernels stream the index with TMA from device memory
        cudaPointerAttributes a{};
        if (cudaPointerGetAttributes(&a, index) != cudaSuccess || a.type != cudaMemoryTypeDevice) {
            cudaGetLastError();
            return fail(KVM_ERR_INVALID_ARG,
                        "index: device memory required (KVM_HOST_PINNED for a host index)");
        }
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (c->cfg.index_location != KVM_DEVICE) {
        // the tiled path orders its staging buffers with events recorded by
        // earlier calls, which a graph launch would not see
        bool capturing = false;
        if ((st = stream_capturing(s, &capturing)) != KVM_OK) return st;
        if (capturing)
            return fail(KVM_ERR_INVALID_ARG,
                        "scoring a host-resident index cannot be captured into a CUDA graph");
    }
    const kvm::ScoreShape sh = shape_of(c, n_queries, c->cfg.max_blocks);
    int64_t c0 = 0, c1 = n_blocks;
    if (c->cfg.candidate_mode == 1) {
        c0 = std::min<int64_t>(c->cfg.sink_blocks, n_blocks);
        c1 = std::max<int64_t>(n_blocks - c->cfg.recent_blocks, c0);
    }
    st = c->cfg.index_location == KVM_DEVICE
             ? score_device(c, sh, q, index, n_blocks, c0, c1, scores_out, s)
             : score_host_tiled(c, sh, q, index, n_blocks, c0, c1, scores_out, s);
    if (st != KVM_OK) return st;
    const cudaError_t e = kvm::launch_select(scores_out, n_blocks, c->cfg.sink_blocks,
                                             c->cfg.recent_blocks, c->cfg.view_blocks,
                                             sel_ids_out, c->sel_scratch, s);
    if (e != cudaSuccess) return cuda_fail(e, "select launch");
    if (n_sel_out) *n_sel_out = (int32_t)std::min<int64_t>(n_blocks, c->cfg.view_blocks);
    return KVM_OK;
}

kvm_status kvm_assemble_view(kvm_ctx *c, const int32_t *sel_ids, const int32_t *page_ids,
                             int32_t n_sel, const void *raw_k_repo, const void *v_repo,
                             void *k_pages, void *v_pages, kvm_stream stream) {
    if (!c) return fail(KVM_ERR_INVALID_ARG, "ctx is NULL");
    if (!sel_ids || !raw_k_repo || !k_pages)
        return fail(KVM_ERR_INVALID_ARG, "sel_ids, raw_k_repo and k_pages are required");
    if ((v_repo == nullptr) != (v_pages == nullptr))
        return fail(KVM_ERR_INVALID_ARG, "v_repo and v_pages must both be set or both be NULL");
    if (n_sel < 0) return fail(KVM_ERR_INVALID_ARG, "n_sel < 0");
    if ((int64_t)n_sel * 32 > c->cfg.max_positions)
        return fail(KVM_ERR_CAPACITY, "view of %d slots beyond max_positions", n_sel);
    if (n_sel == 0) return KVM_OK;
    kvm_status st;
    if ((st = kernel_ptr(sel_ids, &sel_ids, "sel_ids")) != KVM_OK ||
        (st = kernel_ptr(page_ids, &page_ids, "page_ids")) != KVM_OK ||
        (st = kernel_ptr(raw_k_repo, &raw_k_repo, "raw_k_repo")) != KVM_OK ||
        (st = kernel_ptr(v_repo, &v_repo, "v_repo")) != KVM_OK ||
        (st = kernel_ptr(k_pages, &k_pages, "k_pages")) != KVM_OK ||
        (st = kernel_ptr(v_pages, &v_pages, "v_pages")) != KVM_OK)
        return st;
    const cudaError_t e = kvm::launch_assemble_ids(
        c->cfg.kv_dtype, c->cfg.head_dim, sel_ids, page_ids, n_sel, c->cfg.max_blocks,
        raw_k_repo, v_repo, k_pages, v_pages, c->cfg.n_layers * c->cfg.n_kv_heads, c->table,
        c->cfg.max_positions, c->err_dev, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "assemble launch");
    return KVM_OK;
}

kvm_status kvm_bind(kvm_ctx *c, const kvm_buffers *b) {
    if (!c || !b) return fail(KVM_ERR_INVALID_ARG, "ctx and buffers are required");
    if (!b->index || !b->raw_k || !b->v || !b->pool_k || !b->pool_v || !b->page_table ||
        !b->scores || !b->sel_ids)
        return fail(KVM_ERR_INVALID_ARG, "a required buffer is NULL");
    if (c->cfg.repo_location == KVM_HOST_PINNED && c->cfg.h2d_mode == 0 && !b->pool_raw_k)
        return fail(KVM_ERR_INVALID_ARG,
                    "pool_raw_k is required with a host-resident repository and h2d_mode 0");
    c->repo_k_dev = b->raw_k;
    c->repo_v_dev = b->v;
    if (c->cfg.repo_location == KVM_HOST_PINNED && c->cfg.h2d_mode == 1) {
        // device addresses of the pinned host repository (the same pointer under
        // unified addressing; an error if the memory is not pinned and mapped)
        void *dk = nullptr, *dv = nullptr;
        cudaError_t e = cudaHostGetDevicePointer(&dk, const_cast<void *>(b->raw_k), 0);
        if (e == cudaSuccess) e = cudaHostGetDevicePointer(&dv, const_cast<void *>(b->v), 0);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(KVM_ERR_INVALID_ARG,
                        "h2d_mode 1 needs a pinned, device-mapped repository: %s",
                        cudaGetErrorString(e));
        }
        c->repo_k_dev = dk;
        c->repo_v_dev = dv;
    }
    c->bufs = *b;
    c->bound = true;
    reset_pool(c);
    return KVM_OK;
}

kvm_status kvm_stage_out(kvm_ctx *c, const void *raw_k, const void *v, int64_t first_block,
                         int64_t n_blocks, kvm_stream stream) {
    if (!c) return fail(KVM_ERR_INVALID_ARG, "ctx is NULL");
    if (!c->bound) return fail(KVM_ERR_NOT_BOUND, "kvm_stage_out before kvm_bind");
    if (c->cfg.repo_location != KVM_HOST_PINNED)
        return fail(KVM_ERR_INVALID_ARG, "stage-out needs a host-resident repository");
    if (!raw_k || !v) return fail(KVM_ERR_INVALID_ARG, "raw_k and v are required");
    if (first_block < 0 || n_blocks < 0) return fail(KVM_ERR_INVALID_ARG, "negative block range");
    if (first_block + n_blocks > c->cfg.max_blocks)
        return fail(KVM_ERR_CAPACITY, "blocks beyond max_blocks");
    if (n_blocks == 0) return KVM_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the copies run on the context's copy stream, ordered by events that
    // later eager calls wait on: not something a graph launch can replay
    bool capturing = false;
    if (kvm_status cst = stream_capturing(s, &capturing); cst != KVM_OK) return cst;
    if (capturing)
        return fail(KVM_ERR_INVALID_ARG, "kvm_stage_out cannot be captured into a CUDA graph");
    const size_t blk = block_bytes(c->cfg);
    char *dk = const_cast<char *>(static_cast<const char *>(c->bufs.raw_k)) + first_block * blk;
    char *dv = const_cast<char *>(static_cast<const char *>(c->bufs.v)) + first_block * blk;
    KVM_CUDA(cudaEventRecord(c->ev_main, s));
    KVM_CUDA(cudaStreamWaitEvent(c->copy_stream, c->ev_main, 0));
    KVM_CUDA(cudaMemcpyAsync(dk, raw_k, n_blocks * blk, cudaMemcpyDeviceToHost, c->copy_stream));
    KVM_CUDA(cudaMemcpyAsync(dv, v, n_blocks * blk, cudaMemcpyDeviceToHost, c->copy_stream));
    KVM_CUDA(cudaEventRecord(c->ev_stage, c->copy_stream));
    c->staged = true;
    return KVM_OK;
}

kvm_status kvm_reset_pool(kvm_ctx *c) {
    if (!c) return fail(KVM_ERR_INVALID_ARG, "ctx is NULL");
    reset_pool(c);
    return KVM_OK;
}

// The delta working set of [KVMem] §4.4: hits keep their pages; misses take
// the free pages (those not holding a selected block) in ascending page order,
// in ascending slot order.  Fills the page of every slot and whether it is a hit.
static kvm_status assign_pages(kvm_ctx *c, const std::vector<int32_t> &sel,
                               std::vector<int32_t> *page_of_slot, std::vector<uint8_t> *is_hit) {
    const int n_sel = (int)sel.size();
    const int P = c->cfg.pool_pages;
    page_of_slot->assign(n_sel, -1);
    is_hit->assign(n_sel, 0);
    for (int j = 0; j < n_sel; ++j)
        if (sel[j] < 0 || sel[j] >= c->cfg.max_blocks)
            return fail(KVM_ERR_DEVICE, "selected id %d out of range", sel[j]);
    for (int j = 0; j < n_sel; ++j) {
        const int32_t b = sel[j];
        c->mark[b] = 1;
        if (c->page_of_block[b] >= 0) {
            (*page_of_slot)[j] = c->page_of_block[b];
            (*is_hit)[j] = 1;
        }
    }
    std::vector<int32_t> free_pages;
    free_pages.reserve(P);
    for (int p = 0; p < P; ++p) {
        const int64_t b = c->block_of_page[p];
        if (b < 0 || !c->mark[b]) free_pages.push_back(p);
    }
    for (int j = 0; j < n_sel; ++j) c->mark[sel[j]] = 0;
    int n_miss = 0;
    for (int j = 0; j < n_sel; ++j) n_miss += !(*is_hit)[j];
    if (n_miss > (int)free_pages.size())
        return fail(KVM_ERR_CAPACITY, "%d misses but only %zu free pages", n_miss, free_pages.size());
    int f = 0;
    for (int j = 0; j < n_sel; ++j)
        if (!(*is_hit)[j]) (*page_of_slot)[j] = free_pages[f++];
    return KVM_OK;
}

// Records the step's residency once its transfers are enqueued: each missed
// block now owns its page (evicting the block the page held), and every page's
// K is baked at its slot's positions.  Returns the number of evicted blocks.
static int commit_residency(kvm_ctx *c, const std::vector<int32_t> &sel,
                            const std::vector<int32_t> &page_of_slot,
                            const std::vector<int> &miss_slots) {
    int evicted = 0;
    for (int j : miss_slots) {
        const int p = page_of_slot[j];
        const int64_t old = c->block_of_page[p];
        if (old >= 0) {
            c->page_of_block[old] = -1;
            ++evicted;
        }
        c->block_of_page[p] = sel[j];
        c->page_of_block[sel[j]] = p;
    }
    for (size_t j = 0; j < sel.size(); ++j) c->baked_pos[page_of_slot[j]] = (int64_t)j * 32;
    return evicted;
}

// Copies the counters of every step still waiting for them to the caller's
// stats (host tier fields 0); the steps' work must be complete.
// A step's stats from its slot of the counter ring (host tier fields 0).
static void fill_stats(const kvm_ctx *c, const int32_t *k, int64_t n_blocks, int32_t n_sel,
                       kvm_step_stats *st) {
    const bool pull = c->cfg.repo_location == KVM_HOST_PINNED;
    *st = kvm_step_stats{};
    st->n_blocks = n_blocks;
    st->n_sel = n_sel;
    st->hits = k[1];
    st->misses = k[2];
    st->reroped = k[0];
    st->delta_reroped = k[3];
    st->evicted = k[4];
    st->h2d_bytes = pull ? 2 * (int64_t)k[2] * (int64_t)block_bytes(c->cfg) : 0;
}

static kvm_status flush_pending(kvm_ctx *c) {
    if (c->pending.empty()) return KVM_OK;
    int32_t ring[kStatSlots * 8];
    KVM_CUDA(cudaEventSynchronize(c->ev_step));
    KVM_CUDA(cudaMemcpy(ring, c->d_counts, sizeof ring, cudaMemcpyDeviceToHost));
    for (const auto &pd : c->pending)
        fill_stats(c, ring + (pd.step % kStatSlots) * 8, pd.n_blocks, pd.n_sel, pd.out);
    c->pending.clear();
    return KVM_OK;
}

// kvm_step when the residency diff runs on the device (the repository in
// device memory, or in pinned host memory read by the GPU): selection ->
// diff -> assembly, all enqueued on the stream with no wait on the host.
//
// Under stream capture the step becomes part of the caller's CUDA graph, and
// each launch of the graph runs one step.  Its ordering with the host-issued
// work of the context then has to hold at every launch, not at capture time:
// the step waits on the latest pool reset (and stage-out) through external
// event-wait nodes, and records ev_step through an external record node, so
// that a later kvm_reset_pool orders its clearing after the launches already
// enqueued.  Its counters go to a slot of their own and are not reported.
static kvm_status step_device(kvm_ctx *c, int64_t n_blocks, int32_t n_sel,
                              kvm_step_stats *stats, cudaStream_t s, bool capturing) {
    const kvm_config &cfg = c->cfg;
    cudaError_t e;
    const bool pull = cfg.repo_location == KVM_HOST_PINNED;
    if (capturing) {
        KVM_CUDA(cudaStreamWaitEvent(s, c->ev_reset, cudaEventWaitExternal));
        if (pull) KVM_CUDA(cudaStreamWaitEvent(s, c->ev_stage, cudaEventWaitExternal));
    } else {
        if (!c->pending.empty() && c->n_dev_steps - c->pending.front().step >= kStatSlots) {
            // this step's ring slot still holds the counters of a step waiting
            // for them (steps without stats use slots too): copy them out first
            if (kvm_status st = flush_pending(c); st != KVM_OK) return st;
        }
        if (c->reset_pending) {
            KVM_CUDA(cudaStreamWaitEvent(s, c->ev_reset, 0));
            c->reset_pending = false;
        }
    }
    const int slot = capturing ? kStatSlots : (int)(c->n_dev_steps % kStatSlots);
    auto abort_step = [&](kvm_status err) {
        // the diff may have run: forget the whole pool, after this stream's
        // work (a captured step ran nothing: the pool is as it was)
        if (!capturing) reset_pool(c, s, true);
        return err;
    };
    kvm::ResidencyArgs a{};
    a.sel = c->bufs.sel_ids;
    a.n_sel = n_sel;
    a.page_of_block = c->d_page_of_block;
    a.block_of_page = c->d_block_of_page;
    a.baked_pos = c->d_baked_pos;
    a.delta_count = c->d_delta_count;
    a.stamp = c->d_stamp;
    a.epoch = c->d_epoch;
    a.P = cfg.pool_pages;
    a.max_blocks = cfg.max_blocks;
    a.delta_limit = cfg.delta_rerope_limit;
    a.page_table = c->bufs.page_table;
    a.desc = c->desc_dev;
    a.counts = c->d_counts + slot * 8;
    a.slot_page = c->d_slot_page;
    a.free_list = c->d_free_list;
    a.pool_k = static_cast<char *>(c->bufs.pool_k);
    a.pool_v = static_cast<char *>(c->bufs.pool_v);
    a.pool_raw = static_cast<char *>(c->bufs.pool_raw_k);
    a.repo_k = static_cast<const char *>(c->repo_k_dev);
    a.repo_v = static_cast<const char *>(c->repo_v_dev);
    a.blk = block_bytes(cfg);
    a.pull = pull ? 1 : 0;
    a.err = c->err_dev;
    if (injected(c, 2)) return abort_step(fail(KVM_ERR_INJECTED, "injected launch failure"));
    if ((e = kvm::launch_residency_diff(a, s)) != cudaSuccess)
        return abort_step(cuda_fail(e, "residency diff launch"));
    if (pull && c->staged && !capturing) {
        // the kernel reads the host repository: order it after earlier stage-outs
        if ((e = cudaStreamWaitEvent(s, c->ev_stage, 0)) != cudaSuccess)
            return abort_step(cuda_fail(e, "stage-out wait"));
    }
    if (injected(c, 2)) return abort_step(fail(KVM_ERR_INJECTED, "injected launch failure"));
    if ((e = kvm::launch_assemble_desc_dev(cfg.kv_dtype, cfg.head_dim, c->desc_dev, n_sel,
                                           a.counts, cfg.n_layers * cfg.n_kv_heads, c->table,
                                           cfg.max_positions, c->err_dev, s)) != cudaSuccess)
        return abort_step(cuda_fail(e, "assemble launch"));
    if (capturing) {
        KVM_CUDA(cudaEventRecordWithFlags(c->ev_step, s, cudaEventRecordExternal));
        c->graph_steps = true;
        c->graph_n_blocks = n_blocks;
        c->graph_n_sel = n_sel;
        return KVM_OK;
    }
    KVM_CUDA(cudaEventRecord(c->ev_step, s));
    ++c->n_dev_steps;
    if (stats) c->pending.push_back({stats, c->n_dev_steps - 1, n_blocks, n_sel});
    return KVM_OK;
}

static kvm_status step_body(kvm_ctx *c, const void *q, int32_t n_queries, int64_t n_blocks,
                            kvm_step_stats *stats, kvm_stream stream) {
    const kvm_config &cfg = c->cfg;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    bool capturing = false;
    if (kvm_status cst = stream_capturing(s, &capturing); cst != KVM_OK) return cst;
    if (capturing) {
        // only a step that enqueues everything with no wait on the host can
        // become part of a graph
        if (!c->device_diff)
            return fail(KVM_ERR_INVALID_ARG,
                        "kvm_step under stream capture needs the residency diff on the device "
                        "(repository in device memory, or pinned and read by the GPU; no host tier)");
        if (stats)
            return fail(KVM_ERR_INVALID_ARG, "kvm_step under stream capture takes stats = NULL");
    }
    int32_t n_sel = 0;
    kvm_status st = kvm_score_select(c, q, n_queries, c->bufs.index, n_blocks, c->bufs.scores,
                                     c->bufs.sel_ids, &n_sel, stream);
    if (st != KVM_OK) return st;
    if (c->device_diff) return step_device(c, n_blocks, n_sel, stats, s, capturing);

    // the selected ids drive the host-side residency diff
    std::vector<int32_t> sel(n_sel);
    KVM_CUDA(cudaMemcpyAsync(sel.data(), c->bufs.sel_ids, n_sel * sizeof(int32_t),
                             cudaMemcpyDeviceToHost, s));
    KVM_CUDA(cudaStreamSynchronize(s));

    std::vector<int32_t> page_of_slot;
    std::vector<uint8_t> is_hit;
    if ((st = assign_pages(c, sel, &page_of_slot, &is_hit)) != KVM_OK) return st;

    const size_t blk = block_bytes(cfg);
    const bool host_repo = cfg.repo_location == KVM_HOST_PINNED;
    const bool pull = host_repo && cfg.h2d_mode == 1;
    auto P_k = [&](int p) { return static_cast<char *>(c->bufs.pool_k) + (size_t)p * blk; };
    auto P_v = [&](int p) { return static_cast<char *>(c->bufs.pool_v) + (size_t)p * blk; };
    auto P_r = [&](int p) { return static_cast<char *>(c->bufs.pool_raw_k) + (size_t)p * blk; };
    auto R_k = [&](int64_t b) { return static_cast<const char *>(c->bufs.raw_k) + (size_t)b * blk; };
    auto R_v = [&](int64_t b) { return static_cast<const char *>(c->bufs.v) + (size_t)b * blk; };

    // where a page's K is rebuilt from: its own raw-K copy, else the repository
    // (device memory, or the pinned host repository read by the kernel)
    auto raw_src = [&](int64_t b, int p) -> const void * {
        if (c->bufs.pool_raw_k) return P_r(p);
        if (!host_repo) return R_k(b);
        return static_cast<const char *>(c->repo_k_dev) + (size_t)b * blk;
    };
    // descriptors: shifted hits first (no copy to wait for), then misses in slot order
    std::vector<kvm::SlotDesc> desc;
    desc.reserve(n_sel);
    std::vector<int32_t> new_count(c->delta_count);
    int n_rope = 0, evicted = 0, n_delta = 0;
    for (int j = 0; j < n_sel; ++j) {
        if (!is_hit[j]) continue;
        const int p = page_of_slot[j];
        const int64_t want = (int64_t)j * 32;
        if (c->baked_pos[p] == want) continue;
        kvm::SlotDesc d{};
        d.dst_k = P_k(p);
        if (cfg.delta_rerope_limit > 0 && c->delta_count[p] < cfg.delta_rerope_limit) {
            // bounded delta re-RoPE ([KVMem] §4.4): rotate the page's K in place
            d.src_k = P_k(p);
            d.pos0 = want - c->baked_pos[p];
            d.flags = kvm::kSlotDelta;
            new_count[p] = c->delta_count[p] + 1;
            ++n_delta;
        } else {
            d.src_k = raw_src(sel[j], p);
            d.pos0 = want;
            new_count[p] = 0;
        }
        desc.push_back(d);
    }
    const int n_hit_rope = (int)desc.size();
    std::vector<int> miss_slots;
    for (int j = 0; j < n_sel; ++j) {
        if (is_hit[j]) continue;
        miss_slots.push_back(j);
        const int p = page_of_slot[j];
        kvm::SlotDesc d{};
        if (host_repo && pull) {
            // the kernel reads the block from the pinned host repository itself and
            // writes the page's raw K, its K at the slot's positions and its V
            d.src_k = static_cast<const char *>(c->repo_k_dev) + (size_t)sel[j] * blk;
            d.src_v = static_cast<const char *>(c->repo_v_dev) + (size_t)sel[j] * blk;
            d.dst_v = P_v(p);
            d.dst_raw = c->bufs.pool_raw_k ? P_r(p) : nullptr;
        } else if (host_repo) {
            d.src_k = P_r(p);
        } else {
            d.src_k = R_k(sel[j]);
            d.src_v = R_v(sel[j]);
            d.dst_v = P_v(p);
        }
        d.dst_k = P_k(p);
        d.pos0 = (int64_t)j * 32;
        desc.push_back(d);
        new_count[p] = 0;
    }
    n_rope = (int)desc.size();

    auto abort_step = [&](kvm_status err) {
        // pages may be partly overwritten: forget the whole pool
        reset_pool(c);
        return err;
    };
    const int LG = cfg.n_layers * cfg.n_kv_heads;
    int64_t h2d_bytes = 0;
    int h2d_copies = 0;
    cudaError_t e;
    if (n_rope > 0) {
        if ((e = cudaMemcpyAsync(c->desc_dev, desc.data(), desc.size() * sizeof(kvm::SlotDesc),
                                 cudaMemcpyHostToDevice, s)) != cudaSuccess)
            return abort_step(cuda_fail(e, "descriptor upload"));
    }
    if (pull && c->staged) {
        // the kernel reads the host repository: order it after earlier stage-outs
        if ((e = cudaStreamWaitEvent(s, c->ev_stage, 0)) != cudaSuccess)
            return abort_step(cuda_fail(e, "stage-out wait"));
    }
    if (!host_repo || pull) {
        if (n_rope > 0) {
            if (injected(c, 2)) return abort_step(fail(KVM_ERR_INJECTED, "injected launch failure"));
            if ((e = kvm::launch_assemble_desc(cfg.kv_dtype, cfg.head_dim, c->desc_dev, n_rope, LG,
                                               c->table, cfg.max_positions, c->err_dev, s)) != cudaSuccess)
                return abort_step(cuda_fail(e, "assemble launch"));
        }
    } else {
        if (n_hit_rope > 0) {
            if (injected(c, 2)) return abort_step(fail(KVM_ERR_INJECTED, "injected launch failure"));
            if ((e = kvm::launch_assemble_desc(cfg.kv_dtype, cfg.head_dim, c->desc_dev, n_hit_rope,
                                               LG, c->table, cfg.max_positions, c->err_dev, s)) != cudaSuccess)
                return abort_step(cuda_fail(e, "re-RoPE launch"));
        }
        // misses: coalesced H2D of raw K and V straight into their pages on the
        // copy stream, one event per batch; the GPU re-RoPEs batch i while
        // batch i+1 is in flight
        if ((e = cudaEventRecord(c->ev_main, s)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(c->copy_stream, c->ev_main, 0)) != cudaSuccess)
            return abort_step(cuda_fail(e, "stream join"));
        const int nb_batch = cfg.h2d_batch_blocks;
        int batch = 0;
        for (size_t i0 = 0; i0 < miss_slots.size(); i0 += nb_batch, ++batch) {
            const size_t i1 = std::min(miss_slots.size(), i0 + nb_batch);
            size_t i = i0;
            while (i < i1) {
                // a run: consecutive block ids landing in consecutive pages
                size_t k = i + 1;
                while (k < i1 && sel[miss_slots[k]] == sel[miss_slots[k - 1]] + 1 &&
                       page_of_slot[miss_slots[k]] == page_of_slot[miss_slots[k - 1]] + 1)
                    ++k;
                const int64_t b0 = sel[miss_slots[i]];
                const int p0 = page_of_slot[miss_slots[i]];
                const size_t bytes = (k - i) * blk;
                if (injected(c, 1)) return abort_step(fail(KVM_ERR_INJECTED, "injected copy failure"));
                if ((e = cudaMemcpyAsync(P_r(p0), R_k(b0), bytes, cudaMemcpyHostToDevice,
                                         c->copy_stream)) != cudaSuccess ||
                    (e = cudaMemcpyAsync(P_v(p0), R_v(b0), bytes, cudaMemcpyHostToDevice,
                                         c->copy_stream)) != cudaSuccess)
                    return abort_step(cuda_fail(e, "H2D copy"));
                h2d_bytes += 2 * (int64_t)bytes;
                h2d_copies += 2;
                i = k;
            }
            cudaEvent_t ev = c->ev_batch[batch % c->ev_batch.size()];
            if ((e = cudaEventRecord(ev, c->copy_stream)) != cudaSuccess ||
                (e = cudaStreamWaitEvent(s, ev, 0)) != cudaSuccess)
                return abort_step(cuda_fail(e, "batch event"));
            if (injected(c, 2)) return abort_step(fail(KVM_ERR_INJECTED, "injected launch failure"));
            if ((e = kvm::launch_assemble_desc(cfg.kv_dtype, cfg.head_dim,
                                               c->desc_dev + n_hit_rope + i0, (int)(i1 - i0), LG,
                                               c->table, cfg.max_positions, c->err_dev, s)) != cudaSuccess)
                return abort_step(cuda_fail(e, "re-RoPE launch"));
        }
    }
    if ((e = cudaMemcpyAsync(c->bufs.page_table, page_of_slot.data(), n_sel * sizeof(int32_t),
                             cudaMemcpyHostToDevice, s)) != cudaSuccess)
        return abort_step(cuda_fail(e, "page table upload"));

    evicted = commit_residency(c, sel, page_of_slot, miss_slots);
    c->delta_count.swap(new_count);

    kvm_tier_stats ts{};
    if (c->tier) {
        const kvm_status tst = kvm_tier_step(c->tier, sel.data(), n_sel, n_blocks, nullptr, &ts);
        if (tst != KVM_OK) return tst;
    }
    if (stats) {
        stats->host_hits = ts.hits;
        stats->host_misses = ts.misses;
        stats->host_demoted = ts.demoted;
        stats->n_blocks = n_blocks;
        stats->n_sel = n_sel;
        stats->misses = (int32_t)miss_slots.size();
        stats->hits = n_sel - stats->misses;
        stats->reroped = n_rope;
        stats->delta_reroped = n_delta;
        stats->evicted = evicted;
        stats->h2d_copies = h2d_copies;
        // bytes that crossed the host link: by copy engine, or read by the kernel
        stats->h2d_bytes = pull ? 2 * (int64_t)miss_slots.size() * (int64_t)blk : h2d_bytes;
    }
    return KVM_OK;
}

kvm_status kvm_step(kvm_ctx *c, const void *q, int32_t n_queries, int64_t n_blocks,
                    kvm_step_stats *stats, kvm_stream stream) {
    if (!c) return fail(KVM_ERR_INVALID_ARG, "ctx is NULL");
    if (!c->bound) return fail(KVM_ERR_NOT_BOUND, "kvm_step before kvm_bind");
    try {   // no exception crosses the C ABI
        return step_body(c, q, n_queries, n_blocks, stats, stream);
    } catch (...) {
        // out of host memory part-way: forget the pool, as a failed step does
        std::fill(c->mark.begin(), c->mark.end(), 0);
        reset_pool(c);
        return fail(KVM_ERR_CAPACITY, "out of host memory");
    }
}

kvm_status kvm_sync(kvm_ctx *c, kvm_stream stream) {
    if (!c) return fail(KVM_ERR_INVALID_ARG, "ctx is NULL");
    KVM_CUDA(cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)));
    KVM_CUDA(cudaStreamSynchronize(c->copy_stream));
    if (kvm_status st = flush_pending(c); st != KVM_OK) return st;
    int flag = 0;
    KVM_CUDA(cudaMemcpy(&flag, c->err_dev, sizeof(int), cudaMemcpyDeviceToHost));
    if (flag) {
        KVM_CUDA(cudaMemset(c->err_dev, 0, sizeof(int)));
        if (flag & 4) return fail(KVM_ERR_TIMEOUT, "a bounded device wait gave up (flag 0x%x)", flag);
        return fail(KVM_ERR_DEVICE, "device range check raised flag 0x%x", flag);
    }
    return KVM_OK;
}

kvm_status kvm_graph_step_stats(kvm_ctx *c, kvm_step_stats *stats, kvm_stream stream) {
    if (!c || !stats) return fail(KVM_ERR_INVALID_ARG, "ctx and stats are required");
    if (!c->graph_steps)
        return fail(KVM_ERR_INVALID_ARG, "no kvm_step of this context was captured");
    KVM_CUDA(cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)));
    int32_t k[8];
    KVM_CUDA(cudaMemcpy(k, c->d_counts + kStatSlots * 8, sizeof k, cudaMemcpyDeviceToHost));
    fill_stats(c, k, c->graph_n_blocks, c->graph_n_sel, stats);
    return KVM_OK;
}

const char *kvm_status_string(kvm_status s) {
    switch (s) {
        case KVM_OK: return "ok";
        case KVM_ERR_INVALID_ARG: return "invalid argument";
        case KVM_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case KVM_ERR_CAPACITY: return "capacity exceeded";
        case KVM_ERR_CUDA: return "CUDA error";
        case KVM_ERR_TIMEOUT: return "device wait timed out";
        case KVM_ERR_NOT_BOUND: return "buffers not bound";
        case KVM_ERR_INJECTED: return "injected failure";
        case KVM_ERR_DEVICE: return "device range check failed";
    }
    return "unknown status";
}

const char *kvm_last_error(void) { return g_last_error.c_str(); }

int64_t kvm_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

kvm_status kvm_host_alloc(size_t bytes, void **out) {
    if (!out) return fail(KVM_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (bytes == 0) return fail(KVM_ERR_INVALID_ARG, "bytes must be > 0");
    void *p = nullptr;
    const cudaError_t e = cudaHostAlloc(&p, bytes, cudaHostAllocPortable | cudaHostAllocMapped);
    if (e != cudaSuccess) return cuda_fail(e, "cudaHostAlloc");
    *out = p;
    return KVM_OK;
}

kvm_status kvm_host_free(void *ptr) {
    if (!ptr) return KVM_OK;
    const cudaError_t e = cudaFreeHost(ptr);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFreeHost");
    return KVM_OK;
}

kvm_status kvm_debug_inject(kvm_ctx *c, int32_t what, int64_t nth) {
    if (!c) return fail(KVM_ERR_INVALID_ARG, "ctx is NULL");
    if (what < 0 || what > 3 || (what != 0 && nth < 1))
        return fail(KVM_ERR_INVALID_ARG, "what must be 0..3 and nth >= 1");
    c->inject_what = what;
    c->inject_nth = nth;
    c->inject_seen = 0;
    return KVM_OK;
}

}  // extern "C"
