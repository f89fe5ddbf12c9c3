// kvm_score_select_static: block scoring + selection with no device allocation
// by anyone.
//
// kvm_score_select needs a context, and a context needs a caller-allocated
// device workspace.  Some callers cannot allocate device memory at all: a
// plugin inside an inference engine whose memory planner has already handed
// the whole device to its own pools (a cudaMalloc there fails or fragments the
// engine's pool), or a latency-critical caller that cannot pay for
// cudaMalloc / cudaFree, which may synchronise the device.  For them this
// entry point keeps its scratch in a fixed file-scope device array and takes
// only inputs and outputs.
//
// The array is SCRATCH_BYTES (32 MiB) per device.  Every GPU on which the
// library is loaded holds it until the process exits.  It is shared by every
// call: two calls that overlap on the GPU (different streams, or different
// host threads without ordering) race on it and produce garbage.  The array
// keeps whatever the last call left in it.  Every byte a call reads from it is
// written earlier in the same call, except the error word: the one part that
// must start at zero, the histograms of the selection over 16384 blocks or
// more, is cleared on the call's stream before its first use, and the rest is
// fully overwritten.  The error word (the array's first 4 bytes) collects the
// device error flags of every call until kvm_score_select_static_status reads
// and clears it.
#include <cuda.h>

#include <cstdio>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include "kvm.h"
#include "kvm_internal.cuh"

namespace {

constexpr size_t SCRATCH_BYTES = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_scratch[SCRATCH_BYTES];

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

using CtxGetCurrent = CUresult (*)(CUcontext *);

// cuCtxGetCurrent from the driver, looked up once per process.
CtxGetCurrent ctx_get_current() {
    static const CtxGetCurrent fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            return reinterpret_cast<CtxGetCurrent>(p);
        return static_cast<CtxGetCurrent>(nullptr);
    }();
    return fn;
}

std::mutex g_mu;
std::vector<std::pair<CUcontext, void *>> g_addr;   // (CUDA context, address of g_scratch)

CUcontext current_ctx() {
    CUcontext ctx = nullptr;
    CtxGetCurrent fn = ctx_get_current();
    if (fn && fn(&ctx) != CUDA_SUCCESS) ctx = nullptr;
    return ctx;
}

// The device address of g_scratch in the calling thread's current CUDA context
// (the current device's primary context unless the caller made another one
// current).  In host code the name g_scratch is only a host-side stand-in, so
// the address is looked up with cudaGetSymbolAddress the first time a context
// calls, then reused for the life of the process.  A context destroyed and
// re-created (cudaDeviceReset) may leave a stale entry behind.
kvm_status scratch_for_current_context(void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        kvm::set_last_error(std::string("cudaGetDevice: ") + cudaGetErrorString(e));
        return KVM_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    CUcontext ctx = current_ctx();
    if (ctx)
        for (const auto &p : g_addr)
            if (p.first == ctx) {
                *out = p.second;
                return KVM_OK;
            }
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);    // makes the primary context current if none is
    if (e != cudaSuccess || p == nullptr) {
        kvm::set_last_error(std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
        return KVM_ERR_CUDA;
    }
    if (!ctx) ctx = current_ctx();
    if (ctx) g_addr.emplace_back(ctx, p);
    *out = p;
    return KVM_OK;
}

}  // namespace

extern "C" kvm_status kvm_score_select_static(const kvm_config *cfg, const void *q,
                                              int32_t n_queries, const void *index,
                                              int64_t n_blocks, float *scores_out,
                                              int32_t *sel_ids_out, int32_t *n_sel_out,
                                              kvm_stream stream) {
    auto bad = [](kvm_status s, const char *m) { kvm::set_last_error(m); return s; };
    if (!cfg) return bad(KVM_ERR_INVALID_ARG, "config is NULL");
    if (!q || !index || !scores_out || !sel_ids_out)
        return bad(KVM_ERR_INVALID_ARG, "q, index, scores_out and sel_ids_out are required");
    if (cfg->n_layers < 1 || cfg->n_kv_heads < 1 || cfg->n_q_heads < 1 ||
        cfg->n_q_heads % cfg->n_kv_heads != 0)
        return bad(KVM_ERR_INVALID_ARG, "layers / heads invalid");
    if (cfg->head_dim != 64 && cfg->head_dim != 128)
        return bad(KVM_ERR_INVALID_ARG, "head_dim must be 64 or 128");
    for (int dt : {cfg->index_dtype, cfg->q_dtype})
        if (dt != KVM_F32 && dt != KVM_BF16) return bad(KVM_ERR_INVALID_ARG, "dtype invalid");
    if (cfg->index_location != KVM_DEVICE)
        return bad(KVM_ERR_INVALID_ARG, "the index must be in device memory");
    if (cfg->sink_blocks < 0 || cfg->recent_blocks < 0 ||
        cfg->view_blocks < cfg->sink_blocks + cfg->recent_blocks + 1)
        return bad(KVM_ERR_INVALID_ARG, "view_blocks must be >= sink + recent + 1");
    if (cfg->score_variant < 0 || cfg->score_variant > 2)
        return bad(KVM_ERR_INVALID_ARG, "score_variant must be 0, 1 or 2");
    if (cfg->candidate_mode != 0 && cfg->candidate_mode != 1)
        return bad(KVM_ERR_INVALID_ARG, "candidate_mode must be 0 or 1");
    if (n_queries < 1 || n_blocks < 1) return bad(KVM_ERR_INVALID_ARG, "empty input");
    if (n_blocks > cfg->max_blocks)
        return bad(KVM_ERR_CAPACITY, "n_blocks beyond max_blocks (the index row stride)");
    const int gqa = cfg->n_q_heads / cfg->n_kv_heads;
    if ((int64_t)n_queries * gqa > kvm::kMaxRows)
        return bad(KVM_ERR_CAPACITY, "n_queries * (H/G) must be <= 256");

    kvm::ScoreShape sh{};
    sh.L = cfg->n_layers;
    sh.G = cfg->n_kv_heads;
    sh.H = cfg->n_q_heads;
    sh.d = cfg->head_dim;
    sh.n_queries = n_queries;
    sh.gqa = gqa;
    sh.rows = n_queries * gqa;
    sh.index_cap = cfg->max_blocks;
    sh.variant = cfg->score_variant;
    // the candidate set and the chunk count exactly as kvm_score_select takes
    // them, so that both entry points sum in the same order
    int64_t c0 = 0, c1 = n_blocks;
    if (cfg->candidate_mode == 1) {
        c0 = cfg->sink_blocks < n_blocks ? cfg->sink_blocks : n_blocks;
        c1 = n_blocks - cfg->recent_blocks > c0 ? n_blocks - cfg->recent_blocks : c0;
    }
    const int nch = c1 > c0 ? kvm::score_chunks(sh, c1 - c0, kvm::kMaxChunks) : 1;
    sh.chunk_cap = nch;

    const size_t LG = (size_t)sh.L * sh.G;
    const size_t part = up256(LG * nch * sh.rows * sizeof(float));
    const size_t rowb = up256(LG * sh.rows * sizeof(float));
    const size_t partial = up256(LG * (size_t)n_blocks * sizeof(float));
    const size_t selb = up256(kvm::select_scratch_bytes());
    const size_t fused = up256(kvm::fused_scratch_bytes(sh.rows));
    const size_t need = 256 + 2 * part + 2 * rowb + partial + selb + fused;
    if (need > SCRATCH_BYTES) {
        char msg[200];
        snprintf(msg, sizeof msg,
                 "needs %zu bytes of scratch, more than the fixed %zu: layers * kv_heads * "
                 "n_blocks must shrink (use kvm_score_select with a workspace)",
                 need, SCRATCH_BYTES);
        return bad(KVM_ERR_CAPACITY, msg);
    }

    // the kernels take device addresses: the index must be device memory (the
    // tensor-core passes stream it with TMA); q and the outputs may also be
    // pinned host memory, used through its device alias
    {
        cudaPointerAttributes a{};
        if (cudaPointerGetAttributes(&a, index) != cudaSuccess || a.type != cudaMemoryTypeDevice) {
            cudaGetLastError();
            return bad(KVM_ERR_INVALID_ARG, "index: device memory required");
        }
    }
    int rs;
    if ((rs = kvm::resolve_kernel_ptr(q, &q, "q")) != KVM_OK) return (kvm_status)rs;
    {
        const void *p = scores_out;
        if ((rs = kvm::resolve_kernel_ptr(p, &p, "scores_out")) != KVM_OK) return (kvm_status)rs;
        scores_out = static_cast<float *>(const_cast<void *>(p));
        p = sel_ids_out;
        if ((rs = kvm::resolve_kernel_ptr(p, &p, "sel_ids_out")) != KVM_OK) return (kvm_status)rs;
        sel_ids_out = static_cast<int32_t *>(const_cast<void *>(p));
    }

    void *base = nullptr;
    kvm_status st = scratch_for_current_context(&base);
    if (st != KVM_OK) return st;
    char *b = static_cast<char *>(base) + 256;   // the first 256 bytes hold the error word
    kvm::ScoreScratch scr{};
    scr.part_m = reinterpret_cast<float *>(b);
    scr.part_z = reinterpret_cast<float *>(b + part);
    scr.row_m = reinterpret_cast<float *>(b + 2 * part);
    scr.row_invz = reinterpret_cast<float *>(b + 2 * part + rowb);
    scr.partial = reinterpret_cast<float *>(b + 2 * part + 2 * rowb);
    int *sel_scratch = reinterpret_cast<int *>(b + 2 * part + 2 * rowb + partial);
    kvm::fused_scratch_carve(&scr, b + 2 * part + 2 * rowb + partial + selb, sh.rows);
    scr.err = static_cast<int *>(base);
    const bool one_launch = c1 > c0 &&
                            kvm::score_fused_supported(cfg->q_dtype, cfg->index_dtype, sh) &&
                            kvm::fused_q_ok(q);

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if ((one_launch &&
         (e = kvm::launch_score_fused(sh, q, index, c0, c1, scr, n_blocks, s)) != cudaSuccess) ||
        (!one_launch && c1 > c0 &&
         ((e = kvm::launch_score_pass1(cfg->q_dtype, cfg->index_dtype, sh, q, index, 0, c0, c1,
                                       0, nch, scr, s)) != cudaSuccess ||
          (e = kvm::launch_score_combine(sh, nch, scr, s)) != cudaSuccess ||
          (e = kvm::launch_score_pass2(cfg->q_dtype, cfg->index_dtype, sh, q, index, 0, c0, c1,
                                       nch, scr, n_blocks, s)) != cudaSuccess)) ||
        (e = kvm::launch_score_reduce(sh, n_blocks, c0, c1, scr, n_blocks, scores_out, s)) !=
            cudaSuccess ||
        (e = kvm::launch_select(scores_out, n_blocks, cfg->sink_blocks, cfg->recent_blocks,
                                cfg->view_blocks, sel_ids_out, sel_scratch, s)) != cudaSuccess) {
        kvm::set_last_error(std::string("launch: ") + cudaGetErrorString(e));
        return KVM_ERR_CUDA;
    }
    if (n_sel_out) *n_sel_out = (int32_t)(n_blocks < cfg->view_blocks ? n_blocks : cfg->view_blocks);
    return KVM_OK;
}

extern "C" kvm_status kvm_score_select_static_status(kvm_stream stream) {
    void *base = nullptr;
    kvm_status st = scratch_for_current_context(&base);
    if (st != KVM_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int flag = 0;
    cudaError_t e;
    if ((e = cudaMemcpyAsync(&flag, base, sizeof(int), cudaMemcpyDeviceToHost, s)) !=
            cudaSuccess ||
        (e = cudaStreamSynchronize(s)) != cudaSuccess) {
        kvm::set_last_error(std::string("reading the error word: ") + cudaGetErrorString(e));
        return KVM_ERR_CUDA;
    }
    if (flag == 0) return KVM_OK;
    if ((e = cudaMemsetAsync(base, 0, sizeof(int), s)) != cudaSuccess ||
        (e = cudaStreamSynchronize(s)) != cudaSuccess) {
        kvm::set_last_error(std::string("clearing the error word: ") + cudaGetErrorString(e));
        return KVM_ERR_CUDA;
    }
    char msg[96];
    if (flag & 4) {
        snprintf(msg, sizeof msg, "a bounded device wait gave up (flag 0x%x)", flag);
        kvm::set_last_error(msg);
        return KVM_ERR_TIMEOUT;
    }
    snprintf(msg, sizeof msg, "device check raised flag 0x%x", flag);
    kvm::set_last_error(msg);
    return KVM_ERR_DEVICE;
}
