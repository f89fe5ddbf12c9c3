// Host-tier admission and eviction of repository blocks: KVMem (Virtualizing
// Million-Token Agent Workspaces on a Consumer GPU) §4.4, retrieval-aware
// hierarchical reuse.  Host memory keeps a bounded set of blocks; admission
// and eviction weigh recent retrieval and cumulative retrieval frequency, so
// that often-recalled blocks stay in host memory across short idle periods.
//
// The policy is LRFU (Lee et al., IEEE Transactions on Computers 50(12),
// 2001): a block's combined recency and frequency value at step t is
// CRF_t(b) = sum over its references t_i of 2^(-lambda (t - t_i)), kept here
// incrementally as its value at the last reference, decayed on demand.  A step
// first creates its new blocks (resident, one reference each), then references
// the selected blocks (a selected block not resident is a miss and becomes
// resident).  While more than `capacity` blocks are resident, the resident
// block with the smallest CRF_t that was not selected in the step is demoted
// (ties: the lower block id first).  Host-only bookkeeping: no device memory.
#include <math.h>

#include <algorithm>
#include <new>
#include <vector>

#include "kvm.h"
#include "kvm_internal.cuh"

struct kvm_tier {
    int64_t capacity = 0;
    double lambda = 0.0;
    int64_t t = 0;
    int64_t n_blocks = 0;
    int64_t n_resident = 0;
    std::vector<double> crf;       // CRF at the block's last reference
    std::vector<int64_t> last;     // step of the last reference, -1 before any
    std::vector<uint8_t> resident;

    double value(int64_t b) const {
        return last[b] < 0 ? 0.0 : crf[b] * exp2(-lambda * (double)(t - last[b]));
    }
    void reference(int64_t b) {
        crf[b] = value(b) + 1.0;
        last[b] = t;
        if (!resident[b]) {
            resident[b] = 1;
            ++n_resident;
        }
    }
};

extern "C" {

kvm_status kvm_tier_create(int64_t capacity_blocks, double lambda, kvm_tier **out) {
    if (!out) {
        kvm::set_last_error("out is NULL");
        return KVM_ERR_INVALID_ARG;
    }
    *out = nullptr;
    if (capacity_blocks < 1 || !(lambda >= 0.0 && lambda <= 1.0)) {
        kvm::set_last_error("capacity must be >= 1 and lambda in [0, 1]");
        return KVM_ERR_INVALID_ARG;
    }
    kvm_tier *t = new (std::nothrow) kvm_tier;
    if (!t) {
        kvm::set_last_error("out of host memory");
        return KVM_ERR_CAPACITY;
    }
    t->capacity = capacity_blocks;
    t->lambda = lambda;
    *out = t;
    return KVM_OK;
}

kvm_status kvm_tier_step(kvm_tier *t, const int32_t *ids, int32_t n_ids, int64_t n_blocks,
                         int32_t *demoted_out, kvm_tier_stats *stats) {
    if (!t || (n_ids > 0 && !ids) || n_ids < 0 || n_blocks < t->n_blocks) {
        kvm::set_last_error("tier step: invalid arguments (history cannot shrink)");
        return KVM_ERR_INVALID_ARG;
    }
    for (int32_t i = 0; i < n_ids; ++i)
        if (ids[i] < 0 || ids[i] >= n_blocks) {
            kvm::set_last_error("tier step: block id out of range");
            return KVM_ERR_INVALID_ARG;
        }
    // every allocation comes before the first change of state, and none
    // throws across the C ABI
    std::vector<uint8_t> prot;
    std::vector<std::pair<double, int64_t>> cand;
    try {
        std::vector<int32_t> sorted(ids, ids + n_ids);
        std::sort(sorted.begin(), sorted.end());
        if (std::adjacent_find(sorted.begin(), sorted.end()) != sorted.end()) {
            kvm::set_last_error("tier step: block ids must be distinct");
            return KVM_ERR_INVALID_ARG;
        }
        t->crf.resize(n_blocks, 0.0);
        t->last.resize(n_blocks, -1);
        t->resident.resize(n_blocks, 0);
        prot.assign((size_t)n_blocks, 0);
        // at most every block resident after this step's creations and hits
        cand.reserve((size_t)std::min<int64_t>(n_blocks,
                                               t->n_resident + (n_blocks - t->n_blocks) + n_ids));
    } catch (...) {
        kvm::set_last_error("out of host memory");
        return KVM_ERR_CAPACITY;
    }
    t->t += 1;
    for (int64_t b = t->n_blocks; b < n_blocks; ++b) t->reference(b);
    t->n_blocks = n_blocks;
    int32_t hits = 0;
    for (int32_t i = 0; i < n_ids; ++i) {
        if (t->resident[ids[i]]) ++hits;
        t->reference(ids[i]);
    }

    int32_t n_dem = 0;
    const int64_t need = t->n_resident - t->capacity;
    if (need > 0) {
        // candidates: resident and not referenced by the step's selection
        // blocks the step selected are protected; blocks only created are not
        for (int32_t i = 0; i < n_ids; ++i) prot[ids[i]] = 1;
        for (int64_t b = 0; b < n_blocks; ++b)
            if (t->resident[b] && !prot[b]) cand.emplace_back(t->value(b), b);
        const size_t k = (size_t)std::min<int64_t>(need, (int64_t)cand.size());
        std::partial_sort(cand.begin(), cand.begin() + k, cand.end());
        for (size_t i = 0; i < k; ++i) {
            const int64_t b = cand[i].second;
            t->resident[b] = 0;
            --t->n_resident;
            if (demoted_out) demoted_out[n_dem] = (int32_t)b;
            ++n_dem;
        }
    }
    if (stats) {
        stats->hits = hits;
        stats->misses = n_ids - hits;
        stats->demoted = n_dem;
        stats->resident = t->n_resident;
    }
    return KVM_OK;
}

kvm_status kvm_tier_resident(const kvm_tier *t, uint8_t *flags, int64_t n) {
    if (!t || (n > 0 && !flags) || n < 0) {
        kvm::set_last_error("tier resident: invalid arguments");
        return KVM_ERR_INVALID_ARG;
    }
    for (int64_t b = 0; b < n; ++b) flags[b] = b < t->n_blocks ? t->resident[b] : 0;
    return KVM_OK;
}

kvm_status kvm_tier_destroy(kvm_tier *t) {
    delete t;
    return KVM_OK;
}

}  // extern "C"
