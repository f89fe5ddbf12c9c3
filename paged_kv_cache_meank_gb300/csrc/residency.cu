// The residency diff of one kvm_step on the device: the delta working set of
// KVMem (Virtualizing Million-Token Agent Workspaces on a Consumer GPU), §4.4.
// A selected block already held by a pool page is a hit and keeps its page; a
// selected block held by no page is a miss; pages not holding a selected block
// are free, and the misses, in ascending slot order, take the free pages in
// ascending page order.  A hit whose compact position moved is re-RoPE'd (a
// bounded delta rotation of its K while its page has had fewer than `limit`
// in a row, else a rebuild from raw K); every miss is RoPE'd from raw K.
//
// One CTA walks the selection and the pool with block-wide prefix sums, so the
// step needs no selected ids on the host: it writes the page table, one
// assembly descriptor per slot that needs RoPE (in slot order, their count in
// counts[0]) and the new residency, and counts hits, misses, delta rotations
// and evictions.  Which blocks the current step selected is an epoch stamp per
// block, so nothing is cleared between steps.
#include "kvm_internal.cuh"

namespace kvm {

namespace {

constexpr int kThreads = 1024;

// Exclusive prefix sum of flag(i) over i in [0, n) in index order; calls
// out(i, rank) for every i whose flag is set and returns the total.  Every
// thread of the CTA must call it.
template <typename F, typename O>
__device__ int block_scan(int n, F flag, O out, int *warp_tot) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int carry = 0;
    for (int base = 0; base < n; base += kThreads) {
        const int i = base + tid;
        const int f = i < n && flag(i) ? 1 : 0;
        int x = f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_tot[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int t = warp_tot[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, t, o);
                if (lane >= o) t += y;
            }
            warp_tot[lane] = t;                     // inclusive over warps
        }
        __syncthreads();
        const int before = carry + (warp ? warp_tot[warp - 1] : 0) + x - f;
        if (f) out(i, before);
        carry += warp_tot[31];
        __syncthreads();
    }
    return carry;
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1) residency_diff_kernel(ResidencyArgs a) {
    __shared__ int warp_tot[32];
    __shared__ int s_count[4];                      // hits, delta, evicted, bad ids
    __shared__ int32_t s_epoch;
    const int tid = threadIdx.x;
    const int n = a.n_sel, P = a.P;
    if (tid < 4) s_count[tid] = 0;
    // this step's stamp: one more than the last step's, counted on the device
    if (tid == 0) s_epoch = ++*a.epoch;
    __syncthreads();
    const int32_t epoch = s_epoch;
    // hits and the epoch stamp of every selected block
    for (int j = tid; j < n; j += kThreads) {
        const int32_t b = a.sel[j];
        int32_t p = -1;
        if (b >= 0 && b < a.max_blocks) {
            a.stamp[b] = epoch;
            p = a.page_of_block[b];
        } else {
            atomicAdd(&s_count[3], 1);
        }
        a.slot_page[j] = p;
        if (p >= 0) atomicAdd(&s_count[0], 1);
    }
    __syncthreads();
    if (s_count[3]) {                               // an id out of range: change nothing
        if (tid == 0) atomicOr(a.err, 2);
        if (tid < 8) a.counts[tid] = 0;
        return;
    }
    // free pages in ascending order; then the misses take them in slot order
    const int n_free = block_scan(
        P,
        [&](int p) {
            const int32_t b = a.block_of_page[p];
            return b < 0 || a.stamp[b] != epoch;
        },
        [&](int p, int r) { a.free_list[r] = p; }, warp_tot);
    const int n_miss = n - s_count[0];
    if (n_miss > n_free) {                          // cannot happen with pool_pages >= view_blocks
        if (tid == 0) atomicOr(a.err, 2);
        if (tid < 8) a.counts[tid] = 0;
        return;
    }
    block_scan(
        n, [&](int j) { return a.slot_page[j] < 0; },
        [&](int j, int r) { a.slot_page[j] = -2 - a.free_list[r]; }, warp_tot);
    __syncthreads();
    // descriptors (slot order) from the residency as it was before this step
    auto needs_rope = [&](int j) {
        const int32_t p = a.slot_page[j];
        return p < -1 || a.baked_pos[p] != j * kBlockTokens;
    };
    const int n_desc = block_scan(
        n, needs_rope,
        [&](int j, int r) {
            const int32_t sp = a.slot_page[j];
            const bool miss = sp < -1;
            const int32_t p = miss ? -2 - sp : sp;
            const int64_t b = a.sel[j];
            const int64_t want = (int64_t)j * kBlockTokens;
            SlotDesc d{};
            d.dst_k = a.pool_k + (size_t)p * a.blk;
            d.pos0 = want;
            if (!miss) {
                if (a.delta_limit > 0 && a.delta_count[p] < a.delta_limit) {
                    // bounded delta re-RoPE: rotate the page's K in place
                    d.src_k = d.dst_k;
                    d.pos0 = want - a.baked_pos[p];
                    d.flags = kSlotDelta;
                } else {
                    d.src_k = a.pool_raw ? a.pool_raw + (size_t)p * a.blk
                                         : a.repo_k + (size_t)b * a.blk;
                }
            } else {
                d.src_k = a.repo_k + (size_t)b * a.blk;
                d.src_v = a.repo_v + (size_t)b * a.blk;
                d.dst_v = a.pool_v + (size_t)p * a.blk;
                // the GPU reads the block from the pinned host repository and
                // also keeps its raw K in the page
                d.dst_raw = a.pull && a.pool_raw ? a.pool_raw + (size_t)p * a.blk : nullptr;
            }
            a.desc[r] = d;
        },
        warp_tot);
    // the new residency
    for (int j = tid; j < n; j += kThreads) {
        const int32_t sp = a.slot_page[j];
        const bool miss = sp < -1;
        const int32_t p = miss ? -2 - sp : sp;
        const int32_t b = a.sel[j];
        const int32_t want = j * kBlockTokens;
        if (miss) {
            const int32_t old = a.block_of_page[p];
            if (old >= 0) {
                a.page_of_block[old] = -1;
                atomicAdd(&s_count[2], 1);
            }
            a.block_of_page[p] = b;
            a.page_of_block[b] = p;
            a.delta_count[p] = 0;
        } else if (a.baked_pos[p] != want) {
            if (a.delta_limit > 0 && a.delta_count[p] < a.delta_limit) {
                ++a.delta_count[p];
                atomicAdd(&s_count[1], 1);
            } else {
                a.delta_count[p] = 0;
            }
        }
        a.baked_pos[p] = want;
        a.page_table[j] = p;
    }
    __syncthreads();
    if (tid == 0) {
        a.counts[0] = n_desc;
        a.counts[1] = s_count[0];                   // hits
        a.counts[2] = n_miss;
        a.counts[3] = s_count[1];                   // delta rotations
        a.counts[4] = s_count[2];                   // evicted
    }
}

cudaError_t launch_residency_diff(const ResidencyArgs &a, cudaStream_t s) {
    residency_diff_kernel<<<1, kThreads, 0, s>>>(a);
    note_launch();
    return cudaGetLastError();
}

}  // namespace kvm
