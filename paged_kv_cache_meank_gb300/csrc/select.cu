// Budgeted block selection: the default selector of KVMem (Virtualizing
// Million-Token Agent Workspaces on a Consumer GPU), §4.3.  Blocks [0, S) and
// [N-W, N) are always kept; the remaining V_b - S - W slots go to the
// candidates of largest R_b, ties to the lower block id, NaN last; the result
// is written in ascending (chronological) order.
//
// One CTA of 1024 threads.  A radix select over the 32-bit order-preserving
// key of R_b (four 8-bit digits, most significant first) finds the k-th
// largest key T and how many keys equal to T must be taken; a segmented
// scan in block order then takes every key > T, the first `need` keys == T,
// and the reserved blocks, and writes the ids.  Deterministic: no float
// atomics, counts only.
#include <math.h>

#include "kvm_internal.cuh"

namespace kvm {

constexpr int kSelThreads = 1024;

__device__ __forceinline__ uint32_t order_key(float x) {
    if (isnan(x)) return 0u;      // NaN ranks below every number
    if (x == 0.f) x = 0.f;        // -0 and +0 tie
    const uint32_t u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive scan of one int per thread across the CTA; returns the prefix and
// writes the total to *total.
__device__ int block_exclusive_scan(int v, int *warp_sums, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = (lane < (int)(blockDim.x >> 5)) ? warp_sums[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off) w += y;
        }
        warp_sums[lane] = w;  // inclusive
    }
    __syncthreads();
    const int base = warp > 0 ? warp_sums[warp - 1] : 0;
    const int tot = warp_sums[(blockDim.x >> 5) - 1];
    __syncthreads();
    *total = tot;
    return base + x - v;
}

__global__ void __launch_bounds__(kSelThreads)
select_kernel(const float *__restrict__ R, int64_t N, int S, int W, int V,
              int32_t *__restrict__ sel) {
    __shared__ int hist[256];
    __shared__ int warp_sums[32];
    __shared__ uint32_t s_prefix;
    __shared__ int s_remaining;
    const int tid = threadIdx.x;

    if (N <= V) {
        for (int64_t b = tid; b < N; b += blockDim.x) sel[b] = (int32_t)b;
        return;
    }
    const int64_t c0 = S, c1 = N - W;          // candidate range
    const int k = V - S - W;
    uint32_t prefix = 0, mask = 0;
    int remaining = k;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        for (int64_t b = c0 + tid; b < c1; b += blockDim.x) {
            const uint32_t key = order_key(R[b]);
            if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
        }
        __syncthreads();
        if (tid == 0) {
            int acc = 0, dsel = 0;
            for (int dgt = 255; dgt >= 0; --dgt) {
                if (acc + hist[dgt] >= remaining) { dsel = dgt; break; }
                acc += hist[dgt];
            }
            s_prefix = prefix | ((uint32_t)dsel << shift);
            s_remaining = remaining - acc;
        }
        __syncthreads();
        prefix = s_prefix;
        remaining = s_remaining;
        mask |= 255u << shift;
        __syncthreads();
    }
    const uint32_t T = prefix;     // key of the k-th largest candidate
    const int need_eq = remaining; // how many keys == T to take (lowest ids first)

    // Segmented compaction in block order.
    const int64_t seg = (N + blockDim.x - 1) / blockDim.x;
    const int64_t s0 = min(N, (int64_t)tid * seg), s1 = min(N, s0 + seg);
    int n_eq = 0;
    for (int64_t b = s0; b < s1; ++b)
        if (b >= c0 && b < c1 && order_key(R[b]) == T) ++n_eq;
    int total;
    int eq_rank = block_exclusive_scan(n_eq, warp_sums, &total);
    int n_take = 0;
    {
        int r = eq_rank;
        for (int64_t b = s0; b < s1; ++b) {
            if (b < c0 || b >= c1) { ++n_take; continue; }
            const uint32_t key = order_key(R[b]);
            if (key > T) ++n_take;
            else if (key == T) { if (r < need_eq) ++n_take; ++r; }
        }
    }
    int out = block_exclusive_scan(n_take, warp_sums, &total);
    {
        int r = eq_rank;
        for (int64_t b = s0; b < s1; ++b) {
            bool take;
            if (b < c0 || b >= c1) take = true;
            else {
                const uint32_t key = order_key(R[b]);
                if (key > T) take = true;
                else if (key == T) { take = r < need_eq; ++r; }
                else take = false;
            }
            if (take) sel[out++] = (int32_t)b;
        }
    }
}

cudaError_t launch_select(const float *scores, int64_t n_blocks, int sink, int recent,
                          int view_blocks, int32_t *sel_ids, cudaStream_t s) {
    select_kernel<<<1, kSelThreads, 0, s>>>(scores, n_blocks, sink, recent, view_blocks,
                                            sel_ids);
    return cudaGetLastError();
}

}  // namespace kvm
