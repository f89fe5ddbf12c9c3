// Budgeted block selection: the default selector of KVMem (Virtualizing
// Million-Token Agent Workspaces on a Consumer GPU), §4.3.  Blocks [0, S) and
// [N-W, N) are always kept; the remaining V_b - S - W slots go to the
// candidates of largest R_b, ties to the lower block id, NaN last; the result
// is written in ascending (chronological) order.
//
// A radix select over the 32-bit order-preserving key of R_b (four 8-bit
// digits, most significant first) finds the k-th largest key T and how many
// keys equal to T must be taken; a scan in block order then takes every key
// > T, the first `need` keys == T, and the reserved blocks, and writes the
// ids.  Deterministic: no float atomics, counts only.
//
// Short histories run in one CTA of 1024 threads.  Long ones (kSelManyMin
// blocks and more) spread the same steps over many CTAs, so that enough loads
// are in flight: four histogram launches (each CTA first re-derives the digits
// already chosen from the earlier histograms), one launch that counts each
// segment's taken and tied keys, and one that writes each segment's ids at
// the offset the counts of the segments before it give.
#include <math.h>

#include <algorithm>

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

// One CTA, for histories shorter than kSelManyMin blocks: the keys of all N
// blocks are staged in shared memory once (at most 64 KB), and every pass
// reads them there.
__global__ void __launch_bounds__(kSelThreads)
select_kernel(const float *__restrict__ R, int64_t N, int S, int W, int V,
              int32_t *__restrict__ sel) {
    extern __shared__ uint32_t keys[];     // [N] when N > V
    __shared__ int hist[256];
    __shared__ int warp_sums[32];
    __shared__ uint32_t s_prefix;
    __shared__ int s_remaining;
    const int tid = threadIdx.x;

    if (N <= V) {
        for (int64_t b = tid; b < N; b += blockDim.x) sel[b] = (int32_t)b;
        return;
    }
    // all loads of a thread in flight before its first store
    for (int64_t base = 0; base < N; base += 4 * kSelThreads) {
        float v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t b = base + tid + j * kSelThreads;
            v[j] = b < N ? R[b] : 0.f;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t b = base + tid + j * kSelThreads;
            if (b < N) keys[b] = order_key(v[j]);
        }
    }
    __syncthreads();
    const int64_t c0 = S, c1 = N - W;          // candidate range
    const int k = V - S - W;
    uint32_t prefix = 0, mask = 0;
    int remaining = k;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        for (int64_t b = c0 + tid; b < c1; b += blockDim.x) {
            const uint32_t key = keys[b];
            if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
        }
        __syncthreads();
        // the largest digit whose count, with the counts of all larger digits,
        // reaches the remaining rank: thread t < 256 holds digit 255 - t, and
        // a scan gives each the count of the digits above it
        {
            const int r = 255 - tid;
            const int h = tid < 256 ? hist[r] : 0;
            int total;
            const int above = block_exclusive_scan(h, warp_sums, &total);
            if (tid < 256 && above < remaining && (above + h >= remaining || r == 0)) {
                s_prefix = prefix | ((uint32_t)r << shift);
                s_remaining = remaining - (above + h >= remaining ? above : above + h);
            }
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
        if (b >= c0 && b < c1 && keys[b] == T) ++n_eq;
    int total;
    int eq_rank = block_exclusive_scan(n_eq, warp_sums, &total);
    int n_take = 0;
    {
        int r = eq_rank;
        for (int64_t b = s0; b < s1; ++b) {
            if (b < c0 || b >= c1) { ++n_take; continue; }
            const uint32_t key = keys[b];
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
                const uint32_t key = keys[b];
                if (key > T) take = true;
                else if (key == T) { take = r < need_eq; ++r; }
                else take = false;
            }
            if (take) sel[out++] = (int32_t)b;
        }
    }
}

// ---------------------------------------------------------------- many CTAs

constexpr int kMT = 256;               // threads per CTA
constexpr int kPer = 8;                // blocks per thread per sub-chunk
constexpr int kSub = kMT * kPer;       // blocks per sub-chunk
constexpr int kMaxSegs = 1024;         // segments of the count / write launches
constexpr int64_t kSelManyMin = 16384;

// The digits chosen in passes [0, passes), from the global histograms: the
// largest digit whose count, with the counts of all larger digits, reaches
// the remaining rank (the one-CTA kernel's choice, taken by 256 threads at
// once).  Returns the key prefix and the rank left within it.
__device__ void decode_digits(const int *__restrict__ hist, int passes, int k, uint32_t &prefix,
                              int &remaining, int *warp_sums, int *s_pick) {
    prefix = 0;
    remaining = k;
    const int r = kMT - 1 - (int)threadIdx.x;      // thread t holds digit 255 - t
    for (int p = 0; p < passes; ++p) {
        const int h = hist[p * 256 + r];
        int total;
        const int above = block_exclusive_scan(h, warp_sums, &total);   // digits > r
        if (above < remaining && (above + h >= remaining || r == 0)) {
            s_pick[0] = r;
            s_pick[1] = above + h >= remaining ? above : above + h;
        }
        __syncthreads();
        prefix |= (uint32_t)s_pick[0] << (24 - 8 * p);
        remaining -= s_pick[1];
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kMT)
select_hist_kernel(const float *__restrict__ R, int64_t c0, int64_t c1, int k, int pass,
                   int *__restrict__ hist) {
    __shared__ int h[256];
    __shared__ int warp_sums[32];
    __shared__ int s_pick[2];
    uint32_t prefix;
    int remaining;
    decode_digits(hist, pass, k, prefix, remaining, warp_sums, s_pick);
    const uint32_t mask = pass == 0 ? 0u : 0xFFFFFFFFu << (32 - 8 * pass);
    const int shift = 24 - 8 * pass;
    h[threadIdx.x] = 0;
    __syncthreads();
    for (int64_t base = c0 + (int64_t)blockIdx.x * kSub; base < c1;
         base += (int64_t)gridDim.x * kSub) {
        float v[kPer];
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int64_t b = base + threadIdx.x + j * kMT;
            v[j] = b < c1 ? R[b] : 0.f;
        }
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int64_t b = base + threadIdx.x + j * kMT;
            const uint32_t key = order_key(v[j]);
            if (b < c1 && (key & mask) == prefix) atomicAdd(&h[(key >> shift) & 255u], 1);
        }
    }
    __syncthreads();
    const int c = h[threadIdx.x];
    if (c) atomicAdd(&hist[pass * 256 + threadIdx.x], c);
}

// 0: not taken, 1: taken (reserved, or key > T), 2: tied with T
__device__ __forceinline__ int classify(float x, int64_t b, int64_t c0, int64_t c1, uint32_t T) {
    if (b < c0 || b >= c1) return 1;
    const uint32_t key = order_key(x);
    return key > T ? 1 : key == T ? 2 : 0;
}

// Per segment of [0, N): the blocks taken for sure and the blocks tied with T.
__global__ void __launch_bounds__(kMT)
select_count_kernel(const float *__restrict__ R, int64_t N, int64_t c0, int64_t c1, int k,
                    int64_t seg, const int *__restrict__ hist, int *__restrict__ cnt) {
    __shared__ int warp_sums[32];
    __shared__ int s_pick[2];
    uint32_t T;
    int need_eq;
    decode_digits(hist, 4, k, T, need_eq, warp_sums, s_pick);
    const int64_t s0 = (int64_t)blockIdx.x * seg, s1 = min(N, s0 + seg);
    int n_take = 0, n_eq = 0;
    for (int64_t base = s0; base < s1; base += kSub) {
        float v[kPer];
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int64_t b = base + threadIdx.x + j * kMT;
            v[j] = b < s1 ? R[b] : 0.f;
        }
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int64_t b = base + threadIdx.x + j * kMT;
            if (b < s1) {
                const int c = classify(v[j], b, c0, c1, T);
                n_take += c == 1;
                n_eq += c == 2;
            }
        }
    }
    int tot_take, tot_eq;
    block_exclusive_scan(n_take, warp_sums, &tot_take);
    block_exclusive_scan(n_eq, warp_sums, &tot_eq);
    if (threadIdx.x == 0) {
        cnt[blockIdx.x] = tot_take;
        cnt[kMaxSegs + blockIdx.x] = tot_eq;
    }
}

// Writes segment blockIdx.x's ids in block order, at the offset of the blocks
// the earlier segments take; of the tied blocks, the first need_eq in block
// order are taken.
__global__ void __launch_bounds__(kMT)
select_write_kernel(const float *__restrict__ R, int64_t N, int64_t c0, int64_t c1, int k,
                    int64_t seg, const int *__restrict__ hist, const int *__restrict__ cnt,
                    int32_t *__restrict__ sel, int V) {
    __shared__ int warp_sums[32];
    __shared__ int s_pick[2];
    uint32_t T;
    int need_eq;
    decode_digits(hist, 4, k, T, need_eq, warp_sums, s_pick);
    const int t = threadIdx.x, c = blockIdx.x;
    // the segments before this one: ties before each, then what each takes
    const int per = (gridDim.x + kMT - 1) / kMT;
    const int e0 = min(c, t * per), e1 = min(c, e0 + per);
    int leq = 0;
    for (int e = e0; e < e1; ++e) leq += cnt[kMaxSegs + e];
    int eq_seen;
    int eqb = block_exclusive_scan(leq, warp_sums, &eq_seen);
    int ltake = 0;
    for (int e = e0; e < e1; ++e) {
        const int ce = cnt[kMaxSegs + e];
        ltake += cnt[e] + min(max(need_eq - eqb, 0), ce);
        eqb += ce;
    }
    int out;
    block_exclusive_scan(ltake, warp_sums, &out);
    // this segment's blocks, kPer consecutive ones per thread
    const int64_t s0 = (int64_t)c * seg, s1 = min(N, s0 + seg);
    for (int64_t base = s0; base < s1; base += kSub) {
        int cls[kPer];
        int n_eq = 0;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int64_t b = base + (int64_t)t * kPer + j;
            cls[j] = b < s1 ? classify(R[b], b, c0, c1, T) : 0;
            n_eq += cls[j] == 2;
        }
        int sub_eq;
        int r = eq_seen + block_exclusive_scan(n_eq, warp_sums, &sub_eq);
        int n_take = 0;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            if (cls[j] == 2) {
                cls[j] = r < need_eq ? 1 : 0;
                ++r;
            }
            n_take += cls[j];
        }
        int sub_take;
        int o = out + block_exclusive_scan(n_take, warp_sums, &sub_take);
#pragma unroll
        for (int j = 0; j < kPer; ++j)
            if (cls[j]) {
                if (o < V) sel[o] = (int32_t)(base + (int64_t)t * kPer + j);   // V ids in all
                ++o;
            }
        eq_seen += sub_eq;
        out += sub_take;
    }
}

size_t select_scratch_bytes() { return (4 * 256 + 2 * kMaxSegs) * sizeof(int); }

cudaError_t launch_select(const float *scores, int64_t n_blocks, int sink, int recent,
                          int view_blocks, int32_t *sel_ids, int *scratch, cudaStream_t s) {
    if (n_blocks <= view_blocks || n_blocks < kSelManyMin) {
        const cudaError_t e = cudaFuncSetAttribute(    // per device: set on every call
            select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
            (int)(kSelManyMin * sizeof(uint32_t)));
        if (e != cudaSuccess) return e;
        const size_t smem = n_blocks > view_blocks ? (size_t)n_blocks * sizeof(uint32_t) : 0;
        select_kernel<<<1, kSelThreads, smem, s>>>(scores, n_blocks, sink, recent, view_blocks,
                                                   sel_ids);
        note_launch();
        return cudaGetLastError();
    }
    const int64_t c0 = sink, c1 = n_blocks - recent;
    const int k = view_blocks - sink - recent;
    int *hist = scratch, *cnt = scratch + 4 * 256;
    cudaError_t e = cudaMemsetAsync(hist, 0, 4 * 256 * sizeof(int), s);
    if (e != cudaSuccess) return e;
    const int64_t g1 = std::min<int64_t>((c1 - c0 + kSub - 1) / kSub, 4 * (int64_t)sm_count());
    for (int pass = 0; pass < 4; ++pass) {
        select_hist_kernel<<<(unsigned)g1, kMT, 0, s>>>(scores, c0, c1, k, pass, hist);
        note_launch();
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    const int64_t g2 = std::min<int64_t>((n_blocks + kSub - 1) / kSub, kMaxSegs);
    const int64_t seg = (n_blocks + g2 - 1) / g2;
    select_count_kernel<<<(unsigned)g2, kMT, 0, s>>>(scores, n_blocks, c0, c1, k, seg, hist, cnt);
    note_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    select_write_kernel<<<(unsigned)g2, kMT, 0, s>>>(scores, n_blocks, c0, c1, k, seg, hist, cnt,
                                                     sel_ids, view_blocks);
    note_launch();
    return cudaGetLastError();
}

}  // namespace kvm
