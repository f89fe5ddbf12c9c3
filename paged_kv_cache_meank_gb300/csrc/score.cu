// Query-conditioned block scoring, Eq. (10) of KVMem (Virtualizing Million-Token
// Agent Workspaces on a Consumer GPU), §4.3, with the global softmax kept across
// chunks and host-staged tiles (§5, tiled retrieval).
//
// For one (layer l, kv head g) the query rows that read g are the n_queries x
// (H/G) vectors q[l, m, g*(H/G) + hl]; row r = m*(H/G) + hl.  Scores are kept in
// log2 units t = q.kbar * log2(e)/sqrt(d), so that exp(s - M) = 2^(t - M').
//
//   pass 1   per (l, g, chunk): running max and rescaled partition sum per row
//   combine  per (l, g, row): fold the chunks in chunk order -> M, 1/Z
//   pass 2   per (l, g, chunk): for each block, sum over rows of 2^(t - M)/Z
//   reduce   per block: sum over (l, g) in a fixed order, times 1/(L*H)
//
// This file holds the CUDA-core ("SIMT") variant: one thread per query row
// with the row in shared memory, eight Mean-K vectors per step broadcast from
// shared memory, and warp-shuffle reductions across rows for pass 2.  It reads
// any element type.  The tensor-core variant for bf16 lives in score_tc1.cu (pass 1)
// and score_tc.cu (pass 2).
#include <math.h>

#include <algorithm>

#include "kvm_internal.cuh"
#include "kvm_vec.cuh"
#include "score_common.cuh"

namespace kvm {

constexpr int kNB = 8;  // Mean-K vectors per step

template <typename TQ, typename TI, int D, int PASS>
__global__ void score_simt_kernel(const TQ *__restrict__ q, const TI *__restrict__ index,
                                  ScoreShape sh, int64_t b_index0, int64_t b_begin,
                                  int64_t b_end, int chunk0, int64_t chunk_blocks,
                                  ScoreScratch scr, int64_t partial_stride, float scale_log2) {
    extern __shared__ float qs[];                       // [rows][D+1]
    __shared__ __align__(16) float ks[D * kNB];         // [D][kNB]
    __shared__ float red[kMaxRows / 32][kNB];

    const int lg = blockIdx.y;
    const int l = lg / sh.G, g = lg - l * sh.G;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rows = sh.rows;
    const int chunk = blockIdx.x;
    const int64_t cb0 = b_begin + (int64_t)chunk * chunk_blocks;
    const int64_t cb1 = min(b_end, cb0 + chunk_blocks);

    for (int i = tid; i < rows * D; i += blockDim.x) {
        const int r = i / D, k = i - r * D;
        const int m = r / sh.gqa, hl = r - m * sh.gqa;
        qs[r * (D + 1) + k] =
            to_float<TQ>(q[(((size_t)l * sh.n_queries + m) * sh.H + g * sh.gqa + hl) * D + k]);
    }
    const bool valid = tid < rows;
    float m_run = -INFINITY, z_run = 0.f, row_m = 0.f, row_iz = 0.f;
    if (PASS == 2 && valid) {
        row_m = scr.row_m[(size_t)lg * rows + tid];
        row_iz = scr.row_invz[(size_t)lg * rows + tid];
    }
    const TI *ibase = index + (size_t)lg * sh.index_cap * D;

    for (int64_t bb = cb0; bb < cb1; bb += kNB) {
        const int nvalid = (int)min((int64_t)kNB, cb1 - bb);
        __syncthreads();
        for (int i = tid; i < kNB * D; i += blockDim.x) {
            const int nb = i / D, k = i - nb * D;
            float v = 0.f;
            if (nb < nvalid) v = to_float<TI>(ibase[(size_t)(bb + nb - b_index0) * D + k]);
            ks[k * kNB + nb] = v;
        }
        __syncthreads();
        float acc[kNB];
#pragma unroll
        for (int nb = 0; nb < kNB; ++nb) acc[nb] = 0.f;
        if (valid) {
            const float *qr = qs + tid * (D + 1);
            const float4 *k4 = reinterpret_cast<const float4 *>(ks);
#pragma unroll 4
            for (int k = 0; k < D; ++k) {
                const float qv = qr[k];
                const float4 a = k4[2 * k], b = k4[2 * k + 1];
                acc[0] = fmaf(qv, a.x, acc[0]);
                acc[1] = fmaf(qv, a.y, acc[1]);
                acc[2] = fmaf(qv, a.z, acc[2]);
                acc[3] = fmaf(qv, a.w, acc[3]);
                acc[4] = fmaf(qv, b.x, acc[4]);
                acc[5] = fmaf(qv, b.y, acc[5]);
                acc[6] = fmaf(qv, b.z, acc[6]);
                acc[7] = fmaf(qv, b.w, acc[7]);
            }
        }
        if (PASS == 1) {
            if (valid) {
                float tmax = -INFINITY;
#pragma unroll
                for (int nb = 0; nb < kNB; ++nb) {
                    acc[nb] *= scale_log2;
                    if (nb < nvalid) tmax = fmaxf(tmax, acc[nb]);
                }
                const float mn = fmaxf(m_run, tmax);
                float zs = 0.f;
#pragma unroll
                for (int nb = 0; nb < kNB; ++nb)
                    if (nb < nvalid) zs += fast_exp2(acc[nb] - mn);
                z_run = z_run * fast_exp2(m_run - mn) + zs;
                m_run = mn;
            }
        } else {
            float p[kNB];
#pragma unroll
            for (int nb = 0; nb < kNB; ++nb)
                p[nb] = (valid && nb < nvalid)
                            ? fast_exp2(fmaf(acc[nb], scale_log2, -row_m)) * row_iz
                            : 0.f;
#pragma unroll
            for (int nb = 0; nb < kNB; ++nb) {
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    p[nb] += __shfl_xor_sync(0xffffffffu, p[nb], off);
            }
            if (lane == 0) {
#pragma unroll
                for (int nb = 0; nb < kNB; ++nb) red[warp][nb] = p[nb];
            }
            __syncthreads();
            if (tid < nvalid) {
                float s = 0.f;
                const int nw = (int)(blockDim.x >> 5);
                for (int w = 0; w < nw; ++w) s += red[w][tid];
                scr.partial[(size_t)lg * partial_stride + bb + tid] = s;
            }
        }
    }
    if (PASS == 1 && valid) {
        const size_t o = ((size_t)lg * sh.chunk_cap + chunk0 + chunk) * rows + tid;
        scr.part_m[o] = m_run;
        scr.part_z[o] = z_run;
    }
}

int sm_count() {
    // read once per process (thread-safe initialisation of a local static)
    static const int n = [] {
        int dev = 0, v = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
            return v;
        return 152;
    }();
    return n;
}

// Chunks per (layer, kv head).  Each chunk is one CTA and the scoring kernels
// run one CTA per SM, so the pass takes waves = ceil(L*G*chunks / SMs) rounds
// of (tiles per chunk + about four tiles of CTA start-up).  Start from enough
// CTAs for four waves and take the count with the fewest of those tile-times
// among the next 16 (at least 64 blocks per chunk).
int score_chunks(const ScoreShape &sh, int64_t n_blocks, int max_chunks) {
    const int64_t LG = (int64_t)sh.L * sh.G;
    const int64_t sms = sm_count();
    const int64_t by_size = std::max<int64_t>(1, (n_blocks + 63) / 64);
    const int64_t hi = std::min<int64_t>(std::min<int64_t>(by_size, max_chunks), 1 << 20);
    const int64_t lo = std::min<int64_t>(std::max<int64_t>(1, (sms * 4 + LG - 1) / LG), hi);
    int64_t best = lo, best_cost = -1;
    for (int64_t c = lo; c <= std::min(hi, lo + 16); ++c) {
        const int64_t waves = (LG * c + sms - 1) / sms;
        const int64_t tiles = ((n_blocks + c - 1) / c + 127) / 128;
        const int64_t cost = waves * (tiles + 4);
        if (best_cost < 0 || cost < best_cost) {
            best = c;
            best_cost = cost;
        }
    }
    return (int)best;
}

template <typename TQ, typename TI, int D, int PASS>
static cudaError_t simt_t(const ScoreShape &sh, const void *q, const void *index,
                          int64_t b_index0, int64_t b_begin, int64_t b_end, int chunk0,
                          int n_chunks, const ScoreScratch &scr, int64_t partial_stride,
                          cudaStream_t s) {
    const int threads = ((sh.rows + 31) / 32) * 32;
    const size_t smem = (size_t)sh.rows * (D + 1) * sizeof(float);
    auto kern = score_simt_kernel<TQ, TI, D, PASS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t n = b_end - b_begin;
    const int64_t chunk_blocks = (n + n_chunks - 1) / n_chunks;
    dim3 grid((unsigned)n_chunks, (unsigned)(sh.L * sh.G));
    const float scale_log2 = (float)(1.4426950408889634 / sqrt((double)D));
    kern<<<grid, threads, smem, s>>>(static_cast<const TQ *>(q), static_cast<const TI *>(index),
                                     sh, b_index0, b_begin, b_end, chunk0, chunk_blocks, scr,
                                     partial_stride, scale_log2);
    note_launch();
    return cudaGetLastError();
}

template <int PASS>
static cudaError_t simt_dispatch(int q_dtype, int index_dtype, const ScoreShape &sh,
                                 const void *q, const void *index, int64_t b_index0,
                                 int64_t b_begin, int64_t b_end, int chunk0, int n_chunks,
                                 const ScoreScratch &scr, int64_t partial_stride,
                                 cudaStream_t s) {
#define KVM_SIMT(TQ, TI, D)                                                               \
    return simt_t<TQ, TI, D, PASS>(sh, q, index, b_index0, b_begin, b_end, chunk0,        \
                                   n_chunks, scr, partial_stride, s)
    if (q_dtype == F32 && index_dtype == F32) {
        if (sh.d == 128) KVM_SIMT(float, float, 128);
        if (sh.d == 64) KVM_SIMT(float, float, 64);
    } else if (q_dtype == BF16 && index_dtype == BF16) {
        if (sh.d == 128) KVM_SIMT(__nv_bfloat16, __nv_bfloat16, 128);
        if (sh.d == 64) KVM_SIMT(__nv_bfloat16, __nv_bfloat16, 64);
    } else if (q_dtype == F32 && index_dtype == BF16) {
        if (sh.d == 128) KVM_SIMT(float, __nv_bfloat16, 128);
        if (sh.d == 64) KVM_SIMT(float, __nv_bfloat16, 64);
    } else if (q_dtype == BF16 && index_dtype == F32) {
        if (sh.d == 128) KVM_SIMT(__nv_bfloat16, float, 128);
        if (sh.d == 64) KVM_SIMT(__nv_bfloat16, float, 64);
    }
#undef KVM_SIMT
    return cudaErrorInvalidValue;
}

cudaError_t launch_score_pass1_simt(int q_dtype, int index_dtype, const ScoreShape &sh,
                                    const void *q, const void *index, int64_t b_index0,
                                    int64_t b_begin, int64_t b_end, int chunk0, int n_chunks,
                                    const ScoreScratch &scr, cudaStream_t s) {
    return simt_dispatch<1>(q_dtype, index_dtype, sh, q, index, b_index0, b_begin, b_end,
                            chunk0, n_chunks, scr, 0, s);
}

cudaError_t launch_score_pass2_simt(int q_dtype, int index_dtype, const ScoreShape &sh,
                                    const void *q, const void *index, int64_t b_index0,
                                    int64_t b_begin, int64_t b_end, int n_chunks,
                                    const ScoreScratch &scr, int64_t partial_stride,
                                    cudaStream_t s) {
    return simt_dispatch<2>(q_dtype, index_dtype, sh, q, index, b_index0, b_begin, b_end, 0,
                            n_chunks, scr, partial_stride, s);
}

// ---------------------------------------------------------------- combine / reduce

__global__ void score_combine_kernel(ScoreShape sh, int n_chunks, ScoreScratch scr) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const int LG = sh.L * sh.G;
    if (i >= LG * sh.rows) return;
    const int lg = i / sh.rows, r = i - lg * sh.rows;
    const float *pm = scr.part_m + (size_t)lg * sh.chunk_cap * sh.rows + r;
    const float *pz = scr.part_z + (size_t)lg * sh.chunk_cap * sh.rows + r;
    float M = -INFINITY;
    for (int c = 0; c < n_chunks; ++c) M = fmaxf(M, pm[(size_t)c * sh.rows]);
    float Z = 0.f;
    for (int c = 0; c < n_chunks; ++c) Z += pz[(size_t)c * sh.rows] * exp2f(pm[(size_t)c * sh.rows] - M);
    scr.row_m[i] = M;
    scr.row_invz[i] = 1.0f / Z;
}

cudaError_t launch_score_combine(const ScoreShape &sh, int n_chunks_total,
                                 const ScoreScratch &scr, cudaStream_t s) {
    const int n = sh.L * sh.G * sh.rows;
    score_combine_kernel<<<(n + 255) / 256, 256, 0, s>>>(sh, n_chunks_total, scr);
    note_launch();
    return cudaGetLastError();
}

// R_b = (1 / (L H)) * sum over (l, g) of the pass-2 partials, for the scored
// blocks [c0, c1); blocks outside the candidate set get 0.  A CTA takes 32
// blocks, one per lane.  Each of its 16 warps sums a contiguous run of the
// (l, g) pairs into four interleaved accumulators, and the runs are added in
// warp order, so the order of the additions is fixed.
constexpr int kRedWarps = 16;

__global__ void __launch_bounds__(kRedWarps * 32)
score_reduce_kernel(int LG, float inv_lh, int64_t n_blocks, int64_t c0, int64_t c1,
                    const float *__restrict__ partial, int64_t stride, float *__restrict__ out) {
    __shared__ float part[kRedWarps][32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t b = (int64_t)blockIdx.x * 32 + lane;
    const bool scored = b < n_blocks && b >= c0 && b < c1;
    const int lg0 = (int)((int64_t)LG * warp / kRedWarps);
    const int lg1 = (int)((int64_t)LG * (warp + 1) / kRedWarps);
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    if (scored) {
        const float *p = partial + (size_t)lg0 * stride + b;
        int lg = lg0;
        for (; lg + 4 <= lg1; lg += 4, p += 4 * stride) {
            a0 += p[0];
            a1 += p[stride];
            a2 += p[2 * stride];
            a3 += p[3 * stride];
        }
        for (; lg < lg1; ++lg, p += stride) a0 += p[0];
    }
    part[warp][lane] = (a0 + a1) + (a2 + a3);
    __syncthreads();
    if (warp == 0 && b < n_blocks) {
        float s = 0.f;
        for (int w = 0; w < kRedWarps; ++w) s += part[w][lane];
        out[b] = s * inv_lh;
    }
}

cudaError_t launch_score_reduce(const ScoreShape &sh, int64_t n_blocks, int64_t c0, int64_t c1,
                                const ScoreScratch &scr, int64_t partial_stride,
                                float *scores_out, cudaStream_t s) {
    if (n_blocks <= 0) return cudaSuccess;
    const int64_t blocks = (n_blocks + 31) / 32;
    const float inv_lh = (float)(1.0 / ((double)sh.L * sh.H));
    score_reduce_kernel<<<(unsigned)blocks, kRedWarps * 32, 0, s>>>(
        sh.L * sh.G, inv_lh, n_blocks, c0, c1, scr.partial, partial_stride, scores_out);
    note_launch();
    return cudaGetLastError();
}

}  // namespace kvm
