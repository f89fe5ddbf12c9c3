// Pieces shared by the scoring kernels.
#pragma once

#include <cuda.h>

#include "kvm_internal.cuh"

namespace kvm {

// 2^x with the hardware approximation (ex2.approx, relative error about 2^-22);
// 2^-inf = 0.
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Online softmax statistics of one query row over the first nv of NV loaded
// scores: running max m (log2 units) and the partition sum z rescaled to it.
template <int NV>
__device__ __forceinline__ void online_update(const uint32_t *r, int nv, float c, float &m,
                                              float &z) {
    if (nv <= 0) return;
    float mx0 = -INFINITY, mx1 = -INFINITY;
    if (nv == NV) {
#pragma unroll
        for (int k = 0; k < NV; k += 2) {
            mx0 = fmaxf(mx0, __uint_as_float(r[k]));
            mx1 = fmaxf(mx1, __uint_as_float(r[k + 1]));
        }
    } else {
#pragma unroll
        for (int k = 0; k < NV; ++k)
            if (k < nv) mx0 = fmaxf(mx0, __uint_as_float(r[k]));
    }
    const float mn = fmaxf(m, fmaxf(mx0, mx1) * c);
    float zs = 0.f;
#pragma unroll
    for (int k = 0; k < NV; ++k)
        if (k < nv) zs += fast_exp2(fmaf(__uint_as_float(r[k]), c, -mn));
    z = z * fast_exp2(m - mn) + zs;
    m = mn;
}

// Row statistics with the reference held fixed: while every term of a full
// tile stays below 2^64 relative to the row's current reference m, the tile
// only adds its terms to z (no max over the tile).  A larger term, the row's
// first tile and a ragged tile take the exact online update, which moves m to
// the running maximum.  (m, z) stays an exact pair for any m: the partition sum
// is z * 2^m, and pass 2 divides by it through m + log2 z.
template <int NV>
__device__ __forceinline__ void row_update(const uint32_t *r, int nv, float c, float &m,
                                           float &z) {
    if (nv == NV && m != -INFINITY) {
        const float2 c2 = make_float2(c, c), nm2 = make_float2(-m, -m);
        float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < NV; k += 4) {
            const float2 x01 = __ffma2_rn(
                make_float2(__uint_as_float(r[k]), __uint_as_float(r[k + 1])), c2, nm2);
            const float2 x23 = __ffma2_rn(
                make_float2(__uint_as_float(r[k + 2]), __uint_as_float(r[k + 3])), c2, nm2);
            a0 = __fadd2_rn(a0, make_float2(fast_exp2(x01.x), fast_exp2(x01.y)));
            a1 = __fadd2_rn(a1, make_float2(fast_exp2(x23.x), fast_exp2(x23.y)));
        }
        const float zs = (a0.x + a0.y) + (a1.x + a1.y);
        if (zs <= 0x1p64f) {   // false for inf and NaN as well
            z += zs;
            return;
        }
    }
    online_update<NV>(r, nv, c, m, z);
}

// Sum of 2^(v*c + no) over n loaded columns (n a multiple of 16, at most 64;
// no = minus the row offset).  Arguments and partial sums use the packed
// float32x2 FMA / add of sm_100-family GPUs, two elements per instruction.
__device__ __forceinline__ float exp_sum(const uint32_t *r, const float *no, int n, float c) {
    const float2 c2 = make_float2(c, c);
    float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < 64; k += 4) {
        if (k < n) {
            const float4 o4 = *reinterpret_cast<const float4 *>(no + k);
            const float2 x01 = __ffma2_rn(
                make_float2(__uint_as_float(r[k]), __uint_as_float(r[k + 1])), c2,
                make_float2(o4.x, o4.y));
            const float2 x23 = __ffma2_rn(
                make_float2(__uint_as_float(r[k + 2]), __uint_as_float(r[k + 3])), c2,
                make_float2(o4.z, o4.w));
            a0 = __fadd2_rn(a0, make_float2(fast_exp2(x01.x), fast_exp2(x01.y)));
            a1 = __fadd2_rn(a1, make_float2(fast_exp2(x23.x), fast_exp2(x23.y)));
        }
    }
    return (a0.x + a0.y) + (a1.x + a1.y);
}

// exp_sum over a compile-time count of columns (the common shapes), with no
// per-column guards, so that the whole sum is one straight-line schedule.
template <int NC>
__device__ __forceinline__ float exp_sum_n(const uint32_t *r, const float *no, float c) {
    const float2 c2 = make_float2(c, c);
    float2 a[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                   make_float2(0.f, 0.f)};
#pragma unroll
    for (int k = 0; k < NC; k += 4) {
        const float4 o4 = *reinterpret_cast<const float4 *>(no + k);
        const float2 x01 = __ffma2_rn(
            make_float2(__uint_as_float(r[k]), __uint_as_float(r[k + 1])), c2,
            make_float2(o4.x, o4.y));
        const float2 x23 = __ffma2_rn(
            make_float2(__uint_as_float(r[k + 2]), __uint_as_float(r[k + 3])), c2,
            make_float2(o4.z, o4.w));
        const int j = (k >> 2) & 1;
        a[2 * j] = __fadd2_rn(a[2 * j], make_float2(fast_exp2(x01.x), fast_exp2(x01.y)));
        a[2 * j + 1] = __fadd2_rn(a[2 * j + 1], make_float2(fast_exp2(x23.x), fast_exp2(x23.y)));
    }
    const float2 s01 = __fadd2_rn(a[0], a[1]), s23 = __fadd2_rn(a[2], a[3]);
    return (s01.x + s01.y) + (s23.x + s23.y);
}

cudaError_t launch_score_pass1_simt(int q_dtype, int index_dtype, const ScoreShape &sh,
                                    const void *q, const void *index, int64_t b_index0,
                                    int64_t b_begin, int64_t b_end, int chunk0, int n_chunks,
                                    const ScoreScratch &scr, cudaStream_t s);
cudaError_t launch_score_pass2_simt(int q_dtype, int index_dtype, const ScoreShape &sh,
                                    const void *q, const void *index, int64_t b_index0,
                                    int64_t b_begin, int64_t b_end, int n_chunks,
                                    const ScoreScratch &scr, int64_t partial_stride,
                                    cudaStream_t s);

bool score_tc_supported(int q_dtype, int index_dtype, const ScoreShape &sh);
// 2-D tensor map over an index buffer (rows = L * G * index_cap Mean-K
// vectors of d bf16) with 64 x box_rows boxes and 128-byte swizzle.
bool make_index_map(CUtensorMap *m, const void *index, int d, int64_t n_rows, int box_rows);
// 3-D tensor map over the queries [L][n_queries][H][d] (bf16) viewed as
// (d, H, L * n_queries): one 64 x gqa x n_queries box is the 64-element K atom
// of the n_queries * gqa query rows of one (layer, kv head), row
// r = m * gqa + hl, in 128-byte-swizzled rows.
bool make_q_map(CUtensorMap *m, const void *q, int d, int H, int64_t n_lq, int gqa,
                int n_queries);
cudaError_t launch_score_pass1_tc(const ScoreShape &sh, const void *q, const void *index,
                                  int64_t b_index0, int64_t b_begin, int64_t b_end, int chunk0,
                                  int n_chunks, const ScoreScratch &scr, int *err,
                                  cudaStream_t s);
cudaError_t launch_score_pass2_tc(const ScoreShape &sh, const void *q, const void *index,
                                  int64_t b_index0, int64_t b_begin, int64_t b_end, int n_chunks,
                                  const ScoreScratch &scr, int64_t partial_stride, int *err,
                                  cudaStream_t s);

}  // namespace kvm
