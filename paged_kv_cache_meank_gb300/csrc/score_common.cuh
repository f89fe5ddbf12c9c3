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
cudaError_t launch_score_pass1_tc(const ScoreShape &sh, const void *q, const void *index,
                                  int64_t b_index0, int64_t b_begin, int64_t b_end, int chunk0,
                                  int n_chunks, const ScoreScratch &scr, int *err,
                                  cudaStream_t s);
cudaError_t launch_score_pass2_tc(const ScoreShape &sh, const void *q, const void *index,
                                  int64_t b_index0, int64_t b_begin, int64_t b_end, int n_chunks,
                                  const ScoreScratch &scr, int64_t partial_stride, int *err,
                                  cudaStream_t s);

}  // namespace kvm
