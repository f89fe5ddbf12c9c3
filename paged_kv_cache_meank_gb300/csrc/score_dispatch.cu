// Chooses the scoring kernel variant for a call: the tensor-core kernels for
// bf16 queries and index (d = 64 or 128, at most 256 query rows per KV head),
// the CUDA-core kernels otherwise or when the configuration asks for them.
#include "kvm_internal.cuh"
#include "score_common.cuh"

namespace kvm {

bool score_uses_tc(int q_dtype, int index_dtype, const ScoreShape &sh) {
    return (sh.variant == 0 || sh.variant == 2) && score_tc_supported(q_dtype, index_dtype, sh);
}

cudaError_t launch_score_pass1(int q_dtype, int index_dtype, const ScoreShape &sh,
                               const void *q, const void *index, int64_t b_index0,
                               int64_t b_begin, int64_t b_end, int chunk0, int n_chunks,
                               const ScoreScratch &scr, cudaStream_t s) {
    if (score_uses_tc(q_dtype, index_dtype, sh))
        return launch_score_pass1_tc(sh, q, index, b_index0, b_begin, b_end, chunk0, n_chunks,
                                     scr, scr.err, s);
    return launch_score_pass1_simt(q_dtype, index_dtype, sh, q, index, b_index0, b_begin, b_end,
                                   chunk0, n_chunks, scr, s);
}

cudaError_t launch_score_pass2(int q_dtype, int index_dtype, const ScoreShape &sh,
                               const void *q, const void *index, int64_t b_index0,
                               int64_t b_begin, int64_t b_end, int n_chunks,
                               const ScoreScratch &scr, int64_t partial_stride,
                               cudaStream_t s) {
    if (score_uses_tc(q_dtype, index_dtype, sh))
        return launch_score_pass2_tc(sh, q, index, b_index0, b_begin, b_end, n_chunks, scr,
                                     partial_stride, scr.err, s);
    return launch_score_pass2_simt(q_dtype, index_dtype, sh, q, index, b_index0, b_begin, b_end,
                                   n_chunks, scr, partial_stride, s);
}

}  // namespace kvm
