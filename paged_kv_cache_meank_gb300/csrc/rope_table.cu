// RoPE cos/sin table: entry [p][i] = (cos(p * w_i), sin(p * w_i)) evaluated in
// double precision and rounded once to float32.  KVMem (Virtualizing
// Million-Token Agent Workspaces on a Consumer GPU), §4.4: precomputed RoPE
// sine/cosine tables keep reconstruction cheap.
#include "kvm_internal.cuh"

namespace kvm {

__global__ void rope_table_kernel(float2 *__restrict__ table, int64_t n_pos, int half_d,
                                  Omega om) {
    const int64_t total = n_pos * half_d;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t p = idx / half_d;
        const int i = (int)(idx - p * half_d);
        const double a = (double)p * om.w[i];
        double sn, cs;
        sincos(a, &sn, &cs);
        table[idx] = make_float2((float)cs, (float)sn);
    }
}

cudaError_t launch_rope_table(float2 *table, int64_t n_pos, int half_d, const Omega &om,
                              cudaStream_t s) {
    const int64_t total = n_pos * half_d;
    int64_t blocks = (total + 255) / 256;
    if (blocks > (int64_t)sm_count() * 64) blocks = (int64_t)sm_count() * 64;
    if (blocks < 1) blocks = 1;
    rope_table_kernel<<<(unsigned)blocks, 256, 0, s>>>(table, n_pos, half_d, om);
    note_launch();
    return cudaGetLastError();
}

}  // namespace kvm
