// Mean-K index build.
//
// KVMem (Virtualizing Million-Token Agent Workspaces on a Consumer GPU), §4.3:
// each 32-token block is represented, per layer and KV head, by the mean of its
// position-independent K; §5 (incremental indexing): the mean is taken while the
// block's K pages are still on the GPU, RoPE removed first.
//
// One CTA owns one block and a run of (layer, kv head) pairs.  The block's 32
// rows of the cos/sin table are staged in shared memory once and reused for
// every pair.  Each thread moves 16 bytes of the first half of a token row and
// the matching 16 bytes of the second half (rotate-half partners), un-rotates
// them in float32, optionally writes the raw K, and the 32 tokens are summed
// with warp shuffles plus one shared-memory pass across warps.  HBM traffic per
// (layer, kv head, block): 32*d elements read, 32*d written (raw K), d written.
#include "kvm_internal.cuh"
#include "kvm_vec.cuh"

namespace kvm {

template <typename T, typename TI, int D>
__global__ void __launch_bounds__(32 * (D / 2) / VecTraits<T>::N)
meank_kernel(const T *__restrict__ k_pages, T *__restrict__ raw_out, TI *__restrict__ index,
             int64_t index_cap, int64_t first_block, int LG, int lg_per_cta,
             const float2 *__restrict__ table) {
    constexpr int PPT = VecTraits<T>::N;   // rotation pairs per thread
    constexpr int HD = D / 2;
    constexpr int TPT = HD / PPT;          // threads per token row
    constexpr int NT = 32 * TPT;
    constexpr int NW = NT / 32;
    __shared__ float2 tab[kBlockTokens * HD];
    __shared__ float red[NW][D];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int tok = tid / TPT, c = tid % TPT;
    const int64_t b = blockIdx.x;
    const int64_t gb = first_block + b;

    const float2 *trow = table + gb * kBlockTokens * HD;
    for (int i = tid; i < kBlockTokens * HD; i += NT) tab[i] = trow[i];
    __syncthreads();
    float cs[PPT], sn[PPT];
#pragma unroll
    for (int i = 0; i < PPT; ++i) {
        const float2 t = tab[tok * HD + c * PPT + i];
        cs[i] = t.x;
        sn[i] = t.y;
    }

    const int lg0 = blockIdx.y * lg_per_cta;
    const int lg1 = min(LG, lg0 + lg_per_cta);
    const size_t row = (size_t)tok * D + (size_t)c * PPT;
    auto base_of = [&](int lg) { return ((size_t)b * LG + lg) * kBlockTokens * D; };

    uint4 nx = make_uint4(0, 0, 0, 0), ny = nx;
    if (lg0 < lg1) {
        nx = ld_stream(k_pages + base_of(lg0) + row);
        ny = ld_stream(k_pages + base_of(lg0) + row + HD);
    }
    for (int lg = lg0; lg < lg1; ++lg) {
        const uint4 vx = nx, vy = ny;
        if (lg + 1 < lg1) {  // keep the next pair's loads in flight
            nx = ld_stream(k_pages + base_of(lg + 1) + row);
            ny = ld_stream(k_pages + base_of(lg + 1) + row + HD);
        }
        float x[PPT], y[PPT], rx[PPT], ry[PPT];
        VecTraits<T>::unpack(vx, x);
        VecTraits<T>::unpack(vy, y);
#pragma unroll
        for (int i = 0; i < PPT; ++i) {
            // R_{-p}: (x cos + y sin, y cos - x sin), each product rounded
            rx[i] = __fadd_rn(__fmul_rn(x[i], cs[i]), __fmul_rn(y[i], sn[i]));
            ry[i] = __fsub_rn(__fmul_rn(y[i], cs[i]), __fmul_rn(x[i], sn[i]));
        }
        if (raw_out != nullptr) {
            st_stream(raw_out + base_of(lg) + row, VecTraits<T>::pack(rx));
            st_stream(raw_out + base_of(lg) + row + HD, VecTraits<T>::pack(ry));
        }
#pragma unroll
        for (int off = TPT; off < 32; off <<= 1) {
#pragma unroll
            for (int i = 0; i < PPT; ++i) {
                rx[i] += __shfl_xor_sync(0xffffffffu, rx[i], off);
                ry[i] += __shfl_xor_sync(0xffffffffu, ry[i], off);
            }
        }
        if (lane < TPT) {
#pragma unroll
            for (int i = 0; i < PPT; ++i) {
                red[warp][c * PPT + i] = rx[i];
                red[warp][HD + c * PPT + i] = ry[i];
            }
        }
        __syncthreads();
        if (tid < D) {
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) s += red[w][tid];
            index[((size_t)lg * index_cap + gb) * D + tid] =
                from_float<TI>(s * (1.0f / kBlockTokens));
        }
        __syncthreads();
    }
}

template <typename T, typename TI, int D>
static cudaError_t launch_meank_t(const void *k_pages, void *raw_out, void *index,
                                  int64_t index_cap, int64_t first_block, int64_t n_blocks,
                                  int LG, const float2 *table, cudaStream_t s) {
    constexpr int NT = 32 * (D / 2) / VecTraits<T>::N;
    // enough CTAs per block to fill the machine for small runs, long runs of
    // (layer, kv head) pairs per CTA to amortise the table stage otherwise
    int lg_per_cta = LG;
    const int64_t want_ctas = 152 * 16;
    while (lg_per_cta > 8 && n_blocks * ((LG + lg_per_cta - 1) / lg_per_cta) < want_ctas)
        lg_per_cta = (lg_per_cta + 1) / 2;
    if (lg_per_cta > 64) lg_per_cta = 64;
    dim3 grid((unsigned)n_blocks, (unsigned)((LG + lg_per_cta - 1) / lg_per_cta));
    meank_kernel<T, TI, D><<<grid, NT, 0, s>>>(
        static_cast<const T *>(k_pages), static_cast<T *>(raw_out), static_cast<TI *>(index),
        index_cap, first_block, LG, lg_per_cta, table);
    return cudaGetLastError();
}

cudaError_t launch_meank(int kv_dtype, int index_dtype, int d, const void *k_pages,
                         void *raw_out, void *index, int64_t index_cap, int64_t first_block,
                         int64_t n_blocks, int LG, const float2 *table, int *err,
                         cudaStream_t s) {
    (void)err;
    if (n_blocks <= 0) return cudaSuccess;
#define KVM_MEANK(T, TI, D)                                                              \
    return launch_meank_t<T, TI, D>(k_pages, raw_out, index, index_cap, first_block,     \
                                    n_blocks, LG, table, s)
    if (kv_dtype == BF16 && index_dtype == BF16) {
        if (d == 128) KVM_MEANK(__nv_bfloat16, __nv_bfloat16, 128);
        if (d == 64) KVM_MEANK(__nv_bfloat16, __nv_bfloat16, 64);
    } else if (kv_dtype == BF16 && index_dtype == F32) {
        if (d == 128) KVM_MEANK(__nv_bfloat16, float, 128);
        if (d == 64) KVM_MEANK(__nv_bfloat16, float, 64);
    } else if (kv_dtype == F32 && index_dtype == F32) {
        if (d == 128) KVM_MEANK(float, float, 128);
        if (d == 64) KVM_MEANK(float, float, 64);
    } else if (kv_dtype == F32 && index_dtype == BF16) {
        if (d == 128) KVM_MEANK(float, __nv_bfloat16, 128);
        if (d == 64) KVM_MEANK(float, __nv_bfloat16, 64);
    }
#undef KVM_MEANK
    return cudaErrorInvalidValue;
}

}  // namespace kvm
