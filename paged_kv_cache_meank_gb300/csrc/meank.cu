// Mean-K index build.
//
// KVMem (Virtualizing Million-Token Agent Workspaces on a Consumer GPU), §4.3:
// each 32-token block is represented, per layer and KV head, by the mean of its
// position-independent K; §5 (incremental indexing): the mean is taken while the
// block's K pages are still on the GPU, RoPE removed first.
//
// One CTA owns one block and a run of (layer, kv head) pairs; the block's 32
// rows of the cos/sin table are staged in shared memory once.  Each warp then
// owns whole (layer, kv head) pairs, so no CTA barrier sits in the streaming
// loop: a lane owns 16 bytes of the first half of a token row and the matching
// 16 bytes of the second half (rotate-half partners) for a fixed column slice,
// walks its share of the 32 tokens with loads issued in groups of 128 bytes
// per lane, un-rotates them in float32, optionally writes the raw
// K, and keeps the token sum in registers; two shuffle rounds finish the sum
// across the lanes that share a column slice.  HBM traffic per (layer, kv
// head, block): 32*d elements read, 32*d written (raw K), d written.
#include "kvm_internal.cuh"
#include "kvm_vec.cuh"

namespace kvm {

constexpr int kMeanKWarps = 4;
// CTAs per SM the register budget is sized for.  2- and 4-byte pages: four,
// which leave 128 registers a thread, so nothing spills (six capped it at 80
// and spilled 64 bytes at d = 128: the 256K build took 10.53 ms against
// 10.40).  e4m3 pages carry half the bytes per load, and the extra warps of
// six CTAs keep more of them in flight (5.47 ms against 6.20 with four).
template <typename T>
constexpr int meank_min_ctas() { return sizeof(T) == 1 ? 6 : 4; }

template <typename T, typename TI, int D>
__global__ void __launch_bounds__(kMeanKWarps * 32, meank_min_ctas<T>())
meank_kernel(const T *__restrict__ k_pages, T *__restrict__ raw_out, TI *__restrict__ index,
             int64_t index_cap, int64_t first_block, int LG, int lg_per_cta,
             const float2 *__restrict__ table) {
    constexpr int PPT = VecTraits<T>::N;     // rotation pairs per 16-byte vector
    constexpr int HD = D / 2;
    constexpr int TPT = HD / PPT;            // lanes per token row
    constexpr int TOK = 32 / TPT;            // tokens per warp-wide sweep
    constexpr int ITERS = 32 / TOK;          // sweeps over the block's 32 tokens
    // sweeps with loads in flight together: 128 bytes per lane
    constexpr int GROUP = ITERS < 128 / (2 * (int)sizeof(typename VecTraits<T>::V))
                              ? ITERS
                              : 128 / (2 * (int)sizeof(typename VecTraits<T>::V));
    using V = typename VecTraits<T>::V;
    // cos/sin of (token, column slice): PPT pairs padded by 2 so that the eight
    // lanes of one shared-memory phase hit distinct banks
    constexpr int ROW = PPT + 2;
    __shared__ __align__(16) float2 tab[kBlockTokens * TPT * ROW];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = lane % TPT, t0 = lane / TPT;
    const int64_t b = blockIdx.x;
    const int64_t gb = first_block + b;

    const float2 *trow = table + gb * kBlockTokens * HD;
    for (int i = tid; i < kBlockTokens * HD; i += kMeanKWarps * 32) {
        const int t = i / HD, j = i - t * HD;
        tab[(t * TPT + j / PPT) * ROW + j % PPT] = trow[i];
    }
    __syncthreads();

    const int lg0 = blockIdx.y * lg_per_cta;
    const int lg1 = min(LG, lg0 + lg_per_cta);
    for (int lg = lg0 + warp; lg < lg1; lg += kMeanKWarps) {
        const size_t base = ((size_t)b * LG + lg) * kBlockTokens * D;
        const T *src = k_pages + base;
        float ax[PPT], ay[PPT];
#pragma unroll
        for (int k = 0; k < PPT; ++k) ax[k] = ay[k] = 0.f;
#pragma unroll
        for (int g0 = 0; g0 < ITERS; g0 += GROUP) {
            V vx[GROUP], vy[GROUP];
#pragma unroll
            for (int i = 0; i < GROUP; ++i) {
                const int t = t0 + (g0 + i) * TOK;
                const size_t off = (size_t)t * D + (size_t)c * PPT;
                ld_stream_v(src + off, vx[i]);
                ld_stream_v(src + off + HD, vy[i]);
            }
#pragma unroll
            for (int i = 0; i < GROUP; ++i) {
                const int t = t0 + (g0 + i) * TOK;
                float x[PPT], y[PPT], rx[PPT], ry[PPT];
                VecTraits<T>::unpack(vx[i], x);
                VecTraits<T>::unpack(vy[i], y);
                const float4 *cs4 = reinterpret_cast<const float4 *>(tab + (t * TPT + c) * ROW);
                float2 cw[PPT];
#pragma unroll
                for (int k = 0; k < PPT / 2; ++k) {
                    const float4 w4 = cs4[k];
                    cw[2 * k] = make_float2(w4.x, w4.y);
                    cw[2 * k + 1] = make_float2(w4.z, w4.w);
                }
#pragma unroll
                for (int k = 0; k < PPT; ++k) {
                    const float2 w = cw[k];
                    // R_{-p}: (x cos + y sin, y cos - x sin), each product rounded
                    rx[k] = __fadd_rn(__fmul_rn(x[k], w.x), __fmul_rn(y[k], w.y));
                    ry[k] = __fsub_rn(__fmul_rn(y[k], w.x), __fmul_rn(x[k], w.y));
                    ax[k] += rx[k];
                    ay[k] += ry[k];
                }
                if (raw_out != nullptr) {
                    const size_t off = base + (size_t)t * D + (size_t)c * PPT;
                    st_stream_v(raw_out + off, VecTraits<T>::pack(rx));
                    st_stream_v(raw_out + off + HD, VecTraits<T>::pack(ry));
                }
            }
        }
#pragma unroll
        for (int off = TPT; off < 32; off <<= 1) {
#pragma unroll
            for (int k = 0; k < PPT; ++k) {
                ax[k] += __shfl_xor_sync(0xffffffffu, ax[k], off);
                ay[k] += __shfl_xor_sync(0xffffffffu, ay[k], off);
            }
        }
        if (lane < TPT) {
            TI *dst = index + ((size_t)lg * index_cap + gb) * D + (size_t)c * PPT;
#pragma unroll
            for (int k = 0; k < PPT; ++k) {
                dst[k] = from_float<TI>(ax[k] * (1.0f / kBlockTokens));
                dst[HD + k] = from_float<TI>(ay[k] * (1.0f / kBlockTokens));
            }
        }
    }
}

template <typename T, typename TI, int D>
static cudaError_t launch_meank_t(const void *k_pages, void *raw_out, void *index,
                                  int64_t index_cap, int64_t first_block, int64_t n_blocks,
                                  int LG, const float2 *table, cudaStream_t s) {
    // long runs of (layer, kv head) pairs per CTA amortise the table stage (16 KB
    // per CTA at d = 128); short ones keep the machine full when few blocks are
    // built.  The cap was measured on the 256K build: 128 pairs for 2- and
    // 4-byte elements, 256 for e4m3, whose pairs carry half the bytes.
    int lg_per_cta = LG;
    const int64_t want_ctas = (int64_t)sm_count() * 16;
    while (lg_per_cta > kMeanKWarps &&
           n_blocks * ((LG + lg_per_cta - 1) / lg_per_cta) < want_ctas)
        lg_per_cta = (lg_per_cta + 1) / 2;
    constexpr int kCap = (sizeof(T) == 1 ? 64 : 32) * kMeanKWarps;
    if (lg_per_cta > kCap) lg_per_cta = kCap;
    dim3 grid((unsigned)n_blocks, (unsigned)((LG + lg_per_cta - 1) / lg_per_cta));
    meank_kernel<T, TI, D><<<grid, kMeanKWarps * 32, 0, s>>>(
        static_cast<const T *>(k_pages), static_cast<T *>(raw_out), static_cast<TI *>(index),
        index_cap, first_block, LG, lg_per_cta, table);
    note_launch();
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
    } else if (kv_dtype == E4M3 && index_dtype == BF16) {
        if (d == 128) KVM_MEANK(e4m3, __nv_bfloat16, 128);
        if (d == 64) KVM_MEANK(e4m3, __nv_bfloat16, 64);
    } else if (kv_dtype == E4M3 && index_dtype == F32) {
        if (d == 128) KVM_MEANK(e4m3, float, 128);
        if (d == 64) KVM_MEANK(e4m3, float, 64);
    }
#undef KVM_MEANK
    return cudaErrorInvalidValue;
}

}  // namespace kvm
