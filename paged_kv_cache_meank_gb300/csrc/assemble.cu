// Execution-view assembly: gather + re-RoPE + V copy.
//
// KVMem (Virtualizing Million-Token Agent Workspaces on a Consumer GPU), §4.4:
// a block entering the execution view gets RoPE applied to its position-
// independent raw K at its compact position and the result is written into its
// destination page; V is copied unchanged.  InferScale (GPU-Native KV Injection
// for Personalized LLM Serving), Theorem 6: rotating stored pre-RoPE keys at
// any chosen position yields exactly the scores they would have there.
//
// One CTA owns one view slot and a run of (layer, kv head) pairs.  The slot's
// 32 rows of the cos/sin table (positions 32j .. 32j+31) are staged in shared
// memory once.  Each thread rotates 8 (bf16) or 4 (float32) rotate-half pairs
// of one token per pair of 16-byte loads and copies the matching 32 bytes of V.
// HBM traffic per view token: L*G*d elements each of raw K read, K written,
// V read, V written.
#include "kvm_internal.cuh"
#include "kvm_vec.cuh"

namespace kvm {

template <typename T, int D>
struct SlotWork {
    static constexpr int PPT = VecTraits<T>::N;
    static constexpr int HD = D / 2;
    static constexpr int TPT = HD / PPT;
    static constexpr int NT = 32 * TPT;

    // Rotate one block's K to positions pos0 + t for pairs [lg0, lg1) and copy V.
    // src_k and dst_k may be the same block (an in-place delta rotation), so
    // they carry no __restrict__
    // U: (layer, kv head) pairs whose loads are issued before any of them is
    // stored.  Batching pays for sources in device memory; for blocks read
    // from pinned host memory over the host link, one pair at a time was
    // measured faster.
    template <int U>
    __device__ static void run(const T *src_k, const T *__restrict__ src_v,
                               T *dst_k, T *__restrict__ dst_v, int64_t pos0,
                               int lg0, int lg1, const float2 *__restrict__ table,
                               float2 *tab, T *__restrict__ dst_raw = nullptr,
                               bool delta = false) {
        const int tid = threadIdx.x;
        const int tok = tid / TPT, c = tid % TPT;
        if (!delta) {
            const float2 *trow = table + pos0 * HD;
            for (int i = tid; i < kBlockTokens * HD; i += NT) tab[i] = trow[i];
        } else {
            // every token turns by the same angle delta * w_i: row |delta| for all
            // tokens, sin negated for a negative delta
            const int64_t ad = pos0 < 0 ? -pos0 : pos0;
            const float sg = pos0 < 0 ? -1.f : 1.f;
            const float2 *trow = table + ad * HD;
            for (int i = tid; i < kBlockTokens * HD; i += NT) {
                const float2 w = trow[i % HD];
                tab[i] = make_float2(w.x, sg * w.y);
            }
        }
        __syncthreads();
        float cs[PPT], sn[PPT];
#pragma unroll
        for (int i = 0; i < PPT; ++i) {
            const float2 t = tab[tok * HD + c * PPT + i];
            cs[i] = t.x;
            sn[i] = t.y;
        }
        const size_t row = (size_t)tok * D + (size_t)c * PPT;
        const bool do_v = (src_v != nullptr) && (dst_v != nullptr);
        using V = typename VecTraits<T>::V;
        // The loads of U pairs are issued explicitly ahead of their stores
        // because src_k and dst_k may alias (in-place delta rotation);
        // different pairs never overlap, and each element is still read before
        // it is written.
        constexpr int kOuterUnroll = U == 1 ? 2 : 1;
#pragma unroll kOuterUnroll
        for (int lg = lg0; lg < lg1; lg += U) {
            V vx[U], vy[U], wx[U], wy[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (lg + u < lg1) {
                    const size_t off = (size_t)(lg + u) * kBlockTokens * D + row;
                    ld_stream_v(src_k + off, vx[u]);
                    ld_stream_v(src_k + off + HD, vy[u]);
                    if (do_v) {
                        ld_stream_v(src_v + off, wx[u]);
                        ld_stream_v(src_v + off + HD, wy[u]);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (lg + u >= lg1) break;
                const size_t off = (size_t)(lg + u) * kBlockTokens * D + row;
                float x[PPT], y[PPT], ox[PPT], oy[PPT];
                VecTraits<T>::unpack(vx[u], x);
                VecTraits<T>::unpack(vy[u], y);
#pragma unroll
                for (int i = 0; i < PPT; ++i) {
                    // R_p: (x cos - y sin, x sin + y cos), each product rounded
                    ox[i] = __fsub_rn(__fmul_rn(x[i], cs[i]), __fmul_rn(y[i], sn[i]));
                    oy[i] = __fadd_rn(__fmul_rn(x[i], sn[i]), __fmul_rn(y[i], cs[i]));
                }
                st_stream_v(dst_k + off, VecTraits<T>::pack(ox));
                st_stream_v(dst_k + off + HD, VecTraits<T>::pack(oy));
                if (dst_raw != nullptr) {
                    st_stream_v(dst_raw + off, vx[u]);
                    st_stream_v(dst_raw + off + HD, vy[u]);
                }
                if (do_v) {
                    st_stream_v(dst_v + off, wx[u]);
                    st_stream_v(dst_v + off + HD, wy[u]);
                }
            }
        }
    }
};

template <typename T, int D>
__global__ void __launch_bounds__(SlotWork<T, D>::NT)
assemble_ids_kernel(const int32_t *__restrict__ sel_ids, const int32_t *__restrict__ page_ids,
                    int64_t max_blocks, const T *raw_k_repo, const T *v_repo, T *k_pages,
                    T *v_pages, int LG, int lg_per_cta, const float2 *__restrict__ table,
                    int *err) {
    __shared__ float2 tab[kBlockTokens * (D / 2)];
    const int j = blockIdx.x;
    const int64_t b = sel_ids[j];
    const int64_t p = page_ids ? (int64_t)page_ids[j] : (int64_t)j;
    if (b < 0 || b >= max_blocks || p < 0) {
        if (threadIdx.x == 0) atomicOr(err, 1);
        return;
    }
    const size_t blk = (size_t)LG * kBlockTokens * D;
    const int lg0 = blockIdx.y * lg_per_cta, lg1 = min(LG, lg0 + lg_per_cta);
    // 128 bytes of loads in flight per thread whatever the element size
    constexpr int U = 128 / (4 * (int)sizeof(typename VecTraits<T>::V));
    SlotWork<T, D>::template run<U>(raw_k_repo + b * blk, v_repo ? v_repo + b * blk : nullptr,
                        k_pages + p * blk, v_pages ? v_pages + p * blk : nullptr,
                        (int64_t)j * kBlockTokens, lg0, lg1, table, tab);
}

template <typename T, int D>
__global__ void __launch_bounds__(SlotWork<T, D>::NT)
assemble_desc_kernel(const SlotDesc *__restrict__ desc, int LG, int lg_per_cta,
                     const float2 *__restrict__ table, int64_t max_pos, int *err,
                     const int32_t *__restrict__ n_dev) {
    __shared__ float2 tab[kBlockTokens * (D / 2)];
    if (n_dev && (int)blockIdx.x >= *n_dev) return;   // count known on the device only
    const SlotDesc sd = desc[blockIdx.x];
    const bool delta = (sd.flags & kSlotDelta) != 0;
    const bool pos_ok = delta ? (sd.pos0 > -max_pos && sd.pos0 < max_pos)
                              : (sd.pos0 >= 0 && sd.pos0 + kBlockTokens <= max_pos);
    if (!pos_ok || sd.src_k == nullptr || sd.dst_k == nullptr) {
        if (threadIdx.x == 0) atomicOr(err, 2);
        return;
    }
    // a delta rotation runs in place (src_k == dst_k): every thread reads its
    // 16-byte pieces before it writes the same addresses
    const int lg0 = blockIdx.y * lg_per_cta, lg1 = min(LG, lg0 + lg_per_cta);
    SlotWork<T, D>::template run<1>(static_cast<const T *>(sd.src_k),
                                    static_cast<const T *>(sd.src_v),
                        static_cast<T *>(sd.dst_k), static_cast<T *>(sd.dst_v), sd.pos0, lg0,
                        lg1, table, tab, static_cast<T *>(sd.dst_raw), delta);
}

static int lg_split(int n_slots, int LG) {
    int lpc = LG;
    const int64_t want_ctas = (int64_t)sm_count() * 16;
    while (lpc > 8 && (int64_t)n_slots * ((LG + lpc - 1) / lpc) < want_ctas) lpc = (lpc + 1) / 2;
    return lpc > 64 ? 64 : lpc;
}

template <typename T, int D>
static cudaError_t ids_t(const int32_t *sel_ids, const int32_t *page_ids, int n_sel,
                         int64_t max_blocks, const void *rk, const void *v, void *kp, void *vp,
                         int LG, const float2 *table, int *err, cudaStream_t s) {
    const int lpc = lg_split(n_sel, LG);
    dim3 grid((unsigned)n_sel, (unsigned)((LG + lpc - 1) / lpc));
    assemble_ids_kernel<T, D><<<grid, SlotWork<T, D>::NT, 0, s>>>(
        sel_ids, page_ids, max_blocks, static_cast<const T *>(rk), static_cast<const T *>(v),
        static_cast<T *>(kp), static_cast<T *>(vp), LG, lpc, table, err);
    note_launch();
    return cudaGetLastError();
}

template <typename T, int D>
static cudaError_t desc_t(const SlotDesc *desc, int n_desc, const int32_t *n_dev, int LG,
                          const float2 *table, int64_t max_pos, int *err, cudaStream_t s) {
    const int lpc = lg_split(n_desc, LG);
    dim3 grid((unsigned)n_desc, (unsigned)((LG + lpc - 1) / lpc));
    assemble_desc_kernel<T, D><<<grid, SlotWork<T, D>::NT, 0, s>>>(desc, LG, lpc, table,
                                                                     max_pos, err, n_dev);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_assemble_ids(int kv_dtype, int d, const int32_t *sel_ids,
                                const int32_t *page_ids, int n_sel, int64_t max_blocks,
                                const void *raw_k_repo, const void *v_repo, void *k_pages,
                                void *v_pages, int LG, const float2 *table, int64_t max_pos,
                                int *err, cudaStream_t s) {
    (void)max_pos;  // n_sel * 32 <= max_pos is checked on the host
    if (n_sel <= 0) return cudaSuccess;
    if (kv_dtype == BF16 && d == 128)
        return ids_t<__nv_bfloat16, 128>(sel_ids, page_ids, n_sel, max_blocks, raw_k_repo,
                                         v_repo, k_pages, v_pages, LG, table, err, s);
    if (kv_dtype == BF16 && d == 64)
        return ids_t<__nv_bfloat16, 64>(sel_ids, page_ids, n_sel, max_blocks, raw_k_repo,
                                        v_repo, k_pages, v_pages, LG, table, err, s);
    if (kv_dtype == F32 && d == 128)
        return ids_t<float, 128>(sel_ids, page_ids, n_sel, max_blocks, raw_k_repo, v_repo,
                                 k_pages, v_pages, LG, table, err, s);
    if (kv_dtype == F32 && d == 64)
        return ids_t<float, 64>(sel_ids, page_ids, n_sel, max_blocks, raw_k_repo, v_repo,
                                k_pages, v_pages, LG, table, err, s);
    if (kv_dtype == E4M3 && d == 128)
        return ids_t<e4m3, 128>(sel_ids, page_ids, n_sel, max_blocks, raw_k_repo, v_repo,
                                k_pages, v_pages, LG, table, err, s);
    if (kv_dtype == E4M3 && d == 64)
        return ids_t<e4m3, 64>(sel_ids, page_ids, n_sel, max_blocks, raw_k_repo, v_repo,
                               k_pages, v_pages, LG, table, err, s);
    return cudaErrorInvalidValue;
}

static cudaError_t desc_dispatch(int kv_dtype, int d, const SlotDesc *desc, int n_desc,
                                 const int32_t *n_dev, int LG, const float2 *table,
                                 int64_t max_pos, int *err, cudaStream_t s) {
    if (n_desc <= 0) return cudaSuccess;
    if (kv_dtype == BF16 && d == 128)
        return desc_t<__nv_bfloat16, 128>(desc, n_desc, n_dev, LG, table, max_pos, err, s);
    if (kv_dtype == BF16 && d == 64)
        return desc_t<__nv_bfloat16, 64>(desc, n_desc, n_dev, LG, table, max_pos, err, s);
    if (kv_dtype == F32 && d == 128)
        return desc_t<float, 128>(desc, n_desc, n_dev, LG, table, max_pos, err, s);
    if (kv_dtype == F32 && d == 64)
        return desc_t<float, 64>(desc, n_desc, n_dev, LG, table, max_pos, err, s);
    if (kv_dtype == E4M3 && d == 128)
        return desc_t<e4m3, 128>(desc, n_desc, n_dev, LG, table, max_pos, err, s);
    if (kv_dtype == E4M3 && d == 64)
        return desc_t<e4m3, 64>(desc, n_desc, n_dev, LG, table, max_pos, err, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_assemble_desc(int kv_dtype, int d, const SlotDesc *desc, int n_desc, int LG,
                                 const float2 *table, int64_t max_pos, int *err,
                                 cudaStream_t s) {
    return desc_dispatch(kv_dtype, d, desc, n_desc, nullptr, LG, table, max_pos, err, s);
}

cudaError_t launch_assemble_desc_dev(int kv_dtype, int d, const SlotDesc *desc, int n_max,
                                     const int32_t *n_dev, int LG, const float2 *table,
                                     int64_t max_pos, int *err, cudaStream_t s) {
    return desc_dispatch(kv_dtype, d, desc, n_max, n_dev, LG, table, max_pos, err, s);
}

}  // namespace kvm
