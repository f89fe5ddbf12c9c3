// Tensor-core (tcgen05) pass 2 of Eq. (10), KVMem (Virtualizing Million-Token
// Agent Workspaces on a Consumer GPU) §4.3, for bf16 queries and a bf16
// Mean-K index: for every block of a chunk, the sum over the query rows of one
// (layer l, kv head g) of its softmax probability 2^(s*c - M - log2 Z), with
// the per-row M and Z of pass 1 (score_tc1.cu).  Also the host helpers both
// tensor-core passes share.
//
// The scaled scores are the dense contraction D[block][query row] = Kbar . Q_g^T
// (M = 128 blocks, N = rows rounded up to 16).  Products of bf16 values are
// exact in fp32 and the tensor cores accumulate in fp32, so only the summation
// order differs from the CUDA-core variant.
//
// CTA = 18 warps, one SM (the shared-memory ring and the 512 TMEM columns):
//   warp 0       TMA producer: 128-block index tiles into a 4-stage ring of
//                128-byte-swizzled shared memory (one copy per 64-element K atom)
//   warp 1       MMA issuer: one thread issues tcgen05.mma into one of two TMEM
//                accumulators and commits to mbarriers
//   warps 2..17  epilogue in two groups of eight that take alternate tiles
//                (group g owns TMEM accumulator g); in a group, two warps per
//                TMEM lane quadrant each take half of the accumulator's
//                columns.  Each thread owns one block and sums its half of the
//                rows in registers, and the two halves combine in a fixed order
//                through shared memory.  An accumulator goes back to the MMA
//                warp once its last columns are in registers.
// Every mbarrier wait is bounded (one second of global time); on timeout the
// kernel raises the device error flag (bit 4) and winds down: the producer
// waits for the copies it issued, the MMA warp for its last commit, and then
// the TMEM is freed.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include "kvm_internal.cuh"
#include "score_common.cuh"
#include "tc_ptx.cuh"

namespace kvm {

namespace {

constexpr int TB = 128;             // index blocks per tile
constexpr int kStages = 4;
constexpr int kEpiWarps = 16;
constexpr int kThreads = 64 + kEpiWarps * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kWaitNs = 1000000000u;   // 1 s
constexpr int kQRows = 256;         // largest N (query rows per kv head)

template <int D>
struct Lay {
    static constexpr int KA = D / 64;              // 128-byte K atoms per row
    static constexpr int ATOM_TILE = TB * 128;     // one K atom of an index tile
    static constexpr int TILE = KA * ATOM_TILE;
    static constexpr int Q_ATOM = kQRows * 128;
    static constexpr int QB = KA * Q_ATOM;
    static constexpr int OFF_Q = kStages * TILE;
    static constexpr int OFF_O = OFF_Q + QB;       // float[kQRows]
    static constexpr int OFF_X = OFF_O + kQRows * 4;   // warp exchange, 1536 floats
    static constexpr int OFF_BAR = OFF_X + 1536 * 4;
    static constexpr int SMEM = 1024 + OFF_BAR + 512;
};

}  // namespace

// NC: columns per epilogue warp when fixed at compile time (96 for 192 query
// rows), 0 for any row count.
template <int D, int NC>
__global__ void __launch_bounds__(kThreads, 1)
score_tc_pass2_kernel(const __grid_constant__ CUtensorMap tmap,
                      const __nv_bfloat16 *__restrict__ q, ScoreShape sh, int64_t b_index0,
                      int64_t b_begin, int64_t b_end, int64_t chunk_blocks, ScoreScratch scr,
                      int64_t partial_stride, float scale_log2, int *err) {
    using LY = Lay<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *tiles = smem;
    uint8_t *qs = smem + LY::OFF_Q;
    float *o_r = reinterpret_cast<float *>(smem + LY::OFF_O);
    float *xch = reinterpret_cast<float *>(smem + LY::OFF_X);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + LY::OFF_BAR);
    uint64_t *empty = full + kStages;
    uint64_t *tfull = empty + kStages;
    uint64_t *tempty = tfull + 2;
    uint64_t *xfull = tempty + 2;        // [2][4][4]: a warp's partner wrote its partial
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(xfull + 32);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int lg = blockIdx.y;
    const int l = lg / sh.G, g = lg - l * sh.G;
    const int rows = sh.rows;
    const int chunk = blockIdx.x;
    const int64_t cb0 = b_begin + (int64_t)chunk * chunk_blocks;
    const int64_t cb1 = min(b_end, cb0 + chunk_blocks);
    const int n_tiles = cb1 > cb0 ? (int)((cb1 - cb0 + TB - 1) / TB) : 0;
    const int n2 = (rows + 15) & ~15;              // MMA N

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&tfull[b], 1);
            tc::mbar_init(&tempty[b], (kEpiWarps / 2) * 32);
        }
        for (int k = 0; k < 32; ++k) tc::mbar_init(&xfull[k], 32);
        tc::fence_mbar_init();
    }
    // the producer's first ring entries go out now, so that their HBM latency
    // overlaps the staging of the query rows below (the stages are free)
    const int n_load = sh.idle_producer ? 0 : n_tiles;   // an idle producer issues nothing
    const int n_pre = min(n_load, kStages);
    auto issue = [&](int i) {
        const int s = i % kStages;
        tc::mbar_expect_tx(&full[s], LY::TILE);
        const int32_t y =
            (int32_t)((int64_t)lg * sh.index_cap + (cb0 + (int64_t)i * TB - b_index0));
#pragma unroll
        for (int a = 0; a < LY::KA; ++a)
            tc::tma_load_2d(tiles + s * LY::TILE + a * LY::ATOM_TILE, &tmap, &full[s], a * 64, y);
    };
    if (tid == 0)
        for (int i = 0; i < n_pre; ++i) issue(i);
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, kTmemCols);
        tc::tmem_relinquish();
    }
    // Query rows of (l, g) into the swizzled K-major layout; padding rows are 0.
    // Each thread issues all of its loads before the first store.
    {
        const int n_items = n2 * (D / 8);
        constexpr int kPer = (kQRows * (D / 8) + kThreads - 1) / kThreads;
        uint4 v[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int i = tid + k * kThreads;
            v[k] = make_uint4(0, 0, 0, 0);
            const int r = i / (D / 8), c16 = i - r * (D / 8);
            if (i < n_items && r < rows) {
                const int m = r / sh.gqa, hl = r - m * sh.gqa;
                const __nv_bfloat16 *src = q + (((size_t)l * sh.n_queries + m) * sh.H +
                                                (size_t)g * sh.gqa + hl) * D + c16 * 8;
                v[k] = __ldg(reinterpret_cast<const uint4 *>(src));
            }
        }
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int i = tid + k * kThreads;
            if (i < n_items) {
                const int r = i / (D / 8), c16 = i - r * (D / 8);
                const int a = c16 >> 3, cc = c16 & 7;
                *reinterpret_cast<uint4 *>(qs + a * LY::Q_ATOM + r * 128 + ((cc ^ (r & 7)) << 4)) =
                    v[k];
            }
        }
    }
    for (int r = tid; r < kQRows; r += kThreads) {
        float o = INFINITY;
        if (r < rows) {
            const size_t k = (size_t)lg * rows + r;
            o = scr.row_m[k] - log2f(scr.row_invz[k]);   // M + log2 Z, log2 units
        }
        o_r[r] = -o;                                     // stored negated
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            int issued = n_pre;
            for (int i = n_pre; i < n_load; ++i) {
                const int s = i % kStages;
                const uint32_t ph = (i / kStages) & 1;
                if (!tc::mbar_wait(&empty[s], ph ^ 1, kWaitNs)) { atomicOr(err, 4); break; }
                issue(i);
                ++issued;
            }
            // every issued copy lands before the CTA ends: wait for the last
            // use of each ring stage (at once in a run without errors)
            for (int i = max(0, issued - kStages); i < issued; ++i)
                if (!tc::mbar_wait(&full[i % kStages], (i / kStages) & 1, kWaitNs)) {
                    atomicOr(err, 4);
                    break;
                }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t qbase = tc::smem_u32(qs);
            const uint32_t tbase = tc::smem_u32(tiles);
            const uint32_t idesc = tc::idesc_bf16_f32(128, n2);
            int last = -1;
            for (int i = 0; i < n_tiles; ++i) {
                const int s = i % kStages;
                const uint32_t ph = (i / kStages) & 1;
                const int buf = i & 1;
                const uint32_t bph = (i >> 1) & 1;
                if (!tc::mbar_wait(&full[s], ph, kWaitNs)) { atomicOr(err, 4); break; }
                if (!tc::mbar_wait(&tempty[buf], bph ^ 1, kWaitNs)) { atomicOr(err, 4); break; }
                tc::tc_fence_after();
                const uint32_t d = tmem + buf * 256;
                const uint32_t tile = tbase + s * LY::TILE;
#pragma unroll
                for (int a = 0; a < LY::KA; ++a) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = tc::sdesc_sw128(tile + a * LY::ATOM_TILE + kk * 32);
                        const uint64_t bd = tc::sdesc_sw128(qbase + a * LY::Q_ATOM + kk * 32);
                        tc::mma_bf16(d, ad, bd, idesc, (a | kk) != 0);
                    }
                }
                tc::mma_commit(&empty[s]);
                tc::mma_commit(&tfull[buf]);
                last = i;
            }
            // the last commit covers every MMA issued: they are done before
            // the TMEM is freed
            if (last >= 0 && !tc::mbar_wait(&tfull[last & 1], (last >> 1) & 1, kWaitNs))
                atomicOr(err, 4);
        }
    } else {
        // Two groups of eight warps take alternate tiles: group gr owns TMEM
        // buffer gr and the tiles i = gr, gr + 2, ..., so that one group's
        // waits and TMEM loads overlap the other group's exponentials.  In a
        // group two warps share a lane quadrant, each taking half of the n2
        // columns in chunks; the buffer goes back to the MMA warp once its
        // last chunk is in registers.
        const int ew = warp - 2;                    // 0..15
        const int quad = warp & 3;                  // TMEM lanes 32*quad .. 32*quad+31
        const int gr = ew >> 3;                     // group
        const int hf = (ew >> 2) & 1;               // which half of the columns
        const int lrow = quad * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        // the n2 columns in 16-column units, split into two near-equal runs
        const int nu = n2 >> 4;
        const int u0 = (hf * nu) >> 1, u1 = ((hf + 1) * nu) >> 1;
        const int my_c0 = u0 * 16;
        const int my_nc = (u1 - u0) * 16;
        // warp hf = 0 of a quadrant adds its partner's partial of the group's
        // tile jj - 1 while on tile jj, when that partial is long written
        float pend = 0.f;
        auto combine = [&](int jj, float own) -> bool {
            const int bar = (gr * 4 + (jj & 3)) * 4 + quad;
            if (!tc::mbar_wait(&xfull[bar], (jj >> 2) & 1, kWaitNs)) return false;
            const float sum = own + xch[bar * 32 + lane];
            const int64_t gb0 = cb0 + (int64_t)(2 * jj + gr) * TB;
            if (lrow < min((int64_t)TB, cb1 - gb0))
                scr.partial[(size_t)lg * partial_stride + gb0 + lrow] = sum;
            return true;
        };
        bool ok = true;
        int jj = 0;
        for (int i = gr; i < n_tiles; i += 2, ++jj) {
            if (!tc::mbar_wait(&tfull[gr], jj & 1, kWaitNs)) {
                ok = false;
                break;
            }
            tc::tc_fence_after();
            const uint32_t taddr = tmem + lane_base + gr * 256;
            uint32_t r[48];
            float sum;
            if (NC == 96) {   // 192 query rows: 96 columns per warp, two chunks of 48
                tc::tmem_ld32_async(taddr + my_c0, r);
                tc::tmem_ld16_async(taddr + my_c0 + 32, r + 32);
                tc::tmem_wait_ld(r);
                tc::tmem_wait_ld(r + 16);
                tc::tmem_wait_ld(r + 32);
                sum = exp_sum_n<48>(r, o_r + my_c0, scale_log2);
                tc::tmem_ld32_async(taddr + my_c0 + 48, r);
                tc::tmem_ld16_async(taddr + my_c0 + 80, r + 32);
                tc::tmem_wait_ld(r);
                tc::tmem_wait_ld(r + 16);
                tc::tmem_wait_ld(r + 32);
                tc::tc_fence_before();
                tc::mbar_arrive(&tempty[gr]);
                sum += exp_sum_n<48>(r, o_r + my_c0 + 48, scale_log2);
            } else {
                sum = 0.f;
                if (my_nc == 0) {
                    tc::tc_fence_before();
                    tc::mbar_arrive(&tempty[gr]);
                }
                for (int c = 0; c < my_nc; c += 32) {
                    const int n = min(32, my_nc - c);    // 16 or 32
                    if (n == 32) {
                        tc::tmem_ld32_async(taddr + my_c0 + c, r);
                        tc::tmem_wait_ld(r);
                        tc::tmem_wait_ld(r + 16);
                    } else {
                        tc::tmem_ld16_async(taddr + my_c0 + c, r);
                        tc::tmem_wait_ld(r);
                    }
                    if (c + 32 >= my_nc) {
                        tc::tc_fence_before();
                        tc::mbar_arrive(&tempty[gr]);
                    }
                    sum += exp_sum(r, o_r + my_c0 + c, n, scale_log2);
                }
            }
            // the partner's partial goes through a four-deep ring of slots per
            // group.  A slot is not rewritten before warp hf = 0 read it: the
            // group's tile jj + 4 needs that warp's arrival on tempty for tile
            // jj + 3, which follows its read of tile jj's slot.
            const int bar = (gr * 4 + (jj & 3)) * 4 + quad;
            if (hf) {
                xch[bar * 32 + lane] = sum;
                tc::mbar_arrive(&xfull[bar]);
            } else {
                if (jj > 0 && !combine(jj - 1, pend)) {
                    ok = false;
                    break;
                }
                pend = sum;
            }
        }
        if (hf == 0 && jj > 0 && ok && !combine(jj - 1, pend)) ok = false;
        if (!ok) atomicOr(err, 4);
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------- host side

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    // looked up once per process (thread-safe initialisation of a local static)
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    }();
    return fn;
}

bool make_index_map(CUtensorMap *m, const void *index, int d, int64_t n_rows, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)n_rows};
    cuuint64_t strides[1] = {(cuuint64_t)d * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(index), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_q_map(CUtensorMap *m, const void *q, int d, int H, int64_t n_lq, int gqa,
                int n_queries) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)n_lq};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)gqa, (cuuint32_t)n_queries};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool score_tc_supported(int q_dtype, int index_dtype, const ScoreShape &sh) {
    // the TMA row coordinate (l * G + g) * index_cap + block is a 32-bit int:
    // larger indexes take the CUDA-core kernels, which index in 64 bits
    const bool rows_fit = (int64_t)sh.L * sh.G * sh.index_cap <= (int64_t)INT32_MAX;
    return q_dtype == BF16 && index_dtype == BF16 && (sh.d == 64 || sh.d == 128) &&
           sh.rows >= 1 && sh.rows <= kQRows && rows_fit && encode_fn() != nullptr;
}

template <int D, int NC>
static cudaError_t pass2_t(const ScoreShape &sh, const void *q, const void *index,
                           int64_t b_index0, int64_t b_begin, int64_t b_end, int n_chunks,
                           const ScoreScratch &scr, int64_t partial_stride, int *err,
                           cudaStream_t s) {
    CUtensorMap map;
    if (((uintptr_t)index & 15) != 0) return cudaErrorMisalignedAddress;
    if (!make_index_map(&map, index, D, (int64_t)sh.L * sh.G * sh.index_cap, TB))
        return cudaErrorInvalidValue;
    auto kern = score_tc_pass2_kernel<D, NC>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Lay<D>::SMEM);
    if (e != cudaSuccess) return e;
    const int64_t n = b_end - b_begin;
    const int64_t chunk_blocks = (n + n_chunks - 1) / n_chunks;
    dim3 grid((unsigned)n_chunks, (unsigned)(sh.L * sh.G));
    const float scale_log2 = (float)(1.4426950408889634 / sqrt((double)D));
    kern<<<grid, kThreads, Lay<D>::SMEM, s>>>(map, static_cast<const __nv_bfloat16 *>(q), sh,
                                              b_index0, b_begin, b_end, chunk_blocks, scr,
                                              partial_stride, scale_log2, err);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_score_pass2_tc(const ScoreShape &sh, const void *q, const void *index,
                                  int64_t b_index0, int64_t b_begin, int64_t b_end, int n_chunks,
                                  const ScoreScratch &scr, int64_t partial_stride, int *err,
                                  cudaStream_t s) {
    const bool n192 = ((sh.rows + 15) & ~15) == 192;
    if (sh.d == 128)
        return n192 ? pass2_t<128, 96>(sh, q, index, b_index0, b_begin, b_end, n_chunks, scr,
                                       partial_stride, err, s)
                    : pass2_t<128, 0>(sh, q, index, b_index0, b_begin, b_end, n_chunks, scr,
                                      partial_stride, err, s);
    return n192 ? pass2_t<64, 96>(sh, q, index, b_index0, b_begin, b_end, n_chunks, scr,
                                  partial_stride, err, s)
                : pass2_t<64, 0>(sh, q, index, b_index0, b_begin, b_end, n_chunks, scr,
                                 partial_stride, err, s);
}

}  // namespace kvm
