// Tensor-core (tcgen05) pass 1 of Eq. (10), KVMem (Virtualizing Million-Token
// Agent Workspaces on a Consumer GPU) §4.3: for every query row of one (layer
// l, kv head g) the maximum and the partition sum of its scaled scores over a
// chunk of Mean-K blocks, for bf16 queries and a bf16 index.
//
// The contraction is D[query row][block] = Q_g . Kbar^T, M = 128 query rows
// per row tile and N = 256 blocks per index tile, both operands in
// 128-byte-swizzled shared memory.  The tensor pipe runs N = 256 instructions
// near its peak rate where N = 128 ran at about 72% of it.  Work is a sequence
// of slots, one per (index tile, row tile); slot j accumulates into TMEM
// buffer j mod 2 (256 columns each), so the epilogue of one slot overlaps the
// MMAs of the next.  (Keeping Q in TMEM as the A operand was measured slower:
// it needs tiles of at most 96 blocks to fit.)
//
// CTA = 18 warps, one SM:
//   warp 0       TMA producer: each tile's 128-byte K atoms (256 rows, 32 KB
//                each) into a 4-entry ring
//   warp 1       MMA issuer: one thread, per slot 4 * (d / 64) MMAs into one of
//                two TMEM accumulators
//   warps 2..17  epilogue, four warps per TMEM lane quadrant; each thread owns
//                a query row (and, in the second row tile, half of one) and
//                keeps a reference m and the partition sum z relative to it
// For 128 < rows <= 192 the second row tile holds rows 128..191 twice (lanes
// 0-63 and 64-127): quadrants 0-1 take its block columns 0-127, quadrants 2-3
// columns 128-255, and the two halves of a row are merged at the end.  Every
// mbarrier wait is bounded (one second of global time); on timeout the kernel
// raises the device error flag (bit 4) and winds down: the producer waits for
// the copies it issued, the MMA warp for its last commit, and then the TMEM is
// freed.
#include <cuda.h>
#include <math.h>

#include "kvm_internal.cuh"
#include "score_common.cuh"
#include "tc_ptx.cuh"

namespace kvm {

namespace {

constexpr int TB = 256;             // index blocks per tile
constexpr int kEpiWarps = 16;
constexpr int kThreads = 64 + kEpiWarps * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = TB;   // one accumulator: one row tile x one index tile
constexpr uint32_t kWaitNs = 1000000000u;   // 1 s
constexpr int kQRows = 256;         // query rows padded to two row tiles

template <int D>
struct Lay1 {
    static constexpr int KA = D / 64;              // 128-byte K atoms per row
    static constexpr int ATOM_TILE = TB * 128;     // one ring entry: one atom of a tile
    static constexpr int STAGES = 4;
    static constexpr int Q_ATOM = kQRows * 128;
    static constexpr int OFF_Q = STAGES * ATOM_TILE;
    static constexpr int OFF_X = OFF_Q + KA * Q_ATOM;      // 1536 floats
    static constexpr int OFF_D = OFF_X + 1536 * 4;         // 2 x 32 x 2 floats
    static constexpr int OFF_BAR = OFF_D + 2 * 32 * 2 * 4;
    static constexpr int SMEM = 1024 + OFF_BAR + 512;
};

}  // namespace

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
score_tc_pass1_kernel(const __grid_constant__ CUtensorMap tmap,
                      const __nv_bfloat16 *__restrict__ q, ScoreShape sh, int64_t b_index0,
                      int64_t b_begin, int64_t b_end, int chunk0, int64_t chunk_blocks,
                      ScoreScratch scr, float scale_log2, int *err) {
    using LY = Lay1<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *tiles = smem;
    uint8_t *qs = smem + LY::OFF_Q;
    float *xch = reinterpret_cast<float *>(smem + LY::OFF_X);
    float *xdup = reinterpret_cast<float *>(smem + LY::OFF_D);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + LY::OFF_BAR);
    uint64_t *empty = full + LY::STAGES;
    uint64_t *tfull = empty + LY::STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *xfin = tempty + 2;         // [4]: warps 1..3 of a quadrant wrote their (m, z)
    uint64_t *xdbar = xfin + 4;          // [2]: quadrant 2+q handed its half-row stats to q
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(xdbar + 2);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int lg = blockIdx.y;
    const int l = lg / sh.G, g = lg - l * sh.G;
    const int rows = sh.rows;
    const int chunk = blockIdx.x;
    const int64_t cb0 = b_begin + (int64_t)chunk * chunk_blocks;
    const int64_t cb1 = min(b_end, cb0 + chunk_blocks);
    const int n_tiles = cb1 > cb0 ? (int)((cb1 - cb0 + TB - 1) / TB) : 0;
    const int qtiles = rows > 128 ? 2 : 1;
    const bool dup = rows > 128 && rows <= 192;

    if (tid == 0) {
        for (int s = 0; s < LY::STAGES; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&tfull[b], 1);
            tc::mbar_init(&tempty[b], kEpiWarps * 32);
        }
        for (int k = 0; k < 4; ++k) tc::mbar_init(&xfin[k], 96);
        for (int k = 0; k < 2; ++k) tc::mbar_init(&xdbar[k], 32);
        tc::fence_mbar_init();
    }
    // ring entry e = (tile, K atom) = (e / KA, e % KA); the producer's first
    // entries go out now, so that their HBM latency overlaps the staging of the
    // query rows below (the stages are free)
    const int n_entries = (sh.idle_producer ? 0 : n_tiles) * LY::KA;   // an idle producer issues nothing
    const int n_pre = min(n_entries, LY::STAGES);
    auto issue = [&](int e) {
        const int i = e / LY::KA, a = e - i * LY::KA;
        const int s = e % LY::STAGES;
        const int32_t y =
            (int32_t)((int64_t)lg * sh.index_cap + (cb0 + (int64_t)i * TB - b_index0));
        tc::mbar_expect_tx(&full[s], LY::ATOM_TILE);
        tc::tma_load_2d(tiles + s * LY::ATOM_TILE, &tmap, &full[s], a * 64, y);
    };
    if (tid == 0)
        for (int e = 0; e < n_pre; ++e) issue(e);
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, kTmemCols);
        tc::tmem_relinquish();
    }
    // Query rows of (l, g) into the swizzled K-major layout; padding rows are 0
    // and rows 192..255 repeat 128..191 when the second row tile is duplicated.
    // Each thread issues all of its loads before the first store.
    {
        constexpr int kQItems = kQRows * (D / 8);
        constexpr int kPer = (kQItems + kThreads - 1) / kThreads;
        uint4 v[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int i = tid + k * kThreads;
            v[k] = make_uint4(0, 0, 0, 0);
            const int r = i / (D / 8), c16 = i - r * (D / 8);
            const int src_r = (dup && r >= 192) ? r - 64 : r;
            if (i < kQItems && src_r < rows) {
                const int m = src_r / sh.gqa, hl = src_r - m * sh.gqa;
                const __nv_bfloat16 *src = q + (((size_t)l * sh.n_queries + m) * sh.H +
                                                (size_t)g * sh.gqa + hl) * D + c16 * 8;
                v[k] = __ldg(reinterpret_cast<const uint4 *>(src));
            }
        }
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int i = tid + k * kThreads;
            if (i < kQItems) {
                const int r = i / (D / 8), c16 = i - r * (D / 8);
                const int a = c16 >> 3, cc = c16 & 7;
                *reinterpret_cast<uint4 *>(qs + a * LY::Q_ATOM + r * 128 + ((cc ^ (r & 7)) << 4)) =
                    v[k];
            }
        }
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // ring entry of atom a of tile i: (stage, phase parity)
    auto ring = [](int i, int a) {
        const int e = i * LY::KA + a;
        return make_int2(e % LY::STAGES, (e / LY::STAGES) & 1);
    };
    const int n_slots = n_tiles * qtiles;

    if (warp == 0) {
        if (lane == 0) {
            int issued = n_pre;                     // ring entries
            for (int e = n_pre; e < n_entries; ++e) {
                const int2 r = ring(e / LY::KA, e % LY::KA);
                if (!tc::mbar_wait(&empty[r.x], r.y ^ 1, kWaitNs)) {
                    atomicOr(err, 4);
                    break;
                }
                issue(e);
                ++issued;
            }
            // every issued copy lands before the CTA ends: wait for the last
            // use of each ring stage (at once in a run without errors)
            for (int e = max(0, issued - LY::STAGES); e < issued; ++e)
                if (!tc::mbar_wait(&full[e % LY::STAGES], (e / LY::STAGES) & 1, kWaitNs)) {
                    atomicOr(err, 4);
                    break;
                }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t qbase = tc::smem_u32(qs);
            const uint32_t tbase = tc::smem_u32(tiles);
            constexpr uint32_t idesc = tc::idesc_bf16_f32(128, TB);
            bool ok = true;
            int last = -1;
            for (int j = 0; j < n_slots && ok; ++j) {
                const int i = j / qtiles, t = j - i * qtiles;
                const int buf = j & 1;
                const uint32_t bph = (j >> 1) & 1;
                if (t == 0)
                    for (int a = 0; a < LY::KA && ok; ++a) {
                        const int2 e = ring(i, a);
                        ok = tc::mbar_wait(&full[e.x], e.y, kWaitNs);
                    }
                if (!ok || !tc::mbar_wait(&tempty[buf], bph ^ 1, kWaitNs)) { ok = false; break; }
                tc::tc_fence_after();
                const uint32_t d = tmem + buf * kAccCols;
#pragma unroll
                for (int a = 0; a < LY::KA; ++a) {
                    const uint32_t atom = tbase + ring(i, a).x * LY::ATOM_TILE;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad =
                            tc::sdesc_sw128(qbase + a * LY::Q_ATOM + t * 128 * 128 + kk * 32);
                        const uint64_t bd = tc::sdesc_sw128(atom + kk * 32);
                        tc::mma_bf16(d, ad, bd, idesc, (a | kk) != 0);
                    }
                }
                tc::mma_commit(&tfull[buf]);
                if (t == qtiles - 1)
                    for (int a = 0; a < LY::KA; ++a) tc::mma_commit(&empty[ring(i, a).x]);
                last = j;
            }
            // the last commit covers every MMA issued: they are done before
            // the TMEM is freed
            if (last >= 0 && !tc::mbar_wait(&tfull[last & 1], (last >> 1) & 1, kWaitNs))
                ok = false;
            if (!ok) atomicOr(err, 4);
        }
    } else {
        const int ew = warp - 2;                    // 0..15
        const int quad = warp & 3;                  // TMEM lanes 32*quad .. 32*quad+31
        const int sub = ew >> 2;                    // which quarter of the columns
        const int lrow = quad * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        const int my_c0 = sub * 64;                 // a full row tile: 64 block columns
        // second row tile, duplicated: quadrants 0-1 take columns 0-127, 2-3
        // columns 128-255, thirty-two per warp
        const int c1 = (quad >= 2 ? 128 : 0) + sub * 32;
        float m_run[2] = {-INFINITY, -INFINITY}, z_run[2] = {0.f, 0.f};
        for (int j = 0; j < n_slots; ++j) {
            const int i = j / qtiles, t = j - i * qtiles;
            const int buf = j & 1;
            const uint32_t bph = (j >> 1) & 1;
            if (!tc::mbar_wait(&tfull[buf], bph, kWaitNs)) { atomicOr(err, 4); break; }
            tc::tc_fence_after();
            const int64_t gb0 = cb0 + (int64_t)i * TB;
            const int nvalid = (int)min((int64_t)TB, cb1 - gb0);
            const uint32_t taddr = tmem + lane_base + buf * kAccCols;
            const bool half = t == 1 && dup;
            const int c0 = half ? c1 : my_c0;
            uint32_t r[64];
            tc::tmem_ld32_async(taddr + c0, r);
            if (!half) tc::tmem_ld32_async(taddr + c0 + 32, r + 32);
            tc::tmem_wait_ld(r);
            tc::tmem_wait_ld(r + 16);
            if (!half) {
                tc::tmem_wait_ld(r + 32);
                tc::tmem_wait_ld(r + 48);
            }
            // the accumulator is in registers: hand the buffer back to the MMA warp
            tc::tc_fence_before();
            tc::mbar_arrive(&tempty[buf]);
            // explicit branches keep both rows' statistics in registers
            if (half)
                row_update<32>(r, min(32, max(0, nvalid - c0)), scale_log2, m_run[1], z_run[1]);
            else if (t == 0)
                row_update<64>(r, min(64, max(0, nvalid - c0)), scale_log2, m_run[0], z_run[0]);
            else
                row_update<64>(r, min(64, max(0, nvalid - c0)), scale_log2, m_run[1], z_run[1]);
        }
        // the quadrant's four warps merge their (m, z) in a fixed order:
        // [t][quad][sub-1][lane] pairs
        float *slot = xch + ((quad * 3) * 32 + lane) * 2;
        if (sub) {
            for (int t = 0; t < qtiles; ++t) {
                slot[(t * 12 + sub - 1) * 64] = m_run[t];
                slot[(t * 12 + sub - 1) * 64 + 1] = z_run[t];
            }
            tc::mbar_arrive(&xfin[quad]);
        } else if (!tc::mbar_wait(&xfin[quad], 0, kWaitNs)) {
            atomicOr(err, 4);
        } else {
            float M[2], Z[2];
            for (int t = 0; t < qtiles; ++t) {
                M[t] = m_run[t];
                for (int k = 0; k < 3; ++k) M[t] = fmaxf(M[t], slot[(t * 12 + k) * 64]);
                Z[t] = 0.f;
                if (M[t] != -INFINITY) {
                    Z[t] = z_run[t] * fast_exp2(m_run[t] - M[t]);
                    for (int k = 0; k < 3; ++k)
                        Z[t] += slot[(t * 12 + k) * 64 + 1] *
                                fast_exp2(slot[(t * 12 + k) * 64] - M[t]);
                }
            }
            auto emit = [&](int r, float m, float z) {
                if (r < rows) {
                    const size_t o = ((size_t)lg * sh.chunk_cap + chunk0 + chunk) * rows + r;
                    scr.part_m[o] = m;
                    scr.part_z[o] = z;
                }
            };
            emit(lrow, M[0], Z[0]);
            if (qtiles > 1) {
                if (!dup) {
                    emit(128 + lrow, M[1], Z[1]);
                } else if (quad >= 2) {
                    // the other half of row 128 + 32*(quad-2) + lane goes to quadrant quad-2
                    xdup[((quad - 2) * 32 + lane) * 2] = M[1];
                    xdup[((quad - 2) * 32 + lane) * 2 + 1] = Z[1];
                    tc::mbar_arrive(&xdbar[quad - 2]);
                } else if (!tc::mbar_wait(&xdbar[quad], 0, kWaitNs)) {
                    atomicOr(err, 4);
                } else {
                    const float m2 = xdup[(quad * 32 + lane) * 2];
                    const float z2 = xdup[(quad * 32 + lane) * 2 + 1];
                    const float Mx = fmaxf(M[1], m2);
                    float Zx = 0.f;
                    if (Mx != -INFINITY)
                        Zx = Z[1] * fast_exp2(M[1] - Mx) + z2 * fast_exp2(m2 - Mx);
                    emit(128 + lrow, Mx, Zx);
                }
            }
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D>
static cudaError_t pass1_t(const ScoreShape &sh, const void *q, const void *index,
                           int64_t b_index0, int64_t b_begin, int64_t b_end, int chunk0,
                           int n_chunks, const ScoreScratch &scr, int *err, cudaStream_t s) {
    CUtensorMap map;
    if (((uintptr_t)index & 15) != 0) return cudaErrorMisalignedAddress;
    if (!make_index_map(&map, index, D, (int64_t)sh.L * sh.G * sh.index_cap, TB))
        return cudaErrorInvalidValue;
    auto kern = score_tc_pass1_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Lay1<D>::SMEM);
    if (e != cudaSuccess) return e;
    const int64_t n = b_end - b_begin;
    const int64_t chunk_blocks = (n + n_chunks - 1) / n_chunks;
    dim3 grid((unsigned)n_chunks, (unsigned)(sh.L * sh.G));
    const float scale_log2 = (float)(1.4426950408889634 / sqrt((double)D));
    kern<<<grid, kThreads, Lay1<D>::SMEM, s>>>(map, static_cast<const __nv_bfloat16 *>(q), sh,
                                               b_index0, b_begin, b_end, chunk0, chunk_blocks, scr,
                                               scale_log2, err);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_score_pass1_tc(const ScoreShape &sh, const void *q, const void *index,
                                  int64_t b_index0, int64_t b_begin, int64_t b_end, int chunk0,
                                  int n_chunks, const ScoreScratch &scr, int *err,
                                  cudaStream_t s) {
    if (sh.d == 128)
        return pass1_t<128>(sh, q, index, b_index0, b_begin, b_end, chunk0, n_chunks, scr, err, s);
    return pass1_t<64>(sh, q, index, b_index0, b_begin, b_end, chunk0, n_chunks, scr, err, s);
}

}  // namespace kvm
