// Tensor-core (tcgen05) scoring of Eq. (10), KVMem (Virtualizing Million-Token
// Agent Workspaces on a Consumer GPU) §4.3, in one persistent launch
// (score_variant 2): both passes of the exact softmax over all candidate
// blocks, with the second pass re-reading a (layer, kv head) slice of the
// Mean-K index soon after the first, so that it can come from L2.
//
// Measured on GB300 this variant is slower than the two-pass kernels
// (score_tc1.cu, score_tc.cu), which stay the default: with enough slices in
// flight to fill the GPU the data touched between a tile's two reads exceeds
// what L2 keeps (a 1.07 GB index still drew 2.02 GB from DRAM), a 10M-block
// slice alone is 80 MB, and the per-slice group sync costs several
// microseconds.  Even with every second read from L2, the tensor pipe (both
// passes' MMAs) would bind before HBM does.
//
// The softmax of a query row runs over every block of its (layer l, kv head g)
// slice, so pass 2 of a slice can start only once pass 1 has seen the whole
// slice.  The grid (one CTA per SM, launched cooperatively so that all CTAs
// are resident) is split into groups of P CTAs; a group walks its slices
// g0, g0 + n_groups, ... and each CTA of the group takes the same contiguous
// share of every slice:
//   pass 1   the share's 256-block tiles: per query row, running max m and the
//            partition sum z relative to it (as score_tc1.cu)
//   sync     the CTA's (m, z) per row goes to global memory; the group's CTAs
//            count their arrivals on one counter (a bounded spin), then every
//            CTA folds the group's P shares in CTA order into o = M + log2 Z
//   pass 2   the share's 128-block tiles in reverse order, most recently
//            loaded first: for each block, the sum over the rows of
//            2^(s*c - o) (as score_tc.cu), written per (l, g, block)
// P is chosen so that the slices in flight fit in L2 (all CTAs on one slice
// for the 10M-block index, a few CTAs per slice for short histories).  The
// per-block sums over (l, g) are then added in a fixed order by
// score_reduce_kernel, so every result is deterministic.
//
// CTA = 18 warps:
//   warp 0       TMA producer: per slice the query rows (one 3-D box per K
//                atom, prefetched into L2 one slice ahead) and the share's
//                index tiles into a 4-entry ring of 32 KB (a pass-1 tile: one
//                entry per K atom, 256 rows; a pass-2 tile: one entry, 128 rows
//                of every atom)
//   warp 1       MMA issuer: pass 1 D[query row][block] (M = 128 rows, N = 256),
//                pass 2 D[block][query row] (M = 128 blocks, N = rows); slots
//                alternate between two 256-column TMEM accumulators
//   warps 2..17  epilogue: pass 1 as 4 warps per TMEM lane quadrant splitting
//                the columns; pass 2 as two groups of eight taking the slots of
//                their own accumulator
// Query rows: for 128 < rows <= 192 the second row tile starts at row
// t1base = rows - 128 rounded up to 32 (64 for 192 rows), so that no query row
// is stored twice; a row in both tiles takes its first 128 block columns from
// tile 0 and the rest from tile 1, which keeps the four quadrants' work even.
//
// Every wait is bounded by one second of global time, including the spin on
// the group counter.  On timeout the kernel raises the device error flag (bit
// 4) and the CTA's abort flag: the producer and the MMA warp stop issuing, the
// epilogue runs through its remaining steps without waiting (so that its named
// barriers are always reached), the producer waits for the copies it issued,
// the MMA warp for its last commit, and then the TMEM is freed.
#include <cuda.h>
#include <math.h>

#include <algorithm>
#include <cstdlib>

#include "kvm_internal.cuh"
#include "score_common.cuh"
#include "tc_ptx.cuh"

namespace kvm {

namespace {

constexpr int TB1 = 256;            // pass-1 index blocks per tile
constexpr int TB2 = 128;            // pass-2 index blocks per tile
constexpr int kStages = 3;
constexpr int kStageBytes = 32768;
constexpr int kEpiWarps = 16;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kThreads = 64 + kEpiThreads;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kWaitNs = 1000000000u;   // 1 s
constexpr int kEpiBar = 1;                  // named barrier of the epilogue warps
constexpr int kPrefetch = 3;                // pass-1 tiles loaded into L2 ahead of the ring

template <int D>
struct LayF {
    static constexpr int KA = D / 64;                    // 128-byte K atoms per row
    static constexpr int Q_ATOM = kFusedMaxRows * 128;   // one K atom of the query rows
    static constexpr int OFF_Q = kStages * kStageBytes;  // two slices' query rows
    static constexpr int OFF_ST = OFF_Q + 2 * KA * Q_ATOM;   // float2 [2 tiles][4 subs][128 lanes]
    static constexpr int OFF_O = OFF_ST + 2 * 4 * 128 * 8;   // float [256]: -o per row
    static constexpr int OFF_X = OFF_O + 256 * 4;        // float [32][32]: pass-2 partner sums
    static constexpr int OFF_BAR = OFF_X + 32 * 32 * 4;
    static constexpr int SMEM = 1024 + OFF_BAR + 512;
};

struct FusedArgs {
    ScoreShape sh;
    int64_t c0, c1;         // candidate blocks of every slice
    int P;                  // CTAs per slice group
    int n_groups;
    int t1base;             // first row of the second pass-1 row tile (0: one tile)
    float scale_log2;       // log2(e) / sqrt(d)
    float *partial;         // [LG][partial_stride]
    int64_t partial_stride;
    float2 *part;           // [grid][2][rows]: a CTA's (m, z) per row, by slice parity
    float *fo;              // [n_groups][2][rows]: o = M + log2 Z per row, by slice parity
    int *cnt;               // [2][kFusedMaxCtas]: arrivals per group, zero at launch
    int *err;
    int head;               // pass-1 tiles of the next slice run before pass 2
};

// Bounded wait on an mbarrier phase that also gives up once the CTA's abort
// flag is set; a timeout raises the error flag and the abort flag.
__device__ __forceinline__ bool waitb(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                      int *err) {
    uint32_t t0 = 0;
    for (uint32_t n = 0;; ++n) {
        if (tc::mbar_try_wait(bar, parity)) return true;
        if ((n & 63) == 63) {
            if (*abort_flag) return false;
            const uint32_t t = tc::global_ns_lo();
            if (n == 63) {
                t0 = t;
            } else if (t - t0 > kWaitNs) {
                atomicOr(err, 4);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

__device__ __forceinline__ void epi_sync() {
    __syncwarp();
    tc::named_sync(kEpiBar, kEpiThreads);
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
score_fused_kernel(const __grid_constant__ CUtensorMap tidx, const __grid_constant__ CUtensorMap tq,
                   FusedArgs a) {
    using LY = LayF<D>;
    constexpr int KA = LY::KA;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *ring = smem;
    uint8_t *qs = smem + LY::OFF_Q;                 // [2 slices][KA][kFusedMaxRows rows]
    float2 *stat = reinterpret_cast<float2 *>(smem + LY::OFF_ST);
    float *o_neg = reinterpret_cast<float *>(smem + LY::OFF_O);
    float *xch = reinterpret_cast<float *>(smem + LY::OFF_X);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + LY::OFF_BAR);
    uint64_t *empty = full + kStages;
    uint64_t *tfull = empty + kStages;      // [2]: accumulator written (any pass)
    uint64_t *tempty1 = tfull + 2;          // [2]: pass-1 slot read by all 16 warps
    uint64_t *tempty2 = tempty1 + 2;        // [2]: pass-2 slot read by its group of 8
    uint64_t *qfull = tempty2 + 2;          // [2]: query rows of a slice landed
    uint64_t *qempty = qfull + 2;           // [2]: last MMA of a slice done with them
    uint64_t *xfull = qempty + 2;           // [2][4][4]: a warp's partner wrote its sum
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(xfull + 32);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const ScoreShape &sh = a.sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rows = sh.rows;
    const int LG = sh.L * sh.G;
    const int grp = blockIdx.x / a.P, p = blockIdx.x - grp * a.P;
    const int n_slices = grp < LG ? (LG - grp + a.n_groups - 1) / a.n_groups : 0;
    // this CTA's share of every slice: 128-block units [ub, ue) of the
    // candidates, as pass-1 tiles of two units (the last may be one unit)
    // and pass-2 tiles of one
    const int64_t n = a.c1 - a.c0;
    const int64_t U = (n + TB2 - 1) / TB2;
    const int64_t ub = U * p / a.P, ue = U * (p + 1) / a.P;
    const int64_t pb0 = a.c0 + ub * TB2;
    const int64_t pb1 = min(a.c1, a.c0 + ue * TB2);
    const int n2 = (int)(ue - ub);
    const int n1 = (n2 + 1) / 2;
    const bool half_last = (n2 & 1) != 0;   // the last pass-1 tile has 128 blocks
    const int head = min(a.head, n1);       // pass-1 tiles of slice k+1 run before pass 2 of k
    const int qt = a.t1base > 0 ? 2 : 1;    // pass-1 row tiles
    const int n2c = (rows + 15) & ~15;      // pass-2 MMA N

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&tfull[b], 1);
            tc::mbar_init(&tempty1[b], kEpiThreads);
            tc::mbar_init(&tempty2[b], kEpiThreads / 2);
            tc::mbar_init(&qfull[b], 1);
            tc::mbar_init(&qempty[b], 1);
        }
        for (int k = 0; k < 32; ++k) tc::mbar_init(&xfull[k], 32);
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, kTmemCols);
        tc::tmem_relinquish();
    }
    // query rows beyond `rows` are read by the MMAs as zeros: the TMA box
    // writes rows [0, rows) only
    {
        const int pad16 = (kFusedMaxRows - rows) * 8;          // 16-byte chunks per atom
        for (int i = tid; i < 2 * KA * pad16; i += kThreads) {
            const int qa = i / pad16, rr = i - qa * pad16;     // qa = buffer * KA + atom
            *reinterpret_cast<uint4 *>(qs + qa * LY::Q_ATOM + rows * 128 + rr * 16) =
                make_uint4(0, 0, 0, 0);
        }
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // the program every role walks, per slice k:
    //   T(k)    pass-1 tiles [k ? head : 0, n1) of slice k
    //   H(k+1)  pass-1 tiles [0, head) of slice k+1 (if there is one)
    //   P2(k)   pass-2 tiles of slice k, last to first
    auto t_begin = [&](int k) { return k ? head : 0; };

    if (warp == 0) {
        if (lane == 0) {
            int e = 0;                      // ring entries, issued or (idle) skipped
            uint32_t recent = 0;            // bit i: entry e - 1 - i was issued
            int q_last = -1;                // last slice whose query rows were issued
            bool ok = true;
            // the query rows of slice j into buffer j & 1, once the MMAs of
            // slice j - 2 are done with it
            auto q_load = [&](int j) -> bool {
                const int b = j & 1;
                if (!waitb(&qempty[b], ((j >> 1) & 1) ^ 1, abort_flag, a.err)) return false;
                const int lg = grp + j * a.n_groups, l = lg / sh.G, g = lg - l * sh.G;
                tc::mbar_expect_tx(&qfull[b], (uint32_t)(KA * rows * 128));
                for (int at = 0; at < KA; ++at)
                    tc::tma_load_3d(qs + (b * KA + at) * LY::Q_ATOM, &tq, &qfull[b], at * 64,
                                    g * sh.gqa, l * sh.n_queries);
                q_last = j;
                return true;
            };
            // pass-1 tile j of the run T(k) H(k + 1) into L2 ahead of its ring
            // entries, which hides the HBM latency that three ring entries
            // (1.5 pass-1 tiles) cannot
            auto prefetch = [&](int k, int j) {
                const int nT = n1 - t_begin(k), nH = k + 1 < n_slices ? head : 0;
                if (j >= nT + nH || (sh.idle_producer & 1)) return;
                const int kk = j < nT ? k : k + 1;
                const int t = j < nT ? t_begin(k) + j : j - nT;
                const int32_t y = (int32_t)((int64_t)(grp + kk * a.n_groups) * sh.index_cap + pb0 +
                                            (int64_t)t * TB1);
                const bool half = half_last && t == n1 - 1;
                for (int at = 0; at < KA; ++at) {
                    tc::tma_prefetch_2d(&tidx, at * 64, y);
                    if (!half) tc::tma_prefetch_2d(&tidx, at * 64, y + 128);
                }
            };
            if (n_slices > 0) ok = q_load(0);
            for (int j = 0; j < kPrefetch; ++j) prefetch(0, j);
            for (int k = 0; k < n_slices && ok; ++k) {
                // T(k) then H(k + 1) as one run of pass-1 tiles; Q(k + 1) goes
                // in after the first ring entries of T(k), by which time the
                // MMAs of slice k - 1 are issued
                const bool more = k + 1 < n_slices;
                const int nT = n1 - t_begin(k), nH = more ? head : 0;
                bool q_done = !more;
                for (int j = 0; j < nT + nH && ok; ++j) {
                    if (!q_done && (j * KA >= kStages || j == nT)) {
                        if (!(ok = q_load(k + 1))) break;
                        q_done = true;
                    }
                    prefetch(k, j + kPrefetch);
                    const int kk = j < nT ? k : k + 1;
                    const int t = j < nT ? t_begin(k) + j : j - nT;
                    const int lg = grp + kk * a.n_groups;
                    const int32_t y =
                        (int32_t)((int64_t)lg * sh.index_cap + pb0 + (int64_t)t * TB1);
                    const bool half = half_last && t == n1 - 1;
                    for (int at = 0; at < KA && ok; ++at, ++e) {
                        recent <<= 1;
                        if (sh.idle_producer & 1) continue;
                        const int s = e % kStages;
                        if (!(ok = waitb(&empty[s], ((e / kStages) & 1) ^ 1, abort_flag, a.err)))
                            break;
                        tc::mbar_expect_tx(&full[s], half ? kStageBytes / 2 : kStageBytes);
                        tc::tma_load_2d(ring + s * kStageBytes, &tidx, &full[s], at * 64, y);
                        if (!half)
                            tc::tma_load_2d(ring + s * kStageBytes + 16384, &tidx, &full[s],
                                            at * 64, y + 128);
                        recent |= 1;
                    }
                }
                if (ok && !q_done) ok = q_load(k + 1);
                // the next run's first tiles load into L2 during pass 2
                for (int j = 0; more && j < kPrefetch; ++j) prefetch(k + 1, j);
                const int lg = grp + k * a.n_groups;
                for (int i = n2 - 1; i >= 0 && ok; --i, ++e) {
                    recent <<= 1;
                    if (sh.idle_producer & 2) continue;
                    const int s = e % kStages;
                    if (!(ok = waitb(&empty[s], ((e / kStages) & 1) ^ 1, abort_flag, a.err)))
                        break;
                    tc::mbar_expect_tx(&full[s], KA * 16384);
                    const int32_t y =
                        (int32_t)((int64_t)lg * sh.index_cap + pb0 + (int64_t)i * TB2);
                    for (int at = 0; at < KA; ++at)
                        tc::tma_load_2d(ring + s * kStageBytes + at * 16384, &tidx, &full[s],
                                        at * 64, y);
                    recent |= 1;
                }
            }
            // every issued copy lands before the CTA ends: the last use of each
            // stage is among the last kStages entries (earlier uses were
            // consumed before their stage was refilled)
            for (int i = 0; i < kStages; ++i) {
                const int ei = e - 1 - i;
                if (ei >= 0 && ((recent >> i) & 1) &&
                    !tc::mbar_wait(&full[ei % kStages], (ei / kStages) & 1, kWaitNs))
                    atomicOr(a.err, 4);
            }
            for (int j = max(0, q_last - 1); j <= q_last; ++j)
                if (!tc::mbar_wait(&qfull[j & 1], (j >> 1) & 1, kWaitNs)) atomicOr(a.err, 4);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t qbase = tc::smem_u32(qs);
            const uint32_t rbase = tc::smem_u32(ring);
            constexpr uint32_t idesc1 = tc::idesc_bf16_f32(128, TB1);
            constexpr uint32_t idesc1h = tc::idesc_bf16_f32(128, TB2);   // a one-unit tile
            const uint32_t idesc2 = tc::idesc_bf16_f32(128, n2c);
            int e = 0, slot = 0, last_slot = -1, q_seen = 0;
            // per accumulator (bit buf): its last slot was a pass-1 / pass-2
            // slot, and the parity of the pass-1 / pass-2 slots it has held
            uint32_t was1 = 0, was2 = 0, par1 = 0, par2 = 0;
            // the accumulator `buf` is free once its previous slot was read
            auto released = [&](int buf) -> bool {
                if ((was1 >> buf) & 1)
                    return waitb(&tempty1[buf], ((par1 >> buf) & 1) ^ 1, abort_flag, a.err);
                if ((was2 >> buf) & 1)
                    return waitb(&tempty2[buf], ((par2 >> buf) & 1) ^ 1, abort_flag, a.err);
                return true;
            };
            auto mark = [&](int buf, int pass) {
                const uint32_t bit = 1u << buf;
                was1 = pass == 1 ? was1 | bit : was1 & ~bit;
                was2 = pass == 2 ? was2 | bit : was2 & ~bit;
                if (pass == 1) par1 ^= bit;
                else par2 ^= bit;
            };
            // the query rows of slices up to j have landed
            auto q_ready = [&](int j) -> bool {
                for (; q_seen <= j; ++q_seen)
                    if (!waitb(&qfull[q_seen & 1], (q_seen >> 1) & 1, abort_flag, a.err))
                        return false;
                tc::tc_fence_after();
                return true;
            };
            bool ok = true;
            for (int k = 0; k < n_slices && ok; ++k) {
                const bool more = k + 1 < n_slices;
                const int nT = n1 - t_begin(k), nH = more ? head : 0;
                for (int j = 0; j < nT + nH && ok; ++j) {
                    const int kk = j < nT ? k : k + 1;
                    const int t = j < nT ? t_begin(k) + j : j - nT;
                    if (!(ok = q_ready(kk))) break;
                    for (int at = 0; at < KA && ok; ++at)
                        ok = waitb(&full[(e + at) % kStages], ((e + at) / kStages) & 1,
                                   abort_flag, a.err);
                    if (!ok) break;
                    tc::tc_fence_after();
                    const uint32_t id1 = half_last && t == n1 - 1 ? idesc1h : idesc1;
                    const uint32_t qb = qbase + (kk & 1) * KA * LY::Q_ATOM;
                    for (int rt = 0; rt < qt && ok; ++rt) {
                        const int buf = slot & 1;
                        if (!(ok = released(buf))) break;
                        tc::tc_fence_after();
                        const uint32_t d = tmem + buf * 256;
                        const uint32_t row0 = (uint32_t)(rt ? a.t1base : 0) * 128;
#pragma unroll
                        for (int at = 0; at < KA; ++at) {
                            const uint32_t entry = rbase + ((e + at) % kStages) * kStageBytes;
#pragma unroll
                            for (int kq = 0; kq < 4; ++kq) {
                                const uint64_t ad =
                                    tc::sdesc_sw128(qb + at * LY::Q_ATOM + row0 + kq * 32);
                                const uint64_t bd = tc::sdesc_sw128(entry + kq * 32);
                                tc::mma_bf16(d, ad, bd, id1, (at | kq) != 0);
                            }
                        }
                        tc::mma_commit(&tfull[buf]);
                        mark(buf, 1);
                        last_slot = slot++;
                    }
                    if (!ok) break;
                    for (int at = 0; at < KA; ++at) tc::mma_commit(&empty[(e + at) % kStages]);
                    e += KA;
                }
                if (!ok || !(ok = q_ready(k))) break;
                const uint32_t qb = qbase + (k & 1) * KA * LY::Q_ATOM;
                for (int i = 0; i < n2 && ok; ++i, ++e) {
                    const int s = e % kStages;
                    if (!(ok = waitb(&full[s], (e / kStages) & 1, abort_flag, a.err))) break;
                    const int buf = slot & 1;
                    if (!(ok = released(buf))) break;
                    tc::tc_fence_after();
                    const uint32_t d = tmem + buf * 256;
                    const uint32_t entry = rbase + s * kStageBytes;
#pragma unroll
                    for (int at = 0; at < KA; ++at) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t ad = tc::sdesc_sw128(entry + at * 16384 + kk * 32);
                            const uint64_t bd = tc::sdesc_sw128(qb + at * LY::Q_ATOM + kk * 32);
                            tc::mma_bf16(d, ad, bd, idesc2, (at | kk) != 0);
                        }
                    }
                    tc::mma_commit(&empty[s]);
                    tc::mma_commit(&tfull[buf]);
                    mark(buf, 2);
                    last_slot = slot++;
                }
                if (ok) tc::mma_commit(&qempty[k & 1]);
            }
            // the last commit covers every MMA issued: they are done before
            // the TMEM is freed
            if (last_slot >= 0 &&
                !tc::mbar_wait(&tfull[last_slot & 1], (last_slot >> 1) & 1, kWaitNs))
                atomicOr(a.err, 4);
        }
    } else {
        const int ew = warp - 2;                    // 0..15
        const int et = tid - 64;                    // 0..511
        const int quad = warp & 3;                  // TMEM lanes 32*quad .. 32*quad+31
        const int sub = ew >> 2;                    // pass 1: which quarter of the columns
        const int gr = ew >> 3;                     // pass 2: group (= its accumulator)
        const int hf = (ew >> 2) & 1;               // pass 2: which half of the rows
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        const int lrow = quad * 32 + lane;
        // pass 2: the n2c row columns in 16-column units, two near-equal runs
        const int nu = n2c >> 4;
        const int u0 = (hf * nu) >> 1, u1 = ((hf + 1) * nu) >> 1;
        const int my_c0 = u0 * 16, my_nc = (u1 - u0) * 16;
        // pass 1: the block columns this warp reads in row tile rt (width 64,
        // 32 or 0 from column p1c0(rt))
        auto p1row0 = [&](int rt) { return (rt ? a.t1base : 0) + quad * 32; };
        auto p1full = [&](int rt) {
            return qt == 1 || (rt == 0 ? p1row0(0) < a.t1base : p1row0(1) >= 128);
        };
        auto p1w = [&](int rt) { return rt >= qt || p1row0(rt) >= rows ? 0 : (p1full(rt) ? 64 : 32); };
        auto p1c0 = [&](int rt) { return p1full(rt) ? sub * 64 : (rt ? 128 : 0) + sub * 32; };
        int slot = 0, jj = 0;                       // jj: this group's pass-2 tiles so far
        float m_run[2] = {-INFINITY, -INFINITY}, z_run[2] = {0.f, 0.f};   // slice in pass 1
        // the group counter `which` reaches (k + 1) * P: bounded spin by one
        // thread, then the epilogue's named barrier
        auto group_wait = [&](int which, int k) {
            if (et == 0) {
                const int *c = a.cnt + which * kFusedMaxCtas + grp;
                const int target = (k + 1) * a.P;
                const uint32_t t0 = tc::global_ns_lo();
                while (!*abort_flag && tc::ld_acquire_gpu(c) < target) {
                    if (*reinterpret_cast<volatile int *>(a.err) & 4) {
                        *abort_flag = 1;    // another CTA gave up
                        break;
                    }
                    if (tc::global_ns_lo() - t0 > kWaitNs) {
                        atomicOr(a.err, 4);
                        *abort_flag = 1;
                        break;
                    }
                    __nanosleep(32);
                }
                __threadfence();
            }
            epi_sync();
        };
        for (int k = 0; k < n_slices; ++k) {
            const int lg = grp + k * a.n_groups;
            const bool more = k + 1 < n_slices;
            const int nT = n1 - t_begin(k), nH = more ? head : 0;
            const int jA = nT + (nH + 1) / 2;       // the fold of slice k comes here
            // T(k) then H(k + 1) as one run of pass-1 tiles, with the steps of
            // slice k's group sync in between: after T(k) this CTA's (m, z) per
            // row, halfway through H(k + 1) the fold of its rows, after H(k + 1)
            // every row's offset
            for (int j = 0; j <= nT + nH; ++j) {
                if (j == nT) {
                    // ---------------- this CTA's (m, z) per row of slice k
                    stat[sub * 128 + lrow] = make_float2(m_run[0], z_run[0]);
                    stat[(4 + sub) * 128 + lrow] = make_float2(m_run[1], z_run[1]);
                    m_run[0] = m_run[1] = -INFINITY;
                    z_run[0] = z_run[1] = 0.f;
                    epi_sync();
                    if (et < rows) {
                        // the row's entries in a fixed order: tile 0 at lane et,
                        // then tile 1 at lane et - t1base, each by column quarter
                        const bool in0 = et < 128, in1 = qt == 2 && et >= a.t1base;
                        const float2 *s0 = stat + et, *s1 = stat + 4 * 128 + et - a.t1base;
                        float M = -INFINITY;
#pragma unroll
                        for (int s4 = 0; s4 < 4; ++s4) {
                            if (in0) M = fmaxf(M, s0[s4 * 128].x);
                            if (in1) M = fmaxf(M, s1[s4 * 128].x);
                        }
                        float Z = 0.f;
                        if (M != -INFINITY) {
#pragma unroll
                            for (int s4 = 0; s4 < 4; ++s4)
                                if (in0 && s0[s4 * 128].x != -INFINITY)
                                    Z += s0[s4 * 128].y * fast_exp2(s0[s4 * 128].x - M);
#pragma unroll
                            for (int s4 = 0; s4 < 4; ++s4)
                                if (in1 && s1[s4 * 128].x != -INFINITY)
                                    Z += s1[s4 * 128].y * fast_exp2(s1[s4 * 128].x - M);
                        }
                        a.part[((size_t)blockIdx.x * 2 + (k & 1)) * rows + et] = make_float2(M, Z);
                    }
                    // the writes above, ordered by the barrier, are published by
                    // one fence and release of thread 0
                    epi_sync();
                    if (et == 0) {
                        __threadfence();
                        tc::red_release_gpu_add(a.cnt + grp, 1);
                    }
                }
                if (j == jA) {
                    // ---------------- rows p, p + P, ...: fold the group's P shares
                    group_wait(0, k);
                    const int na = p < rows ? (rows - p + a.P - 1) / a.P : 0;
                    float2 *red = stat;             // free until the next (m, z) step
                    if (et < na * a.P && !*abort_flag) {
                        const int i = et / a.P, q = et - i * a.P;
                        red[et] = __ldcg(&a.part[((size_t)(grp * a.P + q) * 2 + (k & 1)) * rows +
                                                 p + i * a.P]);
                    }
                    epi_sync();
                    for (int i = ew; i < na; i += kEpiWarps) {
                        // lane l takes shares l, l + 32, ...; then a fixed tree
                        float M = -INFINITY;
                        for (int q = lane; q < a.P; q += 32) M = fmaxf(M, red[i * a.P + q].x);
#pragma unroll
                        for (int o = 16; o; o >>= 1)
                            M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
                        float Z = 0.f;
                        if (M != -INFINITY)
                            for (int q = lane; q < a.P; q += 32) {
                                const float2 v = red[i * a.P + q];
                                if (v.x != -INFINITY) Z += v.y * fast_exp2(v.x - M);
                            }
#pragma unroll
                        for (int o = 16; o; o >>= 1) Z += __shfl_xor_sync(0xffffffffu, Z, o);
                        if (lane == 0)
                            a.fo[((size_t)grp * 2 + (k & 1)) * rows + p + i * a.P] =
                                M != -INFINITY && Z > 0.f ? M + log2f(Z) : INFINITY;
                    }
                    epi_sync();
                    if (et == 0) {
                        __threadfence();
                        tc::red_release_gpu_add(a.cnt + kFusedMaxCtas + grp, 1);
                    }
                }
                if (j == nT + nH) break;
                // ---------------- one pass-1 tile (of slice k, or of k + 1 in H)
                const int t = j < nT ? t_begin(k) + j : j - nT;
                const int64_t tb0 = pb0 + (int64_t)t * TB1;
                const int nvalid = (int)min((int64_t)TB1, pb1 - tb0);
#pragma unroll
                for (int rt = 0; rt < 2; ++rt) {
                    if (rt >= qt) break;
                    const int buf = slot & 1;
                    const uint32_t ph = (slot >> 1) & 1;
                    ++slot;
                    if (!waitb(&tfull[buf], ph, abort_flag, a.err)) continue;
                    tc::tc_fence_after();
                    const int c0 = p1c0(rt);
                    const int w = nvalid > c0 ? p1w(rt) : 0;   // no valid column: no load
                    const uint32_t taddr = tmem + lane_base + buf * 256 + c0;
                    // 32 columns at a time (fewer live registers); the
                    // accumulator goes back once its last columns are loaded
                    for (int h = 0; h < 2; ++h) {
                        const bool again = h == 0 && w == 64;
                        uint32_t r[32];
                        if (w) {
                            tc::tmem_ld32_async(taddr + h * 32, r);
                            tc::tmem_wait_ld(r);
                            tc::tmem_wait_ld(r + 16);
                        }
                        if (!again) {
                            tc::tc_fence_before();
                            tc::mbar_arrive(&tempty1[buf]);
                        }
                        if (w)
                            row_update<32>(r, min(32, max(0, nvalid - c0 - h * 32)), a.scale_log2,
                                           m_run[rt], z_run[rt]);
                        if (!again) break;
                    }
                }
            }
            // ---------------- every row's offset, kept negated
            group_wait(1, k);
            if (et < 256) {
                float on = -INFINITY;
                if (et < rows && !*abort_flag)
                    on = -__ldcg(&a.fo[((size_t)grp * 2 + (k & 1)) * rows + et]);
                o_neg[et] = on;
            }
            epi_sync();
            // ---------------- P2(k), tiles in reverse order
            // the next slice's row statistics wait in shared memory (fewer live
            // registers in the pass-2 loop); the stat area is free until the
            // next (m, z) step
            stat[et] = make_float2(m_run[0], z_run[0]);
            stat[kEpiThreads + et] = make_float2(m_run[1], z_run[1]);
            bool pend = false;
            float pend_sum = 0.f;
            int64_t pend_b0 = 0;
            int pend_nv = 0, pend_jj = 0;
            auto combine = [&]() {
                const int bar = (gr * 4 + (pend_jj & 3)) * 4 + quad;
                if (!waitb(&xfull[bar], (pend_jj >> 2) & 1, abort_flag, a.err)) return;
                if (lrow < pend_nv)
                    a.partial[(size_t)lg * a.partial_stride + pend_b0 + lrow] =
                        pend_sum + xch[bar * 32 + lane];
            };
            for (int i = 0; i < n2; ++i) {
                const int buf = slot & 1;
                const uint32_t ph = (slot >> 1) & 1;
                ++slot;
                if (buf != gr) continue;            // the other group's tile
                const int ti = n2 - 1 - i;
                const int64_t gb0 = pb0 + (int64_t)ti * TB2;
                const int nvalid = (int)min((int64_t)TB2, pb1 - gb0);
                const int my_jj = jj++;
                if (!waitb(&tfull[buf], ph, abort_flag, a.err)) continue;
                tc::tc_fence_after();
                const uint32_t taddr = tmem + lane_base + buf * 256;
                uint32_t r[32];
                // the row columns in 32-column runs; the accumulator goes back
                // once the last run is loaded
                float sum = 0.f;
                if (my_nc == 0) {
                    tc::tc_fence_before();
                    tc::mbar_arrive(&tempty2[buf]);
                }
                for (int c = 0; c < my_nc; c += 32) {
                    const int nc = min(32, my_nc - c);    // 16 or 32
                    if (nc == 32) {
                        tc::tmem_ld32_async(taddr + my_c0 + c, r);
                        tc::tmem_wait_ld(r);
                        tc::tmem_wait_ld(r + 16);
                    } else {
                        tc::tmem_ld16_async(taddr + my_c0 + c, r);
                        tc::tmem_wait_ld(r);
                    }
                    if (c + 32 >= my_nc) {
                        tc::tc_fence_before();
                        tc::mbar_arrive(&tempty2[buf]);
                    }
                    sum += nc == 32 ? exp_sum_n<32>(r, o_neg + my_c0 + c, a.scale_log2)
                                    : exp_sum(r, o_neg + my_c0 + c, nc, a.scale_log2);
                }
                // the partner's sum goes through a four-deep ring of slots per
                // group (see score_tc.cu for why a slot is read before reuse)
                const int bar = (gr * 4 + (my_jj & 3)) * 4 + quad;
                if (hf) {
                    xch[bar * 32 + lane] = sum;
                    tc::mbar_arrive(&xfull[bar]);
                } else {
                    if (pend) combine();
                    pend = true;
                    pend_sum = sum;
                    pend_b0 = gb0;
                    pend_nv = nvalid;
                    pend_jj = my_jj;
                }
            }
            if (hf == 0 && pend) combine();
            {
                const float2 v0 = stat[et], v1 = stat[kEpiThreads + et];
                m_run[0] = v0.x;
                z_run[0] = v0.y;
                m_run[1] = v1.x;
                z_run[1] = v1.y;
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

// ---------------------------------------------------------------- host side

namespace {

// Tuning overrides, read once from the environment: KVM_SCORE_HEAD (pass-1
// tiles of the next slice that run before pass 2 of the current one; default
// 4) and KVM_SCORE_GROUP (CTAs per slice group; default: plan_groups).
struct Tuning {
    int head, group;
};
const Tuning &tuning() {
    static const Tuning t = [] {
        Tuning v{4, 0};
        if (const char *h = getenv("KVM_SCORE_HEAD")) v.head = std::max(0, atoi(h));
        if (const char *g = getenv("KVM_SCORE_GROUP")) v.group = std::max(0, atoi(g));
        return v;
    }();
    return t;
}

int coop_supported() {
    static const int v = [] {
        int dev = 0, c = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&c, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess)
            return 0;
        return c;
    }();
    return v;
}

// CTAs per slice group.  One CTA per SM; a group of P CTAs takes a slice at a
// time, so about (SMs / P) slices are in flight and pass 2 finds its slice in
// L2 while (SMs / P) * slice bytes stays well inside L2.  Among the P that
// keep the footprint within the budget (or the whole grid on one slice, the
// smallest footprint there is), take the fewest tile-times: rounds of slices
// per group x (pass-1 tiles per CTA + a sync charged as two tiles).
struct Plan {
    int P, n_groups;
};

Plan plan_groups(int64_t n, int LG, int d, int sms) {
    const int64_t U = (n + TB2 - 1) / TB2;         // 128-block units per slice
    const double slice_mb = (double)n * d * 2 / 1048576.0;
    constexpr double kBudgetMB = 64.0;
    Plan best{sms, 1};
    double best_cost = -1;
    for (int P = 1; P <= sms; ++P) {
        if (P > 1 && P > U) break;
        int G = sms / P;
        if (G > LG) G = LG;
        const double foot = G * slice_mb;
        if (foot > kBudgetMB && G > 1) continue;
        const int64_t rounds = (LG + G - 1) / G;
        const int64_t per_cta = (U + P - 1) / P;
        // a unit is about 0.75 us of both passes; the group sync about 3 us
        const double cost = (double)rounds * ((double)per_cta + (P > 1 ? 4.0 : 1.0));
        if (best_cost < 0 || cost < best_cost || (cost == best_cost && P * G > best.P * best.n_groups)) {
            best_cost = cost;
            best = Plan{P, G};
        }
    }
    return best;
}

template <int D>
cudaError_t fused_t(const ScoreShape &sh, const void *q, const void *index, int64_t c0,
                    int64_t c1, const ScoreScratch &scr, int64_t partial_stride,
                    cudaStream_t s) {
    CUtensorMap mi, mq;
    if (!make_index_map(&mi, index, D, (int64_t)sh.L * sh.G * sh.index_cap, TB2))
        return cudaErrorInvalidValue;
    if (!make_q_map(&mq, q, D, sh.H, (int64_t)sh.L * sh.n_queries, sh.gqa, sh.n_queries))
        return cudaErrorInvalidValue;
    auto kern = score_fused_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         LayF<D>::SMEM);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads,
                                                           LayF<D>::SMEM)) != cudaSuccess)
        return e;
    if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
    const int sms = std::min(sm_count(), kFusedMaxCtas);
    const int LG = sh.L * sh.G;
    Plan pl = plan_groups(c1 - c0, LG, D, sms);
    if (tuning().group > 0) {   // a forced group size (tuning override)
        pl.P = std::min(tuning().group, sms);
        pl.n_groups = std::max(1, std::min(sms / pl.P, LG));
    }
    FusedArgs a{};
    a.sh = sh;
    a.c0 = c0;
    a.c1 = c1;
    a.P = pl.P;
    a.n_groups = pl.n_groups;
    a.t1base = sh.rows > 128 ? ((sh.rows - 128 + 31) / 32) * 32 : 0;
    a.scale_log2 = (float)(1.4426950408889634 / sqrt((double)D));
    a.partial = scr.partial;
    a.partial_stride = partial_stride;
    a.part = scr.fpart;
    a.fo = scr.fo;
    a.cnt = scr.fcnt;
    a.err = scr.err;
    a.head = tuning().head;
    if ((e = cudaMemsetAsync(scr.fcnt, 0, sizeof(int) * 2 * kFusedMaxCtas, s)) != cudaSuccess)
        return e;
    void *args[] = {(void *)&mi, (void *)&mq, (void *)&a};
    e = cudaLaunchCooperativeKernel((const void *)kern, dim3((unsigned)(pl.P * pl.n_groups)),
                                    dim3(kThreads), args, LayF<D>::SMEM, s);
    note_launch();
    return e;
}

}  // namespace

bool score_fused_supported(int q_dtype, int index_dtype, const ScoreShape &sh) {
    if (sh.variant != 2 || !score_uses_tc(q_dtype, index_dtype, sh) ||
        sh.rows > kFusedMaxRows || !coop_supported())
        return false;
    // a pass-1 tile reads 256 rows from its first: the TMA row coordinate
    // stays a 32-bit int
    return (int64_t)sh.L * sh.G * sh.index_cap + TB1 <= (int64_t)INT32_MAX;
}

bool fused_q_ok(const void *q) {
    // the queries are read by TMA: device memory, 16-byte aligned
    if (((uintptr_t)q & 15) != 0) return false;
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, q) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeDevice;
}

cudaError_t launch_score_fused(const ScoreShape &sh, const void *q, const void *index,
                               int64_t c0, int64_t c1, const ScoreScratch &scr,
                               int64_t partial_stride, cudaStream_t s) {
    if (c1 <= c0) return cudaSuccess;
    if (((uintptr_t)index & 15) != 0) return cudaErrorMisalignedAddress;
    if (sh.d == 128) return fused_t<128>(sh, q, index, c0, c1, scr, partial_stride, s);
    return fused_t<64>(sh, q, index, c0, c1, scr, partial_stride, s);
}

}  // namespace kvm
