// Grouped-mode (large T) stage-1 and stage-2 group GEMMs on CTA pairs: the
// two-SM form of the tcgen05 tensor core (.cta_group::2) computes one
// 256 x 256 tile per pair, bf16 (QT = 0) or per-token e4m3 (QT = 1) inputs,
// fp32 accumulation in TMEM.
//
// Why pairs: a one-SM 128 x 256 tile moves 384 operand rows through shared
// memory for 128 * 256 products per K step; a pair tile moves 2 x 256 rows
// for 256 * 256, a third fewer bytes per FLOP through the L2 -> SM path,
// which is what limits the one-SM kernel at FP8 rates.
//
// A pair tile is two consecutive 128-row blocks of one expert's sorted rows
// (the token sort of the AITER walk-through, section 3.1, pads every expert
// to whole blocks) against 256 weight rows: stage 1, 128 gate rows and the
// matching 128 up rows (accumulator columns j and 128 + j pair up for
// SwiGLU); stage 2, 256 rows of W_down.  CTA r of the pair holds block r of
// the tokens (A rows) and weight half r (B columns) in its shared memory, and
// block r's 128 accumulator rows in its TMEM.  An expert with an odd block
// count ends on a half-used pair: the second CTA repeats the first block's
// rows and stores nothing.
//
// Roles (192 threads per CTA, one CTA per SM):
//   warp 0      TMA producer in both CTAs: the CTA's own A and B halves; both
//               CTAs' bytes complete on the leader's stage barrier
//   warp 1      TMEM allocation of the pair (both CTAs); in the leader, one
//               thread issues the pair MMAs and commits them to barriers of
//               both CTAs (stage free, accumulator ready)
//   warps 2..5  epilogue in both CTAs on the CTA's own accumulator rows;
//               they release the accumulator on the leader's barrier
// The leader claims tiles from a global counter and publishes each index to
// both CTAs through a small shared-memory queue.  Within an expert, groups of
// up to 8 pairs walk the N tiles together so that one weight tile serves 16
// token blocks from L2.  Every wait is bounded; a CTA that gives up raises the status word
// and both CTAs still meet at the final cluster barrier.
//
// Light experts (LT = 1, stages 1 and 2, bf16): an expert with at most 64
// tokens would waste most of a 256-row pair tile on padding (fine-grained
// routing leaves most experts with a few tokens).  Its tiles swap the
// operands instead: the pair's 256-row MMA side holds weight rows (128 per
// CTA) and the N side its np = ceil32(count) token rows (np / 2 <= 32 per
// CTA, loaded in 16-row boxes).  Each K step issues two MMAs into two
// accumulators of the same TMEM lanes: stage 1 gate rows and the matching
// up rows (SwiGLU still pairs within a thread; a tile covers 256
// intermediate columns), stage 2 two consecutive 256-row ranges of W_down (a
// tile covers 512 output features).  So a light tile streams 32 KB of
// weights per CTA per K step and six 36 KB stages keep 192 KB in flight: a
// light tile is bound by the bytes in flight per SM at the loaded memory
// latency, not by the tensor core (hence the 64-token limit: a 128-token
// light tile would need 40 KB stages, of which only five fit).  The epilogue holds one feature per
// thread and a token per accumulator column.  Heavy and light experts' tiles are claimed from the same counter,
// so tensor-bound and weight-streaming tiles run side by side.
#include <atomic>
#include "gemm_common.cuh"
#include "moe_internal.h"
#include "sm100_ptx.cuh"

namespace moe {

namespace gemm2sm {

constexpr int kHalfBytes = 128 * 128;       // 128 rows x 128 bytes of K
constexpr int kSwapRowsPerLoad = 16;        // token rows per TMA box of a light expert's tile
// Pipeline stage: [A: token rows | B: weight rows]; with light-expert tiles a stage also holds
// [weight rows 0-127 | weight rows 128-255 of the second range | up to 32 token rows], 36 KB.
constexpr int kMaxLightTokens = 64;
template <int STAGE, int LT>
constexpr int kStageBytesT = LT ? 2 * kHalfBytes + kMaxLightTokens / 2 * 128 : 2 * kHalfBytes;
template <int STAGE, int LT>
constexpr int kStagesT = 6;
// Per-expert tables in shared memory: with light tiles the six 36 KB stages leave room for 512.
constexpr int kMaxELight = 512;
constexpr int kAccCols = 256;
constexpr int kTmemCols = 2 * kAccCols;
constexpr int kThreads = 192;
constexpr int kEpiWarps = 4;
constexpr int kMaxE = 1024;
// Pairs of one expert that walk the N tiles together (16 token blocks).  A
// whole-expert group in stage 1 (up to 9 pairs at Mixtral prefill) measured
// slower: 76 clusters then share a smaller set of L2 lines.
template <int STAGE>
constexpr int kGroupPairs = 8;

template <int STAGE, int LT>
struct __align__(1024) Smem {
    static constexpr int kStages = kStagesT<STAGE, LT>;
    static constexpr int kStageBytes = kStageBytesT<STAGE, LT>;
    uint8_t stage[kStages][kStageBytes];
    uint64_t full[kStages];    // leader: both CTAs' TMA bytes of the stage
    uint64_t empty[kStages];   // both: the pair MMAs have read the stage
    uint64_t tfull[2];         // both: accumulator complete
    uint64_t tempty[2];        // leader: both CTAs' epilogues have drained it
    uint64_t drain;
    int qidx[kTileQ];          // tile queue: indices claimed by the leader, published to both CTAs
    uint64_t qfull[kTileQ];    // both: an index is in this CTA's slot
    uint64_t qempty[kTileQ];   // leader: every consumer of both CTAs has read the slot
    uint32_t tmem_base;
    int abort;
    int ntiles;
    int off[(LT ? kMaxELight : kMaxE) + 1];     // expert_offsets (sorted rows)
    int tstart[(LT ? kMaxELight : kMaxE) + 1];  // first pair tile of each expert (LT: among the 256 x 256 tiles)
    int lstart[LT ? kMaxELight + 1 : 1];        // LT: first light-expert tile of each expert
    int nheavy, nlight;        // LT: tiles of each kind
};

template <int STAGE, int LT>
constexpr size_t kSmemBytesT = sizeof(Smem<STAGE, LT>) + 1024;
static_assert(kSmemBytesT<1, 1> <= 227 * 1024 && kSmemBytesT<2, 1> <= 227 * 1024 && kSmemBytesT<1, 0> <= 227 * 1024,
              "a CTA has at most 227 KB of shared memory");

struct PairTile {
    int e;
    int mb0;      // first 128-row block of the pair
    int second;   // the pair's second block is a real block of expert e
    int wrow0;    // weight rows of B half 0 / half 1 (light tile: gate / up rows, or W_down rows, of CTA 0)
    int wrow1;
    int ncol0;    // output column base
    int kb0, kb1; // K blocks (weight gradients: the expert's token positions)
    int swap;     // light-expert tile: weights on the MMA's 256-row side, tokens on N
    int cnt;      // light tile: the expert's token rows
    int np;       // light tile: MMA N = cnt rounded up to 32 (np / 2 rows per CTA)
};

// A light expert: at most kMaxLightTokens tokens (one 128-row block, mostly padding).
__device__ __forceinline__ bool light_expert(int nb, int cnt) { return nb == 1 && cnt <= kMaxLightTokens; }

// Tiles of one expert: ceil(blocks / 2) pairs per N tile; with LT, a light expert has none of
// those and one light tile per 256 (stage 1) or 512 (stage 2) output columns instead.
template <int STAGE, int LT>
__device__ __forceinline__ int heavy_tiles(int nb, int cnt, int nnt)
{
    return (LT && light_expert(nb, cnt)) ? 0 : (nb + 1) / 2 * nnt;
}

template <int STAGE>
constexpr int kLightCols = STAGE == 1 ? 256 : 512;

template <int STAGE, int LT>
__device__ __forceinline__ int light_tiles(const GemmArgs &a, int nb, int cnt)
{
    return (LT && light_expert(nb, cnt)) ? (a.N + kLightCols<STAGE> - 1) / kLightCols<STAGE> : 0;
}

// The last e in [0, E) with start[e] <= t (experts without tiles share their successor's start).
__device__ __forceinline__ int find_expert(const int *start, int E, int t)
{
    int lo = 0, hi = E;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (start[mid] <= t)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

// STAGE 5 (weight gradients): D[e] (M x N) = A_e B_e^T with K over expert e's
// sorted token positions; A and B are transposed activations [rows][P]; a
// pair tile is 256 rows of A (128 per CTA) x 256 rows of B.

template <int STAGE>
__device__ __forceinline__ int n_tiles_n(const GemmArgs &a)
{
    return (STAGE == 1) ? a.N / 128 : (a.N + 255) / 256;
}

template <int STAGE, int LT, class SM>
__device__ __forceinline__ PairTile decode(const SM &sm, const GemmArgs &a, int t)
{
    const int nnt = n_tiles_n<STAGE>(a);
    if (STAGE == 5) {
        const int nmp = a.M / 256;
        PairTile p;
        p.swap = p.cnt = p.np = 0;
        p.e = t / (nmp * nnt);
        const int rem = t - p.e * nmp * nnt;
        // consecutive tiles share the larger operand's rows, so that the smaller one is what each
        // tile re-reads (from L2): the W_gate_up gradient (M = 2I rows of dg | du against N = H
        // of x) walked its 112 row pairs per N tile and read 13.5 GB of DRAM per launch
        const bool m_outer = a.M > a.N;
        const int nt = m_outer ? rem % nnt : rem / nmp;
        p.mb0 = 2 * (m_outer ? rem / nnt : rem % nmp);
        p.second = 1;
        p.wrow0 = nt * 256;
        p.wrow1 = p.wrow0 + 128;
        p.ncol0 = nt * 256;
        p.kb0 = sm.off[p.e] / 64;
        p.kb1 = sm.off[p.e + 1] / 64;
        return p;
    }
    PairTile p;
    p.swap = p.cnt = p.np = 0;
    if (LT) {
        // The two kinds of tile are interleaved in proportion to their counts, so that
        // weight-streaming (light) and tensor-bound (256 x 256) tiles run side by side: tile t is
        // the light tile floor(t * L / (L + H)) when that count steps at t, else heavy tile
        // t - floor(t * L / (L + H)).
        const int L = sm.nlight, tot = sm.nlight + sm.nheavy;
        const int lb = (int)((int64_t)t * L / tot);
        if ((int)((int64_t)(t + 1) * L / tot) > lb) {
            const int lo = find_expert(sm.lstart, a.E, lb);
            p.e = lo;
            // local = the slice of kLightCols output columns
            const int local = lb - sm.lstart[lo];
            p.swap = 1;
            p.mb0 = sm.off[lo] >> 7;
            p.second = 1;
            p.cnt = __ldg(a.expert_counts + lo);
            p.np = (p.cnt + 31) & ~31;
            p.ncol0 = local * kLightCols<STAGE>;
            p.wrow0 = lo * a.rows_per_expert + p.ncol0;  // gate rows (stage 1) / W_down rows ncol0..
            // stage 1: the matching up rows; stage 2: the next 256 rows of W_down
            p.wrow1 = STAGE == 1 ? lo * a.rows_per_expert + a.N + p.ncol0 : p.wrow0 + 256;
            p.kb0 = p.kb1 = 0;
            return p;
        }
        t -= lb;
    }
    const int lo = find_expert(sm.tstart, a.E, t);
    p.e = lo;
    const int local = t - sm.tstart[lo];
    const int nb = (sm.off[lo + 1] - sm.off[lo]) >> 7;
    const int np = (nb + 1) >> 1;
    const int gi = local / (kGroupPairs<STAGE> * nnt);
    const int gsize = min(kGroupPairs<STAGE>, np - gi * kGroupPairs<STAGE>);
    const int wi = local - gi * kGroupPairs<STAGE> * nnt;
    const int nt = wi / gsize;
    const int pi = gi * kGroupPairs<STAGE> + wi % gsize;
    p.mb0 = (sm.off[lo] >> 7) + 2 * pi;
    p.second = (2 * pi + 1 < nb) ? 1 : 0;
    if (STAGE == 1) {
        p.wrow0 = lo * a.rows_per_expert + nt * 128;          // gate rows
        p.wrow1 = lo * a.rows_per_expert + a.N + nt * 128;    // matching up rows
        p.ncol0 = nt * 128;
    } else {
        p.wrow0 = lo * a.rows_per_expert + nt * 256;
        p.wrow1 = p.wrow0 + 128;
        p.ncol0 = nt * 256;
    }
    p.kb0 = p.kb1 = 0;  // the whole K (set by the kernel, which knows the element size)
    return p;
}

// BT = 1 (the backward, bf16): operands read in their stored [K][N] layout (64 x 64 boxes) as
// MN-major operands, so nothing needs a transposed copy -- stages 2 and 3 (dgrad): the weights
// (a.tm_w over [E*K][N]); stage 5 (weight gradients, K = an expert's token positions): both
// activations (a.tm_x over [P][M], a.tm_w over [P][N]).
template <int STAGE, int QT, int LT, int BT>
__global__ void __launch_bounds__(kThreads, 1) gemm_pair_kernel(const __grid_constant__ GemmArgs a)
{
    static_assert(!LT || ((STAGE == 1 || STAGE == 2) && QT == 0), "light-expert tiles: bf16 stages 1 and 2");
    static_assert(!BT || ((STAGE == 2 || STAGE == 3 || STAGE == 5) && QT == 0 && !LT), "MN-major: backward stages");
    using SmemT = Smem<STAGE, LT>;
    constexpr int kStages = SmemT::kStages;
    extern __shared__ uint8_t smem_raw[];
    SmemT &sm = *reinterpret_cast<SmemT *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    volatile int *abort_flag = &sm.abort;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.tfull[i], 1);
            mbar_init(&sm.tempty[i], 2 * kEpiWarps);
        }
        mbar_init(&sm.drain, 1);
        for (int i = 0; i < kTileQ; ++i) {
            mbar_init(&sm.qfull[i], 1);
            mbar_init(&sm.qempty[i], 2 * (1 + kEpiWarps));  // producer/MMA + epilogue warps of each CTA
        }
        sm.abort = 0;
        fence_mbarrier_init();
        tma_prefetch_desc(&a.tm_x);
        tma_prefetch_desc(&a.tm_w);
        if (LT)
            tma_prefetch_desc(&a.tm_x16);
    }
    if (warp == 1) {
        tmem_alloc_pair(&sm.tmem_base, kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers exist before any cross-CTA signal
    tc_fence_after();
    const uint32_t tmem_base = sm.tmem_base;
    pdl_wait();
    pdl_trigger();

    // pair-tile table: tstart[e] = sum over experts before e of ceil(blocks/2) * N tiles
    if (STAGE == 5 && warp == 2) {
        for (int e = lane; e <= a.E; e += 32)
            sm.off[e] = a.expert_offsets[e];
        if (lane == 0)
            sm.ntiles = a.E * (a.M / 256) * n_tiles_n<STAGE>(a);
    } else if (warp == 2) {
        // per-expert tile starts: a warp scan over the experts (light tiles separately with LT)
        const int E = a.E;
        const int nnt = n_tiles_n<STAGE>(a);
        const int per = (E + 31) / 32;
        const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
        int hsum = 0, lsum = 0;
        for (int e = e0; e < e1; ++e) {
            const int o0 = a.expert_offsets[e], o1 = a.expert_offsets[e + 1];
            const int cnt = LT ? a.expert_counts[e] : 0;
            sm.off[e] = o0;
            hsum += heavy_tiles<STAGE, LT>((o1 - o0) >> 7, cnt, nnt);
            lsum += light_tiles<STAGE, LT>(a, (o1 - o0) >> 7, cnt);
        }
        int hincl = hsum, lincl = lsum;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int hv = __shfl_up_sync(0xffffffffu, hincl, d);
            const int lv = __shfl_up_sync(0xffffffffu, lincl, d);
            if (lane >= d) {
                hincl += hv;
                lincl += lv;
            }
        }
        int hrun = hincl - hsum, lrun = lincl - lsum;
        for (int e = e0; e < e1; ++e) {
            const int nb = (a.expert_offsets[e + 1] - a.expert_offsets[e]) >> 7;
            const int cnt = LT ? a.expert_counts[e] : 0;
            sm.tstart[e] = hrun;
            hrun += heavy_tiles<STAGE, LT>(nb, cnt, nnt);
            if (LT) {
                sm.lstart[e] = lrun;
                lrun += light_tiles<STAGE, LT>(a, nb, cnt);
            }
        }
        if (lane == 31) {
            sm.tstart[E] = hincl;
            if (LT)
                sm.lstart[E] = lincl;
            sm.off[E] = a.expert_offsets[E];
            sm.nheavy = hincl;
            sm.nlight = lincl;
            sm.ntiles = hincl + lincl;
        }
    }
    __syncthreads();
    const int ntiles = sm.ntiles;
    const int nkb = a.K / kBK<QT>;
    // consumers of the tile queue: wait for the slot, read it, release it on the leader
    auto pop = [&](int &qs, uint32_t &qph, int &t) -> bool {
        if (!mbar_wait_cluster(&sm.qfull[qs], qph, a.status, abort_flag))
            return false;
        t = *reinterpret_cast<volatile int *>(&sm.qidx[qs]);
        return true;
    };
    auto release = [&](int qs) { mbar_arrive_cluster(cluster_map(&sm.qempty[qs], 0)); };

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer
        if (lane == 0) {
            // Weight tiles of 256 x 256 tiles are read by up to 8 pairs of a group within a few
            // microseconds; streamed as evict-first they were dropped between those reads while
            // light tiles streamed their weights through L2 (fine-grained stage 1: 10.97 GB of
            // DRAM reads per launch against 7.99 GB algorithmic; Mixtral prefill 4.33 GB against
            // 2.5).  Kept as evict-last they are read about once (9.5 and 2.96 GB; fine-grained
            // 3.39 -> 3.24 ms, prefill stage 1 2.48 -> 2.42 ms, same box).  Light tiles read their
            // weights once: evict-first.
            const uint64_t pol_w = l2_policy_evict_first();
            const uint64_t pol_wh = l2_policy_evict_last();
            const uint64_t pol_x = l2_policy_evict_last();
            int s = 0;
            uint32_t ph = 0;
            bool ok = true, any = false;
            int qs = 0;
            uint32_t qph = 0;
            // the leader claims tiles one ahead from the global counter (uneven pair speeds balance out)
            int claim = leader ? atomicAdd(a.tile_counter, 1) : 0;
            for (;;) {
                int t;
                if (leader) {
                    if (!mbar_wait_cluster(&sm.qempty[qs], qph ^ 1, a.status, abort_flag)) {
                        ok = false;
                        break;
                    }
                    t = claim < ntiles ? claim : -1;
                    *reinterpret_cast<volatile int *>(&sm.qidx[qs]) = t;
                    st_cluster_s32(cluster_map(&sm.qidx[qs], 1), t);
                    mbar_arrive(&sm.qfull[qs]);
                    mbar_arrive_cluster(cluster_map(&sm.qfull[qs], 1));
                    if (t >= 0)
                        claim = atomicAdd(a.tile_counter, 1);
                } else {
                    if (!pop(qs, qph, t)) {
                        ok = false;
                        break;
                    }
                    release(qs);
                }
                if (++qs == kTileQ) {
                    qs = 0;
                    qph ^= 1;
                }
                if (t < 0)
                    break;
                const PairTile p = decode<STAGE, LT>(sm, a, t);
                const int xrow = (rank == 1 && p.second) ? (p.mb0 + 1) * 128 : p.mb0 * 128;
                const int wrow = rank == 0 ? p.wrow0 : p.wrow1;
                const int kb0 = STAGE == 5 ? p.kb0 : 0, kb1 = STAGE == 5 ? p.kb1 : nkb;
                // light tile: this CTA's half of the token rows, and the bytes of both CTAs per stage
                const int half = p.swap ? p.np / 2 : 0;
                const uint32_t swap_bytes = 2u * (2 * kHalfBytes + half * 128);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&sm.empty[s], ph ^ 1, a.status, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fullc = cluster_map(&sm.full[s], 0);
                    if (LT && p.swap) {
                        if (leader)
                            mbar_arrive_expect_tx(&sm.full[s], swap_bytes);
                        // weights: rows r*128.. of each of the tile's two 256-row ranges, tokens after them
                        tma_load_2d_pair(sm.stage[s], &a.tm_w, kb * kBK<QT>, p.wrow0 + (int)rank * 128, fullc,
                                         pol_w);
                        tma_load_2d_pair(sm.stage[s] + kHalfBytes, &a.tm_w, kb * kBK<QT>, p.wrow1 + (int)rank * 128,
                                         fullc, pol_w);
                        uint8_t *tok = sm.stage[s] + 2 * kHalfBytes;
                        const int trow = p.mb0 * 128 + (int)rank * half;
                        for (int c = 0; c < half; c += kSwapRowsPerLoad)
                            tma_load_2d_pair(tok + c * 128, &a.tm_x16, kb * kBK<QT>, trow + c, fullc, pol_x);
                    } else {
                        if (leader)
                            mbar_arrive_expect_tx(&sm.full[s], 2 * 2 * kHalfBytes);
                        if (BT && STAGE == 5) {
                            // A: this CTA's 128 gradient rows (columns of [P][M]) at token rows kb*64..
                            tma_load_2d_pair(sm.stage[s], &a.tm_x, xrow, kb * 64, fullc, pol_x);
                            tma_load_2d_pair(sm.stage[s] + kHalfBytes / 2, &a.tm_x, xrow + 64, kb * 64, fullc,
                                             pol_x);
                        } else {
                            tma_load_2d_pair(sm.stage[s], &a.tm_x, kb * kBK<QT>, xrow, fullc, pol_x);
                        }
                        if (BT) {
                            // this CTA's 128 of the tile's 256 N columns at K rows kb*64..: two 64 x 64
                            // boxes, 8 KB apart (weights: expert e's rows of [E*K][N])
                            const int n0 = STAGE == 5 ? wrow : p.ncol0 + (int)rank * 128;
                            const int k0 = (STAGE == 5 ? 0 : p.e * a.K) + kb * 64;
                            tma_load_2d_pair(sm.stage[s] + kHalfBytes, &a.tm_w, n0, k0, fullc, pol_wh);
                            tma_load_2d_pair(sm.stage[s] + kHalfBytes + kHalfBytes / 2, &a.tm_w, n0 + 64, k0, fullc,
                                             pol_wh);
                        } else {
                            tma_load_2d_pair(sm.stage[s] + kHalfBytes, &a.tm_w, kb * kBK<QT>, wrow, fullc, pol_wh);
                        }
                    }
                    any = true;
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1;
                    }
                }
                if (!ok)
                    break;
            }
            if (!ok && any) {
                // copies in flight complete on the leader's barriers: give them a bounded moment to land
                const unsigned long long t0 = global_timer_ns();
                while (global_timer_ns() - t0 < 20000000ull) {
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        if (leader && lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int acc = 0;
            uint32_t aph = 0;
            bool ok = true, any = false;
            const uint32_t idesc = BT ? (make_idesc_bmn(1, 1, 256, 256) | (STAGE == 5 ? 1u << 15 : 0u))  // A MN-major too
                                      : make_idesc(QT ? 0u : 1u, QT ? 0u : 1u, 256, 256);
            int qs = 0;
            uint32_t qph = 0;
            for (;;) {
                int t;
                if (!pop(qs, qph, t)) {
                    ok = false;
                    break;
                }
                release(qs);
                if (++qs == kTileQ) {
                    qs = 0;
                    qph ^= 1;
                }
                if (t < 0)
                    break;
                if (!mbar_wait(&sm.tempty[acc], aph ^ 1, a.status, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + acc * kAccCols;
                int kb0 = 0, kb1 = nkb;
                bool swap = false;
                uint32_t idesc_swap = 0;
                if (STAGE == 5 || LT) {
                    const PairTile p = decode<STAGE, LT>(sm, a, t);
                    kb0 = STAGE == 5 ? p.kb0 : 0;
                    kb1 = STAGE == 5 ? p.kb1 : nkb;
                    swap = p.swap != 0;
                    if (swap)
                        idesc_swap = make_idesc(1, 1, 256, (uint32_t)p.np);
                }
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&sm.full[s], ph, a.status, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t accum0 = kb > kb0 ? 1u : 0u;
                    if (LT && swap) {
                        // A = weight rows (this CTA's 128 of each 256-row range), B = the expert's token
                        // rows; the second range into the second accumulator half
                        const uint8_t *w0 = sm.stage[s];
                        const uint8_t *tok = sm.stage[s] + 2 * kHalfBytes;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint32_t accum = (kk > 0) ? 1u : accum0;
                            mma_pair<QT>(d, smem_desc_sw128(w0 + kk * 32), smem_desc_sw128(tok + kk * 32),
                                         idesc_swap, accum);
                            mma_pair<QT>(d + 128, smem_desc_sw128(w0 + kHalfBytes + kk * 32),
                                         smem_desc_sw128(tok + kk * 32), idesc_swap, accum);
                        }
                    } else {
                        const uint8_t *xa = sm.stage[s];
                        const uint8_t *wb = sm.stage[s] + kHalfBytes;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            // B: K-major 32 bytes further per 16 K, or MN-major 16 rows (2 KB) further
                            const uint64_t bdesc = BT ? smem_desc_sw128_mn(wb + kk * 2048, kHalfBytes / 2)
                                                      : smem_desc_sw128(wb + kk * 32);
                            const uint64_t adesc = (BT && STAGE == 5) ? smem_desc_sw128_mn(xa + kk * 2048, kHalfBytes / 2)
                                                                      : smem_desc_sw128(xa + kk * 32);
                            mma_pair<QT>(d, adesc, bdesc, idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    any = true;
                    mma_commit_pair(&sm.empty[s], 0x3);
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1;
                    }
                }
                if (!ok)
                    break;
                mma_commit_pair(&sm.tfull[acc], 0x3);
                if (++acc == 2) {
                    acc = 0;
                    aph ^= 1;
                }
            }
            if (!ok && any) {
                mma_commit_pair(&sm.drain, 0x1);
                const unsigned long long t0 = global_timer_ns();
                while (!mbar_try_wait(&sm.drain, 0) && global_timer_ns() - t0 < 100000000ull) {
                }
            }
        }
    } else {
        // -------------------------------------------------------- epilogue
        const int q = warp & 3;           // TMEM lane quadrant of this warp
        const int row = q * 32 + lane;    // accumulator row = token row within the CTA's block
        int acc = 0;
        uint32_t aph = 0;
        int qs = 0;
        uint32_t qph = 0;
        for (;;) {
            int t = -1;
            bool qok = pop(qs, qph, t);
            qok = __all_sync(0xffffffffu, qok);
            if (!qok)
                break;
            __syncwarp();
            if (lane == 0)
                release(qs);
            if (++qs == kTileQ) {
                qs = 0;
                qph ^= 1;
            }
            if (t < 0)
                break;
            const PairTile p = decode<STAGE, LT>(sm, a, t);
            const bool store = rank == 0 || p.second;
            const int pos = (p.mb0 + (int)rank) * 128 + row;   // sorted row of this thread
            if (STAGE == 3 && store) {
                // the saved g | u this thread's epilogue reads (2 x 512 bytes of its row, from DRAM):
                // into L2 while the tile's MMAs run, so that the epilogue's loads wait on L2 only
                const __nv_bfloat16 *gr = a.gu_in + (size_t)pos * (2 * a.N) + p.ncol0;
#pragma unroll
                for (int c = 0; c < 256; c += 64) {
                    prefetch_l2(gr + c);
                    prefetch_l2(gr + a.N + c);
                }
            }
            bool ok = mbar_wait(&sm.tfull[acc], aph, a.status, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok)
                break;
            tc_fence_after();
            const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16) + acc * kAccCols;
            if (LT && p.swap) {
                // one output feature per thread, one token per accumulator column
                const int f = p.ncol0 + (int)rank * 128 + row;
                const int row0 = p.mb0 * 128;  // the expert's first sorted row
#pragma unroll 1
                for (int c0 = 0; c0 < p.np; c0 += 32) {
                    float v[32];
                    tmem_ld32(tacc + c0, v);
                    if (STAGE == 1) {
                        float u[32];
                        tmem_ld32(tacc + 128 + c0, u);
                        __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.inter) + (size_t)(row0 + c0) * a.N + f;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            dst[(size_t)j * a.N] = __float2bfloat16_rn(silu(v[j]) * u[j]);
                    } else {
                        // features f (first accumulator half) and f + 256 (second half)
                        float v2[32];
                        tmem_ld32(tacc + 128 + c0, v2);
                        const bool ok0 = f < a.N, ok1 = f + 256 < a.N;
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const int c = c0 + j;
                            if (c < p.cnt) {
                                const int slot = a.sorted_ids[row0 + c];
                                const float wgt = a.sorted_weights[row0 + c];
                                if (ok0)
                                    a.y[(size_t)slot * a.N + f] = __float2bfloat16_rn(wgt * v[j]);
                                if (ok1)
                                    a.y[(size_t)slot * a.N + f + 256] = __float2bfloat16_rn(wgt * v2[j]);
                            }
                        }
                    }
                }
            } else if (STAGE == 1) {
                __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.inter) + (size_t)pos * a.N + p.ncol0;
                const float sx = (QT && store) ? a.x_scales[pos] : 1.0f;
#pragma unroll 1
                for (int c0 = 0; c0 < 128; c0 += 32) {
                    float g[32], u[32], h[32];
                    tmem_ld32(tacc + c0, g);
                    tmem_ld32(tacc + 128 + c0, u);
                    if (!store)
                        continue;
                    if (QT) {
#pragma unroll
                        for (int i = 0; i < 32; i += 4) {
                            const float4 sg = ld_scale4(a.w_scales + p.wrow0 + c0 + i);
                            const float4 su = ld_scale4(a.w_scales + p.wrow1 + c0 + i);
                            g[i] *= sx * sg.x, g[i + 1] *= sx * sg.y, g[i + 2] *= sx * sg.z, g[i + 3] *= sx * sg.w;
                            u[i] *= sx * su.x, u[i + 1] *= sx * su.y, u[i + 2] *= sx * su.z, u[i + 3] *= sx * su.w;
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        h[i] = silu(g[i]) * u[i];
                    store_bf16x32(dst + c0, h);
                    if (a.gu) {  // training: keep the pre-activations for the backward
                        __nv_bfloat16 *gr = a.gu + (size_t)pos * (2 * a.N) + p.ncol0 + c0;
                        store_bf16x32(gr, g);
                        store_bf16x32(gr + a.N, u);
                    }
                }
            } else if (STAGE == 3) {
                // backward of stage 2: dh in the accumulator; SwiGLU's backward with the saved g | u
                const __nv_bfloat16 *gr = a.gu_in + (size_t)pos * (2 * a.N) + p.ncol0;
                __nv_bfloat16 *dr = a.dgu + (size_t)pos * (2 * a.N) + p.ncol0;
#pragma unroll 1
                for (int c0 = 0; c0 < 256; c0 += 32) {
                    float dh[32], dg[32], du[32];
                    tmem_ld32(tacc + c0, dh);
                    if (!store)
                        continue;
#pragma unroll
                    for (int i = 0; i < 32; i += 8) {
                        const uint4 gv = *reinterpret_cast<const uint4 *>(gr + c0 + i);
                        const uint4 uv = *reinterpret_cast<const uint4 *>(gr + a.N + c0 + i);
                        const __nv_bfloat162 *g2 = reinterpret_cast<const __nv_bfloat162 *>(&gv);
                        const __nv_bfloat162 *u2 = reinterpret_cast<const __nv_bfloat162 *>(&uv);
#pragma unroll
                        for (int q2 = 0; q2 < 4; ++q2) {
                            const float2 gf = __bfloat1622float2(g2[q2]);
                            const float2 uf = __bfloat1622float2(u2[q2]);
                            const float gg[2] = {gf.x, gf.y}, uu[2] = {uf.x, uf.y};
#pragma unroll
                            for (int r = 0; r < 2; ++r) {
                                const int ii = i + 2 * q2 + r;
                                const float sg = sigmoid_fast(gg[r]);
                                dg[ii] = dh[ii] * uu[r] * sg * (1.0f + gg[r] * (1.0f - sg));
                                du[ii] = dh[ii] * gg[r] * sg;
                            }
                        }
                    }
                    store_bf16x32(dr + c0, dg);
                    store_bf16x32(dr + a.N + c0, du);
                }
            } else if (STAGE == 5) {
                // weight gradient: rows (mb0 + rank) * 128 + row of expert e's gradient
                float *dst = a.dw_out + ((size_t)p.e * a.M + pos) * a.N + p.ncol0;
                const int ncols = min(256, a.N - p.ncol0);
                const bool empty = p.kb0 == p.kb1;  // an expert without tokens: zero gradient
#pragma unroll 1
                for (int c0 = 0; c0 < ncols; c0 += 32) {
                    float v[32];
                    tmem_ld32(tacc + c0, v);
                    float4 *d4 = reinterpret_cast<float4 *>(dst + c0);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        d4[i] = empty ? make_float4(0.f, 0.f, 0.f, 0.f)
                                      : make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                }
            } else {
                const int slot = store ? a.sorted_ids[pos] : a.S;
                const bool live = slot < a.S;
                // no weights: the unweighted rows (the backward's dx per slot)
                const float wgt =
                    live ? (a.sorted_weights ? a.sorted_weights[pos] : 1.0f) * (QT ? a.x_scales[pos] : 1.0f) : 0.0f;
                __nv_bfloat16 *dst = a.y + (size_t)(live ? slot : 0) * a.N + p.ncol0;
                const int ncols = min(256, a.N - p.ncol0);
#pragma unroll 1
                for (int c0 = 0; c0 < ncols; c0 += 32) {
                    float v[32];
                    tmem_ld32(tacc + c0, v);
                    if (!live)
                        continue;
                    if (QT) {
#pragma unroll
                        for (int i = 0; i < 32; i += 4) {
                            const float4 sw = ld_scale4(a.w_scales + p.wrow0 + c0 + i);
                            v[i] *= sw.x, v[i + 1] *= sw.y, v[i + 2] *= sw.z, v[i + 3] *= sw.w;
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        v[i] *= wgt;
                    store_bf16x32(dst + c0, v);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive_remote(cluster_map(&sm.tempty[acc], 0));
            if (++acc == 2) {
                acc = 0;
                aph ^= 1;
            }
        }
    }

    // both CTAs stay until the pair's last MMA, copy and remote arrive are done
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    if (warp == 1)
        tmem_dealloc_pair(tmem_base, kTmemCols);
}

template <int STAGE, int QT, int LT, int BT = 0>
cudaError_t launch(const GemmArgs &a, int clusters, cudaStream_t st)
{
    auto kern = gemm_pair_kernel<STAGE, QT, LT, BT>;
    constexpr size_t smem = kSmemBytesT<STAGE, LT>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess)
        return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

// Clusters of two that can be resident at once (one CTA per SM), cached per device.
template <int STAGE, int QT, int LT, int BT = 0>
int max_clusters()
{
    static std::atomic<int> cache[64];  // per device, zero until first computed
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 0;
    if (cache[dev].load(std::memory_order_relaxed) == 0) {
        auto kern = gemm_pair_kernel<STAGE, QT, LT, BT>;
        constexpr size_t smem = kSmemBytesT<STAGE, LT>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return 0;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0)
            return 0;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return cache[dev].load(std::memory_order_relaxed);
}

}  // namespace gemm2sm

bool gemm_pair_supported(int E) { return E <= gemm2sm::kMaxE; }
bool gemm_pair_light_supported(int E) { return E <= gemm2sm::kMaxELight; }

cudaError_t launch_gemm_pair(int stage, int qt, const GemmArgs &a, int64_t max_pair_tiles, cudaStream_t st,
                             bool light, bool w_mn_major)
{
    // stages 1, 2 (bf16 or per-token FP8; bf16 optionally with light-expert tiles); 3 and 5
    // (training, bf16): the backward of stage 2 and the weight gradients
    if (light && (qt || (stage != 1 && stage != 2)))
        return cudaErrorInvalidValue;
    if (w_mn_major && (qt || light || (stage != 2 && stage != 3 && stage != 5)))
        return cudaErrorInvalidValue;
    const int key = stage * 4 + (qt ? 1 : 0) + (light ? 2 : 0) + (w_mn_major ? 64 : 0);
    int ncl = 0;
    switch (key) {
    case 4: ncl = gemm2sm::max_clusters<1, 0, 0>(); break;
    case 5: ncl = gemm2sm::max_clusters<1, 1, 0>(); break;
    case 6: ncl = gemm2sm::max_clusters<1, 0, 1>(); break;
    case 8: ncl = gemm2sm::max_clusters<2, 0, 0>(); break;
    case 9: ncl = gemm2sm::max_clusters<2, 1, 0>(); break;
    case 10: ncl = gemm2sm::max_clusters<2, 0, 1>(); break;
    case 12: ncl = gemm2sm::max_clusters<3, 0, 0>(); break;
    case 72: ncl = gemm2sm::max_clusters<2, 0, 0, 1>(); break;
    case 76: ncl = gemm2sm::max_clusters<3, 0, 0, 1>(); break;
    case 84: ncl = gemm2sm::max_clusters<5, 0, 0, 1>(); break;
    case 20: ncl = gemm2sm::max_clusters<5, 0, 0>(); break;
    default: return cudaErrorInvalidValue;
    }
    if (ncl <= 0)
        return cudaErrorInvalidConfiguration;
    if (max_pair_tiles < ncl)
        ncl = (int)(max_pair_tiles > 0 ? max_pair_tiles : 1);
    switch (key) {
    case 4: return gemm2sm::launch<1, 0, 0>(a, ncl, st);
    case 5: return gemm2sm::launch<1, 1, 0>(a, ncl, st);
    case 6: return gemm2sm::launch<1, 0, 1>(a, ncl, st);
    case 8: return gemm2sm::launch<2, 0, 0>(a, ncl, st);
    case 9: return gemm2sm::launch<2, 1, 0>(a, ncl, st);
    case 10: return gemm2sm::launch<2, 0, 1>(a, ncl, st);
    case 12: return gemm2sm::launch<3, 0, 0>(a, ncl, st);
    case 72: return gemm2sm::launch<2, 0, 0, 1>(a, ncl, st);
    case 76: return gemm2sm::launch<3, 0, 0, 1>(a, ncl, st);
    case 84: return gemm2sm::launch<5, 0, 0, 1>(a, ncl, st);
    default: return gemm2sm::launch<5, 0, 0>(a, ncl, st);
    }
}

}  // namespace moe
