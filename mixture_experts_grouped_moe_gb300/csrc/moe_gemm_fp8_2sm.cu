// Block-scaled FP8 (e4m3, fp32 scales per 1x128 activation group and per
// 128x128 weight block) group GEMMs of the fused MoE layer on CTA pairs
// ("per_1x128" quantisation of the AITER walk-through, two-stage path with
// the intermediate re-quantised between the stages, section 3.2).
//
// The one-SM kernel (moe_gemm_fp8.cu) computes 128 token rows x 256 weight
// rows per tile; its tensor core is fed 384 operand rows from shared memory
// per 128 x 256 products, and its K blocks run at about 88 % of the FP8 rate
// with the L2 -> SM path carrying 48 KB per K block.  Here a pair of CTAs
// (tcgen05 .cta_group::2) computes 256 token rows x 256 weight rows: CTA r
// holds token block r (A rows) and weight half r (B columns), 32 KB per K
// block, and keeps its 128 accumulator rows x 256 columns in its own TMEM --
// the same accumulator shape per SM as the one-SM kernel, so the promotion
// and the epilogues are that kernel's, run in both CTAs:
//     acc[row][col] += D_kb[row][col] * s_x[row][kb] * s_w[col_block][kb]
// over two TMEM buffers (the tensor core fills one with K block kb + 1 while
// eight promotion warps per CTA fold the other into registers), then
// stage 1: h = silu(gate) * up, re-quantised per 1x128 group (scale =
// amax / 448); stage 2: rows scaled by their top-k weight into y.  The
// products and the promotion order are the one-SM kernel's, so both give the
// same bits.
//
// Measured on GB300 (Mixtral shapes, T=4096): stage 1 1.14 ms against the
// one-SM kernel's 0.82, stage 2 0.48 against 0.48.  Neither kernel is fed
// too slowly (this one draws 7.8 TB/s from L2, tensor pipe 41 % active): the
// pace is set by the K-block round trip MMA -> promotion -> release, which
// here waits for the promotion warps of both SMs, and the release arrives
// from the other SM.  So the library picks this kernel only on request
// (per-call gemm_pair = 1).  The per-K-block signals use CTA-scope
// semantics: a cluster-scope release there made every release wait for the
// promotion warp's scale loads in flight (stage 1: 2.25 ms).
//
// Pair tiles: two consecutive 128-row blocks of one expert's sorted rows (the
// sort pads every expert to whole blocks, section 3.1) x 256 weight rows
// (stage 1: 128 gate rows and the matching 128 up rows; stage 2: 256 rows of
// W_down).  An expert with an odd block count ends on a half-used pair: the
// second CTA repeats the first block's rows and stores nothing.  Within an
// expert, groups of up to 8 pairs walk the N tiles together (one weight tile
// serves 16 token blocks from L2).  The leader claims tiles from a global
// counter and publishes them to both CTAs through a shared-memory queue.
//
// Roles (320 threads per CTA, one CTA per SM):
//   warp 0      TMA producer in both CTAs (the CTA's own A and B halves; both
//               CTAs' bytes complete on the leader's stage barrier)
//   warp 1      TMEM allocation of the pair; in the leader, one thread issues
//               the pair MMAs and commits them to barriers of both CTAs
//   warps 2..9  promotion + epilogue on the CTA's own accumulator rows: warp w
//               reads TMEM lanes 32*(w%4)..+31, and (w-2)/4 picks half of the
//               256 columns; they release a TMEM buffer on the leader's barrier
// Every wait is bounded; a CTA that gives up raises the status word, and both
// CTAs still meet at the final cluster barrier.
#include <atomic>
#include <cuda_fp8.h>

#include "gemm_common.cuh"
#include "moe_internal.h"
#include "sm100_ptx.cuh"

namespace moe {

namespace fp8pair {

constexpr int kBK = 128;                  // one 128-wide K block (128 bytes of e4m3) per stage
constexpr int kHalfBytes = 128 * 128;     // 128 rows x 128 bytes
constexpr int kStageBytes = 2 * kHalfBytes;
constexpr int kStages = 6;
constexpr int kAccCols = 256;
constexpr int kTmemCols = 2 * kAccCols;
constexpr int kPromoWarps = 8;
constexpr int kLdCols = 16;
constexpr int kSubs = kPromoWarps / 4;
constexpr int kChunk = 256 / (2 * kSubs);
constexpr int kThreads = 64 + 32 * kPromoWarps;
constexpr int kMaxE = 1024;
constexpr int kGroupPairs = 8;
static_assert(kChunk == 64, "each thread owns two 64-column chunks of the 256 accumulator columns");

struct __align__(1024) Smem {
    uint8_t stage[kStages][kStageBytes];  // [A: the CTA's 128 token rows | B: its 128 weight rows]
    uint64_t full[kStages];     // leader: both CTAs' TMA bytes of the stage
    uint64_t empty[kStages];    // both: the pair MMAs have read the stage
    uint64_t tfull[2];          // both: a K block's products are in the TMEM buffer
    uint64_t tempty[2];         // leader: both CTAs' promotion warps have read the buffer
    uint64_t drain;
    int qidx[kTileQ];           // tile queue: indices claimed by the leader, published to both CTAs
    uint64_t qfull[kTileQ];     // both: an index is in this CTA's slot
    uint64_t qempty[kTileQ];    // leader: every consumer of both CTAs has read the slot
    uint64_t ep_bar[4];         // per lane quadrant: one phase per tile once every warp wrote its amax
    uint32_t tmem_base;
    int abort;
    int ntiles;
    int off[kMaxE + 1];         // expert_offsets (sorted rows)
    int tstart[kMaxE + 1];      // first pair tile of each expert
    float amax[2][kSubs][128];  // per tile parity: row amax of each promotion warp's h chunk
    float4 ep_out[kPromoWarps][32][4];  // a warp's 32 rows x 64 bytes on their way to global memory
};

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
static_assert(kSmemBytes <= 227 * 1024, "a CTA has at most 227 KB of shared memory");

struct PairTile {
    int mb0;      // first 128-row block of the pair
    int second;   // the pair's second block is a real block of the expert
    int wrow0;    // weight rows of B half 0 / half 1
    int wrow1;
    int ncol0;    // output column base
};

template <int STAGE>
__device__ __forceinline__ int n_tiles_n(const GemmArgs &a)
{
    return (STAGE == 1) ? a.N / 128 : (a.N + 255) / 256;
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

template <int STAGE>
__device__ __forceinline__ PairTile decode(const Smem &sm, const GemmArgs &a, int t)
{
    const int nnt = n_tiles_n<STAGE>(a);
    const int e = find_expert(sm.tstart, a.E, t);
    const int local = t - sm.tstart[e];
    const int nb = (sm.off[e + 1] - sm.off[e]) >> 7;
    const int np = (nb + 1) >> 1;
    const int gi = local / (kGroupPairs * nnt);
    const int gsize = min(kGroupPairs, np - gi * kGroupPairs);
    const int wi = local - gi * kGroupPairs * nnt;
    const int nt = wi / gsize;
    const int pi = gi * kGroupPairs + wi % gsize;
    PairTile p;
    p.mb0 = (sm.off[e] >> 7) + 2 * pi;
    p.second = (2 * pi + 1 < nb) ? 1 : 0;
    if (STAGE == 1) {
        p.wrow0 = e * a.rows_per_expert + nt * 128;          // gate rows
        p.wrow1 = e * a.rows_per_expert + a.N + nt * 128;    // matching up rows
        p.ncol0 = nt * 128;
    } else {
        p.wrow0 = e * a.rows_per_expert + nt * 256;
        p.wrow1 = p.wrow0 + 128;
        p.ncol0 = nt * 256;
    }
    return p;
}

template <int STAGE>
__global__ void __launch_bounds__(kThreads, 1) gemm_fp8_pair_kernel(const __grid_constant__ GemmArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
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
            mbar_init(&sm.tempty[i], 2 * kPromoWarps);
        }
        mbar_init(&sm.drain, 1);
        for (int i = 0; i < kTileQ; ++i) {
            mbar_init(&sm.qfull[i], 1);
            mbar_init(&sm.qempty[i], 2 * (1 + kPromoWarps));  // producer/MMA + promotion warps of each CTA
        }
        for (int i = 0; i < 4; ++i)
            mbar_init(&sm.ep_bar[i], 32 * kSubs);
        sm.abort = 0;
        fence_mbarrier_init();
        tma_prefetch_desc(&a.tm_x);
        tma_prefetch_desc(&a.tm_w);
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
    // everything above is independent of earlier kernels; from here on their outputs are read
    pdl_wait();
    pdl_trigger();

    if (warp == 2) {
        // per-expert tile starts: tstart[e] = sum over experts before e of ceil(blocks / 2) * N tiles
        const int E = a.E;
        const int nnt = n_tiles_n<STAGE>(a);
        const int per = (E + 31) / 32;
        const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
        int sum = 0;
        for (int e = e0; e < e1; ++e) {
            const int o0 = a.expert_offsets[e], o1 = a.expert_offsets[e + 1];
            sm.off[e] = o0;
            sum += (((o1 - o0) >> 7) + 1) / 2 * nnt;
        }
        int incl = sum;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d)
                incl += v;
        }
        int run = incl - sum;
        for (int e = e0; e < e1; ++e) {
            const int nb = (a.expert_offsets[e + 1] - a.expert_offsets[e]) >> 7;
            sm.tstart[e] = run;
            run += (nb + 1) / 2 * nnt;
        }
        if (lane == 31) {
            sm.tstart[E] = incl;
            sm.off[E] = a.expert_offsets[E];
            sm.ntiles = incl;
        }
    }
    __syncthreads();
    const int ntiles = sm.ntiles;
    const int nkb = a.K / kBK;
    // consumers of the tile queue: wait for the slot, read it, release it on the leader
    auto pop = [&](int qs, uint32_t qph, int &t) -> bool {
        if (!mbar_wait_cluster(&sm.qfull[qs], qph, a.status, abort_flag))
            return false;
        t = *reinterpret_cast<volatile int *>(&sm.qidx[qs]);
        return true;
    };
    auto release = [&](int qs) { mbar_arrive_cluster(cluster_map(&sm.qempty[qs], 0)); };

    if (warp == 0) {
        // ------------------------------------------------------- TMA producer
        if (lane == 0) {
            const uint64_t pol_w = l2_policy_evict_last();  // reused by the group's pairs
            const uint64_t pol_x = l2_policy_evict_last();
            int s = 0;
            uint32_t ph = 0;
            bool ok = true, any = false;
            int qs = 0;
            uint32_t qph = 0;
            int claim = leader ? atomicAdd(a.tile_counter, 1) : 0;
            for (;;) {
                int t = -1;
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
                const PairTile p = decode<STAGE>(sm, a, t);
                const int xrow = (rank == 1 && p.second) ? (p.mb0 + 1) * 128 : p.mb0 * 128;
                const int wrow = rank == 0 ? p.wrow0 : p.wrow1;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(&sm.empty[s], ph ^ 1, a.status, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fullc = cluster_map(&sm.full[s], 0);
                    if (leader)
                        mbar_arrive_expect_tx(&sm.full[s], 2 * kStageBytes);
                    tma_load_2d_pair(sm.stage[s], &a.tm_x, kb * kBK, xrow, fullc, pol_x);
                    tma_load_2d_pair(sm.stage[s] + kHalfBytes, &a.tm_w, kb * kBK, wrow, fullc, pol_w);
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
        // ------------------------------------------------------- MMA issuer
        if (leader && lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int buf = 0;
            uint32_t bph = 0;
            bool ok = true, any = false;
            const uint32_t idesc = make_idesc(0, 0, 256, 256);
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
                for (int kb = 0; kb < nkb; ++kb) {
                    // the stage is normally loaded long before its TMEM buffer is released, so
                    // waiting on it first leaves only the MMA issue after the release
                    if (!mbar_wait(&sm.full[s], ph, a.status, abort_flag) ||
                        !mbar_wait(&sm.tempty[buf], bph ^ 1, a.status, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem_base + buf * kAccCols;
                    const uint8_t *xa = sm.stage[s];
                    const uint8_t *wb = sm.stage[s] + kHalfBytes;
#pragma unroll
                    for (int kk = 0; kk < kBK / 32; ++kk)
                        mma_pair<1>(d, smem_desc_sw128(xa + kk * 32), smem_desc_sw128(wb + kk * 32), idesc,
                                    kk > 0 ? 1u : 0u);
                    any = true;
                    mma_commit_pair(&sm.empty[s], 0x3);
                    mma_commit_pair(&sm.tfull[buf], 0x3);
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1;
                    }
                    if (++buf == 2) {
                        buf = 0;
                        bph ^= 1;
                    }
                }
                if (!ok)
                    break;
            }
            if (!ok && any) {
                mma_commit_pair(&sm.drain, 0x1);
                const unsigned long long t0 = global_timer_ns();
                while (!mbar_try_wait(&sm.drain, 0) && global_timer_ns() - t0 < 100000000ull) {
                }
            }
        }
    } else {
        // ------------------------------------------------- promotion + epilogue
        const int q = warp & 3;
        const int sub = (warp - 2) >> 2;
        const int row = q * 32 + lane;
        const int c0 = (STAGE == 1) ? sub * kChunk : sub * 2 * kChunk;                // first chunk
        const int c1 = (STAGE == 1) ? 128 + sub * kChunk : sub * 2 * kChunk + kChunk;  // second chunk
        const int KB128 = a.K / 128;
        const int nrb = a.E * a.rows_per_expert / 128;
        int buf = 0;
        uint32_t bph = 0;
        bool ok = true;
        int qs = 0;
        uint32_t qph = 0;
        // Next tile and the first scales of its K loop (taken right after the last K block of the
        // current tile in stage 1, so that these dependent loads overlap its epilogue).
        int t = -1;
        PairTile tl{};
        bool store = false;
        int pos = 0;
        const float *sw0 = nullptr, *sw1 = nullptr;
        float sx_n = 0.0f, s0_n = 0.0f, s1_n = 0.0f;
        auto next_tile = [&]() -> bool {
            bool qok = pop(qs, qph, t);
            qok = __all_sync(0xffffffffu, qok);
            if (!qok)
                return false;
            __syncwarp();
            if (lane == 0)
                release(qs);
            if (++qs == kTileQ) {
                qs = 0;
                qph ^= 1;
            }
            if (t >= 0) {
                tl = decode<STAGE>(sm, a, t);
                store = rank == 0 || tl.second;
                // the sorted row of this thread; a half-used pair's second CTA reads the first
                // block's scales again (its products are those rows' too) and stores nothing
                pos = (tl.mb0 + (store ? (int)rank : 0)) * 128 + row;
                int rb0 = (STAGE == 1 ? tl.wrow0 : tl.wrow0 + sub * 2 * kChunk) / 128;
                int rb1 = (STAGE == 1 ? tl.wrow1 : tl.wrow0 + sub * 2 * kChunk) / 128;
                // a stage-2 chunk past the last output feature (H % 256 == 128) reads a valid
                // scale row and is never stored
                rb0 = rb0 < nrb ? rb0 : nrb - 1;
                rb1 = rb1 < nrb ? rb1 : nrb - 1;
                sw0 = a.w_scales + (size_t)rb0 * KB128;
                sw1 = a.w_scales + (size_t)rb1 * KB128;
                sx_n = a.x_scales[pos];
                s0_n = sw0[0];
                s1_n = sw1[0];
            }
            return true;
        };
        int gen = 0;  // epilogues done by this warp
        if (!next_tile())
            t = -1;
        while (t >= 0) {
            float acc0[kChunk], acc1[kChunk];
#pragma unroll
            for (int i = 0; i < kChunk; ++i)
                acc0[i] = 0.0f, acc1[i] = 0.0f;
            // the scales of block kb + 1 are fetched while block kb is still on the tensor core
            for (int kb = 0; kb < nkb; ++kb) {
                const float sx = sx_n, s0 = s0_n, s1 = s1_n;
                if (kb + 1 < nkb) {
                    sx_n = a.x_scales[(size_t)(kb + 1) * a.P_max + pos];
                    s0_n = sw0[kb + 1];
                    s1_n = sw1[kb + 1];
                }
                bool w_ok = mbar_wait(&sm.tfull[buf], bph, a.status, abort_flag);
                w_ok = __all_sync(0xffffffffu, w_ok);
                if (!w_ok) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float f0 = sx * s0;
                const float f1 = sx * s1;
                const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + buf * kAccCols;
#pragma unroll
                for (int c = 0; c < kChunk; c += kLdCols) {
                    float v[kLdCols], u[kLdCols];
                    tmem_ld_nowait(tb + c0 + c, v);
                    tmem_ld_nowait(tb + c1 + c, u);
                    tmem_wait_ld(v, u);
#pragma unroll
                    for (int i = 0; i < kLdCols; i += 2) {
                        ffma2(acc0[c + i], acc0[c + i + 1], v[i], v[i + 1], f0);
                        ffma2(acc1[c + i], acc1[c + i + 1], u[i], u[i + 1], f1);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive_remote(cluster_map(&sm.tempty[buf], 0));
                if (++buf == 2) {
                    buf = 0;
                    bph ^= 1;
                }
            }
            if (!ok)
                break;
            const PairTile ctl = tl;
            const bool cstore = store;
            const int cpos = pos;
            if (STAGE == 1 && !next_tile()) {
                ok = false;
                t = -1;
            }
            ++gen;
            if (STAGE == 1) {
                // h for columns ncol0 + sub*kChunk + i; one 1x128 group spans the quadrant's kSubs
                // warps, which exchange their row amax through shared memory and a bounded mbarrier
                // wait.  The slot alternates with the tile: a warp can be at most one tile ahead.
                float amax = 0.0f;
#pragma unroll
                for (int i = 0; i < kChunk; ++i) {
                    acc0[i] = silu(acc0[i]) * acc1[i];
                    amax = fmaxf(amax, fabsf(acc0[i]));
                }
                sm.amax[gen & 1][sub][row] = amax;
                mbar_arrive(&sm.ep_bar[q]);
                bool x_ok = mbar_wait(&sm.ep_bar[q], (uint32_t)(gen - 1) & 1u, a.status, abort_flag);
                x_ok = __all_sync(0xffffffffu, x_ok);
                if (!x_ok)
                    break;
#pragma unroll
                for (int s2 = 0; s2 < kSubs; ++s2)
                    amax = fmaxf(amax, sm.amax[gen & 1][s2][row]);
                const float sc = amax > 0.0f ? amax / 448.0f : 1.0f;
                const float isc = 1.0f / sc;
                // 64 code bytes per row through the warp's shared block, so that each store writes
                // 8 rows x 64 contiguous bytes
                float4(*ep_rows)[4] = sm.ep_out[warp - 2];
#pragma unroll
                for (int v = 0; v < kChunk / 16; ++v) {
                    uint32_t w[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float *e = &acc0[v * 16 + j * 4];
                        const uint32_t lo =
                            __nv_cvt_float2_to_fp8x2(make_float2(e[0] * isc, e[1] * isc), __NV_SATFINITE, __NV_E4M3);
                        const uint32_t hi =
                            __nv_cvt_float2_to_fp8x2(make_float2(e[2] * isc, e[3] * isc), __NV_SATFINITE, __NV_E4M3);
                        w[j] = lo | (hi << 16);
                    }
                    ep_rows[lane][v ^ ((lane >> 1) & 3)] = make_float4(__uint_as_float(w[0]), __uint_as_float(w[1]),
                                                                   __uint_as_float(w[2]), __uint_as_float(w[3]));
                }
                __syncwarp();
                if (cstore) {
                    const int rr = lane >> 2, cq = lane & 3;
                    const int row0 = cpos - lane;  // sorted row of the warp's lane 0
#pragma unroll
                    for (int it = 0; it < 4; ++it) {
                        const int r = 8 * it + rr;
                        const float4 o = ep_rows[r][cq ^ ((r >> 1) & 3)];
                        *reinterpret_cast<float4 *>(static_cast<uint8_t *>(a.inter) + (size_t)(row0 + r) * a.N +
                                                    ctl.ncol0 + sub * kChunk + 16 * cq) = o;
                    }
                    if (sub == 0)
                        a.inter_scales[(size_t)(ctl.ncol0 / 128) * a.P_max + cpos] = sc;
                }
                __syncwarp();
            } else {
                // rows of y, 32 bf16 columns at a time, through a per-warp shared buffer (16-byte
                // slot j of row r at j ^ ((r >> 1) & 3)), leaving as 8 rows x 64 contiguous bytes
                // per store
                const int slot = cstore ? a.sorted_ids[cpos] : a.S;
                const float wgt = slot < a.S ? a.sorted_weights[cpos] : 0.0f;
                const int n0 = ctl.ncol0 + sub * 2 * kChunk;
                float4(*ep_rows)[4] = sm.ep_out[warp - 2];
                const int rr = lane >> 2, cq = lane & 3;
                if (cstore && n0 < a.N) {
#pragma unroll
                    for (int blk = 0; blk < 2 * kChunk / 32; ++blk) {
                        const float *v = blk < kChunk / 32 ? &acc0[blk * 32] : &acc1[blk * 32 - kChunk];
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            ep_rows[lane][j ^ ((lane >> 1) & 3)] = pack_bf16x8(v + 8 * j, wgt);
                        __syncwarp();
#pragma unroll
                        for (int it = 0; it < 4; ++it) {
                            const int r = 8 * it + rr;
                            const int rslot = __shfl_sync(0xffffffffu, slot, r);
                            const float4 o = ep_rows[r][cq ^ ((r >> 1) & 3)];
                            if (rslot < a.S)
                                *reinterpret_cast<float4 *>(a.y + (size_t)rslot * a.N + n0 + blk * 32 + 8 * cq) = o;
                        }
                        __syncwarp();
                    }
                }
                if (!next_tile())
                    t = -1;
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

template <int STAGE>
cudaError_t launch(const GemmArgs &a, int clusters, cudaStream_t st)
{
    auto kern = gemm_fp8_pair_kernel<STAGE>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (err != cudaSuccess)
        return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_site(a.pdl_mask, STAGE == 1 ? kPdlStage1 : kPdlStage2) ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

// Clusters of two that can be resident at once (one CTA per SM), cached per device.
template <int STAGE>
int max_clusters()
{
    static std::atomic<int> cache[64];  // per device, zero until first computed
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 0;
    if (cache[dev].load(std::memory_order_relaxed) == 0) {
        auto kern = gemm_fp8_pair_kernel<STAGE>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) != cudaSuccess)
            return 0;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kSmemBytes;
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

}  // namespace fp8pair

bool gemm_pair_fp8_supported(int E) { return E <= fp8pair::kMaxE; }

cudaError_t launch_gemm_pair_fp8(int stage, const GemmArgs &a, int64_t max_pair_tiles, cudaStream_t st)
{
    if (stage != 1 && stage != 2)
        return cudaErrorInvalidValue;
    int ncl = stage == 1 ? fp8pair::max_clusters<1>() : fp8pair::max_clusters<2>();
    if (ncl <= 0)
        return cudaErrorInvalidConfiguration;
    if (max_pair_tiles < ncl)
        ncl = (int)(max_pair_tiles > 0 ? max_pair_tiles : 1);
    return stage == 1 ? fp8pair::launch<1>(a, ncl, st) : fp8pair::launch<2>(a, ncl, st);
}

}  // namespace moe
