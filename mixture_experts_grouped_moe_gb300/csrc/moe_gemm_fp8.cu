// Block-scaled FP8 (e4m3) group GEMMs of the fused MoE layer ("per_1x128"
// quantisation of the AITER walk-through; two-stage path with the
// intermediate re-quantised between the stages, section 3.2).
//
// Scales are fp32 per 128x128 weight block and per 1x128 activation group,
// so they are not the power-of-two 32-element scales the tensor core applies
// in hardware.  Each 128-wide K block is therefore accumulated on its own
// by tcgen05.mma kind::f8f6f4 into one of two TMEM buffers, and eight
// promotion warps fold it into fp32 registers:
//     acc[row][col] += D_kb[row][col] * s_x[row][kb] * s_w[col_block][kb]
// while the tensor core fills the other buffer with the next K block.
// After the last K block the same warps run the epilogue from registers:
// stage 1 computes h = silu(gate) * up and re-quantises each 1x128 group of
// h (scale = amax / 448); stage 2 scales rows by their top-k weight.
//
// Warp roles: 0 TMA producer, 1 TMEM allocator + MMA issuer, 2..9
// promotion/epilogue: warp w reads TMEM lanes 32*(w%4)..+31 (its quadrant)
// and sub = (w-2)/4 picks half of the 256 accumulator columns, so two warps
// share each quadrant.  Tiles: M = 128 sorted token rows, N = 256 weight rows
// (stage 1: 128 gate + the matching 128 up rows; stage 2: 256 output
// features).  Each thread owns two 64-column chunks: stage 1 gate columns
// [64s, 64s+64) and up columns [128+64s, ...) so the SwiGLU pairs stay
// inside the thread; stage 2 columns [128s, 128s+128).
//
// Eight warps with 16-column TMEM loads measured faster than sixteen warps
// with 8-column loads (stage 1 of the Mixtral shapes at T=4096: 0.836 vs
// 0.889 ms): sixteen warps leave 96 registers a thread, too few for wider
// loads in flight next to 64 accumulators.
#include <cuda_fp8.h>

#include "gemm_common.cuh"
#include "moe_internal.h"
#include "sm100_ptx.cuh"

namespace moe {

namespace fp8gemm {

constexpr int kBK = 128;                    // one 128-wide K block (128 bytes) per stage
constexpr int kStages = 4;
constexpr int kWBytes = 256 * 128;          // 32 KiB
constexpr int kXBytes = 128 * 128;          // 16 KiB
constexpr int kStageBytes = kWBytes + kXBytes;
constexpr int kAccCols = 256;
constexpr int kTmemCols = 2 * kAccCols;
// Register budget: each SM sub-partition holds 16K registers and gets ceil(warps/4) of
// the CTA's warps, so 2 + 8 warps leave 168 registers a thread: 128 accumulators and two
// 16-column TMEM loads in flight (2 + 16 warps would leave 96).
constexpr int kPromoWarps = 8;
constexpr int kLdCols = 16;                 // TMEM columns per load, two loads per wait
constexpr int kSubs = kPromoWarps / 4;      // promotion warps per TMEM lane quadrant
constexpr int kChunk = 256 / (2 * kSubs);   // columns per chunk, two chunks per thread
constexpr int kThreads = 64 + 32 * kPromoWarps;
constexpr int kGroupM = 16;
static_assert(kChunk * 2 * kSubs == 256, "the quadrant's warps cover the 256 accumulator columns");
static_assert(kChunk == 64, "the epilogue stores move 64-byte (stage 1) and 16-column (stage 2) row pieces");

struct __align__(1024) Smem {
    uint8_t stage[kStages][kStageBytes];
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    TileQueue tq;
    uint32_t tmem_base;
    int abort;
    float amax[2][kSubs][128];  // per tile parity: row amax of each promotion warp's h chunk
    uint64_t ep_bar[4];         // per lane quadrant: one phase per tile once every warp wrote its amax
    float4 ep_out[kPromoWarps][32][4];  // a warp's 32 rows x 64 bytes on their way to global memory
};

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;

struct Tile {
    int e, xrow, wrow0, wrow1, ncol0;
};

template <int STAGE>
__device__ __forceinline__ Tile get_tile(const GemmArgs &a, int t, int nmb, int nnt)
{
    const int group = t / (kGroupM * nnt);
    const int within = t - group * kGroupM * nnt;
    const int gsize = min(kGroupM, nmb - group * kGroupM);
    const int nt = within / gsize;
    const int mb = group * kGroupM + within % gsize;
    Tile tl;
    tl.e = a.sorted_expert_ids[mb];
    tl.xrow = mb * 128;
    if (STAGE == 1) {
        tl.wrow0 = tl.e * a.rows_per_expert + nt * 128;
        tl.wrow1 = tl.e * a.rows_per_expert + a.N + nt * 128;
        tl.ncol0 = nt * 128;
    } else {
        tl.wrow0 = tl.e * a.rows_per_expert + nt * 256;
        tl.wrow1 = tl.wrow0 + 128;
        tl.ncol0 = nt * 256;
    }
    return tl;
}

template <int STAGE>
__global__ void __launch_bounds__(kThreads, 1) gemm_fp8_kernel(const __grid_constant__ GemmArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int *abort_flag = &sm.abort;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.tfull[i], 1);
            mbar_init(&sm.tempty[i], kPromoWarps);
        }
        mbar_init(&sm.drain, 1);
        tq_init(sm.tq, 1 + kPromoWarps);
        sm.abort = 0;
        for (int i = 0; i < 4; ++i)
            mbar_init(&sm.ep_bar[i], 32 * kSubs);
        fence_mbarrier_init();
        tma_prefetch_desc(&a.tm_x);
        tma_prefetch_desc(&a.tm_w);
    }
    if (warp == 1) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = sm.tmem_base;
    // everything above is independent of earlier kernels; from here on their outputs are read
    pdl_wait();
    pdl_trigger();
    const int nmb = *a.num_post_padded / 128;
    const int nnt = (STAGE == 1) ? a.N / 128 : (a.N + 255) / 256;
    const int ntiles = nmb * nnt;
    const int nkb = a.K / kBK;

    if (warp == 0) {
        if (lane == 0) {
            // weight tiles are reused by the 16 blocks of a raster group: evict-normal (evict-first
            // dropped some between uses, 1.41 -> 1.33 GB of DRAM reads per stage-1 launch;
            // evict-last measured 7 % slower per layer call)
            const uint64_t pol_w = l2_policy_evict_normal();
            const uint64_t pol_x = l2_policy_evict_last();
            int s = 0;
            uint32_t ph = 0;
            int issued[kStages];
            uint32_t issued_ph[kStages];
            for (int i = 0; i < kStages; ++i)
                issued[i] = 0, issued_ph[i] = 0;
            bool ok = true;
            int qs = 0;
            uint32_t qph = 0;
            int claim = -2;
            for (;;) {
                int t;
                if (!tq_push_next(sm.tq, qs, qph, a.tile_counter, ntiles, claim, t, a.status, abort_flag)) {
                    ok = false;
                    break;
                }
                if (t < 0)
                    break;
                const Tile tl = get_tile<STAGE>(a, t, nmb, nnt);
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(&sm.empty[s], ph ^ 1, a.status, abort_flag)) {
                        ok = false;
                        break;
                    }
                    uint8_t *wdst = sm.stage[s];
                    mbar_arrive_expect_tx(&sm.full[s], kStageBytes);
                    tma_load_2d(wdst, &a.tm_w, kb * kBK, tl.wrow0, &sm.full[s], pol_w);
                    tma_load_2d(wdst + kWBytes / 2, &a.tm_w, kb * kBK, tl.wrow1, &sm.full[s], pol_w);
                    tma_load_2d(wdst + kWBytes, &a.tm_x, kb * kBK, tl.xrow, &sm.full[s], pol_x);
                    issued[s] = 1;
                    issued_ph[s] = ph;
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1;
                    }
                }
                if (!ok)
                    break;
            }
            if (!ok) {
                for (int i = 0; i < kStages; ++i)
                    if (issued[i]) {
                        const unsigned long long t0 = global_timer_ns();
                        while (!mbar_try_wait(&sm.full[i], issued_ph[i]) && global_timer_ns() - t0 < 100000000ull) {
                        }
                    }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int buf = 0;
            uint32_t bph = 0;
            bool ok = true, any = false;
            const uint32_t idesc = make_idesc(0, 0, 128, 256);
            int qs = 0;
            uint32_t qph = 0;
            for (;;) {
                int t;
                if (!tq_pop(sm.tq, qs, qph, t, a.status, abort_flag)) {
                    ok = false;
                    break;
                }
                mbar_arrive(&sm.tq.empty[qs]);
                tq_advance(qs, qph);
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
                    const uint8_t *w = sm.stage[s];
                    const uint8_t *xs = sm.stage[s] + kWBytes;
#pragma unroll
                    for (int kk = 0; kk < kBK / 32; ++kk)
                        mma_fp8(d, smem_desc_sw128(xs + kk * 32), smem_desc_sw128(w + kk * 32), idesc,
                                kk > 0 ? 1u : 0u);
                    any = true;
                    mma_commit(&sm.empty[s]);
                    mma_commit(&sm.tfull[buf]);
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
                mma_commit(&sm.drain);
                const unsigned long long t0 = global_timer_ns();
                while (!mbar_try_wait(&sm.drain, 0) && global_timer_ns() - t0 < 100000000ull) {
                }
            }
        }
    } else {
        // ------------------------------------------- promotion + epilogue
        const int q = warp & 3;
        const int sub = (warp - 2) >> 2;       // 0 .. kSubs-1
        const int row = q * 32 + lane;
        const int c0 = (STAGE == 1) ? sub * kChunk : sub * 2 * kChunk;                // first chunk
        const int c1 = (STAGE == 1) ? 128 + sub * kChunk : sub * 2 * kChunk + kChunk;  // second chunk
        const int KB128 = a.K / 128;
        int buf = 0;
        uint32_t bph = 0;
        bool ok = true;
        int qs = 0;
        uint32_t qph = 0;
        const int nrb = a.E * a.rows_per_expert / 128;
        // Next tile and the first scales of its K loop.  The next tile is taken from the queue
        // right after the last K block of the current one, before its epilogue, so the
        // dependent global loads (expert id, then scales) overlap the epilogue.
        int t = -1;
        Tile tl{};
        int pos = 0;
        const float *sw0 = nullptr, *sw1 = nullptr;
        float sx_n = 0.0f, s0_n = 0.0f, s1_n = 0.0f;
        auto next_tile = [&]() -> bool {
            bool qok = tq_pop(sm.tq, qs, qph, t, a.status, abort_flag);
            qok = __all_sync(0xffffffffu, qok);
            if (!qok)
                return false;
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sm.tq.empty[qs]);
            tq_advance(qs, qph);
            if (t >= 0) {
                tl = get_tile<STAGE>(a, t, nmb, nnt);
                pos = tl.xrow + row;
                // weight-scale rows of this thread's two column chunks; a stage-2 chunk past the
                // last output feature (H % 256 == 128) reads a valid row and is never stored
                int rb0 = (STAGE == 1 ? tl.wrow0 : tl.wrow0 + sub * 2 * kChunk) / 128;
                int rb1 = (STAGE == 1 ? tl.wrow1 : tl.wrow0 + sub * 2 * kChunk) / 128;
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
            // the scales of block kb+1 are fetched while block kb is still on the tensor core
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
                // two TMEM loads in flight per wait: the promotion latency of a K block is what
                // paces the tensor core (it may refill this buffer only after the arrive below)
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
                    mbar_arrive(&sm.tempty[buf]);
                if (++buf == 2) {
                    buf = 0;
                    bph ^= 1;
                }
            }
            if (!ok)
                break;
            const Tile ctl = tl;
            const int cpos = pos;
            // stage 1 takes the next tile now, so that its expert id and first scales load during
            // the long SwiGLU epilogue; stage 2 (short epilogue) takes it afterwards
            if (STAGE == 1 && !next_tile()) {
                ok = false;
                t = -1;
            }
            ++gen;
            if (STAGE == 1) {
                // h for columns ncol0 + sub*kChunk + i; one 1x128 group spans the quadrant's
                // kSubs warps, which exchange their row amax through shared memory and a bounded
                // mbarrier wait (a named barrier would hang a warp whose partner left on an
                // abort).  The slot alternates with the tile: a warp can be at most one tile
                // ahead of its partners.
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
                // codes = RNE(h * (1/sc)) two at a time; the product can differ from h / sc in the
                // last fp32 bit, which moves a code only for a quotient within that bit of an e4m3
                // rounding midpoint
                const float isc = 1.0f / sc;
                // 64 code bytes per row: through the warp's shared block (same swizzle as stage 2)
                // so that each store writes 8 rows x 64 contiguous bytes instead of 32 rows
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
                {
                    const int rr = lane >> 2, cq = lane & 3;
                    const int row0 = ctl.xrow + q * 32;  // sorted row of the warp's lane 0
#pragma unroll
                    for (int it = 0; it < 4; ++it) {
                        const int r = 8 * it + rr;
                        const float4 o = ep_rows[r][cq ^ ((r >> 1) & 3)];
                        *reinterpret_cast<float4 *>(static_cast<uint8_t *>(a.inter) + (size_t)(row0 + r) * a.N +
                                                    ctl.ncol0 + sub * kChunk + 16 * cq) = o;
                    }
                }
                __syncwarp();
                if (sub == 0)
                    a.inter_scales[(size_t)(ctl.ncol0 / 128) * a.P_max + cpos] = sc;
            } else {
                // Each lane holds one row; stored straight from registers, every store instruction
                // would touch 32 rows of y (32 cache lines).  Blocks of 32 columns (64 bytes of bf16)
                // go through a per-warp shared buffer instead (16-byte slot j of row r at
                // j ^ ((r >> 1) & 3), free of bank conflicts both ways) and leave as 8 rows x 64
                // contiguous bytes.
                const int slot = a.sorted_ids[cpos];
                const float wgt = slot < a.S ? a.sorted_weights[cpos] : 0.0f;
                const int n0 = ctl.ncol0 + sub * 2 * kChunk;
                float4(*ep_rows)[4] = sm.ep_out[warp - 2];
                const int rr = lane >> 2, cq = lane & 3;  // read side: row within 8, float4 column
                if (n0 < a.N) {
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

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        tmem_dealloc(tmem_base, kTmemCols);
}

template <int STAGE>
cudaError_t launch(const GemmArgs &a, int grid, cudaStream_t st)
{
    auto kern = gemm_fp8_kernel<STAGE>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (err != cudaSuccess)
        return err;
    return launch_kernel(pdl_site(a.pdl_mask, STAGE == 1 ? kPdlStage1 : kPdlStage2), kern, dim3(grid),
                         dim3(kThreads), kSmemBytes, st, a);
}

}  // namespace fp8gemm

cudaError_t launch_gemm_grouped_fp8(int stage, const GemmArgs &a, int grid, cudaStream_t st)
{
    return stage == 1 ? fp8gemm::launch<1>(a, grid, st) : fp8gemm::launch<2>(a, grid, st);
}

}  // namespace moe
