// One-kernel (1-stage) decode path: gate/up GEMM -> SwiGLU -> down GEMM in a
// single persistent launch (the "1-stage" execution of the AITER
// walk-through, section 3.2), bf16, swap-AB tiles as in the two-launch decode
// kernels.
//
// Tiles of both stages are claimed from one counter, stage-1 tiles first, so
// every stage-1 tile is owned by a running CTA before any stage-2 tile is
// handed out.  The intermediate h (16-64 token rows x I per expert, a few
// MB) stays on chip in L2 between the phases.  A stage-2 tile's weight loads
// do not depend on h and are issued at once; its first h load waits until
// the count of finished stage-1 epilogue warps reaches its target (a bounded
// wait on a global counter that the epilogues release after their stores),
// so W_down streams from HBM while the last stage-1 tiles finish.  Stage 2
// splits K = I as the two-launch path does; the fixed-order split reduce and
// top-k combine remain a separate pass.  No gather pass precedes the launch:
// the producer warp fetches each stage-1 tile's token rows from x itself.
#include "gemm_common.cuh"
#include "moe_internal.h"
#include "sm100_ptx.cuh"

namespace moe {

namespace fused {

constexpr int kStages = 4;
constexpr int kWRows = 256;
constexpr int kXRows = 128;
constexpr int kWBytes = kWRows * 128;
constexpr int kXBytes = kXRows * 128;
constexpr int kStageBytes = kWBytes + kXBytes;
constexpr int kAccCols = 256;
constexpr int kTmemCols = 2 * kAccCols;
constexpr int kThreads = 192;
constexpr int kEpiWarps = 4;

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
    int xtok[kXRows];  // stage-1 tile: token of each sorted row, -1 for padding
};

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;

struct Tile {
    int stage;      // 1 or 2
    int e, xrow, nx, wrow0, wrow1, ncol0, kb0, kb1, ks;
};

__device__ __forceinline__ int tiles_of(const GemmArgs &a, int stage)
{
    const int nwt = (stage == 1) ? a.N / 128 : (a.N + 255) / 256;
    return *a.num_active * nwt * a.split_k;
}

__device__ __forceinline__ Tile get_tile(const FusedArgs &F, int t, int n1)
{
    Tile tl;
    tl.stage = t < n1 ? 1 : 2;
    const GemmArgs &a = tl.stage == 1 ? F.s1 : F.s2;
    if (tl.stage == 2)
        t -= n1;
    const int nact = *a.num_active;
    const int nwt = (tl.stage == 1) ? a.N / 128 : (a.N + 255) / 256;
    const int ai = t % nact;
    const int r = t / nact;
    const int wt = r % nwt;
    const int ks = r / nwt;
    tl.e = a.active_experts[ai];
    tl.xrow = a.expert_offsets[tl.e];
    tl.nx = a.expert_offsets[tl.e + 1] - tl.xrow;
    if (tl.stage == 1) {
        tl.wrow0 = tl.e * a.rows_per_expert + wt * 128;
        tl.wrow1 = tl.e * a.rows_per_expert + a.N + wt * 128;
        tl.ncol0 = wt * 128;
    } else {
        tl.wrow0 = tl.e * a.rows_per_expert + wt * 256;
        tl.wrow1 = tl.wrow0 + 128;
        tl.ncol0 = wt * 256;
    }
    const int per = (a.K / 64) / a.split_k;
    tl.kb0 = ks * per;
    tl.kb1 = tl.kb0 + per;
    tl.ks = ks;
    return tl;
}

__device__ __forceinline__ int ld_acquire(const int *p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Wait (bounded by limit_ns) until *p >= target; false (status raised) on timeout or abort.
__device__ __forceinline__ bool wait_count(const int *p, int target, unsigned long long limit_ns, int *status,
                                           volatile int *abort)
{
    const unsigned long long t0 = global_timer_ns();
    for (uint32_t it = 0;; ++it) {
        if (ld_acquire(p) >= target)
            return true;
        __nanosleep(256);
        if ((it & 63u) == 63u) {
            if (*abort)
                return false;
            if (global_timer_ns() - t0 > limit_ns) {
                atomicExch(status, -5 /* MOE_ERR_TIMEOUT */);
                *abort = 1;
                return false;
            }
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1) fused_swap_kernel(const __grid_constant__ FusedArgs F)
{
    extern __shared__ uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int *abort_flag = &sm.abort;
    int *status = F.s1.status;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sm.full[i], 1 + 32);  // TMA bytes + the producer lanes' token-row copies
            mbar_init(&sm.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.tfull[i], 1);
            mbar_init(&sm.tempty[i], kEpiWarps);
        }
        mbar_init(&sm.drain, 1);
        tq_init(sm.tq, 1 + kEpiWarps);
        sm.abort = 0;
        fence_mbarrier_init();
        tma_prefetch_desc(&F.s1.tm_x);
        tma_prefetch_desc(&F.s1.tm_w);
        tma_prefetch_desc(&F.s2.tm_x);
        tma_prefetch_desc(&F.s2.tm_w);
    }
    if (warp == 1) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = sm.tmem_base;
    pdl_wait();
    pdl_trigger();
    const int n1 = tiles_of(F.s1, 1);
    const int ntiles = n1 + tiles_of(F.s2, 2);
    const int h_target = n1 * kEpiWarps + F.h_extra;  // epilogue warps of all stage-1 tiles

    if (warp == 0) {
        // ------------------------------------------------- producer (whole warp)
        // Lane 0 claims tiles and issues the weight loads (and stage 2's h rows) by TMA.  The
        // token rows of a stage-1 tile come straight from x: the 32 lanes copy them in 16-byte
        // pieces (cp.async) into the 128-byte-swizzled layout a TMA load would have produced
        // (16-byte chunk c of row r at chunk c ^ (r % 8)), zero-filled for padding rows, so no
        // gather pass runs before this kernel.  Each lane's copies complete on the stage
        // barrier (1 + 32 arrivals per phase).
        const uint64_t pol_w = l2_policy_evict_first();
        const uint64_t pol_x = l2_policy_evict_last();
        int s = 0;
        uint32_t ph = 0;
        int issued[kStages];
        uint32_t issued_ph[kStages];
        for (int i = 0; i < kStages; ++i)
            issued[i] = 0, issued_ph[i] = 0;
        bool ok = true, h_ready = false;
        int qs = 0;
        uint32_t qph = 0;
        int claim = -2;
        const int H = F.s1.K;
        for (;;) {
            int t = -1;
            bool qok = true;
            if (lane == 0)
                qok = tq_push_next(sm.tq, qs, qph, F.tile_counter, ntiles, claim, t, status, abort_flag);
            qok = __shfl_sync(0xffffffffu, (int)qok, 0) != 0;
            t = __shfl_sync(0xffffffffu, t, 0);
            if (!qok) {
                ok = false;
                break;
            }
            if (t < 0)
                break;
            const Tile tl = get_tile(F, t, n1);
            const GemmArgs &a = tl.stage == 1 ? F.s1 : F.s2;
            if (tl.stage == 1) {
                __syncwarp();  // the previous tile's copies have all been issued
                for (int r = lane; r < tl.nx; r += 32) {
                    const int slot = a.sorted_ids[tl.xrow + r];
                    sm.xtok[r] = slot < a.S ? slot / F.k : -1;
                }
                __syncwarp();
            }
            const uint32_t bytes = tl.stage == 1 ? kWBytes : kWBytes + tl.nx * 128;
            for (int kb = tl.kb0; kb < tl.kb1; ++kb) {
                bool w_ok = mbar_wait(&sm.empty[s], ph ^ 1, status, abort_flag);
                w_ok = __all_sync(0xffffffffu, w_ok);
                if (!w_ok) {
                    ok = false;
                    break;
                }
                uint8_t *wdst = sm.stage[s];
                uint8_t *xdst = sm.stage[s] + kWBytes;
                if (tl.stage == 1) {
                    for (int j = lane; j < tl.nx * 8; j += 32) {
                        const int r = j >> 3, c = j & 7;
                        const int tok = sm.xtok[r];
                        const __nv_bfloat16 *src = F.x + (size_t)(tok < 0 ? 0 : tok) * H + kb * 64 + c * 8;
                        cp_async_16_zfill(xdst + r * 128 + ((c ^ (r & 7)) << 4), src, tok >= 0);
                    }
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(&sm.full[s], bytes);
                    tma_load_2d(wdst, &a.tm_w, kb * 64, tl.wrow0, &sm.full[s], pol_w);
                    tma_load_2d(wdst + kWBytes / 2, &a.tm_w, kb * 64, tl.wrow1, &sm.full[s], pol_w);
                    issued[s] = 1;
                    issued_ph[s] = ph;
                }
                if (tl.stage == 2) {
                    if (!h_ready) {
                        // h is written by every stage-1 epilogue: wait for all of them once
                        bool h_ok = true;
                        if (lane == 0) {
                            h_ok = wait_count(F.h_done, h_target, F.h_wait_ns, status, abort_flag);
                            if (h_ok)
                                asm volatile("fence.proxy.async.global;" ::: "memory");
                        }
                        h_ok = __shfl_sync(0xffffffffu, (int)h_ok, 0) != 0;
                        if (!h_ok) {
                            // This stage's phase expects the h rows' bytes and the lanes' copy
                            // arrivals, which will not come now: retire both, so that the phase
                            // completes exactly when its weight copies have landed (the drain
                            // below waits for that before the CTA exits).
                            if (lane == 0)
                                mbar_complete_tx(&sm.full[s], (uint32_t)tl.nx * 128);
                            cp_async_arrive(&sm.full[s]);
                            ok = false;
                            break;
                        }
                        h_ready = true;
                    }
                    if (lane == 0)
                        for (int c = 0; c < tl.nx; c += 16)
                            tma_load_2d(xdst + c * 128, &a.tm_x, kb * 64, tl.xrow + c, &sm.full[s], pol_x);
                }
                cp_async_arrive(&sm.full[s]);
                if (++s == kStages) {
                    s = 0;
                    ph ^= 1;
                }
            }
            if (!ok)
                break;
        }
        cp_async_wait_all();
        if (!ok && lane == 0) {
            for (int i = 0; i < kStages; ++i)
                if (issued[i]) {
                    const unsigned long long t0 = global_timer_ns();
                    while (!mbar_try_wait(&sm.full[i], issued_ph[i]) && global_timer_ns() - t0 < 100000000ull) {
                    }
                }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int acc = 0;
            uint32_t aph = 0;
            bool ok = true, any = false;
            int qs = 0;
            uint32_t qph = 0;
            for (;;) {
                int t;
                if (!tq_pop(sm.tq, qs, qph, t, status, abort_flag)) {
                    ok = false;
                    break;
                }
                mbar_arrive(&sm.tq.empty[qs]);
                tq_advance(qs, qph);
                if (t < 0)
                    break;
                const Tile tl = get_tile(F, t, n1);
                if (!mbar_wait(&sm.tempty[acc], aph ^ 1, status, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + acc * kAccCols;
                const uint32_t idesc = make_idesc(1, 1, 128, (uint32_t)tl.nx);
                for (int kb = tl.kb0; kb < tl.kb1; ++kb) {
                    if (!mbar_wait(&sm.full[s], ph, status, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    fence_proxy_async_smem();  // the token-row copies (generic proxy) before the MMAs read them
                    const uint8_t *w = sm.stage[s];
                    const uint8_t *xs = sm.stage[s] + kWBytes;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t accum = (kb > tl.kb0 || kk > 0) ? 1u : 0u;
                        mma_bf16(d, smem_desc_sw128(w + kk * 32), smem_desc_sw128(xs + kk * 32), idesc, accum);
                        mma_bf16(d + 128, smem_desc_sw128(w + kWBytes / 2 + kk * 32), smem_desc_sw128(xs + kk * 32),
                                 idesc, accum);
                    }
                    any = true;
                    mma_commit(&sm.empty[s]);
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1;
                    }
                }
                if (!ok)
                    break;
                mma_commit(&sm.tfull[acc]);
                if (++acc == 2) {
                    acc = 0;
                    aph ^= 1;
                }
            }
            if (!ok && any) {
                mma_commit(&sm.drain);
                const unsigned long long t0 = global_timer_ns();
                while (!mbar_try_wait(&sm.drain, 0) && global_timer_ns() - t0 < 100000000ull) {
                }
            }
        }
    } else {
        // -------------------------------------------------------- epilogue
        const int q = warp & 3;
        const int row = q * 32 + lane;
        int acc = 0;
        uint32_t aph = 0;
        int qs = 0;
        uint32_t qph = 0;
        for (;;) {
            int t = -1;
            bool qok = tq_pop(sm.tq, qs, qph, t, status, abort_flag);
            qok = __all_sync(0xffffffffu, qok);
            if (!qok)
                break;
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sm.tq.empty[qs]);
            tq_advance(qs, qph);
            if (t < 0)
                break;
            const Tile tl = get_tile(F, t, n1);
            bool ok = mbar_wait(&sm.tfull[acc], aph, status, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok)
                break;
            tc_fence_after();
            const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16) + acc * kAccCols;
            if (tl.stage == 1) {
                const GemmArgs &a = F.s1;
                __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.inter) + (size_t)tl.xrow * a.N + tl.ncol0 + row;
#pragma unroll 1
                for (int c0 = 0; c0 < tl.nx; c0 += 16) {
                    float g[16], u[16];
                    tmem_ld16(tacc + c0, g);
                    tmem_ld16(tacc + 128 + c0, u);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        dst[(size_t)(c0 + j) * a.N] = __float2bfloat16_rn(silu(g[j]) * u[j]);
                }
                // publish this warp's part of h to the stage-2 loads (async proxy, other CTAs)
                asm volatile("fence.proxy.async.global;" ::: "memory");
                __threadfence();
                __syncwarp();
                if (lane == 0)
                    atomicAdd(F.h_done, 1);
            } else {
                const GemmArgs &a = F.s2;
#pragma unroll 1
                for (int half = 0; half < 2; ++half) {
                    const int n = tl.ncol0 + half * 128 + row;
                    const bool nok = n < a.N;
#pragma unroll 1
                    for (int c0 = 0; c0 < tl.nx; c0 += 16) {
                        float v[16];
                        tmem_ld16(tacc + half * 128 + c0, v);
                        if (!nok)
                            continue;
                        if (a.split_k > 1) {
                            float *dst = a.partials + ((size_t)tl.ks * a.P_max + tl.xrow + c0) * a.N + n;
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                dst[(size_t)j * a.N] = v[j];
                        } else {
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                const int pos = tl.xrow + c0 + j;
                                const int slot = a.sorted_ids[pos];
                                if (slot < a.S)
                                    a.y[(size_t)slot * a.N + n] = __float2bfloat16_rn(a.sorted_weights[pos] * v[j]);
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sm.tempty[acc]);
            if (++acc == 2) {
                acc = 0;
                aph ^= 1;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        tmem_dealloc(tmem_base, kTmemCols);
}

}  // namespace fused

cudaError_t launch_fused_decode(const FusedArgs &F, int grid, cudaStream_t st)
{
    auto kern = fused::fused_swap_kernel;
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fused::kSmemBytes);
    if (err != cudaSuccess)
        return err;
    return launch_kernel(pdl_site(F.s1.pdl_mask, kPdlStage1), kern, dim3(grid), dim3(fused::kThreads), fused::kSmemBytes,
                         st, F);
}

}  // namespace moe
