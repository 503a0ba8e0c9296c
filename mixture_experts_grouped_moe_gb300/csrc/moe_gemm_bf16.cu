// Stage-1 and stage-2 group GEMMs of the fused MoE layer on the sm_100-family
// tensor core (tcgen05) fed by TMA, fp32 accumulation in tensor memory, for
// two input types:
//   QT = 0  bf16 activations and weights (kind::f16)
//   QT = 1  e4m3 activations and weights with one fp32 scale per row of each
//           ("per_Token" on the AITER page: a scale per token, a scale per
//           output channel).  Both scales are constant along K, so the whole
//           K sum runs in the tensor core (kind::f8f6f4) and the epilogue
//           multiplies accumulator element (token, channel) by
//           s_token * s_channel -- no per-K-block promotion.
// Every pipeline stage carries 128 bytes of K per row either way (64 bf16 or
// 128 e4m3 elements), so the tiles, the 128-byte swizzle and the descriptor
// steps (32 bytes per MMA: K = 16 bf16 or 32 e4m3) are shared.
//
// The two stages are the "2-stage" path of the AITER walk-through
// (section 3.2: stage 1 = gate/up projection + activation, stage 2 = down
// projection) run as group GEMMs over the blocks produced by the token sort
// (section 3.1), as in the Mixtral group-GEMM talk (group GEMMs in place of
// masked dense GEMMs; SwiGLU).  Each block of sorted rows belongs to one
// expert, so a tile is a dense GEMM against that expert's weights.
//
// Design (one CTA per SM, persistent, warp-specialised):
//   warp 0      TMA producer: weight tile (256 rows x 64 K) and token tile
//               (up to 128 rows x 64 K) per pipeline stage, 128-byte swizzle
//   warp 1      TMEM allocator and MMA issuer (one thread); tcgen05.commit
//               frees a stage when its MMAs finish, and signals a finished
//               accumulator to the epilogue
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (warp w reads TMEM
//               lanes 32*(w%4)..+31), fused SwiGLU (stage 1) or top-k weight
//               scaling (stage 2), stores to global memory
// Two 256-column fp32 accumulators in TMEM let the epilogue of one tile
// overlap the main loop of the next.
//
// Two tile shapes:
//   grouped (large T): M = 128 sorted token rows, N = 256 weight rows.
//     Stage 1's 256 weight rows are 128 gate rows and the matching 128 up
//     rows, so accumulator columns j and 128+j pair up for SwiGLU inside one
//     thread.  Stage 2's are 256 rows of W_down (256 output features).
//   swap (small T, decode): the weights take the MMA's M side.  A tile is
//     one expert's whole padded token segment (N = 16..128 tokens) against
//     256 weight rows issued as two M = 128 MMAs (stage 1: gate rows and the
//     matching up rows; stage 2: two halves of 256 output features), so
//     every weight byte of an active expert is streamed exactly once.
//     Stage 2 may split K (= I) across CTAs; the partial sums then go to a
//     workspace and a separate pass reduces them in a fixed order.
#include "gemm_common.cuh"
#include "moe_internal.h"
#include "sm100_ptx.cuh"

namespace moe {

namespace bf16gemm {

constexpr int kStages = 4;
constexpr int kWRows = 256;
constexpr int kXRows = 128;
constexpr int kWBytes = kWRows * 128;       // 32 KiB
constexpr int kXBytes = kXRows * 128;       // 16 KiB
constexpr int kStageBytes = kWBytes + kXBytes;
constexpr int kAccCols = 256;
constexpr int kTmemCols = 2 * kAccCols;
constexpr int kThreads = 192;
constexpr int kGroupM = 16;                 // raster: 16 M-blocks share each weight tile in turn

struct __align__(1024) Smem {
    uint8_t stage[kStages][kStageBytes];    // [W tile | X tile] per stage, 1024-byte aligned
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    TileQueue tq;
    uint32_t tmem_base;
    int abort;
};

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
constexpr int kEpiWarps = 4;

struct Tile {
    int valid;
    int e;          // expert
    int xrow;       // first token row (sorted position)
    int nx;         // token rows (grouped: 128; swap: padded segment length)
    int wrow0;      // first weight row of W-tile half 0
    int wrow1;      // first weight row of W-tile half 1
    int ncol0;      // output column base (stage 1: h column; stage 2: output feature)
    int kb0, kb1;   // K-block range
    int ks;         // K split index (swap stage 2)
};

// Internal tile shape of the weight-gradient GEMMs (STAGE 5): per expert e,
// D[e] (M x N) = A_e B_e^T with K running over e's sorted token positions;
// A and B are row arrays whose K dimension is the position (transposed
// activations), tiles 128 rows of A x 256 rows of B.  With no
// expert_offsets the a.E "segments" are equal slices of K instead (the
// router's tensor-core logits: D[s] = partial x W_router^T over slice s).
constexpr int kModeSegment = 2;

template <int MODE, int STAGE>
__device__ __forceinline__ int num_tiles(const GemmArgs &a)
{
    if (MODE == kModeSegment)
        return a.E * (a.M / 128) * ((a.N + 255) / 256);
    if (MODE == MOE_MODE_GROUPED) {
        const int nmb = *a.num_post_padded / 128;
        const int nnt = (STAGE == 1) ? a.N / 128 : (a.N + 255) / 256;
        return nmb * nnt;
    } else {
        const int nact = *a.num_active;
        const int nwt = (STAGE == 1) ? a.N / 128 : (a.N + 255) / 256;
        return nact * nwt * a.split_k;
    }
}

template <int MODE, int STAGE, int QT>
__device__ __forceinline__ Tile get_tile(const GemmArgs &a, int t)
{
    Tile tl;
    tl.valid = 1;
    const int nkb = a.K / kBK<QT>;
    if (MODE == kModeSegment) {
        const int nmt = a.M / 128, nnt = (a.N + 255) / 256;
        tl.e = t / (nmt * nnt);
        const int rem = t - tl.e * nmt * nnt;
        const int nt = rem / nmt, mt = rem % nmt;
        tl.xrow = mt * 128;            // A rows (output rows)
        tl.nx = 128;
        tl.wrow0 = nt * 256;           // B rows (output columns)
        tl.wrow1 = tl.wrow0 + 128;
        tl.ncol0 = nt * 256;
        if (a.expert_offsets) {
            tl.kb0 = a.expert_offsets[tl.e] / kBK<QT>;   // segments are whole 128-row blocks
            tl.kb1 = a.expert_offsets[tl.e + 1] / kBK<QT>;
        } else {
            // dense: K = a.K split evenly over the a.E "segments" (the router's logits)
            const int per = nkb / a.E;
            tl.kb0 = tl.e * per;
            tl.kb1 = tl.kb0 + per;
        }
        tl.ks = 0;
        return tl;
    }
    if (MODE == MOE_MODE_GROUPED) {
        const int nmb = *a.num_post_padded / 128;
        const int nnt = (STAGE == 1) ? a.N / 128 : (a.N + 255) / 256;
        const int group = t / (kGroupM * nnt);
        const int within = t - group * kGroupM * nnt;
        const int gsize = min(kGroupM, nmb - group * kGroupM);
        const int nt = within / gsize;
        const int mb = group * kGroupM + within % gsize;
        tl.e = a.sorted_expert_ids[mb];
        tl.xrow = mb * 128;
        tl.nx = 128;
        if (STAGE == 1) {
            tl.wrow0 = tl.e * a.rows_per_expert + nt * 128;          // gate rows
            tl.wrow1 = tl.e * a.rows_per_expert + a.N + nt * 128;    // matching up rows
            tl.ncol0 = nt * 128;
        } else {
            tl.wrow0 = tl.e * a.rows_per_expert + nt * 256;
            tl.wrow1 = tl.wrow0 + 128;
            tl.ncol0 = nt * 256;
        }
        tl.kb0 = 0;
        tl.kb1 = nkb;
        tl.ks = 0;
    } else {
        const int nact = *a.num_active;
        const int nwt = (STAGE == 1) ? a.N / 128 : (a.N + 255) / 256;
        const int ai = t % nact;
        const int r = t / nact;
        const int wt = r % nwt;
        const int ks = r / nwt;
        tl.e = a.active_experts[ai];
        tl.xrow = a.expert_offsets[tl.e];
        tl.nx = a.expert_offsets[tl.e + 1] - tl.xrow;
        if (STAGE == 1) {
            tl.wrow0 = tl.e * a.rows_per_expert + wt * 128;
            tl.wrow1 = tl.e * a.rows_per_expert + a.N + wt * 128;
            tl.ncol0 = wt * 128;
        } else {
            tl.wrow0 = tl.e * a.rows_per_expert + wt * 256;
            tl.wrow1 = tl.wrow0 + 128;
            tl.ncol0 = wt * 256;
        }
        const int per = nkb / a.split_k;
        tl.kb0 = ks * per;
        tl.kb1 = tl.kb0 + per;
        tl.ks = ks;
    }
    return tl;
}

template <int MODE, int STAGE, int QT>
__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const __grid_constant__ GemmArgs a)
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
            mbar_init(&sm.tempty[i], 4);
        }
        mbar_init(&sm.drain, 1);
        tq_init(sm.tq, 1 + kEpiWarps);
        sm.abort = 0;
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
    const int ntiles = num_tiles<MODE, STAGE>(a);

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer
        if (lane == 0) {
            // grouped mode reuses a weight tile across a raster group of blocks: evict-normal;
            // swap mode reads every weight byte once: evict-first
            const uint64_t pol_w = MODE == MOE_MODE_GROUPED ? l2_policy_evict_normal() : l2_policy_evict_first();
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
                const Tile tl = get_tile<MODE, STAGE, QT>(a, t);
                const uint32_t bytes = kWBytes + tl.nx * 128;
                for (int kb = tl.kb0; kb < tl.kb1; ++kb) {
                    if (!mbar_wait(&sm.empty[s], ph ^ 1, a.status, abort_flag)) {
                        ok = false;
                        break;
                    }
                    uint8_t *wdst = sm.stage[s];
                    uint8_t *xdst = sm.stage[s] + kWBytes;
                    mbar_arrive_expect_tx(&sm.full[s], bytes);
                    tma_load_2d(wdst, &a.tm_w, kb * kBK<QT>, tl.wrow0, &sm.full[s], pol_w);
                    tma_load_2d(wdst + kWBytes / 2, &a.tm_w, kb * kBK<QT>, tl.wrow1, &sm.full[s], pol_w);
                    if (MODE != MOE_MODE_SWAP) {
                        tma_load_2d(xdst, &a.tm_x, kb * kBK<QT>, tl.xrow, &sm.full[s], pol_x);
                    } else {
                        for (int c = 0; c < tl.nx; c += 16)
                            tma_load_2d(xdst + c * 128, &a.tm_x, kb * kBK<QT>, tl.xrow + c, &sm.full[s], pol_x);
                    }
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
                // let the copies already in flight land before the CTA exits
                for (int i = 0; i < kStages; ++i)
                    if (issued[i]) {
                        const unsigned long long t0 = global_timer_ns();
                        while (!mbar_try_wait(&sm.full[i], issued_ph[i]) && global_timer_ns() - t0 < 100000000ull) {
                        }
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
            bool ok = true;
            bool any = false;
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
                const Tile tl = get_tile<MODE, STAGE, QT>(a, t);
                if (!mbar_wait(&sm.tempty[acc], aph ^ 1, a.status, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + acc * kAccCols;
                constexpr uint32_t kFmt = QT ? 0u : 1u;  // e4m3 (kind::f8f6f4) or bf16 (kind::f16)
                const uint32_t idesc = (MODE != MOE_MODE_SWAP) ? make_idesc(kFmt, kFmt, 128, 256)
                                                               : make_idesc(kFmt, kFmt, 128, (uint32_t)tl.nx);
                for (int kb = tl.kb0; kb < tl.kb1; ++kb) {
                    if (!mbar_wait(&sm.full[s], ph, a.status, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint8_t *w = sm.stage[s];
                    const uint8_t *xs = sm.stage[s] + kWBytes;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {  // 4 MMAs of 32 bytes of K each
                        const uint32_t accum = (kb > tl.kb0 || kk > 0) ? 1u : 0u;
                        if (MODE != MOE_MODE_SWAP) {
                            mma_kind<QT>(d, smem_desc_sw128(xs + kk * 32), smem_desc_sw128(w + kk * 32), idesc,
                                         accum);
                        } else {
                            mma_kind<QT>(d, smem_desc_sw128(w + kk * 32), smem_desc_sw128(xs + kk * 32), idesc,
                                         accum);
                            mma_kind<QT>(d + 128, smem_desc_sw128(w + kWBytes / 2 + kk * 32),
                                         smem_desc_sw128(xs + kk * 32), idesc, accum);
                        }
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
                // drain: wait (bounded) until every MMA issued so far has finished
                mma_commit(&sm.drain);
                const unsigned long long t0 = global_timer_ns();
                while (!mbar_try_wait(&sm.drain, 0) && global_timer_ns() - t0 < 100000000ull) {
                }
            }
        }
    } else {
        // -------------------------------------------------------- epilogue
        const int q = warp & 3;           // TMEM lane quadrant of this warp
        const int row = q * 32 + lane;    // accumulator row (TMEM lane)
        int acc = 0;
        uint32_t aph = 0;
        int qs = 0;
        uint32_t qph = 0;
        for (;;) {
            int t = -1;
            bool qok = tq_pop(sm.tq, qs, qph, t, a.status, abort_flag);
            qok = __all_sync(0xffffffffu, qok);
            if (!qok)
                break;
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sm.tq.empty[qs]);
            tq_advance(qs, qph);
            if (t < 0)
                break;
            const Tile tl = get_tile<MODE, STAGE, QT>(a, t);
            bool ok = mbar_wait(&sm.tfull[acc], aph, a.status, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok)
                break;
            tc_fence_after();
            const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16) + acc * kAccCols;

            if (MODE == MOE_MODE_GROUPED && STAGE == 1) {
                // row = sorted position; columns j (gate) and 128+j (up) of h column ncol0+j
                __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.inter) + (size_t)(tl.xrow + row) * a.N + tl.ncol0;
                const float sx = QT ? a.x_scales[tl.xrow + row] : 1.0f;
                float hmax = 0.0f;  // per-token FP8: max |h| of the row's 128 columns here
#pragma unroll 1
                for (int c0 = 0; c0 < 128; c0 += 32) {
                    float g[32], u[32], h[32];
                    tmem_ld32(tacc + c0, g);
                    tmem_ld32(tacc + 128 + c0, u);
                    if (QT) {
#pragma unroll
                        for (int i = 0; i < 32; i += 4) {
                            const float4 sg = ld_scale4(a.w_scales + tl.wrow0 + c0 + i);
                            const float4 su = ld_scale4(a.w_scales + tl.wrow1 + c0 + i);
                            g[i] *= sx * sg.x, g[i + 1] *= sx * sg.y, g[i + 2] *= sx * sg.z, g[i + 3] *= sx * sg.w;
                            u[i] *= sx * su.x, u[i + 1] *= sx * su.y, u[i + 2] *= sx * su.z, u[i + 3] *= sx * su.w;
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        h[i] = silu(g[i]) * u[i];
                    if (QT)
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            hmax = fmaxf(hmax, fabsf(h[i]));
                    store_bf16x32(dst + c0, h);
                    if (a.gu) {  // training: keep the pre-activations for the backward
                        __nv_bfloat16 *gr = a.gu + (size_t)(tl.xrow + row) * (2 * a.N) + tl.ncol0 + c0;
                        store_bf16x32(gr, g);
                        store_bf16x32(gr + a.N, u);
                    }
                }
                // the row's max |h| as the quantiser will see it (bf16 rounding is monotonic, so the
                // rounded maximum is the maximum of the rounded values); non-negative floats order
                // as their bits
                if (QT && a.row_amax)
                    atomicMax(reinterpret_cast<int *>(a.row_amax) + tl.xrow + row,
                              __float_as_int(__bfloat162float(__float2bfloat16_rn(hmax))));
            } else if (MODE == MOE_MODE_GROUPED && STAGE == 3) {
                // backward of stage 2 (dh = dY W_down): SwiGLU's backward with the saved g | u,
                // dg = dh u silu'(g), du = dh silu(g), into dgu (g part at column c, u part at I + c)
                const size_t p = (size_t)(tl.xrow + row);
                const __nv_bfloat16 *gr = a.gu_in + p * (2 * a.N) + tl.ncol0;
                __nv_bfloat16 *dr = a.dgu + p * (2 * a.N) + tl.ncol0;
#pragma unroll 1
                for (int c0 = 0; c0 < 256; c0 += 32) {
                    float dh[32], dg[32], du[32];
                    tmem_ld32(tacc + c0, dh);
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
            } else if (MODE == kModeSegment) {
                // weight gradient: output row tl.xrow + row of expert e, columns ncol0 .. +256
                float *dst = a.dw_out + ((size_t)tl.e * a.M + tl.xrow + row) * a.N + tl.ncol0;
                const int ncols = min(256, a.N - tl.ncol0);
                const bool empty = tl.kb0 == tl.kb1;  // an expert without tokens: zero gradient
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
            } else if (MODE == MOE_MODE_GROUPED && STAGE == 2) {
                const int pos = tl.xrow + row;
                const int slot = a.sorted_ids[pos];
                // no weights: the unweighted rows (the backward's dx per slot)
                const float wgt = (a.sorted_weights ? a.sorted_weights[pos] : 1.0f) * (QT ? a.x_scales[pos] : 1.0f);
                const bool live = slot < a.S;
                __nv_bfloat16 *dst = a.y + (size_t)(live ? slot : 0) * a.N + tl.ncol0;
                const int ncols = min(256, a.N - tl.ncol0);
#pragma unroll 1
                for (int c0 = 0; c0 < ncols; c0 += 32) {
                    float v[32];
                    tmem_ld32(tacc + c0, v);
                    if (QT) {
#pragma unroll
                        for (int i = 0; i < 32; i += 4) {
                            const float4 sw = ld_scale4(a.w_scales + tl.wrow0 + c0 + i);
                            v[i] *= sw.x, v[i + 1] *= sw.y, v[i + 2] *= sw.z, v[i + 3] *= sw.w;
                        }
                    }
                    if (live) {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            v[i] *= wgt;
                        store_bf16x32(dst + c0, v);
                    }
                }
            } else if (MODE == MOE_MODE_SWAP && STAGE == 1) {
                // row = h column within the 128-wide tile; TMEM columns = tokens of the segment
                __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.inter) + (size_t)tl.xrow * a.N + tl.ncol0 + row;
                const float swg = QT ? a.w_scales[tl.wrow0 + row] : 1.0f;
                const float swu = QT ? a.w_scales[tl.wrow1 + row] : 1.0f;
#pragma unroll 1
                for (int c0 = 0; c0 < tl.nx; c0 += 16) {
                    float g[16], u[16];
                    tmem_ld16(tacc + c0, g);
                    tmem_ld16(tacc + 128 + c0, u);
                    if (QT) {
#pragma unroll
                        for (int j = 0; j < 16; j += 4) {
                            const float4 sx = ld_scale4(a.x_scales + tl.xrow + c0 + j);
                            g[j] *= swg * sx.x, g[j + 1] *= swg * sx.y, g[j + 2] *= swg * sx.z, g[j + 3] *= swg * sx.w;
                            u[j] *= swu * sx.x, u[j + 1] *= swu * sx.y, u[j + 2] *= swu * sx.z, u[j + 3] *= swu * sx.w;
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        dst[(size_t)(c0 + j) * a.N] = __float2bfloat16_rn(silu(g[j]) * u[j]);
                }
            } else {
                // swap, stage 2: rows = output features ncol0 + half*128 + row; columns = tokens
#pragma unroll 1
                for (int half = 0; half < 2; ++half) {
                    const int n = tl.ncol0 + half * 128 + row;
                    const bool nok = n < a.N;
                    const float sw = (QT && nok) ? a.w_scales[tl.wrow0 + half * 128 + row] : 1.0f;
#pragma unroll 1
                    for (int c0 = 0; c0 < tl.nx; c0 += 16) {
                        float v[16];
                        tmem_ld16(tacc + half * 128 + c0, v);
                        if (!nok)
                            continue;
                        if (QT) {
#pragma unroll
                            for (int j = 0; j < 16; j += 4) {
                                const float4 sx = ld_scale4(a.x_scales + tl.xrow + c0 + j);
                                v[j] *= sw * sx.x, v[j + 1] *= sw * sx.y, v[j + 2] *= sw * sx.z, v[j + 3] *= sw * sx.w;
                            }
                        }
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

template <int MODE, int STAGE, int QT>
cudaError_t launch(const GemmArgs &a, int grid, cudaStream_t st)
{
    auto kern = gemm_kernel<MODE, STAGE, QT>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (err != cudaSuccess)
        return err;
    return launch_kernel(pdl_site(a.pdl_mask, STAGE == 1 ? kPdlStage1 : kPdlStage2), kern,
                         dim3(grid), dim3(kThreads), kSmemBytes, st, a);
}

}  // namespace bf16gemm

cudaError_t launch_gemm_grouped_bf16(int stage, const GemmArgs &a, int grid, cudaStream_t st)
{
    return stage == 1 ? bf16gemm::launch<MOE_MODE_GROUPED, 1, 0>(a, grid, st)
                      : bf16gemm::launch<MOE_MODE_GROUPED, 2, 0>(a, grid, st);
}

cudaError_t launch_gemm_backward_bf16(int which, const GemmArgs &a, int grid, cudaStream_t st)
{
    // 3: backward of stage 2 with SwiGLU's backward; 2: backward of stage 1 (stage 2's
    // tile shape, unit weights); 5: weight gradients over token segments
    if (which == 3)
        return bf16gemm::launch<MOE_MODE_GROUPED, 3, 0>(a, grid, st);
    if (which == 5)
        return bf16gemm::launch<bf16gemm::kModeSegment, 5, 0>(a, grid, st);
    return bf16gemm::launch<MOE_MODE_GROUPED, 2, 0>(a, grid, st);
}

cudaError_t launch_gemm_swap_bf16(int stage, const GemmArgs &a, int grid, cudaStream_t st)
{
    return stage == 1 ? bf16gemm::launch<MOE_MODE_SWAP, 1, 0>(a, grid, st)
                      : bf16gemm::launch<MOE_MODE_SWAP, 2, 0>(a, grid, st);
}

cudaError_t launch_gemm_grouped_fp8_token(int stage, const GemmArgs &a, int grid, cudaStream_t st)
{
    return stage == 1 ? bf16gemm::launch<MOE_MODE_GROUPED, 1, 1>(a, grid, st)
                      : bf16gemm::launch<MOE_MODE_GROUPED, 2, 1>(a, grid, st);
}

cudaError_t launch_gemm_swap_fp8_token(int stage, const GemmArgs &a, int grid, cudaStream_t st)
{
    return stage == 1 ? bf16gemm::launch<MOE_MODE_SWAP, 1, 1>(a, grid, st)
                      : bf16gemm::launch<MOE_MODE_SWAP, 2, 1>(a, grid, st);
}

}  // namespace moe
