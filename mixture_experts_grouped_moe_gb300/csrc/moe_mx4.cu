// MXFP4 ("per_1x32" on the AITER walk-through, section 3.2's quantisation
// types): E2M1 elements with one power-of-two E8M0 scale per 32 consecutive
// elements of a row (OCP microscaling), and the decode-size group GEMMs that
// multiply them on the tensor core's block-scaled path (tcgen05
// kind::mxf4, scales in TMEM).
//
// Storage:
//   codes    two E2M1 codes per byte, element 2j in the low nibble of byte j
//            (code = sign << 3 | magnitude index, magnitudes 0 .5 1 1.5 2 3 4 6)
//   scales   E8M0 bytes (biased exponent, 2^(s - 127)), either row-major
//            [rows][C/32] (activations, the intermediate) or tiled for the
//            weights: [rows/128][C/128][512] with the 512 bytes of a
//            128-row x 4-group tile in the tensor core's blocked order
//            (byte (r % 32) * 16 + (r % 128 / 32) * 4 + g % 4).
// Quantisation (MX rule): e = floor(log2(amax of the 32)) - 2 (0 for an
// all-zero group), element = v * 2^-e rounded to the nearest E2M1 value,
// ties to the even mantissa, clamped to +-6.
//
// GEMMs (swap-AB, T <= 64): weights on the MMA M side (two M = 128 MMAs per K
// step: gate rows and the matching up rows, or two halves of the output
// features), the expert's padded token segment (16..64 rows, MMA N = 64) on N.  A
// pipeline stage carries 256 elements (128 bytes) of K per row plus the
// scales of both operands; the weight scales arrive by bulk copy in their
// tiled order, the token scales are re-tiled by the producer warp with
// asynchronous copies that complete on the stage barrier.  The MMA
// thread copies each stage's scales into a TMEM ring (tcgen05.cp) ahead of
// its MMAs (same thread, so they run in issue order).  Stage 1's epilogue
// computes SwiGLU and re-quantises h per 1x32 group directly: the 32 h
// columns of a group are the 32 lanes of one warp.
#include "gemm_common.cuh"
#include "moe_internal.h"
#include "sm100_ptx.cuh"

namespace moe {

namespace mx4 {

// ------------------------------------------------------------ quantiser

// Nearest E2M1 code of y (|y| < 8 after scaling), ties to the even mantissa.
__device__ __forceinline__ uint32_t e2m1_code(float y)
{
    const uint32_t sign = (__float_as_uint(y) >> 31) << 3;
    const float a = fabsf(y);
    const uint32_t i = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) + (a >= 3.5f) +
                       (a > 5.0f);
    return sign | i;
}

// Eight floats -> eight E2M1 codes in one word, element i in bits 4i..4i+3, by the tensor-format
// conversion instruction (two elements each; round to nearest even, saturating to +-6): the same
// rule as e2m1_code in a sixteenth of the instructions.  The quantiser's codes are compared bit for
// bit with the oracle's on every finite bf16 value of six binades around a group's scale.
__device__ __forceinline__ uint32_t e2m1x8(const float (&v)[8])
{
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(r)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return r;
}

// Shared exponent floor(log2(amax)) - 2, clamped to [-127, 127]; 0 for amax = 0.
__device__ __forceinline__ int mx_exponent(float amax)
{
    const uint32_t b = __float_as_uint(amax) & 0x7FFFFFFFu;
    if (b == 0)
        return 0;
    const int ef = (int)(b >> 23);
    const int fl = ef > 0 ? ef - 127 : (31 - __clz(b & 0x7FFFFF)) - 149;  // subnormal: m * 2^-149
    const int e = fl - 2;
    return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// 2^-e as a float (e in [-127, 125]: a normal number).
__device__ __forceinline__ float pow2_neg(int e) { return __uint_as_float((uint32_t)(127 - e) << 23); }

__device__ __forceinline__ uint32_t tiled_sf_offset(int64_t r, int g, int C)
{
    return (uint32_t)(((r >> 7) * (C >> 7) + (g >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (g & 3));
}

// Rows of X (bf16 [R][C], C % 32 == 0), optionally gathered through
// sorted_ids (row i = token sorted_ids[i] / k, padding -> zero row) with the
// row count read on the device.  4 threads per 32-element group, 8 elements
// (one 16-byte load, one 4-byte store of codes) per thread.
__global__ void __launch_bounds__(256) quant_mx4_kernel(const __nv_bfloat16 *__restrict__ X,
                                                       const int32_t *__restrict__ sorted_ids,
                                                       const int32_t *__restrict__ nrows, int64_t R, int S, int k,
                                                       int C, uint8_t *__restrict__ q, uint8_t *__restrict__ s,
                                                       int tiled)
{
    pdl_wait();
    pdl_trigger();
    const int64_t rows = nrows ? (int64_t)*nrows : R;
    const int nvec = C / 8;
    // one row per block and pass (no per-thread index division); every thread of a warp takes part
    // in the group shuffles, past the row's end with zeros
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        int64_t src = r;
        bool zero = false;
        if (sorted_ids) {
            const int sl = sorted_ids[r];
            zero = sl >= S;
            src = zero ? 0 : sl / k;
        }
        const uint4 *xr = reinterpret_cast<const uint4 *>(X + src * C);
        for (int c0 = 0; c0 < nvec; c0 += blockDim.x) {
            const int c8 = c0 + threadIdx.x;
            const bool ok = c8 < nvec;
            float f[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            if (ok && !zero) {
                const uint4 raw = __ldg(xr + c8);
                const __nv_bfloat162 *p2 = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 t = __bfloat1622float2(p2[i]);
                    f[2 * i] = t.x;
                    f[2 * i + 1] = t.y;
                }
            }
            float m = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                m = fmaxf(m, fabsf(f[i]));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
            const int e = mx_exponent(m);
            const float inv = pow2_neg(e);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                f[i] *= inv;
            const uint32_t packed = e2m1x8(f);
            if (ok) {
                reinterpret_cast<uint32_t *>(q + r * (C / 2))[c8] = packed;
                if ((c8 & 3) == 0) {
                    const int g = c8 >> 2;
                    const uint8_t sb = (uint8_t)(e + 127);
                    if (tiled)
                        s[tiled_sf_offset(r, g, C)] = sb;
                    else
                        s[r * (C / 32) + g] = sb;
                }
            }
        }
    }
}

// ------------------------------------------------------------- GEMMs

constexpr int kStages = 4;
constexpr int kKBytes = 128;                  // bytes of K per row per stage (256 elements)
constexpr int kWHalf = 128 * kKBytes;         // 16 KiB: 128 weight rows
constexpr int kWBytes = 2 * kWHalf;
constexpr int kXBytes = 64 * kKBytes;         // up to 64 token rows
constexpr int kWSf = 4 * 512;                 // 2 halves x 2 tiles of 128 x 4 scales
constexpr int kXSf = 2 * 512;
constexpr int kStageBytes = kWBytes + kXBytes + kWSf + kXSf;  // 44 KiB (a multiple of 1 KiB)
constexpr int kAccCols = 128;                 // half 0 at +0, half 1 at +64 (N <= 64)
constexpr int kSfCols = 24;                   // TMEM columns of one stage's scales
constexpr int kSfBase = 2 * kAccCols;
constexpr int kTmemCols = 512;
constexpr int kThreads = 192;
constexpr int kEpiWarps = 4;
static_assert(kStageBytes % 1024 == 0, "stages must keep 1 KiB alignment");
static_assert(kSfBase + kStages * kSfCols <= kTmemCols, "TMEM budget");

struct __align__(1024) Smem {
    uint8_t stage[kStages][kStageBytes];
    uint64_t full[kStages];    // TMA + bulk bytes, and the producer warp's re-tiled token scales
    uint64_t empty[kStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    TileQueue tq;
    uint32_t tmem_base;
    int abort;
};

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;

struct Tile {
    int e, xrow, nx, wrow0, wrow1, ncol0, kb0, kb1, ks;
};

template <int STAGE>
__device__ __forceinline__ int num_tiles(const GemmArgs &a)
{
    const int nwt = (STAGE == 1) ? a.N / 128 : (a.N + 255) / 256;
    return *a.num_active * nwt * a.split_k;
}

template <int STAGE>
__device__ __forceinline__ Tile get_tile(const GemmArgs &a, int t)
{
    Tile tl;
    const int nkb = a.K / 256;
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
    return tl;
}

// GemmArgs for MXFP4: tm_w / tm_x map the packed codes (bytes, K/2 per row);
// w_scales points at the weights' tiled E8M0 scales and x_scales at the
// token rows' row-major E8M0 scales (both as bytes).  Stage 1 writes h codes
// to inter and its scales to inter_scales (row-major, as bytes).
template <int STAGE>
__global__ void __launch_bounds__(kThreads, 1) gemm_mx4_kernel(const __grid_constant__ GemmArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int *abort_flag = &sm.abort;
    const uint8_t *wsf_g = reinterpret_cast<const uint8_t *>(a.w_scales);
    const uint8_t *xsf_g = reinterpret_cast<const uint8_t *>(a.x_scales);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sm.full[i], 1 + 32);  // TMA bytes + the producer lanes' scale copies
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
    pdl_wait();
    pdl_trigger();
    const int ntiles = num_tiles<STAGE>(a);
    const int kgroups = a.K / 32;     // scale bytes per token row
    const int ktiles = a.K / 128;     // 128-wide K tiles of the weight scales

    if (warp == 0) {
        // ------------------------------------------ producer (whole warp)
        const uint64_t pol_w = l2_policy_evict_first();
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
            int t = -1;
            bool qok = true;
            if (lane == 0)
                qok = tq_push_next(sm.tq, qs, qph, a.tile_counter, ntiles, claim, t, a.status, abort_flag);
            qok = __shfl_sync(0xffffffffu, (int)qok, 0) != 0;
            t = __shfl_sync(0xffffffffu, t, 0);
            if (!qok) {
                ok = false;
                break;
            }
            if (t < 0)
                break;
            const Tile tl = get_tile<STAGE>(a, t);
            const uint32_t bytes = kWBytes + tl.nx * kKBytes + kWSf;
            for (int kb = tl.kb0; kb < tl.kb1; ++kb) {
                bool w_ok = mbar_wait(&sm.empty[s], ph ^ 1, a.status, abort_flag);
                w_ok = __all_sync(0xffffffffu, w_ok);
                if (!w_ok) {
                    ok = false;
                    break;
                }
                uint8_t *st = sm.stage[s];
                if (lane == 0) {
                    mbar_arrive_expect_tx(&sm.full[s], bytes);
                    tma_load_2d(st, &a.tm_w, kb * kKBytes, tl.wrow0, &sm.full[s], pol_w);
                    tma_load_2d(st + kWHalf, &a.tm_w, kb * kKBytes, tl.wrow1, &sm.full[s], pol_w);
                    for (int c = 0; c < tl.nx; c += 16)
                        tma_load_2d(st + kWBytes + c * kKBytes, &a.tm_x, kb * kKBytes, tl.xrow + c, &sm.full[s],
                                    pol_x);
                    // weight scales: tiles (row block, K tiles 2kb and 2kb+1) are 1 KiB contiguous
                    bulk_load(st + kWBytes + kXBytes, wsf_g + ((size_t)(tl.wrow0 >> 7) * ktiles + 2 * kb) * 512,
                              1024, &sm.full[s]);
                    bulk_load(st + kWBytes + kXBytes + 1024,
                              wsf_g + ((size_t)(tl.wrow1 >> 7) * ktiles + 2 * kb) * 512, 1024, &sm.full[s]);
                    issued[s] = 1;
                    issued_ph[s] = ph;
                }
                // token scales: 8 bytes per row for this stage, re-tiled into two 128 x 4 blocks by
                // asynchronous 4-byte copies that complete on the stage barrier
                uint8_t *xsf = st + kWBytes + kXBytes + kWSf;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int j = lane + 32 * h;
                    if (j < tl.nx) {
                        const uint8_t *src = xsf_g + (size_t)(tl.xrow + j) * kgroups + kb * 8;
                        const int off = (j & 31) * 16 + (j >> 5) * 4;
                        cp_async_4(xsf + off, src);
                        cp_async_4(xsf + 512 + off, src + 4);
                    }
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
                if (!tq_pop(sm.tq, qs, qph, t, a.status, abort_flag)) {
                    ok = false;
                    break;
                }
                mbar_arrive(&sm.tq.empty[qs]);
                tq_advance(qs, qph);
                if (t < 0)
                    break;
                const Tile tl = get_tile<STAGE>(a, t);
                if (!mbar_wait(&sm.tempty[acc], aph ^ 1, a.status, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + acc * kAccCols;
                for (int kb = tl.kb0; kb < tl.kb1; ++kb) {
                    if (!mbar_wait(&sm.full[s], ph, a.status, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint8_t *st = sm.stage[s];
                    const uint8_t *sfw = st + kWBytes + kXBytes;
                    const uint8_t *sfx = sfw + kWSf;
                    const uint32_t sf = tmem_base + kSfBase + s * kSfCols;
                    fence_proxy_async_smem();  // the scale copies (generic proxy) before tcgen05.cp reads them
#pragma unroll
                    for (int i = 0; i < 4; ++i)  // weight scales: half i/2, K tile i%2
                        tmem_cp_sf(sf + 4 * i, smem_desc_rows16(sfw + 512 * i));
#pragma unroll
                    for (int i = 0; i < 2; ++i)
                        tmem_cp_sf(sf + 16 + 4 * i, smem_desc_rows16(sfx + 512 * i));
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {  // 4 MMAs of K = 64 (32 bytes) each
                        const uint32_t b = kk >> 1, id = (kk & 1) * 2;
                        // N is always 64 (the token tile's capacity): columns past the segment are
                        // never read, and one MMA shape serves every tile
                        const uint32_t idesc = make_idesc_mx4(128, 64, id, id);
                        const uint32_t accum = (kb > tl.kb0 || kk > 0) ? 1u : 0u;
#pragma unroll
                        for (int h = 0; h < 2; ++h)
                            mma_mx4(d + h * 64, smem_desc_sw128(st + h * kWHalf + kk * 32),
                                    smem_desc_sw128(st + kWBytes + kk * 32), idesc, sf + (2 * h + b) * 4,
                                    sf + 16 + b * 4, accum);
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
            const Tile tl = get_tile<STAGE>(a, t);
            bool ok = mbar_wait(&sm.tfull[acc], aph, a.status, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok)
                break;
            tc_fence_after();
            const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16) + acc * kAccCols;
            if (STAGE == 1) {
                // h column n = ncol0 + row; the warp's 32 lanes are one 1x32 group of h
                const int n = tl.ncol0 + row;
                uint8_t *hq = static_cast<uint8_t *>(a.inter);
                uint8_t *hs = reinterpret_cast<uint8_t *>(a.inter_scales);
#pragma unroll 1
                for (int c0 = 0; c0 < tl.nx; c0 += 16) {
                    float g[16], u[16];
                    tmem_ld16(tacc + c0, g);
                    tmem_ld16(tacc + 64 + c0, u);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float h = silu(g[j]) * u[j];
                        float m = fabsf(h);
#pragma unroll
                        for (int off = 16; off >= 1; off >>= 1)
                            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
                        const int e = mx_exponent(m);
                        const uint32_t code = e2m1_code(h * pow2_neg(e));
                        const uint32_t hi = __shfl_down_sync(0xffffffffu, code, 1);
                        const size_t tok = (size_t)(tl.xrow + c0 + j);
                        if ((lane & 1) == 0)
                            hq[tok * (a.N / 2) + n / 2] = (uint8_t)(code | (hi << 4));
                        if (lane == 0)
                            hs[tok * (a.N / 32) + n / 32] = (uint8_t)(e + 127);
                    }
                }
            } else {
#pragma unroll 1
                for (int half = 0; half < 2; ++half) {
                    const int n = tl.ncol0 + half * 128 + row;
                    const bool nok = n < a.N;
#pragma unroll 1
                    for (int c0 = 0; c0 < tl.nx; c0 += 16) {
                        float v[16];
                        tmem_ld16(tacc + half * 64 + c0, v);
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

// ------------------------------------------------- grouped (T > 64)
//
// Tokens on the MMA M side (128 sorted rows of one expert), weights on N:
// 128 rows per tile -- stage 1, 64 gate rows and the matching 64 up rows
// (accumulator columns j and 64 + j pair up), stage 2, 128 output features.
// N = 128 keeps two accumulators (2 x 128 columns) and the scale ring within
// 512 TMEM columns.  The producer warp assembles both operands' 128 x 4
// scale blocks per K tile: the tokens' from their row-major scales, the
// weights' from the matching words of their tiled scales (a 64-row half of
// a 128-row tile occupies words 0-1 or 2-3 of every lane).  Stage 1's
// epilogue thread holds a whole token row of the tile, so it quantises its
// 64 h values (two 1x32 groups) by itself.
namespace grouped {

constexpr int kStages = 6;
constexpr int kHalf = 128 * kKBytes;                    // 16 KiB: 128 rows x 256 elements
constexpr int kStageBytes = 2 * kHalf + 2 * 1024;      // [A tokens | B weights | A scales | B scales]
constexpr int kAccCols = 128;
constexpr int kSfCols = 16;                            // A: 2 K tiles x 4 columns, B: the same
constexpr int kSfBase = 2 * kAccCols;
constexpr int kGroupM = 16;
static_assert(kStageBytes % 1024 == 0, "stages must keep 1 KiB alignment");
static_assert(kSfBase + kStages * kSfCols <= kTmemCols, "TMEM budget");

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
};

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;

struct GTile {
    int e, mb, wrow0, wrow1, ncol0;
};

template <int STAGE>
__device__ __forceinline__ int nnt_of(const GemmArgs &a)
{
    return (STAGE == 1) ? a.N / 64 : (a.N + 127) / 128;
}

template <int STAGE>
__device__ __forceinline__ GTile get_gtile(const GemmArgs &a, int t)
{
    const int nmb = *a.num_post_padded / 128;
    const int nnt = nnt_of<STAGE>(a);
    const int group = t / (kGroupM * nnt);
    const int within = t - group * kGroupM * nnt;
    const int gsize = min(kGroupM, nmb - group * kGroupM);
    const int nt = within / gsize;
    GTile g;
    g.mb = group * kGroupM + within % gsize;
    g.e = a.sorted_expert_ids[g.mb];
    if (STAGE == 1) {
        g.wrow0 = g.e * a.rows_per_expert + nt * 64;          // gate rows
        g.wrow1 = g.e * a.rows_per_expert + a.N + nt * 64;    // matching up rows
        g.ncol0 = nt * 64;
    } else {
        g.wrow0 = g.e * a.rows_per_expert + nt * 128;
        g.wrow1 = g.wrow0 + 64;
        g.ncol0 = nt * 128;
    }
    return g;
}

// Address of words w0, w0+1 of lane l of tiled scale tile (row block rb, K tile kt).
__device__ __forceinline__ const uint8_t *sf_word_ptr(const uint8_t *sf, int64_t rb, int ktiles, int kt, int l,
                                                      int w0)
{
    return sf + ((size_t)rb * ktiles + kt) * 512 + l * 16 + w0 * 4;
}

template <int STAGE>
__global__ void __launch_bounds__(kThreads, 1) gemm_mx4_grouped_kernel(const __grid_constant__ GemmArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int *abort_flag = &sm.abort;
    const uint8_t *wsf_g = reinterpret_cast<const uint8_t *>(a.w_scales);
    const uint8_t *xsf_g = reinterpret_cast<const uint8_t *>(a.x_scales);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            // TMA bytes (+ the producer lanes' scale copies in stage 1)
            mbar_init(&sm.full[i], STAGE == 2 ? 1 : 1 + 32);
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
        tma_prefetch_desc(&a.tm_x);
        tma_prefetch_desc(&a.tm_w);
        if (STAGE == 2) {
            tma_prefetch_desc(&a.tm_sfa);
            tma_prefetch_desc(&a.tm_sfb);
        }
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
    const int ntiles = (*a.num_post_padded / 128) * nnt_of<STAGE>(a);
    const int nkb = a.K / 256;
    const int ktiles = a.K / 128;

    if (warp == 0) {
        // ------------------------------------------ producer (whole warp)
        const uint64_t pol_w = l2_policy_evict_normal();  // reused across a raster group of blocks
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
            int t = -1;
            bool qok = true;
            if (lane == 0)
                qok = tq_push_next(sm.tq, qs, qph, a.tile_counter, ntiles, claim, t, a.status, abort_flag);
            qok = __shfl_sync(0xffffffffu, (int)qok, 0) != 0;
            t = __shfl_sync(0xffffffffu, t, 0);
            if (!qok) {
                ok = false;
                break;
            }
            if (t < 0)
                break;
            const GTile g = get_gtile<STAGE>(a, t);
            const int xrow = g.mb * 128;
            for (int kb = 0; kb < nkb; ++kb) {
                bool w_ok = mbar_wait(&sm.empty[s], ph ^ 1, a.status, abort_flag);
                w_ok = __all_sync(0xffffffffu, w_ok);
                if (!w_ok) {
                    ok = false;
                    break;
                }
                uint8_t *st = sm.stage[s];
                uint8_t *asf = st + 2 * kHalf;
                uint8_t *bsf = asf + 1024;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&sm.full[s], 2 * kHalf + (STAGE == 2 ? 2048 : 0));
                    tma_load_2d(st, &a.tm_x, kb * kKBytes, xrow, &sm.full[s], pol_x);
                    tma_load_2d(st + kHalf, &a.tm_w, kb * kKBytes, g.wrow0, &sm.full[s], pol_w);
                    tma_load_2d(st + kHalf + kHalf / 2, &a.tm_w, kb * kKBytes, g.wrow1, &sm.full[s], pol_w);
                    if (STAGE == 2) {
                        // stage 2's 128 weight rows are one 128-row tile: both scale blocks are whole
                        // 512-byte tiles of the blocked order (two K tiles, 64 rows of 16 bytes each),
                        // so they come by TMA too and need no proxy fence before tcgen05.cp
                        tma_load_2d(asf, &a.tm_sfa, 0, ((xrow >> 7) * ktiles + 2 * kb) * 32, &sm.full[s], pol_x);
                        tma_load_2d(bsf, &a.tm_sfb, 0, ((g.wrow0 >> 7) * ktiles + 2 * kb) * 32, &sm.full[s], pol_w);
                    }
                    issued[s] = 1;
                    issued_ph[s] = ph;
                }
                if (STAGE == 2) {
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1;
                    }
                    continue;
                }
                // A scales: token rows l + 32 w of the block, 8 bytes each (two K tiles of 4 groups);
                // B scales: rows 0-63 from wrow0's tile, 64-127 from wrow1's (words of a 64-row half).
                // Asynchronous copies that complete on the stage barrier.
                {
                    // the block's scales of K tiles 2kb and 2kb + 1 are two consecutive 512-byte tiles
                    // of the blocked order: one 16-byte copy per lane from each (a warp's copy covers
                    // 512 contiguous bytes, free of shared-memory bank conflicts)
                    const uint8_t *src = xsf_g + ((size_t)(xrow >> 7) * ktiles + 2 * kb) * 512 + lane * 16;
                    cp_async_16_zfill(asf + lane * 16, src, true);
                    cp_async_16_zfill(asf + 512 + lane * 16, src + 512, true);
                }
                // B: blocked row m takes words 0-1 from wrow0's tile and words 2-3 from wrow1's; lanes
                // 2m and 2m + 1 copy the two halves of row m, so each 16-lane phase of a copy writes
                // 128 contiguous bytes (no bank conflicts)
                {
                    const int part = lane & 1;
                    const int wrow = part ? g.wrow1 : g.wrow0;
#pragma unroll
                    for (int kt = 0; kt < 2; ++kt) {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int m = h * 16 + (lane >> 1);
                            cp_async_8(bsf + kt * 512 + m * 16 + part * 8,
                                       sf_word_ptr(wsf_g, wrow >> 7, ktiles, 2 * kb + kt, m, (wrow & 127) >> 5));
                        }
                    }
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
                if (!tq_pop(sm.tq, qs, qph, t, a.status, abort_flag)) {
                    ok = false;
                    break;
                }
                mbar_arrive(&sm.tq.empty[qs]);
                tq_advance(qs, qph);
                if (t < 0)
                    break;
                if (!mbar_wait(&sm.tempty[acc], aph ^ 1, a.status, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + acc * kAccCols;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(&sm.full[s], ph, a.status, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint8_t *st = sm.stage[s];
                    const uint32_t sf = tmem_base + kSfBase + s * kSfCols;
                    if (STAGE == 1)
                        fence_proxy_async_smem();  // the scale copies (generic proxy) before tcgen05.cp reads them
#pragma unroll
                    for (int i = 0; i < 4; ++i)  // A K tiles 0,1 then B K tiles 0,1
                        tmem_cp_sf(sf + 4 * i, smem_desc_rows16(st + 2 * kHalf + 512 * i));
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t b = kk >> 1, id = (kk & 1) * 2;
                        mma_mx4(d, smem_desc_sw128(st + kk * 32), smem_desc_sw128(st + kHalf + kk * 32),
                                make_idesc_mx4(128, 128, id, id), sf + b * 4, sf + 8 + b * 4,
                                (kb > 0 || kk > 0) ? 1u : 0u);
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
        const int row = q * 32 + lane;    // token row within the block (TMEM lane)
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
            const GTile g = get_gtile<STAGE>(a, t);
            bool ok = mbar_wait(&sm.tfull[acc], aph, a.status, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok)
                break;
            tc_fence_after();
            const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16) + acc * kAccCols;
            const int pos = g.mb * 128 + row;
            if (STAGE == 1) {
                uint8_t *hq = static_cast<uint8_t *>(a.inter) + (size_t)pos * (a.N / 2) + g.ncol0 / 2;
                // h's scales in the tensor core's 128 x 4 blocked order, as stage 2's producer copies them
                uint8_t *hs = reinterpret_cast<uint8_t *>(a.inter_scales);
#pragma unroll 1
                for (int c0 = 0; c0 < 64; c0 += 32) {
                    float gv[32], uv[32], h[32];
                    tmem_ld32(tacc + c0, gv);
                    tmem_ld32(tacc + 64 + c0, uv);
                    float m = 0.0f;
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        h[i] = silu(gv[i]) * uv[i];
                        m = fmaxf(m, fabsf(h[i]));
                    }
                    const int e = mx_exponent(m);
                    const float inv = pow2_neg(e);
                    uint32_t w[4];
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        float y[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            y[i] = h[8 * b + i] * inv;
                        w[b] = e2m1x8(y);
                    }
                    *reinterpret_cast<uint4 *>(hq + c0 / 2) = make_uint4(w[0], w[1], w[2], w[3]);
                    hs[tiled_sf_offset(pos, (g.ncol0 + c0) / 32, a.N)] = (uint8_t)(e + 127);
                }
            } else {
                const int slot = a.sorted_ids[pos];
                const float wgt = a.sorted_weights[pos];
                const bool live = slot < a.S;
                __nv_bfloat16 *dst = a.y + (size_t)(live ? slot : 0) * a.N + g.ncol0;
                const int ncols = min(128, a.N - g.ncol0);
#pragma unroll 1
                for (int c0 = 0; c0 < ncols; c0 += 32) {
                    float v[32];
                    tmem_ld32(tacc + c0, v);
                    if (!live)
                        continue;
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        v[i] *= wgt;
                    store_bf16x32(dst + c0, v);
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

template <int STAGE>
cudaError_t launch(const GemmArgs &a, int grid, cudaStream_t st)
{
    auto kern = gemm_mx4_grouped_kernel<STAGE>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (err != cudaSuccess)
        return err;
    return launch_kernel(pdl_site(a.pdl_mask, STAGE == 1 ? kPdlStage1 : kPdlStage2), kern, dim3(grid),
                         dim3(kThreads), kSmemBytes, st, a);
}

}  // namespace grouped

template <int STAGE>
cudaError_t launch(const GemmArgs &a, int grid, cudaStream_t st)
{
    auto kern = gemm_mx4_kernel<STAGE>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (err != cudaSuccess)
        return err;
    return launch_kernel(pdl_site(a.pdl_mask, STAGE == 1 ? kPdlStage1 : kPdlStage2), kern, dim3(grid),
                         dim3(kThreads), kSmemBytes, st, a);
}

}  // namespace mx4

cudaError_t launch_quant_mx4(const __nv_bfloat16 *X, const int32_t *sorted_ids, const int32_t *nrows, int64_t R,
                             int S, int k, int C, uint8_t *q, uint8_t *s, bool tiled, bool pdl, cudaStream_t st)
{
    int64_t grid = R < 152 * 32 ? R : 152 * 32;  // rows per pass (the row count may be read on the device)
    if (grid < 1)
        return cudaSuccess;
    return launch_kernel(pdl, mx4::quant_mx4_kernel, dim3((unsigned)grid), dim3(256), 0, st, X, sorted_ids, nrows,
                         R, S, k, C, q, s, tiled ? 1 : 0);
}

cudaError_t launch_gemm_swap_mx4(int stage, const GemmArgs &a, int grid, cudaStream_t st)
{
    return stage == 1 ? mx4::launch<1>(a, grid, st) : mx4::launch<2>(a, grid, st);
}

cudaError_t launch_gemm_grouped_mx4(int stage, const GemmArgs &a, int grid, cudaStream_t st)
{
    return stage == 1 ? mx4::grouped::launch<1>(a, grid, st) : mx4::grouped::launch<2>(a, grid, st);
}

}  // namespace moe
