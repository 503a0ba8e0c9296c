// Router (gating + warp-shuffle top-k), align-sort by expert, row gathers and
// block-scaled FP8 quantisation of the fused MoE layer.  These are the
// memory- and latency-bound steps before the two group GEMMs (the combine
// after them is in moe_combine.cu).
//
// Sources (fused-MoE pages): AITER walk-through section 3 ("Fused MoE":
// gating -> token reorder -> expert GEMMs -> weighted combine), section 3.1
// (moe_sorting: slots grouped by expert, per-expert padding to the block
// size, buffers of T*k + E*B - k entries), the "per_1x128" quantisation type
// of that page, and the Mixtral group-GEMM talk (top-2 routing, SwiGLU).
#include <cuda_fp8.h>

#include <cfloat>
#include <climits>
#include <cstring>

#include "moe_internal.h"

namespace moe {

__device__ __forceinline__ void bf16x8_to_float(const uint4 &v, float (&f)[8])
{
    const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 t = __bfloat1622float2(p[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

// ================================================================ router
//
// logit[t][e] in fp32, one fixed order: lane L of a warp accumulates (one
// rounding per element; a bf16 x bf16 product is exact in fp32) the
// elements h with (h / 8) mod 32 == L in ascending h, then a xor butterfly
// with strides 16, 8, 4, 2, 1 combines the 32 partials; the bias is added
// last.  Any tiling that keeps each lane's partial in this order gives the
// same bits, so the two kernels below agree with each other and with the
// CPU oracle.

// (c0, c1) = (a0 * b0 + c0, a1 * b1 + c1) in one paired-fp32 instruction of the
// sm_100 family; each lane is rounded once, exactly like fmaf.
__device__ __forceinline__ void fma2(float &c0, float &c1, float a0, float a1, float b0, float b1)
{
    asm("{\n\t.reg .b64 a, b, c, d;\n\t"
        "mov.b64 a, {%2, %3};\n\t"
        "mov.b64 b, {%4, %5};\n\t"
        "mov.b64 c, {%0, %1};\n\t"
        "fma.rn.f32x2 d, a, b, c;\n\t"
        "mov.b64 {%0, %1}, d;\n\t}"
        : "+f"(c0), "+f"(c1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// acc += x[2i] * w[2i], then acc += x[2i+1] * w[2i+1] (the low, then the high bf16 of each word), with
// the mixed-precision fma: the exact product of the two bf16 values plus acc, rounded once --
// the same roundings as fmaf on the widened values, without the conversion instructions.
__device__ __forceinline__ void fma_bf16x2_chain(float &acc, uint32_t xw, uint32_t ww)
{
    // elements 2i (low half) then 2i + 1 (high half)
    asm("{\n\t.reg .b16 xl, xh, wl, wh;\n\t"
        "mov.b32 {xl, xh}, %1;\n\t"
        "mov.b32 {wl, wh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, xl, wl, %0;\n\t"
        "fma.rn.f32.bf16 %0, xh, wh, %0;\n\t}"
        : "+f"(acc)
        : "r"(xw), "r"(ww));
}

__device__ __forceinline__ float butterfly_sum(float v)
{
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

__device__ __forceinline__ void warp_softmax_k(const float *lg, int E, int k, int renorm, int lane, float my_v,
                                               int my_e, int32_t *ids_out, float *w_out);

// Top k of one token's E logits by one warp (larger logit first, the lower
// expert on ties), then the softmax over the k selected (renorm = 1) or over
// all E, evaluated at the selected (renorm = 0).  k <= 32, E <= 1024.
__device__ __forceinline__ void warp_topk_softmax(const float *lg, int E, int k, int renorm, int lane,
                                                  int32_t *ids_out, float *w_out)
{
    uint32_t taken = 0;  // bit m: expert lane + 32m already selected
    float my_v = 0.0f;
    int my_e = 0;
    for (int j = 0; j < k; ++j) {
        float bv = -FLT_MAX;
        int be = INT_MAX;
        for (int m = 0, e = lane; e < E; ++m, e += 32) {
            if (taken & (1u << m))
                continue;
            const float v = lg[e];
            if (be == INT_MAX || v > bv) {  // ascending e: ties keep the lower expert
                bv = v;
                be = e;
            }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oe = __shfl_xor_sync(0xffffffffu, be, off);
            if (oe != INT_MAX && (be == INT_MAX || ov > bv || (ov == bv && oe < be))) {
                bv = ov;
                be = oe;
            }
        }
        if ((be & 31) == lane)
            taken |= 1u << (be >> 5);
        if (lane == j) {
            my_v = bv;
            my_e = be;
        }
    }
    warp_softmax_k(lg, E, k, renorm, lane, my_v, my_e, ids_out, w_out);
}

// Lanes j < k hold the j-th selected logit and expert (largest first): the weights, softmax over
// the k (renorm = 1) or over all E logits lg (renorm = 0), and the outputs.
__device__ __forceinline__ void warp_softmax_k(const float *lg, int E, int k, int renorm, int lane, float my_v,
                                               int my_e, int32_t *ids_out, float *w_out)
{
    const float vmax = __shfl_sync(0xffffffffu, my_v, 0);
    const float ex = (lane < k) ? expf(my_v - vmax) : 0.0f;
    float sum = 0.0f;
    if (renorm) {
        for (int j = 0; j < k; ++j)
            sum += __shfl_sync(0xffffffffu, ex, j);
    } else {
        for (int e = lane; e < E; e += 32)
            sum += expf(lg[e] - vmax);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1)
            sum += __shfl_xor_sync(0xffffffffu, sum, off);
    }
    if (lane < k) {
        ids_out[lane] = my_e;
        w_out[lane] = ex / sum;
    }
}

// Small T*E (decode): a CTA takes TT tokens, each warp groups of EG experts;
// each lane keeps UNR 256-element rounds of loads in flight.  The CTA's
// logits go to shared memory and one warp per token selects the top k.
template <int TT, int EG, int UNR>
__global__ void __launch_bounds__(256) router_small_kernel(const __nv_bfloat16 *__restrict__ x,
                                                           const __nv_bfloat16 *__restrict__ Wr,
                                                           const float *__restrict__ bias, int T, int H, int E,
                                                           int k, int renorm, int32_t *__restrict__ ids,
                                                           float *__restrict__ wts, float *__restrict__ logits_out,
                                                           int *status)
{
    extern __shared__ float s_logit[];  // [TT][E]
    pdl_wait();
    pdl_trigger();
    if (status && blockIdx.x == 0 && threadIdx.x < kStatusWords)
        status[threadIdx.x] = 0;  // status word and the GEMMs' tile counters
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.x * TT;
    const int ngroups = (E + EG - 1) / EG;

    for (int g = warp; g < ngroups; g += 8) {
        float acc[TT][EG];
#pragma unroll
        for (int t = 0; t < TT; ++t)
#pragma unroll
            for (int j = 0; j < EG; ++j)
                acc[t][j] = 0.0f;
        for (int hb = 0; hb < H; hb += 256 * UNR) {
            uint4 wv[UNR][EG], xv[UNR][TT];
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                const int h0 = hb + u * 256 + lane * 8;
#pragma unroll
                for (int j = 0; j < EG; ++j) {
                    const int e = g * EG + j;
                    wv[u][j] = (h0 < H && e < E) ? __ldg(reinterpret_cast<const uint4 *>(Wr + (size_t)e * H + h0))
                                                 : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int t = 0; t < TT; ++t) {
                    const int tok = t0 + t;
                    xv[u][t] = (h0 < H && tok < T)
                                   ? __ldg(reinterpret_cast<const uint4 *>(x + (size_t)tok * H + h0))
                                   : make_uint4(0, 0, 0, 0);
                }
            }
            // (widened to fp32 first: with only TT x EG chains per lane the conversions fill the
            // FMA latency; the mixed-precision fma measured slower here, 11.3 -> 13.5 us)
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                float wf[EG][8];
#pragma unroll
                for (int j = 0; j < EG; ++j)
                    bf16x8_to_float(wv[u][j], wf[j]);
#pragma unroll
                for (int t = 0; t < TT; ++t) {
                    float xf[8];
                    bf16x8_to_float(xv[u][t], xf);
#pragma unroll
                    for (int c = 0; c < 8; ++c)
#pragma unroll
                        for (int j = 0; j < EG; ++j)
                            acc[t][j] = __fmaf_rn(xf[c], wf[j][c], acc[t][j]);
                }
            }
        }
#pragma unroll
        for (int t = 0; t < TT; ++t)
#pragma unroll
            for (int j = 0; j < EG; ++j) {
                float v = butterfly_sum(acc[t][j]);
                const int e = g * EG + j;
                if (lane == 0 && e < E) {
                    if (bias)
                        v = __fadd_rn(v, bias[e]);
                    s_logit[t * E + e] = v;
                }
            }
    }
    __syncthreads();

    for (int t = warp; t < TT; t += 8) {
        const int tok = t0 + t;
        if (tok >= T)
            continue;
        const float *lg = s_logit + t * E;
        if (logits_out)
            for (int e = lane; e < E; e += 32)
                logits_out[(size_t)tok * E + e] = lg[e];
        warp_topk_softmax(lg, E, k, renorm, lane, ids + (size_t)tok * k, wts + (size_t)tok * k);
    }
}

// Large T*E: a CTA computes a (WT*NWT tokens) x (WE*NWE experts) tile of
// logits.  256-element rounds of x and W_router rows are staged in shared
// memory (double-buffered cp.async, zero-filled past T, E or H); warp
// (wt, we) computes WT x WE logits, lane L reading its 16-byte slice of each
// staged row, so every partial keeps the fixed order above.
constexpr int kRouterStages = 4;

template <int WT, int WE, int NWT, int NWE>
constexpr size_t router_tiled_smem()
{
    return (size_t)kRouterStages * (WT * NWT + WE * NWE) * 256 * sizeof(__nv_bfloat16);
}

template <int WT, int WE, int NWT, int NWE>
__global__ void __launch_bounds__(256) router_tiled_kernel(const __nv_bfloat16 *__restrict__ x,
                                                           const __nv_bfloat16 *__restrict__ Wr,
                                                           const float *__restrict__ bias, int T, int H, int E,
                                                           float *__restrict__ logits, int *status)
{
    constexpr int TT = WT * NWT, EC = WE * NWE, ROWS = TT + EC;
    static_assert(NWT * NWE == 8, "8 warps");
    extern __shared__ __align__(16) uint8_t s_raw[];
    auto s_rows = reinterpret_cast<__nv_bfloat16(*)[ROWS][256]>(s_raw);  // [kRouterStages][ROWS][256]
    pdl_wait();
    pdl_trigger();
    if (status && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x < kStatusWords)
        status[threadIdx.x] = 0;  // status word and the GEMMs' tile counters
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.x * TT, e0 = blockIdx.y * EC;
    const int wt = warp / NWE, we = warp % NWE;
    const int nchunks = (H + 255) / 256;

    auto stage = [&](int c, int b) {
        for (int v = threadIdx.x; v < ROWS * 32; v += 256) {
            const int r = v >> 5, col = (v & 31) * 8;
            const int h = c * 256 + col;
            const __nv_bfloat16 *src;
            bool ok;
            if (r < TT) {
                ok = (t0 + r < T) && h < H;
                src = x + (size_t)(ok ? t0 + r : 0) * H + (ok ? h : 0);
            } else {
                ok = (e0 + r - TT < E) && h < H;
                src = Wr + (size_t)(ok ? e0 + r - TT : 0) * H + (ok ? h : 0);
            }
            const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(&s_rows[b][r][col]));
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(ok ? 16 : 0)
                         : "memory");
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };

    float acc[WT][WE];
#pragma unroll
    for (int t = 0; t < WT; ++t)
#pragma unroll
        for (int j = 0; j < WE; ++j)
            acc[t][j] = 0.0f;

    // kRouterStages-deep ring: chunk c lives in buffer c % kRouterStages; one commit group per
    // chunk (empty past the end) so that "all but the newest kRouterStages-1 groups" = chunk c.
    for (int c = 0; c < kRouterStages - 1; ++c) {
        if (c < nchunks)
            stage(c, c);
        else
            asm volatile("cp.async.commit_group;" ::: "memory");
    }
    for (int c = 0; c < nchunks; ++c) {
        const int b = c % kRouterStages;
        const int cn = c + kRouterStages - 1;
        if (cn < nchunks)
            stage(cn, cn % kRouterStages);
        else
            asm volatile("cp.async.commit_group;" ::: "memory");
        asm volatile("cp.async.wait_group %0;" ::"n"(kRouterStages - 1) : "memory");
        __syncthreads();
        float xf[WT][8];
#pragma unroll
        for (int t = 0; t < WT; ++t)
            bf16x8_to_float(*reinterpret_cast<const uint4 *>(&s_rows[b][wt * WT + t][lane * 8]), xf[t]);
        static_assert(WE % 2 == 0, "experts are processed in pairs");
#pragma unroll
        for (int j = 0; j < WE; j += 2) {
            float wf0[8], wf1[8];
            bf16x8_to_float(*reinterpret_cast<const uint4 *>(&s_rows[b][TT + we * WE + j][lane * 8]), wf0);
            bf16x8_to_float(*reinterpret_cast<const uint4 *>(&s_rows[b][TT + we * WE + j + 1][lane * 8]), wf1);
#pragma unroll
            for (int t = 0; t < WT; ++t)
#pragma unroll
                for (int cc = 0; cc < 8; ++cc)
                    fma2(acc[t][j], acc[t][j + 1], xf[t][cc], xf[t][cc], wf0[cc], wf1[cc]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int t = 0; t < WT; ++t)
#pragma unroll
        for (int j = 0; j < WE; ++j) {
            float v = butterfly_sum(acc[t][j]);
            const int tok = t0 + wt * WT + t, e = e0 + we * WE + j;
            if (lane == 0 && tok < T && e < E) {
                if (bias)
                    v = __fadd_rn(v, bias[e]);
                logits[(size_t)tok * E + e] = v;
            }
        }
}

__global__ void __launch_bounds__(256) topk_kernel(const float *__restrict__ logits, int T, int E, int k, int renorm,
                                                  int32_t *__restrict__ ids, float *__restrict__ wts)
{
    pdl_wait();
    pdl_trigger();
    const int tok = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (tok >= T)
        return;
    warp_topk_softmax(logits + (size_t)tok * E, E, k, renorm, threadIdx.x & 31, ids + (size_t)tok * k,
                      wts + (size_t)tok * k);
}

bool router_needs_logits(int T, int E) { return (long)T * E > 64L * 64; }

template <int WT, int WE, int NWT, int NWE>
static cudaError_t launch_router_tiled(const __nv_bfloat16 *x, const __nv_bfloat16 *Wr, const float *bias, int T,
                                       int H, int E, float *logits, int *status, bool pdl, cudaStream_t st)
{
    auto kern = router_tiled_kernel<WT, WE, NWT, NWE>;
    constexpr size_t smem = router_tiled_smem<WT, WE, NWT, NWE>();
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess)
        return err;
    return launch_kernel(pdl, kern, dim3((T + WT * NWT - 1) / (WT * NWT), (E + WE * NWE - 1) / (WE * NWE)),
                         dim3(256), smem, st, x, Wr, bias, T, H, E, logits, status);
}

cudaError_t launch_router(const __nv_bfloat16 *x, const __nv_bfloat16 *Wr, const float *bias, int T, int H, int E,
                          int k, int renorm, int32_t *ids, float *wts, float *logits, int *status, int pdl_mask,
                          cudaStream_t st)
{
    if (T <= 0)
        return cudaSuccess;
    const bool pdl = pdl_site(pdl_mask, kPdlRouter);
    if (!router_needs_logits(T, E) || !logits) {
        if ((long)T * E <= 64L * 64) {
            constexpr int TT = 2;
            return launch_kernel(pdl, router_small_kernel<TT, 1, 8>, dim3((T + TT - 1) / TT), dim3(256),
                                 sizeof(float) * TT * E, st, x, Wr, bias, T, H, E, k, renorm, ids, wts, logits,
                                 status);
        }
        constexpr int TT = 8;
        return launch_kernel(pdl, router_small_kernel<TT, 4, 2>, dim3((T + TT - 1) / TT), dim3(256),
                             sizeof(float) * TT * E, st, x, Wr, bias, T, H, E, k, renorm, ids, wts, logits, status);
    }
    cudaError_t err;
    if (E <= 8)
        err = launch_router_tiled<2, 8, 8, 1>(x, Wr, bias, T, H, E, logits, status, pdl, st);
    else if (E <= 16)
        err = launch_router_tiled<2, 16, 8, 1>(x, Wr, bias, T, H, E, logits, status, pdl, st);
    else
        err = launch_router_tiled<4, 16, 4, 2>(x, Wr, bias, T, H, E, logits, status, pdl, st);
    if (err != cudaSuccess)
        return err;
    return launch_kernel(pdl_site(pdl_mask, kPdlTopk), topk_kernel, dim3((T + 7) / 8), dim3(256), 0, st, logits, T,
                         E, k, renorm, ids, wts);
}

// ============================================== router on the tensor core
//
// With many experts (fine-grained routing: E = 256, H = 7168) the fixed-order
// fp32 logits cost E*H FMAs per token on CUDA cores.  Here the tensor core
// computes all logits (bf16 products, fp32 accumulation in an unspecified
// order, K split into slices whose partial logits are added after), and the
// fixed order is spent only where it decides something:
//   1. the k + kTcExtra experts with the largest tensor-core logits are the
//      candidates; their logits are recomputed in the fixed order (exactly
//      the values the other router kernels produce);
//   2. the k largest candidates by those exact values (ties to the lower
//      expert) are the selection, if every other expert's tensor-core logit
//      plus a bound on the two computations' difference stays below the
//      k-th exact value: then no other expert's exact logit can reach it;
//   3. otherwise (a near tie) all E logits are recomputed in the fixed order
//      and selected as the other kernels do.
// So the ids and weights are the fixed-order ones bit for bit.  The bound:
// both sums consist of the same exact products p_h = x_h * w_h (a bf16 x
// bf16 product fits fp32); the fixed order adds at most H/32 + 5 of them in
// a chain (error <= 2^-16 sum|p| for H <= 2^20 ... far below the next
// term); the tensor core's accumulation is taken to lose at most 2^-12
// sum|p| (an fp32 accumulator, even truncating, loses about 2^-22 per
// addition; a test measures the actual difference); the slice additions and
// the bias add a few fp32 roundings.  Together <= 2^-11 sum|p| + 2^-22 |bias|,
// with sum|p| <= ||x_t|| ||w_e|| (Cauchy-Schwarz; both norms rounded up).
constexpr int kTcExtra = 4;
constexpr int kTcMaxSplits = 8;  // K slices of the tensor-core logits (router_tc_splits)

bool router_tc_eligible(int T, int H, int E, int k)
{
    return E >= 64 && E % 32 == 0 && E <= 1024 && k + kTcExtra <= 32 && T >= 64 && H % 64 == 0;
}

int router_tc_splits(int T, int H, int E, int num_sms)
{
    const int nkb = H / 64;
    const int64_t tiles1 = (int64_t)((T + 127) / 128) * ((E + 255) / 256);
    int s = 1;
    while (s < 8 && tiles1 * s < num_sms / 2 && nkb % (2 * s) == 0)
        s *= 2;
    return s;
}

size_t router_tc_scratch_floats(int T, int H, int E, int num_sms)
{
    return (size_t)router_tc_splits(T, H, E, num_sms) * ((T + 127) / 128 * 128) * E + E;
}

// Upper bound of ||W_router[e]||_2 per expert (one warp per expert); also zeroes the status words.
__global__ void __launch_bounds__(256) router_wnorm_kernel(const __nv_bfloat16 *__restrict__ Wr, int H, int E,
                                                          float *__restrict__ wnorm, int *status)
{
    pdl_wait();
    pdl_trigger();
    if (status && blockIdx.x == 0 && threadIdx.x < kStatusWords)
        status[threadIdx.x] = 0;  // status word, tile counters, router fall-back count
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * 8 + warp;
    if (e >= E)
        return;
    float ss = 0.0f;
#pragma unroll 4
    for (int h0 = lane * 8; h0 < H; h0 += 256) {  // (unrolled: several row loads in flight)
        float f[8];
        bf16x8_to_float(__ldg(reinterpret_cast<const uint4 *>(Wr + (size_t)e * H + h0)), f);
#pragma unroll
        for (int c = 0; c < 8; ++c)
            ss = fmaf(f[c], f[c], ss);
    }
    ss = butterfly_sum(ss);
    // the fp32 sum of squares is within (H/32 + 6) * 2^-24 of the exact one (H <= 2^20)
    if (lane == 0)
        wnorm[e] = sqrtf(ss) * (1.0f + 0x1p-8f);
}

// Fixed-order logits (the order of the other router kernels: lane L adds the elements h with
// (h / 8) mod 32 == L in ascending h, then the butterfly, then the bias) of N <= 8 experts of
// one token, by one warp; every lane returns the values.  Two 256-element rounds are loaded
// before either is added, so more loads are in flight; each lane's chain still adds its
// elements in ascending h (round r before round r + 1).  The products take the bf16 operands
// straight from the loaded words (mixed-precision fma: exact product, one rounding, as fmaf on
// the widened values), so no conversion instructions are spent.
template <int N>
__device__ __forceinline__ void exact_logits_acc(const uint4 &xv, const uint4 (&wv)[N], float (&acc)[N])
{
#pragma unroll
    for (int j = 0; j < N; ++j) {
        fma_bf16x2_chain(acc[j], xv.x, wv[j].x);
        fma_bf16x2_chain(acc[j], xv.y, wv[j].y);
        fma_bf16x2_chain(acc[j], xv.z, wv[j].z);
        fma_bf16x2_chain(acc[j], xv.w, wv[j].w);
    }
}

template <int N>
__device__ __forceinline__ void exact_logits_n(const __nv_bfloat16 *xrow, const __nv_bfloat16 *Wr, const float *bias,
                                               int H, const int (&es)[8], int lane, float (&out)[8])
{
    float acc[N];
    const __nv_bfloat16 *wp[N];
#pragma unroll
    for (int j = 0; j < N; ++j) {
        acc[j] = 0.0f;
        wp[j] = Wr + (size_t)es[j] * H;
    }
    for (int h0 = lane * 8; h0 < H; h0 += 512) {
        const bool two = h0 + 256 < H;
        const uint4 xv0 = __ldg(reinterpret_cast<const uint4 *>(xrow + h0));
        const uint4 xv1 = two ? __ldg(reinterpret_cast<const uint4 *>(xrow + h0 + 256)) : make_uint4(0, 0, 0, 0);
        uint4 wv0[N], wv1[N];
#pragma unroll
        for (int j = 0; j < N; ++j) {
            wv0[j] = __ldg(reinterpret_cast<const uint4 *>(wp[j] + h0));
            wv1[j] = two ? __ldg(reinterpret_cast<const uint4 *>(wp[j] + h0 + 256)) : make_uint4(0, 0, 0, 0);
        }
        exact_logits_acc<N>(xv0, wv0, acc);
        if (two)
            exact_logits_acc<N>(xv1, wv1, acc);
    }
#pragma unroll
    for (int j = 0; j < N; ++j) {
        float v = butterfly_sum(acc[j]);
        if (bias)
            v = __fadd_rn(v, bias[es[j]]);
        out[j] = v;
    }
#pragma unroll
    for (int j = N; j < 8; ++j)
        out[j] = 0.0f;
}

// exact_logits_n for a run-time count n in 1..8 (out[j] for j >= n is unspecified).
__device__ __forceinline__ void exact_logits8(const __nv_bfloat16 *xrow, const __nv_bfloat16 *Wr, const float *bias,
                                              int H, const int (&es)[8], int n, int lane, float (&out)[8])
{
    switch (n) {
    case 1: exact_logits_n<1>(xrow, Wr, bias, H, es, lane, out); break;
    case 2: exact_logits_n<2>(xrow, Wr, bias, H, es, lane, out); break;
    case 3: exact_logits_n<3>(xrow, Wr, bias, H, es, lane, out); break;
    case 4: exact_logits_n<4>(xrow, Wr, bias, H, es, lane, out); break;
    case 5: exact_logits_n<5>(xrow, Wr, bias, H, es, lane, out); break;
    case 6: exact_logits_n<6>(xrow, Wr, bias, H, es, lane, out); break;
    case 7: exact_logits_n<7>(xrow, Wr, bias, H, es, lane, out); break;
    default: exact_logits_n<8>(xrow, Wr, bias, H, es, lane, out); break;
    }
}

// One warp per token: tensor-core logits -> candidates -> exact values -> checked selection.
__global__ void __launch_bounds__(256) router_select_kernel(const __nv_bfloat16 *__restrict__ x,
                                                           const __nv_bfloat16 *__restrict__ Wr,
                                                           const float *__restrict__ bias, int T, int H, int E,
                                                           int k, const float *__restrict__ part, int nsplit,
                                                           int64_t part_rows, const float *__restrict__ wnorm,
                                                           int32_t *__restrict__ ids, float *__restrict__ wts,
                                                           int *fallbacks)
{
    extern __shared__ float s_lg[];  // [8 warps][E]
    pdl_wait();
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    if (t >= T)
        return;
    float *lg = s_lg + warp * E;
    const __nv_bfloat16 *xrow = x + (size_t)t * H;
    // the slices' partial logits, summed in slice order; the loads of four experts' slices are
    // issued before any sum (one L2 round trip per four experts, not one per slice)
    for (int e0 = lane; e0 < E; e0 += 4 * 32) {
        float pv[4][kTcMaxSplits];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int sl = 0; sl < kTcMaxSplits; ++sl)
                pv[j][sl] = (e0 + 32 * j < E && sl < nsplit)
                                ? __ldg(part + ((size_t)sl * part_rows + t) * E + e0 + 32 * j)
                                : 0.0f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = e0 + 32 * j;
            if (e >= E)
                break;
            float v = 0.0f;
#pragma unroll
            for (int sl = 0; sl < kTcMaxSplits; ++sl)
                if (sl < nsplit)
                    v += pv[j][sl];
            if (bias)
                v += bias[e];
            lg[e] = v;
        }
    }
    float ss = 0.0f;
#pragma unroll 4
    for (int h0 = lane * 8; h0 < H; h0 += 256) {  // (unrolled: several row loads in flight)
        float f[8];
        bf16x8_to_float(__ldg(reinterpret_cast<const uint4 *>(xrow + h0)), f);
#pragma unroll
        for (int c = 0; c < 8; ++c)
            ss = fmaf(f[c], f[c], ss);
    }
    const float xnorm = sqrtf(butterfly_sum(ss)) * (1.0f + 0x1p-8f);
    __syncwarp();

    // 1. candidates: the nc largest tensor-core logits (ties to the lower expert); lane c keeps one
    const int nc = min(E, k + kTcExtra);
    uint32_t taken = 0;  // bit m: expert lane + 32m is a candidate
    int my_c = 0;
    // up to 256 experts: the lane's eight logits stay in registers across the rounds
    const bool in_regs = E <= 256;
    float lv[8];
    uint32_t valid = 0;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const int e = lane + 32 * m;
        lv[m] = (in_regs && e < E) ? lg[e] : 0.0f;
        if (e < E)
            valid |= 1u << m;
    }
    for (int c = 0; c < nc; ++c) {
        float bv = -FLT_MAX;
        int be = INT_MAX;
        if (in_regs) {
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                if (!(valid & (1u << m)) || (taken & (1u << m)))
                    continue;
                if (be == INT_MAX || lv[m] > bv) {
                    bv = lv[m];
                    be = lane + 32 * m;
                }
            }
        } else {
            for (int m = 0, e = lane; e < E; ++m, e += 32) {
                if (taken & (1u << m))
                    continue;
                if (be == INT_MAX || lg[e] > bv) {
                    bv = lg[e];
                    be = e;
                }
            }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oe = __shfl_xor_sync(0xffffffffu, be, off);
            if (oe != INT_MAX && (be == INT_MAX || ov > bv || (ov == bv && oe < be))) {
                bv = ov;
                be = oe;
            }
        }
        if ((be & 31) == lane)
            taken |= 1u << (be >> 5);
        if (lane == c)
            my_c = be;
    }
    // 2. their fixed-order logits, up to eight experts per pass over the token's row
    float my_x = 0.0f;
    for (int c0 = 0; c0 < nc; c0 += 8) {
        int es[8];
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            es[j] = __shfl_sync(0xffffffffu, my_c, min(c0 + j, nc - 1));
        exact_logits8(xrow, Wr, bias, H, es, min(8, nc - c0), lane, v);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (lane == c0 + j)
                my_x = v[j];
    }
    // 3. the k largest candidates by exact value (ties to the lower expert), in lanes 0..k-1
    uint32_t sel = 0;  // bit c: candidate c selected
    float my_v = 0.0f;
    int my_e = 0;
    float vk = 0.0f;
    for (int j = 0; j < k; ++j) {
        float bv = -FLT_MAX;
        int be = INT_MAX, bc = -1;
        if (lane < nc && !(sel & (1u << lane))) {
            bv = my_x;
            be = my_c;
            bc = lane;
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oe = __shfl_xor_sync(0xffffffffu, be, off);
            const int oc = __shfl_xor_sync(0xffffffffu, bc, off);
            if (oe != INT_MAX && (be == INT_MAX || ov > bv || (ov == bv && oe < be))) {
                bv = ov;
                be = oe;
                bc = oc;
            }
        }
        sel |= 1u << bc;
        if (lane == j) {
            my_v = bv;
            my_e = be;
        }
        vk = bv;
    }
    // 4. no other expert may reach the k-th exact value
    bool near = false;
    if (nc < E) {
        for (int m = 0, e = lane; e < E; ++m, e += 32) {
            if (taken & (1u << m))
                continue;
            const float margin = 0x1p-11f * xnorm * wnorm[e] + (bias ? 0x1p-22f * fabsf(bias[e]) : 0.0f);
            if (lg[e] + margin * (1.0f + 0x1p-20f) >= vk)
                near = true;
        }
    }
    if (__any_sync(0xffffffffu, near)) {
        // a near tie: every logit in the fixed order, selected as the other router kernels do
        for (int e0 = 0; e0 < E; e0 += 8) {
            int es[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                es[j] = min(e0 + j, E - 1);
            float v[8];
            exact_logits8(xrow, Wr, bias, H, es, min(8, E - e0), lane, v);
            if (lane == 0)
                for (int j = 0; j < 8 && e0 + j < E; ++j)
                    lg[e0 + j] = v[j];
        }
        __syncwarp();
        if (lane == 0 && fallbacks)
            atomicAdd(fallbacks, 1);
        warp_topk_softmax(lg, E, k, 1, lane, ids + (size_t)t * k, wts + (size_t)t * k);
        return;
    }
    warp_softmax_k(lg, E, k, 1, lane, my_v, my_e, ids + (size_t)t * k, wts + (size_t)t * k);
}

cudaError_t launch_router_tc(const __nv_bfloat16 *x, const __nv_bfloat16 *Wr, const float *bias, int T, int H, int E,
                             int k, int32_t *ids, float *wts, float *scratch, int *status, int pdl_mask,
                             cudaStream_t st)
{
    const int nsm = num_sms_current_device();
    if (nsm <= 0)
        return cudaErrorInvalidDevice;
    const int nsplit = router_tc_splits(T, H, E, nsm);
    const int64_t rows = (T + 127) / 128 * 128;
    float *part = scratch;
    float *wnorm = scratch + (size_t)nsplit * rows * E;
    cudaError_t err = launch_kernel(pdl_site(pdl_mask, kPdlRouter), router_wnorm_kernel, dim3((E + 7) / 8),
                                    dim3(256), 0, st, Wr, H, E, wnorm, status);
    if (err != cudaSuccess)
        return err;
    GemmArgs g;
    memset(&g, 0, sizeof g);
    if (!encode_tmap_2d(&g.tm_x, x, 2, H, T, 64, 128) || !encode_tmap_2d(&g.tm_w, Wr, 2, H, E, 64, 128))
        return cudaErrorInvalidValue;
    g.K = H;
    g.M = (int)rows;
    g.N = E;
    g.E = nsplit;            // K slices
    g.expert_offsets = nullptr;
    g.dw_out = part;
    g.status = status;
    g.tile_counter = nullptr;
    const int64_t tiles = (int64_t)nsplit * (rows / 128) * ((E + 255) / 256);
    err = launch_gemm_backward_bf16(5, g, (int)(tiles < nsm ? tiles : nsm), st);
    if (err != cudaSuccess)
        return err;
    return launch_kernel(pdl_site(pdl_mask, kPdlTopk), router_select_kernel, dim3((T + 7) / 8), dim3(256),
                         sizeof(float) * 8 * E, st, x, Wr, bias, T, H, E, k, part, nsplit, rows, wnorm, ids, wts,
                         status ? status + 4 : nullptr);
}

// ============================================================ align-sort
//
// Small S (<= 1024 slots): one CTA.  Thread e counts expert e's slots, the
// padded lengths are scanned over the experts, and thread e writes its own
// segment in ascending slot order followed by its padding.
//
// Larger S: three launches over chunks of kSortChunk consecutive slots:
//  1. count:   per-chunk histogram of expert ids -> cc[chunk][e]; also
//              pre-fills sorted_ids with the sentinel S and sorted_weights
//              with 0 (grid-stride over all max_padded entries).
//  2. scan:    one CTA.  For each expert the chunk histograms become
//              exclusive prefixes (chunk order), the totals are the expert
//              counts, padded segment lengths ceil(cnt/B)*B are scanned over
//              experts (ascending e), block -> expert ids are written, the
//              compact list of experts with slots is built.
//  3. scatter: each chunk ranks its slots stably (warp match + per-warp
//              counts, ascending slot) and writes slot s to
//              offset[e] + prefix[chunk][e] + rank.

constexpr int kSmallSort = 1024;

size_t sort_scratch_bytes(int T, int k, int E)
{
    const long S = (long)T * k;
    const long nchunks = (S + kSortChunk - 1) / kSortChunk;
    return (size_t)(nchunks > 0 ? nchunks : 1) * E * sizeof(int32_t);
}

// Inclusive Hillis-Steele scans of two 1024-entry shared arrays (one per thread).
__device__ __forceinline__ void scan2_1024(int32_t *a, int32_t *b)
{
    const int i = threadIdx.x;
    for (int off = 1; off < 1024; off <<= 1) {
        const int x = (i >= off) ? a[i - off] : 0;
        const int y = (i >= off) ? b[i - off] : 0;
        __syncthreads();
        a[i] += x;
        b[i] += y;
        __syncthreads();
    }
}

__global__ void __launch_bounds__(1024) sort_small_kernel(const int32_t *__restrict__ ids,
                                                         const float *__restrict__ wts, int S, int E, int B,
                                                         int64_t P_max, int64_t NB_max, SortOut o)
{
    __shared__ int32_t s_ids[kSmallSort];
    __shared__ float s_w[kSmallSort];
    __shared__ int32_t s_pad[1024];
    __shared__ int32_t s_act[1024];
    pdl_wait();
    pdl_trigger();
    const int e = threadIdx.x;
    bool bad_id = false;
    if (e < S) {
        s_ids[e] = ids[e];
        s_w[e] = wts[e];  // staged so the per-expert scatter below waits on no global load
        bad_id = (unsigned)s_ids[e] >= (unsigned)E;
    }
    // an id outside [0, E) matches no expert below, so its slot is left out; it is reported
    // through num_post_padded = -1
    const bool any_bad = __syncthreads_or(bad_id);
    int cnt = 0;
    if (e < E)
        for (int s = 0; s < S; ++s)
            cnt += (s_ids[s] == e);
    const int pad = (cnt + B - 1) / B * B;
    s_pad[e] = (e < E) ? pad : 0;
    s_act[e] = (e < E && cnt > 0) ? 1 : 0;
    __syncthreads();
    scan2_1024(s_pad, s_act);
    const int off = s_pad[e] - ((e < E) ? pad : 0);
    const int total = s_pad[1023];
    if (e < E) {
        if (o.expert_counts)
            o.expert_counts[e] = cnt;
        if (o.expert_offsets)
            o.expert_offsets[e] = off;
        if (o.active_experts && cnt > 0)
            o.active_experts[s_act[e] - 1] = e;
        int pos = off;
        for (int s = 0; s < S; ++s)
            if (s_ids[s] == e) {
                o.sorted_ids[pos] = s;
                o.sorted_weights[pos] = s_w[s];
                if (o.slot_pos)
                    o.slot_pos[s] = pos;
                ++pos;
            }
        for (; pos < off + pad; ++pos) {
            o.sorted_ids[pos] = S;
            o.sorted_weights[pos] = 0.0f;
        }
        for (int b = off / B; b < (off + pad) / B; ++b)
            o.sorted_expert_ids[b] = e;
    }
    if (e == 0) {
        *o.num_post_padded = any_bad ? -1 : total;
        if (o.expert_offsets)
            o.expert_offsets[E] = total;
        if (o.num_active)
            *o.num_active = s_act[1023];
    }
    for (int64_t i = total + e; i < P_max; i += 1024) {
        o.sorted_ids[i] = S;
        o.sorted_weights[i] = 0.0f;
    }
    for (int64_t b = total / B + e; b < NB_max; b += 1024)
        o.sorted_expert_ids[b] = -1;
}

// Few experts (E <= 32) and small S: the same outputs as sort_small_kernel, with the
// per-expert counts scanned by one warp's shuffles instead of a 1024-thread block scan
// (twenty block barriers), so the CTA is 256 threads.  Every decode step runs it.
__global__ void __launch_bounds__(256) sort_few_kernel(const int32_t *__restrict__ ids,
                                                       const float *__restrict__ wts, int S, int E, int B,
                                                       int64_t P_max, int64_t NB_max, SortOut o)
{
    __shared__ int32_t s_ids[kSmallSort];
    __shared__ float s_w[kSmallSort];
    __shared__ int s_total;
    pdl_wait();
    pdl_trigger();
    bool bad_id = false;
    for (int i = threadIdx.x; i < S; i += blockDim.x) {
        s_ids[i] = ids[i];
        s_w[i] = wts[i];
        bad_id |= (unsigned)s_ids[i] >= (unsigned)E;  // matches no expert below: left out, reported
    }
    const bool any_bad = __syncthreads_or(bad_id);
    if (threadIdx.x < 32) {
        const int e = threadIdx.x;
        int cnt = 0;
        if (e < E)
            for (int s = 0; s < S; ++s)
                cnt += (s_ids[s] == e);
        const int pad = (e < E) ? (cnt + B - 1) / B * B : 0;
        const int act = (e < E && cnt > 0) ? 1 : 0;
        int ipad = pad, iact = act;  // inclusive scans over the experts
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int vp = __shfl_up_sync(0xffffffffu, ipad, d);
            const int va = __shfl_up_sync(0xffffffffu, iact, d);
            if (e >= d) {
                ipad += vp;
                iact += va;
            }
        }
        const int off = ipad - pad;
        const int total = __shfl_sync(0xffffffffu, ipad, 31);
        const int nact = __shfl_sync(0xffffffffu, iact, 31);
        if (e < E) {
            if (o.expert_counts)
                o.expert_counts[e] = cnt;
            if (o.expert_offsets)
                o.expert_offsets[e] = off;
            if (o.active_experts && cnt > 0)
                o.active_experts[iact - 1] = e;
            int pos = off;
            for (int s = 0; s < S; ++s)
                if (s_ids[s] == e) {
                    o.sorted_ids[pos] = s;
                    o.sorted_weights[pos] = s_w[s];
                    if (o.slot_pos)
                        o.slot_pos[s] = pos;
                    ++pos;
                }
            for (; pos < off + pad; ++pos) {
                o.sorted_ids[pos] = S;
                o.sorted_weights[pos] = 0.0f;
            }
            for (int b = off / B; b < (off + pad) / B; ++b)
                o.sorted_expert_ids[b] = e;
        }
        if (e == 0) {
            *o.num_post_padded = any_bad ? -1 : total;
            if (o.expert_offsets)
                o.expert_offsets[E] = total;
            if (o.num_active)
                *o.num_active = nact;
            s_total = total;
        }
    }
    __syncthreads();
    const int total = s_total;
    for (int64_t i = total + threadIdx.x; i < P_max; i += blockDim.x) {
        o.sorted_ids[i] = S;
        o.sorted_weights[i] = 0.0f;
    }
    for (int64_t b = total / B + threadIdx.x; b < NB_max; b += blockDim.x)
        o.sorted_expert_ids[b] = -1;
}

__global__ void __launch_bounds__(1024) sort_count_kernel(const int32_t *__restrict__ ids, int S, int E,
                                                         int32_t *__restrict__ cc,
                                                         int32_t *__restrict__ sorted_ids,
                                                         float *__restrict__ sorted_w, int64_t P_max)
{
    extern __shared__ int32_t s_hist[];
    pdl_wait();
    pdl_trigger();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        s_hist[e] = 0;
    __syncthreads();
    const int s = blockIdx.x * kSortChunk + threadIdx.x;
    if (s < S) {
        const int e = ids[s];
        if ((unsigned)e < (unsigned)E)  // a bad id is not counted; the scan sees the shortfall
            atomicAdd(&s_hist[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        cc[(size_t)blockIdx.x * E + e] = s_hist[e];
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < P_max; i += (int64_t)gridDim.x * blockDim.x) {
        sorted_ids[i] = S;
        sorted_w[i] = 0.0f;
    }
}

__global__ void __launch_bounds__(1024) sort_scan_kernel(int32_t *__restrict__ cc, int nchunks, int S, int E,
                                                        int B, int64_t NB_max, SortOut o)
{
    __shared__ int32_t s_pad[1024];
    __shared__ int32_t s_act[1024];
    __shared__ int s_counted;
    pdl_wait();
    pdl_trigger();
    const int e = threadIdx.x;
    if (e == 0)
        s_counted = 0;
    int cnt = 0;
    if (e < E) {
        // eight chunk counts in flight per round (each round one L2 round trip, not eight)
        for (int c0 = 0; c0 < nchunks; c0 += 8) {
            int v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                v[j] = c0 + j < nchunks ? cc[(size_t)(c0 + j) * E + e] : 0;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (c0 + j < nchunks) {
                    cc[(size_t)(c0 + j) * E + e] = cnt;
                    cnt += v[j];
                }
        }
    }
    const int pad = (e < E) ? (cnt + B - 1) / B * B : 0;
    s_pad[e] = pad;
    s_act[e] = (e < E && cnt > 0) ? 1 : 0;
    __syncthreads();
    if (cnt)
        atomicAdd(&s_counted, cnt);  // fewer than S counted slots: some id was outside [0, E)
    scan2_1024(s_pad, s_act);
    const int pad_incl = s_pad[e];
    const int pad_excl = pad_incl - pad;
    if (e < E) {
        if (o.expert_counts)
            o.expert_counts[e] = cnt;
        o.expert_offsets[e] = pad_excl;
        if (o.active_experts && cnt > 0)
            o.active_experts[s_act[e] - 1] = e;
        for (int b = pad_excl / B; b < pad_incl / B; ++b)
            o.sorted_expert_ids[b] = e;
    }
    const int total = s_pad[1023];
    if (e == 0) {
        *o.num_post_padded = (s_counted == S) ? total : -1;
        o.expert_offsets[E] = total;
        if (o.num_active)
            *o.num_active = s_act[1023];
    }
    for (int64_t b = total / B + e; b < NB_max; b += blockDim.x)
        o.sorted_expert_ids[b] = -1;
}

__global__ void __launch_bounds__(1024) sort_scatter_kernel(const int32_t *__restrict__ ids,
                                                           const float *__restrict__ wts, int S, int E,
                                                           const int32_t *__restrict__ cc, SortOut o)
{
    extern __shared__ int32_t s_wc[];  // [32 warps][E] per-warp counts -> exclusive prefixes over warps
    pdl_wait();
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < 32 * E; i += blockDim.x)
        s_wc[i] = 0;
    __syncthreads();
    const int s = blockIdx.x * kSortChunk + threadIdx.x;
    const int e_in = s < S ? ids[s] : -1;
    const bool valid = (unsigned)e_in < (unsigned)E;  // past S or a bad id: not placed
    const int e = valid ? e_in : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (valid && rank == 0)
        s_wc[warp * E + e] = __popc(peers);
    __syncthreads();
    for (int ex = threadIdx.x; ex < E; ex += blockDim.x) {
        int run = 0;
        for (int w = 0; w < 32; ++w) {
            const int v = s_wc[w * E + ex];
            s_wc[w * E + ex] = run;
            run += v;
        }
    }
    __syncthreads();
    if (valid) {
        const int pos = o.expert_offsets[e] + cc[(size_t)blockIdx.x * E + e] + s_wc[warp * E + e] + rank;
        o.sorted_ids[pos] = s;
        o.sorted_weights[pos] = wts[s];
        if (o.slot_pos)
            o.slot_pos[s] = pos;
    }
}

// o.expert_offsets must be non-null (the scatter reads it).
cudaError_t launch_align_sort(const int32_t *ids, const float *wts, int T, int k, int E, int block_m,
                              const SortOut &o, void *scratch, bool pdl, bool pdl_inner, cudaStream_t st)
{
    const int S = T * k;
    const int64_t P_max = (int64_t)S + (int64_t)E * block_m - k;
    const int64_t NB_max = (P_max + block_m - 1) / block_m;
    if (S <= kSmallSort && E <= 32)
        return launch_kernel(pdl, sort_few_kernel, dim3(1), dim3(256), 0, st, ids, wts, S, E, block_m, P_max,
                             NB_max, o);
    if (S <= kSmallSort)
        return launch_kernel(pdl, sort_small_kernel, dim3(1), dim3(1024), 0, st, ids, wts, S, E, block_m, P_max,
                             NB_max, o);
    const int nchunks = (S + kSortChunk - 1) / kSortChunk;
    int32_t *cc = static_cast<int32_t *>(scratch);
    cudaError_t err = launch_kernel(pdl, sort_count_kernel, dim3(nchunks), dim3(1024), sizeof(int32_t) * E, st, ids,
                                    S, E, cc, o.sorted_ids, o.sorted_weights, P_max);
    if (err != cudaSuccess)
        return err;
    err = launch_kernel(pdl_inner, sort_scan_kernel, dim3(1), dim3(1024), 0, st, cc, nchunks, S, E, block_m, NB_max,
                        o);
    if (err != cudaSuccess)
        return err;
    const size_t smem = sizeof(int32_t) * 32 * E;
    if (smem > 48 * 1024) {
        err = cudaFuncSetAttribute(sort_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess)
            return err;
    }
    return launch_kernel(pdl_inner, sort_scatter_kernel, dim3(nchunks), dim3(1024), smem, st, ids, wts, S, E, cc, o);
}

// ================================================================ gather

__global__ void __launch_bounds__(256) gather_rows_kernel(const __nv_bfloat16 *__restrict__ x,
                                                         const int32_t *__restrict__ sorted_ids,
                                                         const int32_t *__restrict__ npp, int S, int k, int H,
                                                         __nv_bfloat16 *__restrict__ xs, int zero_padding)
{
    pdl_wait();
    pdl_trigger();
    const int rows = *npp;
    const int nvec = H / 8;
    constexpr int U = 4;  // 16-byte pieces a thread requests before storing any (H <= 8192 in one round)
    for (int i = blockIdx.x; i < rows; i += gridDim.x) {
        const int s = sorted_ids[i];
        if (s >= S && !zero_padding)
            continue;  // a padding row: its GEMM results are discarded, so its contents do not matter
        uint4 *dst = reinterpret_cast<uint4 *>(xs + (size_t)i * H);
        const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)(s < S ? s / k : 0) * H);
        for (int c0 = threadIdx.x; c0 < nvec; c0 += U * blockDim.x) {
            uint4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * blockDim.x;
                v[u] = (s < S && c < nvec) ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * blockDim.x;
                if (c < nvec)
                    dst[c] = v[u];
            }
        }
    }
}

cudaError_t launch_gather_rows(const __nv_bfloat16 *x, const int32_t *sorted_ids, const int32_t *npp, int S, int k,
                               int H, int64_t P_max, __nv_bfloat16 *xs, bool zero_padding, bool pdl, cudaStream_t st)
{
    int grid = (int)(P_max < 8192 ? P_max : 8192);
    if (grid < 1)
        grid = 1;
    return launch_kernel(pdl, gather_rows_kernel, dim3(grid), dim3(256), 0, st, x, sorted_ids, npp, S, k, H, xs,
                         zero_padding ? 1 : 0);
}

// ---------------------------------------------------- FP8 quantisation
//
// Group quantisation with scale = amax / 448 (1 if amax is 0) and codes
// e4m3(v / scale), round-to-nearest-even, saturating (satfinite).  The
// division is IEEE (the library is built without fast-math).

__device__ __forceinline__ float group_scale(float amax) { return amax > 0.0f ? amax / 448.0f : 1.0f; }

__device__ __forceinline__ uint2 encode8(const float (&f)[8], float scale)
{
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t c = __nv_cvt_float_to_fp8(f[i] / scale, __NV_SATFINITE, __NV_E4M3);
        lo |= c << (8 * i);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t c = __nv_cvt_float_to_fp8(f[4 + i] / scale, __NV_SATFINITE, __NV_E4M3);
        hi |= c << (8 * i);
    }
    return make_uint2(lo, hi);
}

// One 16-lane segment handles one 128-column group (8 columns per lane).
__device__ __forceinline__ float seg16_max(float v)
{
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

__device__ __forceinline__ float absmax8(const float (&f)[8])
{
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        m = fmaxf(m, fabsf(f[i]));
    return m;
}

// Rows of X [R][C] quantised per 1x128: codes q [R][C], scales s [R][C/128].
__global__ void __launch_bounds__(256) quant_act_kernel(const __nv_bfloat16 *__restrict__ X, int64_t R, int C,
                                                       uint8_t *__restrict__ q, float *__restrict__ s)
{
    const int nvec = C / 8;
    const int64_t total = R * nvec;
    // 256 threads cover 16 groups; every 16 consecutive vectors form one group
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v - threadIdx.x < total;
         v += (int64_t)gridDim.x * blockDim.x) {
        const bool ok = v < total;
        float f[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (ok)
            bf16x8_to_float(__ldg(reinterpret_cast<const uint4 *>(X) + v), f);
        const float sc = group_scale(seg16_max(absmax8(f)));
        if (ok) {
            reinterpret_cast<uint2 *>(q)[v] = encode8(f, sc);
            if ((v & 15) == 0)
                s[v / 16] = sc;
        }
    }
}

void launch_quant_act(const __nv_bfloat16 *X, int64_t R, int C, uint8_t *q, float *s, cudaStream_t st)
{
    const int64_t total = R * (C / 8);
    int64_t grid = (total + 255) / 256;
    if (grid > 65535)
        grid = 65535;
    if (grid < 1)
        return;
    quant_act_kernel<<<(int)grid, 256, 0, st>>>(X, R, C, q, s);
}

// Gathered rows quantised per 1x128: q [P_max][H] in sorted order, scales
// transposed sT [H/128][P_max] so that a GEMM tile reads them coalesced.
__global__ void __launch_bounds__(256) gather_quant_kernel(const __nv_bfloat16 *__restrict__ x,
                                                          const int32_t *__restrict__ sorted_ids,
                                                          const int32_t *__restrict__ npp, int S, int k, int H,
                                                          int64_t P_max, uint8_t *__restrict__ q,
                                                          float *__restrict__ sT)
{
    pdl_wait();
    pdl_trigger();
    const int rows = *npp;
    const int nvec = H / 8;
    constexpr int U = 2;  // 16-byte pieces a thread requests before encoding any (H <= 4096 in one round)
    for (int i = blockIdx.x; i < rows; i += gridDim.x) {
        const int s = sorted_ids[i];
        const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)(s < S ? s / k : 0) * H);
        for (int c0 = 0; c0 < nvec; c0 += U * blockDim.x) {
            uint4 raw[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * blockDim.x + threadIdx.x;
                raw[u] = (c < nvec && s < S) ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * blockDim.x + threadIdx.x;
                float f[8];
                bf16x8_to_float(raw[u], f);  // zero pieces past the row or for padding convert to 0
                const float sc = group_scale(seg16_max(absmax8(f)));
                if (c < nvec) {
                    reinterpret_cast<uint2 *>(q + (size_t)i * H)[c] = encode8(f, sc);
                    if ((c & 15) == 0)
                        sT[(size_t)(c / 16) * P_max + i] = sc;
                }
            }
        }
    }
}

cudaError_t launch_gather_quant_rows(const __nv_bfloat16 *x, const int32_t *sorted_ids, const int32_t *npp, int S,
                                     int k, int H, int64_t P_max, uint8_t *q, float *sT, bool pdl, cudaStream_t st)
{
    int grid = (int)(P_max < 8192 ? P_max : 8192);
    if (grid < 1)
        grid = 1;
    return launch_kernel(pdl, gather_quant_kernel, dim3(grid), dim3(256), 0, st, x, sorted_ids, npp, S, k, H, P_max,
                         q, sT);
}

// One scale per row ("per_Token"): a CTA per row, amax over the whole row,
// then codes.  With sorted_ids the rows are gathered (row i is token
// sorted_ids[i] / k, a zero row with scale 1 for padding); with nrows the row
// count is read on the device (the rows past it are never used).  NV > 0
// keeps the row in registers between the two passes (C <= 256 * 8 * NV; the
// launch takes the smallest NV of 2, 4, 8 that holds the row, since unused
// register slots cost resident rows: activation rows of 4096 went 55 -> 36 us
// at 8192 rows with NV = 2 instead of 8); NV = 0 reads it twice.
template <int NV>
__global__ void __launch_bounds__(256) quant_rows_kernel(const __nv_bfloat16 *__restrict__ X,
                                                        const int32_t *__restrict__ sorted_ids,
                                                        const int32_t *__restrict__ nrows, int64_t R, int S,
                                                        int k, int C, uint8_t *__restrict__ q,
                                                        float *__restrict__ s, float *__restrict__ zero_rows)
{
    __shared__ float s_red[8];
    pdl_wait();
    pdl_trigger();
    const int64_t rows = nrows ? (int64_t)*nrows : R;
    if (zero_rows && threadIdx.x == 0)
        for (int64_t r = blockIdx.x; r < rows; r += gridDim.x)
            zero_rows[r] = 0.0f;
    const int nvec = C / 8;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        bool zero = false;
        int64_t src_row = r;
        if (sorted_ids) {
            const int sl = sorted_ids[r];
            zero = sl >= S;
            src_row = zero ? 0 : sl / k;
        }
        const uint4 *src = reinterpret_cast<const uint4 *>(X + src_row * C);
        uint2 *dst = reinterpret_cast<uint2 *>(q + r * C);
        float m = 0.0f;
        uint4 v[NV > 0 ? NV : 1];
        if (NV > 0) {
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int c = threadIdx.x + i * 256;
                v[i] = (c < nvec && !zero) ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
                float f[8];
                bf16x8_to_float(v[i], f);
                m = fmaxf(m, absmax8(f));
            }
        } else if (!zero) {
#pragma unroll 4
            for (int c = threadIdx.x; c < nvec; c += 256) {
                float f[8];
                bf16x8_to_float(__ldg(src + c), f);
                m = fmaxf(m, absmax8(f));
            }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1)
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        if (lane == 0)
            s_red[warp] = m;
        __syncthreads();
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            amax = fmaxf(amax, s_red[i]);
        const float sc = group_scale(amax);
        if (NV > 0) {
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int c = threadIdx.x + i * 256;
                if (c < nvec) {
                    float f[8];
                    bf16x8_to_float(v[i], f);
                    dst[c] = encode8(f, sc);
                }
            }
        } else {
#pragma unroll 4
            for (int c = threadIdx.x; c < nvec; c += 256) {
                float f[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                if (!zero)
                    bf16x8_to_float(__ldg(src + c), f);
                dst[c] = encode8(f, sc);
            }
        }
        if (threadIdx.x == 0)
            s[r] = sc;
        __syncthreads();  // s_red is rewritten for the next row
    }
}

cudaError_t launch_quant_rows(const __nv_bfloat16 *X, const int32_t *sorted_ids, const int32_t *nrows, int64_t R,
                              int S, int k, int C, uint8_t *q, float *s, bool pdl, cudaStream_t st, float *zero_rows)
{
    int64_t grid = R < 16384 ? R : 16384;
    if (grid < 1)
        return cudaSuccess;
    if (C <= 256 * 8 * 2)
        return launch_kernel(pdl, quant_rows_kernel<2>, dim3((unsigned)grid), dim3(256), 0, st, X, sorted_ids, nrows,
                             R, S, k, C, q, s, zero_rows);
    if (C <= 256 * 8 * 4)
        return launch_kernel(pdl, quant_rows_kernel<4>, dim3((unsigned)grid), dim3(256), 0, st, X, sorted_ids, nrows,
                             R, S, k, C, q, s, zero_rows);
    if (C <= 256 * 8 * 8)
        return launch_kernel(pdl, quant_rows_kernel<8>, dim3((unsigned)grid), dim3(256), 0, st, X, sorted_ids, nrows,
                             R, S, k, C, q, s, zero_rows);
    return launch_kernel(pdl, quant_rows_kernel<0>, dim3((unsigned)grid), dim3(256), 0, st, X, sorted_ids, nrows, R,
                         S, k, C, q, s, zero_rows);
}

// Rows whose max |v| is already known (the per-token FP8 intermediate: the stage-1 epilogue takes
// each row's max |h| by atomicMax): no reduction, so no barrier between a row's loads and its
// codes; a CTA streams whole rows, several 16-byte loads in flight per thread.
__global__ void __launch_bounds__(256) quant_rows_amax_kernel(const __nv_bfloat16 *__restrict__ X,
                                                             const float *__restrict__ row_amax,
                                                             const int32_t *__restrict__ nrows, int C,
                                                             uint8_t *__restrict__ q, float *__restrict__ s)
{
    pdl_wait();
    pdl_trigger();
    const int64_t rows = *nrows;
    const int nvec = C / 8;
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const float sc = group_scale(row_amax[r]);
        const uint4 *src = reinterpret_cast<const uint4 *>(X + r * C);
        uint2 *dst = reinterpret_cast<uint2 *>(q + r * C);
#pragma unroll 4
        for (int c = threadIdx.x; c < nvec; c += 256) {
            float f[8];
            bf16x8_to_float(__ldg(src + c), f);
            dst[c] = encode8(f, sc);
        }
        if (threadIdx.x == 0)
            s[r] = sc;
    }
}

cudaError_t launch_quant_rows_amax(const __nv_bfloat16 *X, const float *row_amax, const int32_t *nrows, int64_t R,
                                   int C, uint8_t *q, float *s, bool pdl, cudaStream_t st)
{
    const int64_t grid = R < 16384 ? R : 16384;
    if (grid < 1)
        return cudaSuccess;
    return launch_kernel(pdl, quant_rows_amax_kernel, dim3((unsigned)grid), dim3(256), 0, st, X, row_amax, nrows, C,
                         q, s);
}

// One CTA per 128x128 block of W [R][C]: amax over the block, then codes.
__global__ void __launch_bounds__(256) quant_weight_kernel(const __nv_bfloat16 *__restrict__ W, int C,
                                                          uint8_t *__restrict__ q, float *__restrict__ s)
{
    __shared__ float s_red[8];
    const int64_t br = blockIdx.y;
    const int bc = blockIdx.x;
    const int GC = C / 128;
    // thread -> row r = tid / 2 (0..127), half = tid % 2 (64 columns)
    const int r = threadIdx.x >> 1, half = threadIdx.x & 1;
    const __nv_bfloat16 *row = W + (br * 128 + r) * (int64_t)C + bc * 128 + half * 64;
    float f[8][8];
    float m = 0.0f;
#pragma unroll
    for (int v = 0; v < 8; ++v) {
        bf16x8_to_float(__ldg(reinterpret_cast<const uint4 *>(row) + v), f[v]);
        m = fmaxf(m, absmax8(f[v]));
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if ((threadIdx.x & 31) == 0)
        s_red[threadIdx.x >> 5] = m;
    __syncthreads();
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        amax = fmaxf(amax, s_red[i]);
    const float sc = group_scale(amax);
    uint8_t *qrow = q + (br * 128 + r) * (int64_t)C + bc * 128 + half * 64;
#pragma unroll
    for (int v = 0; v < 8; ++v)
        reinterpret_cast<uint2 *>(qrow)[v] = encode8(f[v], sc);
    if (threadIdx.x == 0)
        s[br * GC + bc] = sc;
}

void launch_quant_weights(const __nv_bfloat16 *W, int64_t R, int C, uint8_t *q, float *s, cudaStream_t st)
{
    if (R <= 0)
        return;
    dim3 grid(C / 128, (unsigned)(R / 128));
    quant_weight_kernel<<<grid, 256, 0, st>>>(W, C, q, s);
}


}  // namespace moe
