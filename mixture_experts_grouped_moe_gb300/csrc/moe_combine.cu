// The weighted combine of the fused MoE layer (AITER walk-through, section 3:
// gating -> token reorder -> expert GEMMs -> weighted combine): each token's k
// weighted expert rows summed in a fixed order (j ascending, fp32) and
// rounded to bf16 once; and the split-K form, which also sums the K splits
// of stage 2 and applies the top-k weights.  No atomics, so every result is
// bitwise reproducible.  (A translation unit of its own: code generation of
// the latency-bound router kernels is sensitive to what else a unit holds.)
#include "moe_internal.h"

namespace moe {

__device__ __forceinline__ void unpack_bf16x8(const uint4 &v, float (&f)[8])
{
    const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __bfloat1622float2(p[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ uint2 pack_bf16x4(const float4 &a)
{
    __nv_bfloat162 lo = __floats2bfloat162_rn(a.x, a.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(a.z, a.w);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t *>(&lo);
    pk.y = *reinterpret_cast<uint32_t *>(&hi);
    return pk;
}

// out[t] = sum_j Y[t*k + j] (j ascending, fp32) -> bf16; eight columns per thread (16-byte
// loads of the bf16 slot rows, one 16-byte store)
__global__ void __launch_bounds__(256) combine_kernel(const __nv_bfloat16 *__restrict__ Y, int T, int k, int H,
                                                     __nv_bfloat16 *__restrict__ out)
{
    pdl_wait();
    pdl_trigger();
    const int nv = H / 8;
    const int64_t total = (int64_t)T * nv;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / nv;
        const int c = (int)(i % nv);
        const uint4 *src = reinterpret_cast<const uint4 *>(Y) + (t * k) * nv + c;
        float a[8];
        unpack_bf16x8(__ldg(src), a);
        for (int j = 1; j < k; ++j) {
            float b[8];
            unpack_bf16x8(__ldg(src + (int64_t)j * nv), b);
#pragma unroll
            for (int q = 0; q < 8; ++q)
                a[q] += b[q];
        }
        const uint2 lo = pack_bf16x4(make_float4(a[0], a[1], a[2], a[3]));
        const uint2 hi = pack_bf16x4(make_float4(a[4], a[5], a[6], a[7]));
        reinterpret_cast<uint4 *>(out)[i] = make_uint4(lo.x, lo.y, hi.x, hi.y);
    }
}

cudaError_t launch_combine(const __nv_bfloat16 *Y, int T, int k, int H, __nv_bfloat16 *out, bool pdl,
                           cudaStream_t st)
{
    const int64_t total = (int64_t)T * (H / 8);
    int64_t grid = (total + 255) / 256;
    if (grid > 152 * 16)
        grid = 152 * 16;
    if (grid < 1)
        return cudaSuccess;
    return launch_kernel(pdl, combine_kernel, dim3((unsigned)grid), dim3(256), 0, st, Y, T, k, H, out);
}

__global__ void __launch_bounds__(256) splitk_combine_kernel(const float *__restrict__ P, int SK, int64_t P_rows,
                                                            const int32_t *__restrict__ slot_pos,
                                                            const float *__restrict__ wts, int T, int k, int H,
                                                            __nv_bfloat16 *__restrict__ out)
{
    pdl_wait();
    pdl_trigger();
    const int nv = H / 4;
    const int64_t total = (int64_t)T * nv;
    const int64_t split_stride = P_rows * nv;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / nv;
        const int c = (int)(i % nv);
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < k; ++j) {
            const int64_t s = t * k + j;
            const float4 *src = reinterpret_cast<const float4 *>(P) + (int64_t)slot_pos[s] * nv + c;
            float4 p = __ldg(src);
            for (int ks = 1; ks < SK; ++ks) {
                const float4 b = __ldg(src + ks * split_stride);
                p.x += b.x;
                p.y += b.y;
                p.z += b.z;
                p.w += b.w;
            }
            const float w = wts[s];
            a.x += w * p.x;
            a.y += w * p.y;
            a.z += w * p.z;
            a.w += w * p.w;
        }
        reinterpret_cast<uint2 *>(out)[i] = pack_bf16x4(a);
    }
}

cudaError_t launch_splitk_combine(const float *P, int SK, int64_t P_rows, const int32_t *slot_pos, const float *wts,
                                  int T, int k, int H, __nv_bfloat16 *out, bool pdl, cudaStream_t st)
{
    const int64_t total = (int64_t)T * (H / 4);
    int64_t grid = (total + 255) / 256;
    if (grid > 152 * 16)
        grid = 152 * 16;
    if (grid < 1)
        return cudaSuccess;
    return launch_kernel(pdl, splitk_combine_kernel, dim3((unsigned)grid), dim3(256), 0, st, P, SK, P_rows, slot_pos,
                         wts, T, k, H, out);
}

}  // namespace moe
