// Pieces shared by the group-GEMM kernels (one-SM and two-SM forms): the K
// step of a pipeline stage, the MMA of each input type (bf16 / per-token
// FP8), and the epilogue helpers.
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

#include "sm100_ptx.cuh"

namespace moe {

// K elements per pipeline stage: 128 bytes of a row, i.e. 64 bf16 (QT = 0)
// or 128 e4m3 (QT = 1) elements -- one 128-byte swizzle row either way.
template <int QT>
constexpr int kBK = QT ? 128 : 64;

// One tcgen05 MMA of 32 bytes of K: kind::f16 (bf16) or kind::f8f6f4 (e4m3).
template <int QT>
__device__ __forceinline__ void mma_kind(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t accum)
{
    if (QT)
        mma_fp8(d, ad, bd, idesc, accum);
    else
        mma_bf16(d, ad, bd, idesc, accum);
}

// sigmoid(g) = 0.5 + 0.5 tanh(g / 2) on one special-function instruction (tanh.approx, relative
// error near 2^-11), for epilogues bound by that unit whose results are rounded to bf16 next.
__device__ __forceinline__ float sigmoid_fast(float g)
{
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * g));
    return fmaf(0.5f, t, 0.5f);
}

// silu(g) = g sigmoid(g), the sigmoid as above: every SwiGLU epilogue rounds h to bf16 (or
// quantises it) right after, a relative step of 2^-9 or more against the sigmoid's 2^-11.
__device__ __forceinline__ float silu(float g) { return g * sigmoid_fast(g); }

// 32 fp32 values -> 32 bf16 (round to nearest even) at a 16-byte aligned address.
__device__ __forceinline__ void store_bf16x32(__nv_bfloat16 *dst, const float (&h)[32])
{
    uint4 *d = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 p = __floats2bfloat162_rn(h[q * 8 + 2 * i], h[q * 8 + 2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t *>(&p);
        }
        d[q] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// s * v[0..7] -> 8 bf16 (round to nearest even), returned as the bits of a float4 (one
// 16-byte store or shared-memory slot).
__device__ __forceinline__ float4 pack_bf16x8(const float *v, float s)
{
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 p = __floats2bfloat162_rn(s * v[2 * i], s * v[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t *>(&p);
    }
    return make_float4(__uint_as_float(w[0]), __uint_as_float(w[1]), __uint_as_float(w[2]), __uint_as_float(w[3]));
}

// Per-channel or per-token scales (per-token FP8) of 4 consecutive columns;
// channel and token bases are multiples of 16, so the address is 16-byte aligned.
__device__ __forceinline__ float4 ld_scale4(const float *p) { return __ldg(reinterpret_cast<const float4 *>(p)); }

}  // namespace moe
