// Token rows of x in the experts' sorted order (the token reorder of the AITER
// walk-through, section 3.1, feeding the expert GEMMs), walked token by token:
// each row of x is read once and written to its k sorted positions (the slot ->
// position map of the sort), so x itself is read from memory once however its
// k copies fall in expert order.  Padding positions are not written: a GEMM
// output row depends only on its own input row, and the results of padding
// rows are never stored.  (The training forward, whose weight gradients sum
// over every position, zeroes the padding rows with the position-major gather
// instead.)
#include "moe_internal.h"

namespace moe {

constexpr int kGatherMaxK = 32;

__global__ void __launch_bounds__(256) gather_by_token_kernel(const __nv_bfloat16 *__restrict__ x,
                                                             const int32_t *__restrict__ slot_pos, int T, int k,
                                                             int H, int64_t P_max, __nv_bfloat16 *__restrict__ xs)
{
    __shared__ int s_pos[kGatherMaxK];
    pdl_wait();
    pdl_trigger();
    const int nvec = H / 8;
    constexpr int U = 4;  // 16-byte pieces a thread loads before storing any (H <= 8192 in one round)
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        __syncthreads();  // the previous token's positions are no longer read
        if (threadIdx.x < k)
            s_pos[threadIdx.x] = slot_pos[(size_t)t * k + threadIdx.x];
        __syncthreads();
        const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)t * H);
        for (int c0 = threadIdx.x; c0 < nvec; c0 += U * blockDim.x) {
            uint4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * blockDim.x;
                v[u] = c < nvec ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
            }
            for (int j = 0; j < k; ++j) {
                const int pos = s_pos[j];
                if ((uint32_t)pos >= (uint64_t)P_max)
                    continue;  // not a position of the sort's output (never from a valid sort)
                uint4 *dst = reinterpret_cast<uint4 *>(xs + (size_t)pos * H);
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int c = c0 + u * blockDim.x;
                    if (c < nvec)
                        dst[c] = v[u];
                }
            }
        }
    }
}

cudaError_t launch_gather_by_token(const __nv_bfloat16 *x, const int32_t *slot_pos, int T, int k, int H,
                                   int64_t P_max, __nv_bfloat16 *xs, bool pdl, cudaStream_t st)
{
    if (k > kGatherMaxK)
        return cudaErrorInvalidValue;
    const int grid = T < 8192 ? T : 8192;
    if (grid < 1)
        return cudaSuccess;
    return launch_kernel(pdl, gather_by_token_kernel, dim3(grid), dim3(256), 0, st, x, slot_pos, T, k, H, P_max, xs);
}

}  // namespace moe
