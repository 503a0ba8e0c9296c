// Backward of the bf16 fused MoE layer (training): the "dgrad" of both
// group GEMMs, the "wgrad" of both weight stacks, and the router, for
// loss = sum(dout * out) -- the pages' stated future work for the group-GEMM
// MoE kernels (FlyDSL-JAX talk, outlook; Jaxator talk, weight-gradient pass).
//
// A training forward (moe_fused_forward_train) runs the grouped path and
// keeps, in its workspace, the routing, the sorted activations x_s, the
// pre-activations g | u, h and the weighted stage-2 rows Y.  The backward:
//   dY_p = w_p dout_t (sorted order)          D_s = dout_t . Y_s
//   dl   = softmax backward over the chosen k from the D_s (dlogit, zero elsewhere)
//   dh   = dY W_down            -> SwiGLU backward in the GEMM epilogue -> dg | du
//   dx_s = dg W_gate + du W_up  (stage 2's tile shape, unit weights)
//   dx_t = sum_j dx_{t,j} + sum_j dl_j W_router[e_j]
//   dW_down[e] = dY_e^T h_e, dW_gate_up[e] = (dg|du)_e^T x_e  (K over e's tokens)
//   dW_router = dlogit^T x, dbias = column sums of dlogit
// Every GEMM keeps both operands K-major, the form the tcgen05 kernels take:
// the weights are transposed once per call ([E][I][H] and [E][H][2I]) and
// the activations of the weight gradients are transposed into [rows][P].
#include <cstring>

#include "moe_internal.h"

namespace moe {

namespace {

__device__ __forceinline__ float bf2f(__nv_bfloat16 v) { return __bfloat162float(v); }

// dY rows in sorted order: dY_p = w_p * dout[t_p] (bf16), zero for padding.
__global__ void __launch_bounds__(256) dy_gather_kernel(const __nv_bfloat16 *__restrict__ dout,
                                                       const int32_t *__restrict__ sorted_ids,
                                                       const float *__restrict__ sorted_w,
                                                       const int32_t *__restrict__ npp, int S, int k, int H,
                                                       __nv_bfloat16 *__restrict__ dys)
{
    const int rows = *npp;
    const int nvec = H / 8;
    for (int p = blockIdx.x; p < rows; p += gridDim.x) {
        const int s = sorted_ids[p];
        uint4 *dst = reinterpret_cast<uint4 *>(dys + (size_t)p * H);
        if (s >= S) {
            for (int c = threadIdx.x; c < nvec; c += blockDim.x)
                dst[c] = make_uint4(0, 0, 0, 0);
            continue;
        }
        const float w = sorted_w[p];
        const uint4 *src = reinterpret_cast<const uint4 *>(dout + (size_t)(s / k) * H);
        for (int c = threadIdx.x; c < nvec; c += blockDim.x) {
            uint4 v = src[c];
            __nv_bfloat162 *h2 = reinterpret_cast<__nv_bfloat162 *>(&v);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __bfloat1622float2(h2[i]);
                h2[i] = __floats2bfloat162_rn(w * f.x, w * f.y);
            }
            dst[c] = v;
        }
    }
}

// One warp per token.  With D_j = dout_t . Y_{t,j} (Y holds the weighted rows
// w_j y_j), the softmax backward dl_j = w_j (dw_j - sum_m w_m dw_m), dw_j =
// dout_t . y_j, is dl_j = D_j - w_j sum_m D_m; written to dlogit[t][e_j].
__global__ void __launch_bounds__(256) router_grad_kernel(const __nv_bfloat16 *__restrict__ dout,
                                                         const __nv_bfloat16 *__restrict__ Y,
                                                         const int32_t *__restrict__ ids,
                                                         const float *__restrict__ wts, int T, int k, int E, int H,
                                                         float *__restrict__ dlogit)
{
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= T)
        return;
    const int t = warp;
    float D = 0.0f;    // lane j < k keeps D_j
    float sum = 0.0f;  // sum_m D_m
    for (int j = 0; j < k; ++j) {
        const __nv_bfloat16 *yr = Y + ((size_t)t * k + j) * H;
        const __nv_bfloat16 *dr = dout + (size_t)t * H;
        float acc = 0.0f;
        for (int h0 = lane * 8; h0 < H; h0 += 256) {  // eight columns per lane (H % 8 == 0)
            const uint4 dv = __ldg(reinterpret_cast<const uint4 *>(dr + h0));
            const uint4 yv = __ldg(reinterpret_cast<const uint4 *>(yr + h0));
            const __nv_bfloat16 *d8 = reinterpret_cast<const __nv_bfloat16 *>(&dv);
            const __nv_bfloat16 *y8 = reinterpret_cast<const __nv_bfloat16 *>(&yv);
#pragma unroll
            for (int c = 0; c < 8; ++c)
                acc = fmaf(bf2f(d8[c]), bf2f(y8[c]), acc);
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1)
            acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == j)
            D = acc;
        sum += acc;
    }
    for (int e = lane; e < E; e += 32)
        dlogit[(size_t)t * E + e] = 0.0f;
    __syncwarp();
    if (lane < k)
        dlogit[(size_t)t * E + ids[(size_t)t * k + lane]] = D - wts[(size_t)t * k + lane] * sum;
}

// out[b][c][r] = in[b][r][c] for r < R (rows), c < C (C % 64 == 0); out rows
// have ld_out >= round_up(R, 64) elements (columns R..ld_out-1 of a tile are
// written as 0).  64 x 64 tiles, 16-byte loads and stores.
__global__ void __launch_bounds__(256) transpose_kernel(const __nv_bfloat16 *__restrict__ in,
                                                       __nv_bfloat16 *__restrict__ out, int64_t R, int64_t C,
                                                       int64_t ld_out)
{
    __shared__ uint16_t tile[64][66];
    const int64_t b = blockIdx.z;
    const int64_t r0 = (int64_t)blockIdx.y * 64, c0 = (int64_t)blockIdx.x * 64;
    const uint16_t *src = reinterpret_cast<const uint16_t *>(in) + b * R * C;
    uint16_t *dst = reinterpret_cast<uint16_t *>(out) + b * C * ld_out;
    const int t = threadIdx.x;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int rr = t / 8 + 32 * i, cc = (t % 8) * 8;
        const int64_t r = r0 + rr;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (r < R)
            v = *reinterpret_cast<const uint4 *>(src + r * C + c0 + cc);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint32_t *>(&tile[rr][cc + 2 * q]) = w[q];
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int cc = t / 8 + 32 * i, rr = (t % 8) * 8;
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
            w[q] = (uint32_t)tile[rr + 2 * q][cc] | ((uint32_t)tile[rr + 2 * q + 1][cc] << 16);
        *reinterpret_cast<uint4 *>(dst + (c0 + cc) * ld_out + r0 + rr) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// dx[t] = sum_j dxs[t*k + j] (j ascending) + sum_j dlogit[t][e_j] W_router[e_j]  -> bf16;
// eight consecutive columns per thread (16-byte loads of the bf16 slot rows and router rows)
__global__ void __launch_bounds__(256) dx_kernel(const __nv_bfloat16 *__restrict__ dxs,
                                                const float *__restrict__ dlogit, const int32_t *__restrict__ ids,
                                                const __nv_bfloat16 *__restrict__ Wr, int T, int k, int E, int H,
                                                __nv_bfloat16 *__restrict__ dx)
{
    const int nv = H / 8;
    const int64_t total = (int64_t)T * nv;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / nv;
        const int h0 = (int)(i - t * nv) * 8;
        float acc[8];
#pragma unroll
        for (int c = 0; c < 8; ++c)
            acc[c] = 0.0f;
        for (int j = 0; j < k; ++j) {
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(dxs + (t * k + j) * H + h0));
            const __nv_bfloat16 *b = reinterpret_cast<const __nv_bfloat16 *>(&v);
#pragma unroll
            for (int c = 0; c < 8; ++c)
                acc[c] += bf2f(b[c]);
        }
        for (int j = 0; j < k; ++j) {
            const int e = ids[t * k + j];
            const float d = dlogit[t * E + e];
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(Wr + (size_t)e * H + h0));
            const __nv_bfloat16 *b = reinterpret_cast<const __nv_bfloat16 *>(&v);
#pragma unroll
            for (int c = 0; c < 8; ++c)
                acc[c] = fmaf(d, bf2f(b[c]), acc[c]);
        }
        uint32_t w[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            __nv_bfloat162 p2 = __floats2bfloat162_rn(acc[2 * c], acc[2 * c + 1]);
            w[c] = *reinterpret_cast<uint32_t *>(&p2);
        }
        *reinterpret_cast<uint4 *>(dx + t * H + h0) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// dW_router[e][h] = sum_t dlogit[t][e] x[t][h], dbias[e] = sum_t dlogit[t][e]:
// partial sums over chunks of 128 tokens (t ascending within a chunk; 8
// experts per block, each x element read once; the bias sums alongside),
// then a fixed-order sum of the chunks.
constexpr int kRgChunk = 128;
constexpr int kRgE = 8;

__global__ void __launch_bounds__(256) router_wgrad_partial_kernel(const float *__restrict__ dlogit,
                                                                  const __nv_bfloat16 *__restrict__ x, int T, int E,
                                                                  int H, float *__restrict__ part,
                                                                  float *__restrict__ bpart)
{
    __shared__ float s_dl[kRgChunk][kRgE];
    const int h = blockIdx.x * blockDim.x + threadIdx.x;
    const int e0 = blockIdx.y * kRgE;
    const int t0 = blockIdx.z * kRgChunk;
    for (int i = threadIdx.x; i < kRgChunk * kRgE; i += blockDim.x) {
        const int tt = i / kRgE, ee = i % kRgE;
        s_dl[tt][ee] = (t0 + tt < T && e0 + ee < E) ? dlogit[(size_t)(t0 + tt) * E + e0 + ee] : 0.0f;
    }
    __syncthreads();
    const int tn = min(kRgChunk, T - t0);
    if (blockIdx.x == 0 && threadIdx.x < kRgE && e0 + threadIdx.x < E) {  // the chunk's bias-gradient sums
        float bsum = 0.0f;
        for (int tt = 0; tt < tn; ++tt)
            bsum += s_dl[tt][threadIdx.x];
        bpart[(size_t)blockIdx.z * E + e0 + threadIdx.x] = bsum;
    }
    if (h >= H)
        return;
    float acc[kRgE];
#pragma unroll
    for (int j = 0; j < kRgE; ++j)
        acc[j] = 0.0f;
#pragma unroll 8
    for (int tt = 0; tt < tn; ++tt) {  // (unrolled: several tokens' loads in flight; t ascending)
        const float xv = bf2f(x[(size_t)(t0 + tt) * H + h]);
#pragma unroll
        for (int j = 0; j < kRgE; ++j)
            acc[j] = fmaf(s_dl[tt][j], xv, acc[j]);
    }
#pragma unroll
    for (int j = 0; j < kRgE; ++j)
        if (e0 + j < E)
            part[((size_t)blockIdx.z * E + e0 + j) * H + h] = acc[j];
}

__global__ void __launch_bounds__(256) router_wgrad_reduce_kernel(const float *__restrict__ part,
                                                                 const float *__restrict__ bpart, int E, int H,
                                                                 int nchunks, float *__restrict__ dWr,
                                                                 float *__restrict__ dbias)
{
    const int64_t total = (int64_t)E * H;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        float acc = 0.0f;
        for (int c = 0; c < nchunks; ++c)
            acc += part[(size_t)c * total + i];
        dWr[i] = acc;
    }
    if (dbias && blockIdx.x == 0)
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            float acc = 0.0f;
            for (int c = 0; c < nchunks; ++c)
                acc += bpart[(size_t)c * E + e];
            dbias[e] = acc;
        }
}

cudaError_t transpose(const __nv_bfloat16 *in, __nv_bfloat16 *out, int64_t batches, int64_t R, int64_t C,
                      int64_t ld_out, cudaStream_t st)
{
    if (batches <= 0 || R <= 0 || C <= 0)
        return cudaSuccess;
    dim3 grid((unsigned)((C + 63) / 64), (unsigned)((R + 63) / 64), (unsigned)batches);
    transpose_kernel<<<grid, 256, 0, st>>>(in, out, R, C, ld_out);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_backward_aux(int which, const BackwardAux &b, cudaStream_t st)
{
    switch (which) {
    case 0: {  // dY gather
        const int grid = (int)(b.P_max < 8192 ? b.P_max : 8192);
        dy_gather_kernel<<<grid > 0 ? grid : 1, 256, 0, st>>>(b.dout, b.sorted_ids, b.sorted_w, b.npp, b.T * b.k,
                                                              b.k, b.H, b.dys);
        return cudaGetLastError();
    }
    case 1: {  // routing gradient
        const int grid = (b.T * 32 + 255) / 256;
        router_grad_kernel<<<grid > 0 ? grid : 1, 256, 0, st>>>(b.dout, b.Y, b.topk_ids, b.topk_w, b.T, b.k, b.E,
                                                                b.H, b.dlogit);
        return cudaGetLastError();
    }
    case 2: {  // dx
        int64_t grid = ((int64_t)b.T * (b.H / 8) + 255) / 256;
        if (grid > 65535)
            grid = 65535;
        dx_kernel<<<(int)(grid > 0 ? grid : 1), 256, 0, st>>>(b.dxs, b.dlogit, b.topk_ids, b.Wr, b.T, b.k, b.E, b.H,
                                                            b.dx);
        return cudaGetLastError();
    }
    case 3: {  // router weight gradient
        const int nchunks = (b.T + kRgChunk - 1) / kRgChunk;
        dim3 grid((unsigned)((b.H + 255) / 256), (unsigned)((b.E + kRgE - 1) / kRgE), (unsigned)nchunks);
        float *bpart = b.rg_part + (int64_t)nchunks * b.E * b.H;
        router_wgrad_partial_kernel<<<grid, 256, 0, st>>>(b.dlogit, b.x, b.T, b.E, b.H, b.rg_part, bpart);
        int64_t g2 = ((int64_t)b.E * b.H + 255) / 256;
        if (g2 > 4096)
            g2 = 4096;
        router_wgrad_reduce_kernel<<<(int)g2, 256, 0, st>>>(b.rg_part, bpart, b.E, b.H, nchunks, b.dWr, b.dbias);
        return cudaGetLastError();
    }
    default:
        return cudaErrorInvalidValue;
    }
}

cudaError_t launch_transpose(const __nv_bfloat16 *in, __nv_bfloat16 *out, int64_t batches, int64_t R, int64_t C,
                             int64_t ld_out, cudaStream_t st)
{
    return transpose(in, out, batches, R, C, ld_out, st);
}

}  // namespace moe
