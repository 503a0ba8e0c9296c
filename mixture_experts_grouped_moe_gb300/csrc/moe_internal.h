// Internal declarations shared by the translation units of libmoe_gb300:
// kernel launchers (one per .cu file) called by the C-ABI layer in
// moe_api.cu.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/moe.h"

namespace moe {

// ------------------------------------------------------ route / sort / aux

void launch_router(const __nv_bfloat16 *x, const __nv_bfloat16 *Wr, const float *bias, int T, int H, int E,
                   int k, int32_t *ids, float *wts, float *logits, cudaStream_t st);

// Chunked stable counting sort; ws holds nchunks*E int32 chunk counters.
constexpr int kSortChunk = 1024;
size_t sort_scratch_bytes(int T, int k, int E);

struct SortOut {
    int32_t *sorted_ids;
    float *sorted_weights;
    int32_t *sorted_expert_ids;
    int32_t *num_post_padded;
    int32_t *expert_counts;   // [E]
    int32_t *expert_offsets;  // [E+1] padded segment starts (may be null)
    int32_t *active_experts;  // [E] compact list of experts with slots (may be null)
    int32_t *num_active;      // [1] (may be null)
    int32_t *slot_pos;        // [S] sorted position of each slot (may be null)
};
void launch_align_sort(const int32_t *ids, const float *wts, int T, int k, int E, int block_m,
                       const SortOut &o, void *scratch, cudaStream_t st);

// x rows gathered into sorted order (zero rows for padding), up to *npp rows.
void launch_gather_rows(const __nv_bfloat16 *x, const int32_t *sorted_ids, const int32_t *npp, int S, int k,
                        int H, int64_t P_max, __nv_bfloat16 *xs, cudaStream_t st);
// Same, quantised per 1x128 group: codes [P_max][H], scales transposed [H/128][P_max].
void launch_gather_quant_rows(const __nv_bfloat16 *x, const int32_t *sorted_ids, const int32_t *npp, int S,
                              int k, int H, int64_t P_max, uint8_t *q, float *sT, cudaStream_t st);

void launch_quant_act(const __nv_bfloat16 *X, int64_t R, int C, uint8_t *q, float *s, cudaStream_t st);
void launch_quant_weights(const __nv_bfloat16 *W, int64_t R, int C, uint8_t *q, float *s, cudaStream_t st);

// out[t] = sum_j Y[t*k+j] (j ascending), fp32 -> bf16.
void launch_combine(const float *Y, int T, int k, int H, __nv_bfloat16 *out, cudaStream_t st);
// out[t] = sum_j w[t*k+j] * sum_ks P[ks][slot_pos[t*k+j]]  (split-K stage-2 partials).
void launch_splitk_combine(const float *P, int SK, int64_t P_rows, const int32_t *slot_pos, const float *wts,
                           int T, int k, int H, __nv_bfloat16 *out, cudaStream_t st);

// --------------------------------------------------------------- GEMMs

struct GemmArgs {
    // tensor maps (host-encoded; passed by value as __grid_constant__)
    CUtensorMap tm_x;     // token operand rows [P_max][K]
    CUtensorMap tm_w;     // weight operand rows [E*rows_per_expert][K]
    const int32_t *sorted_ids;
    const float *sorted_weights;
    const int32_t *sorted_expert_ids;
    const int32_t *num_post_padded;
    const int32_t *expert_offsets;
    const int32_t *active_experts;
    const int32_t *num_active;
    const int32_t *expert_counts;
    // FP8 block scales
    const float *x_scales;   // [K/128][P_max]
    const float *w_scales;   // [E*rows_per_expert/128][K/128]
    int K;                   // reduction length
    int N;                   // output columns per expert (stage 1: I, stage 2: H)
    int rows_per_expert;     // weight rows per expert (stage 1: 2I, stage 2: H)
    int S;                   // T*k (sentinel)
    int E;
    int64_t P_max;
    int split_k;             // swap mode: K splits
    // outputs
    void *inter;             // stage 1: [P_max][I] bf16 or e4m3
    float *inter_scales;     // stage 1 FP8: [I/128][P_max]
    float *y;                // stage 2: [S][H] fp32 (weighted)
    float *partials;         // stage 2 split-K: [split][P_max][H]
    int *status;
};

bool encode_tmap_2d(CUtensorMap *map, const void *base, int elem_bytes, uint64_t inner, uint64_t rows,
                    uint32_t box_inner, uint32_t box_rows);

int num_sms_current_device();

cudaError_t launch_gemm_grouped_bf16(int stage, const GemmArgs &a, int grid, cudaStream_t st);
cudaError_t launch_gemm_swap_bf16(int stage, const GemmArgs &a, int grid, cudaStream_t st);
cudaError_t launch_gemm_grouped_fp8(int stage, const GemmArgs &a, int grid, cudaStream_t st);

}  // namespace moe
