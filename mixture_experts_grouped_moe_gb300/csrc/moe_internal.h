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

#include <utility>

namespace moe {

// ------------------------------------------------ programmatic dependent launch
//
// Kernels after the first one of an entry point are launched with
// programmatic stream serialisation: a kernel may be scheduled while its
// predecessor drains, runs its prologue, and blocks in pdl_wait() until the
// predecessor has completed and its writes are visible.  Every kernel calls
// pdl_wait() before reading anything a previous kernel wrote (and before
// writing anything a previous kernel reads), and pdl_trigger() to let its
// own successor be scheduled.  Both are no-ops for a normal launch.

#if defined(__CUDACC__)
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
#endif

// Launch boundaries that may overlap (bit i of moe_options_t::pdl_mask):
enum PdlSite {
    kPdlSort = 0,     // router/top-k -> sort, and inside the sort
    kPdlGather = 1,   // sort -> gather
    kPdlStage1 = 2,   // gather -> stage 1
    kPdlStage2 = 3,   // stage 1 -> stage 2
    kPdlCombine = 4,  // stage 2 -> combine
    kPdlTopk = 5,     // logit pass -> top-k pass
    kPdlRouter = 6,   // whatever precedes the layer -> router (the router waits for its completion
                      // before reading anything; it starts early only after a kernel that
                      // triggers, such as the previous layer call's combine)
};
constexpr int kPdlAll = 0x7f;
// The default set: every boundary, except the two GEMM boundaries in grouped
// mode, where an early-resident persistent GEMM measured slower (Mixtral
// prefill 3.94 ms without vs 4.38 ms with) while swap mode gains from it.
inline int pdl_default_mask(bool grouped)
{
    return grouped ? kPdlAll & ~((1 << kPdlStage1) | (1 << kPdlStage2)) : kPdlAll;
}
inline bool pdl_site(int mask, int site) { return (mask >> site) & 1; }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(bool pdl, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t st, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl ? attr : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ------------------------------------------------------ route / sort / aux

// Words at the start of the fused forward's workspace: [0] status, [1] stage-1
// tile counter, [2] stage-2 tile counter, [3] the one-launch decode's count of
// finished stage-1 epilogue warps, [4] tokens whose tensor-core routing fell
// back to all fixed-order logits, [5..7] spare.  The router zeroes them.
constexpr int kStatusWords = 8;

// Small T*E: one fused launch.  Large T*E: a tiled logit pass into `logits`
// (fp32 [T][E], required then) followed by a warp-per-token top-k pass.
// `status` (nullable) points at kStatusWords words that the first kernel
// zeroes.  `pdl` applies to the first launch.
bool router_needs_logits(int T, int E);
// renorm: 1 softmax over the k selected, 0 softmax over all E evaluated at the selected.
// pdl_mask: sites kPdlRouter (the first launch) and kPdlTopk (the top-k pass).
cudaError_t launch_router(const __nv_bfloat16 *x, const __nv_bfloat16 *Wr, const float *bias, int T, int H, int E,
                          int k, int renorm, int32_t *ids, float *wts, float *logits, int *status, int pdl_mask,
                          cudaStream_t st);

// Router on the tensor core for many experts (ids and weights identical to
// launch_router's with renorm = 1): per-expert norms (+ zeroing the status
// words), logits on the tensor core in K slices, then a warp per token that
// recomputes the leading candidates in the fixed order and checks the rest
// against a bound.  scratch: router_tc_scratch_floats floats.
bool router_tc_eligible(int T, int H, int E, int k);
int router_tc_splits(int T, int H, int E, int num_sms);
size_t router_tc_scratch_floats(int T, int H, int E, int num_sms);
// An upper bound of router_tc_scratch_floats for any SM count (at most 8 K slices).
inline size_t router_tc_scratch_floats_max(int T, int E) { return (size_t)8 * ((T + 127) / 128 * 128) * E + E; }
cudaError_t launch_router_tc(const __nv_bfloat16 *x, const __nv_bfloat16 *Wr, const float *bias, int T, int H, int E,
                             int k, int32_t *ids, float *wts, float *scratch, int *status, int pdl_mask,
                             cudaStream_t st);

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
// pdl_first: the first launch follows another kernel of this library; pdl_inner: the
// chunked sort's second and third launches.  An id outside [0, E) is left out of every
// segment and sets *num_post_padded to -1.
cudaError_t launch_align_sort(const int32_t *ids, const float *wts, int T, int k, int E, int block_m,
                              const SortOut &o, void *scratch, bool pdl_first, bool pdl_inner, cudaStream_t st);

// x rows gathered into sorted order, up to *npp rows.  Padding rows are written as zeros when
// zero_padding is set (the training forward: the weight gradients sum over every position);
// otherwise they are left as they are -- a GEMM output row depends only on its own input row,
// and the results of padding rows are never stored.
cudaError_t launch_gather_rows(const __nv_bfloat16 *x, const int32_t *sorted_ids, const int32_t *npp, int S, int k,
                               int H, int64_t P_max, __nv_bfloat16 *xs, bool zero_padding, bool pdl,
                               cudaStream_t st);
// The same rows (inference: padding rows untouched) walked token by token: x[t] is read once and
// written to sorted positions slot_pos[t*k + j], j < k (k <= 32; positions outside [0, P_max)
// are skipped).
cudaError_t launch_gather_by_token(const __nv_bfloat16 *x, const int32_t *slot_pos, int T, int k, int H,
                                   int64_t P_max, __nv_bfloat16 *xs, bool pdl, cudaStream_t st);
// Same, quantised per 1x128 group: codes [P_max][H], scales transposed [H/128][P_max].
cudaError_t launch_gather_quant_rows(const __nv_bfloat16 *x, const int32_t *sorted_ids, const int32_t *npp, int S,
                                     int k, int H, int64_t P_max, uint8_t *q, float *sT, bool pdl, cudaStream_t st);

void launch_quant_act(const __nv_bfloat16 *X, int64_t R, int C, uint8_t *q, float *s, cudaStream_t st);
// Per-row e4m3 quantisation (scale = row amax / 448); rows gathered through
// sorted_ids (token = slot / k, padding -> zero row) when it is non-null;
// the row count read from nrows (device) when non-null, else R.
cudaError_t launch_quant_rows(const __nv_bfloat16 *X, const int32_t *sorted_ids, const int32_t *nrows, int64_t R,
                              int S, int k, int C, uint8_t *q, float *s, bool pdl, cudaStream_t st,
                              float *zero_rows = nullptr);
// Rows [nrows][C] whose max |v| is known (row_amax, e.g. from the GEMM that wrote them): codes and
// scales as launch_quant_rows gives for the same rows, in one pass.
cudaError_t launch_quant_rows_amax(const __nv_bfloat16 *X, const float *row_amax, const int32_t *nrows, int64_t R,
                                   int C, uint8_t *q, float *s, bool pdl, cudaStream_t st);
void launch_quant_weights(const __nv_bfloat16 *W, int64_t R, int C, uint8_t *q, float *s, cudaStream_t st);

// out[t] = sum_j Y[t*k+j] (j ascending), fp32 -> bf16.
cudaError_t launch_combine(const __nv_bfloat16 *Y, int T, int k, int H, __nv_bfloat16 *out, bool pdl,
                           cudaStream_t st);
// out[t] = sum_j w[t*k+j] * sum_ks P[ks][slot_pos[t*k+j]]  (split-K stage-2 partials).
cudaError_t launch_splitk_combine(const float *P, int SK, int64_t P_rows, const int32_t *slot_pos, const float *wts,
                                  int T, int k, int H, __nv_bfloat16 *out, bool pdl, cudaStream_t st);

// --------------------------------------------------------------- GEMMs

struct GemmArgs {
    // tensor maps (host-encoded; passed by value as __grid_constant__)
    CUtensorMap tm_x;     // token operand rows [P_max][K]
    CUtensorMap tm_w;     // weight operand rows [E*rows_per_expert][K]
    CUtensorMap tm_x16;   // the token operand in 16-row boxes (light-expert pair tiles)
    CUtensorMap tm_sfa;   // grouped MXFP4 stage 2: h's blocked scales as 16-byte rows, 64-row boxes
    CUtensorMap tm_sfb;   // grouped MXFP4 stage 2: W_down's blocked scales, the same
    const int32_t *sorted_ids;
    const float *sorted_weights;
    const int32_t *sorted_expert_ids;
    const int32_t *num_post_padded;
    const int32_t *expert_offsets;
    const int32_t *active_experts;
    const int32_t *num_active;
    const int32_t *expert_counts;
    // FP8 block scales
    const float *x_scales;   // block FP8: [K/128][P_max]; per-token FP8: [P_max]
    const float *w_scales;   // block FP8: [E*rows_per_expert/128][K/128]; per-token FP8: [E*rows_per_expert]
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
    float *row_amax;         // per-token FP8 stage 1 (one-SM grouped): max |h| of each row (bf16-rounded),
                             // by atomicMax on the bits; zeroed by the activation quantiser before
    __nv_bfloat16 *y;        // stage 2: [S][H] bf16, each row its weighted fp32 result rounded once
    float *partials;         // stage 2 split-K: [split][P_max][H]
    int *status;
    int *tile_counter;       // zeroed before the launch; CTAs claim tiles from it
    // training (bf16, grouped mode)
    __nv_bfloat16 *gu;       // stage 1: when set, also the pre-activations [P_max][2I] (g | u)
    const __nv_bfloat16 *gu_in;  // backward of stage 2 (STAGE 3): saved g | u
    __nv_bfloat16 *dgu;      // backward of stage 2: dg | du [P_max][2I]
    float *dw_out;           // weight gradient (STAGE 5, segment mode): [E][M][N] fp32
    int M;                   // segment mode: rows of the A operand (output rows)
    int pdl_mask;            // launch boundaries with programmatic serialisation (PdlSite bits)
};

bool encode_tmap_2d(CUtensorMap *map, const void *base, int elem_bytes, uint64_t inner, uint64_t rows,
                    uint32_t box_inner, uint32_t box_rows);
// A byte buffer of nbytes (a multiple of 16) as rows of 16 bytes, unswizzled, box_rows rows per box.
bool encode_tmap_rows16(CUtensorMap *map, const void *base, uint64_t nbytes, uint32_t box_rows);

int num_sms_current_device();

// The GEMM launchers take their programmatic-serialisation choice from a.pdl_mask.
cudaError_t launch_gemm_grouped_bf16(int stage, const GemmArgs &a, int grid, cudaStream_t st);
cudaError_t launch_gemm_swap_bf16(int stage, const GemmArgs &a, int grid, cudaStream_t st);
cudaError_t launch_gemm_grouped_fp8(int stage, const GemmArgs &a, int grid, cudaStream_t st);
cudaError_t launch_gemm_grouped_fp8_token(int stage, const GemmArgs &a, int grid, cudaStream_t st);
// One-kernel decode (bf16, swap-AB): both stages in one persistent launch;
// tile_counter claims tiles of both stages, h_done counts finished stage-1
// epilogue warps (both zeroed by the router).
struct FusedArgs {
    GemmArgs s1, s2;
    int *tile_counter;
    int *h_done;
    const __nv_bfloat16 *x;  // the layer input [T][H]: stage-1 token rows are fetched from it directly
    int k;                   // top-k (slot s belongs to token s / k)
    unsigned long long h_wait_ns;  // limit of the stage-2 tiles' wait for the intermediate
    int h_extra;             // added to that wait's target (1 only to test the timeout path)
};
cudaError_t launch_fused_decode(const FusedArgs &F, int grid, cudaStream_t st);
// Training (bf16): backward GEMMs -- which = 3: dh = dY W_down with
// SwiGLU's backward epilogue (into dgu); 2: dx per slot = dgu W_gate_up
// (stage 2's tile shape, sorted_weights null = unit weights); 5: weight
// gradients over token segments (A, B transposed activations [rows][P]).
cudaError_t launch_gemm_backward_bf16(int which, const GemmArgs &a, int grid, cudaStream_t st);
struct BackwardAux {
    const __nv_bfloat16 *dout, *x, *Wr;
    const int32_t *sorted_ids;
    const float *sorted_w;
    const int32_t *npp;
    const __nv_bfloat16 *Y;    // forward's weighted stage-2 rows [S][H] bf16
    const int32_t *topk_ids;
    const float *topk_w;
    int T, k, E, H;
    int64_t P_max;
    __nv_bfloat16 *dys;        // [P_max][H]
    float *dlogit;             // [T][E]
    const __nv_bfloat16 *dxs;  // [S][H] bf16
    __nv_bfloat16 *dx;         // [T][H]
    float *dWr, *dbias;        // [E][H], [E] (dbias nullable)
    float *rg_part;            // [ceil(T/128)][E][H] + [ceil(T/128)][E] partial router / bias gradients
};
// Scratch floats of the router weight and bias gradients' partial sums.
inline int64_t router_wgrad_scratch(int T, int E, int H) { return (int64_t)((T + 127) / 128) * E * (H + 1); }
// which: 0 dY gather, 1 routing gradient, 2 dx, 3 router weight gradient
cudaError_t launch_backward_aux(int which, const BackwardAux &b, cudaStream_t st);
// out[b][c][r] = in[b][r][c] (bf16); C % 64 == 0; out rows of ld_out >= round_up(R, 64) elements
cudaError_t launch_transpose(const __nv_bfloat16 *in, __nv_bfloat16 *out, int64_t batches, int64_t R, int64_t C,
                             int64_t ld_out, cudaStream_t st);
// MXFP4: swap-AB GEMMs with hardware block scaling, and the 1x32 quantiser
// (row-major or tiled E8M0 scales; optional gather through sorted_ids).
cudaError_t launch_gemm_swap_mx4(int stage, const GemmArgs &a, int grid, cudaStream_t st);
cudaError_t launch_gemm_grouped_mx4(int stage, const GemmArgs &a, int grid, cudaStream_t st);
cudaError_t launch_quant_mx4(const __nv_bfloat16 *X, const int32_t *sorted_ids, const int32_t *nrows, int64_t R,
                             int S, int k, int C, uint8_t *q, uint8_t *s, bool tiled, bool pdl, cudaStream_t st);
// Grouped-mode GEMM on CTA pairs (two-SM tensor core), bf16 (qt = 0) or
// per-token FP8 (qt = 1); max_pair_tiles bounds the useful cluster count.
// light (bf16 stages 1 and 2; stage 1 needs N % 256 == 0; E <= 512): experts with
// at most 64 tokens take swap-AB pair tiles (a.tm_x16: the token operand in
// 16-row boxes; a.expert_counts required).
bool gemm_pair_supported(int E);
// Block-scaled FP8 group GEMM on CTA pairs (grouped mode, stages 1 and 2).
bool gemm_pair_fp8_supported(int E);
cudaError_t launch_gemm_pair_fp8(int stage, const GemmArgs &a, int64_t max_pair_tiles, cudaStream_t st);
bool gemm_pair_light_supported(int E);  // light-expert tiles: E <= 512
// w_mn_major (bf16 stages 2 and 3, the backward's dgrad GEMMs): a.tm_w covers the weights in their
// stored [E*K][N] layout with 64 x 64 boxes, read as an MN-major operand (no transposed copy).
cudaError_t launch_gemm_pair(int stage, int qt, const GemmArgs &a, int64_t max_pair_tiles, cudaStream_t st,
                             bool light = false, bool w_mn_major = false);
cudaError_t launch_gemm_swap_fp8_token(int stage, const GemmArgs &a, int grid, cudaStream_t st);

}  // namespace moe
