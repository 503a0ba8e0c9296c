/*
 * moe.h -- C ABI of the GB300 (sm_103a) fused Mixture-of-Experts layer.
 *
 * The layer is the fused MoE of the AITER walk-through (section 3, "Fused
 * MoE": gating -> token reorder by expert -> expert GEMMs -> weighted
 * combine) built as the two-stage group-GEMM path of the FlyDSL/Mixtral talk
 * (group GEMMs in place of masked dense GEMMs, SwiGLU activation):
 *
 *   route:   logits = x W_router^T (+ bias), top-k per token, softmax over
 *            the k selected logits (the weights sum to 1)
 *   sort:    the T*k (token, slot) pairs grouped by expert, each expert
 *            padded to whole blocks of block_m rows (section 3.1)
 *   stage 1: per block, gathered rows of x times W_gate_up[e]^T, then
 *            h = silu(gate) * up                              (section 3.2)
 *   stage 2: h times W_down[e]^T, each row scaled by its top-k weight
 *   combine: out[t] = sum over j of the weighted rows of token t
 *
 * Conventions for every entry point:
 *  - Pointers marked (device) are CUDA device pointers, (host) are host
 *    pointers.  All matrices are row-major and contiguous.  bf16 is IEEE
 *    bfloat16 bits in a uint16; e4m3 is the OCP FP8 E4M3 byte.
 *  - Weight layouts: W_router [E][H]; W_gate_up [E][2I][H] with rows 0..I-1
 *    the gate projection and rows I..2I-1 the up projection; W_down [E][H][I]
 *    (each expert matrix is N x K with K contiguous).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Calls are asynchronous on it: no host synchronisation, no
 *    allocation, no exceptions; results are ready when the stream is.
 *  - The caller owns every buffer.  The library keeps no mutable state
 *    that changes what a call computes or launches: only per-device
 *    constants (SM count, how many CTA-pair clusters fit).  Every
 *    choice a caller can make travels in the call's own arguments
 *    (block_m, split_k, and moe_options_t for moe_fused_forward_ex); the
 *    library reads no environment variables.
 *  - Arguments are validated on the host before anything is launched; an
 *    invalid call returns a negative status and launches nothing.  A CUDA
 *    launch error returns MOE_ERR_CUDA.  Kernels that wait on barriers give
 *    up after a bounded time and record MOE_ERR_TIMEOUT in the workspace
 *    status word (read it with moe_workspace_status).
 *
 * Limits: 1 <= k <= min(E, 32); E <= 1024; H and I multiples of 128 (the
 * tile granule of every GEMM kernel here, and the granule the AITER page's
 * stage rules test, inter_dim % 128); T >= 0 (T = 0 is a no-op that
 * returns MOE_OK).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_OK 0
#define MOE_ERR_INVALID_ARG (-1)
#define MOE_ERR_UNSUPPORTED (-2)
#define MOE_ERR_WORKSPACE (-3)
#define MOE_ERR_CUDA (-4)
#define MOE_ERR_TIMEOUT (-5)

#define MOE_BF16 0          /* bf16 weights and activations, fp32 accumulation */
#define MOE_FP8_BLOCK128 1  /* e4m3 weights (fp32 scale per 128x128 block) and
                               activations (fp32 scale per 1x128 group) */
#define MOE_FP8_TOKEN 2     /* e4m3 weights (fp32 scale per output channel) and
                               activations (fp32 scale per token) */
#define MOE_MXFP4 3         /* E2M1 weights and activations, E8M0 scale per 1x32
                               group */

#define MOE_MODE_GROUPED 0  /* tokens on the MMA M side, 128-row blocks */
#define MOE_MODE_SWAP 1     /* weights on the MMA M side, tokens on N (small T) */

/* Text for a status code.  Never NULL. */
const char *moe_status_string(int status);

/* Library version, major*10000 + minor*100 + patch. */
int moe_version(void);

/*
 * Sizes of the align-sort outputs (AITER page, section 3.1):
 * max_padded = T*k + E*block_m - k entries of sorted_ids / sorted_weights,
 * max_blocks = ceil(max_padded / block_m) entries of sorted_expert_ids.
 * Host only.  Returns MOE_OK or MOE_ERR_INVALID_ARG.
 */
int moe_align_sort_sizes(int T, int k, int E, int block_m, int64_t *max_padded, int64_t *max_blocks);

/*
 * The block-size rule of the AITER page (section 3.3, get_block_size_M):
 * among `candidates` (n entries), the block size with the fewest rounds of
 * tiles over `units` compute units, then the fewest idle units in the last
 * round (a full tie keeps the earlier candidate), where the tile count is
 * the page's tgN * (max_padded + BM - 1) // BM evaluated left to right,
 * (tgN * (max_padded + BM - 1)) / BM, with tgN = ceil(inter_dim/128) and
 * max_padded = token*topk + expert*BM - topk.  Host only; returns the chosen
 * block size or a negative status.
 */
int moe_block_size_m_heuristic(int token, int topk, int expert, int inter_dim, int units,
                               const int *candidates, int n);

/*
 * The K-split rule of the AITER page (section 3.4, get_ksplit), with the
 * page's undefined tgN/tgM read as ceil(inter_dim/128) and
 * ceil(token*topk/block_m).  Returns the split (0 = none) or a negative
 * status.  Host only.
 */
int moe_ksplit_heuristic(int token, int topk, int expert, int inter_dim, int model_dim, int units,
                         int block_m);

/* The plan moe_fused_forward follows for a shape. */
typedef struct moe_plan {
    int mode;           /* MOE_MODE_GROUPED or MOE_MODE_SWAP */
    int block_m;        /* sort block size (rows per padded expert block) */
    int split_k1;       /* K splits of stage 1 (1 = none) */
    int split_k2;       /* K splits of stage 2 (1 = none) */
    int64_t max_padded; /* T*k + E*block_m - k */
    int64_t max_blocks; /* ceil(max_padded / block_m) */
    size_t workspace_bytes;
} moe_plan_t;

/*
 * Choose mode, block size and K splits for a layer shape.  block_m = 0 and
 * split_k = 0 mean automatic; otherwise they are used as given (block_m
 * must be 128 in grouped mode and a multiple of 16 up to 128 in swap mode;
 * split_k splits stage 2's K = I and must divide I/64, I/128 for
 * MOE_FP8_TOKEN or I/256 for MOE_MXFP4; MXFP4 swap mode (T <= 64) takes
 * block_m up to 64).  num_sms = 0 asks
 * the current CUDA device; a positive value plans for that many SMs without
 * touching CUDA.  Returns MOE_OK or a negative status.  Host only.
 */
int moe_plan(int dtype, int T, int H, int I, int E, int k, int block_m, int split_k, int num_sms,
             moe_plan_t *plan);

/*
 * Workspace bytes moe_fused_forward needs for this shape (the plan's
 * workspace_bytes, planned for the current device).  0 on invalid input.
 */
size_t moe_fused_workspace_size(int dtype, int T, int H, int I, int E, int k, int block_m, int split_k);

/*
 * Byte offsets of the intermediate buffers inside the workspace of
 * moe_fused_forward (for inspection and tests; -1 = not present).
 */
typedef struct moe_ws_layout {
    int64_t status;          /* int32 status word (MOE_OK or MOE_ERR_TIMEOUT); word 4 after it:
                                tokens whose tensor-core routing fell back to all
                                fixed-order logits */
    int64_t topk_ids;        /* int32 [T][k] */
    int64_t topk_weights;    /* fp32 [T][k] */
    int64_t sorted_ids;      /* int32 [max_padded] */
    int64_t sorted_weights;  /* fp32 [max_padded] */
    int64_t sorted_expert_ids; /* int32 [max_blocks] */
    int64_t num_tokens_post_padded; /* int32 [1] */
    int64_t expert_counts;   /* int32 [E] */
    int64_t x_sorted;        /* bf16 [max_padded][H] or e4m3 [max_padded][H] */
    int64_t x_scales;        /* fp32 [H/128][max_padded] (FP8 block), [max_padded] (FP8 token) */
    int64_t inter;           /* bf16 [max_padded][I] or e4m3 [max_padded][I] */
    int64_t inter_scales;    /* fp32 [I/128][max_padded] (FP8 block), [max_padded] (FP8 token) */
    int64_t inter_h;         /* bf16 [max_padded][I]: SwiGLU output before its per-token
                                quantisation (FP8 token only) */
    int64_t y;               /* bf16 [T*k][H], weighted rows in slot order (each rounded once
                                from its fp32 value) */
    int64_t router_logits;   /* fp32 router logits: [T][E] from the CUDA-core router, or the
                                tensor-core router's per-slice partial sums
                                [splits][ceil(T/128)*128][E] */
    int64_t total;
} moe_ws_layout_t;

int moe_workspace_layout(int dtype, int T, int H, int I, int E, int k, int block_m, int split_k,
                         moe_ws_layout_t *layout);

/*
 * Read the workspace status word (device) into *status (host).  Synchronises
 * `stream`.  Returns MOE_OK or MOE_ERR_CUDA.
 */
int moe_workspace_status(const void *ws, int *status, void *stream);

/*
 * Router (gating + top-k; AITER page section 3, FlyDSL talk "Mixtral"):
 *   logit[t][e] = sum_h x[t][h] * W_router[e][h]  (+ bias[e])
 * in fp32 in one fixed order -- the H products are dealt to 32 partial sums
 * in chunks of 8 elements (element h to partial (h/8) mod 32), each partial
 * adds in ascending h, then the partials are combined by a butterfly with
 * strides 16, 8, 4, 2, 1 -- so the ids are a deterministic function of the
 * bytes.  topk_ids[t] = the k largest logits, largest first, an equal logit
 * going to the lower expert.  topk_weights[t][j]:
 *   renormalize = 1: exp(l_j - l_0) / sum over the k selected (they sum to 1;
 *                    what moe_fused_forward uses);
 *   renormalize = 0: exp(l_j - l_0) / sum over all E experts (the softmax
 *                    over all experts, evaluated at the selected ones).
 *   x (device) bf16 [T][H]; W_router (device) bf16 [E][H];
 *   bias (device) fp32 [E] or NULL; topk_ids (device) int32 [T][k];
 *   topk_weights (device) fp32 [T][k]; logits (device) fp32 [T][E] or NULL.
 * With logits given and T*E > 4096 the logits are computed by a tiled pass
 * and the top-k by a second pass (faster for large T*E); otherwise one fused
 * launch.  Both give the same bits.  H % 8 == 0.
 */
int moe_route_topk(const void *x, const void *W_router, const float *bias, int T, int H, int E, int k,
                   int renormalize, int32_t *topk_ids, float *topk_weights, float *logits, void *stream);

/* Scratch bytes moe_align_sort needs (device memory passed as ws). */
size_t moe_align_sort_workspace_size(int T, int k, int E);

/*
 * Token sort and alignment by expert (AITER page section 3.1, moe_sorting):
 * slot s = t*k + j.  Expert e's segment lists its slots in ascending s and
 * is padded with the sentinel T*k up to a multiple of block_m; segments
 * follow in ascending e; experts without slots take no block.
 *   topk_ids (device) int32 [T][k]; topk_weights (device) fp32 [T][k];
 *   sorted_ids (device) int32 [max_padded]: slot or T*k (padding / unused);
 *   sorted_weights (device) fp32 [max_padded]: topk weight of the slot, 0 on padding;
 *   sorted_expert_ids (device) int32 [max_blocks]: expert of each block, -1 if unused;
 *   num_tokens_post_padded (device) int32 [1]: sum of the padded segment lengths;
 *   expert_counts (device) int32 [E] or NULL: slots per expert;
 *   ws (device) scratch of moe_align_sort_workspace_size bytes.
 * An id outside [0, E) is a caller error.  The kernels check every id: a
 * slot with a bad id is left out of every segment (nothing outside the
 * output buffers is written) and num_tokens_post_padded is set to
 * MOE_ERR_INVALID_ARG (-1), which no valid result can be; check it when the
 * ids come from untrusted code.
 */
int moe_align_sort(const int32_t *topk_ids, const float *topk_weights, int T, int k, int E, int block_m,
                   int32_t *sorted_ids, float *sorted_weights, int32_t *sorted_expert_ids,
                   int32_t *num_tokens_post_padded, int32_t *expert_counts, void *ws, size_t ws_bytes,
                   void *stream);

/*
 * Block-scaled FP8 quantisation ("per_1x128" on the AITER page):
 * activations per 1x128 group of a row, weights per 128x128 block; each
 * group takes scale = amax / 448 (1 for an all-zero group) and codes
 * e4m3(v / scale), rounded to nearest even and saturated to +-448.
 *   moe_quantize_fp8_act: X (device) bf16 [R][C], C % 128 == 0 ->
 *     q (device) e4m3 [R][C], s (device) fp32 [R][C/128].
 *   moe_quantize_fp8_weights: W (device) bf16 [R][C], R and C % 128 == 0
 *     (an expert stack [E][N][K] is R = E*N, C = K) ->
 *     q (device) e4m3 [R][C], s (device) fp32 [R/128][C/128].
 */
int moe_quantize_fp8_act(const void *X, int64_t R, int C, uint8_t *q, float *s, void *stream);
int moe_quantize_fp8_weights(const void *W, int64_t R, int C, uint8_t *q, float *s, void *stream);

/*
 * Per-row FP8 quantisation ("per_Token" on the AITER page, section 3.2's
 * quantisation types): one scale per row -- a token of the activations or
 * an output channel of a weight stack -- scale = amax of the row / 448 (1
 * for an all-zero row), codes e4m3(v / scale), rounded to nearest even and
 * saturated to +-448.
 *   X (device) bf16 [R][C], C % 16 == 0 -> q (device) e4m3 [R][C],
 *   s (device) fp32 [R].  An expert stack [E][N][K] is R = E*N, C = K.
 */
int moe_quantize_fp8_rows(const void *X, int64_t R, int C, uint8_t *q, float *s, void *stream);

/*
 * MXFP4 quantisation ("per_1x32" on the AITER page; OCP microscaling FP4):
 * each group of 32 consecutive elements of a row shares the power-of-two
 * scale 2^e, e = floor(log2(group amax)) - 2 (0 for an all-zero group),
 * stored as the E8M0 byte e + 127; elements are v * 2^-e rounded to the
 * nearest E2M1 value (0, 0.5, 1, 1.5, 2, 3, 4, 6 and negatives; ties to the
 * even mantissa), clamped to +-6, as codes sign << 3 | magnitude index.
 *   X (device) bf16 [R][C], C % 32 == 0 -> q (device) [R][C/2] bytes, two
 *   codes per byte (element 2j in the low nibble of byte j);
 *   s (device) E8M0 bytes: tiled = 0 row-major [R][C/32]; tiled = 1 (R and
 *   C multiples of 128; the weight order moe_fused_forward reads)
 *   [R/128][C/128][512], group g of row r of a 128 x 128 tile at byte
 *   (r % 32) * 16 + (r % 128 / 32) * 4 + g % 4.
 */
int moe_quantize_mxfp4(const void *X, int64_t R, int C, uint8_t *q, uint8_t *s, int tiled, void *stream);

/*
 * Per-call choices of moe_fused_forward_ex and the training entries.  Fill
 * one with moe_options_init (the library's defaults) and change the fields
 * you need; a NULL options pointer means the defaults.  These select among
 * kernels that compute the same layer (each within the same tolerance of
 * the definition) or add instrumentation; none changes the workspace size.
 * (No counterpart on the fused-MoE pages: launch choices of this library.)
 */
typedef struct moe_options {
    /* Grouped-mode GEMM kernel for MOE_BF16, MOE_FP8_TOKEN and
     * MOE_FP8_BLOCK128: -1 automatic (CTA pairs when the average expert
     * holds at least one 128-row token block, T*k >= 128 * min(E, T*k): in
     * both stages for bf16, in stage 2 for per-token FP8, never for block
     * FP8, whose pair kernels are bit-identical to its one-SM kernels but
     * slower in stage 1), 0 always the one-SM kernels, 1 CTA pairs (the
     * two-SM tensor core) wherever supported. */
    int gemm_pair;
    /* bf16 swap mode (T <= 128): 1 runs both GEMM stages in one persistent
     * launch ("1-stage", AITER page section 3.2: tiles of both stages claimed
     * from one counter, stage-1 tiles first, the intermediate kept in L2,
     * the token rows fetched from x by the launch itself), 0 two launches
     * with a gather pass before them.  Both give bit-identical results.
     * Default 1. */
    int one_stage;
    /* Programmatic dependent launch: -1 the library's default set of launch
     * boundaries, otherwise a mask of them (bit 0 router -> sort and inside
     * the sort, 1 sort -> gather, 2 -> stage 1, 3 stage 1 -> stage 2, 4 ->
     * combine, 5 logit pass -> top-k pass, 6 preceding work -> router);
     * 0 turns it off.  Default -1 (all, except bits 2 and 3 in grouped mode,
     * where an early-resident persistent GEMM measured slower). */
    int pdl_mask;
    /* NULL, or 7 CUDA events (cudaEvent_t cast to void*, created by the
     * caller) recorded on the call's stream at [0] entry, [1] after routing,
     * [2] after the sort, [3] after the gather (FP8: gather + quantise),
     * [4] after stage 1, [5] after stage 2 (per-token FP8: including the
     * re-quantisation of the intermediate), [6] after the combine.  With the
     * one-launch decode path [3] follows [2] and [5] follows [4] directly.
     * Events between launches stop their overlap: time whole calls without. */
    void *const *stage_events;
    /* Limit, in microseconds, of the one-launch decode path's wait for the
     * intermediate (stage-2 tiles wait for every stage-1 epilogue); 0 = the
     * default of 2 s.  Every other device wait keeps its 2 s limit. */
    unsigned int h_wait_limit_us;
    /* Test of the timeout path only (0 otherwise): 1 makes the one-launch
     * decode path's stage-2 tiles wait for one more stage-1 epilogue than
     * exists, so that wait runs out after h_wait_limit_us; the call then
     * records MOE_ERR_TIMEOUT in the workspace status word and every CTA
     * returns after its copies and MMAs in flight have completed.  The
     * output of such a call is undefined; the next call on the workspace
     * starts clean. */
    int unsatisfiable_h_wait;
    /* MOE_BF16 on CTA pairs: experts with at most 64 tokens take swap-AB
     * pair tiles (the weights on the pair's 256-row MMA side, the expert's
     * tokens, rounded up to 32, on N) instead of a mostly padded 256 x 256
     * tile; light and 256 x 256 tiles are interleaved so that weight
     * streaming and tensor work overlap.  -1 automatic (default: on when I is
     * a multiple of 256, E <= 512 and the average expert that can hold a slot
     * has fewer than 4 blocks of 128 rows), 0 off, 1 on (needs I % 256 == 0
     * and E <= 512, else MOE_ERR_UNSUPPORTED).  Not used by the training
     * forward. */
    int light_tiles;
    /* Router for many experts (E >= 64, E % 32 == 0, T >= 64, k <= 28):
     * -1 automatic / 1: logits on the tensor core, then the k + 4 leading
     * candidates recomputed in the fixed order and the remaining experts
     * checked against a bound on the difference of the two sums (a near tie
     * recomputes all E logits in the fixed order), so the ids and weights are
     * those of the fixed-order router bit for bit; 0: the fixed-order router
     * on CUDA cores for every logit. */
    int tc_router;
} moe_options_t;

/* Set *options to the defaults (gemm_pair -1, one_stage 1, pdl_mask -1, no
 * events, default wait limit, no test switch).  Returns MOE_OK or
 * MOE_ERR_INVALID_ARG (NULL). */
int moe_options_init(moe_options_t *options);

/*
 * moe_fused_forward with per-call options (NULL = defaults).  Everything else
 * as moe_fused_forward.  Returns MOE_ERR_INVALID_ARG for an option outside
 * its range.
 */
int moe_fused_forward_ex(int dtype, const void *x, const void *W_router, const float *router_bias,
                         const void *W_gate_up, const void *w1_scale, const void *W_down, const void *w2_scale,
                         int T, int H, int I, int E, int k, int block_m, int split_k, void *out, void *ws,
                         size_t ws_bytes, const moe_options_t *options, void *stream);

/*
 * The whole layer: route, align-sort, stage 1 (gate/up group GEMM with the
 * SwiGLU epilogue), stage 2 (down group GEMM scaled by the top-k weights),
 * combine.  out (device) bf16 [T][H].
 *   dtype MOE_BF16: W_gate_up / W_down (device) bf16; w1_scale, w2_scale NULL.
 *   dtype MOE_FP8_BLOCK128: W_gate_up / W_down (device) e4m3 with
 *     w1_scale (device) fp32 [E*2I/128][H/128] and w2_scale (device) fp32
 *     [E*H/128][I/128] (as produced by moe_quantize_fp8_weights); x is
 *     quantised per 1x128 group inside the call, the router runs on bf16 x,
 *     and the SwiGLU output is re-quantised per 1x128 group between stages.
 *   dtype MOE_FP8_TOKEN: W_gate_up / W_down (device) e4m3 with w1_scale
 *     (device) fp32 [E*2I] and w2_scale (device) fp32 [E*H], one per output
 *     channel (as produced by moe_quantize_fp8_rows); x is quantised per
 *     token inside the call, the router runs on bf16 x, and the SwiGLU
 *     output (rounded to bf16) is re-quantised per token between stages.
 *   dtype MOE_MXFP4: W_gate_up / W_down (device) E2M1 codes, two per byte
 *     ([E][2I][H/2] and [E][H][I/2] bytes), with w1_scale / w2_scale
 *     (device) the E8M0 scale bytes in the tiled weight order of
 *     moe_quantize_mxfp4 (tiled = 1); x is quantised per 1x32 group inside
 *     the call, the router runs on bf16 x, and the SwiGLU output is
 *     re-quantised per 1x32 group between stages.  H and I multiples of
 *     256 (MOE_ERR_UNSUPPORTED otherwise).
 *   x (device) bf16 [T][H]; W_router (device) bf16 [E][H]; router_bias
 *   (device) fp32 [E] or NULL; block_m / split_k as in moe_plan;
 *   ws (device) of at least moe_fused_workspace_size bytes, 1024-byte aligned.
 * The result is deterministic: no atomics touch floating-point data.
 */
int moe_fused_forward(int dtype, const void *x, const void *W_router, const float *router_bias,
                      const void *W_gate_up, const void *w1_scale, const void *W_down, const void *w2_scale,
                      int T, int H, int I, int E, int k, int block_m, int split_k, void *out, void *ws,
                      size_t ws_bytes, void *stream);

/*
 * Training (bf16; the pages' stated future work for the group-GEMM MoE
 * kernels: backward "dgrad" and "wgrad" passes).
 *
 * moe_train_workspace_size: bytes of the workspace shared by one training
 * forward and its backward (0 on invalid input; I must be a multiple of 256).
 *
 * moe_fused_forward_train: moe_fused_forward for MOE_BF16 that always runs
 * the grouped (128-row block) path and keeps in ws what the backward needs:
 * the routing and sort, the sorted x rows, the pre-activations g | u, the
 * SwiGLU output h and the weighted stage-2 rows.  Same arguments as
 * moe_fused_forward without dtype, scales, block_m and split_k.
 *
 * moe_fused_backward: gradients for loss = sum(dout * out) of the forward
 * that last ran on ws (same x, weights and shape):
 *   dout (device) bf16 [T][H]  ->  dx (device) bf16 [T][H];
 *   dW_gate_up (device) fp32 [E][2I][H], dW_down (device) fp32 [E][H][I],
 *   dW_router (device) fp32 [E][H], dbias (device) fp32 [E] or NULL.
 * The top-k choice is a selection: the gradient reaches the router through
 * the softmax over the chosen k logits.  Experts without tokens get zero
 * weight gradients.  Every sum runs in a fixed order (no atomics), so the
 * gradients are bitwise reproducible.  Returns MOE_OK or a negative status.
 */
size_t moe_train_workspace_size(int T, int H, int I, int E, int k);
int moe_fused_forward_train(const void *x, const void *W_router, const float *router_bias, const void *W_gate_up,
                            const void *W_down, int T, int H, int I, int E, int k, void *out, void *ws,
                            size_t ws_bytes, const moe_options_t *options, void *stream);
int moe_fused_backward(const void *x, const void *W_router, const float *router_bias, const void *W_gate_up,
                       const void *W_down, const void *dout, int T, int H, int I, int E, int k, void *dx,
                       float *dW_gate_up, float *dW_down, float *dW_router, float *dbias, void *ws, size_t ws_bytes,
                       const moe_options_t *options, void *stream);

/*
 * moe_fused_forward with the activations in host memory: x_host (host) bf16
 * [T][H] is copied to the device inside the call and the result is copied
 * back to out_host (host) bf16 [T][H], all on `stream` (pinned host memory
 * keeps the copies asynchronous).  Device staging lives in ws, which must
 * hold moe_fused_workspace_size(...) + moe_host_staging_bytes(T, H) bytes.
 * out_host is valid once the stream has completed.
 */
size_t moe_host_staging_bytes(int T, int H);
int moe_fused_forward_host(int dtype, const void *x_host, const void *W_router, const float *router_bias,
                           const void *W_gate_up, const void *w1_scale, const void *W_down,
                           const void *w2_scale, int T, int H, int I, int E, int k, int block_m,
                           int split_k, void *out_host, void *ws, size_t ws_bytes, void *stream);

/*
 * moe_align_sort without a caller workspace.  (The fused-MoE pages have no
 * counterpart: this entry exists for callers of this library.)
 *
 * For callers that cannot allocate device memory themselves -- code that
 * must not call cudaMalloc because a host framework owns every device
 * allocation through its own pool, runs under a fixed memory budget, or
 * cannot afford the implicit synchronisation of an allocation on its hot
 * path.  They pass the same inputs and outputs as moe_align_sort, but no ws.
 *
 * The scratch is a fixed array of MOE_NOALLOC_SORT_SCRATCH_BYTES in the
 * library's own device memory; every GPU that loads the library holds it
 * until the process exits.  Every call looks up the array's address on the
 * current device (cudaGetSymbolAddress, which allocates nothing; it stays
 * right after a cudaDeviceReset).  The first call on a device may load the
 * library's device code there, so make that first call before any stream
 * capture.  Nothing is allocated, by this library or any library it calls.
 * Shapes whose scratch (one int32 per expert per 1024 slots, plus E+1
 * offsets) does not fit return MOE_ERR_UNSUPPORTED; use moe_align_sort with
 * a workspace for those.  All calls share the one array and it keeps the
 * last call's contents: calls that overlap on the GPU (on different streams,
 * or from different host threads without ordering) race on it and must be
 * serialised by the caller.  Ids are checked as in moe_align_sort.
 */
#define MOE_NOALLOC_SORT_SCRATCH_BYTES (1 << 20)

int moe_align_sort_noalloc(const int32_t *topk_ids, const float *topk_weights, int T, int k, int E,
                           int block_m, int32_t *sorted_ids, float *sorted_weights,
                           int32_t *sorted_expert_ids, int32_t *num_tokens_post_padded,
                           int32_t *expert_counts, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
