// C ABI of the fused MoE layer (declared in include/moe.h): argument
// validation, the host planner (mode, block size, K split, workspace
// carve-up), TMA descriptor encoding, and the launch sequence
//   route -> align-sort -> gather (FP8: gather + quantise) ->
//   stage-1 group GEMM (per-token FP8: + per-row quantisation of h) ->
//   stage-2 group GEMM -> combine
// on the caller's stream.  Nothing here allocates device memory or
// synchronises (except moe_workspace_status, which reads one word back).
#include <atomic>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "moe_internal.h"

namespace moe {

namespace {

constexpr int64_t kAlign = 1024;

int64_t align_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

bool encode_tmap_2d(CUtensorMap *map, const void *base, int elem_bytes, uint64_t inner, uint64_t rows,
                    uint32_t box_inner, uint32_t box_rows)
{
    auto fn = get_encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {inner * (uint64_t)elem_bytes};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                    const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_tmap_rows16(CUtensorMap *map, const void *base, uint64_t nbytes, uint32_t box_rows)
{
    auto fn = get_encode_fn();
    if (!fn || nbytes % 16 != 0)
        return false;
    cuuint64_t dims[2] = {16, nbytes / 16};
    cuuint64_t strides[1] = {16};
    cuuint32_t box[2] = {16, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Automatic CTA-pair rule (same-box measurements on GB300): pairs pay off once
// the average active expert holds one token block (S >= 128 per expert, E
// standing in for the active count): bf16 Mixtral shapes, one-SM vs pairs,
// T=512 0.656 -> 0.637 ms, T=1024 0.815 -> 0.744, T=2048 1.222 -> 1.186,
// T=8192 stage 1 2.45 -> 2.31 and stage 2 1.38 -> 1.16 ms; the fine-grained
// E=256 workload (2.4 blocks per active expert) is even (4.110 vs 4.123 ms).
// For per-token FP8 only stage 2 gains (Mixtral shapes, T=4096: stage 2
// 0.49 -> 0.42 ms, stage 1 0.77 -> 0.83 ms).  Block-scaled FP8 stays on the
// one-SM kernels: its pair kernels are bit-identical but their per-K-block
// promotion round trip crosses the pair (same shapes: stage 1 0.82 -> 1.14
// ms, stage 2 0.48 -> 0.48 ms).  gemm_pair: the caller's choice (-1
// automatic, 0 never, 1 whenever supported).
static bool use_pair(int dtype, int stage, int T, int k, int E, int gemm_pair)
{
    if (dtype == MOE_MXFP4 || !(dtype == MOE_FP8_BLOCK128 ? gemm_pair_fp8_supported(E) : gemm_pair_supported(E)))
        return false;
    if (gemm_pair >= 0)
        return gemm_pair == 1;
    const int64_t S = (int64_t)T * k;
    const int64_t act = S < E ? S : E;
    if (S < 128 * act || dtype == MOE_FP8_BLOCK128)
        return false;
    return dtype == MOE_BF16 || stage == 2;
}

int num_sms_current_device()
{
    static std::atomic<int> cache[64];  // per device, zero until first computed
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 0;
    if (cache[dev].load(std::memory_order_relaxed) == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return 0;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return cache[dev].load(std::memory_order_relaxed);
}

// Workspace carve-up (byte offsets from ws).
struct Layout {
    int64_t status, logits, topk_ids, topk_w, sort_scratch, counts, offsets, active, num_active, npp;
    int64_t sorted_ids, sorted_w, sorted_eids, slot_pos;
    int64_t x_sorted, x_scales, inter, inter_scales, inter_h, h_amax, y, partials;
    int64_t total;
};

static int validate_shape(int dtype, int T, int H, int I, int E, int k)
{
    if (dtype != MOE_BF16 && dtype != MOE_FP8_BLOCK128 && dtype != MOE_FP8_TOKEN && dtype != MOE_MXFP4)
        return MOE_ERR_INVALID_ARG;
    if (T < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0)
        return MOE_ERR_INVALID_ARG;
    if (E > 1024 || k > E || k > 32)
        return MOE_ERR_UNSUPPORTED;
    if (H % 128 != 0 || I % 128 != 0)
        return MOE_ERR_UNSUPPORTED;
    if (dtype == MOE_MXFP4 && (H % 256 != 0 || I % 256 != 0))
        return MOE_ERR_UNSUPPORTED;  // 256 FP4 elements of K per pipeline stage
    if ((int64_t)T * k > (int64_t)1 << 30 || (int64_t)E * 2 * I > (int64_t)1 << 30 ||
        (int64_t)E * H > (int64_t)1 << 30 || H > (1 << 20) || I > (1 << 20))
        return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

static Layout make_layout(int dtype, int T, int H, int I, int E, int k, const moe_plan_t &p)
{
    Layout L;
    const int64_t S = (int64_t)T * k;
    const int64_t P = p.max_padded, NB = p.max_blocks;
    const int64_t eb = (dtype == MOE_BF16) ? 2 : 1;
    int64_t off = 0;
    auto take = [&](int64_t bytes) {
        const int64_t o = off;
        off = align_up(off + (bytes > 0 ? bytes : 0), kAlign);
        return o;
    };
    L.status = take(kStatusWords * 4);
    {
        int64_t lf = (int64_t)T * E;
        if (router_tc_eligible(T, H, E, k))
            lf = std::max<int64_t>(lf, (int64_t)router_tc_scratch_floats_max(T, E));
        L.logits = take(lf * 4);
    }
    L.topk_ids = take(S * 4);
    L.topk_w = take(S * 4);
    L.sort_scratch = take((int64_t)sort_scratch_bytes(T, k, E));
    L.counts = take(E * 4);
    L.offsets = take((E + 1) * 4);
    L.active = take(E * 4);
    L.num_active = take(4);
    L.npp = take(4);
    L.sorted_ids = take(P * 4);
    L.sorted_w = take(P * 4);
    L.sorted_eids = take(NB * 4);
    L.slot_pos = take(S * 4);
    if (dtype == MOE_MXFP4) {
        L.x_sorted = take(P * H / 2);      // two E2M1 codes per byte
        L.x_scales = take(P * H / 32);     // E8M0 per 1x32 group
        L.inter = take(P * I / 2);
        L.inter_scales = take(P * I / 32);
    } else {
        L.x_sorted = take(P * H * eb);
        L.x_scales = (dtype == MOE_FP8_BLOCK128) ? take((H / 128) * P * 4)
                     : (dtype == MOE_FP8_TOKEN)  ? take(P * 4)
                                                 : -1;
        L.inter = take(P * I * eb);
        L.inter_scales = (dtype == MOE_FP8_BLOCK128) ? take((I / 128) * P * 4)
                         : (dtype == MOE_FP8_TOKEN)  ? take(P * 4)
                                                     : -1;
    }
    L.inter_h = (dtype == MOE_FP8_TOKEN) ? take(P * I * 2) : -1;
    L.h_amax = (dtype == MOE_FP8_TOKEN) ? take(P * 4) : -1;
    if (p.split_k2 > 1) {
        L.y = -1;
        L.partials = take((int64_t)p.split_k2 * P * H * 4);
    } else {
        L.y = take(S * H * 2);
        L.partials = -1;
    }
    L.total = off;
    return L;
}

// GB300 analogue of the AITER page's get_block_size_M (section 3.3) for the swap-AB (decode)
// kernels: the same choice -- fewest rounds of tiles over the compute units, then fewest idle
// units in the last round, a full tie keeping the earlier candidate -- over the swap kernels'
// block sizes {16, 32, 64, 128} (MXFP4: up to 64), with the SM count as the units and the
// tiles those kernels actually run: one stage-1 tile per 128 rows of W_gate_up's gate half for
// every expert that can hold a slot, whatever the block size (the expert's whole padded
// segment is the MMA's N side).  The rounds therefore tie and the first candidate, 16, is
// kept, which is also the measured best: Mixtral decode shapes on GB300 (same box, 400 steps)
// T=1 137 / 149 / 184 / 282 us, T=32 436 / 448 / 525 / 785 us, T=128 476 / 512 / 534 / 794 us
// for block sizes 16 / 32 / 64 / 128 (larger blocks only add padded rows to every tile).
static int swap_block_m(int dtype, int64_t e_act, int I, int units)
{
    const int cands[4] = {16, 32, 64, 128};
    const int n = dtype == MOE_MXFP4 ? 3 : 4;
    int best = cands[0];
    int64_t best_r = 0, best_idle = 0;
    for (int i = 0; i < n; ++i) {
        const int64_t tiles = e_act * (I / 128);  // independent of the block size in swap mode
        const int64_t rounds = (tiles + units - 1) / units;
        const int64_t idle = units - tiles % units;
        if (i == 0 || rounds < best_r || (rounds == best_r && idle < best_idle)) {
            best = cands[i];
            best_r = rounds;
            best_idle = idle;
        }
    }
    return best;
}

// GB300 analogue of the page's get_ksplit (section 3.4) for the swap-AB kernels' stage 2
// (K = I): when its tiles (experts that can hold a slot x 256-feature tiles of H) leave SMs
// idle, split K so that every SM gets work: split_max = ceil(units / tiles) as on the page,
// but the smallest divisor of K's 128-byte blocks that reaches it (the page takes the
// largest one below it, leaving a partial wave).  The page's first test (no split when
// token * topk > expert) is not kept: it concerns its stage-1 split.  Measured (Mixtral decode
// shapes, same box): T >= 8 (128 tiles) split 2 436 us / 4 440 / 7 436 / 14 441 / none 453
// at T=32, and 467 / 474 / 476 / 492 / 500 us at T=128; T=1 (32 tiles) split 4 151 us,
// 7 135 us, 14 135 us, none 190 us.
static int swap_split_k(int64_t tiles, int kblocks, int units)
{
    if (tiles >= units || tiles <= 0)
        return 1;
    const int64_t need = (units + tiles - 1) / tiles;
    int split = 1;
    for (int d = 2; d <= 16 && d <= kblocks; ++d)
        if (kblocks % d == 0) {
            split = d;
            if (d >= need)
                break;
        }
    return split;
}

static int plan_impl(int dtype, int T, int H, int I, int E, int k, int block_m, int split_k, int num_sms,
                     moe_plan_t *plan, bool grouped_only = false)
{
    int st = validate_shape(dtype, T, H, I, E, k);
    if (st != MOE_OK)
        return st;
    if (!plan || block_m < 0 || split_k < 0)
        return MOE_ERR_INVALID_ARG;
    if (num_sms <= 0) {
        num_sms = num_sms_current_device();
        if (num_sms <= 0)
            return MOE_ERR_CUDA;
    }
    moe_plan_t p;
    memset(&p, 0, sizeof p);
    // Swap (weights on the MMA M side) while every expert segment fits one
    // N <= 128 tile, i.e. T <= 128 (MXFP4: N <= 64, T <= 64); block-scaled
    // FP8 always runs the grouped kernel.
    const int swap_max = (dtype == MOE_MXFP4) ? 64 : 128;
    p.mode = (dtype != MOE_FP8_BLOCK128 && T <= swap_max && !grouped_only) ? MOE_MODE_SWAP : MOE_MODE_GROUPED;
    // Experts that can hold a slot (the tile counts below are upper bounds for them).
    const int64_t e_act = ((int64_t)T * k < E) ? (int64_t)T * k : E;
    if (block_m == 0)
        block_m = (p.mode == MOE_MODE_SWAP) ? swap_block_m(dtype, e_act, I, num_sms) : 128;
    if (p.mode == MOE_MODE_GROUPED && block_m != 128)
        return MOE_ERR_UNSUPPORTED;
    if (p.mode == MOE_MODE_SWAP && (block_m % 16 != 0 || block_m > (dtype == MOE_MXFP4 ? 64 : 128)))
        return MOE_ERR_UNSUPPORTED;
    p.block_m = block_m;
    p.split_k1 = 1;
    const int kblocks2 = I / (dtype == MOE_BF16 ? 64 : dtype == MOE_MXFP4 ? 256 : 128);  // 128-byte K blocks
    if (p.mode == MOE_MODE_SWAP) {
        if (split_k == 0)
            split_k = swap_split_k(e_act * ((H + 255) / 256), kblocks2, num_sms);
        else if (kblocks2 % split_k != 0)
            return MOE_ERR_UNSUPPORTED;
        p.split_k2 = split_k;
    } else {
        if (split_k > 1)
            return MOE_ERR_UNSUPPORTED;
        p.split_k2 = 1;
    }
    p.max_padded = (int64_t)T * k + (int64_t)E * block_m - k;
    p.max_blocks = (p.max_padded + block_m - 1) / block_m;
    p.workspace_bytes = (size_t)make_layout(dtype, T, H, I, E, k, p).total;
    *plan = p;
    return MOE_OK;
}

static int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

static moe_options_t default_options()
{
    moe_options_t o;
    memset(&o, 0, sizeof o);
    o.gemm_pair = -1;
    o.one_stage = 1;
    o.pdl_mask = -1;
    o.light_tiles = -1;
    o.tc_router = -1;
    return o;
}

static int check_options(const moe_options_t &o)
{
    if (o.gemm_pair < -1 || o.gemm_pair > 1 || o.one_stage < 0 || o.one_stage > 1 || o.pdl_mask < -1 ||
        o.pdl_mask > kPdlAll || o.unsatisfiable_h_wait < 0 || o.unsatisfiable_h_wait > 1 || o.light_tiles < -1 ||
        o.light_tiles > 1 || o.tc_router < -1 || o.tc_router > 1)
        return MOE_ERR_INVALID_ARG;
    if (o.stage_events)
        for (int i = 0; i < 7; ++i)
            if (!o.stage_events[i])
                return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

// Records stage mark i on the call's stream when the caller asked for stage events.
static void mark(const moe_options_t &o, int i, cudaStream_t st)
{
    if (o.stage_events)
        cudaEventRecord(static_cast<cudaEvent_t>(o.stage_events[i]), st);
}

// gu (training): when set, the grouped path is forced and stage 1 also keeps
// the pre-activations g | u there for the backward.
static int forward_impl(int dtype, const void *x, const void *W_router, const float *router_bias,
                        const void *W_gate_up, const void *w1_scale, const void *W_down, const void *w2_scale,
                        int T, int H, int I, int E, int k, int block_m, int split_k, void *out, void *ws,
                        size_t ws_bytes, const moe_options_t &o, cudaStream_t st, __nv_bfloat16 *gu = nullptr)
{
    int rc = validate_shape(dtype, T, H, I, E, k);
    if (rc != MOE_OK)
        return rc;
    rc = check_options(o);
    if (rc != MOE_OK)
        return rc;
    if (!x || !W_router || !W_gate_up || !W_down || !out || !ws)
        return MOE_ERR_INVALID_ARG;
    if (dtype != MOE_BF16 && (!w1_scale || !w2_scale || !aligned(w1_scale, 16) || !aligned(w2_scale, 16)))
        return MOE_ERR_INVALID_ARG;
    if (dtype == MOE_BF16 && (w1_scale || w2_scale))
        return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(W_router, 16) || !aligned(W_gate_up, 16) || !aligned(W_down, 16) ||
        !aligned(out, 16) || !aligned(ws, 256))
        return MOE_ERR_INVALID_ARG;
    if (T == 0)
        return MOE_OK;
    moe_plan_t p;
    rc = plan_impl(dtype, T, H, I, E, k, block_m, split_k, 0, &p, gu != nullptr);
    if (rc != MOE_OK)
        return rc;
    if (ws_bytes < p.workspace_bytes)
        return MOE_ERR_WORKSPACE;
    const bool train = gu != nullptr;
    const Layout L = make_layout(dtype, T, H, I, E, k, p);
    uint8_t *w = static_cast<uint8_t *>(ws);
    auto at = [&](int64_t off) -> void * { return off < 0 ? nullptr : (void *)(w + off); };
    const int S = T * k;
    const int nsm = num_sms_current_device();

    int *status = static_cast<int *>(at(L.status));
    const int pdl = o.pdl_mask >= 0 ? o.pdl_mask : pdl_default_mask(p.mode == MOE_MODE_GROUPED);
    mark(o, 0, st);
    int32_t *topk_ids = static_cast<int32_t *>(at(L.topk_ids));
    float *topk_w = static_cast<float *>(at(L.topk_w));
    // The first kernel follows arbitrary caller work.  With programmatic dependent launch it
    // still waits (griddepcontrol.wait) for the preceding kernel to complete before it reads x or
    // zeroes the status words; it only starts early after a kernel that triggers its dependents,
    // such as the previous call's combine.
    const bool tc_router = o.tc_router != 0 && router_tc_eligible(T, H, E, k);
    if (tc_router) {
        if (launch_router_tc(static_cast<const __nv_bfloat16 *>(x), static_cast<const __nv_bfloat16 *>(W_router),
                             router_bias, T, H, E, k, topk_ids, topk_w, static_cast<float *>(at(L.logits)), status,
                             pdl, st) != cudaSuccess)
            return MOE_ERR_CUDA;
    } else if (launch_router(static_cast<const __nv_bfloat16 *>(x), static_cast<const __nv_bfloat16 *>(W_router),
                             router_bias, T, H, E, k, 1, topk_ids, topk_w, static_cast<float *>(at(L.logits)), status,
                             pdl, st) != cudaSuccess) {
        return MOE_ERR_CUDA;
    }
    mark(o, 1, st);

    SortOut so;
    so.sorted_ids = static_cast<int32_t *>(at(L.sorted_ids));
    so.sorted_weights = static_cast<float *>(at(L.sorted_w));
    so.sorted_expert_ids = static_cast<int32_t *>(at(L.sorted_eids));
    so.num_post_padded = static_cast<int32_t *>(at(L.npp));
    so.expert_counts = static_cast<int32_t *>(at(L.counts));
    so.expert_offsets = static_cast<int32_t *>(at(L.offsets));
    so.active_experts = static_cast<int32_t *>(at(L.active));
    so.num_active = static_cast<int32_t *>(at(L.num_active));
    so.slot_pos = static_cast<int32_t *>(at(L.slot_pos));
    if (launch_align_sort(topk_ids, topk_w, T, k, E, p.block_m, so, at(L.sort_scratch), pdl_site(pdl, kPdlSort),
                          pdl_site(pdl, kPdlSort), st) != cudaSuccess)
        return MOE_ERR_CUDA;
    mark(o, 2, st);

    const int64_t P = p.max_padded;
    const int eb = (dtype == MOE_BF16) ? 2 : 1;
    // Light-expert (swap-AB) pair tiles: bf16 grouped mode on CTA pairs, I a multiple of 256.
    // Automatic when the average expert that can hold a slot has fewer than 4 token blocks
    // (fine-grained routing): their kernel keeps one pipeline stage fewer in stage 1, which
    // measured 2-4 % slower on Mixtral prefill, where no expert is light.
    if (o.light_tiles == 1 && (dtype != MOE_BF16 || I % 256 != 0 || !gemm_pair_light_supported(E)))
        return MOE_ERR_UNSUPPORTED;
    const int64_t e_can = ((int64_t)S < E) ? S : E;
    const bool light = dtype == MOE_BF16 && !train && I % 256 == 0 && gemm_pair_light_supported(E) &&
                       (o.light_tiles == 1 || (o.light_tiles == -1 && (int64_t)S < 4LL * 128 * e_can));
    // bf16 decode: both GEMM stages in one persistent launch that also fetches the token rows
    // itself (no gather pass)
    const bool fused = p.mode == MOE_MODE_SWAP && dtype == MOE_BF16 && o.one_stage == 1 && !train;
    // per-token FP8 on the one-SM grouped stage 1: its epilogue takes each row's max |h| (into
    // h_amax, zeroed by the activation quantiser), so h's quantiser needs no reduction pass
    float *h_amax = (dtype == MOE_FP8_TOKEN && p.mode == MOE_MODE_GROUPED && !use_pair(dtype, 1, T, k, E, o.gemm_pair))
                        ? static_cast<float *>(at(L.h_amax))
                        : nullptr;
    cudaError_t ge = cudaSuccess;
    if (fused) {
        // nothing to gather
    } else if (dtype == MOE_BF16 && train)
        ge = launch_gather_rows(static_cast<const __nv_bfloat16 *>(x), so.sorted_ids, so.num_post_padded, S, k, H, P,
                                static_cast<__nv_bfloat16 *>(at(L.x_sorted)), true, pdl_site(pdl, kPdlGather), st);
    else if (dtype == MOE_BF16)
        ge = launch_gather_by_token(static_cast<const __nv_bfloat16 *>(x), so.slot_pos, T, k, H, P,
                                    static_cast<__nv_bfloat16 *>(at(L.x_sorted)), pdl_site(pdl, kPdlGather), st);
    else if (dtype == MOE_FP8_TOKEN)
        ge = launch_quant_rows(static_cast<const __nv_bfloat16 *>(x), so.sorted_ids, so.num_post_padded, P, S, k, H,
                               static_cast<uint8_t *>(at(L.x_sorted)), static_cast<float *>(at(L.x_scales)),
                               pdl_site(pdl, kPdlGather), st, h_amax);
    else if (dtype == MOE_MXFP4)
        // grouped mode keeps the token scales in the tensor core's 128 x 4 blocked order (two 16-byte
        // copies per lane and K step in the GEMM's producer instead of eight 4-byte ones: Mixtral
        // shapes at T=4096, stage 1 0.921 -> 0.852 ms); swap mode re-tiles its few rows itself
        ge = launch_quant_mx4(static_cast<const __nv_bfloat16 *>(x), so.sorted_ids, so.num_post_padded, P, S, k, H,
                              static_cast<uint8_t *>(at(L.x_sorted)), static_cast<uint8_t *>(at(L.x_scales)),
                              p.mode == MOE_MODE_GROUPED, pdl_site(pdl, kPdlGather), st);
    else
        ge = launch_gather_quant_rows(static_cast<const __nv_bfloat16 *>(x), so.sorted_ids, so.num_post_padded, S,
                                      k, H, P, static_cast<uint8_t *>(at(L.x_sorted)),
                                      static_cast<float *>(at(L.x_scales)), pdl_site(pdl, kPdlGather), st);
    if (ge != cudaSuccess)
        return MOE_ERR_CUDA;
    mark(o, 3, st);

    GemmArgs g;
    memset(&g, 0, sizeof g);
    g.sorted_ids = so.sorted_ids;
    g.sorted_weights = so.sorted_weights;
    g.sorted_expert_ids = so.sorted_expert_ids;
    g.num_post_padded = so.num_post_padded;
    g.expert_offsets = so.expert_offsets;
    g.active_experts = so.active_experts;
    g.num_active = so.num_active;
    g.expert_counts = so.expert_counts;
    g.S = S;
    g.E = E;
    g.P_max = P;
    g.status = status;
    g.tile_counter = nullptr;
    g.pdl_mask = pdl;
    const uint32_t box_inner = (uint32_t)(128 / eb);  // one 128-byte swizzle row (elements; bytes for MXFP4)
    const uint64_t kdiv = (dtype == MOE_MXFP4) ? 2 : 1;  // packed FP4: K/2 bytes per row
    const uint32_t box_x_rows = (p.mode == MOE_MODE_SWAP) ? 16 : 128;

    // ---------------------------------------------------------- stage 1
    GemmArgs g1 = g;
    // grouped tiles differ in cost (compute- vs memory-bound experts): claim them dynamically;
    // bf16 / FP8 swap-mode tiles are uniform: deal them round-robin; the short MXFP4 decode
    // tiles balance better claimed (same-box A/B: 0.1488 -> 0.1478 ms per Mixtral decode step)
    g1.tile_counter = (p.mode == MOE_MODE_GROUPED || dtype == MOE_MXFP4) ? status + 1 : nullptr;
    // grouped MXFP4 tiles take weights in 64-row halves (gate/up pairs of 64 rows)
    const uint32_t box_w_rows = (dtype == MOE_MXFP4 && p.mode == MOE_MODE_GROUPED) ? 64 : 128;
    if (!encode_tmap_2d(&g1.tm_x, at(L.x_sorted), eb, H / kdiv, P, box_inner, box_x_rows) ||
        !encode_tmap_2d(&g1.tm_w, W_gate_up, eb, H / kdiv, (uint64_t)E * 2 * I, box_inner, box_w_rows))
        return MOE_ERR_CUDA;
    if (light && !encode_tmap_2d(&g1.tm_x16, at(L.x_sorted), eb, H, P, box_inner, 16))
        return MOE_ERR_CUDA;
    g1.K = H;
    g1.N = I;
    g1.rows_per_expert = 2 * I;
    g1.split_k = 1;
    g1.inter = (dtype == MOE_FP8_TOKEN) ? at(L.inter_h) : at(L.inter);
    g1.x_scales = static_cast<float *>(at(L.x_scales));
    g1.w_scales = static_cast<const float *>(w1_scale);
    g1.inter_scales = static_cast<float *>(at(L.inter_scales));
    g1.gu = gu;
    g1.row_amax = h_amax;

    GemmArgs g2 = g;
    g2.tile_counter = (p.mode == MOE_MODE_GROUPED || dtype == MOE_MXFP4) ? status + 2 : nullptr;
    if (!encode_tmap_2d(&g2.tm_x, at(L.inter), eb, I / kdiv, P, box_inner, box_x_rows) ||
        !encode_tmap_2d(&g2.tm_w, W_down, eb, I / kdiv, (uint64_t)E * H, box_inner, box_w_rows))
        return MOE_ERR_CUDA;
    if (light && !encode_tmap_2d(&g2.tm_x16, at(L.inter), eb, I, P, box_inner, 16))
        return MOE_ERR_CUDA;
    g2.K = I;
    g2.N = H;
    g2.rows_per_expert = H;
    g2.split_k = p.split_k2;
    g2.x_scales = static_cast<float *>(at(L.inter_scales));
    g2.w_scales = static_cast<const float *>(w2_scale);
    g2.y = static_cast<__nv_bfloat16 *>(at(L.y));
    g2.partials = static_cast<float *>(at(L.partials));
    const int nt2 = (H + 255) / 256;
    const int64_t e_act = (S < E) ? S : E;
    cudaError_t ce;

    if (fused) {
        // both stages in one persistent launch (status[1]: tile claims, status[3]: h written)
        FusedArgs F;
        F.s1 = g1;
        F.s2 = g2;
        F.tile_counter = status + 1;
        F.h_done = status + 3;
        F.x = static_cast<const __nv_bfloat16 *>(x);
        F.k = k;
        F.h_wait_ns = o.h_wait_limit_us ? (unsigned long long)o.h_wait_limit_us * 1000ull : 2000000000ull;
        F.h_extra = o.unsatisfiable_h_wait;
        const int64_t ub = e_act * ((I / 128) + nt2 * p.split_k2);
        ce = launch_fused_decode(F, (int)(ub < nsm ? ub : nsm), st);
        if (ce != cudaSuccess)
            return MOE_ERR_CUDA;
        mark(o, 4, st);
        mark(o, 5, st);
    } else {
        if (p.mode == MOE_MODE_SWAP) {
            const int64_t ub = e_act * (I / 128);
            const int grid = (int)(ub < nsm ? ub : nsm);
            ce = (dtype == MOE_BF16)    ? launch_gemm_swap_bf16(1, g1, grid, st)
                 : (dtype == MOE_MXFP4) ? launch_gemm_swap_mx4(1, g1, grid, st)
                                        : launch_gemm_swap_fp8_token(1, g1, grid, st);
        } else if (dtype == MOE_MXFP4) {
            const int64_t ub = p.max_blocks * (I / 64);
            ce = launch_gemm_grouped_mx4(1, g1, (int)(ub < nsm ? ub : nsm), st);
        } else if (use_pair(dtype, 1, T, k, E, o.gemm_pair)) {
            const int64_t ub = (p.max_blocks / 2 + E) * (I / 128);
            ce = (dtype == MOE_FP8_BLOCK128) ? launch_gemm_pair_fp8(1, g1, ub, st)
                                             : launch_gemm_pair(1, dtype == MOE_FP8_TOKEN, g1, ub, st, light);
        } else {
            const int64_t ub = p.max_blocks * (I / 128);
            const int grid = (int)(ub < nsm ? ub : nsm);
            ce = (dtype == MOE_BF16)        ? launch_gemm_grouped_bf16(1, g1, grid, st)
                 : (dtype == MOE_FP8_TOKEN) ? launch_gemm_grouped_fp8_token(1, g1, grid, st)
                                            : launch_gemm_grouped_fp8(1, g1, grid, st);
        }
        if (ce != cudaSuccess)
            return MOE_ERR_CUDA;
        mark(o, 4, st);

        // ------------------------------------------------------ stage 2
        if (dtype == MOE_FP8_TOKEN) {
            // h (bf16, sorted order) -> e4m3 codes with one scale per row (stage 2's input)
            ce = h_amax ? launch_quant_rows_amax(static_cast<const __nv_bfloat16 *>(at(L.inter_h)), h_amax,
                                                 so.num_post_padded, P, I, static_cast<uint8_t *>(at(L.inter)),
                                                 static_cast<float *>(at(L.inter_scales)), pdl_site(pdl, kPdlGather),
                                                 st)
                        : launch_quant_rows(static_cast<const __nv_bfloat16 *>(at(L.inter_h)), nullptr,
                                            so.num_post_padded, P, S, k, I, static_cast<uint8_t *>(at(L.inter)),
                                            static_cast<float *>(at(L.inter_scales)), pdl_site(pdl, kPdlGather), st);
            if (ce != cudaSuccess)
                return MOE_ERR_CUDA;
        }
        if (p.mode == MOE_MODE_SWAP) {
            const int64_t ub = e_act * nt2 * p.split_k2;
            const int grid = (int)(ub < nsm ? ub : nsm);
            ce = (dtype == MOE_BF16)    ? launch_gemm_swap_bf16(2, g2, grid, st)
                 : (dtype == MOE_MXFP4) ? launch_gemm_swap_mx4(2, g2, grid, st)
                                        : launch_gemm_swap_fp8_token(2, g2, grid, st);
        } else if (dtype == MOE_MXFP4) {
            // the scale blocks of h and W_down (blocked order, whole 512-byte tiles per K tile) as TMA
            // rows of 16 bytes; the sorted rows fill whole 128-row blocks, at most P / 128 of them
            if (!encode_tmap_rows16(&g2.tm_sfa, at(L.inter_scales), (uint64_t)(P / 128) * 128 * I / 32, 64) ||
                !encode_tmap_rows16(&g2.tm_sfb, w2_scale, (uint64_t)E * H * I / 32, 64))
                return MOE_ERR_CUDA;
            const int64_t ub = p.max_blocks * (H / 128);
            ce = launch_gemm_grouped_mx4(2, g2, (int)(ub < nsm ? ub : nsm), st);
        } else if (use_pair(dtype, 2, T, k, E, o.gemm_pair)) {
            const int64_t ub = (p.max_blocks / 2 + E) * nt2;
            ce = (dtype == MOE_FP8_BLOCK128) ? launch_gemm_pair_fp8(2, g2, ub, st)
                                             : launch_gemm_pair(2, dtype == MOE_FP8_TOKEN, g2, ub, st, light);
        } else {
            const int64_t ub = p.max_blocks * nt2;
            const int grid = (int)(ub < nsm ? ub : nsm);
            ce = (dtype == MOE_BF16)        ? launch_gemm_grouped_bf16(2, g2, grid, st)
                 : (dtype == MOE_FP8_TOKEN) ? launch_gemm_grouped_fp8_token(2, g2, grid, st)
                                            : launch_gemm_grouped_fp8(2, g2, grid, st);
        }
        if (ce != cudaSuccess)
            return MOE_ERR_CUDA;
        mark(o, 5, st);
    }

    // ----------------------------------------------------------- combine
    if (p.split_k2 > 1)
        ce = launch_splitk_combine(g2.partials, p.split_k2, P, so.slot_pos, topk_w, T, k, H,
                                   static_cast<__nv_bfloat16 *>(out), pdl_site(pdl, kPdlCombine), st);
    else
        ce = launch_combine(g2.y, T, k, H, static_cast<__nv_bfloat16 *>(out), pdl_site(pdl, kPdlCombine), st);
    mark(o, 6, st);
    return cuda_status(ce);
}

// ------------------------------------------------------------ training
//
// Workspace of a training forward + backward: the forward's (grouped plan)
// followed by the saved pre-activations and the backward's buffers.
struct TrainLayout {
    moe_plan_t plan;
    Layout L;
    int64_t gu, dys, dgu, dxs, dlogit, wdT, wguT, dysT, hT, dguT, xsT, rg_part, total;
    int64_t Pp;  // row length of the transposed activations (>= max_padded, multiple of 64)
};

static int train_layout(int T, int H, int I, int E, int k, TrainLayout &TL)
{
    int rc = validate_shape(MOE_BF16, T, H, I, E, k);
    if (rc != MOE_OK)
        return rc;
    if (I % 256 != 0)
        return MOE_ERR_UNSUPPORTED;  // the backward of stage 2 works in 256-column tiles of I
    rc = plan_impl(MOE_BF16, T, H, I, E, k, 128, 0, 0, &TL.plan, true);
    if (rc != MOE_OK)
        return rc;
    TL.L = make_layout(MOE_BF16, T, H, I, E, k, TL.plan);
    const int64_t P = TL.plan.max_padded, S = (int64_t)T * k;
    TL.Pp = align_up(P, 64);
    int64_t off = align_up((int64_t)TL.plan.workspace_bytes, kAlign);
    auto take = [&](int64_t bytes) {
        const int64_t o = off;
        off = align_up(off + bytes, kAlign);
        return o;
    };
    TL.gu = take(P * 2 * I * 2);
    TL.dys = take(P * H * 2);
    TL.dgu = take(P * 2 * I * 2);
    TL.dxs = take(S * H * 2);
    TL.dlogit = take((int64_t)T * E * 4);
    TL.wdT = take((int64_t)E * I * H * 2);
    TL.wguT = take((int64_t)E * H * 2 * I * 2);
    TL.dysT = take(H * TL.Pp * 2);
    TL.hT = take(I * TL.Pp * 2);
    TL.dguT = take(2 * I * TL.Pp * 2);
    TL.xsT = take(H * TL.Pp * 2);
    TL.rg_part = take(router_wgrad_scratch(T, E, H) * 4);
    TL.total = off;
    return MOE_OK;
}

static int backward_impl(const void *x, const void *W_router, const void *W_gate_up, const void *W_down,
                         const void *dout, int T, int H, int I, int E, int k, void *dx, float *dW_gate_up,
                         float *dW_down, float *dW_router, float *dbias, void *ws, size_t ws_bytes,
                         const moe_options_t &o, cudaStream_t st)
{
    if (check_options(o) != MOE_OK)
        return MOE_ERR_INVALID_ARG;
    TrainLayout TL;
    int rc = train_layout(T, H, I, E, k, TL);
    if (rc != MOE_OK)
        return rc;
    if (!x || !W_router || !W_gate_up || !W_down || !dout || !dx || !dW_gate_up || !dW_down || !dW_router || !ws)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(dout, 16) || !aligned(dx, 16) || !aligned(W_gate_up, 16) ||
        !aligned(W_down, 16) || !aligned(dW_gate_up, 16) || !aligned(dW_down, 16) || !aligned(ws, 256))
        return MOE_ERR_INVALID_ARG;
    if ((size_t)TL.total > ws_bytes)
        return MOE_ERR_WORKSPACE;
    const Layout &L = TL.L;
    const moe_plan_t &p = TL.plan;
    uint8_t *w = static_cast<uint8_t *>(ws);
    auto at = [&](int64_t off) -> void * { return off < 0 ? nullptr : (void *)(w + off); };
    auto bf = [&](int64_t off) { return static_cast<__nv_bfloat16 *>(at(off)); };
    const int S = T * k;
    const int64_t P = p.max_padded;
    const int nsm = num_sms_current_device();
    int *status = static_cast<int *>(at(L.status));

    BackwardAux b;
    memset(&b, 0, sizeof b);
    b.dout = static_cast<const __nv_bfloat16 *>(dout);
    b.x = static_cast<const __nv_bfloat16 *>(x);
    b.Wr = static_cast<const __nv_bfloat16 *>(W_router);
    b.sorted_ids = static_cast<const int32_t *>(at(L.sorted_ids));
    b.sorted_w = static_cast<const float *>(at(L.sorted_w));
    b.npp = static_cast<const int32_t *>(at(L.npp));
    b.Y = static_cast<const __nv_bfloat16 *>(at(L.y));
    b.topk_ids = static_cast<const int32_t *>(at(L.topk_ids));
    b.topk_w = static_cast<const float *>(at(L.topk_w));
    b.T = T;
    b.k = k;
    b.E = E;
    b.H = H;
    b.P_max = P;
    b.dys = bf(TL.dys);
    b.dlogit = static_cast<float *>(at(TL.dlogit));
    b.dxs = static_cast<const __nv_bfloat16 *>(at(TL.dxs));
    b.dx = static_cast<__nv_bfloat16 *>(dx);
    b.dWr = dW_router;
    b.dbias = dbias;
    b.rg_part = static_cast<float *>(at(TL.rg_part));
    if (launch_backward_aux(0, b, st) != cudaSuccess || launch_backward_aux(1, b, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    // CTA pairs under the same rule as the forward's GEMMs.  The pair kernels read the weights of
    // both backward GEMMs in their stored layout as MN-major operands; the one-SM kernels read
    // K-major rows, from transposed copies.
    const bool pairs = use_pair(MOE_BF16, 1, T, k, E, o.gemm_pair);
    if (!pairs &&
        (launch_transpose(static_cast<const __nv_bfloat16 *>(W_down), bf(TL.wdT), E, H, I, H, st) != cudaSuccess ||
         launch_transpose(static_cast<const __nv_bfloat16 *>(W_gate_up), bf(TL.wguT), E, 2 * I, H, 2 * I, st) !=
             cudaSuccess))
        return MOE_ERR_CUDA;

    GemmArgs g;
    memset(&g, 0, sizeof g);
    g.sorted_ids = b.sorted_ids;
    g.sorted_expert_ids = static_cast<const int32_t *>(at(L.sorted_eids));
    g.num_post_padded = b.npp;
    g.expert_offsets = static_cast<const int32_t *>(at(L.offsets));
    g.active_experts = static_cast<const int32_t *>(at(L.active));
    g.num_active = static_cast<const int32_t *>(at(L.num_active));
    g.expert_counts = static_cast<const int32_t *>(at(L.counts));
    g.S = S;
    g.E = E;
    g.P_max = P;
    g.split_k = 1;
    g.status = status;

    // dh = dY W_down, with SwiGLU's backward in the epilogue -> dg | du
    GemmArgs g3 = g;
    if (!encode_tmap_2d(&g3.tm_x, at(TL.dys), 2, H, P, 64, 128) ||
        !(pairs ? encode_tmap_2d(&g3.tm_w, W_down, 2, I, (uint64_t)E * H, 64, 64)  // [E*H][I]: K rows, N columns
                : encode_tmap_2d(&g3.tm_w, at(TL.wdT), 2, H, (uint64_t)E * I, 64, 128)))
        return MOE_ERR_CUDA;
    g3.K = H;
    g3.N = I;
    g3.rows_per_expert = I;
    g3.gu_in = bf(TL.gu);
    g3.dgu = bf(TL.dgu);
    g3.tile_counter = status + 1;
    if (cudaMemsetAsync(status + 1, 0, sizeof(int), st) != cudaSuccess)
        return MOE_ERR_CUDA;
    int64_t ub = p.max_blocks * (I / 256);
    if ((pairs ? launch_gemm_pair(3, 0, g3, (p.max_blocks / 2 + E) * (I / 256), st, false, true)
               : launch_gemm_backward_bf16(3, g3, (int)(ub < nsm ? ub : nsm), st)) != cudaSuccess)
        return MOE_ERR_CUDA;

    // dx per slot = dg W_gate + du W_up (stage 2's tile shape, unit weights)
    GemmArgs g2 = g;
    if (!encode_tmap_2d(&g2.tm_x, at(TL.dgu), 2, 2 * I, P, 64, 128) ||
        !(pairs ? encode_tmap_2d(&g2.tm_w, W_gate_up, 2, H, (uint64_t)E * 2 * I, 64, 64)  // [E*2I][H]
                : encode_tmap_2d(&g2.tm_w, at(TL.wguT), 2, 2 * I, (uint64_t)E * H, 64, 128)))
        return MOE_ERR_CUDA;
    g2.K = 2 * I;
    g2.N = H;
    g2.rows_per_expert = H;
    g2.sorted_weights = nullptr;
    g2.y = static_cast<__nv_bfloat16 *>(at(TL.dxs));
    g2.tile_counter = status + 1;
    if (cudaMemsetAsync(status + 1, 0, sizeof(int), st) != cudaSuccess)
        return MOE_ERR_CUDA;
    ub = p.max_blocks * ((H + 255) / 256);
    if ((pairs ? launch_gemm_pair(2, 0, g2, (p.max_blocks / 2 + E) * ((H + 255) / 256), st, false, true)
               : launch_gemm_backward_bf16(2, g2, (int)(ub < nsm ? ub : nsm), st)) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (launch_backward_aux(2, b, st) != cudaSuccess)
        return MOE_ERR_CUDA;

    // weight gradients, K over each expert's token positions: on CTA pairs (gradient rows a multiple
    // of 256) both activations are read as stored, [P][rows], as MN-major operands; the one-SM
    // kernel reads K-major rows of transposed copies [rows][P]
    const int64_t Pp = TL.Pp;
    struct WG {
        int64_t a_src, b_src, a_off, b_off;
        int M, N;
        float *out;
    } wg[2] = {{TL.dys, L.inter, TL.dysT, TL.hT, H, I, dW_down}, {TL.dgu, L.x_sorted, TL.dguT, TL.xsT, 2 * I, H, dW_gate_up}};
    for (const WG &q : wg) {
        const bool pair5 = pairs && q.M % 256 == 0;  // pair tiles span 256 gradient rows
        GemmArgs g5 = g;
        if (pair5) {
            if (!encode_tmap_2d(&g5.tm_x, at(q.a_src), 2, q.M, P, 64, 64) ||
                !encode_tmap_2d(&g5.tm_w, at(q.b_src), 2, q.N, P, 64, 64))
                return MOE_ERR_CUDA;
            g5.K = (int)P;
        } else {
            if (launch_transpose(bf(q.a_src), bf(q.a_off), 1, P, q.M, Pp, st) != cudaSuccess ||
                launch_transpose(bf(q.b_src), bf(q.b_off), 1, P, q.N, Pp, st) != cudaSuccess)
                return MOE_ERR_CUDA;
            if (!encode_tmap_2d(&g5.tm_x, at(q.a_off), 2, Pp, q.M, 64, 128) ||
                !encode_tmap_2d(&g5.tm_w, at(q.b_off), 2, Pp, q.N, 64, 128))
                return MOE_ERR_CUDA;
            g5.K = (int)Pp;
        }
        g5.M = q.M;
        g5.N = q.N;
        g5.dw_out = q.out;
        g5.tile_counter = status + 1;  // tiles of unequal K (segment lengths): claimed dynamically
        if (cudaMemsetAsync(status + 1, 0, sizeof(int), st) != cudaSuccess)
            return MOE_ERR_CUDA;
        const int64_t tiles = (int64_t)E * (q.M / 128) * ((q.N + 255) / 256);
        if ((pair5 ? launch_gemm_pair(5, 0, g5, tiles / 2, st, false, true)
                   : launch_gemm_backward_bf16(5, g5, (int)(tiles < nsm ? tiles : nsm), st)) != cudaSuccess)
            return MOE_ERR_CUDA;
    }
    if (launch_backward_aux(3, b, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" {

const char *moe_status_string(int status)
{
    switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or option";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
    }
}

int moe_version(void) { return 100; }

int moe_options_init(moe_options_t *options)
{
    if (!options)
        return MOE_ERR_INVALID_ARG;
    *options = default_options();
    return MOE_OK;
}

int moe_align_sort_sizes(int T, int k, int E, int block_m, int64_t *max_padded, int64_t *max_blocks)
{
    if (T < 0 || k <= 0 || E <= 0 || block_m <= 0 || !max_padded || !max_blocks)
        return MOE_ERR_INVALID_ARG;
    const int64_t p = (int64_t)T * k + (int64_t)E * block_m - k;
    *max_padded = p;
    *max_blocks = (p + block_m - 1) / block_m;
    return MOE_OK;
}

int moe_block_size_m_heuristic(int token, int topk, int expert, int inter_dim, int units, const int *candidates,
                               int n)
{
    if (token < 0 || topk <= 0 || expert <= 0 || inter_dim <= 0 || units <= 0 || !candidates || n <= 0)
        return MOE_ERR_INVALID_ARG;
    const int64_t tgN = (inter_dim + 127) / 128;
    int best = -1;
    int64_t best_r = 0, best_idle = 0;
    for (int i = 0; i < n; ++i) {
        const int bm = candidates[i];
        if (bm <= 0)
            return MOE_ERR_INVALID_ARG;
        const int64_t padded = (int64_t)token * topk + (int64_t)expert * bm - topk;
        // the page's tgN * (max + bm - 1) // bm, grouped as Python groups it (left to right)
        const int64_t tiles = tgN * (padded + bm - 1) / bm;
        const int64_t rounds = (tiles + units - 1) / units;
        const int64_t idle = units - tiles % units;
        // fewest rounds, then fewest idle units; a full tie keeps the earlier candidate
        if (best < 0 || rounds < best_r || (rounds == best_r && idle < best_idle)) {
            best = bm;
            best_r = rounds;
            best_idle = idle;
        }
    }
    return best;
}

int moe_ksplit_heuristic(int token, int topk, int expert, int inter_dim, int model_dim, int units, int block_m)
{
    if (token < 0 || topk <= 0 || expert <= 0 || inter_dim <= 0 || model_dim <= 0 || units <= 0 || block_m <= 0)
        return MOE_ERR_INVALID_ARG;
    if ((int64_t)token * topk > expert)
        return 0;
    const int64_t tgN = (inter_dim + 127) / 128;
    const int64_t tgM = ((int64_t)token * topk + block_m - 1) / block_m;
    const int64_t tiles = tgN * tgM;
    if (tiles >= units || tiles == 0)
        return 0;
    const int64_t split_max = (units + tiles - 1) / tiles;
    for (int64_t i = split_max; i >= 2; --i)
        if (model_dim % i == 0 && (model_dim / i) % 256 == 0)
            return (int)i;
    return 0;
}

int moe_plan(int dtype, int T, int H, int I, int E, int k, int block_m, int split_k, int num_sms, moe_plan_t *plan)
{
    return plan_impl(dtype, T, H, I, E, k, block_m, split_k, num_sms, plan);
}

size_t moe_fused_workspace_size(int dtype, int T, int H, int I, int E, int k, int block_m, int split_k)
{
    moe_plan_t p;
    if (plan_impl(dtype, T, H, I, E, k, block_m, split_k, 0, &p) != MOE_OK)
        return 0;
    return p.workspace_bytes;
}

int moe_workspace_layout(int dtype, int T, int H, int I, int E, int k, int block_m, int split_k,
                         moe_ws_layout_t *out)
{
    if (!out)
        return MOE_ERR_INVALID_ARG;
    moe_plan_t p;
    int rc = plan_impl(dtype, T, H, I, E, k, block_m, split_k, 0, &p);
    if (rc != MOE_OK)
        return rc;
    const Layout L = make_layout(dtype, T, H, I, E, k, p);
    out->status = L.status;
    out->topk_ids = L.topk_ids;
    out->topk_weights = L.topk_w;
    out->sorted_ids = L.sorted_ids;
    out->sorted_weights = L.sorted_w;
    out->sorted_expert_ids = L.sorted_eids;
    out->num_tokens_post_padded = L.npp;
    out->expert_counts = L.counts;
    out->x_sorted = L.x_sorted;
    out->x_scales = L.x_scales;
    out->inter = L.inter;
    out->inter_scales = L.inter_scales;
    out->inter_h = L.inter_h;
    out->y = L.y;
    out->router_logits = L.logits;
    out->total = L.total;
    return MOE_OK;
}

int moe_workspace_status(const void *ws, int *status, void *stream)
{
    if (!ws || !status)
        return MOE_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int v = 0;
    if (cudaMemcpyAsync(&v, ws, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return MOE_ERR_CUDA;
    *status = v;
    return MOE_OK;
}

int moe_route_topk(const void *x, const void *W_router, const float *bias, int T, int H, int E, int k,
                   int renormalize, int32_t *topk_ids, float *topk_weights, float *logits, void *stream)
{
    if (T < 0 || H <= 0 || H % 8 != 0 || E <= 0 || k <= 0 || renormalize < 0 || renormalize > 1)
        return MOE_ERR_INVALID_ARG;
    if (E > 1024 || k > E || k > 32)
        return MOE_ERR_UNSUPPORTED;
    if (T == 0)
        return MOE_OK;
    if (!x || !W_router || !topk_ids || !topk_weights || !aligned(x, 16) || !aligned(W_router, 16))
        return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_router(static_cast<const __nv_bfloat16 *>(x),
                                     static_cast<const __nv_bfloat16 *>(W_router), bias, T, H, E, k, renormalize,
                                     topk_ids, topk_weights, logits, nullptr, 1 << kPdlTopk,
                                     static_cast<cudaStream_t>(stream)));
}

size_t moe_align_sort_workspace_size(int T, int k, int E)
{
    if (T < 0 || k <= 0 || E <= 0)
        return 0;
    return (size_t)align_up((int64_t)sort_scratch_bytes(T, k, E), kAlign) + (size_t)(E + 1) * 4;
}

int moe_align_sort(const int32_t *topk_ids, const float *topk_weights, int T, int k, int E, int block_m,
                   int32_t *sorted_ids, float *sorted_weights, int32_t *sorted_expert_ids,
                   int32_t *num_tokens_post_padded, int32_t *expert_counts, void *ws, size_t ws_bytes, void *stream)
{
    if (T < 0 || k <= 0 || E <= 0 || block_m <= 0)
        return MOE_ERR_INVALID_ARG;
    if (E > 1024 || k > E)
        return MOE_ERR_UNSUPPORTED;
    if ((int64_t)T * k > (int64_t)1 << 30)
        return MOE_ERR_UNSUPPORTED;
    if (!topk_ids || !topk_weights || !sorted_ids || !sorted_weights || !sorted_expert_ids ||
        !num_tokens_post_padded || !ws)
        return MOE_ERR_INVALID_ARG;
    if (ws_bytes < moe_align_sort_workspace_size(T, k, E))
        return MOE_ERR_WORKSPACE;
    SortOut so;
    memset(&so, 0, sizeof so);
    so.sorted_ids = sorted_ids;
    so.sorted_weights = sorted_weights;
    so.sorted_expert_ids = sorted_expert_ids;
    so.num_post_padded = num_tokens_post_padded;
    so.expert_counts = expert_counts;
    so.expert_offsets = reinterpret_cast<int32_t *>(static_cast<uint8_t *>(ws) +
                                                    align_up((int64_t)sort_scratch_bytes(T, k, E), kAlign));
    return cuda_status(launch_align_sort(topk_ids, topk_weights, T, k, E, block_m, so, ws, false, true,
                                         static_cast<cudaStream_t>(stream)));
}

int moe_quantize_fp8_act(const void *X, int64_t R, int C, uint8_t *q, float *s, void *stream)
{
    if (R < 0 || C <= 0 || C % 128 != 0 || !X || !q || !s || !aligned(X, 16) || !aligned(q, 8))
        return MOE_ERR_INVALID_ARG;
    launch_quant_act(static_cast<const __nv_bfloat16 *>(X), R, C, q, s, static_cast<cudaStream_t>(stream));
    return cuda_status(cudaGetLastError());
}

int moe_quantize_fp8_weights(const void *W, int64_t R, int C, uint8_t *q, float *s, void *stream)
{
    if (R < 0 || R % 128 != 0 || C <= 0 || C % 128 != 0 || R / 128 > 65535 || !W || !q || !s || !aligned(W, 16) ||
        !aligned(q, 8))
        return MOE_ERR_INVALID_ARG;
    launch_quant_weights(static_cast<const __nv_bfloat16 *>(W), R, C, q, s, static_cast<cudaStream_t>(stream));
    return cuda_status(cudaGetLastError());
}

int moe_quantize_mxfp4(const void *X, int64_t R, int C, uint8_t *q, uint8_t *s, int tiled, void *stream)
{
    if (R < 0 || C <= 0 || C % 32 != 0 || !X || !q || !s || !aligned(X, 16) || !aligned(q, 4))
        return MOE_ERR_INVALID_ARG;
    if (tiled && (R % 128 != 0 || C % 128 != 0))
        return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_quant_mx4(static_cast<const __nv_bfloat16 *>(X), nullptr, nullptr, R, 0, 1, C, q, s,
                                        tiled != 0, false, static_cast<cudaStream_t>(stream)));
}

int moe_quantize_fp8_rows(const void *X, int64_t R, int C, uint8_t *q, float *s, void *stream)
{
    if (R < 0 || C <= 0 || C % 16 != 0 || !X || !q || !s || !aligned(X, 16) || !aligned(q, 16))
        return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_quant_rows(static_cast<const __nv_bfloat16 *>(X), nullptr, nullptr, R, 0, 1, C, q, s,
                                         false, static_cast<cudaStream_t>(stream)));
}

int moe_fused_forward(int dtype, const void *x, const void *W_router, const float *router_bias,
                      const void *W_gate_up, const void *w1_scale, const void *W_down, const void *w2_scale, int T,
                      int H, int I, int E, int k, int block_m, int split_k, void *out, void *ws, size_t ws_bytes,
                      void *stream)
{
    return forward_impl(dtype, x, W_router, router_bias, W_gate_up, w1_scale, W_down, w2_scale, T, H, I, E, k,
                        block_m, split_k, out, ws, ws_bytes, default_options(), static_cast<cudaStream_t>(stream));
}

int moe_fused_forward_ex(int dtype, const void *x, const void *W_router, const float *router_bias,
                         const void *W_gate_up, const void *w1_scale, const void *W_down, const void *w2_scale, int T,
                         int H, int I, int E, int k, int block_m, int split_k, void *out, void *ws, size_t ws_bytes,
                         const moe_options_t *options, void *stream)
{
    return forward_impl(dtype, x, W_router, router_bias, W_gate_up, w1_scale, W_down, w2_scale, T, H, I, E, k,
                        block_m, split_k, out, ws, ws_bytes, options ? *options : default_options(),
                        static_cast<cudaStream_t>(stream));
}

size_t moe_train_workspace_size(int T, int H, int I, int E, int k)
{
    TrainLayout TL;
    if (train_layout(T, H, I, E, k, TL) != MOE_OK)
        return 0;
    return (size_t)TL.total;
}

int moe_fused_forward_train(const void *x, const void *W_router, const float *router_bias, const void *W_gate_up,
                            const void *W_down, int T, int H, int I, int E, int k, void *out, void *ws,
                            size_t ws_bytes, const moe_options_t *options, void *stream)
{
    if (options && check_options(*options) != MOE_OK)
        return MOE_ERR_INVALID_ARG;
    TrainLayout TL;
    int rc = train_layout(T, H, I, E, k, TL);
    if (rc != MOE_OK)
        return rc;
    if (!ws || (size_t)TL.total > ws_bytes)
        return !ws ? MOE_ERR_INVALID_ARG : MOE_ERR_WORKSPACE;
    return forward_impl(MOE_BF16, x, W_router, router_bias, W_gate_up, nullptr, W_down, nullptr, T, H, I, E, k, 128,
                        0, out, ws, TL.plan.workspace_bytes, options ? *options : default_options(),
                        static_cast<cudaStream_t>(stream),
                        reinterpret_cast<__nv_bfloat16 *>(static_cast<uint8_t *>(ws) + TL.gu));
}

int moe_fused_backward(const void *x, const void *W_router, const float *router_bias, const void *W_gate_up,
                       const void *W_down, const void *dout, int T, int H, int I, int E, int k, void *dx,
                       float *dW_gate_up, float *dW_down, float *dW_router, float *dbias, void *ws, size_t ws_bytes,
                       const moe_options_t *options, void *stream)
{
    if (options && check_options(*options) != MOE_OK)
        return MOE_ERR_INVALID_ARG;
    (void)router_bias;  // enters the backward only through the routing kept by the training forward
    if (T == 0)
        return MOE_OK;
    return backward_impl(x, W_router, W_gate_up, W_down, dout, T, H, I, E, k, dx, dW_gate_up, dW_down, dW_router,
                         dbias, ws, ws_bytes, options ? *options : default_options(),
                         static_cast<cudaStream_t>(stream));
}

size_t moe_host_staging_bytes(int T, int H)
{
    if (T < 0 || H <= 0)
        return 0;
    return (size_t)align_up((int64_t)T * H * 2, kAlign) * 2;
}

int moe_fused_forward_host(int dtype, const void *x_host, const void *W_router, const float *router_bias,
                           const void *W_gate_up, const void *w1_scale, const void *W_down, const void *w2_scale,
                           int T, int H, int I, int E, int k, int block_m, int split_k, void *out_host, void *ws,
                           size_t ws_bytes, void *stream)
{
    int rc = validate_shape(dtype, T, H, I, E, k);
    if (rc != MOE_OK)
        return rc;
    if (!x_host || !out_host || !ws)
        return MOE_ERR_INVALID_ARG;
    if (T == 0)
        return MOE_OK;
    const size_t need = moe_fused_workspace_size(dtype, T, H, I, E, k, block_m, split_k);
    if (need == 0)
        return MOE_ERR_INVALID_ARG;
    const size_t stage = moe_host_staging_bytes(T, H);
    if (ws_bytes < need + stage)
        return MOE_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t *base = static_cast<uint8_t *>(ws) + need;
    void *x_dev = base;
    void *out_dev = base + stage / 2;
    const size_t bytes = (size_t)T * H * 2;
    if (cudaMemcpyAsync(x_dev, x_host, bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    rc = forward_impl(dtype, x_dev, W_router, router_bias, W_gate_up, w1_scale, W_down, w2_scale, T, H, I, E, k,
                      block_m, split_k, out_dev, ws, need, default_options(), st);
    if (rc != MOE_OK)
        return rc;
    if (cudaMemcpyAsync(out_host, out_dev, bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

}  // extern "C"
