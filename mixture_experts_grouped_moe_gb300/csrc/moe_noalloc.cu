// moe_align_sort_noalloc: the token sort by expert for callers that cannot
// allocate device memory themselves.  Its scratch (the per-chunk expert
// histograms and the padded expert offsets) lives in a fixed array in the
// library's own device memory instead of a caller-provided workspace.
//
// The array's name in host code is only a host-side stand-in for the device
// symbol, never a device address, so its address on the current device is
// looked up with cudaGetSymbolAddress and that pointer is what the kernels
// receive.
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int64_t kScratchInts = MOE_NOALLOC_SORT_SCRATCH_BYTES / 4;

// Every GPU that loads the library holds this array until the process exits.
static __device__ __align__(256) int32_t g_sort_scratch[kScratchInts];

// Device address of g_sort_scratch on the current device, looked up on every call: the
// lookup allocates nothing and costs far less than the sort, and a cached address would go
// stale after cudaDeviceReset, when the module (and this array) is loaded again in a new
// primary context, possibly elsewhere.  The first lookup on a device may load the library's
// device code there.
int scratch_on_current_device(int32_t **out)
{
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_sort_scratch) != cudaSuccess || !p)
        return MOE_ERR_CUDA;
    *out = static_cast<int32_t *>(p);
    return MOE_OK;
}

}  // namespace

}  // namespace moe

extern "C" int moe_align_sort_noalloc(const int32_t *topk_ids, const float *topk_weights, int T, int k, int E,
                                      int block_m, int32_t *sorted_ids, float *sorted_weights,
                                      int32_t *sorted_expert_ids, int32_t *num_tokens_post_padded,
                                      int32_t *expert_counts, void *stream)
{
    using namespace moe;
    if (T < 0 || k <= 0 || E <= 0 || block_m <= 0)
        return MOE_ERR_INVALID_ARG;
    if (E > 1024 || k > E || (int64_t)T * k > (int64_t)1 << 30)
        return MOE_ERR_UNSUPPORTED;
    if (!topk_ids || !topk_weights || !sorted_ids || !sorted_weights || !sorted_expert_ids ||
        !num_tokens_post_padded)
        return MOE_ERR_INVALID_ARG;
    // scratch: chunk histograms [nchunks][E], then the E+1 padded offsets (64-int aligned)
    const int64_t cc_ints = (int64_t)sort_scratch_bytes(T, k, E) / 4;
    const int64_t off_at = (cc_ints + 63) / 64 * 64;
    if (off_at + E + 1 > kScratchInts)
        return MOE_ERR_UNSUPPORTED;  // beyond the fixed scratch: use moe_align_sort with a workspace
    int32_t *scratch = nullptr;
    const int rc = scratch_on_current_device(&scratch);
    if (rc != MOE_OK)
        return rc;
    // No word of the scratch needs to start at zero: the count pass writes every histogram
    // entry and the scan pass every offset before anything reads them.
    SortOut so = {};
    so.sorted_ids = sorted_ids;
    so.sorted_weights = sorted_weights;
    so.sorted_expert_ids = sorted_expert_ids;
    so.num_post_padded = num_tokens_post_padded;
    so.expert_counts = expert_counts;
    so.expert_offsets = scratch + off_at;
    const cudaError_t err =
        launch_align_sort(topk_ids, topk_weights, T, k, E, block_m, so, scratch, false, true,
                          static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
