// Inline-PTX wrappers for the Blackwell (sm_100 family, built for sm_103a)
// asynchronous machinery used by the group-GEMM kernels: mbarriers, TMA
// tensor copies, and the 5th-generation tensor core (tcgen05) with its
// tensor memory (TMEM).  Every wait is bounded: after kWaitLimitNs the
// waiting thread records MOE_ERR_TIMEOUT and gives up instead of spinning.
#pragma once

#include <cstdint>

namespace moe {

constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bring the 128-byte line holding p into L2 (no register written, nothing waited for).
__device__ __forceinline__ void prefetch_l2(const void *p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// ------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// try_wait that lets the thread sleep (up to the hint, 0.1 ms) until the phase
// completes, so waiting warps do not take issue slots from working ones.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity), "r"(100000u)
        : "memory");
    return done != 0;
}

// Retire `bytes` of the current phase's expected transaction count without a
// copy (for bytes announced with expect_tx whose copies will not be issued),
// so that the phase completes once the copies that were issued have landed.
__device__ __forceinline__ void mbar_complete_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.complete_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// Wait until the phase with the given parity has completed.  Returns false
// (after recording a timeout in *status and raising *abort) if it does not
// within the limit, or if another role of the CTA has already aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int *status, volatile int *abort)
{
    if (mbar_try_wait(bar, parity))
        return true;
    unsigned long long t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_sleep(bar, parity))
            return true;
        if ((it & 15u) == 0) {
            if (*abort)
                return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                atomicExch(status, -5 /* MOE_ERR_TIMEOUT */);
                *abort = 1;
                return false;
            }
        }
    }
}

// ------------------------------------------------ dynamic tile queue
//
// Persistent GEMM CTAs claim tiles from a global counter (atomicAdd), so
// that tiles of uneven cost (a memory-bound tile of a lightly loaded expert
// next to a compute-bound one) balance across SMs.  The producer thread
// claims; the index reaches the MMA thread and the epilogue warps through a
// ring of kTileQ shared-memory slots guarded by mbarriers (full: 1 producer
// arrival; empty: one arrival per consumer).  Index -1 means "no more tiles".
constexpr int kTileQ = 4;

struct TileQueue {
    int idx[kTileQ];
    uint64_t full[kTileQ];
    uint64_t empty[kTileQ];
};

__device__ __forceinline__ void tq_init(TileQueue &q, uint32_t consumers)
{
    for (int i = 0; i < kTileQ; ++i) {
        mbar_init(&q.full[i], 1);
        mbar_init(&q.empty[i], consumers);
    }
}

// Producer: publish the next tile index t (claimed from *counter, or -1 past ntiles).
// Consumer (tq_pop): read the next index, then arrive on q.empty[slot] once every
// thread of the consumer has read it, and tq_advance.
__device__ __forceinline__ bool tq_push_next(TileQueue &q, int &slot, uint32_t &ph, int *counter, int ntiles,
                                             int &claim, int &t, int *status, volatile int *abort)
{
    // `claim` holds the tile claimed on the previous call (-2 before the first one): the
    // next claim is issued right after publishing, so its latency overlaps this tile's loads.
    // Without a counter the tiles are dealt round-robin (blockIdx.x, + gridDim.x, ...).
    if (claim == -2)
        claim = counter ? atomicAdd(counter, 1) : (int)blockIdx.x;
    if (!mbar_wait(&q.empty[slot], ph ^ 1, status, abort))
        return false;
    t = (claim < ntiles) ? claim : -1;
    *reinterpret_cast<volatile int *>(&q.idx[slot]) = t;
    mbar_arrive(&q.full[slot]);
    if (++slot == kTileQ) {
        slot = 0;
        ph ^= 1;
    }
    if (t >= 0)
        claim = counter ? atomicAdd(counter, 1) : claim + (int)gridDim.x;
    return true;
}

__device__ __forceinline__ bool tq_pop(TileQueue &q, int slot, uint32_t ph, int &t, int *status,
                                       volatile int *abort)
{
    if (!mbar_wait(&q.full[slot], ph, status, abort))
        return false;
    t = *reinterpret_cast<volatile int *>(&q.idx[slot]);
    return true;
}

__device__ __forceinline__ void tq_advance(int &slot, uint32_t &ph)
{
    if (++slot == kTileQ) {
        slot = 0;
        ph ^= 1;
    }
}

// --------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const void *tmap)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_normal()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 2-D tiled load of the box at (x = inner coordinate, y = row) into shared
// memory, completing `bytes` on the mbarrier.
__device__ __forceinline__ void tma_load_2d(void *dst, const void *tmap, int x, int y, uint64_t *bar,
                                            uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Non-tensor bulk copy global -> this CTA's shared memory (16-byte aligned
// addresses, size a multiple of 16), completing `bytes` on the mbarrier.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst)),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

// 4- / 8-byte asynchronous copies global -> shared (cp.async), and an arrival
// on an mbarrier once all of this thread's earlier cp.async copies have
// landed (.noinc: the barrier's expected count includes these arrivals).
__device__ __forceinline__ void cp_async_4(void *dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_8(void *dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}

// 16-byte asynchronous copy global -> shared; with valid == false the 16 bytes are zero-filled
// and nothing is read.
__device__ __forceinline__ void cp_async_16_zfill(void *dst, const void *src, bool valid)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}

__device__ __forceinline__ void cp_async_arrive(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Orders this thread's ordinary shared-memory writes before later reads of
// the async proxy (TMA, tcgen05.cp, tcgen05.mma).
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------- clusters (CTA pairs)
//
// Two-SM tensor-core operations (tcgen05 .cta_group::2) run on a pair of
// CTAs of one cluster whose ranks differ in bit 0.  Rank 0 (the leader)
// issues the MMAs; the pair's shared memories hold one half of each operand
// and each CTA's TMEM one half of the accumulator rows.

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// The shared::cluster address of the same variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(const void *p, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
    return r;
}

// All threads of both CTAs: arrive and wait (release / acquire at cluster scope).
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 32-bit store to a shared::cluster address (possibly in the peer CTA).
__device__ __forceinline__ void st_cluster_s32(uint32_t cluster_addr, int v)
{
    asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// Arrive on an mbarrier given by its shared::cluster address (possibly in the peer CTA).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Arrive on an mbarrier of either CTA of the cluster with the default semantics (release at CTA
// scope), for a signal that publishes no data the other CTA reads -- "this CTA has finished
// reading its TMEM buffer" -- and so needs no cluster-scope release, whose fence would first wait
// for the thread's global loads in flight.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// try_wait with acquire at cluster scope: sees the peer CTA's writes released by its arrive.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity), "r"(100000u)
        : "memory");
    return done != 0;
}

// Bounded wait as mbar_wait, with cluster-scope acquire.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t *bar, uint32_t parity, int *status, volatile int *abort)
{
    unsigned long long t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_cluster(bar, parity))
            return true;
        if ((it & 15u) == 0) {
            if (*abort)
                return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                atomicExch(status, -5 /* MOE_ERR_TIMEOUT */);
                *abort = 1;
                return false;
            }
        }
    }
}

// TMA 2-D load into this CTA's shared memory whose completion (bytes) is
// signalled on an mbarrier of either CTA of the pair (shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void *dst, const void *tmap, int x, int y, uint32_t bar_cluster,
                                                 uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar_cluster), "l"(policy)
        : "memory");
}

// TMEM allocation of the CTA pair (one warp of each CTA, together).
__device__ __forceinline__ void tmem_alloc_pair(uint32_t *dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Two-SM MMA issued by the leader: A rows 0-127 / 128-255 from the two CTAs'
// shared memories, B columns split between them the same way, D rows split
// between the two TMEMs (same descriptors and TMEM address in both CTAs).
template <int QT>
__device__ __forceinline__ void mma_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate)
{
    if (QT)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
}

// Arrive once on the mbarrier at this shared offset in every CTA of `mask`
// when the pair MMAs issued so far have completed.
__device__ __forceinline__ void mma_commit_pair(uint64_t *bar, uint16_t mask)
{
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_addr(bar)),
        "h"(mask)
        : "memory");
}

// ------------------------------------------------------------- tcgen05

// Allocate ncols (power of two >= 32) TMEM columns; the base address is
// written to *dst (shared memory).  Whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 inputs, fp32 accumulate).
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Same with kind::f8f6f4 (e4m3 inputs, fp32 accumulate).
__device__ __forceinline__ void mma_fp8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive (once) on the mbarrier when every tcgen05 operation this thread
// issued before has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(bar))
                 : "memory");
}

// Shared-memory matrix descriptor for a K-major operand stored in the
// 128-byte-swizzled layout that a TMA box of 64 bf16 (128 bytes) per row
// writes: rows at 128-byte pitch, 8-row core groups 1024 bytes apart
// (stride byte offset), descriptor version 1, swizzle mode 128B.
__device__ __forceinline__ uint64_t smem_desc_sw128(const void *base)
{
    uint64_t addr = smem_addr(base);
    uint64_t d = 0;
    d |= (addr >> 4) & 0x3FFFull;           // start address (16-byte units)
    d |= (uint64_t)1 << 16;                 // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;       // stride byte offset
    d |= (uint64_t)1 << 46;                 // descriptor version
    d |= (uint64_t)2 << 61;                 // 128-byte swizzle
    return d;
}

// Shared-memory descriptor of an MN-major operand in 128-byte swizzle: 64 consecutive N (or M)
// elements of one K index per 128-byte row, 8 K rows per 1024-byte atom (stride byte offset
// between the K groups of 8), atoms of 64 N elements `lbo` bytes apart (leading byte offset) --
// the layout of 64 x 64 TMA boxes loaded from a [K][N] row-major matrix, one box per 64 N.
__device__ __forceinline__ uint64_t smem_desc_sw128_mn(const void *base, uint32_t lbo)
{
    uint64_t addr = smem_addr(base);
    uint64_t d = 0;
    d |= (addr >> 4) & 0x3FFFull;               // start address (16-byte units)
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;  // leading byte offset: next 64 elements of N
    d |= (uint64_t)(1024 >> 4) << 32;           // stride byte offset: next 8 rows of K
    d |= (uint64_t)1 << 46;                     // descriptor version
    d |= (uint64_t)2 << 61;                     // 128-byte swizzle
    return d;
}

// Instruction descriptor: dense, fp32 accumulator, both operands K-major.
// a_fmt / b_fmt: kind::f16 -> 1 = bf16; kind::f8f6f4 -> 0 = e4m3.
__host__ __device__ constexpr uint32_t make_idesc(uint32_t a_fmt, uint32_t b_fmt, uint32_t M, uint32_t N)
{
    return (1u << 4)            // D format fp32
           | (a_fmt << 7)       // A format
           | (b_fmt << 10)      // B format
           | ((N >> 3) << 17)   // N / 8
           | ((M >> 4) << 24);  // M / 16
}

// The same with B MN-major (bit 16: B is read as [K][N], N contiguous).
__host__ __device__ constexpr uint32_t make_idesc_bmn(uint32_t a_fmt, uint32_t b_fmt, uint32_t M, uint32_t N)
{
    return make_idesc(a_fmt, b_fmt, M, N) | (1u << 16);
}

// ---------------------------------------------- block-scaled FP4 (MXFP4)
//
// kind::mxf4 multiplies E2M1 operands (two per byte, K-major, 128-byte
// swizzle; one MMA covers K = 64 elements = 32 bytes) and applies one
// UE8M0 scale per 32 elements of K to each row of A and of B
// (scale_vec::2X: two scales per row per MMA).  The scales sit in TMEM in
// the 128 x 4 blocked order: for a block of 128 rows and 4 consecutive
// 32-element groups, row r's four scale bytes are 32-bit word r / 32 of TMEM
// lane r % 32, replicated in all four lane quadrants (tcgen05.cp
// .32x128b.warpx4 from 512 contiguous bytes, byte (r % 32) * 16 + (r / 32) * 4
// + g).  The scale id in the instruction descriptor selects the byte pair
// of the group pair an MMA uses (0: groups 0-1, 2: groups 2-3).

// Instruction descriptor for kind::mxf4: E2M1 A and B (format 1), K-major,
// UE8M0 scales, M x N, scale ids of A and B.
__host__ __device__ constexpr uint32_t make_idesc_mx4(uint32_t M, uint32_t N, uint32_t a_sf_id, uint32_t b_sf_id)
{
    return (b_sf_id << 4)         // B scale factor id
           | (1u << 7)            // A format: E2M1
           | (1u << 10)           // B format: E2M1
           | ((N >> 3) << 17)     // N / 8
           | (1u << 23)           // scale factor type: UE8M0
           | ((M >> 4) << 24)     // M / 16
           | (a_sf_id << 29);     // A scale factor id
}

__device__ __forceinline__ void mma_mx4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Shared-memory descriptor of 32 rows x 16 bytes stored contiguously (no
// swizzle: four 8 x 16-byte core matrices 128 bytes apart).
__device__ __forceinline__ uint64_t smem_desc_rows16(const void *p)
{
    const uint64_t addr = smem_addr(p);
    return ((addr & 0x3FFFFull) >> 4)       // start address
           | ((uint64_t)(128 >> 4) << 32)   // stride between core matrices along the rows
           | (1ull << 46);                  // descriptor version (sm_100 family); layout: no swizzle
}

// Copy 512 bytes of 128 x 4 blocked scale factors from shared memory to the 4
// TMEM columns at taddr, replicated in the four lane quadrants.
__device__ __forceinline__ void tmem_cp_sf(uint32_t taddr, uint64_t sdesc)
{
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// (acc0, acc1) = (v0, v1) * s + (acc0, acc1): the paired fp32 FMA of the
// sm_100 family (one instruction, each lane rounded once like fmaf).
__device__ __forceinline__ void ffma2(float &acc0, float &acc1, float v0, float v1, float s)
{
    asm("{\n\t.reg .b64 a, b, c, d;\n\t"
        "mov.b64 a, {%2, %3};\n\t"
        "mov.b64 b, {%4, %4};\n\t"
        "mov.b64 c, {%0, %1};\n\t"
        "fma.rn.f32x2 d, a, b, c;\n\t"
        "mov.b64 {%0, %1}, d;\n\t}"
        : "+f"(acc0), "+f"(acc1)
        : "f"(v0), "f"(v1), "f"(s));
}

// Load 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i)
        v[i] = __uint_as_float(r[i]);
}

// Issue an 8-column TMEM load without waiting for it (see tmem_wait_ld).
__device__ __forceinline__ void tmem_ld_nowait(uint32_t taddr, float (&v)[8])
{
    uint32_t *r = reinterpret_cast<uint32_t *>(v);
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld(float (&a)[8], float (&b)[8])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+f"(a[0]), "+f"(a[1]), "+f"(a[2]), "+f"(a[3]), "+f"(a[4]), "+f"(a[5]), "+f"(a[6]), "+f"(a[7]),
                   "+f"(b[0]), "+f"(b[1]), "+f"(b[2]), "+f"(b[3]), "+f"(b[4]), "+f"(b[5]), "+f"(b[6]), "+f"(b[7])
                 :
                 : "memory");
}

// Issue a 16-column TMEM load without waiting for it; tmem_wait_ld() must
// follow before the values are used.  The "+f" constraints of tmem_wait_ld
// keep the compiler from reading the registers before the wait.
__device__ __forceinline__ void tmem_ld_nowait(uint32_t taddr, float (&v)[16])
{
    uint32_t *r = reinterpret_cast<uint32_t *>(v);
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld(float (&a)[16], float (&b)[16])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+f"(a[0]), "+f"(a[1]), "+f"(a[2]), "+f"(a[3]), "+f"(a[4]), "+f"(a[5]), "+f"(a[6]), "+f"(a[7]),
                   "+f"(a[8]), "+f"(a[9]), "+f"(a[10]), "+f"(a[11]), "+f"(a[12]), "+f"(a[13]), "+f"(a[14]),
                   "+f"(a[15]), "+f"(b[0]), "+f"(b[1]), "+f"(b[2]), "+f"(b[3]), "+f"(b[4]), "+f"(b[5]),
                   "+f"(b[6]), "+f"(b[7]), "+f"(b[8]), "+f"(b[9]), "+f"(b[10]), "+f"(b[11]), "+f"(b[12]),
                   "+f"(b[13]), "+f"(b[14]), "+f"(b[15])
                 :
                 : "memory");
}

// Load 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i)
        v[i] = __uint_as_float(r[i]);
}

}  // namespace moe
