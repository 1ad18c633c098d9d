// Inline-PTX wrappers for the sm_103a GEMM path: mbarriers, TMA (cp.async.bulk.tensor),
// tcgen05 (TMEM alloc / MMA / commit / ld / fences), cluster helpers and named barriers.
//
// The data path these serve is the one the GEMM pages lay out for Blackwell (page
// "TIRx 与高性能GEMM (上)", section "从 GEMM 公式到数据路径"): operand tiles go from global
// memory into shared memory, tcgen05.mma reads them from shared memory and accumulates into
// Tensor Memory, and the epilogue reads TMEM into registers, converts and writes back.
// Every wait here is bounded (see mbar_wait): a wait that runs out reports failure to the
// caller instead of spinning forever.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace gf16 {

// ------------------------------------------------------------------------------------------
// Addresses and special registers
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_id_x()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t num_clusters_x()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// Address of the same shared-memory offset in CTA `rank` of this cluster (shared::cluster window).
__device__ __forceinline__ uint32_t mapa_shared(uint32_t smem_addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The two halves of cluster_sync(), so that work that needs no other thread's writes can run
// between them.
__device__ __forceinline__ void cluster_arrive()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Programmatic dependent launch.  grid_dep_launch() lets the next kernel on the stream, if it
// was launched with programmatic stream serialization, start once every CTA of this grid has
// called it or exited.  grid_dep_wait() returns once the kernel before this one on the stream
// has completed and its memory writes are visible; it returns at once when this launch had no
// programmatic dependency.
__device__ __forceinline__ void grid_dep_launch()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void grid_dep_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// True in exactly one lane of the (converged) warp: the lowest active lane.
__device__ __forceinline__ bool elect_one_sync()
{
    uint32_t pred = 0;
    asm volatile("{\n\t.reg .pred P;\n\t"
                 "elect.sync _|P, 0xffffffff;\n\t"
                 "selp.u32 %0, 1, 0, P;\n\t}"
                 : "=r"(pred));
    return pred != 0;
}

// Named barrier over `nthreads` threads (a multiple of 32); id 0 is __syncthreads' barrier.
__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also ANDs a predicate over the participating threads: every thread gets
// the same answer, so a decision taken from it is uniform across the group.
__device__ __forceinline__ uint32_t named_barrier_and(uint32_t id, uint32_t nthreads,
                                                      uint32_t pred)
{
    uint32_t out;
    asm volatile("{\n\t.reg .pred p, q;\n\t"
                 "setp.ne.u32 p, %3, 0;\n\t"
                 "bar.red.and.pred q, %1, %2, p;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(out)
                 : "r"(id), "r"(nthreads), "r"(pred)
                 : "memory");
    return out;
}

// ------------------------------------------------------------------------------------------
// mbarrier
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later async-proxy
// (TMA / tensor core) accesses.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// One arrival plus `bytes` of expected transaction (TMA) traffic on the current phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_local(uint32_t bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Arrival on a barrier named by a shared::cluster address (possibly another CTA's), with the
// default CTA-scope release.  The epilogue's "accumulator drained" signal needs no cluster-scope
// ordering of memory: its tensor-memory reads are complete (tcgen05.wait::ld) and fenced with
// tcgen05.fence::before_thread_sync, and the waiting MMA issuer fences after the wait.  Measured
// on GB300 (per-tile timeline probe of the CTA-pair kernel), a .release.cluster arrival on the
// peer's barrier took about 550 ns longer to reach the waiter than this form.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar_cluster)
{
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

// True once the phase of parity `parity` has completed.  A fresh barrier is in phase 0, and
// the phase "before" it (parity 1) counts as completed, so waiting on parity 1 of a fresh
// barrier returns at once (the convention the producer's first pass over the ring uses).
template <bool kClusterScope>
__device__ __forceinline__ uint32_t mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    if constexpr (kClusterScope) {
        asm volatile("{\n\t.reg .pred P;\n\t"
                     "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 P, [%1], %2;\n\t"
                     "selp.u32 %0, 1, 0, P;\n\t}"
                     : "=r"(ok)
                     : "r"(bar), "r"(parity)
                     : "memory");
    } else {
        asm volatile("{\n\t.reg .pred P;\n\t"
                     "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
                     "selp.u32 %0, 1, 0, P;\n\t}"
                     : "=r"(ok)
                     : "r"(bar), "r"(parity)
                     : "memory");
    }
    return ok;
}

// Upper bound on polls of one wait, a backstop behind the wall-clock limit.
constexpr uint32_t kMaxPolls = 1u << 28;

// A flag in global memory that another CTA of the grid raises: a GPU-scope release store by
// the raiser, an acquire load by the waiter.
__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Bounded wait until *p is non-zero (false: the wall-clock limit ran out, or another role of
// this CTA raised `abort_flag`).
static __device__ __noinline__ bool wait_flag(const uint32_t* p, const volatile uint32_t* abort_flag,
                                              uint64_t timeout_ns)
{
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 0; i < kMaxPolls; ++i) {
        if (ld_acquire_gpu(p) != 0u) return true;
        if ((i & 15u) == 15u) {
            if (abort_flag != nullptr && *abort_flag) return false;
            if (globaltimer_ns() - t0 > timeout_ns) return false;
        }
        __nanosleep(64);
    }
    return false;
}

template <bool kClusterScope>
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity,
                                            const volatile uint32_t* abort_flag,
                                            uint64_t timeout_ns)
{
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 0; i < kMaxPolls; ++i) {
        if (mbar_try_wait<kClusterScope>(bar, parity)) return true;
        if ((i & 63u) == 63u) {
            if (abort_flag != nullptr && *abort_flag) return false;
            if (globaltimer_ns() - t0 > timeout_ns) return false;
        }
    }
    return false;
}

// Bounded wait: returns false if the phase did not complete within `timeout_ns`, or if another
// role of this CTA raised `abort_flag` (pass nullptr to ignore it, as the drains after an abort
// do).  The fast path is one try_wait.
template <bool kClusterScope = false>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          const volatile uint32_t* abort_flag, uint64_t timeout_ns)
{
    if (mbar_try_wait<kClusterScope>(bar, parity)) return true;
    return mbar_wait_slow<kClusterScope>(bar, parity, abort_flag, timeout_ns);
}

// ------------------------------------------------------------------------------------------
// TMA
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled load into this CTA's shared memory; completion is counted in bytes on `bar`
// (a barrier of this CTA).  x is the inner (contiguous) coordinate, in elements.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t x, int32_t y)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
                 : "memory");
}

// L2 eviction-priority policy for TMA loads (createpolicy, fraction 1.0).
// priority: 0 = evict_normal, 1 = evict_first, 2 = evict_last.
__device__ __forceinline__ uint64_t make_l2_policy(uint32_t priority)
{
    uint64_t pol;
    if (priority == 1)
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    else if (priority == 2)
        asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    else
        asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 2-D tiled load with an L2 eviction-priority hint.
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                                 int32_t x, int32_t y, uint64_t policy)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "l"(policy)
                 : "memory");
}

// CTA-pair form of tma_load_2d_hint (see tma_load_2d_pair).
__device__ __forceinline__ void tma_load_2d_pair_hint(uint32_t dst, const CUtensorMap* map,
                                                      uint32_t bar_cluster, int32_t x, int32_t y,
                                                      uint64_t policy)
{
    asm volatile("cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile"
                 ".mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(
                     dst),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y),
                 "l"(policy)
                 : "memory");
}

// Same, for a CTA pair: the destination is this CTA's shared memory, and the completion
// barrier may be the peer CTA's (a shared::cluster address from mapa_shared).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int32_t x, int32_t y)
{
    asm volatile("cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile"
                 ".mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
                 : "memory");
}

// 3-D tiled load into this CTA's shared memory (the block-scale chunks); x is the inner
// coordinate in elements.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t x, int32_t y, int32_t z)
{
    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
                 : "memory");
}

// CTA-pair form of tma_load_3d: completes on a barrier that may be the peer CTA's.
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int32_t x, int32_t y,
                                                 int32_t z)
{
    asm volatile("cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile"
                 ".mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y), "r"(z)
                 : "memory");
}

// 2-D tiled store from this CTA's shared memory; elements outside the tensor are not written.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t x,
                                             int32_t y)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(src), "r"(x), "r"(y)
                 : "memory");
}

// The same with an L2 eviction-priority policy (make_l2_policy) for the written lines.
__device__ __forceinline__ void tma_store_2d_hint(const CUtensorMap* map, uint32_t src, int32_t x,
                                                  int32_t y, uint64_t policy)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group.L2::cache_hint "
                 "[%0, {%2, %3}], [%1], %4;"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(src), "r"(x), "r"(y), "l"(policy)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit_group()
{
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N committed bulk groups still read their shared-memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until all committed bulk groups have fully completed (writes included).
__device__ __forceinline__ void bulk_wait_group_all()
{
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ------------------------------------------------------------------------------------------
// tcgen05: Tensor Memory and the fifth-generation tensor core
// ------------------------------------------------------------------------------------------
template <int kCtaGroup>
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols)
{
    if constexpr (kCtaGroup == 1)
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         slot_smem),
                     "r"(ncols)
                     : "memory");
    else
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         slot_smem),
                     "r"(ncols)
                     : "memory");
}

template <int kCtaGroup>
__device__ __forceinline__ void tmem_relinquish()
{
    if constexpr (kCtaGroup == 1)
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    else
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

template <int kCtaGroup>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    if constexpr (kCtaGroup == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
                     "r"(ncols)
                     : "memory");
    else
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr),
                     "r"(ncols)
                     : "memory");
}

__device__ __forceinline__ void tcgen05_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tcgen05_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, fp16 inputs, fp32 accumulator, shape from idesc.
// accumulate == 0 overwrites the accumulator (the first K step of a tile).
template <int kCtaGroup>
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate)
{
    if constexpr (kCtaGroup == 1)
        asm volatile("{\n\t.reg .pred p;\n\t"
                     "setp.ne.b32 p, %4, 0;\n\t"
                     "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                     "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
                     : "memory");
    else
        asm volatile("{\n\t.reg .pred p;\n\t"
                     "setp.ne.b32 p, %4, 0;\n\t"
                     "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                     "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
                     : "memory");
}

// Block-scaled FP8 MMA (kind::mxf8f6f4, one E8M0 scale per 32 K elements):
// D[tmem] (+)= (A * sA) * (B * sB)^T.  sfa_tmem / sfb_tmem are the tensor-memory addresses of the
// scale-factor columns; the idesc's scale-factor IDs pick the byte of each 32-bit column that
// holds this MMA's K block.
template <int kCtaGroup>
__device__ __forceinline__ void mma_mx(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                       uint32_t accumulate)
{
    if constexpr (kCtaGroup == 1)
        asm volatile("{\n\t.reg .pred p;\n\t"
                     "setp.ne.b32 p, %4, 0;\n\t"
                     "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X "
                     "[%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d_tmem),
                     "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem),
                     "r"(sfb_tmem)
                     : "memory");
    else
        asm volatile("{\n\t.reg .pred p;\n\t"
                     "setp.ne.b32 p, %4, 0;\n\t"
                     "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X "
                     "[%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d_tmem),
                     "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem),
                     "r"(sfb_tmem)
                     : "memory");
}

// Copy 32 rows x 128 bits from shared memory (described by `sdesc`) into tensor memory at
// `taddr`, replicated into all four 32-lane windows (lanes r, 32 + r, 64 + r, 96 + r get row r):
// the scale-factor layout of the page "TIRx Layout API", section "Scale Factor 布局".  Runs in
// issue order with the MMAs of the same thread.
template <int kCtaGroup>
__device__ __forceinline__ void tmem_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc)
{
    if constexpr (kCtaGroup == 1)
        asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
                     : "memory");
    else
        asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
                     : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
}

// CTA-pair form: arrive on the barrier at the same shared-memory offset in every CTA of
// `cta_mask` (a completion signal, not a data copy).
__device__ __forceinline__ void mma_commit_pair(uint32_t bar, uint16_t cta_mask)
{
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::"
                 "cluster.b64 [%0], %1;" ::"r"(bar),
                 "h"(cta_mask)
                 : "memory");
}

// Each thread of the warp reads 32 consecutive 32-bit columns of its own TMEM lane.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32], int base)
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
                 "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
                 "[%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
                   "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
                   "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
                   "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr + static_cast<uint32_t>(base)));
}

__device__ __forceinline__ void tmem_ld_wait()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------------------------------------
// Conversion and shared-memory stores
// ------------------------------------------------------------------------------------------
// Two fp32 values -> one f16x2 word, each rounded to nearest even; `lo` lands in bits 15:0.
__device__ __forceinline__ uint32_t pack_f16x2_rn(uint32_t lo_bits, uint32_t hi_bits)
{
    uint32_t out;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;"
        : "=r"(out)
        : "f"(__uint_as_float(hi_bits)), "f"(__uint_as_float(lo_bits)));
    return out;
}

// Two fp32 values -> one bf16x2 word, each rounded to nearest even; `lo` lands in bits 15:0.
__device__ __forceinline__ uint32_t pack_bf16x2_rn(uint32_t lo_bits, uint32_t hi_bits)
{
    uint32_t out;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;"
        : "=r"(out)
        : "f"(__uint_as_float(hi_bits)), "f"(__uint_as_float(lo_bits)));
    return out;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ void st_global_v4(void* ptr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d)
{
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(ptr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

}  // namespace gf16
