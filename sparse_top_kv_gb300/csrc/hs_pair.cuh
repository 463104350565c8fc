// hs_pair.cuh -- inline-PTX wrappers for kernels that run as CTA pairs (a
// thread-block cluster of two CTAs on two SMs): cluster rank and barriers,
// distributed shared memory (mapa, remote mbarrier arrivals, st.async and
// shared-to-shared bulk copies that complete on the receiver's mbarrier),
// and the pair forms of the tcgen05 instructions (PTX ISA, "tcgen05" with
// .cta_group::2; "Distributed shared memory"; "mbarrier").
//
// What the pair forms do (checked on sm_103a with a small-integer product):
//  * tcgen05.alloc/dealloc/relinquish .cta_group::2 are issued by one warp
//    in EACH CTA of the pair and return the same column address in both.
//  * tcgen05.mma.cta_group::2 is issued by one thread of the even CTA: for
//    D[M = 256 x N] = A B^T, each CTA holds its 128 rows of A (rows 128 r ..)
//    and N/2 rows of B (the even CTA rows [0, N/2), the odd one [N/2, N)) at
//    the same shared-memory offsets, and each CTA's TMEM receives its 128
//    rows of D over all N columns.
//  * tcgen05.commit.cta_group::2 ... multicast::cluster arrives on the
//    mbarrier at the same offset in every CTA of the mask.
#pragma once

#include "hs_common.cuh"

namespace hs {
namespace pair {

__device__ __forceinline__ uint32_t cta_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

// Cluster-wide barrier (both CTAs).  Only used where both CTAs arrive
// unconditionally (after set-up and before tear-down).
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// One arrival on an mbarrier of another CTA of the cluster (release at
// cluster scope: this thread's earlier writes are visible to the waiter).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                     cluster_addr)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx_cluster(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cluster.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait with cluster-scope acquire (for barriers that the other CTA
// of the pair, its tensor-core commits or its copies complete).  Returns
// false after `timeout_ns` of wall time or once *abort is non-zero.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns,
                                          const volatile int* abort) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (abort != nullptr && *abort != 0) return false;
            if (global_timer_ns() - t0 > timeout_ns) return false;
        }
    }
}

// 16 bytes into another CTA's shared memory; `bar_cluster_addr`'s tx count
// is decremented by 16 when they have landed.
__device__ __forceinline__ void st_async_v4(uint32_t dst_cluster_addr, uint32_t a, uint32_t b,
                                            uint32_t c, uint32_t d, uint32_t bar_cluster_addr) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, "
        "[%5];" ::"r"(dst_cluster_addr),
        "r"(a), "r"(b), "r"(c), "r"(d), "r"(bar_cluster_addr)
        : "memory");
}

// Bulk copy from this CTA's shared memory into another CTA's (16-byte
// aligned, size a multiple of 16), completing on that CTA's mbarrier.
__device__ __forceinline__ void bulk_s2s(uint32_t dst_cluster_addr, uint32_t src_smem,
                                         uint32_t bytes, uint32_t bar_cluster_addr) {
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, "
        "[%3];" ::"r"(dst_cluster_addr),
        "r"(src_smem), "r"(bytes), "r"(bar_cluster_addr)
        : "memory");
}

__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// The source buffers of this thread's committed bulk copies may be reused.
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Barrier of `count` threads (a multiple of 32) on hardware barrier `id`.
__device__ __forceinline__ void named_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// As named_sync, and returns whether `pred` was true in any participant.
__device__ __forceinline__ bool named_sync_or(int id, int count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "barrier.cta.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(uint32_t(pred)), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void st_remote_u32(uint32_t cluster_addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// Loads from another CTA's shared memory (after a cluster barrier).
__device__ __forceinline__ float ld_remote_f32(uint32_t cluster_addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr) : "memory");
    return v;
}

__device__ __forceinline__ int32_t ld_remote_s32(uint32_t cluster_addr) {
    int32_t v;
    asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(cluster_addr) : "memory");
    return v;
}

__device__ __forceinline__ float4 ld_remote_v4(uint32_t cluster_addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(cluster_addr)
                 : "memory");
    return v;
}

// ---------------------------------------------------------------------------
// tcgen05, pair forms.
__device__ __forceinline__ void tmem_alloc2(uint32_t* smem_dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(smem_dst)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish2() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// D(tmem, both CTAs) (+)= A B^T over the pair, bf16 in, f32 accumulate.
__device__ __forceinline__ void mma2_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// One arrival on `bar` (same offset) in both CTAs of the pair (cluster ranks
// in `pair_mask`) once every pair MMA issued so far by this thread has
// completed.
__device__ __forceinline__ void commit2_both(uint64_t* bar, uint16_t pair_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
        "[%0], %1;" ::"r"(smem_u32(bar)),
        "h"(pair_mask)
        : "memory");
}

}  // namespace pair
}  // namespace hs
