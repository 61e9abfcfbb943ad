// ptx.cuh -- hand-written inline PTX for sm_103a: mbarrier, TMA (tiled,
// gather4, store), tcgen05 (alloc, mma, commit, ld) and the fences between
// them.  Each wrapper issues exactly the named instruction; ordering and
// thread election stay with the caller, as on the TIRX tile-op pages
// ("cp.async.bulk.tensor" page, section "Stores, reductions, and completion":
// the tile call elects no thread and inserts no waits).
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace tcg {

// ---------------------------------------------------------------- basics

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- clusters
// A CTA pair (cluster of 2) shares one tcgen05 MMA: ranks differ in bit 0.

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// shared::cluster address of the same shared-memory offset in CTA `rank`
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// every thread of every CTA in the cluster
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void st_shared_cluster_u32(uint32_t cluster_addr, uint32_t v)
{
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// ---------------------------------------------------------------- dependent launch
// With programmatic dependent launch a kernel may start while the previous
// one in the stream finishes.  wait: block until the grids this one depends
// on have completed and their memory is visible (no-op without the launch
// attribute); every access to inputs or outputs comes after it.
// launch_dependents: let the next such launch begin its own set-up.

// A 32-bit global load with acquire semantics at GPU scope: writes another
// CTA made before releasing the value it reads are visible after it.
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];"
                 : "=r"(v)
                 : "l"(reinterpret_cast<uint64_t>(p))
                 : "memory");
    return v;
}

// Bring a global line into L2 ahead of its use (no register, no wait).
__device__ __forceinline__ void prefetch_l2(const void *p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)));
}

__device__ __forceinline__ void grid_dependency_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- mbarrier
// Loads complete on an mbarrier that is initialised, armed with the expected
// transaction bytes, and waited on by phase ("cp.async.bulk.tensor" page,
// section "Stores, reductions, and completion").

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// arrive on an mbarrier of another CTA of the cluster (shared::cluster address)
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}

// true once the phase with the given parity has completed
// Non-blocking probe: has phase `parity` of `bar` completed?
__device__ __forceinline__ bool mbar_probe(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking probe with acquire at cluster scope (see mbar_test_cluster).
__device__ __forceinline__ bool mbar_probe_cluster(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait with acquire at cluster scope: for a phase completed by arrivals
// from the other CTA of a pair, whose shared-memory writes must be visible.
__device__ __forceinline__ bool mbar_test_cluster(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// ---------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *m)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// One box of a 2-D descriptor at (x = inner, y = outer) into shared memory.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *m, uint32_t bar,
                                            int32_t x, int32_t y)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

// Four rows y0..y3 (any order, repeats allowed) of width box[0] starting at
// column x, into a (4, width) shared image ("cp.async.bulk.tensor" page,
// section "Gather4 and scatter4").
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap *m, uint32_t bar,
                                            int32_t x, int32_t y0, int32_t y1, int32_t y2,
                                            int32_t y3)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3)
        : "memory");
}

// Pair forms: the box lands in this CTA's shared memory, the byte count is
// reported to the mbarrier at `bar` (a shared::cluster address, here the
// leader CTA's), so one barrier tracks the loads of both CTAs of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *m, uint32_t bar,
                                                 int32_t x, int32_t y)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void tma_gather4_pair(uint32_t dst, const CUtensorMap *m, uint32_t bar,
                                                 int32_t x, int32_t y0, int32_t y1, int32_t y2,
                                                 int32_t y3)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3)
        : "memory");
}

// Pair + multicast forms: the box lands at the same offset in every CTA of
// `mask`, and each destination reports its bytes to its own pair's leader:
// `bar` is the issuing CTA's pair-leader barrier, and the destinations all
// play the same role in their pairs as the issuing CTA (same rank parity).
__device__ __forceinline__ void tma_load_2d_pair_multicast(uint32_t dst, const CUtensorMap *m,
                                                           uint32_t bar, int32_t x, int32_t y,
                                                           uint16_t mask)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".multicast::cluster [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y), "h"(mask)
        : "memory");
}

__device__ __forceinline__ void tma_gather4_pair_multicast(uint32_t dst, const CUtensorMap *m,
                                                           uint32_t bar, int32_t x, int32_t y0,
                                                           int32_t y1, int32_t y2, int32_t y3,
                                                           uint16_t mask)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile::gather4"
        ".mbarrier::complete_tx::bytes.multicast::cluster"
        " [%0], [%1, {%3, %4, %5, %6, %7}], [%2], %8;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3),
        "h"(mask)
        : "memory");
}

// Multicast forms: the same box lands at the same shared-memory offset of
// every CTA in `mask` (a cluster of CTAs on this GPU), and each destination's
// mbarrier at the offset of `bar` receives the byte count.
__device__ __forceinline__ void tma_load_2d_multicast(uint32_t dst, const CUtensorMap *m, uint32_t bar,
                                                      int32_t x, int32_t y, uint16_t mask)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y), "h"(mask)
        : "memory");
}

__device__ __forceinline__ void tma_gather4_multicast(uint32_t dst, const CUtensorMap *m, uint32_t bar,
                                                      int32_t x, int32_t y0, int32_t y1, int32_t y2,
                                                      int32_t y3, uint16_t mask)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes.multicast::cluster"
        " [%0], [%1, {%3, %4, %5, %6, %7}], [%2], %8;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3),
        "h"(mask)
        : "memory");
}

// An L2 policy that marks lines as first to evict (for data used once).
__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// tma_load_2d with an L2 cache policy
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap *m, uint32_t bar,
                                                 int32_t x, int32_t y, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y), "l"(policy)
        : "memory");
}

// tma_store_2d with an L2 cache policy
__device__ __forceinline__ void tma_store_2d_hint(const CUtensorMap *m, uint32_t src, int32_t x,
                                                  int32_t y, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group.L2::cache_hint [%0, {%2, %3}], [%1], %4;" ::"l"(
            reinterpret_cast<uint64_t>(m)),
        "r"(src), "r"(x), "r"(y), "l"(policy)
        : "memory");
}

// tma_gather4 with an L2 cache policy
__device__ __forceinline__ void tma_gather4_hint(uint32_t dst, const CUtensorMap *m, uint32_t bar,
                                                 int32_t x, int32_t y0, int32_t y1, int32_t y2,
                                                 int32_t y3, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4, %5, %6, %7}], [%2], %8;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3),
        "l"(policy)
        : "memory");
}

// Four rows of a shared image (box one row high) -> rows y0..y3 of a 2-D
// tensor, starting at column x; the dual of tile::gather4 ("cp.async.bulk.tensor"
// page, section "Gather4 and scatter4").  Completion through bulk groups.
__device__ __forceinline__ void tma_scatter4_hint(const CUtensorMap *m, uint32_t src, int32_t x,
                                                  int32_t y0, int32_t y1, int32_t y2, int32_t y3,
                                                  uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.tile::scatter4.bulk_group.L2::cache_hint"
        " [%0, {%2, %3, %4, %5, %6}], [%1], %7;" ::"l"(reinterpret_cast<uint64_t>(m)),
        "r"(src), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "l"(policy)
        : "memory");
}

// Shared image added element by element into the global box (float32 add at
// L2); the destination holds the starting value ("cp.async.bulk.tensor" page,
// section "Stores, reductions, and completion").  Completion through bulk groups.
__device__ __forceinline__ void tma_reduce_add_2d_hint(const CUtensorMap *m, uint32_t src, int32_t x,
                                                       int32_t y, uint64_t policy)
{
    asm volatile(
        "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group.L2::cache_hint"
        " [%0, {%2, %3}], [%1], %4;" ::"l"(reinterpret_cast<uint64_t>(m)),
        "r"(src), "r"(x), "r"(y), "l"(policy)
        : "memory");
}

// Shared image -> global box; completion through bulk groups.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *m, uint32_t src, int32_t x,
                                             int32_t y)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(m)),
                 "r"(src), "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit_group()
{
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// wait until at most N committed groups still read their shared source
template <int N>
__device__ __forceinline__ void bulk_wait_group_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void bulk_wait_group_all()
{
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// generic-proxy shared writes -> visible to the async proxy (TMA store)
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t dst_slot, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_slot),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// Pair forms: one warp of each CTA of the pair executes them together; the
// same columns are allocated in both CTAs' tensor memory.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_slot, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_slot),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, f16/bf16 inputs, fp32 accumulate.
// accumulate == 0 starts from zero (the first K step), otherwise adds to D.
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T: A's row r in TMEM lane r, K along the
// columns, two f16/bf16 elements per 32-bit column (the lower K index in the
// low half), so one K step of 16 spans 8 columns from a_tmem.
__device__ __forceinline__ void tc_mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                  uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Block-scaled MMA on FP4 E2M1 operands with UE8M0 scales, one scale per 32
// elements along K (the OCP Microscaling grouping that the float4_e2m1fn
// operand format of the "cp.async.bulk.tensor" page, section "Interleave and
// packed FP4", refers to).  A and B come from 128-byte swizzled shared images
// through descriptors, the scales from TMEM at sfa_tmem / sfb_tmem (layout:
// sf_tile_cols below), the byte within each 32-bit scale column chosen by the
// scale-factor ids of the instruction descriptor.
//   mxf4:     codes packed two per byte, K = 64 per instruction (32 bytes of a
//             row), two scales per row per instruction (scale_vec::2X).
//   mxf8f6f4: codes in the 16U4_ALIGN16B image (sixteen codes in the low 8
//             bytes of each 16-byte block), K = 32 per instruction (32 bytes of
//             a row), one scale per row per instruction (scale_vec::1X).
__device__ __forceinline__ void tc_mma_mxf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                            uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_mma_mxf8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Pair forms (issued by the leader CTA): M = 256, A's rows and B's halves from
// both CTAs' shared memory as in tc_mma_f16_pair; each CTA's TMEM holds the
// scales of its own 128 rows of A and of all N rows of B, at the same columns.
__device__ __forceinline__ void tc_mma_mxf4_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                 uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                 uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_mma_mxf8f6f4_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                     uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                     uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Pair form of the scale-tile copy, issued by the leader: each CTA's tile at
// the same shared-memory offset goes to the same TMEM columns of that CTA.
__device__ __forceinline__ void tc_cp_32x128b_warpx4_pair(uint32_t taddr, uint64_t src_desc)
{
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(src_desc)
                 : "memory");
}

// Shared memory -> TMEM copy of one scale tile: 32 rows of 16 bytes, written
// to the four 32-lane quarters alike (lane q*32 + l, columns col .. col+3 get
// row l).  Issued by the MMA thread; it completes in order before the MMAs
// issued after it by the same thread.
__device__ __forceinline__ void tc_cp_32x128b_warpx4(uint32_t taddr, uint64_t src_desc)
{
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(src_desc)
                 : "memory");
}

// Pair MMA, issued by the leader CTA only: M = 256 rows, A's rows 0-127 from
// the leader's shared memory and 128-255 from the peer's (same offsets), B's
// N columns split in halves the same way; each CTA's TMEM receives its rows.
__device__ __forceinline__ void tc_mma_f16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on the mbarrier at the same offset in every CTA of `mask` once the
// pair's earlier tcgen05 ops finish.
__device__ __forceinline__ void tc_commit_pair_multicast(uint32_t bar, uint16_t mask)
{
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}

// Single-CTA MMAs, arrival multicast to the mbarrier at the same offset in
// every CTA of `mask` once this thread's earlier tcgen05 ops finish.
__device__ __forceinline__ void tc_commit_multicast(uint32_t bar, uint16_t mask)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}

// Arrive (once) on an mbarrier when all earlier tcgen05 ops of this thread finish.
__device__ __forceinline__ void tc_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread t gets lane (base + t),
// register j = column (col + j).  Followed by tc_wait_ld on the same array.
__device__ __forceinline__ void tc_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// 32 lanes x 16 consecutive columns.
__device__ __forceinline__ void tc_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// Wait for this thread's tcgen05.ld results.  The registers pass through the
// asm so no use of them can be scheduled above the wait.
__device__ __forceinline__ void tc_wait_ld(uint32_t (&r)[32])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                   "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                   "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                   "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

__device__ __forceinline__ void tc_wait_ld(uint32_t (&r)[16])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
}

__device__ __forceinline__ uint32_t ld_shared_u8(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// Registers -> TMEM, the dual of tc_ld_32x32b_x32: thread t of the warp writes
// lane (taddr lane + t), columns col .. col+31.  Followed by tc_wait_st before
// the values may be read by an MMA (with a fence and barrier in between).
__device__ __forceinline__ void tc_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tc_wait_st()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- descriptors

// Shared-memory matrix descriptor for a K-major operand stored as the 128-byte
// swizzled image a TMA load with CU_TENSOR_MAP_SWIZZLE_128B writes: rows of
// 64 x 16-bit elements (128 B), 8-row groups of 1024 B, the 16-byte chunk
// index XORed with (row % 8).  The base must be 1024-byte aligned; a K step
// of 16 elements inside the 128-byte row is +32 bytes on the start address.
//   bits  0-13  start address >> 4
//   bits 16-29  leading-dimension byte offset >> 4 (unused for this layout; 1)
//   bits 32-45  stride byte offset >> 4 (1024 B between 8-row groups)
//   bits 46-47  descriptor version (1 on sm_100-family)
//   bits 49-51  base offset (0: atoms are 1024-byte aligned)
//   bits 61-63  layout: 2 = 128-byte swizzle
__device__ __forceinline__ uint64_t sdesc_k_sw128(uint32_t smem_addr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1u) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// Shared-memory descriptor of an unswizzled image made of 8-row groups of
// 16-byte rows, the groups 128 bytes apart (the source of tcgen05.cp 32x128b:
// 32 rows of 16 bytes, contiguous).  16-byte aligned base; layout 0 = none.
__device__ __forceinline__ uint64_t sdesc_rows16(uint32_t smem_addr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(128u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    return d;
}

// Instruction descriptor of the block-scaled kinds (mxf4, mxf8f6f4), dense,
// fp32 accumulator, both operands K-major, UE8M0 scales.
//   bits  4-5   B scale-factor id (byte of B's 32-bit scale column)
//   bits  7-9   A format, bits 10-12 B format (E2M1: 1 for mxf4, 5 for mxf8f6f4)
//   bits 17-22  N >> 3
//   bit  23     scale type (1 = UE8M0)
//   bits 24-28  M >> 4
//   bits 29-30  A scale-factor id
__host__ __device__ constexpr uint32_t idesc_mx(uint32_t fmt, uint32_t m, uint32_t n, uint32_t sfa_id,
                                                uint32_t sfb_id)
{
    return (sfb_id << 4) | (fmt << 7) | (fmt << 10) | ((n >> 3) << 17) | (1u << 23) |
           ((m >> 4) << 24) | (sfa_id << 29);
}

// Instruction descriptor of tcgen05.mma kind::f16, dense, fp32 accumulator,
// both operands K-major.
//   bits  4-5   D format (1 = f32)
//   bits  7-9   A format (0 = f16, 1 = bf16)
//   bits 10-12  B format (same code)
//   bit  15/16  A/B major (0 = K-major)
//   bits 17-22  N >> 3
//   bits 24-28  M >> 4
__host__ __device__ constexpr uint32_t idesc_f16_f32acc(bool bf16, uint32_t m, uint32_t n)
{
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((n >> 3) << 17) |
           ((m >> 4) << 24);
}

// ---------------------------------------------------------------- epilogue math
// One rounding each, as the fma page requires: no contraction, no ftz.

__device__ __forceinline__ float fma_rn(float a, float b, float c)
{
    float d;
    asm("fma.rn.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float mul_rn(float a, float b)
{
    float d;
    asm("mul.rn.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

// two floats -> packed 16-bit pair, lo in the low half, round to nearest even
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

__device__ __forceinline__ unsigned short f32_to_bf16_rn(float x)
{
    unsigned short d;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(d) : "f"(x));
    return d;
}

__device__ __forceinline__ unsigned short f32_to_f16_rn(float x)
{
    unsigned short d;
    asm("cvt.rn.f16.f32 %0, %1;" : "=h"(d) : "f"(x));
    return d;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ void ld_shared_v4(uint32_t addr, uint32_t &a, uint32_t &b, uint32_t &c,
                                             uint32_t &d)
{
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
                 : "r"(addr)
                 : "memory");
}

}  // namespace tcg
