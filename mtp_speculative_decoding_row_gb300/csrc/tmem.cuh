// tmem.cuh -- tensor memory (TMEM) as on-chip storage for logit row
// segments on sm_103a (tcgen05.alloc / st / ld / dealloc, cta_group::1).
//
// Every SM has 512 TMEM columns of 128 lanes x 32 bits (256 KB).  A CTA
// allocates a power-of-two number of columns; warp w may touch only lanes
// 32 (w % 4) .. 32 (w % 4) + 31, each thread its own lane.  The kernels here
// use TMEM as a parking place: a 16-byte vector of logits a lane has loaded
// from shared memory is stored into four consecutive columns of its lane and
// read back later for a second (and third) pass, so the row never has to be
// read from HBM or L2 again.  No tensor-core instruction is involved.
//
// Allocation blocks while the SM lacks free columns.  A kernel that uses
// these helpers allocates all TMEM_COLS columns in one CTA and its launch
// asks for more than half of the SM's shared memory, so only one of its CTAs
// is ever resident on an SM and an allocation always finds its columns (a
// CTA of another kernel that holds columns ends by itself and frees them).
#pragma once

#include <stdint.h>

#include "common.cuh"

namespace mtp {

constexpr uint32_t TMEM_COLS = 512;

// Warp-wide: allocate `ncols` columns; the TMEM address lands in *slot
// (shared memory).  Then give up the right to allocate again, so that other
// CTAs waiting for columns are not held back.
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(slot))),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

// Warp-wide: free the columns allocated at `taddr`.
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Order TMEM accesses around a thread synchronisation (__syncthreads or a
// cluster barrier): before_sync on the issuing side, after_sync on the other.
__device__ __forceinline__ void tmem_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Address of lane base `lane0` (a multiple of 32), column `col`.
__device__ __forceinline__ uint32_t tmem_addr(uint32_t base, uint32_t lane0, uint32_t col) {
    return base + (lane0 << 16) + col;
}

// Warp-wide: each thread stores one 16-byte vector into columns col .. col+3
// of its own lane.
__device__ __forceinline__ void tmem_st_v4(uint32_t taddr, const uint4 &v) {
    MTP_DBG_CHECK((taddr & 0xffffu) + 4u <= TMEM_COLS && (taddr >> 16) < 128u, "tmem_st", taddr, 0, (void)0);
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// Warp-wide: each thread loads one 16-byte vector from columns col .. col+3
// of its own lane.  The registers are valid after tmem_wait_ld().
__device__ __forceinline__ void tmem_ld_v4(uint32_t taddr, uint4 &v) {
    MTP_DBG_CHECK((taddr & 0xffffu) + 4u <= TMEM_COLS && (taddr >> 16) < 128u, "tmem_ld", taddr, 0, (void)0);
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(taddr)
                 : "memory");
}

// Block until this thread's earlier tcgen05.st (tcgen05.ld) have completed.
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Wait for this thread's TMEM loads and make the compiler see every loaded
// register as produced after the wait: the loads write their registers
// asynchronously, so no use may be scheduled between tcgen05.ld and
// tcgen05.wait::ld.
template <int N>
__device__ __forceinline__ void tmem_wait_ld_regs(uint4 (&v)[N]) {
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < N; ++i) asm volatile("" : "+r"(v[i].x), "+r"(v[i].y), "+r"(v[i].z), "+r"(v[i].w));
}

}  // namespace mtp
