// common.cuh -- device building blocks shared by the verify, row-statistics
// and TV-loss kernels (sm_103a).
//
// A logit row of V entries is split across the C CTAs of one thread-block
// cluster.  Each CTA bulk-copies (cp.async.bulk, completion on an mbarrier)
// its contiguous slice of the row from HBM into its own shared memory and
// keeps it there while the cluster combines per-CTA partial results through
// distributed shared memory (DSMEM).  Every logit is read from HBM once.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace mtp {

constexpr int MAX_C = 16;      // largest cluster
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;
constexpr unsigned FULL = 0xffffffffu;

// Row flag bits (mirror of the public header).
constexpr int F_NONFINITE = 1, F_BAD_ID = 2, F_BAD_TEMP = 4, F_ZERO_MASS = 8, F_BAD_UNIFORM = 16,
              F_TIMEOUT = 32;

// ------------------------------------------------------------------ PTX --

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------- debug-build checks --
//
// Built with MTP_DEBUG (build.build(debug=True) -> libmtprs_debug.so), the
// primitives below check every access they make against the launch: a shared
// 16-byte vector load, a bulk copy's shared destination (and the 16-byte
// alignment of both ends and of its size), a DSMEM address before it is
// mapped to a peer, and a TMEM column.  A failed check prints one line
// starting with "MTP_DEBUG" and the access is skipped (a load returns zeros):
// nothing traps, and the results go wrong so that the oracle comparison
// fails too.  Stores to global memory are not checked.  In the normal build
// every check compiles to nothing.
#ifdef MTP_DEBUG
}  // namespace mtp
#include <cstdio>
namespace mtp {
__device__ __forceinline__ uint32_t dbg_smem_base() {
    extern __shared__ __align__(16) unsigned char mtp_dbg_dyn_smem[];
    return smem_addr(mtp_dbg_dyn_smem);
}
__device__ __forceinline__ uint32_t dbg_smem_size() {
    uint32_t r;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(r));
    return r;
}
// True when [addr, addr + bytes) lies in this CTA's dynamic shared memory.
__device__ __forceinline__ bool dbg_smem_ok(uint32_t addr, uint32_t bytes) {
    const uint32_t base = dbg_smem_base();
    return addr >= base && addr - base + bytes <= dbg_smem_size();
}
static __device__ __noinline__ void dbg_report(const char *what, uint64_t a, uint64_t b) {
    printf("MTP_DEBUG %s block %d thread %d a=%llu b=%llu\n", what, static_cast<int>(blockIdx.x),
           static_cast<int>(threadIdx.x), static_cast<unsigned long long>(a), static_cast<unsigned long long>(b));
}
#define MTP_DBG_CHECK(cond, what, a, b, onfail) \
    do {                                        \
        if (!(cond)) {                          \
            dbg_report(what, a, b);             \
            onfail;                             \
        }                                       \
    } while (0)
#else
#define MTP_DBG_CHECK(cond, what, a, b, onfail) \
    do {                                        \
    } while (0)
#endif

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// Arrive with an expected transaction count, relaxed: orders none of the
// thread's earlier memory operations (for a producer whose data arrives by
// the bulk copies themselves).
__device__ __forceinline__ void mbar_arrive_expect_tx_relaxed(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.relaxed.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
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

// Non-blocking test of an mbarrier phase.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
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

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for an mbarrier phase with plain try_wait (the hardware suspends the
// thread inside each try_wait for a while, so polling costs few issue
// slots); the clock is read every 32 polls and the wait gives up after 2 s.
__device__ __forceinline__ bool mbar_wait_spin(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > 2000000000ull) return false;
    }
}

// try_wait with a suspend-time hint: a thread whose phase is not complete
// sleeps in the instruction (woken when the phase completes, or after about
// `ns` nanoseconds) instead of re-issuing polls that take issue slots from
// the warps that have work.
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

// Wait for an mbarrier phase, sleeping in try_wait between checks of the
// clock; gives up after limit_ns (default 2 s) and returns false.
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity, uint64_t limit_ns = 2000000000ull) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait_hint(bar, parity, 20000u)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// Wait for an mbarrier phase with a 2 s limit; false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
    return mbar_wait_spin(bar, parity);
}

// Bulk copy global -> own shared memory; completion counted on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    MTP_DBG_CHECK(dbg_smem_ok(dst, bytes) && dbg_smem_ok(bar, 8) && dst % 16 == 0 && bytes % 16 == 0 &&
                      reinterpret_cast<uintptr_t>(src) % 16 == 0 && bar % 8 == 0,
                  "bulk_g2s", dst, bytes, return);
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Order earlier generic-proxy shared-memory accesses before later bulk copies.
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

// Hardware cluster barrier (all threads of all CTAs), release/acquire.
__device__ __forceinline__ void cluster_sync() {
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n\t"
        "barrier.cluster.wait.acquire.aligned;" ::
            : "memory");
}

__device__ __forceinline__ uint32_t map_rank(uint32_t addr, uint32_t rank) {
    MTP_DBG_CHECK(dbg_smem_ok(addr, 4), "map_rank", addr, rank, (void)0);
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ int ld_cluster_s32(uint32_t addr) {
    int v;
    asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// Asynchronous 16-byte store into a peer CTA's shared memory; its bytes are
// counted on the peer's mbarrier (complete_tx).  Both addresses come from
// mapa (shared::cluster window).
__device__ __forceinline__ void st_async_v4(uint32_t raddr, float a, float b, float c, float d, uint32_t rbar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(raddr),
        "r"(__float_as_uint(a)), "r"(__float_as_uint(b)), "r"(__float_as_uint(c)), "r"(__float_as_uint(d)),
        "r"(rbar)
        : "memory");
}

// 4-byte asynchronous global -> shared copy (completion by cp_async_wait_all
// in the issuing thread).
__device__ __forceinline__ void cp_async4(void *smem_dst, const void *gsrc) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(smem_dst)), "l"(gsrc) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// 2^x on the MUFU unit (flushes subnormal results to zero).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// max that propagates NaN (any NaN operand gives NaN).
__device__ __forceinline__ float max_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// max.NaN on two packed bf16 pairs.
__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// ------------------------------------------------------- logit storage ----

struct bf16_t {
    uint16_t bits;
};

template <typename Tin>
struct Store;

template <>
struct Store<float> {
    static constexpr int ES = 4;
    static constexpr int VEC = 4;  // elements per 16-byte vector
    __device__ static __forceinline__ void unpack(const uint4 &r, float (&z)[VEC]) {
        z[0] = __uint_as_float(r.x);
        z[1] = __uint_as_float(r.y);
        z[2] = __uint_as_float(r.z);
        z[3] = __uint_as_float(r.w);
    }
    // max of the vector's elements (NaN if any element is NaN)
    __device__ static __forceinline__ float vmax(const uint4 &r) {
        return max_nan(max_nan(__uint_as_float(r.x), __uint_as_float(r.y)),
                       max_nan(__uint_as_float(r.z), __uint_as_float(r.w)));
    }
    __device__ static __forceinline__ float scalar(const unsigned char *smem, int idx) {
        return reinterpret_cast<const float *>(smem)[idx];
    }
    __device__ static __forceinline__ float scalar_g(const void *g, size_t idx) {
        return __ldg(reinterpret_cast<const float *>(g) + idx);
    }
};

template <>
struct Store<bf16_t> {
    static constexpr int ES = 2;
    static constexpr int VEC = 8;
    __device__ static __forceinline__ void unpack(const uint4 &r, float (&z)[VEC]) {
        z[0] = __uint_as_float(r.x << 16);
        z[1] = __uint_as_float(r.x & 0xffff0000u);
        z[2] = __uint_as_float(r.y << 16);
        z[3] = __uint_as_float(r.y & 0xffff0000u);
        z[4] = __uint_as_float(r.z << 16);
        z[5] = __uint_as_float(r.z & 0xffff0000u);
        z[6] = __uint_as_float(r.w << 16);
        z[7] = __uint_as_float(r.w & 0xffff0000u);
    }
    // max of the vector's elements on packed pairs (exact; NaN if any is NaN)
    __device__ static __forceinline__ float vmax(const uint4 &r) {
        const uint32_t m = bmax2_nan(bmax2_nan(r.x, r.y), bmax2_nan(r.z, r.w));
        return max_nan(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
    }
    __device__ static __forceinline__ float scalar(const unsigned char *smem, int idx) {
        return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t *>(smem)[idx]) << 16);
    }
    __device__ static __forceinline__ float scalar_g(const void *g, size_t idx) {
        const uint16_t b = __ldg(reinterpret_cast<const unsigned short *>(g) + idx);
        return __uint_as_float(static_cast<uint32_t>(b) << 16);
    }
};

// --------------------------------------------------------- row slices -----
//
// The vocabulary is split into C contiguous slices of whole 16-byte vectors:
// CTA r owns elements [lo, hi) with lo = r * nvc * VEC.  The split depends
// only on V and C, so the target and draft slices of a CTA line up element
// by element.  Element v sits at index v - lo of the CTA's shared image,
// which holds nvec = ceil((hi - lo) / VEC) vectors.  When a row starts on a
// 16-byte boundary and V is a whole number of vectors, the slice arrives by
// one bulk copy; otherwise it is loaded element by element and the last
// vector is padded with -inf (probability 0), so all compute loops run over
// whole vectors.
struct Slice {
    int lo, hi;  // element range owned by this CTA
    int nvec;    // vectors in the shared image
};

__host__ __device__ inline int slice_vectors(int V, int vec, int C) {
    const int nv = (V + vec - 1) / vec;
    return (nv + C - 1) / C;
}

// Bytes of shared memory one row slice needs (host and device agree).
__host__ __device__ inline uint32_t slice_buffer_bytes(int V, int es, int C) {
    return static_cast<uint32_t>(slice_vectors(V, 16 / es, C) * 16);
}

template <typename Tin>
__device__ __forceinline__ Slice make_slice(int V, int C, int r) {
    constexpr int VEC = Store<Tin>::VEC;
    const int nvc = slice_vectors(V, VEC, C);
    Slice s;
    s.lo = min(V, r * nvc * VEC);
    s.hi = min(V, (r + 1) * nvc * VEC);
    s.nvec = (s.hi - s.lo + VEC - 1) / VEC;
    return s;
}

// Issue the loads of one row slice into `buf`.  Fast path: thread 0 arms
// `bar` and issues one bulk copy; returns true (same value in all threads).
// Otherwise every thread copies elements and pads; the caller publishes the
// plain stores with __syncthreads().
template <typename Tin, int NTH>
__device__ __forceinline__ bool load_slice(const Slice &s, const void *row, unsigned char *buf, uint32_t bar,
                                           bool row_aligned) {
    constexpr int ES = Store<Tin>::ES, VEC = Store<Tin>::VEC;
    const unsigned char *g = reinterpret_cast<const unsigned char *>(row) + static_cast<size_t>(s.lo) * ES;
    if (s.nvec == 0) return false;
    if (row_aligned) {
        if (threadIdx.x == 0) {
            const uint32_t bytes = static_cast<uint32_t>(s.nvec) * 16u;
            mbar_arrive_expect_tx(bar, bytes);
            bulk_g2s(smem_addr(buf), g, bytes, bar);
        }
        return true;
    }
    const int n = s.hi - s.lo;
    for (int e = threadIdx.x; e < s.nvec * VEC; e += NTH) {
        if (ES == 4) {
            reinterpret_cast<float *>(buf)[e] = (e < n) ? reinterpret_cast<const float *>(g)[e] : -INFINITY;
        } else {
            reinterpret_cast<uint16_t *>(buf)[e] =
                (e < n) ? reinterpret_cast<const uint16_t *>(g)[e] : static_cast<uint16_t>(0xFF80u);
        }
    }
    return false;
}

__device__ __forceinline__ uint4 vec_at(const unsigned char *buf, int j) {
    MTP_DBG_CHECK(!__isShared(buf + 16 * static_cast<ptrdiff_t>(j)) ||
                      (dbg_smem_ok(smem_addr(buf + 16 * static_cast<ptrdiff_t>(j)), 16) &&
                       smem_addr(buf + 16 * static_cast<ptrdiff_t>(j)) % 16 == 0),
                  "vec_at", smem_addr(buf), static_cast<uint32_t>(j), return make_uint4(0u, 0u, 0u, 0u));
    return reinterpret_cast<const uint4 *>(buf)[j];
}

// ------------------------------------------------ online softmax partials --
//
// For one row and one scale k = log2(e)/T: m = max z, s = sum 2^{(z-m)k},
// s1 = sum 2^{(z-m)k} (z-m)k (only when entropy is wanted).  Partials merge
// by rescaling to the larger max.
struct Soft {
    float m, s, s1;
};

__device__ __forceinline__ Soft soft_empty() { return {-INFINITY, 0.f, 0.f}; }

// ---------------------------------------------- packed float pairs (f32x2) --

__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void f2unpack(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ uint64_t f2fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint64_t f2add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// The two elements of a 32-bit word of the image as floats: bf16 pair
// (exact widening) or, for float32 storage, the word itself (lo) and the next.
__device__ __forceinline__ uint64_t bf16pair_f2(uint32_t x) {
    return f2pack(__uint_as_float(x << 16), __uint_as_float(x & 0xffff0000u));
}

// Exact path: softmax partial of this thread's vectors j = tid, tid + NT, ...
// < nvec of one row slice, in two passes over shared memory: (1) the exact
// maximum m (NaN-propagating; a NaN or +inf sets `bad`), (2)
// s = sum 2^{(z - m) k} and, with ENT, s1 = sum 2^{(z - m) k} (z - m) k.
template <typename Tin, bool ENT, int NT>
__device__ __forceinline__ Soft thread_soft_exact(const unsigned char *buf, int nvec, float k, bool &bad) {
    Soft a = soft_empty();
    float m;
    if (Store<Tin>::ES == 2) {
        uint32_t m2 = 0xff80ff80u;  // (-inf, -inf)
        for (int j = threadIdx.x; j < nvec; j += NT) {
            const uint4 r = vec_at(buf, j);
            m2 = bmax2_nan(m2, bmax2_nan(bmax2_nan(r.x, r.y), bmax2_nan(r.z, r.w)));
        }
        m = max_nan(__uint_as_float(m2 << 16), __uint_as_float(m2 & 0xffff0000u));
    } else {
        m = -INFINITY;
        for (int j = threadIdx.x; j < nvec; j += NT) {
            const uint4 r = vec_at(buf, j);
            m = max_nan(m, max_nan(max_nan(__uint_as_float(r.x), __uint_as_float(r.y)),
                                   max_nan(__uint_as_float(r.z), __uint_as_float(r.w))));
        }
    }
    if (!(m < INFINITY)) {  // NaN or +inf in the slice
        bad = true;
        return a;
    }
    if (m == -INFINITY) return a;  // nothing but -inf (or no elements)
    a.m = m;
    const float mk = m * k;
    const uint64_t K2 = f2pack(k, k), NMK2 = f2pack(-mk, -mk);
    uint64_t acc = f2pack(0.f, 0.f), acc1 = f2pack(0.f, 0.f);
    for (int j = threadIdx.x; j < nvec; j += NT) {
        const uint4 r = vec_at(buf, j);
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
        if (Store<Tin>::ES == 2) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint64_t d2 = f2fma(bf16pair_f2(w[q]), K2, NMK2);
                float d0, d1;
                f2unpack(d2, d0, d1);
                if (ENT) {
                    d0 = fmaxf(d0, -256.f);
                    d1 = fmaxf(d1, -256.f);
                }
                const float e0 = ex2(d0), e1 = ex2(d1);
                const uint64_t e2 = f2pack(e0, e1);
                acc = f2add(acc, e2);
                if (ENT) acc1 = f2fma(e2, f2pack(d0, d1), acc1);
            }
        } else {
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const uint64_t z2 = f2pack(__uint_as_float(w[2 * q]), __uint_as_float(w[2 * q + 1]));
                const uint64_t d2 = f2fma(z2, K2, NMK2);
                float d0, d1;
                f2unpack(d2, d0, d1);
                if (ENT) {
                    d0 = fmaxf(d0, -256.f);
                    d1 = fmaxf(d1, -256.f);
                }
                const float e0 = ex2(d0), e1 = ex2(d1);
                const uint64_t e2 = f2pack(e0, e1);
                acc = f2add(acc, e2);
                if (ENT) acc1 = f2fma(e2, f2pack(d0, d1), acc1);
            }
        }
    }
    float s0, s1v, t0, t1;
    f2unpack(acc, s0, s1v);
    a.s = s0 + s1v;
    if (ENT) {
        f2unpack(acc1, t0, t1);
        a.s1 = t0 + t1;
    }
    return a;
}

// Sum of 2^{z k - mk} over the VEC elements of one vector into two
// accumulators (and, with ENT, of 2^{d} d with d = z k - mk, clamped).
template <typename Tin, bool ENT>
__device__ __forceinline__ void vec_expsum(const uint4 &r, float k, float mk, float &s0, float &s1, float &t0,
                                           float &t1) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        float z0, z1;
        if (Store<Tin>::ES == 2) {
            z0 = __uint_as_float(w[q] << 16);
            z1 = __uint_as_float(w[q] & 0xffff0000u);
        } else {
            if (q & 1) continue;
            z0 = __uint_as_float(w[q]);
            z1 = __uint_as_float(w[q + 1]);
        }
        float d0 = fmaf(z0, k, -mk), d1 = fmaf(z1, k, -mk);
        if (ENT) {
            d0 = fmaxf(d0, -256.f);
            d1 = fmaxf(d1, -256.f);
        }
        const float e0 = ex2(d0), e1 = ex2(d1);
        s0 += e0;
        s1 += e1;
        if (ENT) {
            t0 = fmaf(e0, d0, t0);
            t1 = fmaf(e1, d1, t1);
        }
    }
}

// Sum of 2^{z k - mk} over one vector on the packed f32x2 pipe, into two
// pair accumulators (K2 = (k, k), NMK2 = (-mk, -mk)).
template <typename Tin>
__device__ __forceinline__ void vec_expsum2(const uint4 &r, uint64_t K2, uint64_t NMK2, uint64_t &acc0,
                                            uint64_t &acc1) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
    float d0, d1;
    if (Store<Tin>::ES == 2) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            f2unpack(f2fma(bf16pair_f2(w[q]), K2, NMK2), d0, d1);
            if (q & 1) acc1 = f2add(acc1, f2pack(ex2(d0), ex2(d1)));
            else acc0 = f2add(acc0, f2pack(ex2(d0), ex2(d1)));
        }
    } else {
        f2unpack(f2fma(f2pack(__uint_as_float(w[0]), __uint_as_float(w[1])), K2, NMK2), d0, d1);
        acc0 = f2add(acc0, f2pack(ex2(d0), ex2(d1)));
        f2unpack(f2fma(f2pack(__uint_as_float(w[2]), __uint_as_float(w[3])), K2, NMK2), d0, d1);
        acc1 = f2add(acc1, f2pack(ex2(d0), ex2(d1)));
    }
}

template <typename Tin, bool ENT, int NT>
__device__ __noinline__ Soft thread_soft_exact_call(const unsigned char *buf, int nvec, float k, bool &bad) {
    return thread_soft_exact<Tin, ENT, NT>(buf, nvec, k, bad);
}

// Softmax partial of this thread's vectors of one row slice (see
// thread_soft_exact for the definition).  With ENT (entropy) the exact path
// always runs: with a reference below the maximum, ln Z and the entropy sum
// would both be large and cancel.  Otherwise, fast path: one pass with the
// reference m = max of the thread's first vector instead of the exact
// maximum; any reference gives the same normaliser after the rescaled merge,
// and the pass is kept only if its sum stays finite and below 2^64 (no
// overflow; NaN or +inf make it non-finite).  Otherwise the exact two-pass
// path runs, which also flags NaN / +inf.
template <typename Tin, bool ENT, int NT>
__device__ __forceinline__ Soft thread_soft(const unsigned char *buf, int nvec, float k, bool &bad) {
    if (ENT) return thread_soft_exact<Tin, ENT, NT>(buf, nvec, k, bad);
    const int j0 = threadIdx.x;
    if (j0 >= nvec) return soft_empty();
    const uint4 first = vec_at(buf, j0);
    float mref;
    if (Store<Tin>::ES == 2) {
        uint32_t m2;
        asm("max.bf16x2 %0, %1, %2;" : "=r"(m2) : "r"(first.x), "r"(first.y));
        uint32_t m3;
        asm("max.bf16x2 %0, %1, %2;" : "=r"(m3) : "r"(first.z), "r"(first.w));
        asm("max.bf16x2 %0, %1, %2;" : "=r"(m2) : "r"(m2), "r"(m3));
        mref = fmaxf(__uint_as_float(m2 << 16), __uint_as_float(m2 & 0xffff0000u));
    } else {
        mref = fmaxf(fmaxf(__uint_as_float(first.x), __uint_as_float(first.y)),
                     fmaxf(__uint_as_float(first.z), __uint_as_float(first.w)));
    }
    if (mref > -INFINITY && mref < INFINITY) {
        const float mk = mref * k;
        const uint64_t K2 = f2pack(k, k), NMK2 = f2pack(-mk, -mk);
        uint64_t acc0 = f2pack(0.f, 0.f), acc1 = f2pack(0.f, 0.f);
        int j = j0;
        for (; j + 3 * NT < nvec; j += 4 * NT) {
            const uint4 r0 = vec_at(buf, j), r1 = vec_at(buf, j + NT), r2 = vec_at(buf, j + 2 * NT),
                        r3 = vec_at(buf, j + 3 * NT);
            vec_expsum2<Tin>(r0, K2, NMK2, acc0, acc1);
            vec_expsum2<Tin>(r1, K2, NMK2, acc0, acc1);
            vec_expsum2<Tin>(r2, K2, NMK2, acc0, acc1);
            vec_expsum2<Tin>(r3, K2, NMK2, acc0, acc1);
        }
        for (; j < nvec; j += NT) vec_expsum2<Tin>(vec_at(buf, j), K2, NMK2, acc0, acc1);
        float a0, a1, b0, b1;
        f2unpack(acc0, a0, a1);
        f2unpack(acc1, b0, b1);
        const float s = (a0 + a1) + (b0 + b1);
        if (s < 1.8e19f) {  // finite, no NaN, far from overflow after merging
            Soft a;
            a.m = mref;
            a.s = s;
            a.s1 = 0.f;
            return a;
        }
    }
    return thread_soft_exact_call<Tin, ENT, NT>(buf, nvec, k, bad);
}

// Add one vector of logits z (its max vm, NaN if any element is NaN).
template <int N, bool ENT>
__device__ __forceinline__ void soft_add(Soft &a, const float (&z)[N], float vm, float k, bool &bad) {
    if (!(vm < INFINITY)) {  // NaN or +inf
        bad = true;
        return;
    }
    if (vm > a.m) {
        const float dl = (vm - a.m) * k;
        const float sc = ex2(-dl);
        if (ENT) a.s1 = (a.s != 0.f) ? sc * (a.s1 - dl * a.s) : 0.f;
        a.s *= sc;
        a.m = vm;
    }
    if (a.m == -INFINITY) return;
    const float mk = a.m * k;
#pragma unroll
    for (int j = 0; j < N; ++j) {
        if (ENT) {
            const float d = fmaxf(fmaf(z[j], k, -mk), -256.f);
            const float e = ex2(d);
            a.s += e;
            a.s1 = fmaf(e, d, a.s1);
        } else {
            a.s += ex2(fmaf(z[j], k, -mk));
        }
    }
}

// Lane `lane` of warp 0 merges the per-thread partials lane, lane+32, ...
// (NT/32 of them) stored as m[], s[], s1[] columns in shared memory.
template <bool ENT, int NW>
__device__ __forceinline__ Soft soft_lane_merge(const float *m, const float *s, const float *s1, int lane, float k) {
    float M = m[lane];
#pragma unroll
    for (int q = 1; q < NW; ++q) M = fmaxf(M, m[lane + 32 * q]);
    Soft r;
    r.m = M;
    r.s = 0.f;
    r.s1 = 0.f;
    if (M == -INFINITY) return r;
#pragma unroll
    for (int q = 0; q < NW; ++q) {
        const float sq = s[lane + 32 * q];
        if (sq != 0.f) {
            const float dl = (M - m[lane + 32 * q]) * k;
            const float sc = ex2(-dl);
            r.s += sq * sc;
            if (ENT) r.s1 += sc * (s1[lane + 32 * q] - dl * sq);
        }
    }
    return r;
}

// Symmetric butterfly sum (every lane ends with the same bits).
__device__ __forceinline__ float warp_allsum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
    return v;
}

__device__ __forceinline__ float warp_allmax(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, o));
    return v;
}

// Warp reduction of softmax partials: exact max over the lanes, one rescale
// per lane, then butterfly sums.  Every lane ends with the same bits.
template <bool ENT>
__device__ __forceinline__ Soft soft_warp_allreduce(const Soft &a, float k) {
    Soft r;
    r.m = warp_allmax(a.m);
    float s = 0.f, s1 = 0.f;
    if (r.m != -INFINITY && a.s != 0.f) {
        const float dl = (r.m - a.m) * k;
        const float sc = ex2(-dl);
        s = a.s * sc;
        if (ENT) s1 = sc * (a.s1 - dl * a.s);
    }
    r.s = warp_allsum(s);
    r.s1 = ENT ? warp_allsum(s1) : 0.f;
    return r;
}

__device__ __forceinline__ int warp_allor(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v |= __shfl_xor_sync(FULL, v, o);
    return v;
}

// ------------------------------------------------------ cluster exchange --
//
// All-gather of one record (XW words) per CTA.  Warp 0 of every CTA pushes
// its record into slot `round % XR` of every peer with st.async; each CTA
// arms its own mbarrier for C records and waits (bounded).  A round is sent
// only after the previous round of the same CTA completed and every warp
// passed a __syncthreads, so a slot is never overwritten while it is read.
constexpr int XR = 2;   // ring of exchange slots (one round outstanding at a time)
constexpr int XW = 8;   // words per record

struct Xchg {
    float rec[XR][MAX_C][XW];
    unsigned long long bar[XR];
};

__device__ __forceinline__ void xchg_init(Xchg &x) {
    for (int s = 0; s < XR; ++s) mbar_init(smem_addr(&x.bar[s]), 1);
}

// Every thread calls; warp 0 holds the record `v` (same value in all its
// lanes).  Returns the slot to read (records 0..C-1); `ok` is false when the
// wait gave up.
template <int W>
__device__ __forceinline__ int xchg_round(Xchg &x, int &round, const float (&v)[W], int C, int rank, bool &ok) {
    static_assert(W % 4 == 0 && W <= XW, "record width");
    const int slot = round % XR;
    const uint32_t par = static_cast<uint32_t>(round / XR) & 1u;
    const uint32_t bar = smem_addr(&x.bar[slot]);
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        if (lane < C) {
            const uint32_t raddr = map_rank(smem_addr(&x.rec[slot][rank][0]), lane);
            const uint32_t rbar = map_rank(bar, lane);
#pragma unroll
            for (int q = 0; q < W / 4; ++q) st_async_v4(raddr + 16 * q, v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3], rbar);
        }
        if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(C * W * 4));
    }
    ok = __syncthreads_and(mbar_wait_bounded(bar, par) ? 1 : 0) != 0;  // same verdict in every thread
    ++round;
    return slot;
}

// Inclusive prefix sum across the warp (Hillis-Steele).
__device__ __forceinline__ float warp_incl_scan(float v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float n = __shfl_up_sync(FULL, v, o);
        if (lane >= o) v += n;
    }
    return v;
}

}  // namespace mtp
