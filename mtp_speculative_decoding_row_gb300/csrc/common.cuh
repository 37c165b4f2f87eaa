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

constexpr int NT = 512;        // threads per CTA
constexpr int NW = NT / 32;    // warps per CTA
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

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
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

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for an mbarrier phase with a 2 s limit; false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > 2000000000ull) return false;
    }
    return true;
}

// Bulk copy global -> own shared memory; completion counted on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
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
template <typename Tin>
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
    for (int e = threadIdx.x; e < s.nvec * VEC; e += NT) {
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

template <int N, bool ENT>
__device__ __forceinline__ void soft_add(Soft &a, const float (&z)[N], float k, bool &bad) {
    float vm = z[0];
#pragma unroll
    for (int j = 1; j < N; ++j) vm = max_nan(vm, z[j]);
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

// Symmetric merge: merge(a, b) and merge(b, a) are bitwise equal.
template <bool ENT>
__device__ __forceinline__ Soft soft_merge(const Soft &a, const Soft &b, float k) {
    Soft r;
    r.m = fmaxf(a.m, b.m);
    if (r.m == -INFINITY) return soft_empty();
    float sa = 0.f, sb = 0.f, ta = 0.f, tb = 0.f;
    if (a.s != 0.f) {
        const float dl = (r.m - a.m) * k;
        const float sc = ex2(-dl);
        sa = a.s * sc;
        if (ENT) ta = sc * (a.s1 - dl * a.s);
    }
    if (b.s != 0.f) {
        const float dl = (r.m - b.m) * k;
        const float sc = ex2(-dl);
        sb = b.s * sc;
        if (ENT) tb = sc * (b.s1 - dl * b.s);
    }
    r.s = sa + sb;
    r.s1 = ENT ? (ta + tb) : 0.f;
    return r;
}

template <bool ENT>
__device__ __forceinline__ Soft soft_shfl_xor(const Soft &a, int mask) {
    Soft o;
    o.m = __shfl_xor_sync(FULL, a.m, mask);
    o.s = __shfl_xor_sync(FULL, a.s, mask);
    o.s1 = ENT ? __shfl_xor_sync(FULL, a.s1, mask) : 0.f;
    return o;
}

template <bool ENT>
__device__ __forceinline__ Soft soft_warp_allreduce(Soft a, float k) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = soft_merge<ENT>(a, soft_shfl_xor<ENT>(a, o), k);
    return a;
}

// Symmetric butterfly sum (every lane ends with the same bits).
__device__ __forceinline__ float warp_allsum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
    return v;
}

__device__ __forceinline__ int warp_allor(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v |= __shfl_xor_sync(FULL, v, o);
    return v;
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
