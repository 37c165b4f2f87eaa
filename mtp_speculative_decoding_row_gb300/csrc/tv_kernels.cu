// tv_kernels.cu -- fused forward and backward of the end-to-end TV loss on
// sm_103a ("Breaking Entropy Bounds: Accelerating RL Training via MTP with
// Rejection Sampling", §4 "End-to-end TV loss", App. A, App. F).
//
// One thread-block cluster per token position t.  For each draft step k the
// cluster bulk-loads the target and draft row slices into shared memory,
// forms both softmax normalisers (online max/sum, DSMEM combine), then in one
// pass over the on-chip slices accumulates
//     alpha_k = sum_v min(p_v, q_v),   S_k = sum_v 1[q_v <= p_v] q_v
// and records the indicator bits.  The draft slices stay on chip.  After the
// last step every thread evaluates the chain
//     l_t = -sum_{m<=gamma} P_m,  P_m = prod_{i<=m} alpha_i,
//     dl_t/dalpha_k = -P_{k-1} W_k,  W_k = 1 + alpha_{k+1} W_{k+1}, W_gamma = 1
// (no division), and the epilogue streams
//     grad[t,k,j] = grad_scale (dl_t/dalpha_k) (1/T) q_j (1[q_j <= p_j] - S_k)
// from the resident draft slices and bits.  Each logit is read from HBM once
// and each gradient entry written once; the softmax is never materialised.
// When gamma draft slices do not fit on chip, the oldest are re-read from
// global memory in the epilogue.
#include <cstddef>

#include "common.cuh"
#include "kernels.h"

namespace mtp {

struct alignas(16) TRec {
    float tm, ts, dm, ds, x0, x1;
    int bad, pad;
};

struct TVShared {
    TRec rec[2];
    float wred[NW][8];
    float comb[8];
    int combi[4];
    float cd[MAX_GAMMA];
    float Sk[MAX_GAMMA];
    float ak[MAX_GAMMA];
    float gk[MAX_GAMMA];
    float loss;
    unsigned long long bar[2];
};
static_assert(sizeof(TVShared) <= HDR_BYTES, "shared header too large");

// Block + cluster combine of target/draft normalisers.  Results in all threads.
__device__ __forceinline__ void tv_combine_soft(TVShared &sh, Soft at, Soft ad, int bad, float k, int &slot, int C,
                                                Soft &Ct, Soft &Cd, int &cbad) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    at = soft_warp_allreduce<false>(at, k);
    ad = soft_warp_allreduce<false>(ad, k);
    bad = warp_allor(bad);
    if (lane == 0) {
        float *w = sh.wred[warp];
        w[0] = at.m;
        w[1] = at.s;
        w[2] = ad.m;
        w[3] = ad.s;
        w[4] = __int_as_float(bad);
    }
    __syncthreads();
    if (warp == 0) {
        Soft a = soft_empty(), d = soft_empty();
        int bb = 0;
        if (lane < NW) {
            const float *w = sh.wred[lane];
            a = {w[0], w[1], 0.f};
            d = {w[2], w[3], 0.f};
            bb = __float_as_int(w[4]);
        }
        a = soft_warp_allreduce<false>(a, k);
        d = soft_warp_allreduce<false>(d, k);
        bb = warp_allor(bb);
        if (lane == 0) {
            TRec &r = sh.rec[slot];
            r.tm = a.m;
            r.ts = a.s;
            r.dm = d.m;
            r.ds = d.s;
            r.bad = bb;
        }
    }
    cluster_sync();
    if (warp == 0) {
        Soft a = soft_empty(), d = soft_empty();
        int bb = 0;
        if (lane < C) {
            const uint32_t base = map_rank(smem_addr(&sh.rec[slot]), lane);
            a.m = ld_cluster_f32(base + offsetof(TRec, tm));
            a.s = ld_cluster_f32(base + offsetof(TRec, ts));
            d.m = ld_cluster_f32(base + offsetof(TRec, dm));
            d.s = ld_cluster_f32(base + offsetof(TRec, ds));
            bb = ld_cluster_s32(base + offsetof(TRec, bad));
        }
        a = soft_warp_allreduce<false>(a, k);
        d = soft_warp_allreduce<false>(d, k);
        bb = warp_allor(bb);
        if (lane == 0) {
            sh.comb[0] = a.m;
            sh.comb[1] = a.s;
            sh.comb[2] = d.m;
            sh.comb[3] = d.s;
            sh.combi[0] = bb;
        }
    }
    __syncthreads();
    Ct = {sh.comb[0], sh.comb[1], 0.f};
    Cd = {sh.comb[2], sh.comb[3], 0.f};
    cbad = sh.combi[0];
    slot ^= 1;
}

// Block + cluster sums of two values; results in all threads.
__device__ __forceinline__ void tv_cluster_sum2(TVShared &sh, float v0, float v1, int &slot, int C, float &r0,
                                                float &r1) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    v0 = warp_allsum(v0);
    v1 = warp_allsum(v1);
    if (lane == 0) {
        sh.wred[warp][0] = v0;
        sh.wred[warp][1] = v1;
    }
    __syncthreads();
    if (warp == 0) {
        float x0 = (lane < NW) ? sh.wred[lane][0] : 0.f;
        float x1 = (lane < NW) ? sh.wred[lane][1] : 0.f;
        x0 = warp_allsum(x0);
        x1 = warp_allsum(x1);
        if (lane == 0) {
            sh.rec[slot].x0 = x0;
            sh.rec[slot].x1 = x1;
        }
    }
    cluster_sync();
    if (warp == 0) {
        float x0 = 0.f, x1 = 0.f;
        if (lane < C) {
            const uint32_t base = map_rank(smem_addr(&sh.rec[slot]), lane);
            x0 = ld_cluster_f32(base + offsetof(TRec, x0));
            x1 = ld_cluster_f32(base + offsetof(TRec, x1));
        }
        x0 = warp_allsum(x0);
        x1 = warp_allsum(x1);
        if (lane == 0) {
            sh.comb[4] = x0;
            sh.comb[5] = x1;
        }
    }
    __syncthreads();
    r0 = sh.comb[4];
    r1 = sh.comb[5];
    slot ^= 1;
}

// Store VEC gradient values for image vector j of row `out` (elements
// lo + j*VEC ...): 16-byte streaming stores when aligned, else masked scalars.
template <int VEC>
__device__ __forceinline__ void store_grad(float *out, int v0, int V, bool aligned, const float (&gr)[VEC]) {
    if (aligned && v0 + VEC <= V) {
#pragma unroll
        for (int q = 0; q < VEC / 4; ++q)
            __stcs(reinterpret_cast<float4 *>(out + v0) + q,
                   make_float4(gr[4 * q], gr[4 * q + 1], gr[4 * q + 2], gr[4 * q + 3]));
    } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            if (v0 + e < V) out[v0 + e] = gr[e];
    }
}

template <typename Tin>
__global__ void __launch_bounds__(NT, 2) tv_kernel_impl(const TVArgs A) {
    using S = Store<Tin>;
    constexpr int VEC = S::VEC, ES = S::ES;
    extern __shared__ __align__(128) unsigned char smem[];
    TVShared &sh = *reinterpret_cast<TVShared *>(smem);
    const int g = A.gamma, V = A.V, nres = A.nres;
    unsigned char *tb = smem + HDR_BYTES;
    unsigned char *dres = tb + A.slice_bytes;
    unsigned char *bits = dres + static_cast<size_t>(nres) * A.slice_bytes;

    const int tid = threadIdx.x;
    const int C = static_cast<int>(cluster_size());
    const int rank = static_cast<int>(cluster_rank());
    const int t = static_cast<int>(cluster_id_x());
    const uint32_t bar_t = smem_addr(&sh.bar[0]), bar_d = smem_addr(&sh.bar[1]);
    if (tid == 0) {
        mbar_init(bar_t, 1);
        mbar_init(bar_d, 1);
        fence_mbar_init();
    }
    const float T = A.temperature;
    int flags = (!(T > 0.f) || !(T < INFINITY)) ? F_BAD_TEMP : 0;
    __syncthreads();
    cluster_sync();

    const float k = LOG2E / T;
    const Slice s = make_slice<Tin>(V, C, rank);
    const int nvc = slice_vectors(V, VEC, C);  // bit bytes per step
    int slot = 0;
    uint32_t ph_t = 0, ph_d = 0;
    bool pend_t = false, pend_d = false;

    for (int kk = 0; kk < g && !flags; ++kk) {
        const size_t row = (static_cast<size_t>(t) * g + kk) * static_cast<size_t>(V);
        const unsigned char *trow = reinterpret_cast<const unsigned char *>(A.target) + row * ES;
        const unsigned char *drow = reinterpret_cast<const unsigned char *>(A.draft) + row * ES;
        unsigned char *db = dres + static_cast<size_t>(kk % nres) * A.slice_bytes;
        fence_proxy_async();
        const bool arm_t = load_slice<Tin>(s, trow, tb, bar_t, A.aligned != 0);
        const bool arm_d = load_slice<Tin>(s, drow, db, bar_d, A.aligned != 0);
        int tmo = 0;
        if (arm_t) {
            if (!mbar_wait_bounded(bar_t, ph_t)) {
                tmo = 1;
                pend_t = true;
            }
            ph_t ^= 1;
        }
        if (arm_d) {
            if (!mbar_wait_bounded(bar_d, ph_d)) {
                tmo = 1;
                pend_d = true;
            }
            ph_d ^= 1;
        }
        __syncthreads();

        Soft at = soft_empty(), ad = soft_empty();
        bool nonfin = false;
        for (int j = tid; j < s.nvec; j += NT) {
            float zt[VEC], zd[VEC];
            S::unpack(vec_at(tb, j), zt);
            S::unpack(vec_at(db, j), zd);
            soft_add<VEC, false>(at, zt, k, nonfin);
            soft_add<VEC, false>(ad, zd, k, nonfin);
        }
        Soft Ct, Cd;
        int cbad;
        tv_combine_soft(sh, at, ad, (nonfin ? F_NONFINITE : 0) | (tmo ? F_TIMEOUT : 0), k, slot, C, Ct, Cd, cbad);
        int rf = cbad;
        if (!(Ct.m > -INFINITY) || !(Ct.s > 0.f) || !(Ct.s < INFINITY)) rf |= F_NONFINITE;
        if (!(Cd.m > -INFINITY) || !(Cd.s > 0.f) || !(Cd.s < INFINITY)) rf |= F_NONFINITE;
        if (rf) {
            flags |= rf;
            break;
        }
        const float ct = fmaf(Ct.m, k, log2f(Ct.s));
        const float cd = fmaf(Cd.m, k, log2f(Cd.s));

        // overlap, S and indicator bits in one pass over the on-chip slices
        float acc_a = 0.f, acc_s = 0.f;
        unsigned char *bk = bits + static_cast<size_t>(kk) * nvc;
        for (int j = tid; j < s.nvec; j += NT) {
            float zt[VEC], zd[VEC];
            S::unpack(vec_at(tb, j), zt);
            S::unpack(vec_at(db, j), zd);
            unsigned m = 0;
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const float lp = fmaf(zt[e], k, -ct), lq = fmaf(zd[e], k, -cd);
                const float x = ex2(fminf(lp, lq));
                acc_a += x;
                if (lq <= lp) {
                    acc_s += x;
                    m |= 1u << e;
                }
            }
            bk[j] = static_cast<unsigned char>(m);
        }
        float a, sk;
        tv_cluster_sum2(sh, acc_a, acc_s, slot, C, a, sk);
        if (tid == 0) {
            sh.ak[kk] = a;
            sh.Sk[kk] = sk;
            sh.cd[kk] = cd;
        }
        __syncthreads();
    }

    if (!flags) {
        if (tid == 0) {
            // chain of the e2e loss: prefix products forward, W backward
            float P[MAX_GAMMA];
            float prod = 1.f, loss = 0.f;
            for (int kk = 0; kk < g; ++kk) {
                prod *= sh.ak[kk];
                P[kk] = prod;
                loss -= prod;
            }
            float W = 1.f;
            for (int kk = g - 1; kk >= 0; --kk) {
                const float Pprev = kk ? P[kk - 1] : 1.f;
                sh.gk[kk] = -Pprev * W;
                W = fmaf(sh.ak[kk], W, 1.f);
            }
            sh.loss = loss;
        }
        __syncthreads();
        const bool out_aligned = A.aligned != 0;
        for (int kk = 0; kk < g; ++kk) {
            const size_t row = (static_cast<size_t>(t) * g + kk) * static_cast<size_t>(V);
            const unsigned char *db;
            if (kk >= g - nres) {
                db = dres + static_cast<size_t>(kk % nres) * A.slice_bytes;
            } else {  // re-read a draft slice that did not stay on chip
                fence_proxy_async();
                const unsigned char *drow = reinterpret_cast<const unsigned char *>(A.draft) + row * ES;
                if (load_slice<Tin>(s, drow, tb, bar_t, A.aligned != 0)) {
                    if (!mbar_wait_bounded(bar_t, ph_t)) pend_t = true;
                    ph_t ^= 1;
                }
                __syncthreads();
                db = tb;
            }
            const float coef = A.grad_scale * sh.gk[kk] / T;
            const float cd = sh.cd[kk], sk = sh.Sk[kk];
            const float on = coef * (1.f - sk), off = -coef * sk;
            const unsigned char *bk = bits + static_cast<size_t>(kk) * nvc;
            float *out = A.grad + row;
            for (int j = tid; j < s.nvec; j += NT) {
                float zd[VEC], gr[VEC];
                S::unpack(vec_at(db, j), zd);
                const unsigned m = bk[j];
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const float q = ex2(fmaf(zd[e], k, -cd));
                    gr[e] = q * (((m >> e) & 1u) ? on : off);
                }
                store_grad<VEC>(out, s.lo + j * VEC, V, out_aligned, gr);
            }
            __syncthreads();
        }
    } else {
        // flagged position: defined zero gradient
        for (int kk = 0; kk < g; ++kk) {
            float *out = A.grad + (static_cast<size_t>(t) * g + kk) * static_cast<size_t>(V);
            for (int v = s.lo + tid; v < s.hi; v += NT) out[v] = 0.f;
        }
    }

    if (pend_t) mbar_wait_bounded(bar_t, ph_t ^ 1);
    if (pend_d) mbar_wait_bounded(bar_d, ph_d ^ 1);

    if (rank == 0 && tid == 0) {
        const bool err = flags != 0;
        A.loss[t] = err ? NAN : sh.loss;
        if (A.alpha)
            for (int kk = 0; kk < g; ++kk) A.alpha[static_cast<size_t>(t) * g + kk] = err ? NAN : sh.ak[kk];
        if (A.flags) A.flags[t] = flags;
    }
    cluster_sync();
}

const void *tv_kernel(int dtype) {
    return dtype == 0 ? reinterpret_cast<const void *>(&tv_kernel_impl<float>)
                      : reinterpret_cast<const void *>(&tv_kernel_impl<bf16_t>);
}

}  // namespace mtp
