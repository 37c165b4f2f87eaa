// tv_kernels.cu -- fused forward and backward of the end-to-end TV loss on
// sm_103a ("Breaking Entropy Bounds: Accelerating RL Training via MTP with
// Rejection Sampling", §4 "End-to-end TV loss", App. A, App. F).
//
// Persistent thread-block clusters; cluster c handles token positions
// c, c + NC, ...  For each draft step k of a position the cluster bulk-loads
// the target and draft row slices into shared memory (the next step's pair is
// already in flight while this one is reduced), forms both softmax
// normalisers (online max/sum, cluster all-gather by DSMEM push), then in one
// pass over the on-chip slices accumulates
//     alpha_k = sum_v min(p_v, q_v),   S_k = sum_v 1[q_v <= p_v] q_v
// and records the indicator bits.  The draft slices stay on chip.  After the
// last step every thread evaluates the chain
//     l_t = -sum_{m<=gamma} P_m,  P_m = prod_{i<=m} alpha_i,
//     dl_t/dalpha_k = -P_{k-1} W_k,  W_k = 1 + alpha_{k+1} W_{k+1}, W_gamma = 1
// (no division), and the epilogue streams
//     grad[t,k,j] = grad_scale (dl_t/dalpha_k) (1/T) q_j (1[q_j <= p_j] - S_k)
// from the resident draft slices and bits with 16-byte streaming stores.
// Each logit is read from HBM once and each gradient entry written once; the
// softmax is never materialised.  When fewer than gamma draft slices fit on
// chip, the older ones are re-read in the epilogue.
#include <cstddef>

#include "common.cuh"
#include "kernels.h"

namespace mtp {

constexpr int NT = 256;      // threads per CTA
constexpr int NW = NT / 32;  // warps per CTA

struct TVShared {
    Xchg x;
    float tpart[5][NT];  // per-thread partials (columns)
    float cd[MAX_GAMMA];
    float Sk[MAX_GAMMA];
    float ak[MAX_GAMMA];
    float gk[MAX_GAMMA];
    float loss;
    unsigned long long tbar[2];          // target slots
    unsigned long long dbar[MAX_GAMMA];  // draft slots
};
constexpr uint32_t HDR_BYTES = (sizeof(TVShared) + 127u) & ~127u;
uint32_t tv_hdr_bytes() { return HDR_BYTES; }
int tv_threads() { return NT; }

// Per-thread partials of two rows -> CTA partial in every lane of warp 0
// (column layout in shared memory; warp 0 merges NT/32 per lane, then one
// butterfly).
__device__ __forceinline__ void block_soft2(float (*tp)[NT], Soft &at, Soft &ad, int &bad, float k) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    tp[0][tid] = at.m;
    tp[1][tid] = at.s;
    tp[2][tid] = ad.m;
    tp[3][tid] = ad.s;
    tp[4][tid] = __int_as_float(bad);
    __syncthreads();
    if (warp == 0) {
        const Soft a = soft_lane_merge<false, NW>(tp[0], tp[1], tp[1], lane, k);
        const Soft d = soft_lane_merge<false, NW>(tp[2], tp[3], tp[3], lane, k);
        int bb = 0;
#pragma unroll
        for (int q = 0; q < NW; ++q) bb |= __float_as_int(tp[4][lane + 32 * q]);
        at = soft_warp_allreduce<false>(a, k);
        ad = soft_warp_allreduce<false>(d, k);
        bad = warp_allor(bb);
    }
}

__device__ __forceinline__ void block_sum2(float (*tp)[NT], float &v0, float &v1) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    tp[0][tid] = v0;
    tp[1][tid] = v1;
    __syncthreads();
    if (warp == 0) {
        float r0 = 0.f, r1 = 0.f;
#pragma unroll
        for (int q = 0; q < NW; ++q) {
            r0 += tp[0][lane + 32 * q];
            r1 += tp[1][lane + 32 * q];
        }
        v0 = warp_allsum(r0);
        v1 = warp_allsum(r1);
    }
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
__device__ __forceinline__ const unsigned char *tv_row(const void *base, int t, int k, int g, int V) {
    return reinterpret_cast<const unsigned char *>(base) +
           ((static_cast<size_t>(t) * g + k) * static_cast<size_t>(V)) * Store<Tin>::ES;
}

// Target row of pair (t, k): [N, gamma, V], or shared rows [N + gamma - 1, V]
// where pair (t, k) reads row t + k.
template <typename Tin>
__device__ __forceinline__ const unsigned char *tv_trow(const TVArgs &A, int t, int k) {
    if (A.shared_target)
        return reinterpret_cast<const unsigned char *>(A.target) +
               (static_cast<size_t>(t + k) * static_cast<size_t>(A.V)) * Store<Tin>::ES;
    return tv_row<Tin>(A.target, t, k, A.gamma, A.V);
}

// One row slice by bulk copy on `bar` (thread 0); aligned rows only.
template <typename Tin>
__device__ __forceinline__ void issue_row(const Slice &s, const unsigned char *row, unsigned char *buf, uint32_t bar) {
    if (threadIdx.x == 0 && s.nvec > 0) {
        const uint32_t bytes = static_cast<uint32_t>(s.nvec) * 16u;
        fence_proxy_async();
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s(smem_addr(buf), row + static_cast<size_t>(s.lo) * Store<Tin>::ES, bytes, bar);
    }
}

// One pass over a CTA's target and draft slices with the final normalisers
// (log2 p = z_t k - ct, log2 q = z_d k - cd): this thread's share of
// alpha = sum_v min(p_v, q_v) and S = sum_v 1[q_v <= p_v] q_v (min(p, q) is
// 2^{min(log2 p, log2 q)}, and equals q where q <= p), plus one indicator
// byte per vector (bit e: q <= p for element e).
template <typename Tin, int NTH>
__device__ __forceinline__ void overlap_pass(const unsigned char *tb, const unsigned char *db, unsigned char *bk,
                                             int nvec, float k, float ct, float cd, float &acc_a, float &acc_s) {
    const uint64_t K2 = f2pack(k, k), NCT = f2pack(-ct, -ct), NCD = f2pack(-cd, -cd);
    uint64_t aa = f2pack(0.f, 0.f), as = f2pack(0.f, 0.f);
    for (int j = threadIdx.x; j < nvec; j += NTH) {
        const uint4 rt = vec_at(tb, j), rd = vec_at(db, j);
        const uint32_t wt[4] = {rt.x, rt.y, rt.z, rt.w}, wd[4] = {rd.x, rd.y, rd.z, rd.w};
        unsigned m = 0;
#pragma unroll
        for (int q = 0; q < (Store<Tin>::ES == 2 ? 4 : 2); ++q) {
            uint64_t zt2, zd2;
            if (Store<Tin>::ES == 2) {
                zt2 = bf16pair_f2(wt[q]);
                zd2 = bf16pair_f2(wd[q]);
            } else {
                zt2 = f2pack(__uint_as_float(wt[2 * q]), __uint_as_float(wt[2 * q + 1]));
                zd2 = f2pack(__uint_as_float(wd[2 * q]), __uint_as_float(wd[2 * q + 1]));
            }
            float lp0, lp1, lq0, lq1;
            f2unpack(f2fma(zt2, K2, NCT), lp0, lp1);
            f2unpack(f2fma(zd2, K2, NCD), lq0, lq1);
            const float x0 = ex2(fminf(lp0, lq0)), x1 = ex2(fminf(lp1, lq1));
            const bool b0 = lq0 <= lp0, b1 = lq1 <= lp1;
            aa = f2add(aa, f2pack(x0, x1));
            as = f2add(as, f2pack(b0 ? x0 : 0.f, b1 ? x1 : 0.f));
            m |= (b0 ? 1u : 0u) << (2 * q);
            m |= (b1 ? 1u : 0u) << (2 * q + 1);
        }
        bk[j] = static_cast<unsigned char>(m);
    }
    float a0, a1, s0, s1;
    f2unpack(aa, a0, a1);
    f2unpack(as, s0, s1);
    acc_a = a0 + a1;
    acc_s = s0 + s1;
}

// Gradient of one draft row slice (aligned rows): out[j] =
// q_j * (bit_j ? on : off) with q_j = 2^{z_j k - cd}; each thread writes four
// consecutive outputs per iteration, so every warp store covers 512
// contiguous bytes (streaming stores: the gradient is not re-read).
template <typename Tin, int NTH>
__device__ __forceinline__ void grad_pass(const unsigned char *db, const unsigned char *bk, int nvec, float k,
                                          float cd, float on, float off, float *out) {
    constexpr int VEC = Store<Tin>::VEC;
    const uint64_t K2 = f2pack(k, k), NCD = f2pack(-cd, -cd);
    const int nquad = nvec * VEC / 4;
    float4 *o4 = reinterpret_cast<float4 *>(out);
    for (int h = threadIdx.x; h < nquad; h += NTH) {
        uint64_t z01, z23;
        unsigned m;
        if (Store<Tin>::ES == 2) {
            const uint2 r = reinterpret_cast<const uint2 *>(db)[h];
            z01 = bf16pair_f2(r.x);
            z23 = bf16pair_f2(r.y);
            m = static_cast<unsigned>(bk[h >> 1]) >> ((h & 1) * 4);
        } else {
            const uint4 r = reinterpret_cast<const uint4 *>(db)[h];
            z01 = f2pack(__uint_as_float(r.x), __uint_as_float(r.y));
            z23 = f2pack(__uint_as_float(r.z), __uint_as_float(r.w));
            m = bk[h];
        }
        float d0, d1, d2, d3;
        f2unpack(f2fma(z01, K2, NCD), d0, d1);
        f2unpack(f2fma(z23, K2, NCD), d2, d3);
        float4 g;
        g.x = ex2(d0) * ((m & 1u) ? on : off);
        g.y = ex2(d1) * ((m & 2u) ? on : off);
        g.z = ex2(d2) * ((m & 4u) ? on : off);
        g.w = ex2(d3) * ((m & 8u) ? on : off);
        __stcs(o4 + h, g);
    }
}

template <typename Tin>
__global__ void __launch_bounds__(NT, 2) tv_kernel_impl(const TVArgs A) {
    using S = Store<Tin>;
    constexpr int VEC = S::VEC;
    extern __shared__ __align__(128) unsigned char smem[];
    TVShared &sh = *reinterpret_cast<TVShared *>(smem);
    const int g = A.gamma, V = A.V, nres = A.nres;
    const bool aligned = A.aligned != 0;
    unsigned char *tslot[2];
    tslot[0] = smem + HDR_BYTES;
    tslot[1] = tslot[0] + A.slice_bytes;
    unsigned char *dres = tslot[1] + A.slice_bytes;
    unsigned char *bits = dres + static_cast<size_t>(nres) * A.slice_bytes;

    const int tid = threadIdx.x;
    const int C = static_cast<int>(cluster_size());
    const int rank = static_cast<int>(cluster_rank());
    const int cid = static_cast<int>(cluster_id_x());
    const int NC = static_cast<int>(gridDim.x) / C;
    const Slice s = make_slice<Tin>(V, C, rank);
    const int nvc = slice_vectors(V, VEC, C);  // bit bytes per step
    const bool pipe = (nres == g);             // every draft slice stays on chip

    if (tid == 0) {
        xchg_init(sh.x);
        mbar_init(smem_addr(&sh.tbar[0]), 1);
        mbar_init(smem_addr(&sh.tbar[1]), 1);
        for (int d = 0; d < nres; ++d) mbar_init(smem_addr(&sh.dbar[d]), 1);
        fence_mbar_init();
    }
    const float T = A.temperature;
    const bool bad_temp = !(T > 0.f) || !(T < INFINITY);
    const float k = LOG2E / T;
    __syncthreads();
    cluster_sync();

    // Barrier parities (uniform): target slots and draft slots.
    uint32_t tph = 0;        // bit s: parity of target slot s
    uint32_t dph = 0;        // bit d: parity of draft slot d
    uint32_t tarm = 0, darm = 0;  // armed bits
    int round = 0;
    bool dead = false;
    int pc = 0;  // pairs consumed by this CTA (target slot = pc & 1)

    // A slot's phase advances only when its copy has landed: after a wait
    // that gave up the slot stays armed (the CTA is then dead and issues no
    // further copy), and the drain before exit waits for it once more.
    auto wait_t = [&](int sl) -> bool {
        if (!(tarm & (1u << sl))) return true;
        if (!mbar_wait_bounded(smem_addr(&sh.tbar[sl]), (tph >> sl) & 1u)) return false;
        tph ^= 1u << sl;
        tarm &= ~(1u << sl);
        return true;
    };
    auto wait_d = [&](int sl) -> bool {
        if (!(darm & (1u << sl))) return true;
        if (!mbar_wait_bounded(smem_addr(&sh.dbar[sl]), (dph >> sl) & 1u)) return false;
        dph ^= 1u << sl;
        darm &= ~(1u << sl);
        return true;
    };
    auto load_t = [&](int t, int kk, int sl) {
        if (aligned && s.nvec > 0) {
            issue_row<Tin>(s, tv_trow<Tin>(A, t, kk), tslot[sl], smem_addr(&sh.tbar[sl]));
            tarm |= 1u << sl;
        }
    };
    auto load_d = [&](int t, int kk, int sl) {
        if (aligned && s.nvec > 0) {
            issue_row<Tin>(s, tv_row<Tin>(A.draft, t, kk, g, V), dres + static_cast<size_t>(sl) * A.slice_bytes,
                           smem_addr(&sh.dbar[sl]));
            darm |= 1u << sl;
        }
    };

    int t = cid;
    bool d_issued = false;  // the draft slice of the next pair is already requested
    if (!bad_temp && t < A.N) {
        load_t(t, 0, 0);
        load_d(t, 0, 0);
        d_issued = true;
    }

    for (; t < A.N; t += NC) {
        const int tn = t + NC;  // next position of this cluster
        int flags = bad_temp ? F_BAD_TEMP : 0;
        // (alpha, S) partials of the previous step travel with the next
        // step's normaliser record: gamma + 1 exchange rounds per position.
        float pa = 0.f, ps = 0.f;  // CTA partials of the previous step (warp 0)
        bool have_prev = false;
        for (int kk = 0; kk < g; ++kk) {
            const int ts = pc & 1;
            const int ds = kk % nres;
            unsigned char *tb = tslot[ts];
            unsigned char *db = dres + static_cast<size_t>(ds) * A.slice_bytes;
            int tmo = 0;
            if (!bad_temp && !dead && !d_issued) load_d(t, kk, ds);
            if (!bad_temp && !dead) {
                if (!wait_t(ts)) tmo = 1;
                if (!wait_d(ds)) tmo = 1;
                if (!aligned) {
                    load_slice<Tin, NT>(s, tv_trow<Tin>(A, t, kk), tb, 0, false);
                    load_slice<Tin, NT>(s, tv_row<Tin>(A.draft, t, kk, g, V), db, 0, false);
                }
            }
            // one verdict for the CTA: a slice that did not arrive ends its work
            if (__syncthreads_or(tmo)) {
                tmo = 1;
                dead = true;
            }
            // prefetch the next pair: (t, kk+1), or the next position's first target
            if (!bad_temp && !dead) {
                d_issued = false;
                if (kk + 1 < g) {
                    load_t(t, kk + 1, ts ^ 1);
                    if (nres > 1) {
                        load_d(t, kk + 1, (kk + 1) % nres);
                        d_issued = true;
                    }
                } else if (tn < A.N) {
                    load_t(tn, 0, ts ^ 1);
                }
            }
            ++pc;
            if (flags || dead) continue;

            bool nonfin = false;
            Soft at = thread_soft<Tin, false, NT>(tb, s.nvec, k, nonfin);
            Soft ad = thread_soft<Tin, false, NT>(db, s.nvec, k, nonfin);
            int bad = (nonfin ? F_NONFINITE : 0) | (tmo ? F_TIMEOUT : 0);
            block_soft2(sh.tpart, at, ad, bad, k);
            float rec[8] = {at.m, at.s, ad.m, ad.s, __int_as_float(bad), pa, ps, 0.f};
            bool ok;
            const int slot = xchg_round<8>(sh.x, round, rec, C, rank, ok);
            Soft Ct = soft_empty(), Cd = soft_empty();
            int cb = 0;
            float sa = 0.f, ss = 0.f;
            {
                const int lane = tid & 31;
                Soft a = soft_empty(), d = soft_empty();
                if (lane < C) {
                    const float *r = sh.x.rec[slot][lane];
                    a = {r[0], r[1], 0.f};
                    d = {r[2], r[3], 0.f};
                    cb = __float_as_int(r[4]);
                    sa = r[5];
                    ss = r[6];
                }
                Ct = soft_warp_allreduce<false>(a, k);
                Cd = soft_warp_allreduce<false>(d, k);
                cb = warp_allor(cb);
                sa = warp_allsum(sa);
                ss = warp_allsum(ss);
            }
            if (have_prev && tid == 0) {
                sh.ak[kk - 1] = sa;
                sh.Sk[kk - 1] = ss;
            }
            if (!ok) {
                dead = true;
                cb |= F_TIMEOUT;
            }
            if (!(Ct.m > -INFINITY) || !(Ct.s > 0.f) || !(Ct.s < INFINITY)) cb |= F_NONFINITE;
            if (!(Cd.m > -INFINITY) || !(Cd.s > 0.f) || !(Cd.s < INFINITY)) cb |= F_NONFINITE;
            if (cb) {
                flags |= cb;
                have_prev = false;
                continue;
            }
            const float ct = fmaf(Ct.m, k, log2f(Ct.s));
            const float cd = fmaf(Cd.m, k, log2f(Cd.s));
            if (tid == 0) sh.cd[kk] = cd;

            // overlap, S and indicator bits in one pass over the on-chip slices
            unsigned char *bk = bits + static_cast<size_t>(kk) * nvc;
            float acc_a, acc_s;
            overlap_pass<Tin, NT>(tb, db, bk, s.nvec, k, ct, cd, acc_a, acc_s);
            block_sum2(sh.tpart, acc_a, acc_s);
            pa = acc_a;
            ps = acc_s;
            have_prev = true;
        }
        if (!flags && !dead && have_prev) {  // last step's (alpha, S)
            float rec[8] = {0.f, 0.f, 0.f, 0.f, 0.f, pa, ps, 0.f};
            bool ok;
            const int slot = xchg_round<8>(sh.x, round, rec, C, rank, ok);
            const int lane = tid & 31;
            const float sa = warp_allsum(lane < C ? sh.x.rec[slot][lane][5] : 0.f);
            const float ss = warp_allsum(lane < C ? sh.x.rec[slot][lane][6] : 0.f);
            if (tid == 0) {
                sh.ak[g - 1] = sa;
                sh.Sk[g - 1] = ss;
            }
            if (!ok) dead = true;
        }
        if (dead) flags |= F_TIMEOUT;
        __syncthreads();

        float *gbase = A.grad + static_cast<size_t>(t) * g * static_cast<size_t>(V);
        if (!flags) {
            if (tid == 0) {
                float loss = 0.f;
                if (A.loss_kind == 1) {
                    // App. F per-step loss clamp(1 - alpha_k, 0, tau_max): slope -1
                    // strictly inside the clamp, 0 elsewhere
                    for (int kk = 0; kk < g; ++kk) {
                        const float d = 1.f - sh.ak[kk];
                        loss += fminf(fmaxf(d, 0.f), A.tau_max);
                        sh.gk[kk] = (d > 0.f && d < A.tau_max) ? -1.f : 0.f;
                    }
                } else {
                    // chain of the e2e loss: prefix products forward, W backward
                    float P[MAX_GAMMA];
                    float prod = 1.f;
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
                }
                sh.loss = loss;
            }
            __syncthreads();
            for (int kk = 0; kk < g; ++kk) {
                const unsigned char *db;
                if (kk >= g - nres) {
                    db = dres + static_cast<size_t>(kk % nres) * A.slice_bytes;
                } else {  // re-read a draft slice that did not stay on chip
                    const int sl = (pc - 1) & 1;  // the last pair's target slot is free
                    const unsigned char *drow = tv_row<Tin>(A.draft, t, kk, g, V);
                    bool arrived = true;
                    if (aligned) {
                        if (s.nvec > 0) {
                            issue_row<Tin>(s, drow, tslot[sl], smem_addr(&sh.tbar[sl]));
                            tarm |= 1u << sl;
                        }
                        arrived = wait_t(sl);
                    } else {
                        load_slice<Tin, NT>(s, drow, tslot[sl], 0, false);
                    }
                    if (!__syncthreads_and(arrived ? 1 : 0)) {  // the re-read slice did not arrive
                        dead = true;
                        flags |= F_TIMEOUT;
                        break;
                    }
                    db = tslot[sl];
                }
                const float coef = A.grad_scale * sh.gk[kk] / T;
                const float cd = sh.cd[kk], sk = sh.Sk[kk];
                const float on = coef * (1.f - sk), off = -coef * sk;
                const unsigned char *bk = bits + static_cast<size_t>(kk) * nvc;
                float *out = gbase + static_cast<size_t>(kk) * V;
                if (aligned) {
                    grad_pass<Tin, NT>(db, bk, s.nvec, k, cd, on, off, out + s.lo);
                } else {
                    // four consecutive outputs per thread, masked at the row end
                    const int nquad = s.nvec * VEC / 4;
                    for (int h = tid; h < nquad; h += NT) {
                        float zd[4], gr[4];
                        if (S::ES == 2) {
                            const uint2 r = reinterpret_cast<const uint2 *>(db)[h];
                            zd[0] = __uint_as_float(r.x << 16);
                            zd[1] = __uint_as_float(r.x & 0xffff0000u);
                            zd[2] = __uint_as_float(r.y << 16);
                            zd[3] = __uint_as_float(r.y & 0xffff0000u);
                        } else {
                            const uint4 r = reinterpret_cast<const uint4 *>(db)[h];
                            zd[0] = __uint_as_float(r.x);
                            zd[1] = __uint_as_float(r.y);
                            zd[2] = __uint_as_float(r.z);
                            zd[3] = __uint_as_float(r.w);
                        }
                        const unsigned m = static_cast<unsigned>(bk[(4 * h) / VEC]) >> ((4 * h) % VEC);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float q = ex2(fmaf(zd[e], k, -cd));
                            gr[e] = q * (((m >> e) & 1u) ? on : off);
                        }
                        store_grad<4>(out, s.lo + 4 * h, V, false, gr);
                    }
                }
                __syncthreads();
                if (pipe && kk == 0 && tn < A.N && !dead) {
                    load_d(tn, 0, 0);
                    d_issued = true;
                }
            }
        }
        if (flags) {  // a flagged position (also one that timed out above) gets a zero gradient
            for (int kk = 0; kk < g; ++kk) {
                float *out = gbase + static_cast<size_t>(kk) * V;
                for (int v = s.lo + tid; v < s.hi; v += NT) out[v] = 0.f;
            }
            if (pipe && tn < A.N && !dead && !bad_temp) {
                load_d(tn, 0, 0);
                d_issued = true;
            }
        }
        if (!pipe && tn < A.N && !dead && !bad_temp) {
            load_d(tn, 0, 0);
            d_issued = true;
        }

        if (rank == 0 && tid == 0) {
            A.loss[t] = flags ? NAN : sh.loss;
            if (A.alpha)
                for (int kk = 0; kk < g; ++kk) A.alpha[static_cast<size_t>(t) * g + kk] = flags ? NAN : sh.ak[kk];
            if (A.flags) A.flags[t] = flags;
        }
        __syncthreads();
    }

    // Copies that outlived a bounded wait must land before the CTA exits.
    for (int sl = 0; sl < 2; ++sl) wait_t(sl);
    for (int d = 0; d < nres; ++d) wait_d(d);
    cluster_sync();
}

const void *tv_kernel(int dtype) {
    return dtype == 0 ? reinterpret_cast<const void *>(&tv_kernel_impl<float>)
                      : reinterpret_cast<const void *>(&tv_kernel_impl<bf16_t>);
}

}  // namespace mtp
