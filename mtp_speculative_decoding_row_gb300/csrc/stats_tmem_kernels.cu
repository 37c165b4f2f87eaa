// stats_tmem_kernels.cu -- per-position overlap and target entropy with the
// draft rows parked in tensor memory (sm_103a) ("Breaking Entropy Bounds:
// Accelerating RL Training via MTP with Rejection Sampling", §3 and §8:
// alpha = sum_v min(p_v, q_v) = 1 - TV; entropy H(p) = -sum_v p_v ln p_v).
//
// For sequence b, p_i = softmax(target[b,i] / T_b) (i <= gamma) and q_i =
// softmax(draft[b,i] / T_b) (i < gamma):
//     alpha[b,i] = sum_v 2^{min(lp_v, lq_v)},  lp = z_t k - ct, lq = z_d k - cd,
//     H[b,i]     = ln s - ln 2 s1 / s,  s = sum_v 2^{d_v}, s1 = sum_v 2^{d_v} d_v,
// with k = log2(e) / T_b, d = (z_t - m) k and ct, cd the log2 normalisers.
//
// Every logit is read from HBM once.  A kernel that allocates TMEM runs one
// CTA per SM; a persistent cluster of C CTAs x 16 warps handles one sequence
// at a time (c, c + NC, ...), the vocabulary cut into S = 16 C contiguous
// segments of whole 16-byte vectors, one per warp.  Each warp streams its
// segments through a private ring of bulk-copy slots (one row segment per
// slot) in a fixed order:
//   N(i): target row i (softmax and entropy partials) and draft row i
//     (softmax partial), parked in the warp's TMEM columns as it streams;
//     one 32-byte record per warp to every CTA (DSMEM push);
//   O(i), one step behind N: target row i once more (read a few
//     microseconds earlier, so from L2) and the parked draft row i with the
//     final normalisers: the alpha partial, one record per warp;
//   N(gamma): the last target row, entropy only.
// The re-read in O follows the first read closely, so the rows in flight
// between the two stay far below the L2 size; with the draft on chip, the
// only second read of a logit is that L2 hit.  Two draft rows are parked at
// a time (O(i) runs after N(i + 1)); the planner picks C so that they fit
// the warp's 128 of the SM's 512 TMEM columns.  All waits are bounded; the
// ring runs ahead into the next sequence while the exchanges complete.
#include <cstddef>

#include "chunk_math.cuh"
#include "common.cuh"
#include "kernels.h"
#include "tmem.cuh"

namespace mtp {
namespace {

constexpr int NT = 512;          // threads per CTA (one CTA per SM: it holds all TMEM columns)
constexpr int NW = NT / 32;      // warps (segments) per CTA; four per TMEM lane quarter
constexpr int MAXC = 8;          // largest cluster
constexpr int MAXS = MAXC * NW;  // segments per cluster
constexpr int MAXG = 8;          // largest gamma
constexpr int QMAX = 2 * MAXG + 1;  // exchange rounds per sequence
constexpr int MAXR = 8;          // ring slots per warp
constexpr int WCOLS = TMEM_COLS / (NW / 4);  // TMEM columns of one warp
constexpr int PARKED = 2;        // draft rows parked at a time

struct SWarp {
    unsigned long long full[MAXR];  // ring slot barriers
};

// Fixed header; the exchange records ([2 gamma + 1][S][2] float4: rounds
// 0..gamma are N(i), rounds gamma+1.. are O(i)) and the rings ([NW][R][NS *
// 32] vectors) follow.  One bank: a warp pushes a record of the next
// sequence only after every warp of the cluster has pushed (so read) every
// round of this one.
struct SShared {
    unsigned long long xbar[QMAX];
    uint32_t tmem_base;
    SWarp w[NW];
};
constexpr uint32_t HDR_BYTES = (sizeof(SShared) + 127u) & ~127u;

__host__ __device__ constexpr uint32_t srec_bytes(int gamma, int S) {
    return ((static_cast<uint32_t>(2 * gamma + 1) * static_cast<uint32_t>(S) * 32u) + 127u) & ~127u;
}
// A ring slot holds one row segment: NS x 32 vectors.
__host__ __device__ constexpr uint32_t sslot_bytes(int ns) { return static_cast<uint32_t>(ns) * 32u * 16u; }
__host__ __device__ constexpr int sgroup_size(int ns) { return ns % 5 == 0 ? 5 : ns % 4 == 0 ? 4 : ns; }

template <int NS>
struct SGroup {
    static constexpr int GS = sgroup_size(NS);
    static constexpr int NG = NS / GS;
};

enum { U_NT = 0, U_ND = 1, U_OT = 2 };

// Copy u (0 <= u <= 3 gamma) of a sequence: N(0) (target, draft), then N(i)
// and the target re-read of O(i - 1) in turn, then N(gamma) (target alone)
// and O(gamma - 1).
__device__ __forceinline__ void sunit(int u, int g, int &kind, int &i) {
    if (u < 2) {
        kind = u;
        i = 0;
    } else if (u == 3 * g - 1) {
        kind = U_NT;
        i = g;
    } else if (u == 3 * g) {
        kind = U_OT;
        i = g - 1;
    } else {
        const int j = u - 2;
        i = 1 + j / 3;
        kind = j % 3;
        if (kind == U_OT) i -= 1;
    }
}

struct SC {
    int C, rank, warp, lane, sg, S, NC, cid, R, g, Q;
    int seg_lo, seg_n;
    unsigned char *ring;
    SWarp *ws;
    float4 *rec;
    uint32_t tbase;
    // producer
    uint32_t pcount, pslot;
    int p_ord, p_u;
    bool p_done;
    // consumer
    uint32_t ccount, cslot, cphase;
    bool dead;
    uint32_t xpar;  // parity of the exchange barriers
};

template <typename Tin>
__device__ __forceinline__ const unsigned char *srow_ptr(const VerifyArgs &A, int b, int kind, int i) {
    const size_t V = static_cast<size_t>(A.V);
    const size_t g = static_cast<size_t>(A.gamma);
    if (kind == U_ND)
        return reinterpret_cast<const unsigned char *>(A.draft) + ((static_cast<size_t>(b) * g + i) * V) * Store<Tin>::ES;
    return reinterpret_cast<const unsigned char *>(A.target) + ((static_cast<size_t>(b) * (g + 1) + i) * V) * Store<Tin>::ES;
}

// A sequence the statistics cannot cover (temperature not > 0 and finite)
// is skipped by producer and consumer alike.
__device__ __forceinline__ bool stemp_ok(float T) { return T > 0.f && T < INFINITY; }

// Next sequence of this cluster with a usable temperature, from ordinal
// `ord` on (A.B when none is left).
__device__ __forceinline__ int snext(const VerifyArgs &A, const SC &c, int &ord) {
    for (;; ++ord) {
        const int b = c.cid + ord * c.NC;
        if (b >= A.B) return A.B;
        if (stemp_ok(__ldg(A.temp + b))) return b;
    }
}

template <typename Tin, int NS>
__device__ __forceinline__ void sproduce(const VerifyArgs &A, SC &c) {
    if (c.p_done || c.dead) return;
    while (c.pcount - c.ccount < static_cast<uint32_t>(c.R)) {
        const int b = c.cid + c.p_ord * c.NC;
        if (c.lane == 0) {
            int kind, i;
            sunit(c.p_u, c.g, kind, i);
            // no proxy fence: the slot's generic reads completed (their values
            // were consumed) before the consumer released it
            const uint32_t bar = smem_addr(&c.ws->full[c.pslot]);
            const uint32_t dst = smem_addr(c.ring + c.pslot * sslot_bytes(NS));
            const uint32_t bytes = static_cast<uint32_t>(c.seg_n) * 16u;
            mbar_arrive_expect_tx_relaxed(bar, bytes);
            bulk_g2s(dst, srow_ptr<Tin>(A, b, kind, i) + static_cast<size_t>(c.seg_lo) * 16u, bytes, bar);
        }
        ++c.pcount;
        if (++c.pslot == static_cast<uint32_t>(c.R)) c.pslot = 0;
        if (++c.p_u == 3 * c.g + 1) {
            c.p_u = 0;
            ++c.p_ord;
            if (snext(A, c, c.p_ord) >= A.B) {
                c.p_done = true;
                return;
            }
        }
    }
}

__device__ __forceinline__ void sconsumed(SC &c) {
    ++c.ccount;
    if (++c.cslot == static_cast<uint32_t>(c.R)) {
        c.cslot = 0;
        c.cphase ^= 1u;
    }
}

// Bounded wait with one verdict for the whole warp (the tcgen05 accesses
// that follow are warp-wide).
__device__ __forceinline__ bool swait_warp(uint32_t bar, uint32_t parity) {
    return __all_sync(FULL, mbar_wait_sleep(bar, parity) ? 1 : 0) != 0;
}

__device__ __forceinline__ float4 *srec(const SC &c, int round, int q, int half) {
    return c.rec + ((static_cast<size_t>(round) * c.S + q) * 2 + half);
}

__device__ __forceinline__ void spush(SShared &sh, const SC &c, int round, float4 a, float4 b) {
    if (c.lane < c.C) {
        const uint32_t rbar = map_rank(smem_addr(&sh.xbar[round]), c.lane);
        const uint32_t ra = map_rank(smem_addr(srec(c, round, c.sg, 0)), c.lane);
        st_async_v4(ra, a.x, a.y, a.z, a.w, rbar);
        st_async_v4(ra + 16, b.x, b.y, b.z, b.w, rbar);
    }
}

__device__ __forceinline__ bool swait_round(SShared &sh, SC &c, int round) {
    if (c.dead) return false;
    if (!swait_warp(smem_addr(&sh.xbar[round]), c.xpar)) c.dead = true;
    return !c.dead;
}

template <typename Tin, int NS>
__device__ __forceinline__ bool sslot_ready(const VerifyArgs &A, SC &c) {
    sproduce<Tin, NS>(A, c);
    if (c.pcount == c.ccount || !swait_warp(smem_addr(&c.ws->full[c.cslot]), c.cphase)) {
        c.dead = true;
        return false;
    }
    return true;
}

template <typename Tin, int NS>
__device__ __forceinline__ void srelease(const VerifyArgs &A, SC &c) {
    __syncwarp();
    sconsumed(c);
    sproduce<Tin, NS>(A, c);
}

template <typename Tin, int NS>
__device__ __forceinline__ void sload_group(const SC &c, int gi, uint4 (&v)[SGroup<NS>::GS]) {
    constexpr int GS = SGroup<NS>::GS;
    const uint4 NEG = make_uint4(NegInf<Tin>::w, NegInf<Tin>::w, NegInf<Tin>::w, NegInf<Tin>::w);
    const unsigned char *buf = c.ring + c.cslot * sslot_bytes(NS);
#pragma unroll
    for (int q = 0; q < GS; ++q) {
        const int j = (gi * GS + q) * 32 + c.lane;
        v[q] = j < c.seg_n ? vec_at(buf, j) : NEG;
    }
}

// TMEM column of vector slot s of the draft row parked in place `pl`.
template <int NS>
__device__ __forceinline__ uint32_t scol(int pl, int s) {
    return static_cast<uint32_t>((pl * NS + s) * 4);
}

// N pass of one row: the lane's partial (m, s, and with ENT s1) over its
// vectors of the row; a draft row (PARK) is also parked in TMEM place pl.
template <typename Tin, int NS, bool ENT, bool PARK>
__device__ __forceinline__ void snorm_row(const VerifyArgs &A, SC &c, int pl, float k, float &m, float &s, float &s1,
                                          int &bad) {
    constexpr int GS = SGroup<NS>::GS, NG = SGroup<NS>::NG;
    m = -INFINITY;
    s = 0.f;
    s1 = 0.f;
    const bool have = c.seg_n > 0;
    if (have && !sslot_ready<Tin, NS>(A, c)) return;
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
        uint4 v[GS];
        sload_group<Tin, NS>(c, gi, v);
        // the maximum consumes every loaded register: after the last group
        // the slot's reads are complete and it is handed back
        const float cmx = chunk_max<Tin, GS>(v);
        if (have && gi == NG - 1) srelease<Tin, NS>(A, c);
        if (PARK) {
#pragma unroll
            for (int q = 0; q < GS; ++q) tmem_st_v4(c.tbase + scol<NS>(pl, gi * GS + q), v[q]);
        }
        if (ENT) fold_ent<Tin, GS>(v, cmx, k, m, s, s1, bad);
        else fold_regs<Tin, GS>(v, cmx, k, m, s, bad);
    }
    if (PARK) tmem_wait_st();
}

// Overlap sum of one group: sum 2^{min(lp, lq)}.
template <typename Tin, int QV>
__device__ __forceinline__ float alpha_regs(const uint4 (&rt)[QV], const uint4 (&rd)[QV], float k, float ct, float cd) {
    const uint64_t K2 = f2pack(k, k), NCT = f2pack(-ct, -ct), NCD = f2pack(-cd, -cd);
    uint64_t aa = f2pack(0.f, 0.f);
#pragma unroll
    for (int q = 0; q < QV; ++q) {
        const uint32_t wt[4] = {rt[q].x, rt[q].y, rt[q].z, rt[q].w}, wd[4] = {rd[q].x, rd[q].y, rd[q].z, rd[q].w};
#pragma unroll
        for (int h = 0; h < (Store<Tin>::ES == 2 ? 4 : 2); ++h) {
            uint64_t zt2, zd2;
            if (Store<Tin>::ES == 2) {
                zt2 = bf16pair_f2(wt[h]);
                zd2 = bf16pair_f2(wd[h]);
            } else {
                zt2 = f2pack(__uint_as_float(wt[2 * h]), __uint_as_float(wt[2 * h + 1]));
                zd2 = f2pack(__uint_as_float(wd[2 * h]), __uint_as_float(wd[2 * h + 1]));
            }
            float lp0, lp1, lq0, lq1;
            f2unpack(f2fma(zt2, K2, NCT), lp0, lp1);
            f2unpack(f2fma(zd2, K2, NCD), lq0, lq1);
            aa = f2add(aa, f2pack(ex2(fminf(lp0, lq0)), ex2(fminf(lp1, lq1))));
        }
    }
    float a0, a1;
    f2unpack(aa, a0, a1);
    return a0 + a1;
}

// Merged normaliser of one row from the round's records: lane l merges
// segments MAXS/32 l .. (every warp alike); half 0 (target, with s1) or 1.
template <bool ENT>
__device__ __forceinline__ Soft sgather(const SC &c, int round, int half, float k) {
    Soft a = soft_empty();
#pragma unroll
    for (int h = 0; h < MAXS / 32; ++h) {
        const int q = (MAXS / 32) * c.lane + h;
        if (q < c.S) {
            const float4 v = *srec(c, round, q, half);
            if (v.y != 0.f || !(v.y == v.y)) {  // an empty segment adds nothing; a NaN sum propagates
                const float M = fmaxf(a.m, v.x);
                const float da = (M - a.m) * k, dv = (M - v.x) * k;
                const float sa = a.s != 0.f ? ex2(-da) : 0.f, sv = ex2(-dv);
                if (ENT) a.s1 = (a.s != 0.f ? sa * fmaf(-da, a.s, a.s1) : 0.f) + sv * fmaf(-dv, v.y, v.z);
                a.s = a.s * sa + v.y * sv;
                a.m = M;
            }
        }
    }
    return soft_warp_allreduce<ENT>(a, k);
}

template <typename Tin, int NS>
__global__ void __launch_bounds__(NT, 1) stm_kernel_impl(const VerifyArgs A) {
    using St = Store<Tin>;
    constexpr int VEC = St::VEC;
    constexpr int GS = SGroup<NS>::GS, NG = SGroup<NS>::NG;
    extern __shared__ __align__(128) unsigned char smem[];
    SShared &sh = *reinterpret_cast<SShared *>(smem);

    SC c;
    c.C = static_cast<int>(cluster_size());
    c.rank = static_cast<int>(cluster_rank());
    c.cid = static_cast<int>(cluster_id_x());
    c.NC = static_cast<int>(gridDim.x) / c.C;
    c.warp = threadIdx.x >> 5;
    c.lane = threadIdx.x & 31;
    c.S = c.C * NW;
    c.sg = c.rank * NW + c.warp;
    c.R = A.ring;
    c.g = A.gamma;
    c.Q = 2 * A.gamma + 1;
    const int g = c.g;
    const int nv = A.V / VEC;
    const int nvs = A.seg_vectors;
    c.seg_lo = min(nv, c.sg * nvs);
    c.seg_n = min(nv, c.seg_lo + nvs) - c.seg_lo;
    c.ws = &sh.w[c.warp];
    c.rec = reinterpret_cast<float4 *>(smem + HDR_BYTES);
    c.ring = smem + HDR_BYTES + srec_bytes(g, c.S) + static_cast<size_t>(c.warp) * c.R * sslot_bytes(NS);
    c.pcount = c.ccount = 0;
    c.pslot = c.cslot = c.cphase = 0;
    c.p_ord = c.p_u = 0;
    c.dead = false;
    c.xpar = 0;
    c.p_done = c.seg_n <= 0 || snext(A, c, c.p_ord) >= A.B;

    if (c.warp == 0) tmem_alloc(&sh.tmem_base, TMEM_COLS);
    if (c.lane == 0)
        for (int s = 0; s < c.R; ++s) mbar_init(smem_addr(&c.ws->full[s]), 1);
    if (threadIdx.x == 0) {
        for (int i = 0; i < c.Q; ++i) mbar_init(smem_addr(&sh.xbar[i]), 1);
        fence_mbar_init();
        for (int i = 0; i < c.Q; ++i) mbar_arrive_expect_tx(smem_addr(&sh.xbar[i]), static_cast<uint32_t>(c.S) * 32u);
    }
    fence_mbar_init();
    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    c.tbase = tmem_addr(sh.tmem_base, static_cast<uint32_t>((c.warp & 3) * 32),
                        static_cast<uint32_t>((c.warp >> 2) * WCOLS));
    cluster_sync();  // every barrier of the cluster is initialised and armed before any push
    sproduce<Tin, NS>(A, c);

    for (int b = c.cid; b < A.B; b += c.NC) {
        const float T = __ldg(A.temp + b);
        int flags = 0;
        float alpha_l = NAN, ent_l = NAN;  // lane i: alpha_i (i < gamma), H_i (i <= gamma)
        if (!stemp_ok(T)) {
            flags = F_BAD_TEMP;  // the statistics need T > 0 (T = 0, greedy, included)
        } else if (c.dead) {
            flags = F_TIMEOUT;
        } else {
            const float k = LOG2E / T;
            float ctl = 0.f, cdl = 0.f;  // the previous step's log2 normalisers (for O)
            // ---- N(i) for i < gamma, then O(i - 1); N(gamma) (target only) before O(gamma - 1)
            for (int u = 0; u <= g && !c.dead; ++u) {
                float mt, st, s1t, md = -INFINITY, sd = 0.f, s1d;
                int bad = 0;
                snorm_row<Tin, NS, true, false>(A, c, 0, k, mt, st, s1t, bad);
                if (c.dead) break;
                if (u < g) {
                    snorm_row<Tin, NS, false, true>(A, c, u % PARKED, k, md, sd, s1d, bad);
                    if (c.dead) break;
                }
                Soft a;
                a.m = mt;
                a.s = st;
                a.s1 = s1t;
                // the lane partials to the warp's record (exact merge, s1 with it)
                const Soft wt = soft_warp_allreduce<true>(a, k);
                a.m = md;
                a.s = sd;
                a.s1 = 0.f;
                const Soft wd = soft_warp_allreduce<false>(a, k);
                const bool wbad = warp_allor(bad) != 0;
                spush(sh, c, u, make_float4(wt.m, wbad ? NAN : wt.s, wt.s1, 0.f),
                      make_float4(wd.m, wbad ? NAN : wd.s, 0.f, 0.f));
                if (u == 0) continue;
                // ---- O(u - 1): the final normalisers of step u - 1, the target
                // row again (from L2) and the parked draft row
                const int i = u - 1;
                if (!swait_round(sh, c, i)) break;
                const Soft Ct = sgather<true>(c, i, 0, k), Cd = sgather<false>(c, i, 1, k);
                if (!(Ct.m > -INFINITY) || !(Ct.s > 0.f) || !(Ct.s < INFINITY) || !(Cd.m > -INFINITY) ||
                    !(Cd.s > 0.f) || !(Cd.s < INFINITY))
                    flags |= F_NONFINITE;
                ctl = fmaf(Ct.m, k, log2f(Ct.s));
                cdl = fmaf(Cd.m, k, log2f(Cd.s));
                if (c.lane == i) ent_l = logf(Ct.s) - LN2 * Ct.s1 / Ct.s;
                const bool have = c.seg_n > 0;
                if (have && !sslot_ready<Tin, NS>(A, c)) break;
                float acc = 0.f;
#pragma unroll
                for (int gi = 0; gi < NG; ++gi) {
                    uint4 rt[GS], rd[GS];
#pragma unroll
                    for (int q = 0; q < GS; ++q) tmem_ld_v4(c.tbase + scol<NS>(i % PARKED, gi * GS + q), rd[q]);
                    sload_group<Tin, NS>(c, gi, rt);
                    tmem_wait_ld_regs<GS>(rd);
                    if (have && gi == NG - 1) {
                        // consume the slot's values before handing it back
                        const uint32_t x = consume_regs<GS>(rt);
                        asm volatile("" ::"r"(x));
                        srelease<Tin, NS>(A, c);
                    }
                    acc += alpha_regs<Tin, GS>(rt, rd, k, ctl, cdl);
                }
                spush(sh, c, g + 1 + i, make_float4(warp_allsum(acc), 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f));
            }
            // ---- row gamma's entropy and the overlaps: every warp from the records
            if (!c.dead && swait_round(sh, c, g)) {
                const Soft Ct = sgather<true>(c, g, 0, k);
                if (!(Ct.m > -INFINITY) || !(Ct.s > 0.f) || !(Ct.s < INFINITY)) flags |= F_NONFINITE;
                if (c.lane == g) ent_l = logf(Ct.s) - LN2 * Ct.s1 / Ct.s;
            }
            for (int i = 0; i < g && !c.dead; ++i) {
                if (!swait_round(sh, c, g + 1 + i)) break;
                float a0 = 0.f;
#pragma unroll
                for (int h = 0; h < MAXS / 32; ++h) {
                    const int q = (MAXS / 32) * c.lane + h;
                    if (q < c.S) a0 += srec(c, g + 1 + i, q, 0)->x;
                }
                const float al = warp_allsum(a0);
                if (c.lane == i) alpha_l = al;
            }
            if (c.dead) flags |= F_TIMEOUT;
            // warp 0 re-arms every round of this sequence (all complete); a
            // push of the next sequence comes only after every warp of the
            // cluster has read them
            if (c.warp == 0 && !c.dead) {
                if (c.lane == 0)
                    for (int i = 0; i < c.Q; ++i)
                        mbar_arrive_expect_tx(smem_addr(&sh.xbar[i]), static_cast<uint32_t>(c.S) * 32u);
                __syncwarp();
            }
            c.xpar ^= 1u;
        }
        if (c.sg == 0) {
            const bool err = (flags & ~F_ZERO_MASS) != 0;
            if (c.lane < g) A.alpha[static_cast<size_t>(b) * g + c.lane] = err ? NAN : alpha_l;
            if (c.lane <= g) A.entropy[static_cast<size_t>(b) * (g + 1) + c.lane] = err ? NAN : ent_l;
            if (c.lane == 0 && A.flags) A.flags[b] = flags;
        }
    }

    // copies still in flight (after a bounded wait gave up) land before the CTA leaves
    while (c.ccount != c.pcount) {
        (void)mbar_wait_sleep(smem_addr(&c.ws->full[c.cslot]), c.cphase);
        sconsumed(c);
    }
    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    if (c.warp == 0) tmem_dealloc(sh.tmem_base, TMEM_COLS);
    cluster_sync();  // no CTA leaves while a peer may still push into it
}

}  // namespace

uint32_t stm_smem_bytes(int gamma, int C, int ns, int ring) {
    return HDR_BYTES + srec_bytes(gamma, C * NW) + static_cast<uint32_t>(NW * ring) * sslot_bytes(ns);
}
int stm_threads() { return NT; }
int stm_max_gamma() { return MAXG; }
int stm_max_ring() { return MAXR; }
int stm_warp_cols() { return WCOLS; }
int stm_max_cluster() { return MAXC; }
int stm_parked() { return PARKED; }

const void *stm_kernel(int dtype, int ns) {
#define MTP_STM_PICK(T)                                                                     \
    switch (ns) {                                                                           \
        case 2: return reinterpret_cast<const void *>(&stm_kernel_impl<T, 2>);              \
        case 4: return reinterpret_cast<const void *>(&stm_kernel_impl<T, 4>);              \
        case 5: return reinterpret_cast<const void *>(&stm_kernel_impl<T, 5>);              \
        case 8: return reinterpret_cast<const void *>(&stm_kernel_impl<T, 8>);              \
        case 10: return reinterpret_cast<const void *>(&stm_kernel_impl<T, 10>);            \
        case 15: return reinterpret_cast<const void *>(&stm_kernel_impl<T, 15>);            \
        default: return nullptr;                                                            \
    }
    if (dtype == 0) {
        MTP_STM_PICK(float)
    }
    MTP_STM_PICK(bf16_t)
#undef MTP_STM_PICK
}

}  // namespace mtp
