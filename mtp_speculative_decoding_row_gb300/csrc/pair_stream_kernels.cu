// pair_stream_kernels.cu -- per-position statistics of (target, draft) row
// pairs as a streaming kernel on sm_103a ("Breaking Entropy Bounds:
// Accelerating RL Training via MTP with Rejection Sampling", §2 "Acceptance
// methods", §3, §8 "Robustness of acceptance methods", App. E "Rejection
// Sampling Decision Boundary Derivation").
//
// For sequence b and position i, p_i = softmax(z_t[b, i] / T_b) and, for
// i < gamma, q_i = softmax(z_d[b, i] / T_b):
//   statistics:   alpha_i = sum_v min(p_i, q_i)   (= 1 - d_TV(p_i, q_i)),
//                 H(p_i) for i = 0..gamma;
//   diagnostics:  in addition H(q_i), D_KL(q_i || p_i), the draft arg max
//                 yhat_i (ties to the smaller index), p_i(yhat_i) and
//                 rs_better_i = [d_TV(p_i, q_i) < 1 - p_i(yhat_i)], i.e.
//                 [p_i(yhat_i) < alpha_i]: rejection sampling accepts more
//                 often than target-only acceptance of the arg max draft.
//
// Layout of the work.  A persistent cluster of C CTAs x NW warps handles one
// sequence at a time (c, c + NC, ...); the vocabulary is cut into S = C * NW
// contiguous segments, one per warp, and each warp streams its segment of
// the rows through a private ring of bulk-copy chunk slots.  The schedule of
// a sequence is fixed, so the producer (lane 0) simply runs ahead through it:
//   pass N(i), i <= gamma: target row i (and draft row i) from HBM; every
//     one-pass quantity (online softmax partials with the entropy sums, the
//     draft-weighted logit gap for the KL divergence, the draft arg max),
//     pushed as records to every CTA of the cluster (DSMEM);
//   pass O(i), one step behind N: rows i again (now in L2) with the final
//     normalisers: the alpha partial, one record per warp.
// Order: N(0), N(1), O(0), N(2), O(1), ..., N(gamma), O(gamma - 1).  Every
// warp gathers the records itself (same records, same order: the same
// values everywhere); warp 0 of CTA 0 writes the outputs.
//
// Log2 domain: with k = log2(e) / T, a logit z has weight 2^{(z - m) k}
// against the reference m; s = sum of weights, s1 = sum of weight x
// log2(weight), so H = ln s - ln 2 * s1 / s (nats).  The KL divergence is
// ln 2 * (E_q[k (z_d - z_t)] + ct - cd) with ct = m_t k + log2 s_t (and cd
// likewise): the draft-weighted gap x = sum w_d k (z_d - z_t) is a one-pass
// sum that scales like s.
#include <cstddef>

#include "chunk_math.cuh"
#include "common.cuh"
#include "kernels.h"

namespace mtp {
namespace {

constexpr int NT = 128;              // threads per CTA
constexpr int NW = NT / 32;          // warps (segments) per CTA
constexpr int MAXS = 64;             // segments per cluster
constexpr int MAXG = 8;              // largest gamma
constexpr int QMAX = 2 * MAXG + 1;   // exchange rounds per sequence
constexpr int MAXR = 8;              // ring slots per warp

struct PWarp {
    unsigned long long full[MAXR];  // ring slot barriers
};

// Fixed header; the exchange records and the rings follow it.
struct PShared {
    unsigned long long xbar[2][QMAX];
    PWarp w[NW];
};
constexpr uint32_t HDR_BYTES = (sizeof(PShared) + 127u) & ~127u;

// Records per segment in a normaliser round: statistics 2 (target, draft),
// diagnostics 3 (target, draft, arg max).
__host__ __device__ constexpr int nrec_of(int mode) { return mode == PAIR_DIAG ? 3 : 2; }

// float4 records in one bank: (gamma + 1) normaliser rounds of RN per
// segment, gamma overlap rounds of one per segment.
__host__ __device__ constexpr uint32_t bank_recs(int gamma, int S, int mode) {
    return static_cast<uint32_t>((gamma + 1) * nrec_of(mode) + gamma) * static_cast<uint32_t>(S);
}
__host__ __device__ constexpr uint32_t prec_bytes(int gamma, int S, int mode) {
    return ((2u * bank_recs(gamma, S, mode) * 16u) + 127u) & ~127u;
}

enum { P_NORM = 0, P_OVL = 1 };

struct PC {
    int C, rank, warp, lane, sg, S, NC, cid, R, g, Q, cv, RN;
    int seg_lo, seg_n, nch;
    unsigned char *ring;
    PWarp *ws;
    float4 *rec;
    uint32_t bk;  // float4 records per bank
    // producer
    uint32_t pcount, pslot;
    int p_ord, p_u, p_c;
    bool p_done;
    const unsigned char *p_t, *p_d;
    // consumer
    uint32_t ccount, cslot, cphase;
    bool dead;
    int bank;
    uint32_t bpar;
};

__device__ __forceinline__ int pchunk(const PC &c, int ch) { return min(c.cv, c.seg_n - ch * c.cv); }

// Pass u (0 <= u <= 2 gamma) of a sequence: N(0), then N(j) and O(j - 1)
// in turn; the last pass is O(gamma - 1).
__device__ __forceinline__ void punit_of(int u, int &kind, int &i) {
    if (u == 0) {
        kind = P_NORM;
        i = 0;
        return;
    }
    const int j = (u + 1) >> 1;
    kind = (u & 1) ? P_NORM : P_OVL;
    i = (u & 1) ? j : j - 1;
}

template <typename Tin>
__device__ __forceinline__ const unsigned char *prow(const void *base, size_t row, int V) {
    return reinterpret_cast<const unsigned char *>(base) + row * static_cast<size_t>(V) * Store<Tin>::ES;
}

// Issue chunk copies while ring slots are free, in the order of punit_of,
// then the next sequence of the cluster.
template <typename Tin>
__device__ __forceinline__ void pproduce(const PairArgs &A, PC &c) {
    if (c.p_done || c.dead) return;
    while (c.pcount - c.ccount < static_cast<uint32_t>(c.R)) {
        if (c.p_c == 0) {
            const int b = c.cid + c.p_ord * c.NC;
            int kind, i;
            punit_of(c.p_u, kind, i);
            const size_t off = static_cast<size_t>(c.seg_lo) * 16u;
            c.p_t = prow<Tin>(A.target, static_cast<size_t>(b) * (c.g + 1) + i, A.V) + off;
            c.p_d = i < c.g ? prow<Tin>(A.draft, static_cast<size_t>(b) * c.g + i, A.V) + off : nullptr;
        }
        const int cnt = pchunk(c, c.p_c);
        if (c.lane == 0) {
            // no proxy fence: the slot's generic reads completed (their
            // values were consumed) before the consumer released it
            const uint32_t bar = smem_addr(&c.ws->full[c.pslot]);
            const uint32_t dst = smem_addr(c.ring + c.pslot * (2u * c.cv * 16u));
            const uint32_t bytes = static_cast<uint32_t>(cnt) * 16u;
            const size_t off = static_cast<size_t>(c.p_c) * (c.cv * 16);
            mbar_arrive_expect_tx_relaxed(bar, c.p_d ? 2u * bytes : bytes);
            bulk_g2s(dst, c.p_t + off, bytes, bar);
            if (c.p_d) bulk_g2s(dst + c.cv * 16, c.p_d + off, bytes, bar);
        }
        ++c.pcount;
        if (++c.pslot == static_cast<uint32_t>(c.R)) c.pslot = 0;
        if (++c.p_c == c.nch) {
            c.p_c = 0;
            if (++c.p_u == 2 * c.g + 1) {
                c.p_u = 0;
                ++c.p_ord;
                if (c.cid + c.p_ord * c.NC >= A.B) {
                    c.p_done = true;
                    return;
                }
            }
        }
    }
}

__device__ __forceinline__ bool pwait_slot(PC &c) {
    if (c.pcount == c.ccount) c.dead = true;  // nothing issued: never wait on it
    if (c.dead) return false;
    if (!mbar_wait_spin(smem_addr(&c.ws->full[c.cslot]), c.cphase)) {
        c.dead = true;
        return false;
    }
    return true;
}

__device__ __forceinline__ void pconsumed(PC &c) {
    ++c.ccount;
    if (++c.cslot == static_cast<uint32_t>(c.R)) {
        c.cslot = 0;
        c.cphase ^= 1u;
    }
}

__device__ __forceinline__ void pdrain(PC &c) {
    while (c.ccount != c.pcount) {
        if (!mbar_wait_spin(smem_addr(&c.ws->full[c.cslot]), c.cphase)) c.dead = true;
        pconsumed(c);
    }
}

// Record j of segment `seg` in round r of the current bank.
__device__ __forceinline__ float4 *prec(const PC &c, int r, int j, int seg) {
    const uint32_t base = r <= c.g ? static_cast<uint32_t>(r * c.RN) * c.S
                                   : static_cast<uint32_t>((c.g + 1) * c.RN + (r - c.g - 1)) * c.S;
    return c.rec + c.bank * c.bk + base + static_cast<uint32_t>(j * c.S + seg);
}

__device__ __forceinline__ uint32_t pround_bytes(const PC &c, int r) {
    return static_cast<uint32_t>((r <= c.g ? c.RN : 1) * c.S) * 16u;
}

// Push record j of this warp for round r into every CTA of the cluster.
__device__ __forceinline__ void ppush(PShared &sh, const PC &c, int r, int j, float4 v) {
    if (c.lane < c.C) {
        const uint32_t rbar = map_rank(smem_addr(&sh.xbar[c.bank][r]), c.lane);
        const uint32_t ra = map_rank(smem_addr(prec(c, r, j, c.sg)), c.lane);
        st_async_v4(ra, v.x, v.y, v.z, v.w, rbar);
    }
}

__device__ __forceinline__ bool pwait_round(PShared &sh, PC &c, int r) {
    if (c.dead) return false;
    if (!mbar_wait_spin(smem_addr(&sh.xbar[c.bank][r]), (c.bpar >> c.bank) & 1u)) c.dead = true;
    return !c.dead;
}

// ------------------------------------------------------- chunk arithmetic --

// The draft row's fold for the diagnostics: fold_ent over the draft and the
// gap sum x = sum 2^{d} k (z_d - z_t) against the target chunk rt.
template <typename Tin, int QV>
__device__ __forceinline__ void fold_diag(const uint4 (&rd)[QV], const uint4 (&rt)[QV], float cmx, float k, float &m,
                                          float &s, float &s1, float &x, int &bad) {
    using St = Store<Tin>;
    bad |= !(cmx < INFINITY);
    const float nm = fmaxf(m, cmx);
    const float mr = nm > -INFINITY ? nm : 0.f;
    const float dl = (mr - m) * k;
    const float sc = ex2(-dl);
    s1 = (s != 0.f) ? sc * fmaf(-dl, s, s1) : 0.f;
    x = (s != 0.f) ? x * sc : 0.f;
    s *= sc;
    m = nm;
    const float mk = mr * k;
    const uint64_t K2 = f2pack(k, k), NK2 = f2pack(-k, -k), NMK2 = f2pack(-mk, -mk), Z2 = f2pack(0.f, 0.f);
    uint64_t as = Z2, a1 = Z2, ax = Z2;
#pragma unroll
    for (int q = 0; q < QV; ++q) {
        const uint32_t wd[4] = {rd[q].x, rd[q].y, rd[q].z, rd[q].w}, wt[4] = {rt[q].x, rt[q].y, rt[q].z, rt[q].w};
#pragma unroll
        for (int h = 0; h < (St::ES == 2 ? 4 : 2); ++h) {
            uint64_t zd2, zt2;
            if (St::ES == 2) {
                zd2 = bf16pair_f2(wd[h]);
                zt2 = bf16pair_f2(wt[h]);
            } else {
                zd2 = f2pack(__uint_as_float(wd[2 * h]), __uint_as_float(wd[2 * h + 1]));
                zt2 = f2pack(__uint_as_float(wt[2 * h]), __uint_as_float(wt[2 * h + 1]));
            }
            float d0, d1, g0, g1;
            f2unpack(f2fma(zd2, K2, NMK2), d0, d1);
            f2unpack(f2fma(zd2, K2, f2fma(zt2, NK2, Z2)), g0, g1);  // k z_d - k z_t
            d0 = fmaxf(d0, -256.f);
            d1 = fmaxf(d1, -256.f);
            const float e0 = ex2(d0), e1 = ex2(d1);
            const uint64_t e2 = f2pack(e0, e1);
            as = f2add(as, e2);
            a1 = f2fma(e2, f2pack(d0, d1), a1);
            // a zero weight adds nothing (also when both logits are -inf)
            ax = f2fma(e2, f2pack(e0 > 0.f ? g0 : 0.f, e1 > 0.f ? g1 : 0.f), ax);
        }
    }
    float p0, p1;
    f2unpack(as, p0, p1);
    s += p0 + p1;
    f2unpack(a1, p0, p1);
    s1 += p0 + p1;
    f2unpack(ax, p0, p1);
    x += p0 + p1;
}

// alpha partial of one chunk: sum 2^{min(z_t k - ct, z_d k - cd)}.
template <typename Tin, int QV>
__device__ __forceinline__ float overlap_regs(const uint4 (&rt)[QV], const uint4 (&rd)[QV], float k, float ct,
                                              float cd) {
    using St = Store<Tin>;
    const uint64_t K2 = f2pack(k, k), NCT = f2pack(-ct, -ct), NCD = f2pack(-cd, -cd);
    uint64_t aa = f2pack(0.f, 0.f);
#pragma unroll
    for (int q = 0; q < QV; ++q) {
        const uint32_t wt[4] = {rt[q].x, rt[q].y, rt[q].z, rt[q].w}, wd[4] = {rd[q].x, rd[q].y, rd[q].z, rd[q].w};
#pragma unroll
        for (int h = 0; h < (St::ES == 2 ? 4 : 2); ++h) {
            uint64_t zt2, zd2;
            if (St::ES == 2) {
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

// Fold every word of the lane's chunk registers into one value: consuming
// the registers completes the shared-memory loads that filled them, so the
// slot can be handed back before the chunk is processed.
template <int QV>
__device__ __forceinline__ uint32_t consume_words(const uint4 (&r)[QV]) {
    uint32_t x = 0;
#pragma unroll
    for (int q = 0; q < QV; ++q) x ^= r[q].x ^ r[q].y ^ r[q].z ^ r[q].w;
    return x;
}

// ----------------------------------------------------------- partials -----

// Softmax partial with the entropy sum and one more sum that scales like s.
struct SoftX {
    float m, s, s1, x;
};

__device__ __forceinline__ SoftX softx_empty() { return {-INFINITY, 0.f, 0.f, 0.f}; }

// a += b; a NaN sum propagates.
__device__ __forceinline__ void softx_merge(SoftX &a, const SoftX &b, float k) {
    const float M = fmaxf(a.m, b.m);
    SoftX r = {M, 0.f, 0.f, 0.f};
    if (a.s != 0.f) {
        const float dl = (M - a.m) * k, sc = ex2(-dl);
        r.s += a.s * sc;
        r.s1 += sc * fmaf(-dl, a.s, a.s1);
        r.x += a.x * sc;
    }
    if (b.s != 0.f) {
        const float dl = (M - b.m) * k, sc = ex2(-dl);
        r.s += b.s * sc;
        r.s1 += sc * fmaf(-dl, b.s, b.s1);
        r.x += b.x * sc;
    }
    a = r;
}

// Warp all-reduce: exact maximum, one rescale per lane, butterfly sums
// (every lane ends with the same bits).
__device__ __forceinline__ SoftX softx_allreduce(const SoftX &a, float k) {
    SoftX r;
    r.m = warp_allmax(a.m);
    float s = 0.f, s1 = 0.f, x = 0.f;
    if (r.m != -INFINITY && a.s != 0.f) {
        const float dl = (r.m - a.m) * k, sc = ex2(-dl);
        s = a.s * sc;
        s1 = sc * fmaf(-dl, a.s, a.s1);
        x = a.x * sc;
    }
    r.s = warp_allsum(s);
    r.s1 = warp_allsum(s1);
    r.x = warp_allsum(x);
    return r;
}

// Arg max merge: larger value, ties to the smaller index (index -1: none).
__device__ __forceinline__ void amax_merge(float &v, int &i, float &x, float ov, int oi, float ox) {
    if (oi >= 0 && (i < 0 || ov > v || (ov == v && oi < i))) {
        v = ov;
        i = oi;
        x = ox;
    }
}

__device__ __forceinline__ void amax_allreduce(float &v, int &i, float &x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(FULL, v, o), ox = __shfl_xor_sync(FULL, x, o);
        const int oi = __shfl_xor_sync(FULL, i, o);
        amax_merge(v, i, x, ov, oi, ox);
    }
}

// Everything a normaliser round gives for one position.
struct PosNorm {
    SoftX t, d;       // cluster totals (d: diagnostics carry the gap sum in x)
    float yv, zt_at;  // draft arg max value and the target logit there
    int yi;           // draft arg max (-1: none)
};

template <int MODE>
__device__ __forceinline__ PosNorm gather_norm(const PC &c, int i, float k) {
    SoftX lt = softx_empty(), ld = softx_empty();
    float av = -INFINITY, ax = 0.f;
    int ai = -1;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int q = 2 * c.lane + h;
        if (q < c.S) {
            const float4 a = *prec(c, i, 0, q), b = *prec(c, i, 1, q);
            softx_merge(lt, SoftX{a.x, a.y, a.z, 0.f}, k);
            softx_merge(ld, SoftX{b.x, b.y, b.z, b.w}, k);
            if (MODE == PAIR_DIAG) {
                const float4 e = *prec(c, i, 2, q);
                amax_merge(av, ai, ax, b.x, __float_as_int(e.y), e.x);
            }
        }
    }
    PosNorm r;
    r.t = softx_allreduce(lt, k);
    r.d = softx_allreduce(ld, k);
    if (MODE == PAIR_DIAG) amax_allreduce(av, ai, ax);
    r.yv = av;
    r.yi = ai;
    r.zt_at = ax;
    return r;
}

__device__ __forceinline__ bool norm_ok(const SoftX &a) {
    return a.m > -INFINITY && a.s > 0.f && a.s < INFINITY;
}

template <typename Tin, int CV, int MODE>
__global__ void __launch_bounds__(NT, 4) pair_kernel_impl(const PairArgs A) {
    using St = Store<Tin>;
    constexpr int QV = CV / 32;
    static_assert(CV % 32 == 0, "chunk layout: whole vectors per lane");
    constexpr uint32_t SLOT_BYTES = 2u * CV * 16u;
    constexpr bool DIAG = MODE == PAIR_DIAG;
    extern __shared__ __align__(128) unsigned char smem[];
    PShared &sh = *reinterpret_cast<PShared *>(smem);

    PC c;
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
    c.cv = CV;
    c.RN = nrec_of(MODE);
    const int g = c.g;
    const int nv = A.V / St::VEC;
    const int nvs = A.seg_vectors;
    c.seg_lo = min(nv, c.sg * nvs);
    c.seg_n = min(nv, c.seg_lo + nvs) - c.seg_lo;
    c.nch = (c.seg_n + CV - 1) / CV;
    c.ws = &sh.w[c.warp];
    c.rec = reinterpret_cast<float4 *>(smem + HDR_BYTES);
    c.bk = bank_recs(g, c.S, MODE);
    c.ring = smem + HDR_BYTES + prec_bytes(g, c.S, MODE) + static_cast<size_t>(c.warp) * c.R * SLOT_BYTES;
    c.pcount = c.ccount = 0;
    c.pslot = c.cslot = c.cphase = 0;
    c.p_ord = c.p_u = c.p_c = 0;
    c.p_done = c.nch == 0 || c.cid >= A.B;
    c.p_t = c.p_d = nullptr;
    c.dead = false;
    c.bank = 0;
    c.bpar = 0;

    if (c.lane == 0)
        for (int s = 0; s < c.R; ++s) mbar_init(smem_addr(&c.ws->full[s]), 1);
    if (threadIdx.x == 0) {
        for (int bk = 0; bk < 2; ++bk)
            for (int r = 0; r < c.Q; ++r) mbar_init(smem_addr(&sh.xbar[bk][r]), 1);
        fence_mbar_init();
        for (int bk = 0; bk < 2; ++bk)
            for (int r = 0; r < c.Q; ++r) mbar_arrive_expect_tx(smem_addr(&sh.xbar[bk][r]), pround_bytes(c, r));
    }
    fence_mbar_init();
    __syncthreads();
    cluster_sync();  // every barrier of the cluster is initialised and armed before any push
    pproduce<Tin>(A, c);

    for (int b = c.cid; b < A.B; b += c.NC) {
        const float T = A.temp[b];
        int flags = (T > 0.f && T < INFINITY) ? 0 : F_BAD_TEMP;
        const float k = flags ? LOG2E : LOG2E / T;  // a flagged sequence still runs the schedule
        // lane i keeps position i
        float o_alpha = NAN, o_hp = NAN, o_hq = NAN, o_kl = NAN, o_py = NAN;
        int o_y = -1;
        if (c.dead) {
            flags |= F_TIMEOUT;
        } else {
            for (int u = 0; u <= 2 * g && !c.dead; ++u) {
                int kind, i;
                punit_of(u, kind, i);
                const bool has_d = i < g;
                if (kind == P_NORM) {
                    float mt = -INFINITY, st = 0.f, s1t = 0.f, md = -INFINITY, sd = 0.f, s1d = 0.f, xd = 0.f;
                    float av = -INFINITY, ax = 0.f;
                    int ai = -1, bad = 0;
                    for (int ch = 0; ch < c.nch; ++ch) {
                        pproduce<Tin>(A, c);
                        if (!pwait_slot(c)) break;
                        const unsigned char *tb = c.ring + c.cslot * SLOT_BYTES;
                        const unsigned char *db = tb + CV * 16;
                        const int cnt = pchunk(c, ch);
                        uint4 rt[QV], rd[QV];
                        if (cnt == CV) {
                            load_chunk<Tin, true, QV>(tb, cnt, c.lane, rt);
                            if (has_d) load_chunk<Tin, true, QV>(db, cnt, c.lane, rd);
                        } else {
                            load_chunk<Tin, false, QV>(tb, cnt, c.lane, rt);
                            if (has_d) load_chunk<Tin, false, QV>(db, cnt, c.lane, rd);
                        }
                        // the maxima consume every loaded register: the slot's
                        // reads are complete before it is handed back
                        const float cmt = chunk_max<Tin, QV>(rt);
                        const float cmd = has_d ? chunk_max<Tin, QV>(rd) : -INFINITY;
                        __syncwarp();
                        pconsumed(c);
                        pproduce<Tin>(A, c);
                        fold_ent<Tin, QV>(rt, cmt, k, mt, st, s1t, bad);
                        if (has_d) {
                            if (DIAG) {
                                fold_diag<Tin, QV>(rd, rt, cmd, k, md, sd, s1d, xd, bad);
                                argmax_warp<Tin, QV, true>(rd, rt, cmd, c.seg_lo + ch * CV + c.lane, av, ai, ax);
                            } else {
                                fold_regs<Tin, QV>(rd, cmd, k, md, sd, bad);
                            }
                        }
                    }
                    if (c.dead) continue;
                    const bool wbad = warp_allor(bad) != 0;
                    const SoftX wt = softx_allreduce(SoftX{mt, st, s1t, 0.f}, k);
                    const SoftX wd = softx_allreduce(SoftX{md, sd, s1d, xd}, k);
                    ppush(sh, c, i, 0, make_float4(wt.m, wbad ? NAN : wt.s, wt.s1, 0.f));
                    ppush(sh, c, i, 1, make_float4(wd.m, wbad ? NAN : wd.s, wd.s1, wd.x));
                    if (DIAG) {
                        amax_allreduce(av, ai, ax);
                        ppush(sh, c, i, 2, make_float4(ax, __int_as_float(ai), 0.f, 0.f));
                    }
                } else {
                    // ---- O(i): the normalisers of position i, then alpha
                    if (!pwait_round(sh, c, i)) continue;
                    const PosNorm r = gather_norm<MODE>(c, i, k);
                    // a bad temperature is the row's only error (nothing else is examined)
                    if (!(flags & F_BAD_TEMP) && (!norm_ok(r.t) || !norm_ok(r.d) || (DIAG && r.yi < 0)))
                        flags |= F_NONFINITE;
                    const float ct = fmaf(r.t.m, k, log2f(r.t.s)), cd = fmaf(r.d.m, k, log2f(r.d.s));
                    if (c.lane == i) {
                        o_hp = logf(r.t.s) - LN2 * (r.t.s1 / r.t.s);
                        if (DIAG) {
                            o_hq = logf(r.d.s) - LN2 * (r.d.s1 / r.d.s);
                            o_kl = fmaxf(LN2 * (r.d.x / r.d.s + ct - cd), 0.f);
                            o_y = r.yi;
                            o_py = ex2(fmaf(r.zt_at, k, -ct));
                        }
                    }
                    float acc = 0.f;
                    for (int ch = 0; ch < c.nch; ++ch) {
                        pproduce<Tin>(A, c);
                        if (!pwait_slot(c)) break;
                        const unsigned char *tb = c.ring + c.cslot * SLOT_BYTES;
                        const unsigned char *db = tb + CV * 16;
                        const int cnt = pchunk(c, ch);
                        uint4 rt[QV], rd[QV];
                        if (cnt == CV) {
                            load_chunk<Tin, true, QV>(tb, cnt, c.lane, rt);
                            load_chunk<Tin, true, QV>(db, cnt, c.lane, rd);
                        } else {
                            load_chunk<Tin, false, QV>(tb, cnt, c.lane, rt);
                            load_chunk<Tin, false, QV>(db, cnt, c.lane, rd);
                        }
                        const uint32_t x = consume_words<QV>(rt) ^ consume_words<QV>(rd);
                        asm volatile("" ::"r"(x));
                        __syncwarp();
                        pconsumed(c);
                        pproduce<Tin>(A, c);
                        acc += overlap_regs<Tin, QV>(rt, rd, k, ct, cd);
                    }
                    if (c.dead) break;
                    ppush(sh, c, g + 1 + i, 0, make_float4(warp_allsum(acc), 0.f, 0.f, 0.f));
                }
            }
            // ---- H(p_gamma) and the alpha totals
            if (pwait_round(sh, c, g)) {
                const PosNorm r = gather_norm<PAIR_STATS>(c, g, k);
                if (!(flags & F_BAD_TEMP) && !norm_ok(r.t)) flags |= F_NONFINITE;
                if (c.lane == g) o_hp = logf(r.t.s) - LN2 * (r.t.s1 / r.t.s);
            }
            for (int i = 0; i < g; ++i) {
                if (!pwait_round(sh, c, g + 1 + i)) break;
                float a0 = 0.f;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int q = 2 * c.lane + h;
                    if (q < c.S) a0 += prec(c, g + 1 + i, 0, q)->x;
                }
                const float a = warp_allsum(a0);
                if (c.lane == i) o_alpha = a;
            }
            if (c.dead) flags |= F_TIMEOUT;
            // warp 0 closes the bank: every round of this sequence complete, re-armed
            if (c.warp == 0 && !c.dead) {
                for (int r = 0; r < c.Q; ++r) {
                    if (!pwait_round(sh, c, r)) break;
                    if (c.lane == 0) mbar_arrive_expect_tx(smem_addr(&sh.xbar[c.bank][r]), pround_bytes(c, r));
                }
                __syncwarp();
            }
            c.bpar ^= 1u << c.bank;
            c.bank ^= 1;
        }
        if (c.sg == 0) {
            const bool err = flags != 0;
            const int l = c.lane;
            const size_t o = static_cast<size_t>(b) * g + l;
            if (l < g) {
                if (A.alpha) A.alpha[o] = err ? NAN : o_alpha;
                if (DIAG) {
                    if (A.ent_q) A.ent_q[o] = err ? NAN : o_hq;
                    if (A.kl) A.kl[o] = err ? NAN : o_kl;
                    if (A.yhat) A.yhat[o] = err ? -1 : o_y;
                    if (A.p_yhat) A.p_yhat[o] = err ? NAN : o_py;
                    if (A.rs_better) A.rs_better[o] = err ? -1 : (o_py < o_alpha ? 1 : 0);
                }
            }
            if (l <= g && A.ent_p) A.ent_p[static_cast<size_t>(b) * (g + 1) + l] = err ? NAN : o_hp;
            if (l == 0 && A.flags) A.flags[b] = flags;
        }
    }

    pdrain(c);
    __syncthreads();
    cluster_sync();  // no CTA leaves while a peer may still push into it
}

}  // namespace

uint32_t pair_hdr_bytes() { return HDR_BYTES; }
uint32_t pair_rec_bytes(int gamma, int S, int mode) { return prec_bytes(gamma, S, mode); }
int pair_threads() { return NT; }
int pair_max_gamma() { return MAXG; }
int pair_max_segments() { return MAXS; }
int pair_max_ring() { return MAXR; }

const void *pair_kernel(int dtype, int cv, int mode) {
// the diagnostics run on 128- or 160-vector chunks (the 192 variant spills)
#define MTP_PAIR_PICK(T)                                                                              \
    if (mode == PAIR_DIAG)                                                                            \
        return cv == 160 ? reinterpret_cast<const void *>(&pair_kernel_impl<T, 160, PAIR_DIAG>)       \
                         : reinterpret_cast<const void *>(&pair_kernel_impl<T, 128, PAIR_DIAG>);      \
    return cv == 192   ? reinterpret_cast<const void *>(&pair_kernel_impl<T, 192, PAIR_STATS>)        \
           : cv == 160 ? reinterpret_cast<const void *>(&pair_kernel_impl<T, 160, PAIR_STATS>)        \
                       : reinterpret_cast<const void *>(&pair_kernel_impl<T, 128, PAIR_STATS>);
    if (dtype == 0) {
        MTP_PAIR_PICK(float)
    }
    MTP_PAIR_PICK(bf16_t)
#undef MTP_PAIR_PICK
}

}  // namespace mtp
