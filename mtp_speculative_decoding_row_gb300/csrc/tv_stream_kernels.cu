// tv_stream_kernels.cu -- fused forward and backward of the end-to-end TV
// loss as a streaming kernel on sm_103a ("Breaking Entropy Bounds:
// Accelerating RL Training via MTP with Rejection Sampling", §4 "End-to-end
// TV loss", App. A, App. F).
//
// For token position t with draft steps k = 0..gamma-1, p_k = softmax(z_t/T),
// q_k = softmax(z_d/T):
//     alpha_k = sum_v min(p_v, q_v),   S_k = sum_v 1[q_v <= p_v] q_v,
//     l_t = -sum_k P_k,  P_k = prod_{i<=k} alpha_i,
//     dl_t/dalpha_k = -P_{k-1} W_k,  W_k = 1 + alpha_{k+1} W_{k+1}, W_last = 1,
//     grad[t,k,j] = grad_scale (dl_t/dalpha_k) (1/T) q_j (1[q_j <= p_j] - S_k).
//
// Layout of the work.  A persistent cluster of C CTAs x NW warps handles one
// position at a time (c, c + NC, ...); the vocabulary is cut into S = C * NW
// contiguous segments, one per warp, and each warp streams its segment of
// the rows through a private ring of bulk-copy chunk slots.  The schedule of
// a position is fixed (no early exit), so the producer (lane 0) simply runs
// ahead through it:
//   pass N(k), k < gamma: target and draft rows from HBM; online softmax
//     partials, one 16-byte record per warp to every CTA (DSMEM push);
//   pass O(k), one step behind N: the same rows again (now in L2) with the
//     final normalisers: alpha and S partials and one indicator byte per
//     vector kept in shared memory; one record per warp;
//   pass G(k), after every O, latest step first: the draft row again and
//     the indicator bytes: the gradient, written with streaming stores.
// Every warp gathers the records itself and evaluates the chain (same
// records, same order: the same values everywhere).  The number of
// positions in flight is capped so that the rows being re-read stay in L2.
#include <cstddef>

#include "chunk_math.cuh"
#include "common.cuh"
#include "kernels.h"

namespace mtp {
namespace {

constexpr int NT = 128;          // threads per CTA
constexpr int NW = NT / 32;      // warps (segments) per CTA
constexpr int MAXS = 64;         // segments per cluster
constexpr int MAXG = 8;          // largest gamma
constexpr int QMAX = 2 * MAXG;   // exchange rounds per position
constexpr int MAXR = 8;          // ring slots per warp

struct TWarp {
    unsigned long long full[MAXR];  // ring slot barriers
    float ct[MAXG], cd[MAXG];       // log2 normalisers of each step
    float on[MAXG], off[MAXG];      // gradient coefficients of each step
};

// Fixed header; the exchange records ([2][2 gamma][S] float4), the indicator
// bytes ([NW][gamma][segment vectors]) and the rings follow it.
struct TShared {
    unsigned long long xbar[2][QMAX];
    TWarp w[NW];
};
constexpr uint32_t HDR_BYTES = (sizeof(TShared) + 127u) & ~127u;

__host__ __device__ constexpr uint32_t trec_bytes(int gamma, int S) {
    return ((2u * static_cast<uint32_t>(2 * gamma) * static_cast<uint32_t>(S) * 16u) + 127u) & ~127u;
}
__host__ __device__ constexpr uint32_t tbits_bytes(int gamma, int nvs) {
    return ((static_cast<uint32_t>(NW) * static_cast<uint32_t>(gamma) * static_cast<uint32_t>(nvs)) + 127u) & ~127u;
}

enum { P_NORM = 0, P_OVL = 1, P_GRAD = 2 };

struct TC {
    int C, rank, warp, lane, sg, S, NC, cid, R, g, Q, cv;
    int seg_lo, seg_n, nch;
    unsigned char *ring;
    unsigned char *bits;  // this warp's indicator bytes [gamma][seg_n]
    TWarp *ws;
    float4 *rec;
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

template <typename Tin>
__device__ __forceinline__ const unsigned char *tv_row_ptr(const void *base, int t, int k, int g, int V) {
    return reinterpret_cast<const unsigned char *>(base) +
           ((static_cast<size_t>(t) * g + k) * static_cast<size_t>(V)) * Store<Tin>::ES;
}

__device__ __forceinline__ int tchunk(const TC &c, int ch) { return min(c.cv, c.seg_n - ch * c.cv); }

// Pass u (0 <= u < 3 g) of a position: N(0), then N(k) and O(k - 1) in
// turn, then O(g - 1), then G(g-1), ..., G(0).
__device__ __forceinline__ void unit_of(int u, int g, int &kind, int &k) {
    if (u == 0) {
        kind = P_NORM;
        k = 0;
    } else if (u < 2 * g - 1) {
        const int j = (u + 1) >> 1;
        kind = (u & 1) ? P_NORM : P_OVL;
        k = (u & 1) ? j : j - 1;
    } else if (u == 2 * g - 1) {
        kind = P_OVL;
        k = g - 1;
    } else {
        kind = P_GRAD;
        k = 3 * g - 1 - u;  // latest step first: its draft row is the most recently read
    }
}

// Issue chunk copies while ring slots are free, in the order of unit_of,
// then the next position.
template <typename Tin, bool TOPK>
__device__ __forceinline__ void tproduce(const TVArgs &A, TC &c) {
    if (c.p_done || c.dead) return;
    while (c.pcount - c.ccount < static_cast<uint32_t>(c.R)) {
        if (c.p_c == 0) {
            const int t = c.cid + c.p_ord * c.NC;
            int kind, k;
            unit_of(c.p_u, c.g, kind, k);
            if (TOPK && kind == P_OVL) {  // top-K overlap passes stream no row
                if (++c.p_u == 3 * c.g) {
                    c.p_u = 0;
                    ++c.p_ord;
                    if (c.cid + c.p_ord * c.NC >= A.N) {
                        c.p_done = true;
                        return;
                    }
                }
                continue;
            }
            const size_t off = static_cast<size_t>(c.seg_lo) * 16u;
            c.p_t = (kind == P_GRAD || TOPK) ? nullptr
                                             : (A.shared_target ? tv_row_ptr<Tin>(A.target, t + k, 0, 1, A.V)
                                                                : tv_row_ptr<Tin>(A.target, t, k, c.g, A.V)) +
                                                   off;
            c.p_d = tv_row_ptr<Tin>(A.draft, t, k, c.g, A.V) + off;
        }
        const int cnt = tchunk(c, c.p_c);
        if (c.lane == 0) {
            // no proxy fence: the slot's generic reads completed (their
            // values were consumed) before the consumer released it
            const uint32_t bar = smem_addr(&c.ws->full[c.pslot]);
            const uint32_t dst = smem_addr(c.ring + c.pslot * (2u * c.cv * 16u));
            const uint32_t bytes = static_cast<uint32_t>(cnt) * 16u;
            const size_t off = static_cast<size_t>(c.p_c) * (c.cv * 16);
            mbar_arrive_expect_tx_relaxed(bar, c.p_t ? 2u * bytes : bytes);
            if (c.p_t) bulk_g2s(dst, c.p_t + off, bytes, bar);
            bulk_g2s(dst + c.cv * 16, c.p_d + off, bytes, bar);
        }
        ++c.pcount;
        if (++c.pslot == static_cast<uint32_t>(c.R)) c.pslot = 0;
        if (++c.p_c == c.nch) {
            c.p_c = 0;
            if (++c.p_u == 3 * c.g) {
                c.p_u = 0;
                ++c.p_ord;
                if (c.cid + c.p_ord * c.NC >= A.N) {
                    c.p_done = true;
                    return;
                }
            }
        }
    }
}

__device__ __forceinline__ bool twait_slot(TC &c) {
    if (c.pcount == c.ccount) c.dead = true;  // nothing issued: never wait on it
    if (c.dead) return false;
    if (!mbar_wait_spin(smem_addr(&c.ws->full[c.cslot]), c.cphase)) {
        c.dead = true;
        return false;
    }
    return true;
}

__device__ __forceinline__ void tconsumed(TC &c) {
    ++c.ccount;
    if (++c.cslot == static_cast<uint32_t>(c.R)) {
        c.cslot = 0;
        c.cphase ^= 1u;
    }
}

__device__ __forceinline__ void tdrain(TC &c) {
    while (c.ccount != c.pcount) {
        if (!mbar_wait_spin(smem_addr(&c.ws->full[c.cslot]), c.cphase)) c.dead = true;
        tconsumed(c);
    }
}

__device__ __forceinline__ float4 *trec(const TC &c, int i, int r) {
    return c.rec + (static_cast<size_t>(c.bank * c.Q + i) * c.S + r);
}

__device__ __forceinline__ void tpush(TShared &sh, const TC &c, int i, float4 v) {
    if (c.lane < c.C) {
        const uint32_t rbar = map_rank(smem_addr(&sh.xbar[c.bank][i]), c.lane);
        const uint32_t ra = map_rank(smem_addr(trec(c, i, c.sg)), c.lane);
        st_async_v4(ra, v.x, v.y, v.z, v.w, rbar);
    }
}

__device__ __forceinline__ bool twait_round(TShared &sh, TC &c, int i) {
    if (c.dead) return false;
    if (!mbar_wait_spin(smem_addr(&sh.xbar[c.bank][i]), (c.bpar >> c.bank) & 1u)) c.dead = true;
    return !c.dead;
}

// Zero this warp's segment of one gradient row (flagged positions).
template <typename Tin>
__device__ __forceinline__ void zero_segment(const TC &c, float *row) {
    constexpr int VEC = Store<Tin>::VEC;
    float4 *o = reinterpret_cast<float4 *>(row + static_cast<size_t>(c.seg_lo) * VEC);
    const int n4 = c.seg_n * VEC / 4;
    for (int i = c.lane; i < n4; i += 32) __stcs(o + i, make_float4(0.f, 0.f, 0.f, 0.f));
}

template <typename Tin, int CV, bool TOPK>
__global__ void __launch_bounds__(NT, 4) tvs_kernel_impl(const TVArgs A) {
    using St = Store<Tin>;
    constexpr int VEC = St::VEC;
    constexpr int QV = CV / 32;
    static_assert(CV % 32 == 0, "chunk layout: whole vectors per lane");
    constexpr uint32_t SLOT_BYTES = 2u * CV * 16u;
    extern __shared__ __align__(128) unsigned char smem[];
    TShared &sh = *reinterpret_cast<TShared *>(smem);

    TC c;
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
    c.Q = 2 * A.gamma;
    c.cv = CV;
    const int g = c.g;
    const int nv = A.V / VEC;
    const int nvs = A.seg_vectors;
    c.seg_lo = min(nv, c.sg * nvs);
    c.seg_n = min(nv, c.seg_lo + nvs) - c.seg_lo;
    c.nch = (c.seg_n + CV - 1) / CV;
    c.ws = &sh.w[c.warp];
    c.rec = reinterpret_cast<float4 *>(smem + HDR_BYTES);
    c.bits = smem + HDR_BYTES + trec_bytes(g, c.S) + static_cast<size_t>(c.warp) * g * nvs;
    c.ring = smem + HDR_BYTES + trec_bytes(g, c.S) + tbits_bytes(g, nvs) +
             static_cast<size_t>(c.warp) * c.R * SLOT_BYTES;
    const float T = A.temperature;
    const bool bad_temp = !(T > 0.f) || !(T < INFINITY);
    const float k = LOG2E / T;
    c.pcount = c.ccount = 0;
    c.pslot = c.cslot = c.cphase = 0;
    c.p_ord = c.p_u = c.p_c = 0;
    c.p_done = bad_temp || c.nch == 0 || c.cid >= A.N;
    c.p_t = c.p_d = nullptr;
    c.dead = false;
    c.bank = 0;
    c.bpar = 0;

    if (c.lane == 0)
        for (int s = 0; s < c.R; ++s) mbar_init(smem_addr(&c.ws->full[s]), 1);
    if (threadIdx.x == 0) {
        for (int bk = 0; bk < 2; ++bk)
            for (int i = 0; i < c.Q; ++i) mbar_init(smem_addr(&sh.xbar[bk][i]), 1);
        fence_mbar_init();
        for (int bk = 0; bk < 2; ++bk)
            for (int i = 0; i < c.Q; ++i)
                mbar_arrive_expect_tx(smem_addr(&sh.xbar[bk][i]), static_cast<uint32_t>(c.S) * 16u);
    }
    fence_mbar_init();
    __syncthreads();
    cluster_sync();  // every barrier of the cluster is initialised and armed before any push
    tproduce<Tin, TOPK>(A, c);

    for (int t = c.cid; t < A.N; t += c.NC) {
        float *grow = A.grad + static_cast<size_t>(t) * g * static_cast<size_t>(A.V);
        int flags = 0;
        float loss = NAN;
        float alpha_l = NAN;  // lane kk < g: alpha_kk
        if (bad_temp || c.dead) {
            flags = bad_temp ? F_BAD_TEMP : F_TIMEOUT;
            for (int kk = 0; kk < g; ++kk) zero_segment<Tin>(c, grow + static_cast<size_t>(kk) * A.V);
        } else {
            // ---- N(k) and O(k), the overlap pass one step behind the
            // normaliser pass: N(0), N(1), O(0), N(2), O(1), ..., O(g-1).
            // O(k) re-reads rows k right after N(k+1), while they are in L2,
            // and the all-gather of N(k) overlaps the streaming of N(k+1).
            for (int u = 0; u < 2 * g && !c.dead; ++u) {
                int kind, kk;
                unit_of(u, g, kind, kk);
                if (kind == P_NORM) {
                    float mt = -INFINITY, st = 0.f, md = -INFINITY, sd = 0.f;
                    int bad = 0;
                    for (int ch = 0; ch < c.nch; ++ch) {
                        tproduce<Tin, TOPK>(A, c);
                        if (!twait_slot(c)) break;
                        const unsigned char *tb = c.ring + c.cslot * SLOT_BYTES;
                        const unsigned char *db = tb + CV * 16;
                        const int cnt = tchunk(c, ch);
                        uint4 rt[QV], rd[QV];
                        if (cnt == CV) {
                            if (!TOPK) load_chunk<Tin, true, QV>(tb, cnt, c.lane, rt);
                            load_chunk<Tin, true, QV>(db, cnt, c.lane, rd);
                        } else {
                            if (!TOPK) load_chunk<Tin, false, QV>(tb, cnt, c.lane, rt);
                            load_chunk<Tin, false, QV>(db, cnt, c.lane, rd);
                        }
                        // the maxima consume every loaded register: the slot's
                        // reads are complete before it is handed back
                        const float cmt = TOPK ? -INFINITY : chunk_max<Tin, QV>(rt), cmd = chunk_max<Tin, QV>(rd);
                        __syncwarp();
                        tconsumed(c);
                        tproduce<Tin, TOPK>(A, c);
                        if (!TOPK) fold_regs<Tin, QV>(rt, cmt, k, mt, st, bad);
                        fold_regs<Tin, QV>(rd, cmd, k, md, sd, bad);
                    }
                    if (c.dead) continue;
                    Soft a;
                    a.m = mt;
                    a.s = st;
                    a.s1 = 0.f;
                    const Soft wt = soft_warp_allreduce<false>(a, k);
                    a.m = md;
                    a.s = sd;
                    const Soft wd = soft_warp_allreduce<false>(a, k);
                    const bool wbad = warp_allor(bad) != 0;
                    tpush(sh, c, kk, make_float4(wt.m, wbad ? NAN : wt.s, wd.m, wbad ? NAN : wd.s));
                } else if (TOPK) {
                    // ---- O(k), top-K target: no row streams.  The draft
                    // normaliser from the round, the target normaliser over
                    // the K cached entries (every warp alike), then the
                    // entries that fall in this warp's segment
                    if (!twait_round(sh, c, kk)) continue;
                    Soft ld = soft_empty();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int q = 2 * c.lane + h;
                        if (q < c.S) {
                            const float4 v = *trec(c, kk, q);
                            Soft r;
                            r.m = v.z;
                            r.s = v.w;
                            r.s1 = 0.f;
                            ld = soft_pair_merge(ld, r, k);
                        }
                    }
                    const Soft Cd = soft_warp_allreduce<false>(ld, k);
                    const size_t kb = (static_cast<size_t>(t) * g + kk) * static_cast<size_t>(A.K);
                    const Tin *vals = reinterpret_cast<const Tin *>(A.target) + kb;
                    const int32_t *ids = A.topk_idx + kb;
                    float tm = -INFINITY;
                    int tbad = 0;
                    for (int e = c.lane; e < A.K; e += 32) {
                        const float z = St::scalar_g(vals, e);
                        const int v = __ldg(ids + e);
                        tbad |= !(z < INFINITY) ? F_NONFINITE : 0;
                        tbad |= (v < 0 || v >= A.V) ? F_BAD_ID : 0;
                        tm = fmaxf(tm, z);
                    }
                    tm = warp_allmax(tm);
                    tbad = warp_allor(tbad);
                    float ts = 0.f;
                    if (tm > -INFINITY)
                        for (int e = c.lane; e < A.K; e += 32)
                            ts += ex2((St::scalar_g(vals, e) - tm) * k);
                    ts = warp_allsum(ts);
                    if (!(tm > -INFINITY) || !(ts > 0.f) || !(ts < INFINITY) || !(Cd.m > -INFINITY) || !(Cd.s > 0.f) ||
                        !(Cd.s < INFINITY))
                        tbad |= F_NONFINITE;
                    if (tbad & F_BAD_ID) tbad = F_BAD_ID;  // the first error of the pair, as the oracle reports it
                    flags |= tbad;
                    const float ct = fmaf(tm, k, log2f(ts)), cd = fmaf(Cd.m, k, log2f(Cd.s));
                    if (c.lane == 0) {
                        c.ws->ct[kk] = ct;
                        c.ws->cd[kk] = cd;
                    }
                    float acc_a = 0.f, acc_s = 0.f;
                    if (!tbad) {
                        const unsigned char *drow = tv_row_ptr<Tin>(A.draft, t, kk, g, A.V);
                        const int v_lo = c.seg_lo * VEC, v_hi = (c.seg_lo + c.seg_n) * VEC;
                        for (int e = c.lane; e < A.K; e += 32) {
                            const int v = __ldg(ids + e);
                            if (v < v_lo || v >= v_hi) continue;
                            const float lp = fmaf(St::scalar_g(vals, e), k, -ct);
                            const float lq = fmaf(St::scalar_g(drow, v), k, -cd);
                            const float x = ex2(fminf(lp, lq));
                            acc_a += x;
                            if (lq <= lp) acc_s += x;
                        }
                    }
                    tpush(sh, c, g + kk, make_float4(warp_allsum(acc_a), warp_allsum(acc_s), 0.f, 0.f));
                } else {
                    if (!twait_round(sh, c, kk)) continue;
                    // gather: lane l holds segments 2l and 2l + 1
                    Soft lt = soft_empty(), ld = soft_empty();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int q = 2 * c.lane + h;
                        if (q < c.S) {
                            const float4 v = *trec(c, kk, q);
                            Soft r;
                            r.m = v.x;
                            r.s = v.y;
                            r.s1 = 0.f;
                            lt = soft_pair_merge(lt, r, k);
                            r.m = v.z;
                            r.s = v.w;
                            ld = soft_pair_merge(ld, r, k);
                        }
                    }
                    const Soft Ct = soft_warp_allreduce<false>(lt, k), Cd = soft_warp_allreduce<false>(ld, k);
                    if (!(Ct.m > -INFINITY) || !(Ct.s > 0.f) || !(Ct.s < INFINITY) || !(Cd.m > -INFINITY) ||
                        !(Cd.s > 0.f) || !(Cd.s < INFINITY))
                        flags |= F_NONFINITE;
                    const float ct = fmaf(Ct.m, k, log2f(Ct.s)), cd = fmaf(Cd.m, k, log2f(Cd.s));
                    if (c.lane == 0) {
                        c.ws->ct[kk] = ct;
                        c.ws->cd[kk] = cd;
                    }
                    float acc_a = 0.f, acc_s = 0.f;
                    unsigned char *bk = c.bits + static_cast<size_t>(kk) * nvs;
                    for (int ch = 0; ch < c.nch; ++ch) {
                        tproduce<Tin, TOPK>(A, c);
                        if (!twait_slot(c)) break;
                        const unsigned char *tb = c.ring + c.cslot * SLOT_BYTES;
                        const unsigned char *db = tb + CV * 16;
                        const int cnt = tchunk(c, ch);
                        uint4 rt[QV], rd[QV];
                        if (cnt == CV) {
                            load_chunk<Tin, true, QV>(tb, cnt, c.lane, rt);
                            load_chunk<Tin, true, QV>(db, cnt, c.lane, rd);
                        } else {
                            load_chunk<Tin, false, QV>(tb, cnt, c.lane, rt);
                            load_chunk<Tin, false, QV>(db, cnt, c.lane, rd);
                        }
                        // hand the slot back once every loaded register is consumed
                        const uint32_t x = consume_regs<QV>(rt) ^ consume_regs<QV>(rd);
                        asm volatile("" ::"r"(x));
                        __syncwarp();
                        tconsumed(c);
                        tproduce<Tin, TOPK>(A, c);
                        uint32_t m[QV];
                        ovl_regs<Tin, QV>(rt, rd, k, ct, cd, acc_a, acc_s, m);
#pragma unroll
                        for (int q = 0; q < QV; ++q) {
                            const int j = q * 32 + c.lane;
                            if (j < cnt) bk[ch * CV + j] = static_cast<unsigned char>(m[q]);
                        }
                    }
                    if (c.dead) break;
                    tpush(sh, c, g + kk, make_float4(warp_allsum(acc_a), warp_allsum(acc_s), 0.f, 0.f));
                }
            }
            // ---- the chain: every warp from the gathered records
            if (!c.dead) {
                float av[MAXG], sv[MAXG];
#pragma unroll
                for (int kk = 0; kk < MAXG; ++kk) {
                    av[kk] = 0.f;
                    sv[kk] = 0.f;
                    if (kk < g) {
                        if (!twait_round(sh, c, g + kk)) break;
                        float a0 = 0.f, s0 = 0.f;
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int q = 2 * c.lane + h;
                            if (q < c.S) {
                                const float4 v = *trec(c, g + kk, q);
                                a0 += v.x;
                                s0 += v.y;
                            }
                        }
                        av[kk] = warp_allsum(a0);
                        sv[kk] = warp_allsum(s0);
                    }
                }
                if (!c.dead && !flags) {
                    float P[MAXG];
                    float prod = 1.f, ls = 0.f;
                    const bool clamped = A.loss_kind == 1;
#pragma unroll
                    for (int kk = 0; kk < MAXG; ++kk) {
                        if (kk < g) {
                            prod *= av[kk];
                            P[kk] = prod;
                            // e2e: -sum of the prefix products; clamped: sum of clamp(1 - alpha, 0, tau_max)
                            ls += clamped ? fminf(fmaxf(1.f - av[kk], 0.f), A.tau_max) : -prod;
                        }
                    }
                    float W = 1.f;
#pragma unroll
                    for (int kk = MAXG - 1; kk >= 0; --kk) {
                        if (kk < g) {
                            const float Pprev = kk ? P[kk - 1] : 1.f;
                            const float d = 1.f - av[kk];
                            const float dl = clamped ? ((d > 0.f && d < A.tau_max) ? -1.f : 0.f) : -Pprev * W;
                            const float coef = A.grad_scale * dl / T;
                            if (c.lane == 0) {
                                c.ws->on[kk] = coef * (1.f - sv[kk]);
                                c.ws->off[kk] = -coef * sv[kk];
                            }
                            W = fmaf(av[kk], W, 1.f);
                        }
                    }
                    loss = ls;
#pragma unroll
                    for (int kk = 0; kk < MAXG; ++kk)
                        if (kk < g && c.lane == kk) alpha_l = av[kk];
                }
            }
            if (c.dead) flags |= F_TIMEOUT;
            __syncwarp();
            // ---- G(k): the gradient, latest step first (the order of unit_of)
            for (int kk = g - 1; kk >= 0; --kk) {
                float *orow = grow + static_cast<size_t>(kk) * A.V;
                const float cd = c.ws->cd[kk], on = c.ws->on[kk], off = c.ws->off[kk];
                const unsigned char *bk = c.bits + static_cast<size_t>(kk) * nvs;
                for (int ch = 0; ch < c.nch; ++ch) {
                    tproduce<Tin, TOPK>(A, c);
                    if (!twait_slot(c)) break;
                    const unsigned char *db = c.ring + c.cslot * SLOT_BYTES + CV * 16;
                    const int cnt = tchunk(c, ch);
                    uint4 rd[QV];
                    load_chunk<Tin, false, QV>(db, cnt, c.lane, rd);
                    const uint32_t x = consume_regs<QV>(rd);
                    asm volatile("" ::"r"(x));
                    __syncwarp();
                    tconsumed(c);
                    tproduce<Tin, TOPK>(A, c);
#pragma unroll
                    for (int q = 0; q < QV; ++q) {
                        const int j = q * 32 + c.lane;
                        if (j < cnt) {
                            float *out = orow + (static_cast<size_t>(c.seg_lo) + ch * CV + j) * VEC;
                            if (flags) {
                                __stcs(reinterpret_cast<float4 *>(out), make_float4(0.f, 0.f, 0.f, 0.f));
                                if (VEC == 8) __stcs(reinterpret_cast<float4 *>(out) + 1, make_float4(0.f, 0.f, 0.f, 0.f));
                            } else {
                                // two 16-byte stores: measured slightly faster here than one 32-byte store
                                grad_vec<Tin, false>(rd[q], TOPK ? 0u : bk[ch * CV + j], k, cd, on, off, out);
                            }
                        }
                    }
                }
                if (c.dead) break;
                if (TOPK && !flags) {
                    // the cached entries of this segment: 1[q <= p~] where it holds
                    __syncwarp();  // the segment's streamed values are visible to every lane
                    const size_t kb = (static_cast<size_t>(t) * g + kk) * static_cast<size_t>(A.K);
                    const unsigned char *vals =
                        reinterpret_cast<const unsigned char *>(A.target) + kb * St::ES;
                    const int32_t *ids = A.topk_idx + kb;
                    const unsigned char *drow = tv_row_ptr<Tin>(A.draft, t, kk, g, A.V);
                    const float ct = c.ws->ct[kk];
                    const int v_lo = c.seg_lo * VEC, v_hi = (c.seg_lo + c.seg_n) * VEC;
                    for (int e = c.lane; e < A.K; e += 32) {
                        const int v = __ldg(ids + e);
                        if (v < v_lo || v >= v_hi) continue;
                        const float lp = fmaf(St::scalar_g(vals, e), k, -ct);
                        const float lq = fmaf(St::scalar_g(drow, v), k, -cd);
                        orow[v] = ex2(lq) * (lq <= lp ? on : off);
                    }
                }
            }
            if (c.dead) {
                flags |= F_TIMEOUT;
                for (int kk = 0; kk < g; ++kk) zero_segment<Tin>(c, grow + static_cast<size_t>(kk) * A.V);
            }
            // warp 0 closes the bank: every round of this position complete, re-armed
            if (c.warp == 0 && !c.dead) {
                for (int i = 0; i < c.Q; ++i) {
                    if (!twait_round(sh, c, i)) break;
                    if (c.lane == 0) mbar_arrive_expect_tx(smem_addr(&sh.xbar[c.bank][i]), static_cast<uint32_t>(c.S) * 16u);
                }
                __syncwarp();
            }
            c.bpar ^= 1u << c.bank;
            c.bank ^= 1;
        }
        if (c.sg == 0) {
            const bool err = flags != 0;
            if (c.lane == 0) {
                A.loss[t] = err ? NAN : loss;
                if (A.flags) A.flags[t] = flags;
            }
            if (A.alpha && c.lane < g) A.alpha[static_cast<size_t>(t) * g + c.lane] = err ? NAN : alpha_l;
        }
    }

    tdrain(c);
    __syncthreads();
    cluster_sync();  // no CTA leaves while a peer may still push into it
}

}  // namespace

uint32_t tvs_hdr_bytes() { return HDR_BYTES; }
uint32_t tvs_rec_bytes(int gamma, int S) { return trec_bytes(gamma, S); }
uint32_t tvs_bits_bytes(int gamma, int nvs) { return tbits_bytes(gamma, nvs); }
int tvs_threads() { return NT; }
int tvs_max_gamma() { return MAXG; }
int tvs_max_segments() { return MAXS; }

const void *tvs_kernel(int dtype, int cv, bool topk) {
#define MTP_TVS_PICK(T, K)                                                                        \
    return cv == 192   ? reinterpret_cast<const void *>(&tvs_kernel_impl<T, 192, K>)              \
           : cv == 160 ? reinterpret_cast<const void *>(&tvs_kernel_impl<T, 160, K>)              \
                       : reinterpret_cast<const void *>(&tvs_kernel_impl<T, 128, K>);
    if (topk) {
        if (dtype == 0) {
            MTP_TVS_PICK(float, true)
        }
        MTP_TVS_PICK(bf16_t, true)
    }
    if (dtype == 0) {
        MTP_TVS_PICK(float, false)
    }
    MTP_TVS_PICK(bf16_t, false)
#undef MTP_TVS_PICK
}

}  // namespace mtp
