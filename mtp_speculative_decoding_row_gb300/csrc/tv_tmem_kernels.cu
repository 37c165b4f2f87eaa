// tv_tmem_kernels.cu -- fused forward and backward of the end-to-end TV loss
// with the draft rows of a position parked in tensor memory (sm_103a)
// ("Breaking Entropy Bounds: Accelerating RL Training via MTP with Rejection
// Sampling", §4 "End-to-end TV loss", App. A, App. F "Fused TV Loss Kernel":
// the backward pass reuses the quantities the forward pass cached).
//
// For token position t with draft steps k = 0..gamma-1, p_k = softmax(z_t/T),
// q_k = softmax(z_d/T):
//     alpha_k = sum_v min(p_v, q_v),   S_k = sum_v 1[q_v <= p_v] q_v,
//     l_t = -sum_k P_k,  P_k = prod_{i<=k} alpha_i,
//     dl_t/dalpha_k = -P_{k-1} W_k,  W_k = 1 + alpha_{k+1} W_{k+1}, W_last = 1,
//     grad[t,k,j] = grad_scale (dl_t/dalpha_k) (1/T) q_j (1[q_j <= p_j] - S_k).
//
// Every logit is read from HBM once.  A kernel that allocates TMEM runs one
// CTA per SM, so the 16 warps of a CTA form TEAMS independent teams; team
// i of the C CTAs of a cluster handles one position at a time, and the
// teams of an SM work on different positions, so one team's exchange waits
// are covered by the other's work.  The vocabulary is cut into S = C x (16 /
// TEAMS) contiguous segments of whole 16-byte vectors, one per warp of the
// team, and each warp streams its segments through a private ring of
// bulk-copy slots, one row segment per slot, in a fixed order per position:
//   N(k): target row k and draft row k from HBM: softmax partials, one
//     16-byte record per warp to every CTA (DSMEM push); the draft segment
//     is parked in the warp's TMEM columns as it streams;
//   O(k), one step behind N: target row k once more (read a few
//     microseconds earlier, so from L2) and draft row k from TMEM, with the
//     final normalisers: alpha and S partials and one indicator byte per
//     vector kept in shared memory; one record per warp;
//   G(k), after the chain: draft row k from TMEM and the indicator bytes:
//     the gradient, written with streaming stores.
// Keeping the drafts in TMEM takes the gradient pass off HBM and L2
// altogether, and the only re-read (the target in O) follows its first read
// closely, so the rows in flight between the two stay far below the L2
// size.  The planner picks C so that a warp's gamma draft segments fit its
// 128 of the SM's 512 TMEM columns.  All waits are bounded; the ring runs
// ahead into the next position while a position's exchanges, overlap and
// gradient passes complete, so HBM reads continue through them.
#include <cstddef>

#include "chunk_math.cuh"
#include "common.cuh"
#include "kernels.h"
#include "tmem.cuh"

namespace mtp {
namespace {

constexpr int NT = 512;          // threads per CTA (one CTA per SM: it holds all TMEM columns)
constexpr int NW = NT / 32;      // warps per CTA; four per TMEM lane quarter
constexpr int TEAMS = 1;         // independent warp teams per CTA, each on its own position
constexpr int TW = NW / TEAMS;   // warps (segments) per team and CTA
constexpr int MAXC = 8;          // largest cluster
constexpr int MAXS = MAXC * TW;  // segments per team and cluster
constexpr int MAXG = 8;          // largest gamma
constexpr int QMAX = 2 * MAXG;   // exchange rounds per position
constexpr int MAXR = 8;          // ring slots per warp
constexpr int WCOLS = TMEM_COLS / (NW / 4);  // TMEM columns of one warp

struct MWarp {
    unsigned long long full[MAXR];  // ring slot barriers
    float cd[MAXG];                 // draft log2 normaliser of each step
    float on[MAXG], off[MAXG];      // gradient coefficients of each step
};

// Fixed header; the exchange records ([TEAMS][2][2 gamma][S] float4), the
// indicator bytes ([NW][gamma][NS * 32]) and the rings ([NW][R][NS * 32]
// vectors) follow.
struct MShared {
    // [team][bank][round]: N rounds 0..gamma-1, O rounds gamma..2 gamma-1
    unsigned long long xbar[TEAMS][2][QMAX];
    uint32_t tmem_base;
    MWarp w[NW];
};
constexpr uint32_t HDR_BYTES = (sizeof(MShared) + 127u) & ~127u;

__host__ __device__ constexpr uint32_t mrec_bytes(int gamma, int S) {
    return ((2u * static_cast<uint32_t>(2 * gamma) * static_cast<uint32_t>(S) * 16u) + 127u) & ~127u;
}
__host__ __device__ constexpr uint32_t mbits_bytes(int gamma, int ns) {
    return ((static_cast<uint32_t>(NW) * static_cast<uint32_t>(gamma) * static_cast<uint32_t>(ns) * 32u) + 127u) &
           ~127u;
}
// A ring slot holds one row segment: NS x 32 vectors.
__host__ __device__ constexpr uint32_t mslot_bytes(int ns) { return static_cast<uint32_t>(ns) * 32u * 16u; }

// Vectors a lane handles at once: its NS vectors of a row segment are taken
// in NS / GS groups, so that a group of two rows fits in registers.
__host__ __device__ constexpr int group_size(int ns) { return ns % 5 == 0 ? 5 : ns % 4 == 0 ? 4 : ns; }

template <int NS>
struct Group {
    static constexpr int GS = group_size(NS);
    static constexpr int NG = NS / GS;
};

struct MC {
    int C, rank, warp, lane, team, tw, sg, S, NT_, vc, R, g, Q;  // vc: the team's place among NT_ teams
    int seg_lo, seg_n;  // this warp's vectors
    unsigned char *ring;
    unsigned char *bits;  // this warp's indicator bytes [gamma][NS * 32]
    MWarp *ws;
    float4 *rec;
    uint32_t tbase;  // TMEM address of this warp's lane quarter and columns
    uint64_t wait_ns;  // limit of every wait
    // producer
    uint32_t pcount, pslot;
    int p_ord, p_r;  // next copy: position ordinal, unit (munit)
    bool p_done;
    // consumer
    uint32_t ccount, cslot, cphase;
    bool dead;
    int bank;
    uint32_t bpar;
};

enum { U_NT = 0, U_ND = 1, U_OT = 2 };

// Copy u (0 <= u < 3 gamma) of a position: N(0) (target, draft), then N(k)
// and the target re-read of O(k - 1) in turn, then O(gamma - 1).
__device__ __forceinline__ void munit(int u, int g, int &kind, int &k) {
    if (u < 2) {
        kind = u;
        k = 0;
    } else if (u == 3 * g - 1) {
        kind = U_OT;
        k = g - 1;
    } else {
        const int j = u - 2;
        k = 1 + j / 3;
        kind = j % 3;
        if (kind == U_OT) k -= 1;
    }
}

template <typename Tin>
__device__ __forceinline__ const unsigned char *mrow_ptr(const TVArgs &A, int t, int kind, int k, int g) {
    const size_t V = static_cast<size_t>(A.V);
    const unsigned char *base;
    size_t row;
    if (kind == U_ND) {
        base = reinterpret_cast<const unsigned char *>(A.draft);
        row = static_cast<size_t>(t) * g + k;
    } else {
        base = reinterpret_cast<const unsigned char *>(A.target);
        row = A.shared_target ? static_cast<size_t>(t) + k : static_cast<size_t>(t) * g + k;
    }
    return base + row * V * Store<Tin>::ES;
}

// Issue row-segment copies while ring slots are free, in the order of
// munit, then the team's next position.
template <typename Tin, int NS>
__device__ __forceinline__ void mproduce(const TVArgs &A, MC &c) {
    if (c.p_done || c.dead) return;
    while (c.pcount - c.ccount < static_cast<uint32_t>(c.R)) {
        const int t = c.vc + c.p_ord * c.NT_;
        if (c.lane == 0) {
            int kind, k;
            munit(c.p_r, c.g, kind, k);
            // no proxy fence: the slot's generic reads completed (their values
            // were consumed) before the consumer released it
            const uint32_t bar = smem_addr(&c.ws->full[c.pslot]);
            const uint32_t dst = smem_addr(c.ring + c.pslot * mslot_bytes(NS));
            const uint32_t bytes = static_cast<uint32_t>(c.seg_n) * 16u;
            mbar_arrive_expect_tx_relaxed(bar, bytes);
            bulk_g2s(dst, mrow_ptr<Tin>(A, t, kind, k, c.g) + static_cast<size_t>(c.seg_lo) * 16u, bytes, bar);
        }
        ++c.pcount;
        if (++c.pslot == static_cast<uint32_t>(c.R)) c.pslot = 0;
        if (++c.p_r == 3 * c.g) {
            c.p_r = 0;
            ++c.p_ord;
            if (c.vc + c.p_ord * c.NT_ >= A.N) {
                c.p_done = true;
                return;
            }
        }
    }
}

__device__ __forceinline__ void mconsumed(MC &c) {
    ++c.ccount;
    if (++c.cslot == static_cast<uint32_t>(c.R)) {
        c.cslot = 0;
        c.cphase ^= 1u;
    }
}

__device__ __forceinline__ float4 *mrec(const MC &c, int i, int q) {
    return c.rec + (static_cast<size_t>(c.bank * c.Q + i) * c.S + q);
}

__device__ __forceinline__ void mpush(MShared &sh, const MC &c, int i, float4 v) {
    if (c.lane < c.C) {
        const uint32_t rbar = map_rank(smem_addr(&sh.xbar[c.team][c.bank][i]), c.lane);
        const uint32_t ra = map_rank(smem_addr(mrec(c, i, c.sg)), c.lane);
        st_async_v4(ra, v.x, v.y, v.z, v.w, rbar);
    }
}

// Bounded wait with one verdict for the whole warp (the tcgen05 accesses
// that follow are warp-wide: no lane may take another path).
__device__ __forceinline__ bool mwait_warp(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    return __all_sync(FULL, mbar_wait_sleep(bar, parity, limit_ns) ? 1 : 0) != 0;
}

__device__ __forceinline__ bool mwait_round(MShared &sh, MC &c, int i) {
    if (c.dead) return false;
    if (!mwait_warp(smem_addr(&sh.xbar[c.team][c.bank][i]), (c.bpar >> c.bank) & 1u, c.wait_ns)) c.dead = true;
    return !c.dead;
}

// TMEM column of vector slot s of parked draft row k (within this warp's
// columns).
template <int NS>
__device__ __forceinline__ uint32_t mcol(int k, int s) {
    return static_cast<uint32_t>((k * NS + s) * 4);
}

// Wait for the ring slot of the next copy; false (and the warp dead) when the
// bounded wait gave up.
template <typename Tin, int NS>
__device__ __forceinline__ bool mslot_ready(const TVArgs &A, MC &c) {
    mproduce<Tin, NS>(A, c);
    if (c.pcount == c.ccount || !mwait_warp(smem_addr(&c.ws->full[c.cslot]), c.cphase, c.wait_ns)) {
        c.dead = true;
        return false;
    }
    return true;
}

// Group gi of this lane's vectors, from the current ring slot.  A slot's
// vectors past the segment (all of them for a warp without vectors) hold
// -inf logits: mfill_tails writes them once, and the copies never reach
// them.
template <typename Tin, int NS>
__device__ __forceinline__ void mload_group(const MC &c, int gi, uint4 (&v)[Group<NS>::GS]) {
    constexpr int GS = Group<NS>::GS;
    const unsigned char *buf = c.ring + c.cslot * mslot_bytes(NS);
#pragma unroll
    for (int q = 0; q < GS; ++q) v[q] = vec_at(buf, (gi * GS + q) * 32 + c.lane);
}

// Fill every ring slot's vectors past this warp's segment with -inf logits
// (probability 0 in every pass), so that loading a group needs no bound
// test.  Generic-proxy stores to bytes no bulk copy writes.
template <typename Tin, int NS>
__device__ __forceinline__ void mfill_tails(const MC &c) {
    const uint4 NEG = make_uint4(NegInf<Tin>::w, NegInf<Tin>::w, NegInf<Tin>::w, NegInf<Tin>::w);
    for (int s = 0; s < c.R; ++s) {
        uint4 *slot = reinterpret_cast<uint4 *>(c.ring + s * mslot_bytes(NS));
        for (int j = max(c.seg_n, 0) + c.lane; j < NS * 32; j += 32) slot[j] = NEG;
    }
    __syncwarp();
}

// Hand the current ring slot back (every value read from it is consumed).
template <typename Tin, int NS>
__device__ __forceinline__ void mrelease(const TVArgs &A, MC &c) {
    __syncwarp();
    mconsumed(c);
    mproduce<Tin, NS>(A, c);
}

// N pass of one row: this lane's softmax partial (m, s) over its vectors of
// the row; a draft row (PARK) is also parked in TMEM as row k.
template <typename Tin, int NS, bool PARK>
__device__ __forceinline__ void mnorm_row(const TVArgs &A, MC &c, int k, float kk2, float &m, float &s, int &bad) {
    constexpr int GS = Group<NS>::GS, NG = Group<NS>::NG;
    m = -INFINITY;
    s = 0.f;
    const bool have = c.seg_n > 0;
    if (have && !mslot_ready<Tin, NS>(A, c)) return;
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
        uint4 v[GS];
        mload_group<Tin, NS>(c, gi, v);
        // the maximum consumes every loaded register: after the last group
        // the slot's reads are complete and it is handed back
        const float cmx = chunk_max<Tin, GS>(v);
        if (have && gi == NG - 1) mrelease<Tin, NS>(A, c);
        if (PARK) {
#pragma unroll
            for (int q = 0; q < GS; ++q) tmem_st_v4(c.tbase + mcol<NS>(k, gi * GS + q), v[q]);
        }
        fold_regs<Tin, GS>(v, cmx, kk2, m, s, bad);
    }
    if (PARK) tmem_wait_st();
}

// Zero this warp's segment of one gradient row (flagged positions).
template <typename Tin>
__device__ __forceinline__ void mzero_segment(const MC &c, float *row) {
    constexpr int VEC = Store<Tin>::VEC;
    float4 *o = reinterpret_cast<float4 *>(row + static_cast<size_t>(c.seg_lo) * VEC);
    const int n4 = c.seg_n * VEC / 4;
    for (int i = c.lane; i < n4; i += 32) __stcs(o + i, make_float4(0.f, 0.f, 0.f, 0.f));
}

// G(k) of position t: the gradient row k of this warp's segment from the
// parked draft row k and the indicator bytes (a flagged position: zeros).
// The warp's cd, on and off of step k and the bytes belong to position t.
template <typename Tin, int NS>
__device__ __forceinline__ void mgrad_row(const TVArgs &A, const MC &c, int t, int kk, int pflags, float k) {
    constexpr int VEC = Store<Tin>::VEC;
    constexpr int GS = Group<NS>::GS, NG = Group<NS>::NG;
    float *orow = A.grad + (static_cast<size_t>(t) * c.g + kk) * static_cast<size_t>(A.V);
    if (pflags) {
        mzero_segment<Tin>(c, orow);
        return;
    }
    const float cd = c.ws->cd[kk], on = c.ws->on[kk], off = c.ws->off[kk];
    const unsigned char *bk = c.bits + static_cast<size_t>(kk) * NS * 32;
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
        uint4 rd[GS];
#pragma unroll
        for (int q = 0; q < GS; ++q) tmem_ld_v4(c.tbase + mcol<NS>(kk, gi * GS + q), rd[q]);
        tmem_wait_ld_regs<GS>(rd);
#pragma unroll
        for (int q = 0; q < GS; ++q) {
            const int j = (gi * GS + q) * 32 + c.lane;
            if (j < c.seg_n) {
                float *out = orow + (static_cast<size_t>(c.seg_lo) + j) * VEC;
                if (A.grad32)
                    grad_vec<Tin, true>(rd[q], bk[j], k, cd, on, off, out);
                else
                    grad_vec<Tin, false>(rd[q], bk[j], k, cd, on, off, out);
            }
        }
    }
}

template <typename Tin, int NS>
__global__ void __launch_bounds__(NT, 1) tvm_kernel_impl(const TVArgs A) {
    using St = Store<Tin>;
    constexpr int VEC = St::VEC;
    extern __shared__ __align__(128) unsigned char smem[];
    MShared &sh = *reinterpret_cast<MShared *>(smem);

    MC c;
    c.C = static_cast<int>(cluster_size());
    c.rank = static_cast<int>(cluster_rank());
    c.warp = threadIdx.x >> 5;
    c.lane = threadIdx.x & 31;
    c.team = c.warp / TW;
    c.tw = c.warp % TW;
    // team `team` of cluster `cid` handles positions vc, vc + NT_, ...
    c.NT_ = static_cast<int>(gridDim.x) / c.C * TEAMS;
    c.vc = static_cast<int>(cluster_id_x()) * TEAMS + c.team;
    c.S = c.C * TW;
    c.sg = c.rank * TW + c.tw;
    c.R = A.ring;
    c.g = A.gamma;
    c.Q = 2 * A.gamma;
    const int g = c.g;
    const int nv = A.V / VEC;
    const int nvs = A.seg_vectors;
    c.seg_lo = min(nv, c.sg * nvs);
    c.seg_n = min(nv, c.seg_lo + nvs) - c.seg_lo;
    c.ws = &sh.w[c.warp];
    c.rec = reinterpret_cast<float4 *>(smem + HDR_BYTES + static_cast<size_t>(c.team) * mrec_bytes(g, c.S));
    c.bits = smem + HDR_BYTES + TEAMS * mrec_bytes(g, c.S) + static_cast<size_t>(c.warp) * g * NS * 32;
    c.ring = smem + HDR_BYTES + TEAMS * mrec_bytes(g, c.S) + mbits_bytes(g, NS) +
             static_cast<size_t>(c.warp) * c.R * mslot_bytes(NS);
    const float T = A.temperature;
    const bool bad_temp = !(T > 0.f) || !(T < INFINITY);
    const float k = LOG2E / T;
    c.pcount = c.ccount = 0;
    c.pslot = c.cslot = c.cphase = 0;
    c.p_ord = c.p_r = 0;
    c.p_done = bad_temp || c.seg_n <= 0 || c.vc >= A.N;
    c.dead = false;
    c.bank = 0;
    c.bpar = 0;
    c.wait_ns = A.wait_ns ? A.wait_ns : 2000000000ull;

    if (c.warp == 0) tmem_alloc(&sh.tmem_base, TMEM_COLS);
    mfill_tails<Tin, NS>(c);
    if (c.lane == 0)
        for (int s = 0; s < c.R; ++s) mbar_init(smem_addr(&c.ws->full[s]), 1);
    if (threadIdx.x == 0) {
        for (int tm = 0; tm < TEAMS; ++tm)
            for (int bk = 0; bk < 2; ++bk)
                for (int i = 0; i < c.Q; ++i) mbar_init(smem_addr(&sh.xbar[tm][bk][i]), 1);
        fence_mbar_init();
        for (int tm = 0; tm < TEAMS; ++tm)
            for (int bk = 0; bk < 2; ++bk)
                for (int i = 0; i < c.Q; ++i)
                    mbar_arrive_expect_tx(smem_addr(&sh.xbar[tm][bk][i]), static_cast<uint32_t>(c.S) * 16u);
    }
    fence_mbar_init();
    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    // lane quarter of this warp, and its share of the quarter's columns
    c.tbase = tmem_addr(sh.tmem_base, static_cast<uint32_t>((c.warp & 3) * 32),
                        static_cast<uint32_t>((c.warp >> 2) * WCOLS));
    cluster_sync();  // every barrier of the cluster is initialised and armed before any push
    mproduce<Tin, NS>(A, c);

    // The gradient pass of a position runs interleaved with the next
    // position's first passes: G(k) of the previous position right before
    // N(k) of this one, which parks its draft row k in the columns G(k) has
    // just read.  So the stores of one position overlap the loads and
    // arithmetic of the next instead of every warp storing at once.
    int prev_t = -1, prev_flags = 0, prev_done = 0;  // pending G: position, its flags, rows done
    // The next position's target row 0 is folded before this position's
    // chain waits for the overlap records, so that its streaming covers the
    // wait for the cluster's slowest warp (the ring's copy order is the same).
    bool pre_nt = false;  // the fold below already holds target row 0 of position t
    float pre_mt = -INFINITY, pre_st = 0.f;
    int pre_bad = 0;
    for (int t = c.vc; t < A.N; t += c.NT_) {
        float *grow = A.grad + static_cast<size_t>(t) * g * static_cast<size_t>(A.V);
        int flags = 0;
        float loss = NAN;
        float alpha_l = NAN;  // lane kk < g: alpha_kk
        if (bad_temp || c.dead) {
            for (; prev_t >= 0 && prev_done < g; ++prev_done) mgrad_row<Tin, NS>(A, c, prev_t, prev_done, prev_flags, k);
            prev_t = -1;
            flags = bad_temp ? F_BAD_TEMP : F_TIMEOUT;
            for (int kk = 0; kk < g; ++kk) mzero_segment<Tin>(c, grow + static_cast<size_t>(kk) * A.V);
        } else {
            // ---- N(k), and O(k - 1) right after it: the all-gather of N(k - 1)
            // had the streaming of N(k) to complete
            for (int u = 0; u <= g && !c.dead; ++u) {
                if (u < g && prev_t >= 0) {
                    mgrad_row<Tin, NS>(A, c, prev_t, u, prev_flags, k);
                    prev_done = u + 1;
                }
                if (u < g) {
                    float mt, st, md, sd;
                    int bad = 0;
                    if (u == 0 && pre_nt) {
                        mt = pre_mt;
                        st = pre_st;
                        bad = pre_bad;
                    } else {
                        mnorm_row<Tin, NS, false>(A, c, u, k, mt, st, bad);
                    }
                    pre_nt = false;
                    if (c.dead) break;
                    mnorm_row<Tin, NS, true>(A, c, u, k, md, sd, bad);
                    if (c.dead) break;
                    Soft a;
                    a.m = mt;
                    a.s = st;
                    a.s1 = 0.f;
                    const Soft wt = soft_warp_allreduce<false>(a, k);
                    a.m = md;
                    a.s = sd;
                    const Soft wd = soft_warp_allreduce<false>(a, k);
                    const bool wbad = warp_allor(bad) != 0;
                    // fault injection (tests): the cluster's first warp leaves out one record
                    if (!(t == A.skip_t && u == 0 && c.sg == 0))
                        mpush(sh, c, u, make_float4(wt.m, wbad ? NAN : wt.s, wd.m, wbad ? NAN : wd.s));
                }
                if (u == 0) continue;
                // ---- O(kk): the final normalisers, then the parked pair
                const int kk = u - 1;
                if (!mwait_round(sh, c, kk)) break;
                // the cluster's normalisers from the S warp records: the maxima
                // first, then every record's sum rescaled once (a NaN sum, a
                // flagged row, propagates; an empty record adds nothing)
                float4 rv[MAXS / 32];
                float mtl = -INFINITY, mdl = -INFINITY;
#pragma unroll
                for (int h = 0; h < MAXS / 32; ++h) {
                    const int q = (MAXS / 32) * c.lane + h;
                    rv[h] = q < c.S ? *mrec(c, kk, q) : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
                    mtl = fmaxf(mtl, rv[h].x);
                    mdl = fmaxf(mdl, rv[h].z);
                }
                Soft Ct, Cd;
                Ct.m = warp_allmax(mtl);
                Cd.m = warp_allmax(mdl);
                float stl = 0.f, sdl = 0.f;
#pragma unroll
                for (int h = 0; h < MAXS / 32; ++h) {
                    if (rv[h].y != 0.f) stl = fmaf(rv[h].y, ex2((rv[h].x - Ct.m) * k), stl);
                    if (rv[h].w != 0.f) sdl = fmaf(rv[h].w, ex2((rv[h].z - Cd.m) * k), sdl);
                }
                Ct.s = warp_allsum(stl);
                Cd.s = warp_allsum(sdl);
                Ct.s1 = Cd.s1 = 0.f;
                if (!(Ct.m > -INFINITY) || !(Ct.s > 0.f) || !(Ct.s < INFINITY) || !(Cd.m > -INFINITY) ||
                    !(Cd.s > 0.f) || !(Cd.s < INFINITY))
                    flags |= F_NONFINITE;
                const float ct = fmaf(Ct.m, k, log2f(Ct.s)), cd = fmaf(Cd.m, k, log2f(Cd.s));
                if (c.lane == 0) c.ws->cd[kk] = cd;
                // the target row again (from L2) and the parked draft row
                const bool have = c.seg_n > 0;
                if (have && !mslot_ready<Tin, NS>(A, c)) break;
                float acc_a = 0.f, acc_s = 0.f;
                unsigned char *bk = c.bits + static_cast<size_t>(kk) * NS * 32;
                constexpr int GS = Group<NS>::GS, NG = Group<NS>::NG;
#pragma unroll
                for (int gi = 0; gi < NG; ++gi) {
                    uint4 rt[GS], rd[GS];
#pragma unroll
                    for (int q = 0; q < GS; ++q) tmem_ld_v4(c.tbase + mcol<NS>(kk, gi * GS + q), rd[q]);
                    mload_group<Tin, NS>(c, gi, rt);
                    tmem_wait_ld_regs<GS>(rd);
                    if (have && gi == NG - 1) {
                        // consume the slot's values before handing it back
                        const uint32_t x = consume_regs<GS>(rt);
                        asm volatile("" ::"r"(x));
                        mrelease<Tin, NS>(A, c);
                    }
                    uint32_t mb[GS];
                    ovl_regs<Tin, GS>(rt, rd, k, ct, cd, acc_a, acc_s, mb);
#pragma unroll
                    for (int q = 0; q < GS; ++q) bk[(gi * GS + q) * 32 + c.lane] = static_cast<unsigned char>(mb[q]);
                }
                mpush(sh, c, g + kk, make_float4(warp_allsum(acc_a), warp_allsum(acc_s), 0.f, 0.f));
            }
            // rows of the previous position still pending (the loop above
            // stopped early): before the chain overwrites their coefficients
            for (; prev_t >= 0 && prev_done < g; ++prev_done) mgrad_row<Tin, NS>(A, c, prev_t, prev_done, prev_flags, k);
            // the next position's target row 0, while the overlap records arrive
            if (!c.dead && t + c.NT_ < A.N) {
                pre_bad = 0;
                mnorm_row<Tin, NS, false>(A, c, 0, k, pre_mt, pre_st, pre_bad);
                pre_nt = !c.dead;
            }
            // ---- the chain: every warp from the gathered records
            if (!c.dead) {
                float av[MAXG], sv[MAXG];
#pragma unroll
                for (int kk = 0; kk < MAXG; ++kk) {
                    av[kk] = 0.f;
                    sv[kk] = 0.f;
                    if (kk < g) {
                        if (!mwait_round(sh, c, g + kk)) break;
                        float a0 = 0.f, s0 = 0.f;
#pragma unroll
                        for (int h = 0; h < MAXS / 32; ++h) {
                            const int q = (MAXS / 32) * c.lane + h;
                            if (q < c.S) {
                                const float4 v = *mrec(c, g + kk, q);
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
            // ---- G(k) of this position: with the next position's N passes
            prev_t = t;
            prev_flags = flags;
            prev_done = 0;
            // the team's warp 0 closes the bank: every round of this position
            // complete, re-armed
            if (c.tw == 0 && !c.dead) {
                for (int i = 0; i < c.Q; ++i) {
                    if (!mwait_round(sh, c, i)) break;
                    if (c.lane == 0)
                        mbar_arrive_expect_tx(smem_addr(&sh.xbar[c.team][c.bank][i]),
                                              static_cast<uint32_t>(c.S) * 16u);
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

    for (; prev_t >= 0 && prev_done < g; ++prev_done) mgrad_row<Tin, NS>(A, c, prev_t, prev_done, prev_flags, k);
    // copies still in flight (after a bounded wait gave up, or issued ahead
    // past a dead position) land before the CTA leaves
    while (c.ccount != c.pcount) {
        (void)mbar_wait_sleep(smem_addr(&c.ws->full[c.cslot]), c.cphase, c.wait_ns);
        mconsumed(c);
    }
    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    if (c.warp == 0) tmem_dealloc(sh.tmem_base, TMEM_COLS);
    cluster_sync();  // no CTA leaves while a peer may still push into it
}

}  // namespace

uint32_t tvm_smem_bytes(int gamma, int C, int ns, int ring) {
    return HDR_BYTES + TEAMS * mrec_bytes(gamma, C * TW) + mbits_bytes(gamma, ns) +
           static_cast<uint32_t>(NW * ring) * mslot_bytes(ns);
}
int tvm_team_warps() { return TW; }
int tvm_teams() { return TEAMS; }
int tvm_threads() { return NT; }
int tvm_max_gamma() { return MAXG; }
int tvm_max_ring() { return MAXR; }
int tvm_warp_cols() { return WCOLS; }
int tvm_max_cluster() { return MAXC; }

const void *tvm_kernel(int dtype, int ns) {
#define MTP_TVM_PICK(T)                                                                     \
    switch (ns) {                                                                           \
        case 2: return reinterpret_cast<const void *>(&tvm_kernel_impl<T, 2>);              \
        case 4: return reinterpret_cast<const void *>(&tvm_kernel_impl<T, 4>);              \
        case 5: return reinterpret_cast<const void *>(&tvm_kernel_impl<T, 5>);              \
        case 8: return reinterpret_cast<const void *>(&tvm_kernel_impl<T, 8>);              \
        case 10: return reinterpret_cast<const void *>(&tvm_kernel_impl<T, 10>);            \
        default: return nullptr;                                                            \
    }
    if (dtype == 0) {
        MTP_TVM_PICK(float)
    }
    MTP_TVM_PICK(bf16_t)
#undef MTP_TVM_PICK
}

}  // namespace mtp
