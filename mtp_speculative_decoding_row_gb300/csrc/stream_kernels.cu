// stream_kernels.cu -- batched MTP rejection-sampling verification (no
// statistics) as a streaming kernel on sm_103a.
//
// Method ("Breaking Entropy Bounds: Accelerating RL Training via MTP with
// Rejection Sampling", §2 "Acceptance methods" and App. G.1; "EntMTP",
// Related Work "Speculative Decoding"): with p_i = softmax(z_t[i] / T) and
// q_i = softmax(z_d[i] / T), draft y_i is accepted iff u_i q_i(y_i) <
// p_i(y_i); checking stops at the first rejection j, whose replacement is
// drawn from norm(max(0, p_j - q_j)) by inverse CDF with u_gamma; after
// gamma accepts the bonus token is drawn from p_gamma the same way.
//
// Layout of the work.  A persistent cluster of C CTAs x NW warps verifies
// one sequence at a time (sequences cid, cid + NC, ...).  The vocabulary is
// cut into S = C * NW contiguous segments of whole 16-byte vectors, one per
// warp, and every warp works on its own segment only:
//   - it streams its segment of each needed row through a private ring of
//     R chunk slots (CV vectors of the target row + CV of the draft row per
//     slot), filled by cp.async.bulk on one mbarrier per slot; lane 0 is the
//     producer, the whole warp the consumer, and there is no CTA-wide barrier
//     on the streaming path;
//   - per position it folds each chunk into per-lane online softmax partials
//     (exact running maximum, so no overflow path), reduces them across the
//     warp and pushes a 16-byte record (plus the logits at the draft token,
//     from the warp whose segment holds it) to every CTA of the cluster with
//     st.async onto that position's exchange mbarrier;
//   - it runs up to `depth` positions ahead of the last decided one, so the
//     all-gather of one position overlaps the streaming of the next; every
//     warp gathers the S records of a position and takes the accept decision
//     itself (same records, same reduction order: the same verdict
//     everywhere).  A rejection drops the look-ahead.
// Sampling: after a rejection every warp re-streams its segment of rows j
// (now mostly in L2) to form per-chunk residual sums, the segment totals are
// all-gathered, and the warp owning the selected segment walks its chunk sums
// and then the elements of one chunk (fetched again from global memory).
// For the bonus token the per-chunk (max, sum) records taken while streaming
// row gamma give the chunk weights directly, so row gamma is read only once.
//
// Exchange slots: each sequence uses gamma + 2 rounds (one per position and
// one for the residual totals) in one of two banks, alternating by sequence.
// Every warp pushes into every round of its sequence (a zero record where a
// position was not needed), so every slot completes one phase per use; warp
// 0 waits for all of them and re-arms the bank before it pushes anything for
// the next sequence, and a bank is reused two sequences later, after every
// warp has read it.
#include <cstddef>

#include "chunk_math.cuh"
#include "common.cuh"
#include "philox.cuh"
#include "kernels.h"
#include "gsample.h"

namespace mtp {
namespace {

constexpr int NT = 128;          // threads per CTA
constexpr int NW = NT / 32;      // warps (segments) per CTA
// Chunk geometry is a template parameter of the kernel: CV vectors of each
// row per ring slot (128, 160 or 192: 2, 2.5 or 3 KB), CV / 32 per lane.
constexpr int MAXCH = 64;        // chunks per segment
constexpr int MAXS = 64;         // segments per cluster (C * NW)
constexpr int MAXG = 8;          // largest gamma
constexpr int QMAX = MAXG + 2;   // exchange rounds per sequence
constexpr int MAXR = 8;          // ring slots per warp

enum { K_NORM = 0, K_RES = 1 };

struct WarpShared {
    unsigned long long full[MAXR];  // ring slot barriers
    float cm[MAXCH];                // per-chunk maxima (bonus records)
    float cs[MAXCH];                // per-chunk sums
};

// Fixed header; the exchange records follow it, then the warps' rings.
struct StreamShared {
    unsigned long long xbar[2][QMAX];
    WarpShared w[NW];
};
constexpr uint32_t HDR_BYTES = (sizeof(StreamShared) + 127u) & ~127u;

// Exchange records: two float4 per warp per round (a main and an auxiliary
// record, [2][gamma + 2][2 S] float4), so every round carries the same bytes
// whatever the sequence's mode.
__host__ __device__ constexpr uint32_t rec_bytes(int gamma, int S) {
    return ((2u * static_cast<uint32_t>(gamma + 2) * static_cast<uint32_t>(2 * S) * 16u) + 127u) & ~127u;
}

// rejection sampling with an inverse-CDF final draw / target-only acceptance /
// rejection sampling with a Gumbel-max final draw
enum { M_RS = 0, M_TO = 1, M_GB = 2 };

constexpr int ERR_BITS = F_NONFINITE | F_BAD_ID | F_BAD_TEMP | F_BAD_UNIFORM | F_TIMEOUT;

// Per-warp state (warp-uniform).
struct Ctx {
    // geometry
    int C, rank, warp, lane, sg, S, NC, cid, R, depth, g, Q;
    int cv;       // vectors of each row per chunk
    int seg_lo;   // first vector of the segment
    int seg_n;    // vectors in the segment
    int nch;      // chunks in the segment
    unsigned char *ring;
    WarpShared *ws;
    float4 *rec;  // exchange records
    // producer cursor: next chunk to issue
    uint32_t pcount, pslot;
    int p_ord, p_i, p_kind, p_c;
    bool p_done;
    const unsigned char *p_t, *p_d;  // segment start of the unit's rows (p_d null: target only)
    // consumer
    uint32_t ccount, cslot, cphase;
    int c_ord, c_conf;  // consumer's sequence (order in the cluster list) and highest needed position
    bool dead;
    int bank;           // exchange bank of the current sequence
    uint32_t bpar;      // bit b: phase parity of bank b's current use
};

__device__ __forceinline__ int seq_of(const Ctx &c, int ord) { return c.cid + ord * c.NC; }

// What the sampling helpers need of a warp's segment (passed by value).
struct Seg {
    WarpShared *ws;
    int seg_lo, seg_n, nch, cv;
};

__device__ __forceinline__ Seg seg_of(const Ctx &c) { return {c.ws, c.seg_lo, c.seg_n, c.nch, c.cv}; }

// Point the producer at the first row of the sequence after `ord`.
__device__ __forceinline__ void redirect_next(Ctx &c, int ord, int B) {
    c.p_ord = ord + 1;
    c.p_i = 0;
    c.p_kind = K_NORM;
    c.p_c = 0;
    c.p_done = c.dead || c.nch == 0 || seq_of(c, ord + 1) >= B;
}

template <typename Tin>
__device__ __forceinline__ const unsigned char *row_base(const VerifyArgs &A, bool target, int b, int i) {
    const size_t row = target ? static_cast<size_t>(b) * (A.gamma + 1) + i : static_cast<size_t>(b) * A.gamma + i;
    return reinterpret_cast<const unsigned char *>(target ? A.target : A.draft) +
           row * static_cast<size_t>(A.V) * Store<Tin>::ES;
}

__device__ __forceinline__ int chunk_count(const Ctx &c, int ch) { return min(c.cv, c.seg_n - ch * c.cv); }
__device__ __forceinline__ int chunk_count(const Seg &c, int ch) { return min(c.cv, c.seg_n - ch * c.cv); }

// ------------------------------------------------------------ producer ----

// Enter the producer's next unit: apply the look-ahead rule (positions up
// to c_conf + depth of the consumer's sequence; a later sequence only once
// the current one's path is fixed) and set the unit's row pointers.  False
// when the producer has to wait or has no work left.
template <typename Tin, int MODE>
__device__ __forceinline__ bool enter_unit(const VerifyArgs &A, Ctx &c) {
    const int g = c.g;
    if (c.p_kind == K_NORM) {
        if (c.p_i > g) {  // end of the sequence's rows
            if (c.p_ord == c.c_ord && c.c_conf < g) return false;
            c.p_ord += 1;
            c.p_i = 0;
            if (seq_of(c, c.p_ord) >= A.B) {
                c.p_done = true;
                return false;
            }
        }
        const int lim = (c.p_ord == c.c_ord) ? c.c_conf + c.depth : c.depth;
        if (c.p_i > lim) return false;
    }
    const int b = seq_of(c, c.p_ord);
    const size_t off = static_cast<size_t>(c.seg_lo) * 16u;
    c.p_t = row_base<Tin>(A, true, b, c.p_i) + off;
    // target-only residual passes need the target row alone
    const bool want_d = c.p_i < g && !(MODE == M_TO && c.p_kind == K_RES);
    c.p_d = want_d ? row_base<Tin>(A, false, b, c.p_i) + off : nullptr;
    return true;
}

// Issue chunk copies while ring slots are free and the next chunk is needed
// or inside the look-ahead.  With DBL (one-row sequences: draft sampling), a
// target-only row of the main pass fills both halves of a slot with two
// consecutive chunks, so each slot carries a full slot's bytes.
template <typename Tin, int MODE, bool DBL>
__device__ __forceinline__ void produce(const VerifyArgs &A, Ctx &c) {
    if (c.p_done || c.dead) return;
    while (c.pcount - c.ccount < static_cast<uint32_t>(c.R)) {
        if (c.p_c == 0 && !enter_unit<Tin, MODE>(A, c)) break;
        const int cnt = chunk_count(c, c.p_c);
        const bool dbl = DBL && !c.p_d && c.p_kind == K_NORM;
        const int cnt2 = (dbl && c.p_c + 1 < c.nch) ? chunk_count(c, c.p_c + 1) : 0;
        if (c.lane == 0) {
            // No proxy fence: every generic read of this slot has completed
            // (its value was consumed) before the consumer released it.
            const uint32_t bar = smem_addr(&c.ws->full[c.pslot]);
            const uint32_t dst = smem_addr(c.ring + c.pslot * (2u * c.cv * 16u));
            const uint32_t bytes = static_cast<uint32_t>(cnt) * 16u;
            const uint32_t bytes2 = c.p_d ? bytes : static_cast<uint32_t>(cnt2) * 16u;
            const size_t off = static_cast<size_t>(c.p_c) * (c.cv * 16);
            mbar_arrive_expect_tx_relaxed(bar, bytes + bytes2);
            bulk_g2s(dst, c.p_t + off, bytes, bar);
            if (c.p_d) bulk_g2s(dst + c.cv * 16, c.p_d + off, bytes, bar);
            else if (bytes2) bulk_g2s(dst + c.cv * 16, c.p_t + off + c.cv * 16, bytes2, bar);
        }
        ++c.pcount;
        if (++c.pslot == static_cast<uint32_t>(c.R)) c.pslot = 0;
        c.p_c += dbl ? 2 : 1;
        if (c.p_c >= c.nch) {
            c.p_c = 0;
            if (c.p_kind == K_NORM) {
                c.p_i += 1;  // p_i == g + 1 marks the end of the rows
            } else {
                c.p_kind = K_NORM;
                c.p_i = c.g + 1;  // residual pass done: the sequence's path is fixed
            }
        }
    }
}

// Wait for the next ring slot; false (and dead) on timeout.
__device__ __forceinline__ bool slot_wait(Ctx &c) {
    if (!mbar_wait_spin(smem_addr(&c.ws->full[c.cslot]), c.cphase)) {
        c.dead = true;
        return false;
    }
    return true;
}

__device__ __forceinline__ void consumed(Ctx &c) {
    ++c.ccount;
    if (++c.cslot == static_cast<uint32_t>(c.R)) {
        c.cslot = 0;
        c.cphase ^= 1u;
    }
}

// Drop every issued chunk that has not been consumed (waits for each copy).
__device__ __forceinline__ void drain(Ctx &c) {
    while (c.ccount != c.pcount) {
        if (!mbar_wait_spin(smem_addr(&c.ws->full[c.cslot]), c.cphase)) c.dead = true;
        consumed(c);
    }
}

// ------------------------------------------------------------ exchange ----

// Record r of round i in `bank`: main records at r = segment, auxiliary
// records at r = S + segment.
__device__ __forceinline__ float4 *rec_at(const Ctx &c, int bank, int i, int r) {
    return c.rec + (static_cast<size_t>(bank * c.Q + i) * (2 * c.S) + r);
}

// Bytes every CTA receives in one round: two records per warp.
__device__ __forceinline__ uint32_t round_bytes(const Ctx &c) { return static_cast<uint32_t>(2 * c.S) * 16u; }

// Push this warp's main and auxiliary records for round i of the current
// bank into every CTA of the cluster.
__device__ __forceinline__ void xpush(StreamShared &sh, const Ctx &c, int i, float4 v, float4 aux) {
    if (c.lane < c.C) {
        const uint32_t rbar = map_rank(smem_addr(&sh.xbar[c.bank][i]), c.lane);
        const uint32_t ra = map_rank(smem_addr(rec_at(c, c.bank, i, c.sg)), c.lane);
        const uint32_t xa = map_rank(smem_addr(rec_at(c, c.bank, i, c.S + c.sg)), c.lane);
        st_async_v4(ra, v.x, v.y, v.z, v.w, rbar);
        st_async_v4(xa, aux.x, aux.y, aux.z, aux.w, rbar);
    }
}

// Blocking (bounded) wait for round i of the current bank.
__device__ __forceinline__ bool xwait(StreamShared &sh, Ctx &c, int i) {
    if (!mbar_wait_spin(smem_addr(&sh.xbar[c.bank][i]), (c.bpar >> c.bank) & 1u)) c.dead = true;
    return !c.dead;
}

// Non-blocking test of round i of the current bank.
__device__ __forceinline__ bool xtest(StreamShared &sh, const Ctx &c, int i) {
    return mbar_test_wait(smem_addr(&sh.xbar[c.bank][i]), (c.bpar >> c.bank) & 1u);
}

// ------------------------------------------------------------ sampling ----

// Inverse CDF over the S segment totals held two per lane (segments 2l and
// 2l + 1 in lane l, zero beyond S): the first segment whose running sum
// exceeds u * R, in ascending order; if rounding leaves none, the last
// segment with positive weight (and `last` is set so the walk below takes
// the last positive element).  Returns -1 if R == 0.
__device__ __forceinline__ int pick_segment(float t0, float t1, float u, float &rem, int &last) {
    const int lane = threadIdx.x & 31;
    const float tl = t0 + t1;
    const float inc = warp_incl_scan(tl);
    const float R = __shfl_sync(FULL, inc, 31);
    last = 0;
    rem = 0.f;
    if (!(R > 0.f)) return -1;
    const float x = u * R;
    const unsigned bal = __ballot_sync(FULL, inc > x);
    if (bal) {
        const int L = __ffs(bal) - 1;
        const float excl = __shfl_sync(FULL, inc - tl, L);
        const float a0 = __shfl_sync(FULL, t0, L);
        const float r = x - excl;
        if (a0 > r) {
            rem = r;
            return 2 * L;
        }
        rem = r - a0;
        return 2 * L + 1;
    }
    last = 1;
    const unsigned pos = __ballot_sync(FULL, tl > 0.f);
    const int L = 31 - __clz(pos);
    const float a1 = __shfl_sync(FULL, t1, L);
    (void)lane;
    return a1 > 0.f ? 2 * L + 1 : 2 * L;
}

// Weights of one vector: residual max(0, p - q) (RES) or p relative to the
// row maximum (otherwise).  p = 2^{z_t k - ct}, q = 2^{z_d k - cd}.
template <typename Tin, bool RES>
__device__ __forceinline__ void vweights(const uint4 &rt, const uint4 &rd, float k, float ct, float cd,
                                         float (&w)[Store<Tin>::VEC]) {
    constexpr int VEC = Store<Tin>::VEC;
    float zt[VEC];
    Store<Tin>::unpack(rt, zt);
    if (RES) {
        float zd[VEC];
        Store<Tin>::unpack(rd, zd);
#pragma unroll
        for (int e = 0; e < VEC; ++e) w[e] = fmaxf(ex2(fmaf(zt[e], k, -ct)) - ex2(fmaf(zd[e], k, -cd)), 0.f);
    } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) w[e] = ex2(fmaf(zt[e], k, -ct));
    }
}

// Walk inside the owning warp: chunk sums (cs[c] * 2^{(cm[c] - ref) k} when
// `scaled`), then the elements of the selected chunk fetched from global
// memory, in ascending index order (chunk, 32-vector round, lane, element).
// `rem` is the remaining mass inside this segment.  Falls back to the last
// positive weight of the selected unit when rounding leaves no index.
template <typename Tin, bool RES, int QV>
__device__ __noinline__ int walk_segment(const Seg c, const unsigned char *trow, const unsigned char *drow,
                                         bool scaled, float ref, float k, float ct, float cd, float rem, int last,
                                         int excl) {
    constexpr int VEC = Store<Tin>::VEC;
    const int lane = threadIdx.x & 31;
    // chunk selection
    int ch = -1;
    if (!last) {
        for (int base = 0; base < c.nch && ch < 0; base += 32) {
            const int q = base + lane;
            float w = 0.f;
            if (q < c.nch) w = scaled ? c.ws->cs[q] * ex2((c.ws->cm[q] - ref) * k) : c.ws->cs[q];
            if (scaled && !(w == w)) w = 0.f;
            const float inc = warp_incl_scan(w);
            const float tot = __shfl_sync(FULL, inc, 31);
            if (tot > rem) {
                const unsigned bal = __ballot_sync(FULL, inc > rem);
                const int L = __ffs(bal) - 1;
                rem -= __shfl_sync(FULL, inc - w, L);
                ch = base + L;
            } else {
                rem -= tot;
            }
        }
    }
    if (ch < 0) {
        last = 1;
        for (int base = 0; base < c.nch; base += 32) {
            const int q = base + lane;
            float w = 0.f;
            if (q < c.nch) w = scaled ? c.ws->cs[q] * ex2((c.ws->cm[q] - ref) * k) : c.ws->cs[q];
            const unsigned pos = __ballot_sync(FULL, w > 0.f);
            if (pos) ch = base + 31 - __clz(pos);
        }
        if (ch < 0) return -1;
    }
    // element walk inside chunk ch
    const int cnt = chunk_count(c, ch);
    const size_t v0 = static_cast<size_t>(c.seg_lo) + static_cast<size_t>(ch) * c.cv;
    const uint4 *gt = reinterpret_cast<const uint4 *>(trow) + v0;
    const uint4 *gd = RES ? reinterpret_cast<const uint4 *>(drow) + v0 : gt;
    float w[QV][VEC];
#pragma unroll
    for (int r = 0; r < QV; ++r) {
        const int j = r * 32 + lane;
        if (j < cnt) {
            const uint4 rt = __ldg(gt + j);
            const uint4 rd = RES ? __ldg(gd + j) : rt;
            vweights<Tin, RES>(rt, rd, k, ct, cd, w[r]);
            if (excl >= 0 && static_cast<size_t>(excl / VEC) == v0 + j) w[r][excl % VEC] = 0.f;
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) w[r][e] = 0.f;
        }
    }
    if (!last) {
#pragma unroll
        for (int r = 0; r < QV; ++r) {
            float vs = w[r][0];
#pragma unroll
            for (int e = 1; e < VEC; ++e) vs += w[r][e];
            const float inc = warp_incl_scan(vs);
            const float tot = __shfl_sync(FULL, inc, 31);
            if (tot > rem) {
                const unsigned bal = __ballot_sync(FULL, inc > rem);
                const int L = __ffs(bal) - 1;
                const float excl = __shfl_sync(FULL, inc - vs, L);
                int tk = -1;
                if (lane == L) {
                    float r2 = rem - excl;
                    int ef = -1;
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        if (ef < 0) {
                            if (w[r][e] > r2) ef = e;
                            else r2 -= w[r][e];
                        }
                    }
                    if (ef < 0) {
#pragma unroll
                        for (int e = 0; e < VEC; ++e)
                            if (w[r][e] > 0.f) ef = e;
                    }
                    tk = static_cast<int>((v0 + r * 32 + L) * VEC) + ef;
                }
                return __shfl_sync(FULL, tk, L);
            }
            rem -= tot;
        }
    }
    // last positive element of the chunk
    int best = -1;
#pragma unroll
    for (int r = 0; r < QV; ++r)
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            if (w[r][e] > 0.f) best = max(best, static_cast<int>((v0 + r * 32 + lane) * VEC) + e);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) best = max(best, __shfl_xor_sync(FULL, best, o));
    return best;
}

// Per-chunk sums of p (relative to `ref`) of this warp's segment of `trow`,
// read straight from global memory (used when the residual mass rounds to 0).
template <typename Tin>
__device__ __noinline__ void direct_chunk_sums(const Seg c, const unsigned char *trow, float k, float ref) {
    constexpr int VEC = Store<Tin>::VEC;
    const int lane = threadIdx.x & 31;
    for (int ch = 0; ch < c.nch; ++ch) {
        const int cnt = chunk_count(c, ch);
        const uint4 *gt = reinterpret_cast<const uint4 *>(trow) + c.seg_lo + static_cast<size_t>(ch) * c.cv;
        float s = 0.f;
        for (int j = lane; j < cnt; j += 32) {
            float w[VEC];
            vweights<Tin, false>(__ldg(gt + j), __ldg(gt + j), k, ref * k, 0.f, w);
#pragma unroll
            for (int e = 0; e < VEC; ++e) s += w[e];
        }
        s = warp_allsum(s);
        if (lane == 0) {
            c.ws->cs[ch] = s;
            c.ws->cm[ch] = ref;
        }
    }
    __syncwarp();
}

// ------------------------------------------------------------ chunk math --

// This lane's residual mass sum max(0, p - q) over one chunk (registers;
// -inf padding contributes 0).
template <typename Tin, int QV>
__device__ __forceinline__ float res_regs(const uint4 (&rt)[QV], const uint4 (&rd)[QV], float k, float ct,
                                          float cd) {
    constexpr int VEC = Store<Tin>::VEC;
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int q = 0; q < QV; ++q) {
        float w[VEC];
        vweights<Tin, true>(rt[q], rd[q], k, ct, cd, w);
#pragma unroll
        for (int e = 0; e < VEC; e += 2) {
            ps0 += w[e];
            ps1 += w[e + 1];
        }
    }
    return ps0 + ps1;
}

// ----------------------------------------------------------------- kernel --

// One position's round, gathered: log2 normalisers (log2 p = z k - ct),
// target maximum, flags, and this lane's two target segment records
// (segments 2 lane and 2 lane + 1).  Rejection sampling: the logits at the
// draft token (Zty, Zdy).  Target-only: the draft arg max yhat and the target
// logit at it (Zty).
struct Norm {
    float ct, cd, Mt, Zty, Zdy;
    int yhat;
    int rf;
    float m0, s0, m1, s1;
};

template <int MODE>
__device__ __forceinline__ Norm gather_norm(const Ctx &c, int i, float k, bool has_d) {
    Norm r;
    r.m0 = r.m1 = -INFINITY;
    r.s0 = r.s1 = 0.f;
    r.yhat = -1;
    float dm = -INFINITY, ds = 0.f;
    float zt_l = 0.f, zd_l = 0.f;
    int hy = 0;
    float av = -INFINITY, ax = 0.f;  // target-only: draft arg max and target logit there
    int ai = -1;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int q = 2 * c.lane + h;
        if (q < c.S) {
            const float4 v = *rec_at(c, c.bank, i, q);
            const float4 x = *rec_at(c, c.bank, i, c.S + q);
            if (h == 0) {
                r.m0 = v.x;
                r.s0 = v.y;
            } else {
                r.m1 = v.x;
                r.s1 = v.y;
            }
            if (MODE != M_TO) {
                if (v.w != 0.f) {  // draft partial of this lane (NaN propagates)
                    if (v.z > dm) {
                        ds = (ds != 0.f ? ds * ex2((dm - v.z) * k) : 0.f) + v.w;
                        dm = v.z;
                    } else {
                        ds += v.w * ex2((v.z - dm) * k);
                    }
                }
                if (x.z != 0.f) {
                    hy = 1;
                    zt_l = x.x;
                    zd_l = x.y;
                }
            } else {
                argmax_merge(av, ai, ax, v.z, __float_as_int(x.x), v.w);
            }
        }
    }
    Soft lt;
    lt.m = fmaxf(r.m0, r.m1);
    lt.s = 0.f;
    lt.s1 = 0.f;
    if (lt.m > -INFINITY) {
        if (r.s0 != 0.f) lt.s += r.s0 * ex2((r.m0 - lt.m) * k);
        if (r.s1 != 0.f) lt.s += r.s1 * ex2((r.m1 - lt.m) * k);
    } else if (r.s0 != 0.f || r.s1 != 0.f) {
        lt.s = NAN;  // a flagged segment with no finite maximum
    }
    const Soft Ct = soft_warp_allreduce<false>(lt, k);
    r.rf = 0;
    if (!(Ct.m > -INFINITY) || !(Ct.s > 0.f) || !(Ct.s < INFINITY)) r.rf |= F_NONFINITE;
    r.Mt = Ct.m;
    r.ct = fmaf(Ct.m, k, log2f(Ct.s));
    r.cd = 0.f;
    r.Zty = r.Zdy = 0.f;
    if (has_d) {
        if (MODE != M_TO) {
            Soft ld;
            ld.m = dm;
            ld.s = ds;
            ld.s1 = 0.f;
            const Soft Cd = soft_warp_allreduce<false>(ld, k);
            if (!(Cd.m > -INFINITY) || !(Cd.s > 0.f) || !(Cd.s < INFINITY)) r.rf |= F_NONFINITE;
            r.cd = fmaf(Cd.m, k, log2f(Cd.s));
            const unsigned hm = __ballot_sync(FULL, hy != 0);
            const int src = hm ? (__ffs(hm) - 1) : 0;
            r.Zty = __shfl_sync(FULL, zt_l, src);
            r.Zdy = __shfl_sync(FULL, zd_l, src);
        } else {
            argmax_allreduce(av, ai, ax);
            if (ai < 0) r.rf |= F_NONFINITE;  // an all -inf draft row
            r.yhat = ai;
            r.Zty = ax;
        }
    }
    return r;
}

// Greedy round (T = 0): target arg max and, target-only, the draft arg max.
struct Greedy {
    int tidx, didx, bad;
};

__device__ __forceinline__ Greedy gather_greedy(const Ctx &c, int i) {
    float tv = -INFINITY, dv = -INFINITY, dummy = 0.f;
    int ti = -1, di = -1, bad = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int q = 2 * c.lane + h;
        if (q < c.S) {
            const float4 v = *rec_at(c, c.bank, i, q);
            const float4 x = *rec_at(c, c.bank, i, c.S + q);
            argmax_merge(tv, ti, dummy, v.x, __float_as_int(v.y), 0.f);
            argmax_merge(dv, di, dummy, v.z, __float_as_int(v.w), 0.f);
            bad |= x.x != 0.f;
        }
    }
    argmax_allreduce(tv, ti, dummy);
    argmax_allreduce(dv, di, dummy);
    Greedy r;
    r.tidx = ti;
    r.didx = di;
    r.bad = __any_sync(FULL, bad) ? 1 : 0;
    return r;
}

// Element e of a 16-byte logit vector set to -inf (probability 0).
template <typename Tin>
__device__ __forceinline__ void vec_set_neginf(uint4 &v, int e) {
    if (Store<Tin>::ES == 4) {
        const uint32_t w = 0xff800000u;
        if (e == 0) v.x = w;
        else if (e == 1) v.y = w;
        else if (e == 2) v.z = w;
        else v.w = w;
    } else {
        const int wi = e >> 1;
        const uint32_t mask = (e & 1) ? 0xffff0000u : 0x0000ffffu, val = (e & 1) ? 0xff800000u : 0x0000ff80u;
        uint32_t *p = wi == 0 ? &v.x : wi == 1 ? &v.y : wi == 2 ? &v.z : &v.w;
        *p = (*p & ~mask) | val;
    }
}

// This lane's sum of p = 2^{z k - ct} over one chunk of the target row.
template <typename Tin, int QV>
__device__ __forceinline__ float psum_regs(const uint4 (&rt)[QV], float k, float ct) {
    constexpr int VEC = Store<Tin>::VEC;
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int q = 0; q < QV; ++q) {
        float w[VEC];
        vweights<Tin, false>(rt[q], rt[q], k, ct, 0.f, w);
#pragma unroll
        for (int e = 0; e < VEC; e += 2) {
            s0 += w[e];
            s1 += w[e + 1];
        }
    }
    return s0 + s1;
}

// Bounds of the Gumbel term g = -log2(-log2 U) (log2 units) over the
// generator's U in [2^-25, 1 - 2^-25]: g <= 24.47 and g >= -log2(25) =
// -4.64, widened for the approximate logarithms.
constexpr float GUMBEL2_MAX = 25.5f;
constexpr float GUMBEL2_MIN = -6.f;
// Keys (log2 units) within this gap of the best are near-ties: the single
// precision keys (approximate logarithms, noise within 4e-5) may order them
// wrongly, so the two best candidates of a draw are re-keyed in double
// precision whenever their gap is below it.  The filters below keep every
// index that can come within the gap of the best key.
constexpr float GUMBEL_TIE = 1e-3f;

// Gumbel noise of index v in row j of sequence b in double precision,
// G = -ln(-ln U), U = (floor(x / 2^8) + 1/2) 2^-24 from word v mod 4 of
// Philox4x32-10 at counter (v / 4, j, b, offset).
__device__ __forceinline__ double gumbel_noise_d(int v, int j, uint32_t b, uint32_t offset, uint32_t seed_lo,
                                                 uint32_t seed_hi) {
    const uint4 x = philox4x32_10(make_uint4(static_cast<uint32_t>(v / 4), static_cast<uint32_t>(j), b, offset), seed_lo,
                                  seed_hi);
    const uint32_t w = (v & 3) == 0 ? x.x : (v & 3) == 1 ? x.y : (v & 3) == 2 ? x.z : x.w;
    const double u = (static_cast<double>(w >> 8) + 0.5) * 5.9604644775390625e-8;
    return -log(-log(u));
}

// Gumbel-max keys of one chunk (registers; vbase: vector index of the lane's
// first vector) into the lane's running arg maxes, first index among equals,
// and the lane's runner-up keys kp2 and kr2 (the best key other than the
// arg max's; its index is recovered by warp_top2 only on a near-tie):
// p keys z_v k + g_v into (kp, ip) and, with RESID, residual keys
// log2(p_v - q_v) + g_v over the v with p_v > q_v into (kr, ir) (p =
// 2^{z_t k - ct}, q = 2^{z_d k - cd}; g_v the noise of index v in row j of
// sequence b).  Two exact filters keep the work to the indices that can
// still win; bp and br are bounds that a winning key must reach (the
// warp's best keys so far; kp and kr themselves at the least):
//   - a group of four indices (one generator call) is skipped when none of
//     them can reach a bound even with the largest noise (for the residual,
//     log2(p - q) <= log2 p = z k - ct);
//   - without RESID (the p keys alone), an index's noise is formed only if
//     its raw word can give enough noise: g >= bp - z k needs L = -log2 U <=
//     2^{z k - bp}, and L >= W / ln 2 with W = 1 - U, so W <= ln 2 2^{mx - bp}
//     (mx: the group's largest z k) is necessary; W is read off the word
//     exactly, and the bound is widened for the approximate exponential.
// kp starts at a lower bound of the row's best p key, so skipped indices
// never hold a draw.
template <typename Tin, int QV, bool RESID>
__device__ __forceinline__ void gumbel_regs(const uint4 (&rt)[QV], const uint4 (&rd)[QV], int cnt, int lane, float k,
                                            float ct, float cd, int vbase, uint32_t seed_lo, uint32_t seed_hi, int j,
                                            uint32_t b, uint32_t offset, float bp, float br, float &kr, int &ir,
                                            float &kr2, float &kp, int &ip, float &kp2) {
    constexpr int VEC = Store<Tin>::VEC;
#pragma unroll
    for (int q = 0; q < QV; ++q) {
        if (q * 32 + lane >= cnt) break;
        const int vv = vbase + q * 32;  // vector index in the row
        float zt[VEC], zd[VEC];
        Store<Tin>::unpack(rt[q], zt);
        if (RESID) Store<Tin>::unpack(rd[q], zd);
#pragma unroll
        for (int h = 0; h < VEC / 4; ++h) {
            float zk[4];
            float mx = -INFINITY;
#pragma unroll
            for (int e4 = 0; e4 < 4; ++e4) {
                zk[e4] = zt[h * 4 + e4] * k;
                mx = fmaxf(mx, zk[e4]);
            }
            // a key must come within GUMBEL_TIE of the best to matter
            const float bpv = fmaxf(kp, bp) - GUMBEL_TIE, brv = fmaxf(kr, br) - GUMBEL_TIE;
            const bool want_p = mx + GUMBEL2_MAX >= bpv;
            const bool want_r = RESID && mx - ct + GUMBEL2_MAX >= brv;
            if (!want_p && !want_r) continue;  // no index of the group can win either draw
            const uint4 x = philox4x32_10(
                make_uint4(static_cast<uint32_t>(vv * (VEC / 4) + h), static_cast<uint32_t>(j), b, offset), seed_lo,
                seed_hi);
            const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
            // largest W = 1 - U (in units of 2^-24) that can still reach the p
            // bound (the bonus draw; a residual pass keeps every index of the
            // group: its bound rises late, and the filter would only cost).
            // W 2^24 >= 2^24 - 1 - floor(x / 2^8), so an index with W 2^24 <=
            // wlim has floor(x / 2^8) >= 2^24 - 1 - wlim: the test is one
            // integer comparison of x against the group's threshold, taken
            // from 2^24 - 2 - wlim rounded down (at most that plus 1/2, a
            // larger kept set: the filter stays exact).  2 <= wlim < 2^54
            // keeps the clamped threshold in [0, 2^24 - 4].
            const float wlim =
                RESID ? INFINITY : fmaf(ex2(fminf(mx - bpv, 30.f)), 0.69314724f * 16777216.f * 1.000002f, 2.f);
            const uint32_t xmin = RESID ? 0u : static_cast<uint32_t>(fmaxf(16777214.f - wlim, 0.f)) << 8;
#pragma unroll
            for (int e4 = 0; e4 < 4; ++e4) {
                if (!RESID && xs[e4] < xmin) continue;  // too little noise to reach the bound
                const int e = h * 4 + e4;
                const float gv = gumbel2(xs[e4]);
                const float key_p = zk[e4] + gv;
                kp2 = fmaxf(kp2, fminf(key_p, kp));  // the runner-up key (its index is found only if needed)
                if (key_p > kp) {
                    kp = key_p;
                    ip = vv * VEC + e;
                }
                if (RESID && want_r) {
                    // both terms in the same form, so equal logits give exactly 0
                    const float w = ex2(fmaf(zt[e], k, -ct)) - ex2(fmaf(zd[e], k, -cd));
                    if (w > 0.f) {
                        const float key_r = __log2f(w) + gv;
                        kr2 = fmaxf(kr2, fminf(key_r, kr));
                        if (key_r > kr) {
                            kr = key_r;
                            ir = vv * VEC + e;
                        }
                    }
                }
            }
        }
    }
}

// The warp's best two Gumbel-max keys of one draw, {K1, I1, K2, I2}, from
// every lane's arg max (k1, i1) and runner-up key k2 (index -1: no
// candidate).  The runner-up is another lane's arg max or, when it is the
// best lane's own runner-up, a key whose index no lane kept; that index is
// found only when it matters, a near-tie (K1 - K2 < GUMBEL_TIE): the warp
// keys the best lane's vectors of the segment once more (vector seg_lo + L +
// 32 t for lane L, with the pass's own arithmetic) and takes their arg max
// other than I1.  Indices the pass skipped have keys below K1 - GUMBEL_TIE,
// so they cannot be that runner-up.  Otherwise the runner-up's index is
// left at -1: it is never needed.  RKEY: residual keys log2(p - q) + g
// (target row trow, draft row drow); else p keys z k + g of trow.  Out of
// line: it runs once per draw, off the streaming path.
constexpr int TOP2_NONE = 0x7fffffff;      // no candidate
constexpr int TOP2_HIDDEN = 0x7ffffffe;    // the best lane's runner-up

template <typename Tin, bool RKEY>
__device__ __noinline__ float4 warp_top2(float k1, int i1, float k2, const unsigned char *trow,
                                         const unsigned char *drow, int seg_lo, int seg_n, int j, uint32_t b, float k,
                                         float ct, float cd, uint32_t seed_lo, uint32_t seed_hi, uint32_t offset) {
    constexpr int VEC = Store<Tin>::VEC;
    const int lane = threadIdx.x & 31;
    // larger key first; at equal keys the smaller index (TOP2_HIDDEN after
    // every index, TOP2_NONE last)
    auto reduce = [](float &key, int &idx) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ok = __shfl_xor_sync(FULL, key, o);
            const int oi = __shfl_xor_sync(FULL, idx, o);
            if (ok > key || (ok == key && oi < idx)) {
                key = ok;
                idx = oi;
            }
        }
    };
    float K1 = k1;
    int I1 = i1 >= 0 ? i1 : TOP2_NONE;
    reduce(K1, I1);
    const unsigned holder = __ballot_sync(FULL, I1 != TOP2_NONE && i1 == I1);
    const int L1 = holder ? __ffs(holder) - 1 : -1;
    float K2 = lane == L1 ? k2 : k1;
    int I2 = lane == L1 ? TOP2_HIDDEN : (i1 >= 0 ? i1 : TOP2_NONE);
    reduce(K2, I2);
    if (I2 == TOP2_HIDDEN && K1 - K2 < GUMBEL_TIE) {  // warp-uniform
        float bk = -INFINITY;
        int bi = TOP2_NONE;
        const uint4 *gt = reinterpret_cast<const uint4 *>(trow) + seg_lo;
        const uint4 *gd = reinterpret_cast<const uint4 *>(drow) + seg_lo;
        for (int t = lane; L1 + 32 * t < seg_n; t += 32) {
            const int jv = L1 + 32 * t, vv = seg_lo + jv;
            float zt[VEC], zd[VEC];
            Store<Tin>::unpack(__ldg(gt + jv), zt);
            if (RKEY) Store<Tin>::unpack(__ldg(gd + jv), zd);
#pragma unroll
            for (int h = 0; h < VEC / 4; ++h) {
                const uint4 x = philox4x32_10(
                    make_uint4(static_cast<uint32_t>(vv * (VEC / 4) + h), static_cast<uint32_t>(j), b, offset),
                    seed_lo, seed_hi);
                const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int e4 = 0; e4 < 4; ++e4) {
                    const int e = h * 4 + e4, idx = vv * VEC + e;
                    const float zk = zt[e] * k, gv = gumbel2(xs[e4]);
                    float key = zk + gv;
                    if (RKEY) {
                        const float w = ex2(fmaf(zt[e], k, -ct)) - ex2(fmaf(zd[e], k, -cd));
                        key = w > 0.f ? __log2f(w) + gv : -INFINITY;
                    }
                    if (idx != I1 && key > -INFINITY && (key > bk || (key == bk && idx < bi))) {
                        bk = key;
                        bi = idx;
                    }
                }
            }
        }
        reduce(bk, bi);
        I2 = bi;
    }
    return make_float4(K1, __int_as_float(I1 == TOP2_NONE ? -1 : I1), K2,
                       __int_as_float(I2 >= TOP2_HIDDEN ? -1 : I2));
}

// The Gumbel-max pass of one warp over its segment [seg_lo, seg_lo + seg_n)
// of row j (target row trow, draft row drow), read directly from global
// memory (the rows were streamed moments ago and mostly sit in L2): the
// warp's two best residual and p keys with their indices (index -1: no
// candidate, or a runner-up far from the best; the p keys start at the
// bound lb).  Out of line and by value: it runs once per sequence, and
// neither its generator state nor the warp's streaming state should crowd
// the other's registers.
struct Top2x2 {
    float4 best;    // {key_r, idx_r, key_p, idx_p}
    float4 second;  // the runners-up, same layout
};

template <typename Tin, bool RESID>
__device__ __noinline__ Top2x2 gumbel_pass(const unsigned char *trow, const unsigned char *drow, int seg_lo,
                                           int seg_n, int j, uint32_t b, float k, float ct, float cd, float lb,
                                           uint32_t seed_lo, uint32_t seed_hi, uint32_t offset) {
    constexpr int QV = 2;  // vectors per lane per tile
    const int lane = threadIdx.x & 31;
    const uint4 *gt = reinterpret_cast<const uint4 *>(trow) + seg_lo;
    const uint4 *gd = reinterpret_cast<const uint4 *>(drow) + seg_lo;
    float kr = -INFINITY, kp = lb, bp = lb, br = -INFINITY, kr2 = -INFINITY, kp2 = -INFINITY;
    int ir = -1, ip = -1;
    // The pass is bound by load latency, not arithmetic: the next tile's
    // loads are in flight while a tile is keyed.
    uint4 rt[QV], rd[QV], nt[QV], nd[QV];
    auto load_tile = [&](int base, uint4 (&t)[QV], uint4 (&d)[QV]) {
#pragma unroll
        for (int q = 0; q < QV; ++q) {
            const int jv = base + q * 32 + lane;
            if (jv < seg_n) {
                t[q] = __ldg(gt + jv);
                if (RESID) d[q] = __ldg(gd + jv);
            }
        }
    };
    load_tile(0, rt, rd);
    for (int base = 0; base < seg_n; base += QV * 32) {
        if (base + QV * 32 < seg_n) load_tile(base + QV * 32, nt, nd);
        gumbel_regs<Tin, QV, RESID>(rt, rd, min(QV * 32, seg_n - base), lane, k, ct, cd, seg_lo + base + lane,
                                    seed_lo, seed_hi, j, b, offset, bp, br, kr, ir, kr2, kp, ip, kp2);
        // the warp's best p key so far bounds every lane's filters
        if (!RESID) bp = warp_allmax(kp);
#pragma unroll
        for (int q = 0; q < QV; ++q) {
            rt[q] = nt[q];
            if (RESID) rd[q] = nd[q];
        }
    }
    const float4 r2 = RESID ? warp_top2<Tin, true>(kr, ir, kr2, trow, drow, seg_lo, seg_n, j, b, k, ct, cd, seed_lo,
                                                   seed_hi, offset)
                            : make_float4(-INFINITY, __int_as_float(-1), -INFINITY, __int_as_float(-1));
    const float4 p2 =
        warp_top2<Tin, false>(kp, ip, kp2, trow, drow, seg_lo, seg_n, j, b, k, ct, cd, seed_lo, seed_hi, offset);
    Top2x2 r;
    r.best = make_float4(r2.x, r2.y, p2.x, p2.y);
    r.second = make_float4(r2.z, r2.w, p2.z, p2.w);
    return r;
}

// Gumbel-max p keys of one chunk of row j held in a ring slot (target
// vectors at tb; cnt vectors; chunk_v0: the chunk's first vector in the row)
// into the lane's running arg max and runner-up key, passed and returned by
// value as {kp, ip, kp2, -}; bp is the warp's best p key so far.  Out of
// line: it runs once per chunk of the bonus draw, and neither its generator
// state nor the warp's streaming state should crowd the other's registers.
template <typename Tin, int CV>
__device__ __noinline__ float4 gumbel_slot(const unsigned char *tb, int cnt, int chunk_v0, float k, int j, uint32_t b,
                                           uint32_t seed_lo, uint32_t seed_hi, uint32_t offset, float bp, float4 top) {
    const int lane = threadIdx.x & 31;
    float kr = -INFINITY, kr2 = -INFINITY, kp = top.x, kp2 = top.z;
    int ir = -1, ip = __float_as_int(top.y);
    for (int q = 0; q < CV / 32 && q * 32 + lane < cnt; ++q) {
        const uint4 v[1] = {vec_at(tb, q * 32 + lane)};
        gumbel_regs<Tin, 1, false>(v, v, 32, lane, k, 0.f, 0.f, chunk_v0 + q * 32 + lane, seed_lo, seed_hi, j, b,
                                   offset, bp, -INFINITY, kr, ir, kr2, kp, ip, kp2);
    }
    return make_float4(kp, __int_as_float(ip), kp2, 0.f);
}

// A near-tie of a Gumbel-max draw: the two best candidates t1 and t2 (fp32
// keys within GUMBEL_TIE) keyed once more in double precision, ln w_v + G_v
// with w the residual weight max(0, p - q) (resid) or p; the larger key wins,
// ties to the smaller index.  Every warp passes the same inputs in the same
// order and so takes the same token.  Out of line: it runs for about one
// draw in a thousand, and its double-precision code should not weigh on the
// kernel's registers.
template <typename Tin>
__device__ __noinline__ int gumbel_retie(const unsigned char *trow, const unsigned char *drow, bool resid, int t1,
                                         int t2, int j, uint32_t b, float k, float ct, float cd, uint32_t seed_lo,
                                         uint32_t seed_hi, uint32_t offset) {
    auto key_d = [&](int v) {
        const double zt = static_cast<double>(Store<Tin>::scalar_g(trow, static_cast<size_t>(v)));
        double w = exp2(zt * static_cast<double>(k) - static_cast<double>(ct));
        if (resid) {
            const double zd = static_cast<double>(Store<Tin>::scalar_g(drow, static_cast<size_t>(v)));
            w -= exp2(zd * static_cast<double>(k) - static_cast<double>(cd));
        }
        return (w > 0.0 ? log(w) : -static_cast<double>(INFINITY)) + gumbel_noise_d(v, j, b, offset, seed_lo, seed_hi);
    };
    const double a1 = key_d(t1), a2 = key_d(t2);
    return (a2 > a1 || (a2 == a1 && t2 < t1)) ? t2 : t1;
}

// The final token of a Gumbel-max draw from the S warps' records of the
// draw's round (rec: S best records, then S runner-up records, each {key_r,
// idx_r, key_p, idx_p}): the best residual key (at a rejection, resid) or
// the best p key, the two best candidates re-keyed by gumbel_retie on a
// near-tie.  Returns {token, flags}: F_ZERO_MASS when every residual weight
// rounded to zero (the p draw stands in).  Every warp reads the same records
// in the same order and so takes the same token.  Out of line: it runs once
// per sequence, after the streaming.
template <typename Tin>
__device__ __noinline__ int2 gumbel_select(const float4 *rec, int S, int lane, bool resid, const unsigned char *trow,
                                           const unsigned char *drow, int j, uint32_t b, float k, float ct, float cd,
                                           uint32_t seed_lo, uint32_t seed_hi, uint32_t offset) {
    float vr = -INFINITY, vp = -INFINITY, d0 = 0.f;
    int jr = -1, jp = -1;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int q = 2 * lane + h;
        if (q < S) {
            const float4 v = rec[q];
            argmax_merge(vr, jr, d0, v.x, __float_as_int(v.y), 0.f);
            argmax_merge(vp, jp, d0, v.z, __float_as_int(v.w), 0.f);
        }
    }
    argmax_allreduce(vr, jr, d0);
    argmax_allreduce(vp, jp, d0);
    int flags = 0;
    if (resid && jr < 0) flags |= F_ZERO_MASS;  // every residual weight rounded to zero
    const bool use_r = resid && jr >= 0;
    int tok = use_r ? jr : jp;
    if (tok < 0) return make_int2(tok, flags);
    // the runner-up: every warp's best other than the winner, and the
    // winning warp's own runner-up; its key first, its index only on a
    // near-tie
    auto cand = [&](int q, float &key, int &idx) {
        const float4 v = rec[q], w = rec[S + q];
        const float kb = use_r ? v.x : v.z, kw = use_r ? w.x : w.z;
        const int ib = __float_as_int(use_r ? v.y : v.w), iw = __float_as_int(use_r ? w.y : w.w);
        key = ib == tok ? kw : kb;
        idx = ib == tok ? iw : ib;
    };
    float k2 = -INFINITY;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int q = 2 * lane + h;
        if (q < S) {
            float key;
            int idx;
            cand(q, key, idx);
            if (idx >= 0) k2 = fmaxf(k2, key);
        }
    }
    k2 = warp_allmax(k2);
    if ((use_r ? vr : vp) - k2 < GUMBEL_TIE) {  // warp-uniform
        float v2 = -INFINITY;
        int t2 = -1;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int q = 2 * lane + h;
            if (q < S) {
                float key;
                int idx;
                cand(q, key, idx);
                argmax_merge(v2, t2, d0, key, idx, 0.f);
            }
        }
        argmax_allreduce(v2, t2, d0);
        if (t2 >= 0) tok = gumbel_retie<Tin>(trow, drow, use_r, tok, t2, j, b, k, ct, cd, seed_lo, seed_hi, offset);
    }
    return make_int2(tok, flags);
}

// Programmatic dependent launch.  The streaming kernel is launched with
// programmatic stream serialization: the next launch on the stream may start
// once every CTA of the running one has signalled (each signals as it
// starts), so its CTAs take SMs as the running grid's CTAs retire and set up
// their shared memory meanwhile.  Before its first global-memory access the
// kernel waits until every prerequisite grid has completed and its writes
// are visible, so the results are those of plain stream order.  (The
// one-pass Gumbel-max kernel below is launched plainly: it is bound by
// arithmetic in a single wave, and CTAs of the next launch placed early on
// whichever SMs free up first made it slower.)
__device__ __forceinline__ void pdl_allow_next() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_prior() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------ Gumbel-max draft sampling ----
//
// mtp_draft_sample with the Gumbel-max method.  Row r's token is arg max_v
// [z_v k + g_v] (k = log2(e) / T_r; g_v the noise of index v in row 0 of
// sequence r), which needs no normaliser, so every row is read once, with
// no ring and no shared-memory staging: a cluster of C CTAs x GS_NW warps
// cuts the row into warp segments read straight from global memory.  Each
// warp keys its segment with the exact filters of gumbel_regs (bounded by
// the warp's best key so far) and also takes the segment's exact maximum
// with its first index (greedy rows, the all -inf check) and whether it holds
// a NaN or +inf.  The warps' records are all-gathered through distributed
// shared memory behind one cluster barrier, and warp 0 of CTA 0 takes the
// token (gumbel_select: the two best candidates re-keyed in double precision
// on a near-tie) and writes the outputs.  Persistent clusters take rows cid,
// cid + NC, ...; the records alternate between two buffers by row, so a
// row's records are overwritten only after the barrier of the row after it,
// which CTA 0 passes once it has read them.
constexpr int GS_NT = 256;
constexpr int GS_NW = GS_NT / 32;
constexpr int GS_MAXC = 8;                 // largest cluster
constexpr int GS_MAXS = GS_MAXC * GS_NW;   // segments per row (gumbel_select: two per lane)

// [row parity][best records (S), runner-up records (S), {max z, its index,
// NaN or +inf seen, -} (S)], S = C * GS_NW used of each GS_MAXS.
struct GsShared {
    float4 rec[2][3 * GS_MAXS];
};

__device__ __forceinline__ void st_cluster_v4(uint32_t raddr, float4 v) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(raddr), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w)
                 : "memory");
}

// One warp's pass over its segment [seg_lo, seg_lo + seg_n) of row r (vector
// seg_lo + L + 32 t for lane L, as warp_top2 expects): the p-key arg max and
// runner-up when sampling, the exact maximum with its first index, and the
// NaN / +inf test.  Tiles of two vectors per lane; the next tile's loads are
// in flight while a tile is keyed.
template <typename Tin>
__device__ __forceinline__ void gsample_pass(const unsigned char *row, int seg_lo, int seg_n, bool sample, float k,
                                             uint32_t r, uint32_t seed_lo, uint32_t seed_hi, uint32_t offset,
                                             float4 &best, float4 &second, float4 &mrec) {
    constexpr int QV = 2;
    constexpr int VEC = Store<Tin>::VEC;
    const int lane = threadIdx.x & 31;
    const uint4 *g = reinterpret_cast<const uint4 *>(row) + seg_lo;
    float kr = -INFINITY, kr2 = -INFINITY, kp = -INFINITY, kp2 = -INFINITY, bp = -INFINITY;
    int ir = -1, ip = -1;
    float mz = -INFINITY;
    int mi = -1, bad = 0;
    uint4 rt[QV], nt[QV];
    auto load_tile = [&](int base, uint4 (&t)[QV]) {
#pragma unroll
        for (int q = 0; q < QV; ++q) {
            const int jv = base + q * 32 + lane;
            if (jv < seg_n) t[q] = __ldg(g + jv);
        }
    };
    load_tile(0, rt);
    for (int base = 0; base < seg_n; base += QV * 32) {
        if (base + QV * 32 < seg_n) load_tile(base + QV * 32, nt);
#pragma unroll
        for (int q = 0; q < QV; ++q) {
            const int jv = base + q * 32 + lane;
            if (jv < seg_n) {
                const float vm = Store<Tin>::vmax(rt[q]);  // NaN if the vector holds one
                if (!(vm < INFINITY)) {
                    bad = 1;
                } else if (vm > mz) {  // first index of the lane's maximum (its vectors ascend)
                    float z[VEC];
                    Store<Tin>::unpack(rt[q], z);
                    int e0 = VEC - 1;
#pragma unroll
                    for (int e = VEC - 1; e >= 0; --e)
                        if (z[e] == vm) e0 = e;
                    mz = vm;
                    mi = (seg_lo + jv) * VEC + e0;
                }
            }
        }
        if (sample) {
            gumbel_regs<Tin, QV, false>(rt, rt, min(QV * 32, seg_n - base), lane, k, 0.f, 0.f, seg_lo + base + lane,
                                        seed_lo, seed_hi, 0, r, offset, bp, -INFINITY, kr, ir, kr2, kp, ip, kp2);
            bp = warp_allmax(kp);  // the warp's best key so far bounds every lane's filters
        }
#pragma unroll
        for (int q = 0; q < QV; ++q) rt[q] = nt[q];
    }
    const float4 t2 = sample ? warp_top2<Tin, false>(kp, ip, kp2, row, nullptr, seg_lo, seg_n, 0, r, k, 0.f, 0.f,
                                                     seed_lo, seed_hi, offset)
                             : make_float4(-INFINITY, __int_as_float(-1), -INFINITY, __int_as_float(-1));
    float dummy = 0.f;
    argmax_allreduce(mz, mi, dummy);
    bad = warp_allor(bad);
    best = make_float4(-INFINITY, __int_as_float(-1), t2.x, t2.y);
    second = make_float4(-INFINITY, __int_as_float(-1), t2.z, t2.w);
    mrec = make_float4(mz, __int_as_float(mi), __int_as_float(bad), 0.f);
}

template <typename Tin>
__global__ void __launch_bounds__(GS_NT, 4) gsample_kernel_impl(const VerifyArgs A) {
    constexpr int VEC = Store<Tin>::VEC;
    extern __shared__ __align__(128) unsigned char smem[];
    GsShared &sh = *reinterpret_cast<GsShared *>(smem);
    const int C = static_cast<int>(cluster_size());
    const int rank = static_cast<int>(cluster_rank());
    const int cid = static_cast<int>(cluster_id_x());
    const int NC = static_cast<int>(gridDim.x) / C;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = C * GS_NW, sg = rank * GS_NW + warp;
    const int nv = A.V / VEC;
    const int nvs = (nv + S - 1) / S;
    const int seg_lo = min(nv, sg * nvs), seg_n = min(nv, seg_lo + nvs) - seg_lo;
    int par = 0;
    for (int r = cid; r < A.B; r += NC) {
        const float T = __ldg(A.temp + r);
        const bool bad_t = !(T >= 0.f) || !(T < INFINITY);
        const bool sample = !bad_t && T != 0.f;
        const float k = sample ? LOG2E / T : 0.f;
        const unsigned char *row =
            reinterpret_cast<const unsigned char *>(A.target) + static_cast<size_t>(r) * A.V * Store<Tin>::ES;
        float4 best = make_float4(-INFINITY, __int_as_float(-1), -INFINITY, __int_as_float(-1)), second = best;
        float4 mrec = make_float4(-INFINITY, __int_as_float(-1), __int_as_float(0), 0.f);
        if (!bad_t)
            gsample_pass<Tin>(row, seg_lo, seg_n, sample, k, static_cast<uint32_t>(r), A.seed_lo, A.seed_hi,
                              A.offset, best, second, mrec);
        // lane q < C stores this warp's three records into CTA q
        if (lane < C) {
            float4 *base = sh.rec[par];
            st_cluster_v4(map_rank(smem_addr(base + sg), lane), best);
            st_cluster_v4(map_rank(smem_addr(base + S + sg), lane), second);
            st_cluster_v4(map_rank(smem_addr(base + 2 * S + sg), lane), mrec);
        }
        cluster_sync();  // every record of the row is in every CTA
        if (rank == 0 && warp == 0) {
            const float4 *rec = sh.rec[par];
            float mz = -INFINITY, dummy = 0.f;
            int mi = -1, bad = 0;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int q = 2 * lane + h;
                if (q < S) {
                    const float4 v = rec[2 * S + q];
                    argmax_merge(mz, mi, dummy, v.x, __float_as_int(v.y), 0.f);
                    bad |= __float_as_int(v.z);
                }
            }
            argmax_allreduce(mz, mi, dummy);
            bad = warp_allor(bad);
            int flags = 0, tok = -1;
            if (bad_t) {
                flags |= F_BAD_TEMP;
            } else if (bad || mi < 0) {
                flags |= F_NONFINITE;  // a NaN or +inf logit, or nothing but -inf
            } else if (!sample) {
                tok = mi;  // greedy: the arg max, ties to the smallest index
            } else {
                const int2 sel = gumbel_select<Tin>(rec, S, lane, false, row, nullptr, 0, static_cast<uint32_t>(r), k,
                                                    mz * k, 0.f, A.seed_lo, A.seed_hi, A.offset);
                tok = sel.x;
                flags |= sel.y;
                if (tok < 0) flags |= F_NONFINITE;
            }
            if (lane == 0) {
                A.tokens[r] = flags ? -1 : tok;
                if (A.flags) A.flags[r] = flags;
            }
        }
        par ^= 1;
    }
}

template <typename Tin, int CV, int MODE, bool DBL>
__global__ void __launch_bounds__(NT, 4) stream_kernel_impl(const VerifyArgs A) {
    using St = Store<Tin>;
    constexpr int VEC = St::VEC;
    constexpr int QV = CV / 32;
    static_assert(CV % 32 == 0, "chunk layout: whole vectors per lane");
    constexpr uint32_t SLOT_BYTES = 2u * CV * 16u;
    extern __shared__ __align__(128) unsigned char smem[];
    StreamShared &sh = *reinterpret_cast<StreamShared *>(smem);
    pdl_allow_next();

    Ctx c;
    c.C = static_cast<int>(cluster_size());
    c.rank = static_cast<int>(cluster_rank());
    c.cid = static_cast<int>(cluster_id_x());
    c.NC = static_cast<int>(gridDim.x) / c.C;
    c.warp = threadIdx.x >> 5;
    c.lane = threadIdx.x & 31;
    c.S = c.C * NW;
    c.sg = c.rank * NW + c.warp;
    c.R = A.ring;
    c.depth = A.depth;
    c.g = A.gamma;
    c.Q = A.gamma + 2;
    const int g = c.g;
    const int nv = A.V / VEC;  // aligned rows only
    const int nvs = A.seg_vectors;
    c.seg_lo = min(nv, c.sg * nvs);
    c.seg_n = min(nv, c.seg_lo + nvs) - c.seg_lo;
    c.cv = CV;
    c.nch = (c.seg_n + CV - 1) / CV;
    c.ws = &sh.w[c.warp];
    c.rec = reinterpret_cast<float4 *>(smem + HDR_BYTES);
    c.ring = smem + HDR_BYTES + rec_bytes(g, c.S) + static_cast<size_t>(c.warp) * c.R * SLOT_BYTES;
    c.pcount = c.ccount = 0;
    c.pslot = c.cslot = c.cphase = 0;
    c.p_ord = 0;
    c.p_i = 0;
    c.p_kind = K_NORM;
    c.p_c = 0;
    c.p_done = (c.nch == 0) || (c.cid >= A.B);
    c.p_t = c.p_d = nullptr;
    c.c_ord = 0;
    c.c_conf = 0;
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
            for (int i = 0; i < c.Q; ++i) mbar_arrive_expect_tx(smem_addr(&sh.xbar[bk][i]), round_bytes(c));
    }
    fence_mbar_init();
    __syncthreads();
    cluster_sync();  // every barrier of the cluster is initialised and armed before any push
    pdl_wait_prior();  // inputs and outputs of earlier launches on the stream: settled from here on

    // sequence parameters, prefetched one sequence ahead (lane l: u_l, y_l)
    auto load_params = [&](int b, float &u, int &y, float &T) {
        u = 2.f;
        y = 0;
        T = 1.f;
        if (b < A.B) {
            if (A.unif && c.lane <= g) u = __ldg(A.unif + static_cast<size_t>(b) * (g + 1) + c.lane);
            if (MODE != M_TO && c.lane < g) y = __ldg(A.ids + static_cast<size_t>(b) * g + c.lane);
            T = __ldg(A.temp + b);
        }
    };
    float nu, nT;
    int ny;
    load_params(c.cid, nu, ny, nT);
    produce<Tin, MODE, DBL>(A, c);

    const float4 ZERO4 = make_float4(0.f, 0.f, 0.f, 0.f);

    for (int ord = 0;; ++ord) {
        const int b = seq_of(c, ord);
        if (b >= A.B) break;
        const float my_u = nu, T = nT;
        int my_y = ny;  // lane l: draft token of position l (target-only: filled at its decision)
        load_params(seq_of(c, ord + 1), nu, ny, nT);
        c.c_ord = ord;
        c.c_conf = 0;

        int flags = 0;
        if (c.dead) flags |= F_TIMEOUT;
        if (!(T >= 0.f) || !(T < INFINITY)) flags |= F_BAD_TEMP;
        const bool greedy = (T == 0.f);
        if (MODE == M_TO) my_y = -1;
        {
            const bool bad_y = MODE != M_TO && (c.lane < g) && (my_y < 0 || my_y >= A.V);
            // the Gumbel-max final draw uses no uniform u_gamma
            const bool bad_u = (c.lane < g || (MODE != M_GB && c.lane == g)) && !(my_u >= 0.f && my_u < 1.f);
            if (__any_sync(FULL, bad_y)) flags |= F_BAD_ID;
            if (__any_sync(FULL, bad_u)) flags |= F_BAD_UNIFORM;
        }
        const float k = greedy ? 0.f : LOG2E / T;
        int n = 0;          // accepted drafts
        int tok = -1;       // drawn token (owner warp; every warp when greedy)
        int owner = 0;      // segment whose warp writes the outputs
        int reached = 0;    // positions whose decision was taken
        // lanes l < gamma: does this warp's segment hold draft token y_l?
        const int yv_l = my_y / VEC - c.seg_lo;
        const bool own_l = MODE != M_TO && (c.lane < g) && yv_l >= 0 && yv_l < c.seg_n;
        const unsigned own_mask = __ballot_sync(FULL, own_l);

        if (flags) {
            drain(c);
            redirect_next(c, ord, A.B);
        } else {
            int dec = 0;      // next position to decide
            int pushed = -1;  // last position whose record this warp pushed
            int rej = -1;     // rejected position
            int rej_y = -1;   // target-only: the draft token rejected there
            bool fin = false; // decisions over (rejection, error or greedy stop)
            auto decide = [&](int i) {
                ++reached;
                if (greedy) {
                    const Greedy r = gather_greedy(c, i);
                    if (r.bad || r.tidx < 0 || (MODE == M_TO && r.didx < 0)) {
                        flags |= F_NONFINITE;
                        fin = true;
                        return;
                    }
                    const int y = MODE != M_TO ? __shfl_sync(FULL, my_y, i) : r.didx;
                    if (MODE == M_TO && c.lane == i) my_y = y;
                    if (y == r.tidx) {
                        ++n;
                        ++dec;
                        c.c_conf = dec;
                    } else {
                        tok = r.tidx;
                        fin = true;
                    }
                    return;
                }
                const Norm r = gather_norm<MODE>(c, i, k, true);
                if (r.rf) {
                    flags |= r.rf;
                    fin = true;
                    return;
                }
                const float ui = __shfl_sync(FULL, my_u, i);
                bool acc;
                if (MODE != M_TO) {
                    acc = log2f(ui) + fmaf(r.Zdy, k, -r.cd) < fmaf(r.Zty, k, -r.ct);
                } else {
                    if (c.lane == i) my_y = r.yhat;
                    acc = log2f(ui) < fmaf(r.Zty, k, -r.ct);
                }
                if (acc) {
                    ++n;
                    ++dec;
                    c.c_conf = dec;
                } else {
                    rej = i;
                    rej_y = r.yhat;
                    fin = true;
                }
            };
            for (int p = 0; p <= g && !fin && !c.dead; ++p) {
                while (!fin && p > c.c_conf + c.depth) {
                    if (!xwait(sh, c, dec)) break;
                    decide(dec);
                }
                if (fin || c.dead) break;
                const bool has_d = p < g;
                const bool use_d = has_d && !(greedy && MODE != M_TO);  // a greedy RS draft row is never read
                const int y = MODE != M_TO ? __shfl_sync(FULL, my_y, has_d ? p : 0) : 0;
                const bool owns_y = MODE != M_TO && has_d && !greedy && ((own_mask >> p) & 1u);
                const int yv = y / VEC - c.seg_lo;
                // ---- stream the segment of rows (t_p, d_p)
                float mt = -INFINITY, st = 0.f, md = -INFINITY, sd = 0.f;
                float zty = 0.f, zdy = 0.f;  // RS: logits at y; TO: zty = target logit at the draft arg max
                int tix = -1, dix = -1;      // running arg max indices (greedy target, greedy / TO draft)
                int bad = 0;
                // a target-only row takes two chunks per slot under DBL
                const bool dbl = DBL && !has_d;
                // per-chunk record of row gamma for the bonus draw
                auto record = [&](int chi, float csum) {
                    Soft a;
                    a.m = mt;
                    a.s = csum;
                    a.s1 = 0.f;
                    const Soft r = soft_warp_allreduce<false>(a, k);
                    if (c.lane == 0) {
                        c.ws->cm[chi] = r.m;
                        c.ws->cs[chi] = r.s;
                    }
                };
                for (int ch = 0; ch < c.nch; ch += dbl ? 2 : 1) {
                    // a decision may already be out: stop streaming a position
                    // that will not be used
                    if (dec < p && xtest(sh, c, dec)) {
                        decide(dec);
                        if (fin) break;
                    }
                    produce<Tin, MODE, DBL>(A, c);
                    if (c.pcount == c.ccount) c.dead = true;  // nothing issued: never wait on it
                    if (c.dead || !slot_wait(c)) break;
                    const unsigned char *tb = c.ring + c.cslot * SLOT_BYTES;
                    const unsigned char *db = tb + CV * 16;
                    const int cnt = chunk_count(c, ch);
                    const int cnt2 = (dbl && ch + 1 < c.nch) ? chunk_count(c, ch + 1) : 0;
                    const bool two = cnt2 > 0;  // rd holds chunk ch + 1 of the target row
                    uint4 rt[QV], rd[QV];
                    if (cnt == CV) {
                        load_chunk<Tin, true, QV>(tb, cnt, c.lane, rt);
                        if (use_d) load_chunk<Tin, true, QV>(db, cnt, c.lane, rd);
                    } else {
                        load_chunk<Tin, false, QV>(tb, cnt, c.lane, rt);
                        if (use_d) load_chunk<Tin, false, QV>(db, cnt, c.lane, rd);
                    }
                    if (two) {
                        if (cnt2 == CV) load_chunk<Tin, true, QV>(db, cnt2, c.lane, rd);
                        else load_chunk<Tin, false, QV>(db, cnt2, c.lane, rd);
                    }
                    // the maxima consume every loaded register: the slot's
                    // reads are complete before it is handed back
                    const float cmt = chunk_max<Tin, QV>(rt);
                    const float cmd = (use_d || two) ? chunk_max<Tin, QV>(rd) : 0.f;
                    __syncwarp();
                    consumed(c);  // the slot refills while this chunk is reduced
                    produce<Tin, MODE, DBL>(A, c);
                    const int vbase = c.seg_lo + ch * CV + c.lane;
                    if (greedy) {
                        bad |= !(cmt < INFINITY) || ((use_d || two) && !(cmd < INFINITY));
                        float dummy = 0.f;
                        argmax_warp<Tin, QV, false>(rt, rt, cmt, vbase, mt, tix, dummy);
                        if (use_d) argmax_warp<Tin, QV, false>(rd, rd, cmd, vbase, md, dix, dummy);
                        else if (two) argmax_warp<Tin, QV, false>(rd, rd, cmd, vbase + CV, mt, tix, dummy);
                        continue;
                    }
                    if (owns_y && yv >= ch * CV && yv < ch * CV + cnt) {
                        const int jv = yv - ch * CV, q = jv >> 5, e = y % VEC;
                        uint4 vt = rt[0], vd = rd[0];
#pragma unroll
                        for (int qq = 1; qq < QV; ++qq) {
                            if (q == qq) {
                                vt = rt[qq];
                                vd = rd[qq];
                            }
                        }
                        zty = __shfl_sync(FULL, vec_elem<Tin>(vt, e), jv & 31);
                        zdy = __shfl_sync(FULL, vec_elem<Tin>(vd, e), jv & 31);
                    }
                    const float csum = fold_regs<Tin, QV>(rt, cmt, k, mt, st, bad);
                    if (has_d) {
                        if (MODE != M_TO) {
                            fold_regs<Tin, QV>(rd, cmd, k, md, sd, bad);
                        } else {
                            bad |= !(cmd < INFINITY);
                            argmax_warp<Tin, QV, true>(rd, rt, cmd, vbase, md, dix, zty);
                        }
                    }
                    if (!has_d && MODE != M_GB) record(ch, csum);
                    if (two) {  // DBL: never the Gumbel-max mode
                        const float csum2 = fold_regs<Tin, QV>(rd, cmd, k, mt, st, bad);
                        record(ch + 1, csum2);
                    }
                }
                if (c.dead || fin) break;  // fin: position p abandoned, its round gets a zero record
                // ---- warp records -> every CTA of the cluster
                const bool wbad = warp_allor(bad) != 0;
                if (greedy) {
                    float dummy = 0.f;
                    argmax_allreduce(mt, tix, dummy);
                    argmax_allreduce(md, dix, dummy);
                    xpush(sh, c, p, make_float4(mt, __int_as_float(tix), md, __int_as_float(dix)),
                          make_float4(wbad ? 1.f : 0.f, 0.f, 0.f, 0.f));
                } else {
                    Soft a;
                    a.m = mt;
                    a.s = st;
                    a.s1 = 0.f;
                    const Soft wt = soft_warp_allreduce<false>(a, k);
                    if (MODE != M_TO) {
                        a.m = md;
                        a.s = sd;
                        const Soft wd = soft_warp_allreduce<false>(a, k);
                        xpush(sh, c, p, make_float4(wt.m, wbad ? NAN : wt.s, wd.m, wbad ? NAN : wd.s),
                              make_float4(zty, zdy, owns_y ? 1.f : 0.f, 0.f));
                    } else {
                        argmax_allreduce(md, dix, zty);
                        xpush(sh, c, p, make_float4(wt.m, wbad ? NAN : wt.s, md, zty),
                              make_float4(__int_as_float(dix), 0.f, 0.f, 0.f));
                    }
                }
                pushed = p;
                produce<Tin, MODE, DBL>(A, c);
                // decisions whose rounds are already complete
                while (!fin && dec < g && dec <= p && xtest(sh, c, dec)) decide(dec);
            }
            while (!fin && !c.dead && dec < g) {
                if (!xwait(sh, c, dec)) break;
                decide(dec);
            }
            // zero records for the rounds this warp did not fill
            if (!c.dead)
                for (int p = pushed + 1; p <= g; ++p) xpush(sh, c, p, ZERO4, ZERO4);
            if (c.dead) {
                flags |= F_TIMEOUT;
            } else if ((flags & ERR_BITS) || (greedy && fin)) {
                xpush(sh, c, g + 1, ZERO4, ZERO4);
            } else if (greedy) {
                // ---- greedy bonus: the arg max of row gamma
                xpush(sh, c, g + 1, ZERO4, ZERO4);
                if (xwait(sh, c, g)) {
                    ++reached;
                    const Greedy r = gather_greedy(c, g);
                    if (r.bad || r.tidx < 0) flags |= F_NONFINITE;
                    else tok = r.tidx;
                } else {
                    flags |= F_TIMEOUT;
                }
            } else if (MODE == M_GB) {
                // ---- Gumbel-max final draw: one pass over row j (the rejected
                // position: residual weights, with the p keys as the zero-mass
                // fallback; after gamma accepts: row gamma, p keys), one round
                const bool resid = rej >= 0;
                const int j = resid ? rej : g;
                bool ok = true;
                Norm r{};
                if (!resid) {
                    ok = xwait(sh, c, g);  // row gamma's normaliser flags
                    if (ok) {
                        ++reached;
                        r = gather_norm<MODE>(c, g, k, false);
                        flags |= r.rf;
                    }
                } else {
                    r = gather_norm<MODE>(c, j, k, true);
                }
                if (!ok) flags |= F_TIMEOUT;
                // one pass: residual keys (at a rejection) and p keys; the p
                // draw is the bonus, or the residual's fallback when every
                // residual weight rounded to zero (ZERO_MASS)
                float4 best = make_float4(-INFINITY, __int_as_float(-1), -INFINITY, __int_as_float(-1));
                float4 second = best;
                if (!(flags & ERR_BITS)) {
                    const uint32_t bb = static_cast<uint32_t>(b);
                    const float kp = fmaf(r.Mt, k, GUMBEL2_MIN);  // the best p key is at least max z k + min g
                    const int ip = -1;
                    const float kp2 = -INFINITY;
                    if (resid) {
                        // drop the look-ahead rows past the rejection (the producer
                        // moves on to the next sequence's first row) and read row j
                        // directly, mostly from L2
                        drain(c);
                        redirect_next(c, ord, A.B);
                        c.c_conf = g;  // the path is fixed
                        produce<Tin, MODE, DBL>(A, c);
                        const Top2x2 kk = gumbel_pass<Tin, true>(row_base<Tin>(A, true, b, j),
                                                                 row_base<Tin>(A, false, b, j), c.seg_lo, c.seg_n, j,
                                                                 bb, k, r.ct, r.cd, kp, A.seed_lo, A.seed_hi, A.offset);
                        best = kk.best;
                        second = kk.second;
                    } else {
                        // the bonus: row gamma streams through the ring once more
                        // (mostly from L2) as a residual unit of the target row
                        // alone, after which the producer moves on to the next
                        // sequence's first row
                        drain(c);
                        c.p_ord = ord;
                        c.p_i = j;
                        c.p_kind = K_RES;
                        c.p_c = 0;
                        c.p_done = (c.nch == 0);
                        c.c_conf = g;  // the path is fixed
                        float bp = kp;
                        float4 top = make_float4(kp, __int_as_float(ip), kp2, 0.f);
                        for (int ch = 0; ch < c.nch; ++ch) {
                            produce<Tin, MODE, DBL>(A, c);
                            if (c.pcount == c.ccount) c.dead = true;
                            if (c.dead || !slot_wait(c)) break;
                            const unsigned char *tb = c.ring + c.cslot * SLOT_BYTES;
                            top = gumbel_slot<Tin, CV>(tb, chunk_count(c, ch), c.seg_lo + ch * CV, k, j, bb, A.seed_lo,
                                                       A.seed_hi, A.offset, bp, top);
                            __syncwarp();
                            consumed(c);
                            produce<Tin, MODE, DBL>(A, c);
                            bp = warp_allmax(top.x);  // the warp's best p key so far bounds every lane's filters
                        }
                        const float4 p2 = warp_top2<Tin, false>(top.x, __float_as_int(top.y), top.z,
                                                                row_base<Tin>(A, true, b, j), nullptr, c.seg_lo,
                                                                c.seg_n, j, bb, k, 0.f, 0.f, A.seed_lo, A.seed_hi,
                                                                A.offset);
                        best = make_float4(-INFINITY, __int_as_float(-1), p2.x, p2.y);
                        second = make_float4(-INFINITY, __int_as_float(-1), p2.z, p2.w);
                    }
                }
                // every warp fills round gamma + 1 with its two best candidates
                // of each draw (none when the row is flagged)
                if (!c.dead) {
                    xpush(sh, c, g + 1, best, second);
                    xwait(sh, c, g + 1);
                }
                if (c.dead) {
                    flags |= F_TIMEOUT;
                } else if (!(flags & ERR_BITS)) {
                    const int2 sel = gumbel_select<Tin>(rec_at(c, c.bank, g + 1, 0), c.S, c.lane, resid,
                                                        row_base<Tin>(A, true, b, j), row_base<Tin>(A, false, b, j), j,
                                                        static_cast<uint32_t>(b), k, r.ct, r.cd, A.seed_lo, A.seed_hi,
                                                        A.offset);
                    tok = sel.x;
                    flags |= sel.y;
                    if (tok < 0) flags |= F_NONFINITE;
                }
                owner = 0;
            } else if (rej >= 0) {
                // ---- rejection at rej: residual pass over rows (t_rej, d_rej);
                // target-only: over t_rej with the rejected token excluded
                drain(c);
                c.p_ord = ord;
                c.p_i = rej;
                c.p_kind = K_RES;
                c.p_c = 0;
                c.p_done = (c.nch == 0);
                c.c_conf = g;  // the path is fixed: the producer may move on after the pass
                const Norm r = gather_norm<MODE>(c, rej, k, true);
                const int ex_v = MODE == M_TO ? rej_y / VEC - c.seg_lo : -1;  // excluded vector in the segment
                float Rw = 0.f;
                for (int ch = 0; ch < c.nch; ++ch) {
                    produce<Tin, MODE, DBL>(A, c);
                    if (c.pcount == c.ccount) c.dead = true;
                    if (c.dead || !slot_wait(c)) break;
                    const unsigned char *tb = c.ring + c.cslot * SLOT_BYTES;
                    const unsigned char *db = tb + CV * 16;
                    const int cnt = chunk_count(c, ch);
                    uint4 rt[QV], rd[QV];
                    if (cnt == CV) {
                        load_chunk<Tin, true, QV>(tb, cnt, c.lane, rt);
                        if (MODE == M_RS) load_chunk<Tin, true, QV>(db, cnt, c.lane, rd);
                    } else {
                        load_chunk<Tin, false, QV>(tb, cnt, c.lane, rt);
                        if (MODE == M_RS) load_chunk<Tin, false, QV>(db, cnt, c.lane, rd);
                    }
                    float ps;
                    if (MODE == M_RS) {
                        ps = warp_allsum(res_regs<Tin, QV>(rt, rd, k, r.ct, r.cd));
                    } else {
                        if (ex_v >= ch * CV && ex_v < ch * CV + cnt && ((ex_v - ch * CV) & 31) == c.lane) {
                            const int q = (ex_v - ch * CV) >> 5;
#pragma unroll
                            for (int qq = 0; qq < QV; ++qq)
                                if (qq == q) vec_set_neginf<Tin>(rt[qq], rej_y % VEC);
                        }
                        ps = warp_allsum(psum_regs<Tin, QV>(rt, k, r.ct));
                    }
                    __syncwarp();
                    consumed(c);
                    produce<Tin, MODE, DBL>(A, c);
                    if (c.lane == 0) c.ws->cs[ch] = ps;
                    Rw += ps;
                }
                if (!c.dead) {
                    xpush(sh, c, g + 1, make_float4(Rw, 0.f, 0.f, 0.f), ZERO4);
                    xwait(sh, c, g + 1);
                }
                if (c.dead) {
                    flags |= F_TIMEOUT;
                } else {
                    const int q0 = 2 * c.lane, q1 = 2 * c.lane + 1;
                    const float t0 = q0 < c.S ? rec_at(c, c.bank, g + 1, q0)->x : 0.f;
                    const float t1 = q1 < c.S ? rec_at(c, c.bank, g + 1, q1)->x : 0.f;
                    const float uf = __shfl_sync(FULL, my_u, g);
                    float rem;
                    int last;
                    const int sel = pick_segment(t0, t1, uf, rem, last);
                    if (sel >= 0) {
                        owner = sel;
                        if (sel == c.sg) {
                            if (MODE == M_RS)
                                tok = walk_segment<Tin, true, QV>(seg_of(c), row_base<Tin>(A, true, b, rej),
                                                                  row_base<Tin>(A, false, b, rej), false, 0.f, k, r.ct,
                                                                  r.cd, rem, last, -1);
                            else
                                tok = walk_segment<Tin, false, QV>(seg_of(c), row_base<Tin>(A, true, b, rej), nullptr,
                                                                   false, 0.f, k, r.ct, 0.f, rem, last, rej_y);
                        }
                    } else {
                        // residual mass rounded to zero: draw from p_rej
                        flags |= F_ZERO_MASS;
                        const float a0 = (r.s0 != 0.f) ? r.s0 * ex2((r.m0 - r.Mt) * k) : 0.f;
                        const float a1 = (r.s1 != 0.f) ? r.s1 * ex2((r.m1 - r.Mt) * k) : 0.f;
                        const int sp = pick_segment(a0, a1, uf, rem, last);
                        if (sp < 0) {
                            flags |= F_NONFINITE;
                        } else {
                            owner = sp;
                            if (sp == c.sg) {
                                direct_chunk_sums<Tin>(seg_of(c), row_base<Tin>(A, true, b, rej), k, r.Mt);
                                tok = walk_segment<Tin, false, QV>(seg_of(c), row_base<Tin>(A, true, b, rej), nullptr,
                                                                   true, r.Mt, k, r.Mt * k, 0.f, rem, last, -1);
                            }
                        }
                    }
                }
            } else {
                // ---- bonus: all gamma drafts accepted, draw from p_gamma
                xpush(sh, c, g + 1, ZERO4, ZERO4);
                if (xwait(sh, c, g)) {
                    const Norm r = gather_norm<MODE>(c, g, k, false);
                    if (r.rf) {
                        flags |= r.rf;
                    } else {
                        const float a0 = (r.s0 != 0.f) ? r.s0 * ex2((r.m0 - r.Mt) * k) : 0.f;
                        const float a1 = (r.s1 != 0.f) ? r.s1 * ex2((r.m1 - r.Mt) * k) : 0.f;
                        const float uf = __shfl_sync(FULL, my_u, g);
                        float rem;
                        int last;
                        const int sp = pick_segment(a0, a1, uf, rem, last);
                        if (sp < 0) {
                            flags |= F_NONFINITE;
                        } else {
                            owner = sp;
                            if (sp == c.sg)
                                tok = walk_segment<Tin, false, QV>(seg_of(c), row_base<Tin>(A, true, b, g), nullptr,
                                                                   true, r.Mt, k, r.Mt * k, 0.f, rem, last, -1);
                        }
                    }
                } else {
                    flags |= F_TIMEOUT;
                }
            }
            if ((flags & ERR_BITS) || (greedy && fin)) {
                // drop the look-ahead (rows past an error or a greedy stop);
                // the next sequence starts from its first row
                drain(c);
                redirect_next(c, ord, A.B);
            }
            // warp 0 closes the bank: every round of this sequence complete, re-armed
            if (c.warp == 0 && !c.dead) {
                for (int i = 0; i < c.Q; ++i) {
                    if (!xwait(sh, c, i)) break;
                    if (c.lane == 0) mbar_arrive_expect_tx(smem_addr(&sh.xbar[c.bank][i]), round_bytes(c));
                }
                __syncwarp();
            }
            c.bpar ^= 1u << c.bank;
            c.bank ^= 1;
        }
        if ((flags & ERR_BITS) || greedy) owner = 0;
        if (tok < 0 && !(flags & ERR_BITS) && c.sg == owner) flags |= F_NONFINITE;
        // ---- outputs, written by the owning warp
        if (c.sg == owner || (c.dead && c.sg == 0)) {
            const bool err = (flags & ERR_BITS) != 0;
            if (c.lane <= g) {
                int v = -1;
                if (!err) v = (c.lane < n) ? my_y : (c.lane == n ? tok : -1);
                A.tokens[static_cast<size_t>(b) * (g + 1) + c.lane] = v;
            }
            if (MODE == M_TO && A.yhat && c.lane < g)
                A.yhat[static_cast<size_t>(b) * g + c.lane] = (!err && c.lane < reached) ? my_y : -1;
            if (c.lane == 0) {
                if (A.accept_len) A.accept_len[b] = err ? -1 : n;
                if (A.flags) A.flags[b] = flags;
            }
        }
        produce<Tin, MODE, DBL>(A, c);
    }

    drain(c);
    __syncthreads();
    cluster_sync();  // no CTA leaves while a peer may still push into it
}

}  // namespace

const void *gsample_kernel(int dtype) {
    return dtype == 0 ? reinterpret_cast<const void *>(&gsample_kernel_impl<float>)
                      : reinterpret_cast<const void *>(&gsample_kernel_impl<bf16_t>);
}
int gsample_threads() { return GS_NT; }
int gsample_max_cluster() { return GS_MAXC; }
uint32_t gsample_smem_bytes() { return static_cast<uint32_t>(sizeof(GsShared)); }

uint32_t stream_hdr_bytes() { return HDR_BYTES; }
uint32_t stream_rec_bytes(int gamma, int S) { return rec_bytes(gamma, S); }
int stream_threads() { return NT; }
uint32_t stream_slot_bytes(int cv) { return 2u * static_cast<uint32_t>(cv) * 16u; }
int stream_max_chunks() { return MAXCH; }
int stream_max_segments() { return MAXS; }
int stream_max_ring() { return MAXR; }
int stream_max_gamma() { return MAXG; }

const void *stream_kernel(int dtype, int cv, int mode, bool dbl) {
    if (dbl && mode == 0 && cv == 160)  // one-row sequences, inverse-CDF draw
        return dtype == 0 ? reinterpret_cast<const void *>(&stream_kernel_impl<float, 160, M_RS, true>)
                          : reinterpret_cast<const void *>(&stream_kernel_impl<bf16_t, 160, M_RS, true>);
    if (mode == 1)  // target-only: 2 KB chunks (the arg max keeps two rows of registers live)
        return dtype == 0 ? reinterpret_cast<const void *>(&stream_kernel_impl<float, 128, M_TO, false>)
                          : reinterpret_cast<const void *>(&stream_kernel_impl<bf16_t, 128, M_TO, false>);
    if (mode == 2) {  // Gumbel-max final draw
        if (dtype == 0)
            return cv == 192 ? reinterpret_cast<const void *>(&stream_kernel_impl<float, 192, M_GB, false>)
                             : reinterpret_cast<const void *>(&stream_kernel_impl<float, 128, M_GB, false>);
        return cv == 192 ? reinterpret_cast<const void *>(&stream_kernel_impl<bf16_t, 192, M_GB, false>)
                         : reinterpret_cast<const void *>(&stream_kernel_impl<bf16_t, 128, M_GB, false>);
    }
    if (dtype == 0)
        return cv == 192   ? reinterpret_cast<const void *>(&stream_kernel_impl<float, 192, M_RS, false>)
               : cv == 160 ? reinterpret_cast<const void *>(&stream_kernel_impl<float, 160, M_RS, false>)
                           : reinterpret_cast<const void *>(&stream_kernel_impl<float, 128, M_RS, false>);
    return cv == 192   ? reinterpret_cast<const void *>(&stream_kernel_impl<bf16_t, 192, M_RS, false>)
           : cv == 160 ? reinterpret_cast<const void *>(&stream_kernel_impl<bf16_t, 160, M_RS, false>)
                       : reinterpret_cast<const void *>(&stream_kernel_impl<bf16_t, 128, M_RS, false>);
}

}  // namespace mtp
