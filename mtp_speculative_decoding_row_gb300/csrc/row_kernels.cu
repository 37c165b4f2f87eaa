// row_kernels.cu -- batched MTP rejection-sampling verification and
// per-position row statistics on sm_103a.
//
// Persistent thread-block clusters of C CTAs.  Cluster c owns sequences
// c, c + NC, c + 2 NC, ... and keeps two of them ("streams") in flight: while
// one stream's unit (the target row, plus the draft row, of one position) is
// being reduced and decided, the other stream's next unit is arriving by bulk
// copy.  Each CTA holds its vocabulary slice of the unit in shared memory,
// forms the temperature-scaled softmax normalisers in one online pass, and
// the cluster all-gathers the CTA partials with DSMEM pushes (st.async onto
// the peers' mbarriers).  Then (method: "Breaking Entropy Bounds:
// Accelerating RL Training via MTP with Rejection Sampling", §2 "Acceptance
// methods" and App. G.1; "EntMTP", Related Work "Speculative Decoding"):
//   - draft y_i is accepted iff u_i q_i(y_i) < p_i(y_i), tested as
//     log2 u_i + log2 q_i(y_i) < log2 p_i(y_i);
//   - at the first rejection the replacement is drawn from
//     norm(max(0, p - q)) by a two-pass inverse CDF over the slices still
//     held on chip; after gamma accepts the bonus token is drawn from p_gamma;
//   - optionally alpha_i = sum_v min(p_i, q_i) (§3, §8) and
//     H(p_i) = -sum_v p log p are formed for every position.
// Without statistics no row after the stop is ever loaded.
#include <cstddef>

#include "common.cuh"
#include "kernels.h"

namespace mtp {

constexpr int NT = 256;      // threads per CTA
constexpr int NW = NT / 32;  // warps per CTA

struct StreamSt {
    int active;   // stream holds a sequence
    int b;        // sequence
    int i;        // position of the unit in flight
    int n;        // accepted drafts
    int stopped;  // decision chain finished
    int flags;    // row flags
    int drawn;    // residual / bonus token
    int armed;    // a bulk copy is in flight on the stream's barrier
    uint32_t ph;  // parity of the stream's load barrier
    int writer;   // cluster rank that writes the sequence's outputs
    int pad[2];
};

struct RowShared {
    Xchg x;
    float tpart[6][NT];     // per-thread partials (columns)
    float segtot[NW];       // per-warp CDF segment totals
    int sampi[4];
    float sampf[4];
    StreamSt st[2];
    int tok[2][MAX_GAMMA + 1];
    float alpha[2][MAX_GAMMA];
    float ent[2][MAX_GAMMA + 1];
    // per-stream sequence parameters, prefetched when the stream takes a sequence
    float T[2];
    int ids[2][MAX_GAMMA];
    float u[2][MAX_GAMMA + 1];
    unsigned long long lbar[2][2];  // load barriers: [stream][target slice, draft slice]
};
constexpr uint32_t HDR_BYTES = (sizeof(RowShared) + 127u) & ~127u;
uint32_t row_hdr_bytes() { return HDR_BYTES; }
int row_threads() { return NT; }

constexpr int ERR_BITS = F_NONFINITE | F_BAD_ID | F_BAD_TEMP | F_BAD_UNIFORM | F_TIMEOUT;

// ------------------------------------------------------------ reductions ---

// Per-thread softmax partials -> CTA partial in every lane of warp 0: every
// thread stores its partials (column layout), warp 0 merges NT/32 of them per
// lane and finishes with one butterfly.
template <bool ENT>
__device__ __forceinline__ void block_soft(float (*tp)[NT], Soft &at, Soft &ad, int &bad, float k) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    tp[0][tid] = at.m;
    tp[1][tid] = at.s;
    tp[2][tid] = at.s1;
    tp[3][tid] = ad.m;
    tp[4][tid] = ad.s;
    tp[5][tid] = __int_as_float(bad);
    __syncthreads();
    if (warp == 0) {
        const Soft a = soft_lane_merge<ENT, NW>(tp[0], tp[1], tp[2], lane, k);
        const Soft d = soft_lane_merge<false, NW>(tp[3], tp[4], tp[4], lane, k);
        int bb = 0;
#pragma unroll
        for (int q = 0; q < NW; ++q) bb |= __float_as_int(tp[5][lane + 32 * q]);
        at = soft_warp_allreduce<ENT>(a, k);
        ad = soft_warp_allreduce<false>(d, k);
        bad = warp_allor(bb);
    }
}

// Arg max across the warp: the largest value, ties to the smallest index
// (index -1: none).  Same result in every lane.
__device__ __forceinline__ void warp_argmax(float &v, int &i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(FULL, v, o);
        const int oi = __shfl_xor_sync(FULL, i, o);
        if (oi >= 0 && (i < 0 || ov > v || (ov == v && oi < i))) {
            v = ov;
            i = oi;
        }
    }
}

// Per-thread arg max (and flag bits) -> CTA arg max in every lane of warp 0.
__device__ __forceinline__ void block_argmax(float (*tp)[NT], float &v, int &i, int &bad) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    tp[0][tid] = v;
    tp[1][tid] = __int_as_float(i);
    tp[2][tid] = __int_as_float(bad);
    __syncthreads();
    if (warp == 0) {
        float bv = -INFINITY;
        int bi = -1, bb = 0;
#pragma unroll
        for (int q = 0; q < NW; ++q) {
            const float ov = tp[0][lane + 32 * q];
            const int oi = __float_as_int(tp[1][lane + 32 * q]);
            if (oi >= 0 && (bi < 0 || ov > bv || (ov == bv && oi < bi))) {
                bv = ov;
                bi = oi;
            }
            bb |= __float_as_int(tp[2][lane + 32 * q]);
        }
        warp_argmax(bv, bi);
        v = bv;
        i = bi;
        bad = warp_allor(bb);
    }
}

// Per-thread sum -> CTA sum in every lane of warp 0.
__device__ __forceinline__ float block_sum(float (*tp)[NT], float v) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    tp[0][tid] = v;
    __syncthreads();
    float r = 0.f;
    if (warp == 0) {
#pragma unroll
        for (int q = 0; q < NW; ++q) r += tp[0][lane + 32 * q];
        r = warp_allsum(r);
    }
    return r;
}

// Combine the C softmax records of an exchange slot (every warp, every lane).
template <bool ENT>
__device__ __forceinline__ void gather_soft(const Xchg &x, int slot, int C, float k, Soft &Ct, Soft &Cd, int &bits,
                                            float &zty, float &zdy) {
    const int lane = threadIdx.x & 31;
    Soft a = soft_empty(), d = soft_empty();
    int bb = 0;
    float zt = 0.f, zd = 0.f;
    if (lane < C) {
        const float *r = x.rec[slot][lane];
        a = {r[0], r[1], r[2]};
        d = {r[3], r[4], 0.f};
        zt = r[5];
        zd = r[6];
        bb = __float_as_int(r[7]);
    }
    Ct = soft_warp_allreduce<ENT>(a, k);
    Cd = soft_warp_allreduce<false>(d, k);
    const unsigned hm = __ballot_sync(FULL, (bb & 0x100) != 0);
    const int src = hm ? (__ffs(hm) - 1) : 0;
    zty = __shfl_sync(FULL, zt, src);
    zdy = __shfl_sync(FULL, zd, src);
    bits = warp_allor(bb & 0xff);
}

__device__ __forceinline__ float gather_sum(const Xchg &x, int slot, int C) {
    const int lane = threadIdx.x & 31;
    return warp_allsum(lane < C ? x.rec[slot][lane][0] : 0.f);
}

// Draft partial of the statistics modes: the sum pass of thread_soft_exact
// (same loop, same accumulation order) against the reference m, the target's
// exact maximum over the same vectors, instead of a maximum of the draft's
// own.  Where the draft row equals the target row away from elements whose
// weight underflows, the two partials, and so the cluster's normalisers, come
// out bit for bit the same; a rejection's residual max(0, p - q) is then
// exactly zero there, as it is in exact arithmetic (up to the underflowing
// terms), and the draw falls back to p with the row flagged ZERO_MASS,
// instead of drawing from rounding noise.  Falls back to thread_soft_exact
// when m is not finite or the sum leaves the safe range (a NaN or +inf logit
// included, which that path flags).
template <typename Tin, int NT>
__device__ __forceinline__ Soft draft_soft_at(const unsigned char *buf, int nvec, float k, float m, bool &bad) {
    if (m > -INFINITY && m < INFINITY) {
        const float mk = m * k;
        const uint64_t K2 = f2pack(k, k), NMK2 = f2pack(-mk, -mk);
        uint64_t acc = f2pack(0.f, 0.f);
        for (int j = threadIdx.x; j < nvec; j += NT) {
            const uint4 r = vec_at(buf, j);
            const uint32_t w[4] = {r.x, r.y, r.z, r.w};
            if (Store<Tin>::ES == 2) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float d0, d1;
                    f2unpack(f2fma(bf16pair_f2(w[q]), K2, NMK2), d0, d1);
                    acc = f2add(acc, f2pack(ex2(d0), ex2(d1)));
                }
            } else {
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    float d0, d1;
                    f2unpack(f2fma(f2pack(__uint_as_float(w[2 * q]), __uint_as_float(w[2 * q + 1])), K2, NMK2), d0, d1);
                    acc = f2add(acc, f2pack(ex2(d0), ex2(d1)));
                }
            }
        }
        float s0, s1;
        f2unpack(acc, s0, s1);
        const float sum = s0 + s1;
        if (sum < 1.8e19f) {  // finite, no NaN, far from overflow after merging
            Soft a;
            a.m = m;
            a.s = sum;
            a.s1 = 0.f;
            return a;
        }
    }
    return thread_soft_exact<Tin, false, NT>(buf, nvec, k, bad);
}

// ------------------------------------------------------------- sampling ----

// Sampling weights of one image vector: WMODE 0 = residual max(0, p - q),
// WMODE 1 = p.  p = 2^{z_t k - ct}, q = 2^{z_d k - cd}.
template <typename Tin, int WMODE>
__device__ __forceinline__ void vec_weights(const unsigned char *tb, const unsigned char *db, int j, float k,
                                            float ct, float cd, float (&w)[Store<Tin>::VEC]) {
    constexpr int VEC = Store<Tin>::VEC;
    float zt[VEC];
    Store<Tin>::unpack(vec_at(tb, j), zt);
    if (WMODE == 0) {
        float zd[VEC];
        Store<Tin>::unpack(vec_at(db, j), zd);
#pragma unroll
        for (int e = 0; e < VEC; ++e) w[e] = fmaxf(ex2(fmaf(zt[e], k, -ct)) - ex2(fmaf(zd[e], k, -cd)), 0.f);
    } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) w[e] = ex2(fmaf(zt[e], k, -ct));
    }
}

template <int VEC>
__device__ __forceinline__ float vec_sum(const float (&w)[VEC]) {
    float s = w[0];
#pragma unroll
    for (int e = 1; e < VEC; ++e) s += w[e];
    return s;
}

struct SampleOut {
    int status;  // 0 drawn, -2 the weights sum to zero, -3 an exchange gave up
    int writer;  // rank of the CTA that found the token (same in every CTA)
    int token;   // the token, valid in the writer CTA
};

// Two-pass inverse CDF over the row held by the cluster.  Pass one forms the
// per-warp segment totals, the CTA total and (exchange) every CTA's total;
// the draw is the smallest vocabulary index whose running sum exceeds u * R,
// in ascending index order (CTA rank, warp segment, 32-vector round, lane,
// element).  If rounding leaves no such index in the selected unit, the last
// index of that unit with positive weight is taken.  Only the selected CTA
// walks its segment; it keeps the token and writes the sequence's outputs.
template <typename Tin, int WMODE>
__device__ __noinline__ SampleOut cluster_sample(RowShared &sh, int &round, const unsigned char *tb,
                                                 const unsigned char *db, const Slice &s, float k, float ct, float cd,
                                                 float u, int C, int rank) {
    constexpr int VEC = Store<Tin>::VEC;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nvw = (s.nvec + NW - 1) / NW;
    const int a0 = min(s.nvec, warp * nvw), a1 = min(s.nvec, a0 + nvw);
    SampleOut out = {0, 0, -1};

    // pass one: per-thread sums, one reduction per warp segment
    float part = 0.f;
    for (int j = a0 + lane; j < a1; j += 32) {
        float w[VEC];
        vec_weights<Tin, WMODE>(tb, db, j, k, ct, cd, w);
        part += vec_sum<VEC>(w);
    }
    part = warp_allsum(part);
    if (lane == 0) sh.segtot[warp] = part;
    __syncthreads();
    float tot = 0.f;
    if (warp == 0)
        for (int w = 0; w < NW; ++w) tot += sh.segtot[w];
    float rec[4] = {tot, 0.f, 0.f, 0.f};
    bool ok;
    const int slot = xchg_round<4>(sh.x, round, rec, C, rank, ok);
    if (!ok) {
        out.status = -3;
        return out;
    }
    // every thread: rank-ordered scan of the CTA totals
    float R = 0.f;
    for (int r = 0; r < C; ++r) R += sh.x.rec[slot][r][0];
    int rs = -1, last = 0;
    float rem = u * R;
    if (R > 0.f) {
        for (int r = 0; r < C; ++r) {
            const float vr = sh.x.rec[slot][r][0];
            if (vr > rem) {
                rs = r;
                break;
            }
            rem -= vr;
        }
        if (rs < 0) {
            last = 1;
            for (int r = 0; r < C; ++r)
                if (sh.x.rec[slot][r][0] > 0.f) rs = r;
        }
    }
    if (rs < 0) {
        out.status = -2;
        return out;
    }
    out.writer = rs;
    if (rank == rs) {
        // warp segment (same scan in every thread of this CTA)
        int lm = last, ws = -1;
        if (!lm) {
            for (int w = 0; w < NW; ++w) {
                const float t = sh.segtot[w];
                if (t > rem) {
                    ws = w;
                    break;
                }
                rem -= t;
            }
        }
        if (ws < 0) {
            lm = 1;
            for (int w = 0; w < NW; ++w)
                if (sh.segtot[w] > 0.f) ws = w;
        }
        if (warp == ws) {
            const int b0 = min(s.nvec, ws * nvw), b1 = min(s.nvec, b0 + nvw);
            int tok = -1;
            if (!lm) {
                for (int base = b0; base < b1; base += 32) {
                    const int j = base + lane;
                    float w[VEC];
                    float vs = 0.f;
                    if (j < b1) {
                        vec_weights<Tin, WMODE>(tb, db, j, k, ct, cd, w);
                        vs = vec_sum<VEC>(w);
                    } else {
#pragma unroll
                        for (int e = 0; e < VEC; ++e) w[e] = 0.f;
                    }
                    const float inc = warp_incl_scan(vs);
                    const float t = __shfl_sync(FULL, inc, 31);
                    if (t > rem) {
                        const unsigned bal = __ballot_sync(FULL, inc > rem);
                        const int L = __ffs(bal) - 1;
                        float exc = __shfl_up_sync(FULL, inc, 1);
                        if (lane == 0) exc = 0.f;
                        int tk = -1;
                        if (lane == L) {
                            float r2 = rem - exc;
                            int ef = -1;
#pragma unroll
                            for (int e = 0; e < VEC; ++e) {
                                if (ef < 0) {
                                    if (w[e] > r2)
                                        ef = e;
                                    else
                                        r2 -= w[e];
                                }
                            }
                            if (ef < 0) {
#pragma unroll
                                for (int e = 0; e < VEC; ++e)
                                    if (w[e] > 0.f) ef = e;
                            }
                            tk = s.lo + j * VEC + ef;
                        }
                        tok = __shfl_sync(FULL, tk, L);
                        break;
                    }
                    rem -= t;
                }
                if (tok < 0) lm = 1;
            }
            if (lm) {
                int best = -1;
                for (int base = b0; base < b1; base += 32) {
                    const int j = base + lane;
                    if (j < b1) {
                        float w[VEC];
                        vec_weights<Tin, WMODE>(tb, db, j, k, ct, cd, w);
#pragma unroll
                        for (int e = 0; e < VEC; ++e)
                            if (w[e] > 0.f) best = max(best, s.lo + j * VEC + e);
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) best = max(best, __shfl_xor_sync(FULL, best, o));
                tok = best;
            }
            if (lane == 0) sh.sampi[0] = tok;
        }
        __syncthreads();  // CTA-uniform branch
        out.token = sh.sampi[0];
    }
    return out;
}

// ----------------------------------------------------------- unit loads ----

template <typename Tin>
__device__ __forceinline__ const unsigned char *row_ptr(const void *base, size_t row, int V) {
    return reinterpret_cast<const unsigned char *>(base) + row * static_cast<size_t>(V) * Store<Tin>::ES;
}

// Start the loads of unit (b, i) of stream `st` (aligned rows: one bulk copy
// per row slice on the stream's barrier; otherwise loads happen at use).
template <typename Tin>
__device__ __forceinline__ void issue_unit(const VerifyArgs &A, StreamSt &st, const Slice &s, unsigned char *tb,
                                           unsigned char *db, uint32_t bar) {
    st.armed = 0;
    if (!A.aligned || s.nvec == 0) return;
    const int g = A.gamma;
    const uint32_t bytes = static_cast<uint32_t>(s.nvec) * 16u;
    const bool has_d = st.i < g;
    if (threadIdx.x == 0) {
        fence_proxy_async();
        const size_t lo = static_cast<size_t>(s.lo) * Store<Tin>::ES;
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s(smem_addr(tb), row_ptr<Tin>(A.target, static_cast<size_t>(st.b) * (g + 1) + st.i, A.V) + lo, bytes,
                 bar);
        // the draft slice on its own barrier (completed at once without a draft
        // row), so that the target's first pass overlaps the draft's arrival
        mbar_arrive_expect_tx(bar + 8u, has_d ? bytes : 0u);
        if (has_d)
            bulk_g2s(smem_addr(db), row_ptr<Tin>(A.draft, static_cast<size_t>(st.b) * g + st.i, A.V) + lo, bytes,
                     bar + 8u);
    }
    st.armed = 1;
}

// Wait for both slices of a unit (target barrier `bar`, draft barrier next
// to it); false when a bounded wait gave up.
__device__ __forceinline__ bool wait_unit(uint32_t bar, uint32_t ph) {
    const bool a = mbar_wait_bounded(bar, ph);
    const bool b = mbar_wait_bounded(bar + 8u, ph);
    return a && b;
}

// Argument checks of stream si's sequence, from its prefetched parameters
// (the same in every CTA of the cluster).
__device__ __forceinline__ int validate_seq(const RowShared &sh, int si, int g, int V, bool decide, bool greedy_ok) {
    const float T = sh.T[si];
    int f = 0;
    if (!(greedy_ok ? T >= 0.f : T > 0.f) || !(T < INFINITY)) f |= F_BAD_TEMP;
    if (decide) {
        for (int i = 0; i < g; ++i) {
            const int y = sh.ids[si][i];
            if (y < 0 || y >= V) f |= F_BAD_ID;
        }
        for (int i = 0; i <= g; ++i) {
            const float u = sh.u[si][i];
            if (!(u >= 0.f && u < 1.f)) f |= F_BAD_UNIFORM;
        }
    }
    return f;
}

// Stream si takes sequence b: state reset and asynchronous copies of the
// sequence's temperature, draft ids and uniforms into shared memory (waited
// for by the issuing threads at the start of the stream's next step).
__device__ __forceinline__ StreamSt start_seq(const VerifyArgs &A, RowShared &sh, int si, int b, bool decide,
                                              uint32_t ph) {
    StreamSt st = {};
    st.ph = ph;
    if (b >= A.B) return st;
    st.active = 1;
    st.b = b;
    st.drawn = -1;
    const int g = A.gamma, tid = threadIdx.x;
    if (decide && tid <= g) cp_async4(&sh.u[si][tid], A.unif + static_cast<size_t>(b) * (g + 1) + tid);
    if (decide && tid >= 64 && tid < 64 + g) cp_async4(&sh.ids[si][tid - 64], A.ids + static_cast<size_t>(b) * g + (tid - 64));
    if (tid == NT - 1) cp_async4(&sh.T[si], A.temp + b);
    return st;
}

// ---------------------------------------------------------------- kernel ---

template <typename Tin, int MODE>
__global__ void __launch_bounds__(NT, 2) row_kernel_impl(const VerifyArgs A) {
    using S = Store<Tin>;
    constexpr int VEC = S::VEC;
    constexpr bool STATS = (MODE != MODE_VERIFY);
    constexpr bool DECIDE = (MODE != MODE_STATS);
    extern __shared__ __align__(128) unsigned char smem[];
    RowShared &sh = *reinterpret_cast<RowShared *>(smem);

    const int tid = threadIdx.x;
    const int C = static_cast<int>(cluster_size());
    const int rank = static_cast<int>(cluster_rank());
    const int cid = static_cast<int>(cluster_id_x());
    const int NC = static_cast<int>(gridDim.x) / C;
    const int g = A.gamma;
    const Slice s = make_slice<Tin>(A.V, C, rank);

    // stream si: target slice at tbuf(si), draft slice right after it
    auto tbuf = [&](int si) { return smem + HDR_BYTES + static_cast<size_t>(si) * 2 * A.slice_bytes; };

    if (tid == 0) {
        xchg_init(sh.x);
        for (int q = 0; q < 2; ++q) {
            mbar_init(smem_addr(&sh.lbar[q][0]), 1);
            mbar_init(smem_addr(&sh.lbar[q][1]), 1);
        }
        fence_mbar_init();
    }
    const int NS = A.streams;  // sequences in flight per CTA
    int next_seq = cid + NS * NC;
    StreamSt st0 = start_seq(A, sh, 0, cid, DECIDE, 0);
    StreamSt st1 = NS > 1 ? start_seq(A, sh, 1, cid + NC, DECIDE, 0) : StreamSt{};
    __syncthreads();
    cluster_sync();  // peers' barriers are initialised before any push
    if (st0.active) issue_unit<Tin>(A, st0, s, tbuf(0), tbuf(0) + A.slice_bytes, smem_addr(&sh.lbar[0][0]));
    if (st1.active) issue_unit<Tin>(A, st1, s, tbuf(1), tbuf(1) + A.slice_bytes, smem_addr(&sh.lbar[1][0]));
    if (tid == 0) {
        sh.st[0] = st0;
        sh.st[1] = st1;
    }
    int round = 0;
    bool dead = false;  // an exchange gave up: finish without further work
    __syncthreads();

    for (;;) {
        bool any = false;
        for (int si = 0; si < NS; ++si) {
            cp_async_wait_all();  // sequence parameters issued by this thread
            StreamSt st = sh.st[si];
            __syncthreads();  // state and parameters visible; everyone has read the state
            if (!st.active) continue;
            any = true;
            unsigned char *tb = tbuf(si), *db = tb + A.slice_bytes;
            const uint32_t lbar = smem_addr(&sh.lbar[si][0]);
            const int b = st.b, i = st.i;
            bool finish = false;
            bool issued_early = false;  // the stream's next unit is already in flight
            if (i == 0) st.flags |= validate_seq(sh, si, g, A.V, DECIDE, MODE == MODE_VERIFY);

            if ((st.flags & ERR_BITS) || dead) {
                finish = true;
                if (dead) st.flags |= F_TIMEOUT;
                if (st.armed) {  // drain the copy before the buffers change hands
                    wait_unit(lbar, st.ph);
                    st.ph ^= 1u;
                    st.armed = 0;
                }
            } else if (MODE == MODE_VERIFY && sh.T[si] == 0.f) {
                // ---- greedy (T = 0): the target's arg max decides
                int tmo = 0;
                if (st.armed) {
                    if (!wait_unit(lbar, st.ph)) tmo = 1;
                    st.ph ^= 1u;
                    st.armed = 0;
                } else if (!A.aligned) {
                    load_slice<Tin, NT>(s, row_ptr<Tin>(A.target, static_cast<size_t>(b) * (g + 1) + i, A.V), tb, 0, false);
                }
                __syncthreads();
                float bv = -INFINITY;
                int bi = -1, bad = tmo ? F_TIMEOUT : 0;
                for (int j = tid; j < s.nvec; j += NT) {
                    float z[VEC];
                    S::unpack(vec_at(tb, j), z);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        const int v = s.lo + j * VEC + e;
                        if (v >= s.hi) break;
                        if (!(z[e] < INFINITY) || z[e] != z[e]) bad |= F_NONFINITE;
                        else if (z[e] > bv) {
                            bv = z[e];
                            bi = v;
                        }
                    }
                }
                block_argmax(sh.tpart, bv, bi, bad);
                float rec[4] = {bv, __int_as_float(bi), __int_as_float(bad), 0.f};
                bool ok;
                const int slot = xchg_round<4>(sh.x, round, rec, C, rank, ok);
                float gv = -INFINITY;
                int gi = -1, gb = ok ? 0 : F_TIMEOUT;
                {
                    const int lane = tid & 31;
                    float v = -INFINITY;
                    int ix = -1, bb = 0;
                    if (lane < C) {
                        v = sh.x.rec[slot][lane][0];
                        ix = __float_as_int(sh.x.rec[slot][lane][1]);
                        bb = __float_as_int(sh.x.rec[slot][lane][2]);
                    }
                    warp_argmax(v, ix);
                    gv = v;
                    gi = ix;
                    gb |= warp_allor(bb);
                }
                (void)gv;
                if (!ok) dead = true;
                if (gi < 0) gb |= F_NONFINITE;
                if (gb) {
                    st.flags |= gb;
                    finish = true;
                } else if (i < g && sh.ids[si][i] == gi) {
                    if (tid == 0) sh.tok[si][st.n] = gi;
                    ++st.n;
                } else {
                    st.stopped = 1;
                    st.drawn = gi;
                    st.writer = 0;
                    finish = true;
                }
                if (!(i < g)) finish = true;
            } else {
                const float T = sh.T[si];
                const float k = LOG2E / T;
                const bool has_d = i < g;
                int tmo = 0;
                const bool split = st.armed;  // the draft slice is waited for after the target's pass
                if (st.armed) {
                    if (!mbar_wait_bounded(lbar, st.ph)) tmo = 1;
                } else if (!A.aligned) {
                    load_slice<Tin, NT>(s, row_ptr<Tin>(A.target, static_cast<size_t>(b) * (g + 1) + i, A.V), tb, 0, false);
                    if (has_d) load_slice<Tin, NT>(s, row_ptr<Tin>(A.draft, static_cast<size_t>(b) * g + i, A.V), db, 0, false);
                    __syncthreads();
                }

                // pass A: online max / normaliser (and entropy sum) per row
                bool nonfin = false;
                Soft at = thread_soft<Tin, STATS, NT>(tb, s.nvec, k, nonfin);
                if (split) {
                    if (!mbar_wait_bounded(lbar + 8u, st.ph)) tmo = 1;
                    st.ph ^= 1u;
                    st.armed = 0;
                }
                Soft ad = !has_d ? soft_empty()
                          : STATS ? draft_soft_at<Tin, NT>(db, s.nvec, k, at.m, nonfin)
                                  : thread_soft<Tin, false, NT>(db, s.nvec, k, nonfin);
                const bool want_y = DECIDE && has_d && !st.stopped;
                const int y = want_y ? sh.ids[si][i] : -1;
                int bad = (nonfin ? F_NONFINITE : 0) | (tmo ? F_TIMEOUT : 0);
                block_soft<STATS>(sh.tpart, at, ad, bad, k);
                float rec[8];
                {
                    float zty = 0.f, zdy = 0.f;
                    int hasy = 0;
                    if (want_y && y >= s.lo && y < s.hi) {
                        zty = S::scalar(tb, y - s.lo);
                        zdy = S::scalar(db, y - s.lo);
                        hasy = 0x100;
                    }
                    rec[0] = at.m;
                    rec[1] = at.s;
                    rec[2] = at.s1;
                    rec[3] = ad.m;
                    rec[4] = ad.s;
                    rec[5] = zty;
                    rec[6] = zdy;
                    rec[7] = __int_as_float(bad | hasy);
                }
                bool ok;
                int slot = xchg_round<8>(sh.x, round, rec, C, rank, ok);
                Soft Ct, Cd;
                int cbits;
                float Zty, Zdy;
                gather_soft<STATS>(sh.x, slot, C, k, Ct, Cd, cbits, Zty, Zdy);
                int rf = cbits | (ok ? 0 : F_TIMEOUT);
                if (!(Ct.m > -INFINITY) || !(Ct.s > 0.f) || !(Ct.s < INFINITY)) rf |= F_NONFINITE;
                if (has_d && (!(Cd.m > -INFINITY) || !(Cd.s > 0.f) || !(Cd.s < INFINITY))) rf |= F_NONFINITE;
                if (!ok) dead = true;
                if (rf) {
                    st.flags |= rf;
                    finish = true;
                } else {
                    const float ct = fmaf(Ct.m, k, log2f(Ct.s));
                    const float cd = has_d ? fmaf(Cd.m, k, log2f(Cd.s)) : 0.f;
                    if (STATS) {
                        if (tid == 0) sh.ent[si][i] = logf(Ct.s) - LN2 * (Ct.s1 / Ct.s);
                        if (has_d) {
                            float acc = 0.f;
                            for (int j = tid; j < s.nvec; j += NT) {
                                float zt[VEC], zd[VEC];
                                S::unpack(vec_at(tb, j), zt);
                                S::unpack(vec_at(db, j), zd);
#pragma unroll
                                for (int e = 0; e < VEC; ++e)
                                    acc += ex2(fminf(fmaf(zt[e], k, -ct), fmaf(zd[e], k, -cd)));
                            }
                            const float part = block_sum(sh.tpart, acc);  // every read of the slices is done
                            // the slices are not needed again unless this position draws
                            // the final token (a rejection here): otherwise the next
                            // position's slices load while the overlap exchange completes
                            bool no_draw = MODE == MODE_STATS || st.stopped;
                            if (DECIDE && !st.stopped) {
                                const float lp = fmaf(Zty, k, -ct), lq = fmaf(Zdy, k, -cd);
                                no_draw = log2f(sh.u[si][i]) + lq < lp;  // the accept test taken below
                            }
                            if (no_draw && !dead) {
                                StreamSt nx = st;
                                nx.i = i + 1;
                                issue_unit<Tin>(A, nx, s, tb, db, lbar);
                                st.armed = nx.armed;
                                issued_early = true;
                            }
                            float r4[4] = {part, 0.f, 0.f, 0.f};
                            const int sl2 = xchg_round<4>(sh.x, round, r4, C, rank, ok);
                            const float a = gather_sum(sh.x, sl2, C);
                            if (tid == 0) sh.alpha[si][i] = a;
                            if (!ok) {
                                dead = true;
                                st.flags |= F_TIMEOUT;
                                finish = true;
                                if (issued_early && st.armed) {  // the early copy lands before the buffers change hands
                                    wait_unit(lbar, st.ph);
                                    st.ph ^= 1u;
                                    st.armed = 0;
                                }
                                issued_early = false;
                            }
                        }
                    }
                    if (DECIDE && !st.stopped && !finish) {
                        const float uf = sh.u[si][g];
                        SampleOut so = {0, 0, -1};
                        if (has_d) {
                            const float lp = fmaf(Zty, k, -ct), lq = fmaf(Zdy, k, -cd);
                            const float u = sh.u[si][i];
                            if (log2f(u) + lq < lp) {
                                if (tid == 0) sh.tok[si][st.n] = y;
                                ++st.n;
                            } else {
                                st.stopped = 1;
                                so = cluster_sample<Tin, 0>(sh, round, tb, db, s, k, ct, cd, uf, C, rank);
                                if (so.status == -2) {
                                    st.flags |= F_ZERO_MASS;
                                    so = cluster_sample<Tin, 1>(sh, round, tb, db, s, k, ct, cd, uf, C, rank);
                                }
                            }
                        } else {
                            st.stopped = 1;
                            so = cluster_sample<Tin, 1>(sh, round, tb, db, s, k, ct, cd, uf, C, rank);
                        }
                        if (st.stopped) {
                            st.drawn = so.token;  // meaningful in the writer CTA
                            st.writer = so.writer;
                            if (so.status == -3) {
                                dead = true;
                                st.flags |= F_TIMEOUT;
                            } else if (so.status < 0) {
                                st.flags |= F_NONFINITE;
                            }
                        }
                    }
                    if (st.flags & ERR_BITS) finish = true;
                    if (!(i < g && (STATS || !st.stopped))) finish = true;
                }
            }

            __syncthreads();  // every read of this stream's slices and shared outputs is done
            if (finish) {
                if (rank == st.writer && tid == 0) {
                    const int f = st.flags;
                    const bool err = (f & ERR_BITS) != 0;
                    if (DECIDE) {
                        for (int j = 0; j <= g; ++j) {
                            int v = -1;
                            if (!err) v = (j < st.n) ? sh.tok[si][j] : (j == st.n ? st.drawn : -1);
                            A.tokens[static_cast<size_t>(b) * (g + 1) + j] = v;
                        }
                        A.accept_len[b] = err ? -1 : st.n;
                    }
                    if (STATS && A.alpha) {
                        for (int j = 0; j < g; ++j) A.alpha[static_cast<size_t>(b) * g + j] = err ? NAN : sh.alpha[si][j];
                        for (int j = 0; j <= g; ++j)
                            A.entropy[static_cast<size_t>(b) * (g + 1) + j] = err ? NAN : sh.ent[si][j];
                    }
                    if (A.flags) A.flags[b] = f;
                }
                st = start_seq(A, sh, si, next_seq, DECIDE, st.ph);
                next_seq += NC;
            } else {
                st.i = i + 1;
            }
            if (st.active && !dead && !issued_early) issue_unit<Tin>(A, st, s, tb, db, lbar);
            if (tid == 0) sh.st[si] = st;
        }
        __syncthreads();
        if (!any) break;
    }

    // Copies that outlived a bounded wait must land before the CTA exits.
    for (int si = 0; si < NS; ++si) {
        const StreamSt st = sh.st[si];
        if (st.armed) wait_unit(smem_addr(&sh.lbar[si][0]), st.ph);
    }
    cluster_sync();  // no CTA leaves while a peer may still push into it
}

const void *row_kernel(int dtype, int mode) {
    if (dtype == 0) {
        if (mode == MODE_VERIFY) return reinterpret_cast<const void *>(&row_kernel_impl<float, MODE_VERIFY>);
        if (mode == MODE_VERIFY_STATS)
            return reinterpret_cast<const void *>(&row_kernel_impl<float, MODE_VERIFY_STATS>);
        return reinterpret_cast<const void *>(&row_kernel_impl<float, MODE_STATS>);
    }
    if (mode == MODE_VERIFY) return reinterpret_cast<const void *>(&row_kernel_impl<bf16_t, MODE_VERIFY>);
    if (mode == MODE_VERIFY_STATS)
        return reinterpret_cast<const void *>(&row_kernel_impl<bf16_t, MODE_VERIFY_STATS>);
    return reinterpret_cast<const void *>(&row_kernel_impl<bf16_t, MODE_STATS>);
}

}  // namespace mtp
