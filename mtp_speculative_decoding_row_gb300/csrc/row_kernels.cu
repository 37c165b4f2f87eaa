// row_kernels.cu -- batched MTP rejection-sampling verification and
// per-position row statistics on sm_103a.
//
// One thread-block cluster of C CTAs per sequence.  For each position the
// cluster bulk-loads the target row (and the draft row) slice by slice into
// shared memory, forms the temperature-scaled softmax normalisers with an
// online max/sum pass, combines the CTA partials through DSMEM, and then
// (method: "Breaking Entropy Bounds: Accelerating RL Training via MTP with
// Rejection Sampling", §2 "Acceptance methods" and App. G.1; "EntMTP",
// Related Work "Speculative Decoding"):
//   - accepts draft y_i iff u_i q_i(y_i) < p_i(y_i), tested as
//     log2 u_i + log2 q_i(y_i) < log2 p_i(y_i);
//   - at the first rejection draws the replacement from norm(max(0, p - q))
//     by a two-pass inverse CDF over the slices still held on chip;
//   - after gamma accepts draws the bonus token from p_gamma the same way;
//   - optionally forms alpha_i = sum_v min(p_i, q_i) (§3, §8) and
//     H(p_i) = -sum_v p log p for every position.
// Rows after the stop are never loaded unless statistics are requested.
#include <cstddef>

#include "common.cuh"
#include "kernels.h"

namespace mtp {

struct alignas(16) Rec {
    float tm, ts, ts1, dm, ds, zty, zdy, x0;
    int hasy, bad, tok, pad0;
    float x1, pad1, pad2, pad3;
};
static_assert(sizeof(Rec) == 64, "record layout");

struct RowShared {
    Rec rec[2];               // cluster exchange slots (alternating)
    float wred[NW][8];        // per-warp partials
    float comb[8];            // cluster-combined values (broadcast)
    int combi[4];
    float segtot[NW];         // per-warp CDF segment totals
    float ctatot[MAX_C];      // per-CTA residual totals (rank order)
    float sampf[4];
    int sampi[8];
    int tok[MAX_GAMMA + 1];   // accepted draft ids
    float alpha[MAX_GAMMA];
    float ent[MAX_GAMMA + 1];
    unsigned long long bar[2];
};
static_assert(sizeof(RowShared) <= HDR_BYTES, "shared header too large");

// ------------------------------------------------------------ combines -----

// Block + cluster combine of the target/draft softmax partials and of the
// logits at the draft id (held by exactly one CTA).  Results in all threads.
template <bool ENT>
__device__ __forceinline__ void combine_soft(RowShared &sh, Soft at, Soft ad, int bad, float zty, float zdy,
                                             int hasy, float k, int &slot, int C, Soft &Ct, Soft &Cd, int &cbad,
                                             float &Zty, float &Zdy) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    at = soft_warp_allreduce<ENT>(at, k);
    ad = soft_warp_allreduce<false>(ad, k);
    bad = warp_allor(bad);
    if (lane == 0) {
        float *w = sh.wred[warp];
        w[0] = at.m;
        w[1] = at.s;
        w[2] = at.s1;
        w[3] = ad.m;
        w[4] = ad.s;
        w[5] = __int_as_float(bad);
    }
    __syncthreads();
    if (warp == 0) {
        Soft a = soft_empty(), d = soft_empty();
        int bb = 0;
        if (lane < NW) {
            const float *w = sh.wred[lane];
            a = {w[0], w[1], w[2]};
            d = {w[3], w[4], 0.f};
            bb = __float_as_int(w[5]);
        }
        a = soft_warp_allreduce<ENT>(a, k);
        d = soft_warp_allreduce<false>(d, k);
        bb = warp_allor(bb);
        if (lane == 0) {
            Rec &r = sh.rec[slot];
            r.tm = a.m;
            r.ts = a.s;
            r.ts1 = a.s1;
            r.dm = d.m;
            r.ds = d.s;
            r.zty = zty;
            r.zdy = zdy;
            r.hasy = hasy;
            r.bad = bb;
        }
    }
    cluster_sync();
    if (warp == 0) {
        Soft a = soft_empty(), d = soft_empty();
        int bb = 0, hy = 0;
        float zt = 0.f, zd = 0.f;
        if (lane < C) {
            const uint32_t base = map_rank(smem_addr(&sh.rec[slot]), lane);
            a.m = ld_cluster_f32(base + offsetof(Rec, tm));
            a.s = ld_cluster_f32(base + offsetof(Rec, ts));
            a.s1 = ld_cluster_f32(base + offsetof(Rec, ts1));
            d.m = ld_cluster_f32(base + offsetof(Rec, dm));
            d.s = ld_cluster_f32(base + offsetof(Rec, ds));
            zt = ld_cluster_f32(base + offsetof(Rec, zty));
            zd = ld_cluster_f32(base + offsetof(Rec, zdy));
            hy = ld_cluster_s32(base + offsetof(Rec, hasy));
            bb = ld_cluster_s32(base + offsetof(Rec, bad));
        }
        a = soft_warp_allreduce<ENT>(a, k);
        d = soft_warp_allreduce<false>(d, k);
        bb = warp_allor(bb);
        const unsigned hm = __ballot_sync(FULL, hy != 0);
        const int src = hm ? (__ffs(hm) - 1) : 0;
        zt = __shfl_sync(FULL, zt, src);
        zd = __shfl_sync(FULL, zd, src);
        if (lane == 0) {
            sh.comb[0] = a.m;
            sh.comb[1] = a.s;
            sh.comb[2] = a.s1;
            sh.comb[3] = d.m;
            sh.comb[4] = d.s;
            sh.comb[5] = zt;
            sh.comb[6] = zd;
            sh.combi[0] = bb;
        }
    }
    __syncthreads();
    Ct = {sh.comb[0], sh.comb[1], sh.comb[2]};
    Cd = {sh.comb[3], sh.comb[4], 0.f};
    Zty = sh.comb[5];
    Zdy = sh.comb[6];
    cbad = sh.combi[0];
    slot ^= 1;
}

// Block + cluster sum of one value; result in all threads.
__device__ __forceinline__ float cluster_sum(RowShared &sh, float v, int &slot, int C) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    v = warp_allsum(v);
    if (lane == 0) sh.wred[warp][0] = v;
    __syncthreads();
    if (warp == 0) {
        float x = (lane < NW) ? sh.wred[lane][0] : 0.f;
        x = warp_allsum(x);
        if (lane == 0) sh.rec[slot].x0 = x;
    }
    cluster_sync();
    if (warp == 0) {
        float x = (lane < C) ? ld_cluster_f32(map_rank(smem_addr(&sh.rec[slot].x0), lane)) : 0.f;
        x = warp_allsum(x);
        if (lane == 0) sh.comb[7] = x;
    }
    __syncthreads();
    slot ^= 1;
    return sh.comb[7];
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

// Two-pass inverse CDF over the whole row held by the cluster: pass one
// forms the per-warp, per-CTA and total masses; the draw is the smallest
// vocabulary index whose running sum exceeds u * R (ascending index order:
// CTA rank, warp segment, 32-vector round, lane, element).  If rounding
// leaves no such index, the last index with positive weight in the selected
// unit is taken.  Returns the token in every thread, or -2 when R == 0.
template <typename Tin, int WMODE>
__device__ int cluster_sample(RowShared &sh, const unsigned char *tb, const unsigned char *db, const Slice &s,
                              float k, float ct, float cd, float u, int &slot, int C, int rank) {
    constexpr int VEC = Store<Tin>::VEC;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nvw = (s.nvec + NW - 1) / NW;
    const int a0 = min(s.nvec, warp * nvw), a1 = min(s.nvec, a0 + nvw);

    // pass one: segment totals
    float run = 0.f;
    for (int base = a0; base < a1; base += 32) {
        const int j = base + lane;
        float vs = 0.f;
        if (j < a1) {
            float w[VEC];
            vec_weights<Tin, WMODE>(tb, db, j, k, ct, cd, w);
            vs = vec_sum<VEC>(w);
        }
        const float inc = warp_incl_scan(vs);
        run += __shfl_sync(FULL, inc, 31);
    }
    if (lane == 0) sh.segtot[warp] = run;
    __syncthreads();
    if (tid == 0) {
        float tot = 0.f;
        for (int w = 0; w < NW; ++w) tot += sh.segtot[w];
        sh.rec[slot].x0 = tot;
    }
    cluster_sync();
    if (warp == 0) {
        if (lane < C) sh.ctatot[lane] = ld_cluster_f32(map_rank(smem_addr(&sh.rec[slot].x0), lane));
        __syncwarp();
        if (lane == 0) {
            float R = 0.f;
            for (int r = 0; r < C; ++r) R += sh.ctatot[r];
            int rs = -1, last = 0;
            float rem = u * R;
            if (R > 0.f) {
                for (int r = 0; r < C; ++r) {
                    const float vr = sh.ctatot[r];
                    if (vr > rem) {
                        rs = r;
                        break;
                    }
                    rem -= vr;
                }
                if (rs < 0) {
                    last = 1;
                    for (int r = 0; r < C; ++r)
                        if (sh.ctatot[r] > 0.f) rs = r;
                }
            }
            sh.sampi[0] = rs;
            sh.sampi[1] = last;
            sh.sampf[0] = rem;
        }
    }
    __syncthreads();
    slot ^= 1;
    const int rs = sh.sampi[0];
    if (rs < 0) return -2;

    int found = -1;
    if (rank == rs) {
        if (tid == 0) {
            int lm = sh.sampi[1];
            float rem = sh.sampf[0];
            int ws = -1;
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
            sh.sampi[2] = ws;
            sh.sampi[3] = lm;
            sh.sampf[1] = rem;
        }
        __syncthreads();
        const int ws = sh.sampi[2];
        if (warp == ws) {
            int lm = sh.sampi[3];
            float rem = sh.sampf[1];
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
                    const float tot = __shfl_sync(FULL, inc, 31);
                    if (tot > rem) {
                        const unsigned bal = __ballot_sync(FULL, inc > rem);
                        const int L = __ffs(bal) - 1;
                        float exc = __shfl_up_sync(FULL, inc, 1);
                        if (lane == 0) exc = 0.f;
                        int t = -1;
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
                            t = s.lo + j * VEC + ef;
                        }
                        tok = __shfl_sync(FULL, t, L);
                        break;
                    }
                    rem -= tot;
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
            if (lane == 0) sh.sampi[4] = tok;
        }
        __syncthreads();
        found = sh.sampi[4];
    }
    // publish the token to every CTA
    if (tid == 0) sh.rec[slot].tok = (rank == rs) ? found : -1;
    cluster_sync();
    if (warp == 0) {
        int t = (lane < C) ? ld_cluster_s32(map_rank(smem_addr(&sh.rec[slot].tok), lane)) : -1;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t = max(t, __shfl_xor_sync(FULL, t, o));
        if (lane == 0) sh.sampi[5] = t;
    }
    __syncthreads();
    slot ^= 1;
    return sh.sampi[5];
}

// ---------------------------------------------------------------- kernel ---

template <typename Tin, int MODE>
__global__ void __launch_bounds__(NT, 2) row_kernel_impl(const VerifyArgs A) {
    using S = Store<Tin>;
    constexpr int VEC = S::VEC, ES = S::ES;
    constexpr bool STATS = (MODE != MODE_VERIFY);
    constexpr bool DECIDE = (MODE != MODE_STATS);
    extern __shared__ __align__(128) unsigned char smem[];
    RowShared &sh = *reinterpret_cast<RowShared *>(smem);
    unsigned char *tb = smem + HDR_BYTES;
    unsigned char *db = tb + A.slice_bytes;

    const int tid = threadIdx.x;
    const int C = static_cast<int>(cluster_size());
    const int rank = static_cast<int>(cluster_rank());
    const int b = static_cast<int>(cluster_id_x());
    const int g = A.gamma, V = A.V;
    const uint32_t bar_t = smem_addr(&sh.bar[0]), bar_d = smem_addr(&sh.bar[1]);
    if (tid == 0) {
        mbar_init(bar_t, 1);
        mbar_init(bar_d, 1);
        fence_mbar_init();
    }

    // Argument checks that are the same in every CTA of the cluster.
    const float T = A.temp[b];
    int flags = 0;
    if (!(T > 0.f) || !(T < INFINITY)) flags |= F_BAD_TEMP;
    if (DECIDE) {
        for (int i = 0; i < g; ++i) {
            const int y = A.ids[static_cast<size_t>(b) * g + i];
            if (y < 0 || y >= V) flags |= F_BAD_ID;
        }
        for (int i = 0; i <= g; ++i) {
            const float u = A.unif[static_cast<size_t>(b) * (g + 1) + i];
            if (!(u >= 0.f && u < 1.f)) flags |= F_BAD_UNIFORM;
        }
    }
    __syncthreads();
    cluster_sync();  // every CTA has started: DSMEM is safe from here on

    const float k = LOG2E / T;
    const Slice s = make_slice<Tin>(V, C, rank);
    int slot = 0, n = 0, drawn = -1;
    uint32_t ph_t = 0, ph_d = 0;
    bool stopped = false, pend_t = false, pend_d = false;

    if (!flags) {
        for (int i = 0; i <= g; ++i) {
            if (!STATS && stopped) break;
            const bool has_d = i < g;
            const unsigned char *trow = reinterpret_cast<const unsigned char *>(A.target) +
                                        (static_cast<size_t>(b) * (g + 1) + i) * static_cast<size_t>(V) * ES;
            const unsigned char *drow = reinterpret_cast<const unsigned char *>(A.draft) +
                                        (static_cast<size_t>(b) * g + i) * static_cast<size_t>(V) * ES;
            fence_proxy_async();
            const bool arm_t = load_slice<Tin>(s, trow, tb, bar_t, A.aligned != 0);
            const bool arm_d = has_d && load_slice<Tin>(s, drow, db, bar_d, A.aligned != 0);
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

            // pass A: online max / normaliser (and entropy sum) per row
            Soft at = soft_empty(), ad = soft_empty();
            bool nonfin = false;
            for (int j = tid; j < s.nvec; j += NT) {
                float zt[VEC];
                S::unpack(vec_at(tb, j), zt);
                soft_add<VEC, STATS>(at, zt, k, nonfin);
                if (has_d) {
                    float zd[VEC];
                    S::unpack(vec_at(db, j), zd);
                    soft_add<VEC, false>(ad, zd, k, nonfin);
                }
            }
            const bool want_y = DECIDE && has_d && !stopped;
            const int y = want_y ? A.ids[static_cast<size_t>(b) * g + i] : -1;
            float zty = 0.f, zdy = 0.f;
            int hasy = 0;
            if (tid == 0 && want_y && y >= s.lo && y < s.hi) {
                zty = S::scalar(tb, y - s.lo);
                zdy = S::scalar(db, y - s.lo);
                hasy = 1;
            }
            Soft Ct, Cd;
            int cbad;
            float Zty, Zdy;
            combine_soft<STATS>(sh, at, ad, (nonfin ? F_NONFINITE : 0) | (tmo ? F_TIMEOUT : 0), zty, zdy, hasy,
                                k, slot, C, Ct, Cd, cbad, Zty, Zdy);
            int rf = cbad;
            if (!(Ct.m > -INFINITY) || !(Ct.s > 0.f) || !(Ct.s < INFINITY)) rf |= F_NONFINITE;
            if (has_d && (!(Cd.m > -INFINITY) || !(Cd.s > 0.f) || !(Cd.s < INFINITY))) rf |= F_NONFINITE;
            if (rf) {
                flags |= rf;
                break;
            }
            const float ct = fmaf(Ct.m, k, log2f(Ct.s));
            const float cd = has_d ? fmaf(Cd.m, k, log2f(Cd.s)) : 0.f;

            if (STATS) {
                if (tid == 0) sh.ent[i] = logf(Ct.s) - LN2 * (Ct.s1 / Ct.s);
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
                    const float a = cluster_sum(sh, acc, slot, C);
                    if (tid == 0) sh.alpha[i] = a;
                }
            }

            if (DECIDE && !stopped) {
                const float uf = A.unif[static_cast<size_t>(b) * (g + 1) + g];
                if (has_d) {
                    const float lp = fmaf(Zty, k, -ct), lq = fmaf(Zdy, k, -cd);
                    const float u = A.unif[static_cast<size_t>(b) * (g + 1) + i];
                    if (log2f(u) + lq < lp) {
                        if (tid == 0) sh.tok[n] = y;
                        ++n;
                    } else {
                        stopped = true;
                        int t = cluster_sample<Tin, 0>(sh, tb, db, s, k, ct, cd, uf, slot, C, rank);
                        if (t == -2) {
                            flags |= F_ZERO_MASS;
                            t = cluster_sample<Tin, 1>(sh, tb, db, s, k, ct, cd, uf, slot, C, rank);
                        }
                        drawn = t;
                    }
                } else {
                    stopped = true;
                    drawn = cluster_sample<Tin, 1>(sh, tb, db, s, k, ct, cd, uf, slot, C, rank);
                }
                if (stopped && drawn < 0) {
                    flags |= F_NONFINITE;
                    break;
                }
            }
            __syncthreads();  // every read of the slices is done before they are reloaded
        }
    }

    // A copy that outlived its wait must land before this CTA may exit.
    if (pend_t) mbar_wait_bounded(bar_t, ph_t ^ 1);
    if (pend_d) mbar_wait_bounded(bar_d, ph_d ^ 1);

    if (rank == 0 && tid == 0) {
        const bool err = (flags & (F_NONFINITE | F_BAD_ID | F_BAD_TEMP | F_BAD_UNIFORM | F_TIMEOUT)) != 0;
        if (DECIDE) {
            for (int j = 0; j <= g; ++j) {
                int v = -1;
                if (!err) v = (j < n) ? sh.tok[j] : (j == n ? drawn : -1);
                A.tokens[static_cast<size_t>(b) * (g + 1) + j] = v;
            }
            A.accept_len[b] = err ? -1 : n;
        }
        if (STATS && A.alpha) {
            for (int i = 0; i < g; ++i) A.alpha[static_cast<size_t>(b) * g + i] = err ? NAN : sh.alpha[i];
            for (int i = 0; i <= g; ++i) A.entropy[static_cast<size_t>(b) * (g + 1) + i] = err ? NAN : sh.ent[i];
        }
        if (A.flags) A.flags[b] = flags;
    }
    cluster_sync();  // no CTA leaves while a peer may still read its shared memory
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
