// chunk_math.cuh -- per-lane arithmetic on chunks of logit rows held in
// registers, shared by the streaming kernels: loading a chunk from its ring
// slot, the chunk maximum, the branch-free online softmax fold and the
// running and warp-wide arg max.
//
// A chunk row is CV = 32 * QV 16-byte vectors; lane l holds vectors
// q * 32 + l (q < QV).
#pragma once

#include "common.cuh"

namespace mtp {

// Bit pattern of four (float) or eight (bf16) -inf logits in one 32-bit word.
template <typename Tin>
struct NegInf;
template <>
struct NegInf<float> {
    static constexpr uint32_t w = 0xff800000u;
};
template <>
struct NegInf<bf16_t> {
    static constexpr uint32_t w = 0xff80ff80u;
};

// This lane's vectors q * 32 + lane (q < QV) of one chunk row, -inf beyond
// the chunk's `cnt` vectors unless FULL.
template <typename Tin, bool FULL, int QV>
__device__ __forceinline__ void load_chunk(const unsigned char *buf, int cnt, int lane, uint4 (&r)[QV]) {
    const uint4 NEG = make_uint4(NegInf<Tin>::w, NegInf<Tin>::w, NegInf<Tin>::w, NegInf<Tin>::w);
#pragma unroll
    for (int q = 0; q < QV; ++q) {
        const int j = q * 32 + lane;
        r[q] = (FULL || j < cnt) ? vec_at(buf, j) : NEG;
    }
}

// Element e (0 <= e < VEC) of a 16-byte vector of logits, as float.
template <typename Tin>
__device__ __forceinline__ float vec_elem(const uint4 &v, int e) {
    if (Store<Tin>::ES == 4) {
        const uint32_t w = e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
        return __uint_as_float(w);
    }
    const int wi = e >> 1;
    const uint32_t w = wi == 0 ? v.x : wi == 1 ? v.y : wi == 2 ? v.z : v.w;
    return __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
}

// Maximum over the chunk row's elements held by this lane (NaN if any is).
template <typename Tin, int QV>
__device__ __forceinline__ float chunk_max(const uint4 (&r)[QV]) {
    if constexpr (Store<Tin>::ES == 2) {
        uint32_t a = bmax2_nan(r[0].x, r[0].y), b = bmax2_nan(r[0].z, r[0].w);
#pragma unroll
        for (int q = 1; q < QV; ++q) {
            a = bmax2_nan(a, bmax2_nan(r[q].x, r[q].y));
            b = bmax2_nan(b, bmax2_nan(r[q].z, r[q].w));
        }
        a = bmax2_nan(a, b);
        return max_nan(__uint_as_float(a << 16), __uint_as_float(a & 0xffff0000u));
    } else {
        float a = max_nan(__uint_as_float(r[0].x), __uint_as_float(r[0].y));
        float b = max_nan(__uint_as_float(r[0].z), __uint_as_float(r[0].w));
#pragma unroll
        for (int q = 1; q < QV; ++q) {
            a = max_nan(a, max_nan(__uint_as_float(r[q].x), __uint_as_float(r[q].y)));
            b = max_nan(b, max_nan(__uint_as_float(r[q].z), __uint_as_float(r[q].w)));
        }
        return max_nan(a, b);
    }
}

// Fold one chunk row (its lane maximum cmx from chunk_max) into the lane's
// running softmax partial without branches: exact running maximum m (a NaN
// or +inf sets `bad`, the values that follow are then meaningless),
// s = sum 2^{z k - m k}.  Returns the chunk's own sum relative to the
// updated m.
template <typename Tin, int QV>
__device__ __forceinline__ float fold_regs(const uint4 (&r)[QV], float cmx, float k, float &m, float &s, int &bad) {
    using St = Store<Tin>;
    bad |= !(cmx < INFINITY);
    const float nm = fmaxf(m, cmx);
    const float mr = nm > -INFINITY ? nm : 0.f;  // all -inf so far: any finite reference
    s *= ex2((m - mr) * k);
    m = nm;
    const float mk = mr * k;
    // element pairs on the packed f32x2 pipe: one FMA and one add per pair
    const uint64_t K2 = f2pack(k, k), NMK2 = f2pack(-mk, -mk);
    uint64_t acc0 = f2pack(0.f, 0.f), acc1 = f2pack(0.f, 0.f);
#pragma unroll
    for (int q = 0; q < QV; ++q) {
        const uint32_t w[4] = {r[q].x, r[q].y, r[q].z, r[q].w};
#pragma unroll
        for (int h = 0; h < 4; h += 2) {
            uint64_t z0, z1;
            if (St::ES == 2) {
                z0 = bf16pair_f2(w[h]);
                z1 = bf16pair_f2(w[h + 1]);
            } else {
                z0 = f2pack(__uint_as_float(w[h]), __uint_as_float(w[h + 1]));
                z1 = 0;
            }
            float d0, d1;
            f2unpack(f2fma(z0, K2, NMK2), d0, d1);
            acc0 = f2add(acc0, f2pack(ex2(d0), ex2(d1)));
            if (St::ES == 2) {
                f2unpack(f2fma(z1, K2, NMK2), d0, d1);
                acc1 = f2add(acc1, f2pack(ex2(d0), ex2(d1)));
            }
        }
    }
    float a0, a1, b0, b1;
    f2unpack(acc0, a0, a1);
    f2unpack(acc1, b0, b1);
    const float cs = (a0 + a1) + (b0 + b1);
    s += cs;
    return cs;
}

// Fold one chunk row into the lane's running partial with the entropy sum:
// exact running maximum m (NaN or +inf sets `bad`), s = sum 2^{d},
// s1 = sum 2^{d} d with d = z k - m k (clamped at -256 so that -inf logits
// add exactly zero).
template <typename Tin, int QV>
__device__ __forceinline__ void fold_ent(const uint4 (&r)[QV], float cmx, float k, float &m, float &s, float &s1,
                                         int &bad) {
    using St = Store<Tin>;
    bad |= !(cmx < INFINITY);
    const float nm = fmaxf(m, cmx);
    const float mr = nm > -INFINITY ? nm : 0.f;
    const float dl = (mr - m) * k;  // +inf while nothing finite was seen (s == 0)
    const float sc = ex2(-dl);
    s1 = (s != 0.f) ? sc * fmaf(-dl, s, s1) : 0.f;
    s *= sc;
    m = nm;
    const float mk = mr * k;
    const uint64_t K2 = f2pack(k, k), NMK2 = f2pack(-mk, -mk);
    uint64_t as = f2pack(0.f, 0.f), a1 = f2pack(0.f, 0.f);
#pragma unroll
    for (int q = 0; q < QV; ++q) {
        const uint32_t w[4] = {r[q].x, r[q].y, r[q].z, r[q].w};
#pragma unroll
        for (int h = 0; h < (St::ES == 2 ? 4 : 2); ++h) {
            const uint64_t z2 = St::ES == 2 ? bf16pair_f2(w[h])
                                            : f2pack(__uint_as_float(w[2 * h]), __uint_as_float(w[2 * h + 1]));
            float d0, d1;
            f2unpack(f2fma(z2, K2, NMK2), d0, d1);
            d0 = fmaxf(d0, -256.f);
            d1 = fmaxf(d1, -256.f);
            const uint64_t e2 = f2pack(ex2(d0), ex2(d1));
            as = f2add(as, e2);
            a1 = f2fma(e2, f2pack(d0, d1), a1);
        }
    }
    float x0, x1, y0, y1;
    f2unpack(as, x0, x1);
    f2unpack(a1, y0, y1);
    s += x0 + x1;
    s1 += y0 + y1;
}

// Running arg max of one chunk row kept warp-uniform: the warp maximum of
// the lanes' chunk maxima (cmx from chunk_max; a NaN or +inf lane takes no
// part, it is flagged elsewhere) replaces (m, idx, x) only when it exceeds
// m, so an equal value in a later chunk keeps the earlier index.  Then only
// the lanes holding the new maximum look for it, each finds its first
// element equal to it, and the smallest such index wins (first index among
// equals in ascending vocabulary order).  A per-lane running arg max would
// scan a chunk whenever any lane's own maximum rises, which early in a row is
// almost every chunk; the warp maximum rises far less often.  vbase:
// vocabulary index of this lane's first vector in the chunk.  With OTHER, x
// receives the other row's logit at the new arg max.
template <typename Tin, int QV, bool OTHER>
__device__ __forceinline__ void argmax_warp(const uint4 (&r)[QV], const uint4 (&o)[QV], float cmx, int vbase,
                                            float &m, int &idx, float &x) {
    constexpr int VEC = Store<Tin>::VEC;
    const float c = (cmx < INFINITY) ? cmx : -INFINITY;  // NaN and +inf: no part
    float wm = c;
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) wm = fmaxf(wm, __shfl_xor_sync(FULL, wm, o2));
    if (!(wm > m)) return;  // warp-uniform
    int li = 0x7fffffff;
    float lx = 0.f;
    if (c == wm) {
        bool found = false;
#pragma unroll
        for (int q = 0; q < QV; ++q) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                if (!found && vec_elem<Tin>(r[q], e) == wm) {
                    found = true;
                    li = (vbase + q * 32) * VEC + e;
                    if (OTHER) lx = vec_elem<Tin>(o[q], e);
                }
            }
        }
    }
    int mi = li;
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) mi = min(mi, __shfl_xor_sync(FULL, mi, o2));
    const int src = __ffs(__ballot_sync(FULL, li == mi)) - 1;
    if (OTHER) x = __shfl_sync(FULL, lx, src);
    idx = mi;
    m = wm;
}

// Arg max across the warp: the largest value, ties to the smallest index
// (index -1: no element); `x` travels with the winner.  Same result in every
// lane.
__device__ __forceinline__ void argmax_allreduce(float &v, int &i, float &x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(FULL, v, o), ox = __shfl_xor_sync(FULL, x, o);
        const int oi = __shfl_xor_sync(FULL, i, o);
        if (oi >= 0 && (i < 0 || ov > v || (ov == v && oi < i))) {
            v = ov;
            i = oi;
            x = ox;
        }
    }
}

__device__ __forceinline__ void argmax_merge(float &v, int &i, float &x, float ov, int oi, float ox) {
    if (oi >= 0 && (i < 0 || ov > v || (ov == v && oi < i))) {
        v = ov;
        i = oi;
        x = ox;
    }
}

// ------------------------------------------- TV loss: overlap and gradient --

// Fold every word of the lane's chunk registers into one value.  Consuming
// the registers completes the shared-memory loads that filled them, so the
// slot can be handed back to the producer before the chunk is processed.
template <int QV>
__device__ __forceinline__ uint32_t consume_regs(const uint4 (&r)[QV]) {
    uint32_t x = 0;
#pragma unroll
    for (int q = 0; q < QV; ++q) x ^= r[q].x ^ r[q].y ^ r[q].z ^ r[q].w;
    return x;
}

// Merge two softmax partials (m, s); a NaN sum propagates.
__device__ __forceinline__ Soft soft_pair_merge(const Soft &a, const Soft &b, float k) {
    Soft r;
    r.m = fmaxf(a.m, b.m);
    r.s = 0.f;
    r.s1 = 0.f;
    if (a.s != 0.f) r.s += a.s * ex2((a.m - r.m) * k);
    if (b.s != 0.f) r.s += b.s * ex2((b.m - r.m) * k);
    return r;
}

// One lane's partial overlap sums over one chunk (registers): alpha =
// sum 2^{min(lp, lq)}, S = sum over lq <= lp of the same, and the indicator
// byte of each vector (bit e: q <= p for element e).
template <typename Tin, int QV>
__device__ __forceinline__ void ovl_regs(const uint4 (&rt)[QV], const uint4 (&rd)[QV], float k, float ct, float cd,
                                         float &acc_a, float &acc_s, uint32_t (&m)[QV]) {
    const uint64_t K2 = f2pack(k, k), NCT = f2pack(-ct, -ct), NCD = f2pack(-cd, -cd);
    uint64_t aa = f2pack(0.f, 0.f), as = f2pack(0.f, 0.f);
#pragma unroll
    for (int q = 0; q < QV; ++q) {
        const uint32_t wt[4] = {rt[q].x, rt[q].y, rt[q].z, rt[q].w}, wd[4] = {rd[q].x, rd[q].y, rd[q].z, rd[q].w};
        uint32_t bb = 0;
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
            const float x0 = ex2(fminf(lp0, lq0)), x1 = ex2(fminf(lp1, lq1));
            const bool b0 = lq0 <= lp0, b1 = lq1 <= lp1;
            aa = f2add(aa, f2pack(x0, x1));
            as = f2add(as, f2pack(b0 ? x0 : 0.f, b1 ? x1 : 0.f));
            bb |= (b0 ? 1u : 0u) << (2 * h);
            bb |= (b1 ? 1u : 0u) << (2 * h + 1);
        }
        m[q] = bb;
    }
    float a0, a1, s0, s1;
    f2unpack(aa, a0, a1);
    f2unpack(as, s0, s1);
    acc_a += a0 + a1;
    acc_s += s0 + s1;
}

// 32-byte streaming store of eight floats (one 256-bit store instruction:
// a warp writes 1 KB contiguous, half the store instructions of two 16-byte
// stores).  `out` must be 32-byte aligned.
__device__ __forceinline__ void stcs_v8(float *out, const float (&g)[8]) {
    asm volatile("st.global.cs.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(out), "f"(g[0]), "f"(g[1]),
                 "f"(g[2]), "f"(g[3]), "f"(g[4]), "f"(g[5]), "f"(g[6]), "f"(g[7])
                 : "memory");
}

// Gradient of one 16-byte draft vector: out[e] = 2^{z_e k - cd} (bit e ? on : off).
// W32: `out` is 32-byte aligned (bf16 rows then take one 256-bit store).
template <typename Tin, bool W32 = false>
__device__ __forceinline__ void grad_vec(const uint4 &r, uint32_t m, float k, float cd, float on, float off,
                                         float *out) {
    const uint64_t K2 = f2pack(k, k), NCD = f2pack(-cd, -cd);
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
    if (Store<Tin>::ES == 2) {
        float g[8];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            float d0, d1;
            f2unpack(f2fma(bf16pair_f2(w[h]), K2, NCD), d0, d1);
            g[2 * h] = ex2(d0) * ((m >> (2 * h)) & 1u ? on : off);
            g[2 * h + 1] = ex2(d1) * ((m >> (2 * h + 1)) & 1u ? on : off);
        }
        if (W32) {
            stcs_v8(out, g);
        } else {
            __stcs(reinterpret_cast<float4 *>(out), make_float4(g[0], g[1], g[2], g[3]));
            __stcs(reinterpret_cast<float4 *>(out) + 1, make_float4(g[4], g[5], g[6], g[7]));
        }
    } else {
        float d0, d1, d2, d3;
        f2unpack(f2fma(f2pack(__uint_as_float(w[0]), __uint_as_float(w[1])), K2, NCD), d0, d1);
        f2unpack(f2fma(f2pack(__uint_as_float(w[2]), __uint_as_float(w[3])), K2, NCD), d2, d3);
        __stcs(reinterpret_cast<float4 *>(out),
               make_float4(ex2(d0) * (m & 1u ? on : off), ex2(d1) * (m & 2u ? on : off),
                           ex2(d2) * (m & 4u ? on : off), ex2(d3) * (m & 8u ? on : off)));
    }
}

}  // namespace mtp
