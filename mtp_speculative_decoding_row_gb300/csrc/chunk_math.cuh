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

}  // namespace mtp
