// philox.cuh -- the counter-based generator Philox4x32-10 (Salmon, Moraes,
// Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011) and
// the standard Gumbel noise drawn from it for the Gumbel-max final draw of
// verification ("Breaking Entropy Bounds: Accelerating RL Training via MTP
// with Rejection Sampling", App. G.2 "Gumbel-Max Trick (vLLM)").
//
// Stream layout: key = the caller's 64-bit seed (low word first); counter =
// (v / 4, row, sequence, offset); vocabulary index v takes word v mod 4 of
// the output.  U = (floor(x / 2^8) + 1/2) 2^-24 lies strictly inside (0, 1).
#pragma once

#include <cstdint>

namespace mtp {

// Ten Philox rounds: each multiplies counter words 0 and 2 by the round
// multipliers (64-bit products split into high and low words), mixes the
// high words with words 1 and 3 and the key, and bumps the key by the Weyl
// increments.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        // one widening multiply per product: high and low words together
        const uint64_t pa = static_cast<uint64_t>(0xD2511F53u) * c.x;
        const uint64_t pb = static_cast<uint64_t>(0xCD9E8D57u) * c.z;
        const uint32_t ha = static_cast<uint32_t>(pa >> 32), la = static_cast<uint32_t>(pa);
        const uint32_t hb = static_cast<uint32_t>(pb >> 32), lb = static_cast<uint32_t>(pb);
        c = make_uint4(hb ^ c.y ^ k0, lb, ha ^ c.w ^ k1, la);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

// Gumbel noise in log2 units up to a constant: -log2(-log2 U) =
// G log2(e) + log2(ln 2) for G = -ln(-ln U).  The constant is the same for
// every index, so arg max_v [log2 w_v + gumbel2(x_v)] is the Gumbel-max draw.
//
// Single precision cannot hold U itself near 1 (1 - 2^-25 rounds to 1 and
// the noise would come out infinite), but it holds exactly whichever of U
// and W = 1 - U is at most 1/2: with m = floor(x / 2^8), U = (m + 1/2) 2^-24
// for m < 2^23, and W = (2^24 - 1 - m + 1/2) 2^-24 otherwise.  Then
// -log2 U = -log2(t) on the lower half; on the upper half
// -log2(1 - W) = log2(e) (W + W^2/2 + W^3/3 + ...), taken as its first two
// terms when W < 2^-7 and as -log2 of 1 - W rounded to single precision
// otherwise.  Either keeps the noise within 4e-5 of its exact value: the
// series' relative error is below W^2 / 3 < 2e-5, and rounding 1 - W (by at
// most 2^-25) moves -log2(1 - W) >= 0.011 by under 8e-6 of itself.
__device__ __forceinline__ float gumbel2(uint32_t x) {
    const uint32_t m = x >> 8;
    const bool hi = m >= (1u << 23);
    const float t = (__uint2float_rn(hi ? (1u << 24) - 1u - m : m) + 0.5f) * 5.9604644775390625e-8f;  // exact
    const float lg = -__log2f(hi ? 1.f - t : t);
    const float series = t * fmaf(t, 0.72134752044448170f, 1.4426950408889634f);  // log2(e) (t + t^2 / 2)
    const float L = (hi && t < 0.0078125f) ? series : lg;  // -log2 U > 0
    return -__log2f(L);
}

}  // namespace mtp
