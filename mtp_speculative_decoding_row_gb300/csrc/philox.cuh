// philox.cuh -- the counter-based generator Philox4x32-10 (Salmon, Moraes,
// Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011) and
// the standard Gumbel noise drawn from it for the Gumbel-max final draw of
// verification ("Breaking Entropy Bounds: Accelerating RL Training via MTP
// with Rejection Sampling", App. G.2 "Gumbel-Max Trick (vLLM)").
//
// Stream layout: key = the caller's 64-bit seed (low word first); counter =
// (v / 4, row, sequence, offset); vocabulary index v takes word v mod 4 of
// the output.  U = (floor(x / 2^8) + 1/2) 2^-24 is exact in float and lies
// strictly inside (0, 1).
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
        const uint32_t a = c.x, b = c.z;
        const uint32_t ha = __umulhi(0xD2511F53u, a), la = 0xD2511F53u * a;
        const uint32_t hb = __umulhi(0xCD9E8D57u, b), lb = 0xCD9E8D57u * b;
        c = make_uint4(hb ^ c.y ^ k0, lb, ha ^ c.w ^ k1, la);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

// Gumbel noise in log2 units up to a constant: -log2(-log2 U) =
// G log2(e) + log2(ln 2) for G = -ln(-ln U).  The constant is the same for
// every index, so arg max_v [log2 w_v + gumbel2(x_v)] is the Gumbel-max draw.
__device__ __forceinline__ float gumbel2(uint32_t x) {
    const float u = (__uint2float_rn(x >> 8) + 0.5f) * 5.9604644775390625e-8f;  // 2^-24
    return -__log2f(-__log2f(u));
}

}  // namespace mtp
