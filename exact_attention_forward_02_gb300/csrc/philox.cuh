// philox.cuh -- the dropout mask of libfa: Philox-4x32-10 and the 15-bit keep test.
//
// Dropout ("Flash Attention" page, "Algorithm 2": P_dropped = dropout(P, p), O =
// P_dropped V; "Algorithm 4" regenerates the same mask in the backward pass) needs a
// mask that can be recomputed anywhere from a few integers. The pages name no generator;
// this library uses the counter-based Philox-4x32 with 10 rounds of J. K. Salmon,
// M. A. Moraes, R. O. Dror and D. E. Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3"
// (SC'11), section 3.3, and this layout (also stated in include/fa_fwd.h):
//   t = round(p * 32768), a 15-bit threshold;
//   element (bh, i, j) -- head bh = b*H + h, query row i, key j -- draws
//     words = Philox(counter = (j >> 3, i, bh, offset), key = (seed lo, seed hi)),
//     x = low 15 bits of words[(j >> 1) & 3] (j even) or of its high half (j odd),
//     kept iff x >= t, and a kept entry is scaled by 32768 / (32768 - t).
// One generator call covers eight consecutive keys of one query row.
#pragma once

#include <cstdint>

namespace fa {

// One Philox-4x32-10 block. A round maps (c0, c1, c2, c3) under the round key (k0, k1)
// to (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)); the key then
// advances by the Weyl increments.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
  constexpr uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  constexpr uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    const uint64_t a = (uint64_t)M0 * c.x;
    const uint64_t b = (uint64_t)M1 * c.z;
    c = make_uint4((uint32_t)(b >> 32) ^ c.y ^ k0, (uint32_t)b, (uint32_t)(a >> 32) ^ c.w ^ k1,
                   (uint32_t)a);
    k0 += W0;
    k1 += W1;
  }
  return c;
}

__device__ __forceinline__ uint32_t uint4_word(const uint4& v, int w) {
  return w == 0 ? v.x : w == 1 ? v.y : w == 2 ? v.z : v.w;
}

// Keep masks of the two keys of one generator word, as 16-bit lanes: 0xFFFF in a half
// whose low 15 bits are >= t, 0 otherwise. `bias` = (0x8000 - t) * 0x00010001: adding it
// to the 15-bit halves sets bit 15 of a half exactly when x >= t (no carry crosses into
// the other half), and the byte permute copies each half's bit 15 over the half.
__device__ __forceinline__ uint32_t keep_mask2(uint32_t word, uint32_t bias) {
  const uint32_t y = (word & 0x7FFF7FFFu) + bias;
  uint32_t m;
  asm("prmt.b32 %0, %1, 0, 0xBB99;" : "=r"(m) : "r"(y));
  return m;
}

// The generator words of keys [8 g, 8 g + 8) of query row i of head bh.
__device__ __forceinline__ uint4 dropout_words(uint32_t g, uint32_t i, uint32_t bh, uint32_t offset,
                                               uint32_t k0, uint32_t k1) {
  return philox4x32_10(make_uint4(g, i, bh, offset), k0, k1);
}

}  // namespace fa
