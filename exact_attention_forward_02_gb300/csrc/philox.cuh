// philox.cuh -- the dropout mask of libfa: Philox-4x32-10 and the 8-bit keep test.
//
// Dropout ("Flash Attention" page, "Algorithm 2": P_dropped = dropout(P, p), O =
// P_dropped V; "Algorithm 4" regenerates the same mask in the backward pass) needs a
// mask that can be recomputed anywhere from a few integers. The pages name no generator;
// this library uses the counter-based Philox-4x32 with 10 rounds of J. K. Salmon,
// M. A. Moraes, R. O. Dror and D. E. Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3"
// (SC'11), section 3.3, and this layout (also stated in include/fa_fwd.h):
//   t = round(p * 256), an 8-bit threshold;
//   element (bh, i, j) -- head bh = b*H + h, query row i, key j -- draws
//     words = Philox(counter = (j >> 4, i, bh, offset), key = (seed lo, seed hi)),
//     x = byte 2 (j & 1) + ((j >> 1) & 1) of words[(j >> 2) & 3] (the low bytes of a
//         word's 16-bit halves serve its first key pair, the high bytes its second),
//     kept iff x >= t, and a kept entry is scaled by 256 / (256 - t).
// One generator call covers sixteen consecutive keys of one query row.
#pragma once

#include <cstdint>

namespace fa {

constexpr uint32_t PHILOX_M0 = 0xD2511F53u, PHILOX_M1 = 0xCD9E8D57u;
constexpr uint32_t PHILOX_W0 = 0x9E3779B9u, PHILOX_W1 = 0xBB67AE85u;

// The ten round keys of a seed: rk[2r] = k0 + r W0, rk[2r + 1] = k1 + r W1 (the key
// schedule does not depend on the counter, so it is computed once, on the host).
struct PhiloxKeys {
  uint32_t rk[20];
};

__host__ __device__ inline PhiloxKeys philox_keys(unsigned long long seed) {
  PhiloxKeys k;
  uint32_t k0 = (uint32_t)(seed & 0xFFFFFFFFull), k1 = (uint32_t)(seed >> 32);
  for (int r = 0; r < 10; ++r) {
    k.rk[2 * r] = k0;
    k.rk[2 * r + 1] = k1;
    k0 += PHILOX_W0;
    k1 += PHILOX_W1;
  }
  return k;
}

// One Philox-4x32-10 block. A round maps (c0, c1, c2, c3) under the round key (k0, k1)
// to (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)).
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, const PhiloxKeys& k) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t a = (uint64_t)PHILOX_M0 * c.x;
    const uint64_t b = (uint64_t)PHILOX_M1 * c.z;
    c = make_uint4((uint32_t)(b >> 32) ^ c.y ^ k.rk[2 * r], (uint32_t)b,
                   (uint32_t)(a >> 32) ^ c.w ^ k.rk[2 * r + 1], (uint32_t)a);
  }
  return c;
}

__device__ __forceinline__ uint32_t uint4_word(const uint4& v, int w) {
  return w == 0 ? v.x : w == 1 ? v.y : w == 2 ? v.z : v.w;
}

// Keep flags of the four keys of one generator word, as two key pairs: bit 8 of `first`
// for key 0 and bit 24 for key 1 (bytes 0 and 2), bit 8 of `second` for key 2 and bit 24
// for key 3 (bytes 1 and 3); other bits are don't-care. `bias` = (0x100 - t) * 0x00010001:
// added to a byte held in a 16-bit lane it sets bit 8 exactly when the byte is >= t, and
// no carry leaves the lane (x + 0x100 - t <= 0x1FF).
__device__ __forceinline__ void keep_flags4(uint32_t word, uint32_t bias, uint32_t& first,
                                            uint32_t& second) {
  uint32_t hi_bytes;
  asm("prmt.b32 %0, %1, 0, 0x4341;" : "=r"(hi_bytes) : "r"(word));  // bytes 1, 3 -> lanes
  first = (word & 0x00FF00FFu) + bias;
  second = hi_bytes + bias;
}

// 16-bit lane masks from flags at bits 15 and 31: the byte permute replicates the sign
// bit of byte 1 over the low half and that of byte 3 over the high half.
__device__ __forceinline__ uint32_t spread_flags2(uint32_t flags) {
  uint32_t m;
  asm("prmt.b32 %0, %1, 0, 0xBB99;" : "=r"(m) : "r"(flags));
  return m;
}

// The generator words of keys [16 g, 16 g + 16) of query row i of head bh.
__device__ __forceinline__ uint4 dropout_words(uint32_t g, uint32_t i, uint32_t bh, uint32_t offset,
                                               const PhiloxKeys& k) {
  return philox4x32_10(make_uint4(g, i, bh, offset), k);
}

// The keep bits of one query row over 32 NW consecutive keys starting at 16 g0, packed for
// the masking of 16-bit probability pairs: word q holds key pairs (32q + 2kk, 32q + 2kk + 1)
// for kk = 0..15 as bit kk (even key) and bit 16 + kk (odd key).
template <int NW = 4>
__device__ __forceinline__ void dropout_row_bits(uint32_t g0, uint32_t i, uint32_t bh,
                                                 uint32_t offset, const PhiloxKeys& k,
                                                 uint32_t bias, uint32_t* bits) {
#pragma unroll
  for (int q = 0; q < NW; ++q) {
    uint4 r2[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) r2[h] = dropout_words(g0 + 2 * q + h, i, bh, offset, k);
    uint32_t acc = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        uint32_t f0, f1;
        keep_flags4(uint4_word(r2[h], m), bias, f0, f1);
        const int kk0 = 8 * h + 2 * m, kk1 = kk0 + 1;  // pairs of keys 4m.., 4m+2.. of call h
        acc |= (kk0 <= 8 ? f0 >> (8 - kk0) : f0 << (kk0 - 8)) & (0x10001u << kk0);
        acc |= (kk1 <= 8 ? f1 >> (8 - kk1) : f1 << (kk1 - 8)) & (0x10001u << kk1);
      }
    bits[q] = acc;
  }
}

// The 16-bit lane mask of key pair kk of a word of dropout_row_bits.
__device__ __forceinline__ uint32_t pair_mask(uint32_t bits_word, int kk) {
  return spread_flags2(bits_word << (15 - kk));
}

// Whether key e (0..63) of a dropout_row_bits row is kept, as 0 or 1.
__device__ __forceinline__ uint32_t row_bit(const uint32_t* bits, int e) {
  const int pr = e >> 1, kk = pr & 15;
  return (bits[pr >> 4] >> ((e & 1) ? 16 + kk : kk)) & 1u;
}

// The keep mask of the sixteen keys of one generator call: bit e for key 16 g + e.
__device__ __forceinline__ uint32_t keep16(const uint4& w, uint32_t bias) {
  uint32_t m = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t f0, f1;
    keep_flags4(uint4_word(w, q), bias, f0, f1);
    m |= ((f0 >> 8) & 1u) << (4 * q) | ((f0 >> 24) & 1u) << (4 * q + 1) |
         ((f1 >> 8) & 1u) << (4 * q + 2) | ((f1 >> 24) & 1u) << (4 * q + 3);
  }
  return m;
}

}  // namespace fa
