// dropout.cuh -- dropout decisions for the attention kernels.
//
// Dropout of the attention probabilities (page "Flash Attention V2大模型时代的
// 算力救星", section 4.2, the dropout_p argument of the call; page
// "FlashAttention-2：GPU利用率从50%干到90%", improvement 2, dropout done inside
// the kernel).  The pages name no generator; the decisions are drawn from the
// counter-based Philox4x32-10 of Salmon, Moraes, Dror and Shaw, "Parallel
// Random Numbers: As Easy as 1, 2, 3" (SC 2011), so that the backward pass
// recomputes exactly the forward's decisions without storing them:
//
//   counter (query row i, key j / 16, b * H + h, offset), key (seed low 32
//   bits, seed high 32 bits); byte j % 16 of the 16 output bytes (word
//   (j % 16) / 4, least significant byte first) keeps score (i, j) iff it is
//   below the threshold t = floor(256 (1 - p) + 1/2), 1 <= t <= 255.  Kept
//   probabilities are scaled by 256 / t.
#pragma once

#include <cstdint>

#include "kernels.h"

namespace attn {

// Philox4x32-10 (SC 2011, section 3.2): ten rounds of two 32 x 32 -> 64-bit
// products of x0, x2 with the multipliers, the other words and the round key
// xor-ed into the high halves; the key takes a Weyl step per round.
__device__ __forceinline__ uint4 philox_round(uint4 c, uint32_t k0, uint32_t k1) {
  const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
  const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
  return make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
}
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    c = philox_round(c, k0, k1);
    k0 += kPhiloxW0;
    k1 += kPhiloxW1;
  }
  return c;
}
// The same with the round keys taken from the precomputed schedule dk.rk.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, const DropoutArgs& dk) {
#pragma unroll
  for (int r = 0; r < 10; ++r) c = philox_round(c, dk.rk[2 * r], dk.rk[2 * r + 1]);
  return c;
}

// Bit b (0..3) = byte b of x is below t, for cmp = (256 - t) * 0x00010001:
// the even and the odd bytes sit in two 16-bit lanes each, where
// byte + 256 - t carries into bit 8 exactly when byte >= t.
__device__ __forceinline__ uint32_t keep_bits4(uint32_t x, uint32_t cmp) {
  const uint32_t e = x & 0x00FF00FFu, o = (x >> 8) & 0x00FF00FFu;
  const uint32_t ge = (((e + cmp) >> 8) & 0x00010001u) | ((((o + cmp) >> 8) & 0x00010001u) << 1);
  return ~(ge | (ge >> 14)) & 0xFu;
}

// Keep bits of keys 16 g .. 16 g + 15 of query row i: bit m for key 16 g + m.
__device__ __forceinline__ uint32_t keep_bits16(const DropoutArgs& dk, uint32_t head, uint32_t i,
                                                uint32_t g) {
  const uint4 x = philox4x32_10(make_uint4(i, g, head, dk.offset), dk);
  return keep_bits4(x.x, dk.cmp) | (keep_bits4(x.y, dk.cmp) << 4) | (keep_bits4(x.z, dk.cmp) << 8) |
         (keep_bits4(x.w, dk.cmp) << 12);
}

// 32 x 32 bit transpose across a warp: bit m of lane l becomes bit l of
// lane m.  Five butterfly stages; at stage j the lanes l and l ^ j swap the
// off-diagonal j x j blocks of every 2j x 2j block.
__device__ __forceinline__ uint32_t warp_transpose32(uint32_t x, int lane) {
  uint32_t m = 0x0000FFFFu;
#pragma unroll
  for (int j = 16; j > 0; j >>= 1) {
    const uint32_t y = __shfl_xor_sync(0xffffffffu, x, j);
    x = (lane & j) ? ((x & ~m) | ((y >> j) & m)) : ((x & m) | ((y << j) & ~m));
    if (j > 1) m ^= m << (j >> 1);
  }
  return x;
}

}  // namespace attn
