// Philox4x32-10 draws of one position's Gumbel stream with the per-position
// work hoisted out of the per-element loop.
//
// A position's Gumbel draws come from the counters (x, p, (block<<16)|step,
// GUMBEL_ORDER) under the canvas seed, with x = 8 j + k / 2 for step k of the
// order statistics of vocabulary group j the only word that changes.  In the
// first two rounds of the Philox bijection (Salmon, Moraes, Dror, Shaw,
// "Parallel random numbers: as easy as 1, 2, 3", SC'11) half of the products
// and XORs involve only the fixed words, so they are computed once per
// position; the round keys of the remaining eight rounds are kept as well.
// draw(x) returns exactly the block philox((x, p, bs, GUMBEL_ORDER), seed), at
// 37 integer operations instead of 60.
#pragma once

#include <stdint.h>

namespace dg {

struct GumbelStream {
  static constexpr uint32_t kM0 = 0xD2511F53u, kM1 = 0xCD9E8D57u;
  static constexpr uint32_t kW0 = 0x9E3779B9u, kW1 = 0xBB67AE85u;
  uint32_t c1;      // round 0: word 3 ^ key1
  uint32_t d2, e2;  // round 1: lo(M1 z) ^ key0', hi(M0 x1) ^ key1'
  uint32_t f2;      // round 1: lo(M0 x1)
  uint32_t k0[8], k1[8];  // round keys of rounds 2..9

  __host__ __device__ __forceinline__ static uint32_t mulhi(uint32_t a, uint32_t b) {
#ifdef __CUDA_ARCH__
    return __umulhi(a, b);
#else
    return (uint32_t)(((uint64_t)a * b) >> 32);
#endif
  }

  __host__ __device__ __forceinline__ void init(uint64_t seed, uint32_t p, uint32_t bs, uint32_t purpose) {
    const uint32_t key0 = (uint32_t)seed, key1 = (uint32_t)(seed >> 32);
    // round 0 on (x, p, bs, purpose): the M1 * bs product is fixed
    const uint32_t x1 = mulhi(kM1, bs) ^ p ^ key0;  // word 0 after round 0 (fixed)
    const uint32_t y1 = kM1 * bs;                   // word 1 after round 0 (fixed)
    c1 = purpose ^ key1;                            // word 2 after round 0 = hi(M0 x) ^ c1
    // round 1: the M0 * x1 product is fixed
    d2 = y1 ^ (key0 + kW0);                         // word 0 after round 1 = hi(M1 z1) ^ d2
    e2 = mulhi(kM0, x1) ^ (key1 + kW1);             // word 2 after round 1 = lo(M0 x) ^ e2
    f2 = kM0 * x1;                                  // word 3 after round 1
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      k0[r] = key0 + (uint32_t)(r + 2) * kW0;
      k1[r] = key1 + (uint32_t)(r + 2) * kW1;
    }
  }

  // The high and low halves of each product are formed by two 32-bit
  // multiplies rather than one 64-bit product: the same words, fewer issue
  // cycles on the integer multiplier.
  __host__ __device__ __forceinline__ void draw(uint32_t x, uint32_t (&out)[4]) const {
    const uint32_t z1 = mulhi(kM0, x) ^ c1, w1 = kM0 * x;
    uint32_t a = mulhi(kM1, z1) ^ d2, b = kM1 * z1, c = w1 ^ e2, d = f2;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const uint32_t na = mulhi(kM1, c) ^ b ^ k0[r];
      const uint32_t nc = mulhi(kM0, a) ^ d ^ k1[r];
      b = kM1 * c;
      d = kM0 * a;
      a = na;
      c = nc;
    }
    out[0] = a;
    out[1] = b;
    out[2] = c;
    out[3] = d;
  }
};

}  // namespace dg
