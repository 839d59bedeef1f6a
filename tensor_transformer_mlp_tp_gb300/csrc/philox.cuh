// Philox4x64-10 and the dropout keep decision of the sequence-parallel region.
//
// Generator: Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy
// as 1, 2, 3" (SC 2011), the Philox4x64 variant with 10 rounds.  One round
// multiplies counter words 0 and 2 by the round multipliers, takes the high
// and low 64-bit halves of the two 128-bit products, and mixes the high
// halves with counter words 1 and 3 and the key; the key advances by the
// Weyl increments between rounds.
//
// Dropout decision (the pages name Dropout in the sequence-split region but
// give no generator): element e = r*d + c of the gathered [T x d] output
// belongs to block e/8, one generator call with counter (e/8, offset, 0, 0)
// and key (seed, 0).  Element e takes 32 bits of that block: word (e%8)/2,
// low half for even e, high half for odd e.  It is kept when those bits, as
// an unsigned integer, are below thr = floor((1 - p) 2^32); thr = 2^32 keeps
// everything.
#pragma once

#include <stdint.h>

namespace tpmlp {

constexpr unsigned long long kPhiloxM0 = 0xD2E7470EE14C6C93ull;
constexpr unsigned long long kPhiloxM1 = 0xCA5A826395121157ull;
constexpr unsigned long long kPhiloxW0 = 0x9E3779B97F4A7C15ull;
constexpr unsigned long long kPhiloxW1 = 0xBB67AE8584CAA73Bull;
constexpr unsigned long long kKeepAll = 1ull << 32;

__device__ __forceinline__ void philox4x64_10(unsigned long long c0, unsigned long long c1, unsigned long long c2,
                                              unsigned long long c3, unsigned long long k0, unsigned long long k1,
                                              unsigned long long (&out)[4]) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += kPhiloxW0;
      k1 += kPhiloxW1;
    }
    const unsigned long long hi0 = __umul64hi(kPhiloxM0, c0), lo0 = kPhiloxM0 * c0;
    const unsigned long long hi1 = __umul64hi(kPhiloxM1, c2), lo1 = kPhiloxM1 * c2;
    c0 = hi1 ^ c1 ^ k0;
    c1 = lo1;
    c2 = hi0 ^ c3 ^ k1;
    c3 = lo0;
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

// Keep bits of the 8 elements of block q: bit j is element 8 q + j.
__device__ __forceinline__ uint32_t dropout_keep8(unsigned long long q, unsigned long long offset,
                                                  unsigned long long seed, unsigned long long thr) {
  unsigned long long w[4];
  philox4x64_10(q, offset, 0ull, 0ull, seed, 0ull, w);
  uint32_t m = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const unsigned long long u = (w[j >> 1] >> (32 * (j & 1))) & 0xFFFFFFFFull;
    m |= (u < thr ? 1u : 0u) << j;
  }
  return m;
}

}  // namespace tpmlp
