// Device side of attention dropout: the Philox4x32-10 counter-based generator and the map
// from an attention element (head, query row, key) to one byte of its output.
//
// Dropout is listed among the steps fused into the one attention kernel (reading guide,
// arXiv 2205.14135, "Key ideas", kernel fusion); the backward does not read a stored mask
// but regenerates it, as it regenerates S and P (answer page "How FlashAttention works for
// training", section 3.1).  Element (bh, i, j) is dropped when its byte u is below the
// 8-bit threshold t (probability t / 256); kept elements are scaled by 256 / (256 - t).
//
// Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel Random Numbers: As Easy as 1,
// 2, 3", SC 2011): four 32-bit counter words and two key words; each of ten rounds takes
// the 64-bit products of the first and third counter words with two fixed multipliers and
// recombines their halves with the other words and the key; the key advances by two Weyl
// constants between rounds.
//
// Which byte belongs to which element:
//   key     = (seed low word, seed high word),  counter = (kappa, rho, bh, offset)
//   rho     = 8 (i >> 4) + (i & 7)              query rows i and i + 8 of a 16-row block
//   kappa   = 4 (j >> 5) + ((j >> 1) & 3)       keys 32a + 2c + {0, 1} + {0, 8, 16, 24}
//   u(i, j) = byte 2 ((i >> 3) & 1) + (j & 1) of output word (j >> 3) & 3.
// A forward softmax thread of the tensor-core kernel holds rows A and A + 8 (A % 16 < 8) and
// keys 8c + 2(t % 4) + {0, 1}: one call gives it the bytes of four of its key chunks, word c
// holding [row A even key, row A odd key, row B even key, row B odd key].
#pragma once

#include <stdint.h>

#include "fa_internal.cuh"

namespace fa {
namespace philox {

// High 32 bits of a 32 x 32-bit product: __umulhi on the device, the same value on the host
// (the generator functions below also compile as host code, for the CPU tests).
__host__ __device__ __forceinline__ uint32_t mulhi32(uint32_t a, uint32_t b) {
#ifdef __CUDA_ARCH__
  return __umulhi(a, b);
#else
  return static_cast<uint32_t>((static_cast<uint64_t>(a) * b) >> 32);
#endif
}

struct Words {
  uint32_t w[4];
};

__host__ __device__ __forceinline__ Words philox4x32_10(uint32_t x0, uint32_t x1,
                                                        uint32_t x2, uint32_t x3,
                                                        uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t hi0 = mulhi32(0xD2511F53u, x0), lo0 = 0xD2511F53u * x0;
    const uint32_t hi1 = mulhi32(0xCD9E8D57u, x2), lo1 = 0xCD9E8D57u * x2;
    x0 = hi1 ^ x1 ^ k0;
    x1 = lo1;
    x2 = hi0 ^ x3 ^ k1;
    x3 = lo0;
  }
  return Words{{x0, x1, x2, x3}};
}

// The same generator for a stream of calls in which only x0 changes (x1, x2, x3 and the key
// fixed): the 4 multiplies of rounds 1-2 that depend on the fixed words alone are formed once.
struct PrefixX0 {
  uint32_t x3k1;  // round 1: x3 ^ k1
  uint32_t c1;    // round 1: x1'
  uint32_t h0;    // round 2: high product of x0'
  uint32_t l0;    // round 2: low product of x0'
  uint32_t k0, k1;
};

__host__ __device__ __forceinline__ PrefixX0 prefix_x0(uint32_t x1, uint32_t x2,
                                                        uint32_t x3, uint32_t k0,
                                                        uint32_t k1) {
  PrefixX0 s;
  s.k0 = k0;
  s.k1 = k1;
  s.x3k1 = x3 ^ k1;
  s.c1 = 0xCD9E8D57u * x2;
  const uint32_t c0 = mulhi32(0xCD9E8D57u, x2) ^ x1 ^ k0;   // round 1: x0'
  s.h0 = mulhi32(0xD2511F53u, c0);
  s.l0 = 0xD2511F53u * c0;
  return s;
}

__host__ __device__ __forceinline__ Words run_x0(const PrefixX0& s, uint32_t x0) {
  // round 1
  const uint32_t y2 = mulhi32(0xD2511F53u, x0) ^ s.x3k1;
  const uint32_t y3 = 0xD2511F53u * x0;
  // round 2
  uint32_t k0 = s.k0 + 0x9E3779B9u, k1 = s.k1 + 0xBB67AE85u;
  uint32_t z0 = mulhi32(0xCD9E8D57u, y2) ^ s.c1 ^ k0;
  uint32_t z1 = 0xCD9E8D57u * y2;
  uint32_t z2 = s.h0 ^ y3 ^ k1;
  uint32_t z3 = s.l0;
#pragma unroll
  for (int r = 2; r < 10; ++r) {
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
    const uint32_t hi0 = mulhi32(0xD2511F53u, z0), lo0 = 0xD2511F53u * z0;
    const uint32_t hi1 = mulhi32(0xCD9E8D57u, z2), lo1 = 0xCD9E8D57u * z2;
    z0 = hi1 ^ z1 ^ k0;
    z1 = lo1;
    z2 = hi0 ^ z3 ^ k1;
    z3 = lo0;
  }
  return Words{{z0, z1, z2, z3}};
}

__host__ __device__ __forceinline__ uint32_t row_pair(int i) {
  return static_cast<uint32_t>(8 * (i >> 4) + (i & 7));
}

__host__ __device__ __forceinline__ uint32_t key_octet(int j) {
  return static_cast<uint32_t>(4 * (j >> 5) + ((j >> 1) & 3));
}

// The generator call that holds element (bh, i, j)'s byte.
__device__ __forceinline__ Words call(const Problem& p, int bh, int i, int j) {
  return philox4x32_10(key_octet(j), row_pair(i), static_cast<uint32_t>(bh), p.drop_offset,
                       p.drop_seed_lo, p.drop_seed_hi);
}

// Byte u(i, j) out of the words of its call.
__device__ __forceinline__ uint32_t byte_of(const Words& r, int i, int j) {
  const uint32_t w = r.w[(j >> 3) & 3];
  return (w >> (8 * (2 * ((i >> 3) & 1) + (j & 1)))) & 0xFFu;
}

// Per-byte keep masks of a word: 0xFF in each byte that is >= the threshold, else 0.
__device__ __forceinline__ uint32_t keep_bytes(uint32_t word, uint32_t thr4) {
  return __vcmpgeu4(word, thr4);
}

}  // namespace philox
}  // namespace fa
