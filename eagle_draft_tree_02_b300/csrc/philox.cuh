// Philox4x64-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
// as 1, 2, 3", SC'11), device side, and the verify step's two draws.
//
// key = (seed, 0); counter = (round_id, b * 2^32 + node, idx, stream);
// stream 0 gives the acceptance uniform U = (w0 >> 40) 2^-24, stream 1 the
// Gumbel noise -log(-log U'), U' = ((w0 >> 40) + 0.5) 2^-24.
#pragma once
#include <stdint.h>

namespace e3 {

__device__ __forceinline__ uint64_t philox4x64_w0(uint64_t c0, uint64_t c1, uint64_t c2, uint64_t c3,
                                                  uint64_t k0, uint64_t k1) {
  const uint64_t mA = 0xD2E7470EE14C6C93ull, mB = 0xCA5A826395121157ull;
  const uint64_t wA = 0x9E3779B97F4A7C15ull, wB = 0xBB67AE8584CAA73Bull;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += wA;
      k1 += wB;
    }
    uint64_t hi0 = __umul64hi(mA, c0), lo0 = mA * c0;
    uint64_t hi1 = __umul64hi(mB, c2), lo1 = mB * c2;
    uint64_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
  }
  return c0;
}

__device__ __forceinline__ uint64_t verify_word(unsigned long long seed, unsigned long long round_id,
                                                int b, int node, uint64_t idx, int stream) {
  return philox4x64_w0(round_id, ((uint64_t)(uint32_t)b << 32) | (uint32_t)node, idx,
                       (uint64_t)stream, seed, 0ull);
}

// acceptance uniform in [0, 1), exact in fp32 (24 bits)
__device__ __forceinline__ float verify_uniform(unsigned long long seed, unsigned long long round_id,
                                                int b, int node, int i) {
  uint64_t m = verify_word(seed, round_id, b, node, (uint64_t)i, 0) >> 40;
  return (float)m * 5.9604644775390625e-08f;  // 2^-24
}

// Gumbel noise.  -log U' is evaluated from an exactly representable operand:
// U' itself when U' < 1/2, else 1 - U' through log1p, so U' never rounds to 1.
__device__ __forceinline__ float verify_gumbel(unsigned long long seed, unsigned long long round_id,
                                               int b, int node, int x) {
  uint32_t m = (uint32_t)(verify_word(seed, round_id, b, node, (uint64_t)x, 1) >> 40);
  float e;
  if (m < (1u << 23)) {
    float u = ((float)m + 0.5f) * 5.9604644775390625e-08f;
    e = -logf(u);
  } else {
    float t = ((float)((1u << 24) - m) - 0.5f) * 5.9604644775390625e-08f;  // 1 - U'
    e = -log1pf(-t);
  }
  return -logf(e);
}

}  // namespace e3
