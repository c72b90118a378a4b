// Philox4x64-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
// as 1, 2, 3", SC'11), device side, and the verify step's two draws.
//
// key = (seed, 0).  Acceptance test i at node (b, node): counter
// (round_id, b * 2^32 + node, i, 0), U = (w0 >> 40) 2^-24.  Gumbel noise of
// token x: counter (round_id, b * 2^32 + node, x / 4, 1), word x % 4 of the
// block gives U' = ((w >> 40) + 0.5) 2^-24 and the noise -log(-log U').  The
// four words of a block are independent, so one block serves four tokens.
#pragma once
#include <stdint.h>

namespace e3 {

// all four output words of one block
__device__ __forceinline__ void philox4x64(uint64_t c0, uint64_t c1, uint64_t c2, uint64_t c3, uint64_t k0,
                                           uint64_t k1, uint64_t (&w)[4]) {
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
  w[0] = c0;
  w[1] = c1;
  w[2] = c2;
  w[3] = c3;
}

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

// Gumbel noise from one output word.  -log U' is evaluated from an exactly
// representable operand: U' itself when U' < 1/2, else 1 - U' through log1p,
// so U' never rounds to 1.  The outer log uses the fast intrinsic: its error
// (about 1e-6 relative) can only move a Gumbel argmax whose two best scores
// are that close, a near-tie that the parity rule counts.
__device__ __forceinline__ float gumbel_from_u24(uint32_t m) {  // m = word >> 40
  float e;
  if (m < (1u << 23)) {
    float u = ((float)m + 0.5f) * 5.9604644775390625e-08f;
    e = -__logf(u);
  } else {
    float t = ((float)((1u << 24) - m) - 0.5f) * 5.9604644775390625e-08f;  // 1 - U'
    e = -log1pf(-t);
  }
  return -__logf(e);
}
__device__ __forceinline__ float gumbel_from_word(uint64_t w) {
  return gumbel_from_u24((uint32_t)(w >> 40));
}

// the Philox block that holds the Gumbel words of tokens 4 blk .. 4 blk + 3
__device__ __forceinline__ void gumbel_block(unsigned long long seed, unsigned long long round_id, int b,
                                             int node, uint64_t blk, uint64_t (&w)[4]) {
  philox4x64(round_id, ((uint64_t)(uint32_t)b << 32) | (uint32_t)node, blk, 1ull, seed, 0ull, w);
}

// Gumbel noise of token x (one block per call: for paths that need a single token)
__device__ __forceinline__ float verify_gumbel(unsigned long long seed, unsigned long long round_id,
                                               int b, int node, int x) {
  uint64_t w[4];
  gumbel_block(seed, round_id, b, node, (uint64_t)(x >> 2), w);
  return gumbel_from_word(w[x & 3]);
}

}  // namespace e3
