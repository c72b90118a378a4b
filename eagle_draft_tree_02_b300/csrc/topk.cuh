// Warp-level top-k helpers shared by the vocabulary heads and the merge of
// their per-CTA partials: 64-bit keys ordered like (value desc, token asc),
// a warp-wide bitonic sort of one key per lane, and the rank merge of a
// sorted run into a sorted k-list in shared memory.
#pragma once

#include <stdint.h>

namespace e3 {

// 64-bit keys ordered like (value desc, token asc): larger key = better
__device__ __forceinline__ unsigned long long topk_key(float v, int i) {
  const uint32_t u = __float_as_uint(v);
  const uint32_t o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)o << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)i);
}
__device__ __forceinline__ float key_val(unsigned long long k) {
  const uint32_t o = (uint32_t)(k >> 32);
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}
__device__ __forceinline__ int key_tok(unsigned long long k) {
  return (int)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull));
}

// Warp-wide bitonic sort of one 64-bit key per lane, descending: lane j ends
// with the j-th largest key.
__device__ __forceinline__ unsigned long long warp_sort_desc(unsigned long long a, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const unsigned long long p = __shfl_xor_sync(0xffffffffu, a, stride);
      const bool keep_max = ((lane & stride) == 0) == ((lane & size) == 0);
      a = keep_max ? (a > p ? a : p) : (a < p ? a : p);
    }
  }
  return a;
}

// Merge a sorted key list A (lane j holds A_j, 0 = empty) into the sorted
// k-list (vals, idx) in shared memory: element j of either list lands at j
// plus the number of strictly larger keys in the other list; positions >= k
// drop out.
__device__ __forceinline__ void list_merge(float* vals, int* idx, int k, unsigned long long a,
                                           int lane) {
  const unsigned long long l = lane < k ? topk_key(vals[lane], idx[lane]) : 0ull;
  int ra = 0, rl = 0;
  for (int i = 0; i < k; ++i) {
    const unsigned long long li = __shfl_sync(0xffffffffu, l, i);
    const unsigned long long ai = __shfl_sync(0xffffffffu, a, i);
    ra += li > a;
    rl += ai > l;
  }
  __syncwarp();  // every lane has read the old list
  if (lane < k) {
    const int pa = lane + ra, pl = lane + rl;
    if (pa < k && a != 0ull) {
      vals[pa] = key_val(a);
      idx[pa] = key_tok(a);
    }
    if (pl < k) {
      vals[pl] = key_val(l);
      idx[pl] = key_tok(l);
    }
  }
  __syncwarp();
}

}  // namespace e3
