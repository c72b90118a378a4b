// Verification walk over the kept tree ("EAGLE-3 精读" §5 正确性、复现与风险:
// with the target's standard verifier, greedy keeps the target's sequence and
// sampling keeps its distribution when the residual correction is done).
//
// Greedy: from the root, descend into the child whose token is the target's
// argmax at the current node; stop when no child matches; the argmax at the
// stop node is the bonus token.
//
// Sampling: the tree's children are deterministic top-k picks, i.e. point-mass
// proposals, so the exact acceptance rule is: child c_i (canonical order) is
// accepted iff U_i (1 - R) < p(c_i), where p = softmax(z / T) and R is the
// target mass of the children already rejected at this node; when none is
// accepted (or the node is a leaf) the bonus token is the Gumbel-argmax of z/T
// over the node's non-children, an exact draw from the residual distribution.
// One thread per request; all per-node quantities come from the target head.
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "philox.cuh"

namespace e3 {

__global__ void walk_kernel(WalkArgs a) {
  pdl_begin();
  int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= a.B) return;
  if (a.bonus_best) a.bonus_best[b] = 0ull;
  const unsigned long long rid = a.round_ptr ? *a.round_ptr : a.round_id;
  const size_t tb = (size_t)b * a.M1;
  int u = 0, n = 0;
  int* path = a.path + (size_t)b * a.D;
  int* out = a.out_tokens + (size_t)b * (a.D + 1);
  for (int i = 0; i < a.D; ++i) path[i] = -1;
  for (int i = 0; i <= a.D; ++i) out[i] = -1;
  while (true) {
    const size_t r = tb + u;
    int nc = a.n_child[r];
    int next = -1;
    if (!a.sampling) {
      int tgt = a.z_arg[r];
      for (int i = 0; i < nc; ++i) {
        int c = a.child_node[r * a.kmax + i];
        if (a.t_tok[tb + c] == tgt) { next = c; break; }
      }
    } else {
      float lse = a.lse[r], rej = 0.f;
      for (int i = 0; i < nc; ++i) {
        float p = expf(a.child_z[r * a.kmax + i] * a.inv_t - lse);
        float U = verify_uniform(a.seed, rid, b, u, i);
        if (U * (1.f - rej) < p) { next = a.child_node[r * a.kmax + i]; break; }
        rej += p;
      }
    }
    if (next < 0 || n >= a.D) {
      out[n] = a.sampling ? a.g_arg[r] : a.z_arg[r];
      break;
    }
    path[n] = next;
    out[n] = a.t_tok[tb + next];
    ++n;
    u = next;
  }
  a.accept_len[b] = n;
}

void launch_walk(const WalkArgs& a, cudaStream_t st) {
  launch_pdl(walk_kernel, dim3((a.B + 63) / 64), dim3(64), 0, st, a);
}

// Deferred bonus draw.  The noise of token x at (request b, node u) is the
// same Philox word the head's epilogue would have drawn (block x / 4, word
// x % 4), so the draw is the one that epilogue makes, taken at one node.
// A (score, token) pair packs into a key whose unsigned order is score
// ascending, then token descending: the largest key is the Gumbel-argmax with
// ties to the lowest token.
__device__ __forceinline__ unsigned long long bonus_key(float s, int x) {
  const uint32_t u = __float_as_uint(s);
  const uint32_t o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)o << 32) | (0xFFFFFFFFu - (uint32_t)x);
}

__device__ __forceinline__ int bonus_stop(const BonusArgs& a, int b, int& n) {
  n = min(max(a.accept_len[b], 0), a.D);
  int u = n == 0 ? 0 : a.path[(size_t)b * a.D + n - 1];
  return (u < 0 || u >= a.M1) ? 0 : u;  // cannot fail after a walk; keeps the reads in bounds
}

__global__ void __launch_bounds__(256) bonus_gumbel_kernel(BonusArgs a) {
  pdl_begin();
  __shared__ int kids[32];
  __shared__ unsigned long long best_s[8];
  const int b = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned long long rid = a.round_ptr ? *a.round_ptr : a.round_id;
  int n;
  const int u = bonus_stop(a, b, n);
  const size_t r = (size_t)b * a.M1 + u;
  const int nk = min(a.kmax, 32);
  if (tid < nk) kids[tid] = a.child_tok[r * a.kmax + tid];
  __syncthreads();
  const float* z = a.logits + r * a.V;
  unsigned long long best = 0ull;
  for (int blk = blockIdx.x * blockDim.x + tid; blk * 4 < a.V; blk += gridDim.x * blockDim.x) {
    uint64_t w[4];
    gumbel_block(a.seed, rid, b, u, (uint64_t)blk, w);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int x = blk * 4 + e;
      if (x >= a.V) break;
      bool child = false;
      for (int i = 0; i < nk; ++i) child |= kids[i] == x;
      if (child) continue;
      const float s = __fmaf_rn(z[x], a.inv_t, gumbel_from_u24((uint32_t)(w[e] >> 40)));
      const unsigned long long key = bonus_key(s, x);
      best = key > best ? key : best;
    }
  }
  for (int o = 16; o; o >>= 1) {
    const unsigned long long ob = __shfl_xor_sync(0xffffffffu, best, o);
    best = ob > best ? ob : best;
  }
  if (lane == 0) best_s[warp] = best;
  __syncthreads();
  if (tid == 0) {
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) best = best_s[w] > best ? best_s[w] : best;
    if (best) atomicMax(a.best + b, best);
  }
}

__global__ void bonus_write_kernel(BonusArgs a) {
  pdl_begin();
  for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < a.B; b += gridDim.x * blockDim.x) {
    int n;
    const int u = bonus_stop(a, b, n);
    const unsigned long long key = a.best[b];
    const int t = key ? (int)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull)) : -1;
    a.out_tokens[(size_t)b * (a.D + 1) + n] = t;
    a.g_arg[(size_t)b * a.M1 + u] = t;
  }
}

void launch_bonus_gumbel(const BonusArgs& a, cudaStream_t st) {
  // about two waves of 256-thread blocks over all requests' vocabularies
  const int per_req = (a.V / 4 + 255) / 256;
  const int n_blk = std::max(1, std::min(per_req, (2 * 148 * 4 + a.B - 1) / a.B));
  launch_pdl(bonus_gumbel_kernel, dim3(n_blk, a.B), dim3(256), 0, st, a);
  launch_pdl(bonus_write_kernel, dim3((a.B + 127) / 128), dim3(128), 0, st, a);
}

__global__ void set_u64_kernel(unsigned long long* p, unsigned long long v) { pdl_begin(); *p = v; }

void launch_set_u64(unsigned long long* p, unsigned long long v, cudaStream_t st) {
  launch_pdl(set_u64_kernel, dim3(1), dim3(1), 0, st, p, v);
}

}  // namespace e3
