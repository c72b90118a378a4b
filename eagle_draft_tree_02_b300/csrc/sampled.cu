// Sampled drafting with q-ratio verification (a variant of the round; the
// EAGLE-3 pages' sampling verification, "EAGLE-3 精读" §5: the target
// distribution is kept when the residual correction is done).
//
// Drafting: a node's k children are drawn from the draft distribution q
// without replacement, as the k largest keys log q(x) + G(x) (Gumbel-top-k;
// G from the Philox stream 2 counter of the node's slot), in draw order, with
// their true log q and the row's largest log q, from which the expansion
// scores the draws (each from the draws before it only).
//
// Verification at a node: the draws c_1 .. c_m in draw order are tested in
// turn; c_i is accepted when U_i q_i(c_i) < p_i(c_i); on a rejection
// p_{i+1} = norm(max(0, p_i - q_i)) and q_{i+1} = q_i without c_i; with no
// acceptance the bonus token is the Gumbel-argmax (stream 1) of log p over the
// last residual's support.  p = softmax(z / T) of the target logits, q =
// softmax of the draft logits at the node.
//
// Unlike the fused heads, this variant keeps a pass's logits in HBM (rows x V
// fp32, written by the tensor-core GEMM): the verify step needs q and p over
// the whole vocabulary at every node it visits.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "philox.cuh"

namespace e3 {

namespace {
constexpr int kThreads = 1024;
constexpr int kMaxK = 16;

// larger key = better under (value desc, token asc)
__device__ __forceinline__ unsigned long long skey(float v, int tok) {
  const uint32_t u = __float_as_uint(v == 0.f ? 0.f : v);
  const uint32_t o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)o << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)tok);
}

__device__ float block_max(float v, float* red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  v = warp_max(v);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  float t = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : -INFINITY;
  if (wid == 0) t = warp_max(t);
  if (threadIdx.x == 0) red[0] = t;
  __syncthreads();
  const float r = red[0];
  __syncthreads();
  return r;
}

__device__ unsigned long long block_max_u64(unsigned long long v, unsigned long long* red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long p = __shfl_xor_sync(0xffffffffu, v, o);
    v = p > v ? p : v;
  }
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  if (wid == 0) {
    unsigned long long t = lane < (int)(blockDim.x >> 5) ? red[lane] : 0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long p = __shfl_xor_sync(0xffffffffu, t, o);
      t = p > t ? p : t;
    }
    if (lane == 0) red[0] = t;
  }
  __syncthreads();
  const unsigned long long r = red[0];
  __syncthreads();
  return r;
}
}  // namespace

// ----------------------------------------------------------------------------- drafting
// One block per row of the pass: log-sum-exp of the row's logits, then the k
// best keys logit + G (the same order as log q + G), by k rounds of a block
// argmax over each thread's sorted short list.
__global__ void __launch_bounds__(kThreads) sample_children_kernel(SampleArgs a) {
  pdl_begin();
  __shared__ float redf[32];
  __shared__ unsigned long long redk[32];
  const int row = blockIdx.x;
  const float* ell = a.logits + (size_t)row * a.V;
  float m = -INFINITY;
  for (int x = threadIdx.x; x < a.V; x += blockDim.x) m = fmaxf(m, ell[x]);
  m = block_max(m, redf);
  float s = 0.f;
  for (int x = threadIdx.x; x < a.V; x += blockDim.x) s += __expf(ell[x] - m);
  s = block_sum(s, redf);
  const float lse = m + logf(s);
  if (threadIdx.x == 0) a.lmax[row] = m - lse;  // log of the row's largest probability
  // Gumbel keys: thread t takes the 4-token groups t, t + blockDim, ...
  const int b = row / a.rows_per_req, slot = a.slot0 + row % a.rows_per_req;
  const unsigned long long rid = a.round_ptr ? *a.round_ptr : a.round_id;
  unsigned long long mine[kMaxK];
  for (int j = 0; j < a.k; ++j) mine[j] = 0ull;
  for (int g4 = threadIdx.x; 4 * g4 < a.V; g4 += blockDim.x) {
    uint64_t w[4];
    philox4x64(rid, ((uint64_t)(uint32_t)b << 32) | (uint32_t)slot, (uint64_t)g4, 2ull, a.seed,
               0ull, w);
    for (int j = 0; j < 4; ++j) {
      const int x = 4 * g4 + j;
      if (x >= a.V) break;
      const unsigned long long key = skey(ell[x] + gumbel_from_word(w[j]), x);
      if (key > mine[a.k - 1]) {  // insert into the sorted list
        int p = a.k - 1;
        while (p > 0 && mine[p - 1] < key) {
          mine[p] = mine[p - 1];
          --p;
        }
        mine[p] = key;
      }
    }
  }
  int head = 0;
  for (int j = 0; j < a.k; ++j) {
    const unsigned long long cand = head < a.k ? mine[head] : 0ull;
    const unsigned long long best = block_max_u64(cand, redk);
    if (head < a.k && cand == best && best != 0ull) ++head;  // keys are unique (token in the low bits)
    if (threadIdx.x == 0) {
      const int tok = best ? (int)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFull)) : 0;
      a.tok[(size_t)row * a.k + j] = tok;
      a.logq[(size_t)row * a.k + j] = best ? ell[tok] - lse : -INFINITY;
    }
    __syncthreads();
  }
}

void launch_sample_children(const SampleArgs& a, int R, cudaStream_t st) {
  if (R <= 0) return;
  launch_pdl(sample_children_kernel, dim3(R), dim3(kThreads), 0, st, a);
}

// ----------------------------------------------------------------------------- verification
// One block per request walks the tree from the root; p and q of the current
// node live in this request's work rows pw, qw [V].
__global__ void __launch_bounds__(kThreads) qratio_walk_kernel(QratioArgs a) {
  pdl_begin();
  __shared__ float redf[32];
  __shared__ unsigned long long redk[32];
  __shared__ int s_next, s_kids[kMaxK], s_nk;
  const int b = blockIdx.x;
  const unsigned long long rid = a.round_ptr ? *a.round_ptr : a.round_id;
  const size_t tb = (size_t)b * a.M1;
  float* pw = a.pw + (size_t)b * a.V;
  float* qw = a.qw + (size_t)b * a.V;
  int* path = a.path + (size_t)b * a.D;
  int* out = a.out_tokens + (size_t)b * (a.D + 1);
  for (int i = threadIdx.x; i < a.D; i += blockDim.x) path[i] = -1;
  for (int i = threadIdx.x; i <= a.D; i += blockDim.x) out[i] = -1;
  __syncthreads();
  int u = 0, n = 0;
  for (int step = 0; step <= a.D; ++step) {
    const float* z = a.z + (tb + u) * a.V;
    const float* ell = a.ell + (tb + u) * a.V;
    // p = softmax(z / T), q = softmax(ell)
    float mz = -INFINITY, me = -INFINITY;
    for (int x = threadIdx.x; x < a.V; x += blockDim.x) {
      mz = fmaxf(mz, z[x] * a.inv_t);
      me = fmaxf(me, ell[x]);
    }
    mz = block_max(mz, redf);
    me = block_max(me, redf);
    float sz = 0.f, se = 0.f;
    for (int x = threadIdx.x; x < a.V; x += blockDim.x) {
      const float pz = __expf(z[x] * a.inv_t - mz), pe = __expf(ell[x] - me);
      pw[x] = pz;
      qw[x] = pe;
      sz += pz;
      se += pe;
    }
    sz = block_sum(sz, redf);
    se = block_sum(se, redf);
    for (int x = threadIdx.x; x < a.V; x += blockDim.x) {
      pw[x] /= sz;
      qw[x] /= se;
    }
    // the node's draws in draw order (pool index)
    if (threadIdx.x == 0) {
      const int nc = min(a.n_child[tb + u], kMaxK);
      for (int c = 0; c < nc; ++c) s_kids[c] = a.child_node[(tb + u) * a.kmax + c];
      for (int i = 1; i < nc; ++i)  // insertion sort by pool index
        for (int j = i; j > 0 && a.pidx[tb + s_kids[j - 1]] > a.pidx[tb + s_kids[j]]; --j) {
          const int t = s_kids[j];
          s_kids[j] = s_kids[j - 1];
          s_kids[j - 1] = t;
        }
      s_nk = nc;
      s_next = -1;
    }
    __syncthreads();
    const int nk = s_nk;
    for (int i = 0; i < nk; ++i) {
      const int c = s_kids[i];
      const int x = a.t_tok[tb + c];
      if (threadIdx.x == 0) {
        const float U = verify_uniform(a.seed, rid, b, u, i);
        if (U * qw[x] < pw[x]) s_next = c;
      }
      __syncthreads();
      if (s_next >= 0) break;
      // rejected: p <- norm(max(0, p - q)) (kept if that is empty), q <- q
      // without x, renormalised
      float zr = 0.f;
      for (int y = threadIdx.x; y < a.V; y += blockDim.x) zr += fmaxf(pw[y] - qw[y], 0.f);
      zr = block_sum(zr, redf);
      const float qx = qw[x];
      __syncthreads();
      for (int y = threadIdx.x; y < a.V; y += blockDim.x) {
        if (zr > 0.f) pw[y] = fmaxf(pw[y] - qw[y], 0.f) / zr;
        qw[y] = (y == x) ? 0.f : (qx < 1.f ? qw[y] / (1.f - qx) : qw[y]);
      }
      __syncthreads();
    }
    const int next = s_next;
    if (next >= 0) {
      if (threadIdx.x == 0) {
        path[n] = next;
        out[n] = a.t_tok[tb + next];
      }
      ++n;
      u = next;
      __syncthreads();
      continue;
    }
    // bonus: Gumbel-argmax of log p over the residual's support (stream 1)
    unsigned long long best = 0ull;
    for (int g4 = threadIdx.x; 4 * g4 < a.V; g4 += blockDim.x) {
      uint64_t w[4];
      gumbel_block(a.seed, rid, b, u, (uint64_t)g4, w);
      for (int j = 0; j < 4; ++j) {
        const int y = 4 * g4 + j;
        if (y >= a.V) break;
        const float py = pw[y];
        if (py > 0.f) {
          const unsigned long long key = skey(__logf(py) + gumbel_from_word(w[j]), y);
          best = key > best ? key : best;
        }
      }
    }
    best = block_max_u64(best, redk);
    if (threadIdx.x == 0) {
      out[n] = best ? (int)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFull)) : 0;
      a.accept_len[b] = n;
    }
    return;
  }
  if (threadIdx.x == 0) a.accept_len[b] = n;  // not reached: every path ends within D steps
}

void launch_qratio_walk(const QratioArgs& a, cudaStream_t st) {
  if (a.B <= 0) return;
  launch_pdl(qratio_walk_kernel, dim3(a.B), dim3(kThreads), 0, st, a);
}

}  // namespace e3
