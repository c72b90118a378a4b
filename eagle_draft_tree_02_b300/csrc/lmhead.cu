// LM heads with fused epilogues, CUDA-core version (fp32 storage).
//
// Draft head (EAGLE-4 blog, section 关于 Efficient LM Head: the draft LM head
// is the costly part of a one-layer drafter): each block computes a 64-token x
// 64-row tile of logits and immediately reduces it to, per row, the tile's
// running (max, sum of exp) and its k best (logit, token).  A merge kernel
// combines the tiles into log-sum-exp and the global top-k, so the full logits
// never reach HBM.
//
// Target head of the verify step: per row (tree node) the tile's best logit
// and token, (max, sum exp) of z/T, the Gumbel-argmax of z/T over tokens that
// are not children of the node, and the logits at the children's tokens.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "philox.cuh"

namespace e3 {

namespace {
constexpr int TB = 64, TK = 16;  // tile (rows and tokens), K slice
}

int lm_head_simt_parts(int V) { return (V + TB - 1) / TB; }
int verify_head_simt_parts(int V) { return (V + TB - 1) / TB; }

// 64x64 tile of logits L[row][token] = H[r0 + row] . W[n0 + token] into shared memory.
template <typename T>
__device__ void logits_tile(const T* __restrict__ H, const T* __restrict__ W, int R, int V, int d,
                            int r0, int n0, float (*Lt)[TB + 1], float (*Hs)[TB + 4],
                            float (*Ws)[TB + 4]) {
  int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  int lr = tid >> 2, lk = (tid & 3) * 4;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < d; k0 += TK) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      int kk = k0 + lk + i;
      Hs[lk + i][lr] = (r0 + lr < R && kk < d) ? ldf(H + (size_t)(r0 + lr) * d + kk) : 0.f;
      Ws[lk + i][lr] = (n0 + lr < V && kk < d) ? ldf(W + (size_t)(n0 + lr) * d + kk) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = Hs[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Ws[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) Lt[ty * 4 + i][tx * 4 + j] = acc[i][j];
  __syncthreads();
}

template <typename T>
__global__ void __launch_bounds__(256) lm_head_simt_kernel(const T* __restrict__ H,
                                                           const T* __restrict__ W, int R, int V,
                                                           int d, HeadParts hp) {
  pdl_begin();
  __shared__ float Lt[TB][TB + 1];
  __shared__ float Hs[TK][TB + 4];
  __shared__ float Ws[TK][TB + 4];
  int part = blockIdx.x, r0 = blockIdx.y * TB, n0 = part * TB;
  logits_tile<T>(H, W, R, V, d, r0, n0, Lt, Hs, Ws);
  int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int rl = wid; rl < TB; rl += 8) {
    int r = r0 + rl;
    if (r >= R) break;
    int i0 = n0 + lane, i1 = n0 + lane + 32;
    float v0 = i0 < V ? Lt[rl][lane] : -INFINITY;
    float v1 = i1 < V ? Lt[rl][lane + 32] : -INFINITY;
    float m = warp_max(fmaxf(v0, v1));
    float s = warp_sum(expf(v0 - m) + expf(v1 - m));
    size_t pr = (size_t)part * R + r;
    if (lane == 0) {
      hp.ms[pr * 2] = m;
      hp.ms[pr * 2 + 1] = s;
    }
    if (i0 >= V) i0 = 0x7fffffff;
    if (i1 >= V) i1 = 0x7fffffff;
    for (int j = 0; j < hp.k; ++j) {
      float bv;
      int bi;
      if (better(v0, i0, v1, i1)) { bv = v0; bi = i0; } else { bv = v1; bi = i1; }
      warp_best(bv, bi);
      if (lane == 0) {
        hp.val[pr * hp.k + j] = bv;
        hp.idx[pr * hp.k + j] = bi == 0x7fffffff ? -1 : bi;
      }
      if (bi == i0) { v0 = -INFINITY; i0 = 0x7fffffff; }
      if (bi == i1) { v1 = -INFINITY; i1 = 0x7fffffff; }
    }
  }
}

template <typename T>
void launch_lm_head_simt(const void* H, const void* W, int R, int V, int d, const HeadParts& hp,
                         cudaStream_t st) {
  if (R <= 0) return;
  dim3 grid(lm_head_simt_parts(V), (R + TB - 1) / TB);
  launch_pdl(lm_head_simt_kernel<T>, dim3(grid), dim3(256), 0, st, (const T*)H, (const T*)W, R, V, d, hp);
}

// ----------------------------------------------------------------------------- merge: LSE + top-k
// One block per row.  Each thread folds a strided subset of the partials into
// an online (max, sum-exp) and a sorted register list of its best k (value,
// token); partial lists are sorted best-first, so a list is abandoned at its
// first entry that does not beat the thread's current k-th.  Then k block-wide
// rounds each take the best list head, and its owner pops it.  Token ids are
// unique across partials, so (value desc, token asc) is a strict order.
namespace {
constexpr int kMergeThreads = 512;

// (m, s) <- (m, s) (+) (m2, s2) for s = sum exp(x - m)
__device__ __forceinline__ void lse_fold(float& m, float& s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m2 > m) {
    s = s * expf(m - m2) + s2;  // exp(-inf) = 0 covers the empty state
    m = m2;
  } else {
    s += s2 * expf(m2 - m);
  }
}

__device__ __forceinline__ void warp_lse(float& m, float& s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    lse_fold(m, s, m2, s2);
  }
}
}  // namespace

template <int K>
__global__ void __launch_bounds__(kMergeThreads) topk_merge_kernel(HeadParts hp, int* tok, float* logq,
                                                                   float* lse_out) {
  pdl_begin();
  if (hp.skip && *hp.skip == 0) return;
  __shared__ float red_m[32], red_s[32];
  const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int nw = blockDim.x >> 5, k = K;
  float m = -INFINITY, s = 0.f;
  float lv[K];
  int li[K];
#pragma unroll
  for (int j = 0; j < K; ++j) {
    lv[j] = -INFINITY;
    li[j] = 0x7fffffff;
  }
  float tv = -INFINITY;  // current k-th kept (value, token)
  int ti = 0x7fffffff;
  for (int p = tid; p < hp.n_parts; p += blockDim.x) {
    const size_t pr = (size_t)p * hp.R + r;
    const float* pv = hp.val + pr * k;
    const int* pi = hp.idx + pr * k;
    // the partial's whole list first: independent loads, one round trip
    float pvs[K];
    int pis[K];
#pragma unroll
    for (int q = 0; q < K; ++q) {
      pvs[q] = pv[q];
      pis[q] = pi[q];
    }
    lse_fold(m, s, hp.ms[pr * 2], hp.ms[pr * 2 + 1]);
#pragma unroll
    for (int q = 0; q < K; ++q) {
      const int i = pis[q];
      const float v = pvs[q];
      if (i < 0 || !better(v, i, tv, ti)) break;
      float cv = v;
      int ci = i;
#pragma unroll
      for (int j = 0; j < K; ++j) {
        if (better(cv, ci, lv[j], li[j])) {
          const float t = lv[j];
          const int u = li[j];
          lv[j] = cv;
          li[j] = ci;
          cv = t;
          ci = u;
        }
      }
      tv = lv[K - 1];
      ti = li[K - 1];
    }
  }
  // block log-sum-exp
  warp_lse(m, s);
  if (lane == 0) {
    red_m[wid] = m;
    red_s[wid] = s;
  }
  // each warp's k best: k rounds of a warp argmax over its lanes' list heads
  __shared__ float wv[kMergeThreads / 32][K];
  __shared__ int wi_s[kMergeThreads / 32][K];
#pragma unroll
  for (int j = 0; j < K; ++j) {
    float bv = lv[0];
    int bi = li[0];
    warp_best(bv, bi);
    if (bi != 0x7fffffff && li[0] == bi) {  // the owner pops its head
#pragma unroll
      for (int q = 0; q < K - 1; ++q) {
        lv[q] = lv[q + 1];
        li[q] = li[q + 1];
      }
      lv[K - 1] = -INFINITY;
      li[K - 1] = 0x7fffffff;
    }
    if (lane == 0) {
      wv[wid][j] = bv;
      wi_s[wid][j] = bi;
    }
  }
  __syncthreads();
  if (wid != 0) return;
  float m2 = lane < nw ? red_m[lane] : -INFINITY;
  float s2 = lane < nw ? red_s[lane] : 0.f;
  warp_lse(m2, s2);
  const float lse = m2 + logf(s2);
  if (lane == 0 && lse_out) lse_out[r] = lse;
  // the block's k best: k rounds of a warp argmax over the warps' sorted lists
  int head = 0;  // lane j walks warp j's list
#pragma unroll
  for (int j = 0; j < K; ++j) {
    float bv = (lane < nw && head < K) ? wv[lane][head] : -INFINITY;
    int bi = (lane < nw && head < K) ? wi_s[lane][head] : 0x7fffffff;
    const int mine = bi;
    warp_best(bv, bi);
    if (bi != 0x7fffffff && mine == bi) ++head;
    if (lane == 0) {
      tok[(size_t)r * k + j] = bi == 0x7fffffff ? -1 : bi;
      logq[(size_t)r * k + j] = bv - lse;
    }
  }
}

void launch_topk_merge(const HeadParts& hp, int* tok, float* logq, float* lse, int /*unused*/,
                       cudaStream_t st) {
  if (hp.R <= 0) return;
  switch (hp.k) {
#define E3_MERGE_CASE(K) \
  case K:                \
    launch_pdl(topk_merge_kernel<K>, dim3(hp.R), dim3(kMergeThreads), 0, st, hp, tok, logq, lse); \
    break;
    E3_MERGE_CASE(1) E3_MERGE_CASE(2) E3_MERGE_CASE(3) E3_MERGE_CASE(4) E3_MERGE_CASE(5)
    E3_MERGE_CASE(6) E3_MERGE_CASE(7) E3_MERGE_CASE(8) E3_MERGE_CASE(9) E3_MERGE_CASE(10)
    E3_MERGE_CASE(11) E3_MERGE_CASE(12) E3_MERGE_CASE(13) E3_MERGE_CASE(14) E3_MERGE_CASE(15)
    E3_MERGE_CASE(16)
#undef E3_MERGE_CASE
    default:
      break;  // k is checked to lie in 1..16 before any launch
  }
}

// ----------------------------------------------------------------------------- verify head
template <typename T>
__global__ void __launch_bounds__(256) verify_head_simt_kernel(const T* __restrict__ H,
                                                               const T* __restrict__ W,
                                                               VerifyHeadArgs a) {
  pdl_begin();
  __shared__ float Lt[TB][TB + 1];
  __shared__ float Hs[TK][TB + 4];
  __shared__ float Ws[TK][TB + 4];
  int part = blockIdx.x, r0 = blockIdx.y * TB, n0 = part * TB;
  logits_tile<T>(H, W, a.R, a.V, a.d, r0, n0, Lt, Hs, Ws);
  int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int rl = wid; rl < TB; rl += 8) {
    int r = r0 + rl;
    if (r >= a.R) break;
    int b = r / a.M1, u = r % a.M1;
    float zb = -INFINITY, gb = -INFINITY, m = -INFINITY;
    int zi = 0x7fffffff, gi = 0x7fffffff;
    float zz[2];
    int xx[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      int x = n0 + lane + 32 * h;
      xx[h] = x;
      zz[h] = -INFINITY;
      if (x >= a.V) continue;
      float z = Lt[rl][lane + 32 * h];
      zz[h] = z;
      if (better(z, x, zb, zi)) { zb = z; zi = x; }
      m = fmaxf(m, z * a.inv_t);
      bool child = false;
      for (int c = 0; c < a.kmax; ++c) {
        int ct = a.child_tok[(size_t)r * a.kmax + c];
        if (ct == x) {
          child = true;
          a.child_z[(size_t)r * a.kmax + c] = z;
        }
      }
      if (a.sampling && !child) {
        const unsigned long long rid = a.round_ptr ? *a.round_ptr : a.round_id;
        float g = z * a.inv_t + verify_gumbel(a.seed, rid, b, u, x);
        if (better(g, x, gb, gi)) { gb = g; gi = x; }
      }
    }
    m = warp_max(m);
    float s = 0.f;
#pragma unroll
    for (int h = 0; h < 2; ++h)
      if (xx[h] < a.V) s += expf(zz[h] * a.inv_t - m);
    s = warp_sum(s);
    warp_best(zb, zi);
    warp_best(gb, gi);
    if (lane == 0) {
      float* o = a.part + ((size_t)part * a.R + r) * 6;
      o[0] = zb;
      o[1] = __int_as_float(zi);
      o[2] = m;
      o[3] = s;
      o[4] = gb;
      o[5] = __int_as_float(gi);
    }
  }
}

template <typename T>
void launch_verify_head_simt(const void* H, const void* W, const VerifyHeadArgs& a, cudaStream_t st) {
  if (a.R <= 0) return;
  dim3 grid(verify_head_simt_parts(a.V), (a.R + TB - 1) / TB);
  launch_pdl(verify_head_simt_kernel<T>, dim3(grid), dim3(256), 0, st, (const T*)H, (const T*)W, a);
}

// One block per tree node: best target logit (ties: lowest token), log-sum-exp
// of z/T and the Gumbel-argmax over the partials of every vocabulary tile.
__global__ void __launch_bounds__(256) verify_merge_kernel(VerifyHeadArgs a, float* z_max, int* z_arg,
                                                           float* lse, int* g_arg, float* g_max) {
  pdl_begin();
  __shared__ float sh_zb[32], sh_m[32], sh_s[32], sh_gb[32];
  __shared__ int sh_zi[32], sh_gi[32];
  const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int nw = blockDim.x >> 5;
  float zb = -INFINITY, gb = -INFINITY, m = -INFINITY, s = 0.f;
  int zi = 0x7fffffff, gi = 0x7fffffff;
  for (int p = tid; p < a.n_parts; p += blockDim.x) {
    const float* o = a.part + ((size_t)p * a.R + r) * 6;
    const float v0 = o[0], v2 = o[2], v3 = o[3], v4 = o[4];
    const int i1 = __float_as_int(o[1]), i5 = __float_as_int(o[5]);
    if (better(v0, i1, zb, zi)) { zb = v0; zi = i1; }
    if (better(v4, i5, gb, gi)) { gb = v4; gi = i5; }
    lse_fold(m, s, v2, v3);
  }
  warp_best(zb, zi);
  warp_best(gb, gi);
  warp_lse(m, s);
  if (lane == 0) {
    sh_zb[wid] = zb; sh_zi[wid] = zi; sh_gb[wid] = gb; sh_gi[wid] = gi; sh_m[wid] = m; sh_s[wid] = s;
  }
  __syncthreads();
  if (wid == 0) {
    zb = lane < nw ? sh_zb[lane] : -INFINITY;
    zi = lane < nw ? sh_zi[lane] : 0x7fffffff;
    gb = lane < nw ? sh_gb[lane] : -INFINITY;
    gi = lane < nw ? sh_gi[lane] : 0x7fffffff;
    m = lane < nw ? sh_m[lane] : -INFINITY;
    s = lane < nw ? sh_s[lane] : 0.f;
    warp_best(zb, zi);
    warp_best(gb, gi);
    warp_lse(m, s);
    if (lane == 0) {
      z_max[r] = zb;
      z_arg[r] = zi == 0x7fffffff ? -1 : zi;
      lse[r] = m + logf(s);
      g_arg[r] = gi == 0x7fffffff ? -1 : gi;
      if (g_max) g_max[r] = gb;
    }
  }
}

void launch_verify_merge(const VerifyHeadArgs& a, float* z_max, int* z_arg, float* lse, int* g_arg,
                         float* g_max, cudaStream_t st) {
  if (a.R <= 0) return;
  launch_pdl(verify_merge_kernel, dim3(a.R), dim3(256), 0, st, a, z_max, z_arg, lse, g_arg, g_max);
}

template void launch_lm_head_simt<float>(const void*, const void*, int, int, int, const HeadParts&,
                                         cudaStream_t);
template void launch_verify_head_simt<float>(const void*, const void*, const VerifyHeadArgs&,
                                             cudaStream_t);

}  // namespace e3
