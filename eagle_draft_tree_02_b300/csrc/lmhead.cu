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
  lm_head_simt_kernel<T><<<grid, 256, 0, st>>>((const T*)H, (const T*)W, R, V, d, hp);
}

// ----------------------------------------------------------------------------- merge: LSE + top-k
__global__ void topk_merge_kernel(HeadParts hp, int* tok, float* logq, float* lse_out) {
  __shared__ float red_v[32];
  __shared__ int red_i[32];
  __shared__ float sh_lse;
  int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = blockDim.x >> 5;
  // log-sum-exp over parts
  float m = -INFINITY;
  for (int p = tid; p < hp.n_parts; p += blockDim.x) m = fmaxf(m, hp.ms[((size_t)p * hp.R + r) * 2]);
  m = warp_max(m);
  if (lane == 0) red_v[wid] = m;
  __syncthreads();
  if (wid == 0) {
    float t = lane < nw ? red_v[lane] : -INFINITY;
    t = warp_max(t);
    if (lane == 0) red_v[0] = t;
  }
  __syncthreads();
  m = red_v[0];
  __syncthreads();
  float s = 0.f;
  for (int p = tid; p < hp.n_parts; p += blockDim.x) {
    const float* ms = hp.ms + ((size_t)p * hp.R + r) * 2;
    if (ms[0] != -INFINITY) s += ms[1] * expf(ms[0] - m);
  }
  s = block_sum(s, red_v);
  if (tid == 0) sh_lse = m + logf(s);
  __syncthreads();
  float lse = sh_lse;
  if (tid == 0 && lse_out) lse_out[r] = lse;
  // k rounds: best candidate strictly after the previous winner in (value desc, token asc)
  float pv = INFINITY;
  int pi = -1;
  for (int j = 0; j < hp.k; ++j) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int c = tid; c < hp.n_parts * hp.k; c += blockDim.x) {
      int p = c / hp.k, q = c % hp.k;
      size_t o = ((size_t)p * hp.R + r) * hp.k + q;
      int i = hp.idx[o];
      if (i < 0) continue;
      float v = hp.val[o];
      if (better(pv, pi, v, i) && better(v, i, bv, bi)) { bv = v; bi = i; }
    }
    warp_best(bv, bi);
    if (lane == 0) { red_v[wid] = bv; red_i[wid] = bi; }
    __syncthreads();
    if (wid == 0) {
      float tv = lane < nw ? red_v[lane] : -INFINITY;
      int ti = lane < nw ? red_i[lane] : 0x7fffffff;
      warp_best(tv, ti);
      if (lane == 0) { red_v[0] = tv; red_i[0] = ti; }
    }
    __syncthreads();
    pv = red_v[0];
    pi = red_i[0];
    __syncthreads();
    if (tid == 0) {
      tok[(size_t)r * hp.k + j] = pi == 0x7fffffff ? -1 : pi;
      logq[(size_t)r * hp.k + j] = pv - lse;
    }
  }
}

void launch_topk_merge(const HeadParts& hp, int* tok, float* logq, float* lse, int /*unused*/,
                       cudaStream_t st) {
  if (hp.R <= 0) return;
  topk_merge_kernel<<<hp.R, 256, 0, st>>>(hp, tok, logq, lse);
}

// ----------------------------------------------------------------------------- verify head
template <typename T>
__global__ void __launch_bounds__(256) verify_head_simt_kernel(const T* __restrict__ H,
                                                               const T* __restrict__ W,
                                                               VerifyHeadArgs a) {
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
        float g = z * a.inv_t + verify_gumbel(a.seed, a.round_id, b, u, x);
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
  verify_head_simt_kernel<T><<<grid, 256, 0, st>>>((const T*)H, (const T*)W, a);
}

__global__ void verify_merge_kernel(VerifyHeadArgs a, float* z_max, int* z_arg, float* lse,
                                    int* g_arg, float* g_max) {
  int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= a.R) return;
  float zb = -INFINITY, gb = -INFINITY, m = -INFINITY;
  int zi = 0x7fffffff, gi = 0x7fffffff;
  for (int p = 0; p < a.n_parts; ++p) {
    const float* o = a.part + ((size_t)p * a.R + r) * 6;
    int i = __float_as_int(o[1]);
    if (better(o[0], i, zb, zi)) { zb = o[0]; zi = i; }
    int j = __float_as_int(o[5]);
    if (better(o[4], j, gb, gi)) { gb = o[4]; gi = j; }
    m = fmaxf(m, o[2]);
  }
  float s = 0.f;
  for (int p = 0; p < a.n_parts; ++p) {
    const float* o = a.part + ((size_t)p * a.R + r) * 6;
    if (o[2] != -INFINITY) s += o[3] * expf(o[2] - m);
  }
  z_max[r] = zb;
  z_arg[r] = zi == 0x7fffffff ? -1 : zi;
  lse[r] = m + logf(s);
  g_arg[r] = gi == 0x7fffffff ? -1 : gi;
  if (g_max) g_max[r] = gb;
}

void launch_verify_merge(const VerifyHeadArgs& a, float* z_max, int* z_arg, float* lse, int* g_arg,
                         float* g_max, cudaStream_t st) {
  if (a.R <= 0) return;
  verify_merge_kernel<<<(a.R + 127) / 128, 128, 0, st>>>(a, z_max, z_arg, lse, g_arg, g_max);
}

template void launch_lm_head_simt<float>(const void*, const void*, int, int, int, const HeadParts&,
                                         cudaStream_t);
template void launch_verify_head_simt<float>(const void*, const void*, const VerifyHeadArgs&,
                                             cudaStream_t);

}  // namespace e3
