// Two-stage draft head: low-rank recall, exact rerank (EAGLE-4 blog, section
// 关于 Efficient LM Head, and the paragraph on the Efficient LM Head: a
// low-rank head scores the whole vocabulary, its top candidates are scored
// again with the full LM head).
//
// Reading of the pages (they give no formula): l = U (V_lr h) scores the
// vocabulary; C = the lr_cand best tokens by (l desc, token asc); the exact
// logits W_lm[c] . h of c in C give log q normalised over C ("recall +
// rerank"), and the node's children are the k best of C.
//
// The low-rank scores never reach HBM.  A sample of the vocabulary (its first
// kLrSampleTokens tokens) yields the maximum of every 32-token group; since C
// groups each hold a score at least as large as the C-th largest group
// maximum, that maximum is a lower bound of the C-th best score over the whole
// vocabulary.  The full pass then appends only the tokens that reach it (a few
// hundred per row for the workloads here), and one block per row sorts them.
// If a row's buffer overflows (for instance when many scores tie), the block
// finds the exact top C again by a radix select over recomputed scores.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "lowrank.h"

namespace e3 {

namespace {
constexpr int kSelThreads = 512;

__device__ __forceinline__ uint32_t ord_f32(float f) {  // order-preserving map to uint32
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
// larger key = better under (score desc, token asc)
__device__ __forceinline__ unsigned long long lr_key(float v, int tok) {
  return ((unsigned long long)ord_f32(v) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)tok);
}

template <typename T>
__device__ __forceinline__ float act_at(const T* base, int r, int K, int j, bool split) {
  const T* row = base + act_row(r, K, split);
  float v = ldf(row + j);
  if (split) v += ldf(row + K + j);
  return v;
}
}  // namespace

// ----------------------------------------------------------------------------- reduce + store
template <typename T>
__global__ void reduce_store_kernel(int R, int N, int S, const float* __restrict__ part, T* out,
                                    bool split) {
  pdl_begin();
  const size_t n = (size_t)R * N;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    float v = part[i];
    for (int s = 1; s < S; ++s) v += part[(size_t)s * n + i];
    const int r = (int)(i / N), c = (int)(i % N);
    st_act(out + act_row(r, N, split), N, c, v, split);
  }
}

template <typename T>
void launch_reduce_store(int R, int N, int S, const float* part, void* out, bool split,
                         cudaStream_t st) {
  const size_t n = (size_t)R * N;
  if (!n) return;
  int blocks = (int)std::min<size_t>((n + 255) / 256, 148 * 8);
  launch_pdl(reduce_store_kernel<T>, dim3(blocks), dim3(256), 0, st, R, N, S, part, (T*)out, split);
}

// ----------------------------------------------------------------------------- fp32 low-rank pass
// One warp per (32-token group, row): lane = token.  mode 0: group maxima of
// the sample; mode 1: append tokens whose score reaches the row's threshold.
int lowrank_simt_groups(int V) { return (std::min(V, kLrSampleTokens) + 31) / 32; }

template <typename T>
__global__ void lowrank_simt_kernel(int mode, LowRankArgs a) {
  pdl_begin();
  const int g = blockIdx.x, r = blockIdx.y, lane = threadIdx.x;
  const int x = g * 32 + lane;
  const bool valid = x < a.V;
  float v = -INFINITY;
  if (valid) {
    const T* u = (const T*)a.U + (size_t)x * a.r;
    float acc = 0.f;
    for (int j = 0; j < a.r; ++j) acc = fmaf(ldf(u + j), act_at((const T*)a.t, r, a.r, j, a.t_split), acc);
    v = acc;
  }
  if (mode == 0) {
    const float m = warp_max(v);
    if (lane == 0) a.gmax[(size_t)g * a.R + r] = m;
    return;
  }
  const bool q = valid && v >= a.thr[r];
  const unsigned bal = __ballot_sync(0xffffffffu, q);
  if (!bal) return;
  int base = 0;
  if (lane == 0) base = atomicAdd(a.cnt + r, __popc(bal));
  base = __shfl_sync(0xffffffffu, base, 0);
  if (q) {
    const int pos = base + __popc(bal & ((1u << lane) - 1u));
    if (pos < kLrCap) {
      a.cval[(size_t)r * kLrCap + pos] = v;
      a.ctok[(size_t)r * kLrCap + pos] = x;
    }
  }
}

template <typename T>
void launch_lowrank_simt(int mode, const LowRankArgs& a, cudaStream_t st) {
  const int groups = mode == 0 ? lowrank_simt_groups(a.V) : (a.V + 31) / 32;
  dim3 grid(groups, a.R);
  launch_pdl(lowrank_simt_kernel<T>, dim3(grid), dim3(32), 0, st, mode, a);
}

// ----------------------------------------------------------------------------- threshold
__global__ void __launch_bounds__(512) lowrank_threshold_kernel(LowRankArgs a) {
  pdl_begin();
  __shared__ float sv[1024];
  __shared__ float result;
  const int r = blockIdx.x, tid = threadIdx.x, G = a.n_groups;
  if (tid == 0) {
    result = -INFINITY;
    a.cnt[r] = 0;
  }
  if (G < a.C) {  // fewer groups than candidates: every token qualifies
    __syncthreads();
    if (tid == 0) a.thr[r] = -INFINITY;
    return;
  }
  for (int g = tid; g < G; g += blockDim.x) sv[g] = a.gmax[(size_t)g * a.R + r];
  __syncthreads();
  // the element of rank C-1 under (value desc, group asc)
  for (int g = tid; g < G; g += blockDim.x) {
    const float v = sv[g];
    int rank = 0;
    for (int h = 0; h < G; ++h) rank += (sv[h] > v) || (sv[h] == v && h < g);
    if (rank == a.C - 1) result = v;
  }
  __syncthreads();
  if (tid == 0) a.thr[r] = result;
}

void launch_lowrank_threshold(const LowRankArgs& a, cudaStream_t st) {
  launch_pdl(lowrank_threshold_kernel, dim3(a.R), dim3(512), 0, st, a);
}

// ----------------------------------------------------------------------------- select + rescore
// Bitonic sort of n = 2^p keys in shared memory, best first.
__device__ void sort_keys_desc(unsigned long long* key, int n) {
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      __syncthreads();
      for (int i = threadIdx.x; i < (n >> 1); i += blockDim.x) {
        const int lo = 2 * stride * (i / stride) + (i % stride);
        const int hi = lo + stride;
        const bool desc = ((lo & size) == 0);
        const unsigned long long a = key[lo], b = key[hi];
        if ((a < b) == desc) {
          key[lo] = b;
          key[hi] = a;
        }
      }
    }
  }
  __syncthreads();
}

// Exact top-C keys of one row by a most-significant-digit radix select over
// scores recomputed on CUDA cores (used only when the row's buffer
// overflowed).  Writes the C keys, sorted best first, to key[0, C).
template <typename T>
__device__ void exact_topc(const LowRankArgs& a, int r, const float* t_s, unsigned long long* key,
                           unsigned* hist, int* sh_n, unsigned long long* sh_prefix) {
  const int tid = threadIdx.x;
  unsigned long long prefix = 0ull;  // fixed high digits of the C-th key
  int need = a.C;                    // rank of that key among keys with this prefix
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0u;
    __syncthreads();
    for (int x = tid; x < a.V; x += blockDim.x) {
      const T* u = (const T*)a.U + (size_t)x * a.r;
      float acc = 0.f;
      for (int j = 0; j < a.r; ++j) acc = fmaf(ldf(u + j), t_s[j], acc);
      const unsigned long long k = lr_key(acc, x);
      if (shift == 56 || (k >> (shift + 8)) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid == 0) {
      int acc = 0, b = 255;
      for (; b > 0; --b) {
        if (acc + (int)hist[b] >= need) break;
        acc += hist[b];
      }
      *sh_prefix = (prefix << 8) | (unsigned long long)b;
      *sh_n = need - acc;
    }
    __syncthreads();
    prefix = *sh_prefix;
    need = *sh_n;
    __syncthreads();
  }
  // prefix is now the C-th best key: collect every key >= it (exactly C)
  if (tid == 0) *sh_n = 0;
  for (int i = tid; i < 128; i += blockDim.x) key[i] = 0ull;
  __syncthreads();
  for (int x = tid; x < a.V; x += blockDim.x) {
    const T* u = (const T*)a.U + (size_t)x * a.r;
    float acc = 0.f;
    for (int j = 0; j < a.r; ++j) acc = fmaf(ldf(u + j), t_s[j], acc);
    const unsigned long long k = lr_key(acc, x);
    if (k >= prefix) {
      const int pos = atomicAdd(sh_n, 1);
      if (pos < a.C) key[pos] = k;
    }
  }
  __syncthreads();
  sort_keys_desc(key, 128);
}

// Per row: the C candidates in low-rank order (score desc, token asc) from the
// appended buffer (or, after an overflow, the exact radix select), written to
// sel_tok and, when asked, to the exported candidate lists.  Resets the row's
// rescoring counter.
template <typename T>
__global__ void __launch_bounds__(kSelThreads) lowrank_select_kernel(LowRankArgs a) {
  pdl_begin();
  extern __shared__ unsigned long long sel_smem[];
  unsigned long long* key = sel_smem;                   // [kLrCap]
  float* t_s = reinterpret_cast<float*>(key + kLrCap);  // [r]
  __shared__ unsigned hist[256];
  __shared__ int sh_n;
  __shared__ unsigned long long sh_prefix;
  const int r = blockIdx.x, tid = threadIdx.x, C = a.C;

  const int n = a.cnt[r];
  if (n <= kLrCap - 128) {
    // the buffer's keys are distinct (one per token): the key of rank i (by
    // count of larger keys) goes to top[i] for i < C.  top[] sits past the
    // n buffered keys (n <= kLrCap - 128 here, see the overflow test below).
    for (int i = tid; i < n; i += blockDim.x)
      key[i] = lr_key(a.cval[(size_t)r * kLrCap + i], a.ctok[(size_t)r * kLrCap + i]);
    unsigned long long* top = key + (kLrCap - 128);
    for (int i = tid; i < 128; i += blockDim.x) top[i] = 0ull;
    __syncthreads();
    for (int i = tid; i < n; i += blockDim.x) {
      const unsigned long long ki = key[i];
      int rank = 0;
      for (int j = 0; j < n; ++j) rank += key[j] > ki;
      if (rank < C) top[rank] = ki;
    }
    __syncthreads();
    for (int i = tid; i < C; i += blockDim.x) key[i] = top[i];
    __syncthreads();
  } else {
    for (int j = tid; j < a.r; j += blockDim.x) t_s[j] = act_at((const T*)a.t, r, a.r, j, a.t_split);
    __syncthreads();
    exact_topc<T>(a, r, t_s, key, hist, &sh_n, &sh_prefix);
  }
  int* out = a.sel_tok + (size_t)r * C;
  for (int i = tid; i < C; i += blockDim.x) out[i] = (int)(0xFFFFFFFFu - (uint32_t)(key[i] & 0xFFFFFFFFull));
  if (a.cand_out) {
    const int b = r / a.cand_rpr, j = r % a.cand_rpr;
    int* dst = a.cand_out + ((size_t)b * a.cand_n_exp + a.cand_slot0 + j) * C;
    for (int i = tid; i < C; i += blockDim.x) dst[i] = (int)(0xFFFFFFFFu - (uint32_t)(key[i] & 0xFFFFFFFFull));
  }
  if (tid == 0) a.sel_done[r] = 0;
}

// Exact logits of the candidates: block (row, group of kRescoreWarps
// candidates), one warp per candidate, every load of the head row in flight
// before the products.  The last block of a row to finish takes log q over
// the C candidates and the k best of them.
constexpr int kRescoreWarps = 8;

template <typename T>
__global__ void __launch_bounds__(32 * kRescoreWarps) lowrank_rescore_kernel(LowRankArgs a) {
  pdl_begin();
  extern __shared__ float h_s[];  // [d]
  __shared__ int s_last;
  __shared__ float red[32];
  const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int C = a.C;
  for (int j = tid; j < a.d; j += blockDim.x) h_s[j] = act_at((const T*)a.H, r, a.d, j, a.h_split);
  __syncthreads();
  const int c = blockIdx.y * kRescoreWarps + wid;
  if (c < C) {
    const int x = a.sel_tok[(size_t)r * C + c];
    float z = -INFINITY;
    if (x < 0 || x >= a.V) {  // only after an aborted low-rank pass
      if (lane == 0) raise_flag(a.flags, FLAG_TOKEN_RANGE);
    } else {
      const T* w = (const T*)a.W + (size_t)x * a.d;
      constexpr int VEC = 16 / sizeof(T);
      constexpr int U = 8;  // 16-byte loads in flight per lane
      float acc[U];
#pragma unroll
      for (int u = 0; u < U; ++u) acc[u] = 0.f;
      if (a.d % VEC == 0 && ((uintptr_t)w & 15) == 0) {
        for (int j0 = lane * VEC; j0 < a.d; j0 += 32 * VEC * U) {
          uint4 raw[U];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int j = j0 + u * 32 * VEC;
            raw[u] = j < a.d ? __ldg(reinterpret_cast<const uint4*>(w + j)) : make_uint4(0u, 0u, 0u, 0u);
          }
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int j = j0 + u * 32 * VEC;
            if (j < a.d) {
              const T* e = reinterpret_cast<const T*>(&raw[u]);
#pragma unroll
              for (int v = 0; v < VEC; ++v) acc[u] = fmaf(ldf(e + v), h_s[j + v], acc[u]);
            }
          }
        }
      } else {
        for (int j = lane; j < a.d; j += 32) acc[0] = fmaf(ldf(w + j), h_s[j], acc[0]);
      }
      float t = 0.f;
#pragma unroll
      for (int u = 0; u < U; ++u) t += acc[u];
      z = warp_sum(t);
    }
    if (lane == 0) a.sel_z[(size_t)r * C + c] = z;
  }
  // the last block of this row to finish: log q over the C candidates, top k
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(a.sel_done + r, 1) == (int)gridDim.y - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const float* ex = a.sel_z + (size_t)r * C;
  const int* ctk = a.sel_tok + (size_t)r * C;
  float m = -INFINITY;
  for (int i = tid; i < C; i += blockDim.x) m = fmaxf(m, ex[i]);
  m = warp_max(m);
  if (lane == 0) red[wid] = m;
  __syncthreads();
  if (tid < 32) {
    float v = tid < kRescoreWarps ? red[tid] : -INFINITY;
    v = warp_max(v);
    if (tid == 0) red[0] = v;
  }
  __syncthreads();
  m = red[0];
  float s = 0.f;
  for (int i = tid; i < C; i += blockDim.x) s += expf(ex[i] - m);
  s = block_sum(s, red);
  const float lse = m + logf(s);
  // the k best of C by (exact logit desc, token asc)
  for (int i = tid; i < C; i += blockDim.x) {
    const float v = ex[i];
    const int x = ctk[i];
    int rank = 0;
    for (int o = 0; o < C; ++o) rank += better(ex[o], ctk[o], v, x);
    if (rank < a.k) {
      a.tok[(size_t)r * a.k + rank] = x;
      a.logq[(size_t)r * a.k + rank] = v - lse;
    }
  }
  if (tid == 0 && a.lse) a.lse[r] = lse;
}

template <typename T>
void launch_lowrank_select(const LowRankArgs& a, cudaStream_t st) {
  const size_t smem = (size_t)kLrCap * 8 + (size_t)a.r * 4;
  smem_limit((const void*)lowrank_select_kernel<T>, 200 * 1024);  // refusal: the launch fails
  launch_pdl(lowrank_select_kernel<T>, dim3(a.R), dim3(kSelThreads), smem, st, a);
  smem_limit((const void*)lowrank_rescore_kernel<T>, 200 * 1024);
  launch_pdl(lowrank_rescore_kernel<T>, dim3(a.R, (a.C + kRescoreWarps - 1) / kRescoreWarps),
             dim3(32 * kRescoreWarps), (size_t)a.d * 4, st, a);
}

template void launch_reduce_store<float>(int, int, int, const float*, void*, bool, cudaStream_t);
template void launch_reduce_store<bf16>(int, int, int, const float*, void*, bool, cudaStream_t);
template void launch_lowrank_simt<float>(int, const LowRankArgs&, cudaStream_t);
template void launch_lowrank_select<float>(const LowRankArgs&, cudaStream_t);
template void launch_lowrank_select<bf16>(const LowRankArgs&, cudaStream_t);

}  // namespace e3
