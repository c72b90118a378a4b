// Decoder-layer kernels around the GEMMs of the one-layer EAGLE-3 drafter.
//
// "EAGLE-3 精读" §1 (paragraph 2): the decoder combines the fused target
// feature g (or, along draft paths, its own state: §2 Training-Time Test) with
// the token embedding.  This build reads that as x = [rms(E[y]); rms(hid)],
// followed by one pre-norm Llama-style layer:
//   q, k, v = W_q x, W_k x, W_v x   (rotate-half RoPE on q, k)
//   r = hid + W_o attn(q, K, V);  z = rms(r)
//   s = r + W_down(silu(W_gate z) * W_up z);  h = rms(s)
// Every GEMM writes fp32 split-K partials [S][R][N]; the kernels here sum the
// partials and apply the element-wise parts.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace e3 {

namespace cg = cooperative_groups;

// Row kernels (the ones with a norm over a whole row) give each of a few rows
// a cluster of CL = 8 CTAs, each taking one slice of the row's columns; the
// slices' sums of squares meet in distributed shared memory.  (With one block
// per row, the few rows of a draft pass ran on as many SMs, each pulling its
// row's split-K partials alone.)  From kRowClusterMaxRows rows on -- prefill
// chunks, wide verify passes -- one 1024-thread block per row (CL = 1)
// already fills the GPU and costs less.
constexpr int kRowCluster = 8;
constexpr int kRowClusterMaxRows = 148;
constexpr int kRowThreads = 256;      // with clusters
constexpr int kRowThreadsWide = 1024;  // one block per row

struct RowSlice {
  int r, c0, c1;  // row, columns [c0, c1)
};
template <int CL>
__device__ __forceinline__ RowSlice row_slice(int n) {
  const int cw = (n + CL - 1) / CL;
  RowSlice sl;
  sl.r = blockIdx.x / CL;
  sl.c0 = min(n, (int)(blockIdx.x % CL) * cw);
  sl.c1 = min(n, sl.c0 + cw);
  return sl;
}
// v[i] := the sum of v[i] over every thread of the row's CL CTAs, the same
// value (same summation order) in every CTA.  The second cluster barrier keeps
// each CTA alive until its peers have read its sums.
template <int CL, int N>
__device__ __forceinline__ void cluster_sum(float (&v)[N], float* red) {
  __shared__ float mine[N];
#pragma unroll
  for (int i = 0; i < N; ++i) v[i] = block_sum(v[i], red);
  if (CL == 1) return;
  if (threadIdx.x == 0)
#pragma unroll
    for (int i = 0; i < N; ++i) mine[i] = v[i];
  cg::cluster_group cl = cg::this_cluster();
  cl.sync();
#pragma unroll
  for (int i = 0; i < N; ++i) {
    float t = 0.f;
#pragma unroll
    for (int k = 0; k < CL; ++k) t += cl.map_shared_rank(mine, k)[i];
    v[i] = t;
  }
  cl.sync();
}

// ----------------------------------------------------------------------------- x = [rms(E[y]); rms(hid)]
template <typename T, int CL>
__global__ void build_input_kernel(int R, int d, int V, float eps, const int* __restrict__ tok,
                                   const float* __restrict__ hid_base, const int* __restrict__ hid_row,
                                   const T* __restrict__ E, const T* __restrict__ g_emb,
                                   const T* __restrict__ g_hid, T* __restrict__ x, bool split,
                                   int* flags) {
  pdl_begin();
  __shared__ float red[32];
  const RowSlice sl = row_slice<CL>(d);
  const int r = sl.r;
  int t = tok[r];
  if (t < 0 || t >= V) {
    if (threadIdx.x == 0 && sl.c0 == 0) raise_flag(flags, FLAG_TOKEN_RANGE);
    t = t < 0 ? 0 : V - 1;
  }
  const T* e = E + (size_t)t * d;
  const float* h = hid_base + (size_t)hid_row[r] * d;
  float ss[2] = {0.f, 0.f};  // embedding row, hidden row
  for (int j = sl.c0 + threadIdx.x; j < sl.c1; j += blockDim.x) {
    float a = ldf(e + j), b = h[j];
    ss[0] += a * a;
    ss[1] += b * b;
  }
  cluster_sum<CL, 2>(ss, red);
  float ie = rsqrtf(ss[0] / d + eps), ih = rsqrtf(ss[1] / d + eps);
  T* xr = x + act_row(r, 2 * d, split);
  for (int j = sl.c0 + threadIdx.x; j < sl.c1; j += blockDim.x) {
    st_act(xr, 2 * d, j, ldf(e + j) * ie * ldf(g_emb + j), split);
    st_act(xr, 2 * d, d + j, h[j] * ih * ldf(g_hid + j), split);
  }
}

// ----------------------------------------------------------------------------- split-K sum
__device__ __forceinline__ float sum_parts(const float* p, size_t stride, int S) {
  // eight partials' loads in flight at a time
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  int s = 0;
  for (; s + 8 <= S; s += 8) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = p[(size_t)(s + u) * stride];
#pragma unroll
    for (int u = 0; u < 8; ++u) acc[u] += v[u];
  }
  for (; s < S; ++s) acc[0] += p[(size_t)s * stride];
  return ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
}

// g = sum of fusion partials (fp32 [R, d])
__global__ void reduce_parts_kernel(int R, int N, int S, const float* __restrict__ part,
                                    float* __restrict__ out) {
  pdl_begin();
  size_t n = (size_t)R * N;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    out[i] = sum_parts(part + i, n, S);
}

// g = rms(sum of fusion partials) * g_fc: the FC-norm variant, one cluster per row
template <typename T, int CL>
__global__ void reduce_norm_kernel(int R, int N, int S, float eps, const float* __restrict__ part,
                                   const T* __restrict__ g_fc, float* __restrict__ out) {
  pdl_begin();
  __shared__ float red[32];
  const RowSlice sl = row_slice<CL>(N);
  const int r = sl.r;
  const size_t n = (size_t)R * N;
  float ss[1] = {0.f};
  for (int j = sl.c0 + threadIdx.x; j < sl.c1; j += blockDim.x) {
    const float v = sum_parts(part + (size_t)r * N + j, n, S);
    out[(size_t)r * N + j] = v;
    ss[0] += v * v;
  }
  cluster_sum<CL, 1>(ss, red);
  const float inv = rsqrtf(ss[0] / N + eps);
  for (int j = sl.c0 + threadIdx.x; j < sl.c1; j += blockDim.x)
    out[(size_t)r * N + j] *= inv * ldf(g_fc + j);
}

// ----------------------------------------------------------------------------- RoPE + KV write
// One thread per rotate-half pair (j, j + dh/2) of one head.  Heads are laid
// out [q heads | k heads | v heads] in the partials when has_q, else [k | v].
template <typename T>
__global__ void qkv_epilogue_kernel(QkvEpi p) {
  pdl_begin();
  int r = blockIdx.y;
  int half = p.dh / 2;
  int nh = (p.has_q ? p.Hq : 0) + 2 * p.Hkv;
  int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= nh * half) return;
  int hh = idx / half, j = idx % half;
  int ld = nh * p.dh;
  size_t stride = (size_t)p.R * ld;
  const float* base = p.part + (size_t)r * ld + (size_t)hh * p.dh;
  float x1 = sum_parts(base + j, stride, p.S);
  float x2 = sum_parts(base + j + half, stride, p.S);
  int pos = p.row_pos[r];
  if (pos < 0 || pos >= p.rope_rows) {
    if (idx == 0) raise_flag(p.flags, FLAG_POS_RANGE);
    return;
  }
  int qh = p.has_q ? p.Hq : 0;
  if (hh < qh + p.Hkv) {  // q or k head: rotate
    float2 cs = p.rope[(size_t)pos * half + j];
    float y1 = x1 * cs.x - x2 * cs.y;
    float y2 = x2 * cs.x + x1 * cs.y;
    x1 = y1;
    x2 = y2;
  }
  if (hh < qh) {
    float* q = p.q_out + (size_t)r * p.Hq * p.dh + (size_t)hh * p.dh;
    q[j] = x1;
    q[j + half] = x2;
    return;
  }
  bool is_v = hh >= qh + p.Hkv;
  int kvh = is_v ? hh - qh - p.Hkv : hh - qh;
  int b = p.row_b[r];
  int dst = p.row_dst[r];
  if (dst >= 0) {  // tree scratch slot of this request: fp32, the library's own format
    size_t off = (((size_t)b * p.tree_slots + dst) * p.Hkv + kvh) * p.dh;
    float* tout = (float*)(is_v ? p.tree_v : p.tree_k) + off;
    tout[j] = x1;
    tout[j + half] = x2;
    return;
  }
  T* out;
  {  // prefix cache at `pos`, in the cache's storage type
    size_t row;
    if (p.page_table) {
      int lp = pos / p.page_size;
      if (lp >= p.max_pages) {
        if (j == 0) raise_flag(p.flags, FLAG_POS_RANGE);
        return;
      }
      int pg = p.page_table[(size_t)b * p.max_pages + lp];
      if (pg < 0 || pg >= p.n_pages) {
        if (j == 0) raise_flag(p.flags, FLAG_PAGE_RANGE);
        return;
      }
      row = (size_t)pg * p.page_size + pos % p.page_size;
    } else {
      if (pos >= p.max_prefix) {
        if (j == 0) raise_flag(p.flags, FLAG_POS_RANGE);
        return;
      }
      row = (size_t)b * p.max_prefix + pos;
    }
    out = (T*)(is_v ? p.cache_v : p.cache_k) + (row * p.Hkv + kvh) * p.dh;
  }
  stf(out + j, x1);
  stf(out + j + half, x2);
}

// ----------------------------------------------------------------------------- r = hid + W_o o;  z = rms(r)
template <typename T, int CL>
__global__ void o_epilogue_kernel(int R, int d, int S, float eps, const float* __restrict__ part,
                                  const float* __restrict__ hid_base, const int* __restrict__ hid_row,
                                  const T* __restrict__ g_post, float* __restrict__ r_out,
                                  T* __restrict__ z_out, bool split, bool post) {
  pdl_begin();
  __shared__ float red[32];
  const RowSlice sl = row_slice<CL>(d);
  const int r = sl.r;
  const float* h = hid_base + (size_t)hid_row[r] * d;
  size_t stride = (size_t)R * d;
  float ss[1] = {0.f};
  for (int j = sl.c0 + threadIdx.x; j < sl.c1; j += blockDim.x) {
    float v = h[j] + sum_parts(part + (size_t)r * d + j, stride, S);
    r_out[(size_t)r * d + j] = v;
    ss[0] += v * v;
  }
  cluster_sum<CL, 1>(ss, red);
  float inv = rsqrtf(ss[0] / d + eps);
  T* zr = z_out + act_row(r, d, split);
  for (int j = sl.c0 + threadIdx.x; j < sl.c1; j += blockDim.x) {
    const float z = r_out[(size_t)r * d + j] * inv * ldf(g_post + j);
    if (post) r_out[(size_t)r * d + j] = z;  // post-norm: the residual stream is normalised too
    st_act(zr, d, j, z, split);
  }
}

// ----------------------------------------------------------------------------- a = silu(W_g z) * (W_u z)
// part: [S][R][2F], gate in columns [0, F), up in [F, 2F)
template <typename T>
__global__ void swiglu_kernel(int R, int F, int S, const float* __restrict__ part, T* __restrict__ a,
                              bool split) {
  pdl_begin();
  size_t n = (size_t)R * F;
  size_t stride = (size_t)R * 2 * F;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    size_t r = i / F, c = i % F;
    const float* p = part + r * 2 * F + c;
    float g = sum_parts(p, stride, S);
    float u = sum_parts(p + F, stride, S);
    st_act(a + act_row((int)r, F, split), F, (int)c, g / (1.f + expf(-g)) * u, split);
  }
}

// ----------------------------------------------------------------------------- s = r + W_down a;  h = rms(s)
template <typename T, int CL>
__global__ void down_epilogue_kernel(int R, int d, int S, float eps, const float* __restrict__ part,
                                     const float* __restrict__ r_in, const T* __restrict__ g_final,
                                     const int* __restrict__ s_dst, float* __restrict__ s_base,
                                     const int* __restrict__ h_dst, T* __restrict__ h_base,
                                     bool split, bool post) {
  pdl_begin();
  __shared__ float red[32];
  extern __shared__ float srow[];  // this CTA's slice of s
  const RowSlice sl = row_slice<CL>(d);
  const int r = sl.r;
  size_t stride = (size_t)R * d;
  float ss[1] = {0.f};
  for (int j = sl.c0 + threadIdx.x; j < sl.c1; j += blockDim.x) {
    float v = r_in[(size_t)r * d + j] + sum_parts(part + (size_t)r * d + j, stride, S);
    srow[j - sl.c0] = v;
    ss[0] += v * v;
  }
  cluster_sum<CL, 1>(ss, red);
  float inv = rsqrtf(ss[0] / d + eps);
  int sd = s_dst ? s_dst[r] : -1;
  int hd = h_dst ? h_dst[r] : r;
  T* hr = h_base + act_row(hd, d, split);
  for (int j = sl.c0 + threadIdx.x; j < sl.c1; j += blockDim.x) {
    const float h = srow[j - sl.c0] * inv * ldf(g_final + j);
    if (sd >= 0) s_base[(size_t)sd * d + j] = post ? h : srow[j - sl.c0];  // post-norm: the state is h
    st_act(hr, d, j, h, split);
  }
}

// ----------------------------------------------------------------------------- host launchers

template <typename T>
void launch_build_input(int R, int d, int V, float eps, const int* tok, const float* hid_base,
                        const int* hid_row, const void* E, const void* g_emb, const void* g_hid,
                        void* x, bool split, int* flags, cudaStream_t st) {
  if (R <= 0) return;
  if (R < kRowClusterMaxRows)
    launch_pdl_cluster(build_input_kernel<T, kRowCluster>, dim3(R * kRowCluster), dim3(kRowThreads), 0, st,
                       kRowCluster, R, d, V, eps, tok, hid_base, hid_row, (const T*)E, (const T*)g_emb,
                       (const T*)g_hid, (T*)x, split, flags);
  else
    launch_pdl(build_input_kernel<T, 1>, dim3(R), dim3(kRowThreadsWide), 0, st, R, d, V, eps, tok, hid_base,
               hid_row, (const T*)E, (const T*)g_emb, (const T*)g_hid, (T*)x, split, flags);
}

void launch_reduce_parts(int R, int N, int S, const float* part, float* out, cudaStream_t st) {
  size_t n = (size_t)R * N;
  if (!n) return;
  int blocks = (int)((n + 255) / 256);
  if (blocks > 148 * 8) blocks = 148 * 8;
  launch_pdl(reduce_parts_kernel, dim3(blocks), dim3(256), 0, st, R, N, S, part, out);
}

template <typename T>
void launch_reduce_norm(int R, int N, int S, float eps, const float* part, const void* g_fc,
                        float* out, cudaStream_t st) {
  if (R <= 0) return;
  if (R < kRowClusterMaxRows)
    launch_pdl_cluster(reduce_norm_kernel<T, kRowCluster>, dim3(R * kRowCluster), dim3(kRowThreads), 0, st,
                       kRowCluster, R, N, S, eps, part, (const T*)g_fc, out);
  else
    launch_pdl(reduce_norm_kernel<T, 1>, dim3(R), dim3(kRowThreadsWide), 0, st, R, N, S, eps, part,
               (const T*)g_fc, out);
}

template <typename T>
void launch_qkv_epilogue(const QkvEpi& p, cudaStream_t st) {
  if (p.R <= 0) return;
  int nh = (p.has_q ? p.Hq : 0) + 2 * p.Hkv;
  int pairs = nh * p.dh / 2;
  dim3 grid((pairs + 255) / 256, p.R);
  launch_pdl(qkv_epilogue_kernel<T>, dim3(grid), dim3(256), 0, st, p);
}

template <typename T>
void launch_o_epilogue(int R, int d, int S, float eps, const float* part, const float* hid_base,
                       const int* hid_row, const void* g_post, float* r_out, void* z_out,
                       bool split, bool post, cudaStream_t st) {
  if (R <= 0) return;
  if (R < kRowClusterMaxRows)
    launch_pdl_cluster(o_epilogue_kernel<T, kRowCluster>, dim3(R * kRowCluster), dim3(kRowThreads), 0, st,
                       kRowCluster, R, d, S, eps, part, hid_base, hid_row, (const T*)g_post, r_out,
                       (T*)z_out, split, post);
  else
    launch_pdl(o_epilogue_kernel<T, 1>, dim3(R), dim3(kRowThreadsWide), 0, st, R, d, S, eps, part, hid_base,
               hid_row, (const T*)g_post, r_out, (T*)z_out, split, post);
}

template <typename T>
void launch_swiglu(int R, int F, int S, const float* part, void* a, bool split, cudaStream_t st) {
  size_t n = (size_t)R * F;
  if (!n) return;
  int blocks = (int)((n + 255) / 256);
  if (blocks > 148 * 16) blocks = 148 * 16;
  launch_pdl(swiglu_kernel<T>, dim3(blocks), dim3(256), 0, st, R, F, S, part, (T*)a, split);
}

template <typename T>
void launch_down_epilogue(int R, int d, int S, float eps, const float* part, const float* r_in,
                          const void* g_final, const int* s_dst, float* s_base, const int* h_dst,
                          void* h_base, bool split, bool post, cudaStream_t st) {
  if (R <= 0) return;
  if (R < kRowClusterMaxRows) {
    const size_t slice = (size_t)((d + kRowCluster - 1) / kRowCluster) * sizeof(float);
    launch_pdl_cluster(down_epilogue_kernel<T, kRowCluster>, dim3(R * kRowCluster), dim3(kRowThreads), slice,
                       st, kRowCluster, R, d, S, eps, part, r_in, (const T*)g_final, s_dst, s_base, h_dst,
                       (T*)h_base, split, post);
  } else {
    launch_pdl(down_epilogue_kernel<T, 1>, dim3(R), dim3(kRowThreadsWide), d * sizeof(float), st, R, d, S,
               eps, part, r_in, (const T*)g_final, s_dst, s_base, h_dst, (T*)h_base, split, post);
  }
}

#define E3_INST(T)                                                                                   \
  template void launch_build_input<T>(int, int, int, float, const int*, const float*, const int*,   \
                                      const void*, const void*, const void*, void*, bool, int*,     \
                                      cudaStream_t);                                                 \
  template void launch_qkv_epilogue<T>(const QkvEpi&, cudaStream_t);                                 \
  template void launch_reduce_norm<T>(int, int, int, float, const float*, const void*, float*,     \
                                      cudaStream_t);                                                 \
  template void launch_o_epilogue<T>(int, int, int, float, const float*, const float*, const int*,  \
                                     const void*, float*, void*, bool, bool, cudaStream_t);          \
  template void launch_swiglu<T>(int, int, int, const float*, void*, bool, cudaStream_t);            \
  template void launch_down_epilogue<T>(int, int, int, float, const float*, const float*,           \
                                        const void*, const int*, float*, const int*, void*, bool,   \
                                        bool, cudaStream_t);
E3_INST(float)
E3_INST(bf16)
#undef E3_INST

}  // namespace e3
