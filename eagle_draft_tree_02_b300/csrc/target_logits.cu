// Verification of a kept tree against target logits that the caller supplies
// ("EAGLE-3 精读" §5 正确性、复现与风险: strict verification against the
// target's own distribution -- greedy keeps the target's greedy sequence,
// sampling keeps its distribution with the residual correction).
//
// A real target model scores every tree node in one forward pass and hands
// over its logits [B, M+1, V] (row u of request b: the distribution of the
// token after the root-to-u path).  Three kernels turn those rows into the
// acceptance walk's inputs and share the walk with eagle3_verify:
//   plan_children_kernel  the children of every node from the tree's parents;
//   logits_scan_kernel    per (row, vocabulary chunk): argmax of z, the
//                         online (max, sum exp) of z/T and, when sampling, the
//                         Gumbel-argmax of z/T over the node's non-children;
//                         the chunk holding a child token stores its logit;
//   verify_merge_kernel   (lmhead.cu) folds the chunk partials per row.
// The logits stream from HBM once, 16 bytes per load, with an evict-first
// hint; the Gumbel noise takes one Philox block per four tokens, the same
// counter layout as the fused verify head, so both paths draw identical
// numbers for identical logits.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "philox.cuh"

namespace e3 {
namespace {

constexpr int kScanThreads = 256;
constexpr int kBitmapWords = 64;  // 2048-bit filter of a row's child tokens

// children of each node, ascending tree index (the canonical order the walk
// tests them in); padding slots (token < 0) are nobody's children
__global__ void plan_children_kernel(LogitsVerifyArgs a) {
  pdl_begin();
  const int b = blockIdx.x;
  const int* tok = a.t_tok + (size_t)b * a.M1;
  const int* par = a.t_parent + (size_t)b * a.M1;
  for (int u = threadIdx.x; u < a.M1; u += blockDim.x) {
    const size_t r = (size_t)b * a.M1 + u;
    int cnt = 0;
    const bool real = u == 0 || tok[u] >= 0;
    if (real) {
      if (tok[u] >= a.V || (u == 0 && tok[u] < 0)) raise_flag(a.flags, FLAG_TOKEN_RANGE);
      const int pu = par[u];
      if ((u == 0 && pu != -1) || (u > 0 && (pu < 0 || pu >= a.M1 || pu == u)))
        raise_flag(a.flags, FLAG_TREE_NOT_CLOSED);
      for (int c = 0; c < a.M1; ++c) {
        if (c == u || tok[c] < 0 || par[c] != u) continue;
        if (cnt < a.kmax) {
          a.child_node[r * a.kmax + cnt] = c;
          a.child_tok[r * a.kmax + cnt] = tok[c];
          ++cnt;
        } else {
          raise_flag(a.flags, FLAG_ROWS_RANGE);  // more children than the walk can hold
        }
      }
    }
    for (int i = cnt; i < a.kmax; ++i) {
      a.child_node[r * a.kmax + i] = -1;
      a.child_tok[r * a.kmax + i] = -1;
    }
    a.n_child[r] = cnt;
  }
}

struct ScanState {
  float zb, m, s, gb;
  int zi, gi;
};

__device__ __forceinline__ void scan_token(ScanState& st, int x, float z, float inv_t, bool sampling,
                                           float g, bool child) {
  if (better(z, x, st.zb, st.zi)) {
    st.zb = z;
    st.zi = x;
  }
  const float t = z * inv_t;
  if (t > st.m) {
    st.s = st.s * expf(st.m - t) + 1.f;  // exp(-inf) = 0 covers the empty state
    st.m = t;
  } else {
    st.s += expf(t - st.m);
  }
  if (sampling && !child) {
    const float gs = t + g;
    if (better(gs, x, st.gb, st.gi)) {
      st.gb = gs;
      st.gi = x;
    }
  }
}

__device__ __forceinline__ void lse_fold2(float& m, float& s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m2 > m) {
    s = s * expf(m - m2) + s2;
    m = m2;
  } else {
    s += s2 * expf(m2 - m);
  }
}

template <int VW>
__device__ __forceinline__ void load_vec(const void* row, size_t x, float (&z)[VW]);
template <>
__device__ __forceinline__ void load_vec<4>(const void* row, size_t x, float (&z)[4]) {
  const float4 v = __ldcs(reinterpret_cast<const float4*>(static_cast<const float*>(row) + x));
  z[0] = v.x;
  z[1] = v.y;
  z[2] = v.z;
  z[3] = v.w;
}
template <>
__device__ __forceinline__ void load_vec<8>(const void* row, size_t x, float (&z)[8]) {
  const uint4 v = __ldcs(reinterpret_cast<const uint4*>(static_cast<const bf16*>(row) + x));
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    z[2 * i] = __uint_as_float(w[i] << 16);
    z[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

template <typename T>
__device__ __forceinline__ float load_one(const void* row, size_t x) {
  return ldf<T>(static_cast<const T*>(row) + x);
}

template <typename T>
__global__ void __launch_bounds__(kScanThreads) logits_scan_kernel(LogitsVerifyArgs a) {
  pdl_begin();
  constexpr int VW = 16 / (int)sizeof(T);  // tokens per 16-byte load
  __shared__ int s_ctok[16];
  __shared__ uint32_t s_bits[kBitmapWords];
  __shared__ float sh[4][kScanThreads / 32];
  __shared__ int shi[2][kScanThreads / 32];
  const int r = blockIdx.y, chunk = blockIdx.x, tid = threadIdx.x;
  const int b = r / a.M1, u = r - b * a.M1;
  float* out = a.part + ((size_t)chunk * a.R + r) * 6;
  if (u > 0 && a.t_tok[r] < 0) {  // padding slot: never visited by the walk
    if (tid == 0) {
      out[0] = -INFINITY;
      out[1] = __int_as_float(0x7fffffff);
      out[2] = -INFINITY;
      out[3] = 0.f;
      out[4] = -INFINITY;
      out[5] = __int_as_float(0x7fffffff);
    }
    return;
  }
  const int nc = a.n_child[r];
  if (tid < kBitmapWords) s_bits[tid] = 0u;
  __syncthreads();
  if (tid < nc) {
    const int ct = a.child_tok[(size_t)r * a.kmax + tid];
    s_ctok[tid] = ct;
    if (ct >= 0) atomicOr(&s_bits[(ct >> 5) & (kBitmapWords - 1)], 1u << (ct & 31));
  }
  __syncthreads();
  const void* row = static_cast<const char*>(a.logits) + (size_t)r * a.ld * sizeof(T);
  // the child logits, once per row (the walk's acceptance tests read them)
  if (chunk == 0 && tid < nc) {
    const int ct = s_ctok[tid];
    a.child_z[(size_t)r * a.kmax + tid] = (ct >= 0 && ct < a.V) ? load_one<T>(row, ct) : -INFINITY;
  }
  const bool sampling = a.sampling != 0;
  const unsigned long long rid = a.round_ptr ? *a.round_ptr : a.round_id;
  auto is_child = [&](int x) {
    if (!((s_bits[(x >> 5) & (kBitmapWords - 1)] >> (x & 31)) & 1u)) return false;
    for (int i = 0; i < nc; ++i)
      if (s_ctok[i] == x) return true;
    return false;
  };
  ScanState st{-INFINITY, -INFINITY, 0.f, -INFINITY, 0x7fffffff, 0x7fffffff};
  const int x0 = chunk * a.chunk;
  const int x1 = min(a.V, x0 + a.chunk);
  const int nv = x1 > x0 ? (x1 - x0) / VW : 0;
  for (int v = tid; v < nv; v += kScanThreads) {
    const int x = x0 + v * VW;
    float z[VW];
    load_vec<VW>(row, (size_t)x, z);
    uint64_t w[VW];
    if (sampling) {
#pragma unroll
      for (int h = 0; h < VW / 4; ++h) {
        uint64_t wb[4];
        gumbel_block(a.seed, rid, b, u, (uint64_t)((x >> 2) + h), wb);
#pragma unroll
        for (int j = 0; j < 4; ++j) w[4 * h + j] = wb[j];
      }
    }
#pragma unroll
    for (int j = 0; j < VW; ++j) {
      const float g = sampling ? gumbel_from_word(w[j]) : 0.f;
      scan_token(st, x + j, z[j], a.inv_t, sampling, g, sampling && is_child(x + j));
    }
  }
  for (int x = x0 + nv * VW + tid; x < x1; x += kScanThreads) {  // ragged end of the vocabulary
    const float z = load_one<T>(row, (size_t)x);
    const float g = sampling ? verify_gumbel(a.seed, rid, b, u, x) : 0.f;
    scan_token(st, x, z, a.inv_t, sampling, g, sampling && is_child(x));
  }
  // block reduction: argmax, (max, sum exp), Gumbel-argmax
  warp_best(st.zb, st.zi);
  warp_best(st.gb, st.gi);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, st.m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, st.s, o);
    lse_fold2(st.m, st.s, m2, s2);
  }
  const int lane = tid & 31, wid = tid >> 5;
  if (lane == 0) {
    sh[0][wid] = st.zb;
    sh[1][wid] = st.m;
    sh[2][wid] = st.s;
    sh[3][wid] = st.gb;
    shi[0][wid] = st.zi;
    shi[1][wid] = st.gi;
  }
  __syncthreads();
  if (wid == 0) {
    constexpr int NW = kScanThreads / 32;
    float zb = lane < NW ? sh[0][lane] : -INFINITY, m = lane < NW ? sh[1][lane] : -INFINITY;
    float s = lane < NW ? sh[2][lane] : 0.f, gb = lane < NW ? sh[3][lane] : -INFINITY;
    int zi = lane < NW ? shi[0][lane] : 0x7fffffff, gi = lane < NW ? shi[1][lane] : 0x7fffffff;
    warp_best(zb, zi);
    warp_best(gb, gi);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
      lse_fold2(m, s, m2, s2);
    }
    if (lane == 0) {
      out[0] = zb;
      out[1] = __int_as_float(zi);
      out[2] = m;
      out[3] = s;
      out[4] = gb;
      out[5] = __int_as_float(gi);
    }
  }
}

}  // namespace

int logits_verify_chunks(int R, int V, int max_parts) {
  // about eight blocks per SM in all, chunks of at least 2048 tokens
  int n = (8 * 148 + R - 1) / R;
  n = min(n, (V + 2047) / 2048);
  n = max(1, min(n, max_parts));
  return n;
}

void launch_logits_verify(LogitsVerifyArgs a, bool bf, cudaStream_t st) {
  if (a.R <= 0) return;
  launch_pdl(plan_children_kernel, dim3(a.B), dim3(128), 0, st, a);
  // chunk starts on a multiple of 8 tokens keep every 16-byte load aligned
  a.chunk = ((a.V + a.n_chunks - 1) / a.n_chunks + 7) / 8 * 8;
  dim3 grid(a.n_chunks, a.R);
  if (bf)
    launch_pdl(logits_scan_kernel<bf16>, grid, dim3(kScanThreads), 0, st, a);
  else
    launch_pdl(logits_scan_kernel<float>, grid, dim3(kScanThreads), 0, st, a);
}

}  // namespace e3
