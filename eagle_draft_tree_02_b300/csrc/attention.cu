// Tree attention of the draft decoder (split-KV, shared-memory staged).
//
// A tree node attends to every prefix row of its request and to its own
// ancestors-or-self among the tree nodes — the tree mask ("EAGLE-3 精读" §2
// Training-Time Test: the draft sees its own path, never a sibling's; §5: the
// rollout nodes cannot see what is not on their path).  Query head h reads KV
// head h / (Hq / Hkv) (grouped-query attention).
//
// Work split: one block per (request, KV head, group of <= 32 query heads,
// key split).  Key splits 0..n_prefix_splits-1 cover the prefix in ranges of
// keys_per_split rows; the remaining splits cover the tree slots, where each
// query keeps only the slots whose bit is set in its row of the mask.  Each
// block streams 64-key chunks of K and V through shared memory (converted to
// fp32 once), keeps an online softmax per query and writes an unnormalised
// partial (o, max, sum).  A second kernel merges the splits.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace e3 {

namespace {
constexpr int QG = 32;   // query heads per block
constexpr int KC = 64;   // keys per chunk
constexpr int NT = 256;  // threads
}

int attention_qgroups(int rows_per_req, int Hq, int Hkv) {
  int per = rows_per_req * (Hq / Hkv);
  return (per + QG - 1) / QG;
}

template <typename T>
__device__ __forceinline__ const T* kv_row_ptr(const AttnArgs& a, const void* cache, int b, int pos,
                                               int kvh) {
  size_t row;
  if (a.page_table) {
    int pg = a.page_table[(size_t)b * a.max_pages + pos / a.page_size];
    if (pg < 0 || pg >= a.n_pages) return nullptr;
    row = (size_t)pg * a.page_size + pos % a.page_size;
  } else {
    row = (size_t)b * a.max_prefix + pos;
  }
  return (const T*)cache + (row * a.Hkv + kvh) * a.dh;
}

template <typename T>
__global__ void __launch_bounds__(NT) tree_attention_kernel(AttnArgs a) {
  extern __shared__ float sm[];
  const int dh = a.dh;
  const int G = a.Hq / a.Hkv;
  float* Qs = sm;                       // [QG][dh+1]
  float* Ks = Qs + QG * (dh + 1);       // [KC][dh+1]
  float* Vs = Ks + KC * (dh + 1);       // [KC][dh]
  float* Ps = Vs + KC * dh;             // [QG][KC]
  float* Ms = Ps + QG * KC;             // [QG] running max
  float* Ls = Ms + QG;                  // [QG] running sum
  float* As = Ls + QG;                  // [QG] rescale factor of this chunk

  const int b = blockIdx.x / a.Hkv, kvh = blockIdx.x % a.Hkv;
  const int qg = blockIdx.y, split = blockIdx.z;
  const int nq_req = a.rows_per_req * G;
  const int q0 = qg * QG;
  const int nq = min(QG, nq_req - q0);
  const int tid = threadIdx.x;
  const int R = a.B * a.rows_per_req;
  const int n_splits = a.n_prefix_splits + a.n_tree_splits;
  const float scale = rsqrtf((float)dh);

  // queries: local index qi -> (row, head)
  for (int i = tid; i < QG * dh; i += NT) {
    int qi = i / dh, dd = i % dh;
    float v = 0.f;
    if (qi < nq) {
      int ql = q0 + qi;
      int row = b * a.rows_per_req + ql / G;
      int head = kvh * G + ql % G;
      v = a.q[(size_t)a.q_row[row] * a.Hq * dh + (size_t)head * dh + dd] * scale;
    }
    Qs[qi * (dh + 1) + dd] = v;
  }
  if (tid < QG) {
    Ms[tid] = -INFINITY;
    Ls[tid] = 0.f;
  }

  int key_lo, key_hi;
  bool tree = split >= a.n_prefix_splits;
  if (!tree) {
    int np = a.n_prefix[b];
    int cap = a.page_table ? a.max_pages * a.page_size : a.max_prefix;
    if (np > cap || np < 0) {
      if (tid == 0 && split == 0 && kvh == 0 && qg == 0) raise_flag(a.flags, FLAG_POS_RANGE);
      np = np < 0 ? 0 : cap;
    }
    key_lo = split * a.keys_per_split;
    key_hi = min(np, key_lo + a.keys_per_split);
  } else {
    key_lo = (split - a.n_prefix_splits) * KC;
    key_hi = min(a.tree_slots, key_lo + KC);
  }

  const int qi_s = tid >> 3, kk_s = tid & 7;  // score phase: query, key lane
  const int dper = dh / 8;                     // PV phase: outputs per thread
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;

  for (int c0 = key_lo; c0 < key_hi; c0 += KC) {
    int nk = min(KC, key_hi - c0);
    __syncthreads();
    // stage K and V of this chunk
    for (int i = tid; i < KC * dh; i += NT) {
      int kk = i / dh, dd = i % dh;
      float kv = 0.f, vv = 0.f;
      if (kk < nk) {
        if (!tree) {
          const T* kp = kv_row_ptr<T>(a, a.cache_k, b, c0 + kk, kvh);
          const T* vp = kv_row_ptr<T>(a, a.cache_v, b, c0 + kk, kvh);
          if (kp && vp) {
            kv = ldf(kp + dd);
            vv = ldf(vp + dd);
          } else if (dd == 0) {
            raise_flag(a.flags, FLAG_PAGE_RANGE);
          }
        } else {  // tree scratch is fp32
          size_t off = (((size_t)b * a.tree_slots + c0 + kk) * a.Hkv + kvh) * dh;
          kv = ((const float*)a.tree_k)[off + dd];
          vv = ((const float*)a.tree_v)[off + dd];
        }
      }
      Ks[kk * (dh + 1) + dd] = kv;
      Vs[kk * dh + dd] = vv;
    }
    __syncthreads();
    // scores: thread -> (query qi_s, keys kk_s + 8 m)
    float s[8];
    float mx = -INFINITY;
    int ql = q0 + qi_s;
    int row = b * a.rows_per_req + ql / G;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      int kk = kk_s + 8 * m;
      float v = -INFINITY;
      bool ok = kk < nk && qi_s < nq;
      if (ok && tree) {
        int slot = c0 + kk;
        ok = (a.mask[(size_t)row * a.mask_words + (slot >> 5)] >> (slot & 31)) & 1u;
      }
      if (ok) {
        float acc_s = 0.f;
        const float* qp = Qs + qi_s * (dh + 1);
        const float* kp = Ks + kk * (dh + 1);
        for (int dd = 0; dd < dh; ++dd) acc_s = fmaf(qp[dd], kp[dd], acc_s);
        v = acc_s;
      }
      s[m] = v;
      mx = fmaxf(mx, v);
    }
    // row max over the 8 lanes that share a query
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    float m_old = Ms[qi_s];
    float m_new = fmaxf(m_old, mx);
    float psum = 0.f;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      float p = (m_new == -INFINITY) ? 0.f : expf(s[m] - m_new);
      Ps[qi_s * KC + kk_s + 8 * m] = p;
      psum += p;
    }
    psum += __shfl_xor_sync(0xffffffffu, psum, 1);
    psum += __shfl_xor_sync(0xffffffffu, psum, 2);
    psum += __shfl_xor_sync(0xffffffffu, psum, 4);
    __syncthreads();  // everyone has read Ms before it changes
    if (kk_s == 0) {
      float alpha = (m_old == -INFINITY) ? 0.f : expf(m_old - m_new);
      As[qi_s] = alpha;
      Ls[qi_s] = Ls[qi_s] * alpha + psum;
      Ms[qi_s] = m_new;
    }
    __syncthreads();
    // o = o * alpha + P V ; thread -> (query qi_s, dims kk_s + 8 i)
    float alpha = As[qi_s];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] *= alpha;
    for (int kk = 0; kk < nk; ++kk) {
      float p = Ps[qi_s * KC + kk];
      const float* vp = Vs + kk * dh + kk_s;
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (i < dper) acc[i] = fmaf(p, vp[8 * i], acc[i]);
    }
  }
  __syncthreads();
  if (qi_s < nq) {
    int ql = q0 + qi_s;
    int row = b * a.rows_per_req + ql / G;
    int head = kvh * G + ql % G;
    size_t base = ((size_t)split * R + row) * a.Hq + head;
    float* op = a.o_part + base * dh;
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if (i < dper) op[kk_s + 8 * i] = acc[i];
    if (kk_s == 0) {
      a.ml_part[base * 2] = Ms[qi_s];
      a.ml_part[base * 2 + 1] = Ls[qi_s];
    }
  }
  (void)n_splits;
}

// merge the key splits of one (row, head): o = sum_s o_s e^{m_s - m} / sum_s l_s e^{m_s - m}
template <typename T>
__global__ void attention_combine_kernel(AttnArgs a) {
  int row = blockIdx.x, head = blockIdx.y;
  int R = a.B * a.rows_per_req;
  int n_splits = a.n_prefix_splits + a.n_tree_splits;
  float m = -INFINITY;
  for (int s = 0; s < n_splits; ++s)
    m = fmaxf(m, a.ml_part[(((size_t)s * R + row) * a.Hq + head) * 2]);
  float l = 0.f;
  for (int s = 0; s < n_splits; ++s) {
    const float* ml = a.ml_part + (((size_t)s * R + row) * a.Hq + head) * 2;
    if (ml[0] != -INFINITY) l += ml[1] * expf(ml[0] - m);
  }
  float inv = l > 0.f ? 1.f / l : 0.f;
  for (int dd = threadIdx.x; dd < a.dh; dd += blockDim.x) {
    float o = 0.f;
    for (int s = 0; s < n_splits; ++s) {
      size_t base = ((size_t)s * R + row) * a.Hq + head;
      float ms = a.ml_part[base * 2];
      if (ms != -INFINITY) o += a.o_part[base * a.dh + dd] * expf(ms - m);
    }
    st_act((T*)a.out + act_row(row, a.Hq * a.dh, a.split), a.Hq * a.dh, head * a.dh + dd, o * inv,
           a.split);
  }
}

template <typename T>
void launch_tree_attention(const AttnArgs& a, cudaStream_t st) {
  int R = a.B * a.rows_per_req;
  if (R <= 0) return;
  int n_splits = a.n_prefix_splits + a.n_tree_splits;
  size_t smem = (size_t)(QG * (a.dh + 1) + KC * (a.dh + 1) + KC * a.dh + QG * KC + 3 * QG) *
                sizeof(float);
  static bool attr_set[2] = {false, false};
  int ti = sizeof(T) == 4 ? 0 : 1;
  if (!attr_set[ti]) {
    cudaFuncSetAttribute(tree_attention_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         160 * 1024);
    attr_set[ti] = true;
  }
  dim3 grid(a.B * a.Hkv, attention_qgroups(a.rows_per_req, a.Hq, a.Hkv), n_splits);
  tree_attention_kernel<T><<<grid, NT, smem, st>>>(a);
  dim3 g2(R, a.Hq);
  attention_combine_kernel<T><<<g2, a.dh, 0, st>>>(a);
}

template void launch_tree_attention<float>(const AttnArgs&, cudaStream_t);
template void launch_tree_attention<bf16>(const AttnArgs&, cudaStream_t);

}  // namespace e3
