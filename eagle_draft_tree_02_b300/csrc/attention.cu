// Tree attention of the draft decoder (split-KV, shared-memory staged).
//
// A tree node attends to every prefix row of its request and to its own
// ancestors-or-self among the tree nodes — the tree mask ("EAGLE-3 精读" §2
// Training-Time Test: the draft sees its own path, never a sibling's; §5: the
// rollout nodes cannot see what is not on their path).  Query head h reads KV
// head h / (Hq / Hkv) (grouped-query attention).
//
// Work split: key splits 0..n_prefix_splits-1 cover the prefix in ranges of
// keys_per_split rows; the remaining splits cover the tree slots, where each
// query keeps only the slots whose bit is set in its row of the mask.  Every
// split block keeps an online softmax per query and writes an unnormalised
// partial (o, max, sum); a second kernel merges the splits.
//
// bf16 cache, prefix splits: one block of 4 warps per (request, KV head, group
// of <= 64 queries, split); 64-key chunks of K and V stream through a 3-stage
// ring in shared memory as tensor-map boxes (64 dims x 1 KV head x 64 tokens,
// or a page's share of them; 128-byte swizzle), a few per chunk from lanes of
// warp 0, completing on the stage's mbarrier.  (One 256-byte bulk copy per
// row and thread, 128 per chunk, held the batch-64 paged pass to 2.2 TB/s:
// the copies, not the bytes, set the pace.)  The 16 queries of a warp take Q K^T
// and P V on the tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate).
// Q and P enter as hi + lo bf16 pairs (two MMAs each), so the products keep
// about 16 significant bits, and K, V are the cache's exact values.  (With P
// as one bf16, the 70B-shaped tree's log q error grew from 2e-4 to 1e-3 at no
// measurable gain in time.  With fp16 operands -- K and V converted exactly
// after each chunk lands, Q and P one fp16 each, one MMA per product -- the
// 8B-shaped launch fell from 19 to 15 us, but the 70B-shaped log q error grew
// from 2.5e-4 to 8.5e-3; splitting Q as fp16 hi + lo brought the error back and
// the time with it, and the conversion pass slowed the paged batch of chains.)
// A tree split stages its 64 fp32 slots as bf16
// (hi, lo) pairs and adds the lo products (three MMAs per fragment), with the
// ancestor mask applied per query row.  The fp32 cache uses the CUDA-core kernel: 32
// queries per block, K and V staged as fp32.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace e3 {

namespace {
constexpr int QG = 32;   // query heads per block (CUDA-core kernel)
constexpr int QGM = 64;  // queries per block (queries-as-M kernel: 4 warps x 16)
constexpr int QKT = 16;  // at most this many queries per KV head: the keys-as-M kernel
constexpr int QTC = 128; // more than this many: the tcgen05 kernel, 128 queries per block
constexpr int KC = 64;   // keys per chunk
constexpr int KST = 3;   // prefix stages in flight (tensor-core kernel)
constexpr int NT = 256;  // threads (CUDA-core kernel)
}

bool attention_uses_tc(int rows_per_req, int Hq, int Hkv) { return rows_per_req * (Hq / Hkv) > QTC; }

int attention_qgroups(int rows_per_req, int Hq, int Hkv, bool mma) {
  int per = rows_per_req * (Hq / Hkv);
  if (mma && per <= QKT) return 1;
  const int q = !mma ? QG : per <= QTC ? QGM : QTC;
  return (per + q - 1) / q;
}

// The tensor-core kernel loads whole boxes of at least 8 tokens, so a paged
// cache needs pages of a multiple of 8 tokens; other page sizes (and fp32)
// take the CUDA-core kernel.
bool attention_uses_mma(int elem_bytes, int dh, int page_size) {
  return elem_bytes == 2 && (dh == 64 || dh == 128) && page_size >= 0 && page_size % 8 == 0;
}

int attention_box_rows(int page_size) {
  if (page_size <= 0) return KC;
  int a = KC, b = page_size;
  while (b) {
    const int t = a % b;
    a = b;
    b = t;
  }
  return a;
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
__global__ void __launch_bounds__(NT) tree_attention_kernel(AttnArgs a, int z_off) {
  pdl_begin();
  if (a.skip && *a.skip == 0) return;
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
  const int qg = blockIdx.y, split = blockIdx.z + z_off;
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


// ----------------------------------------------------------------------------- tensor-core prefix splits
namespace {
__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                              uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// Transpose of an 8 x 8 matrix of 16-bit pairs held one pair per lane in the
// fragment layout (row lane / 4, columns 2 (lane % 4) and + 1).
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
// One box of a three-dimensional tensor map global -> shared, completing on an mbarrier.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x,
                                            int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void att_mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void att_arrive_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
// Bounded wait for the phase with the given parity: false (and the timeout
// flag) after about two seconds.
__device__ __forceinline__ bool att_wait(uint32_t bar, uint32_t parity, int* flags) {
  const long long t0 = clock64();
  for (uint32_t it = 0;; ++it) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
    if ((it & 63) == 63 && clock64() - t0 > 4000000000LL) {
      raise_flag(flags, FLAG_TIMEOUT);
      return false;
    }
  }
}
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint32_t bf2_bits(__nv_bfloat162 v) {
  return *reinterpret_cast<uint32_t*>(&v);
}
// (x0, x1) -> hi = bf16 pair, lo = bf16 pair of the rounding remainders
__device__ __forceinline__ void split_pair(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  hi = bf2_bits(h);
  lo = bf2_bits(__floats2bfloat162_rn(x0 - hf.x, x1 - hf.y));
}

// ---- tcgen05 pieces of the wide-group kernel (one CTA issues, TMEM holds S and O)
__device__ __forceinline__ void utc_alloc(uint32_t slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void utc_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void utc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void utc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void utc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void utc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// generic-proxy writes to shared memory, made visible to the tensor core's reads
__device__ __forceinline__ void async_proxy_fence() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// 32 consecutive TMEM columns of this thread's lane (load, and its wait)
__device__ __forceinline__ void utc_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void utc_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}
// Shared-memory operand descriptor, 128-byte swizzle, 8-row groups 1024 bytes
// apart.  K-major: rows of 64 K-elements (128 B).  MN-major: rows of 64
// MN-elements, one row per K index; with N = 64 per MMA the operand is one
// swizzle atom wide, so the leading offset (between atoms along MN) is unused.
__device__ __forceinline__ uint64_t att_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);  // start address
  d |= (uint64_t)1 << 16;                    // leading byte offset (unused here)
  d |= (uint64_t)(1024 >> 4) << 32;          // stride byte offset: next 8-row group
  d |= (uint64_t)1 << 46;                    // descriptor version
  d |= (uint64_t)2 << 61;                    // 128-byte swizzle
  return d;
}
// MN-major operand one swizzle atom wide (64 elements along MN): both offset
// fields carry the 8-row group stride, so the descriptor holds whichever of
// the two the hardware takes as the stride along K.
__device__ __forceinline__ uint64_t att_desc_mn(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)(1024 >> 4) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// Instruction descriptor of kind::f16: bf16 A and B, fp32 accumulator, M = 128;
// b_mn: B is MN-major.
__host__ __device__ constexpr uint32_t att_idesc(int n, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn ? (1u << 16) : 0u) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(128 >> 4) << 24);
}
// bounded mbarrier wait of the wide-group kernel: false (flag raised) after ~2 s
__device__ __forceinline__ bool att_wait_abort(uint32_t bar, uint32_t parity, int* flags,
                                               volatile int* abort_f) {
  const long long t0 = clock64();
  for (uint32_t it = 0;; ++it) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
    if ((it & 63) == 63) {
      if (*abort_f) return false;
      if (clock64() - t0 > 4000000000LL) {
        *abort_f = 1;
        raise_flag(flags, FLAG_TIMEOUT);
        return false;
      }
    }
  }
}

// The key range of split blockIdx.z: prefix splits take keys
// [split * keys_per_split, +keys_per_split) of the cache, tree splits 64 tree
// slots each.
struct SplitKeys {
  bool tree;
  int lo, hi, n_chunks;
};
__device__ __forceinline__ SplitKeys split_keys(const AttnArgs& a, int b, int split, bool report) {
  SplitKeys k;
  k.tree = split >= a.n_prefix_splits;
  if (!k.tree) {
    int np = a.n_prefix[b];
    const int cap = a.page_table ? a.max_pages * a.page_size : a.max_prefix;
    if (np > cap || np < 0) {
      if (report) raise_flag(a.flags, FLAG_POS_RANGE);
      np = np < 0 ? 0 : cap;
    }
    k.lo = split * a.keys_per_split;
    k.hi = min(np, k.lo + a.keys_per_split);
  } else {
    k.lo = (split - a.n_prefix_splits) * KC;
    k.hi = min(a.tree_slots, k.lo + KC);
  }
  k.n_chunks = k.hi > k.lo ? (k.tree ? 1 : (k.hi - k.lo + KC - 1) / KC) : 0;
  return k;
}
}  // namespace

// The K/V ring of the tensor-core kernels.  KST stages each hold one 64-key
// chunk: the K halves, then the V halves (NH halves of 128 bytes per row).
// Half h of key row n sits at h * HB + n * 128 and its 16-byte piece j at
// ((j ^ (n & 7)) << 4) within the row -- the tensor map's 128-byte swizzle --
// so fragment loads of 8 consecutive rows touch 8 distinct bank groups.
//
// A chunk arrives as tensor-map boxes of tm_rows tokens x 64 dims of one KV
// head: KC / tm_rows token groups, 2 * NH boxes each (K and V, per half).
// Lane l < n_ops of warp 0 copies box l of every chunk; lane 0 arms the
// stage's mbarrier with the chunk's bytes.  A group past the split's end, or
// on a bad page, is read at token row tm_T, past the tensor, which fills
// zeros.  Each lane fetches its page-table entry one chunk ahead.
template <int DH>
struct KvRing {
  static constexpr int NH = DH / 64;
  static constexpr int HB = KC * 128;
  static constexpr int STB = 2 * NH * HB;
  static constexpr int SMEM = 1024 + KST * STB + 8 * KST;  // with alignment slack

  unsigned char* sb;  // stage 0, 1024-aligned
  uint32_t sb32, bar0;
  int b, kvh, lane, warp;
  SplitKeys k;
  int my_grp, my_box, n_ops, pg_next;

  __device__ __forceinline__ void init(unsigned char* smem, int b_, int kvh_, const SplitKeys& k_) {
    const uint32_t raw = smem_u32(smem);
    sb = smem + (((raw + 1023u) & ~1023u) - raw);
    sb32 = smem_u32(sb);
    bar0 = sb32 + KST * STB;
    b = b_;
    kvh = kvh_;
    k = k_;
    lane = threadIdx.x & 31;
    warp = threadIdx.x >> 5;
    pg_next = 0;
  }
  __device__ __forceinline__ unsigned char* kstage(int st) const { return sb + st * STB; }
  __device__ __forceinline__ uint32_t kstage32(int st) const { return sb32 + st * STB; }
  __device__ __forceinline__ uint32_t vstage32(int st) const { return sb32 + st * STB + NH * HB; }

  __device__ __forceinline__ int page_of(const AttnArgs& a, int ci) const {
    const int pos = k.lo + ci * KC + my_grp * a.tm_rows;
    if (warp != 0 || lane >= n_ops || !a.page_table || ci >= k.n_chunks || pos >= k.hi) return 0;
    return a.page_table[(size_t)b * a.max_pages + pos / a.page_size];
  }
  __device__ __forceinline__ void issue(const AttnArgs& a, int ci, int pg) const {  // warp 0 only
    const int st = ci % KST, pos = k.lo + ci * KC + my_grp * a.tm_rows;
    const uint32_t bar = bar0 + 8u * st;
    if (lane == 0) att_arrive_tx(bar, (uint32_t)STB);  // every box lands in full
    __syncwarp();
    if (lane < n_ops) {
      int row = a.tm_T;
      if (pos < k.hi) {
        if (!a.page_table)
          row = b * a.max_prefix + pos;
        else if (pg >= 0 && pg < a.n_pages)
          row = pg * a.page_size + pos % a.page_size;
        else
          raise_flag(a.flags, FLAG_PAGE_RANGE);
      }
      const int v = my_box / NH, h = my_box % NH;
      tma_load_3d(kstage32(st) + (v * NH + h) * HB + my_grp * a.tm_rows * 128, v ? &a.tm_v : &a.tm_k,
                  bar, h * 64, kvh, row);
    }
  }
  // Barriers, then the first KST - 1 chunks (all threads of the block call it).
  __device__ __forceinline__ void start(const AttnArgs& a) {
    const int per_group = 2 * NH;
    n_ops = (KC / a.tm_rows) * per_group;  // <= 32 for tm_rows >= 8
    my_grp = lane / per_group;
    my_box = lane % per_group;
    if (threadIdx.x == 0) {
      for (int st = 0; st < KST; ++st) att_mbar_init(bar0 + 8u * st, 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (warp != 0) return;
    for (int ci = 0; ci < KST - 1 && ci < k.n_chunks; ++ci) issue(a, ci, page_of(a, ci));
    pg_next = page_of(a, KST - 1);
  }
  // Let the chunks that start() requested land (a block that leaves early).
  __device__ __forceinline__ void drain_start(const AttnArgs& a) const {
    for (int ci = 0; ci < KST - 1 && ci < k.n_chunks; ++ci) att_wait(bar0 + 8u * ci, 0u, a.flags);
  }
  // Refill the stage that chunk ci - 1 used, wait for chunk ci, and give V
  // zero rows past the split's end (stale cache rows there meet P = 0, and 0
  // times a non-finite value would not be 0).  Ends with a block barrier;
  // false, once the copies still in flight have landed, if a copy never did.
  __device__ __forceinline__ bool next(const AttnArgs& a, int ci) {
    const int cn = ci + KST - 1;
    if (warp == 0 && cn < k.n_chunks) {
      issue(a, cn, pg_next);
      pg_next = page_of(a, cn + 1);
    }
    const int st = ci % KST, c0 = k.lo + ci * KC;
    const bool ok = att_wait(bar0 + 8u * st, (uint32_t)(ci / KST) & 1u, a.flags);
    if (ok && c0 + KC > k.hi) {
      unsigned char* vz = kstage(st) + NH * HB;
      for (int i = threadIdx.x; i < (c0 + KC - k.hi) * NH * 8; i += blockDim.x) {
        const int n = k.hi - c0 + i / (NH * 8), h = (i / 8) % NH, piece = i % 8;
        *reinterpret_cast<uint4*>(vz + h * HB + n * 128 + piece * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // for tensor-core reads of V
    }
    if (__syncthreads_and(ok)) return true;
    for (int c = ci + 1; c < k.n_chunks && c < ci + KST; ++c)
      att_wait(bar0 + 8u * (c % KST), (uint32_t)(c / KST) & 1u, a.flags);
    return false;
  }
  // A tree split's 64 fp32 slots as bf16 hi (stage 0) + lo (stage 1), in the
  // ring's row layout; slots past the end are zero rows.
  __device__ __forceinline__ void load_tree(const AttnArgs& a) {
    constexpr int PIECES = DH / 8;
    for (int i = threadIdx.x; i < KC * PIECES; i += blockDim.x) {
      const int kk = i / PIECES, piece = i % PIECES, slot = k.lo + kk;
      float kx[8], vx[8];
      if (slot < k.hi) {
        const size_t off = (((size_t)b * a.tree_slots + slot) * a.Hkv + kvh) * DH + piece * 8;
        const float4* kq = reinterpret_cast<const float4*>((const float*)a.tree_k + off);
        const float4* vq = reinterpret_cast<const float4*>((const float*)a.tree_v + off);
        const float4 k0 = kq[0], k1 = kq[1], v0 = vq[0], v1 = vq[1];
        kx[0] = k0.x; kx[1] = k0.y; kx[2] = k0.z; kx[3] = k0.w;
        kx[4] = k1.x; kx[5] = k1.y; kx[6] = k1.z; kx[7] = k1.w;
        vx[0] = v0.x; vx[1] = v0.y; vx[2] = v0.z; vx[3] = v0.w;
        vx[4] = v1.x; vx[5] = v1.y; vx[6] = v1.z; vx[7] = v1.w;
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) kx[e] = vx[e] = 0.f;
      }
      uint32_t khi[4], klo[4], vhi[4], vlo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        split_pair(kx[2 * e], kx[2 * e + 1], khi[e], klo[e]);
        split_pair(vx[2 * e], vx[2 * e + 1], vhi[e], vlo[e]);
      }
      const int o0 = (piece >> 3) * HB + kk * 128 + (((piece & 7) ^ (kk & 7)) << 4);
      *reinterpret_cast<uint4*>(sb + o0) = make_uint4(khi[0], khi[1], khi[2], khi[3]);
      *reinterpret_cast<uint4*>(sb + STB + o0) = make_uint4(klo[0], klo[1], klo[2], klo[3]);
      *reinterpret_cast<uint4*>(sb + NH * HB + o0) = make_uint4(vhi[0], vhi[1], vhi[2], vhi[3]);
      *reinterpret_cast<uint4*>(sb + STB + NH * HB + o0) = make_uint4(vlo[0], vlo[1], vlo[2], vlo[3]);
    }
  }
};

// Queries as the MMA's M dimension: one warp per 16 queries of a KV head
// (groups of more than 16 queries: the tree frontiers, the verify passes of
// wide trees).  S = Q K^T and O += P V, m16n8k16, Q and P as bf16 hi + lo.
template <int DH>
__global__ void __launch_bounds__(128) prefix_attention_mma_kernel(const __grid_constant__ AttnArgs a) {
  constexpr int NKT = KC / 8;      // key tiles of 8 per chunk
  constexpr int NDT = DH / 8;      // output tiles of 8 dims
  constexpr int NKS = DH / 16;     // k16 steps over dh
  using Ring = KvRing<DH>;
  extern __shared__ __align__(16) unsigned char att_smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int b = blockIdx.x / a.Hkv, kvh = blockIdx.x % a.Hkv, split = blockIdx.z;
  const int G = a.Hq / a.Hkv, nq = a.rows_per_req * G;
  const int R = a.B * a.rows_per_req;
  const int qw = blockIdx.y * QGM + warp * 16;  // first query of this warp
  const SplitKeys sk = split_keys(a, b, split, tid == 0 && split == 0 && kvh == 0 && blockIdx.y == 0);
  Ring ring;
  ring.init(att_smem, b, kvh, sk);
  // When no kernel of this pass writes the prefix cache (every pass after the
  // root's), the first chunks are requested before the wait for the previous
  // kernel, so their latency overlaps its tail; the queries and tree rows follow.
  const bool early = a.prefix_stable && !sk.tree && sk.n_chunks > 0;
  if (early) ring.start(a);
  pdl_begin();
  if (a.skip && *a.skip == 0) {
    if (early) ring.drain_start(a);  // the requested chunks land before the shared memory is released
    return;
  }

  // this thread's two query rows (g and g + 8 of the warp's 16), scaled by 1/sqrt(dh)
  const int qr[2] = {qw + g, qw + g + 8};
  const float* qp[2];
  const uint32_t* mrow_bits[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    qp[h] = nullptr;
    mrow_bits[h] = nullptr;
    if (qr[h] < nq) {
      const int row = b * a.rows_per_req + qr[h] / G, head = kvh * G + qr[h] % G;
      qp[h] = a.q + (size_t)a.q_row[row] * a.Hq * DH + (size_t)head * DH;
      mrow_bits[h] = a.mask + (size_t)row * a.mask_words;
    }
  }
  const float scale = rsqrtf((float)DH);
  uint32_t qh[NKS][4], ql[NKS][4];
#pragma unroll
  for (int ks = 0; ks < NKS; ++ks) {
#pragma unroll
    for (int f = 0; f < 4; ++f) {  // fragment f: row g (+8 if f odd), cols +8 if f >= 2
      const float* p = qp[f & 1];
      const int c = ks * 16 + t4 * 2 + (f >> 1) * 8;
      const float x0 = p ? p[c] * scale : 0.f, x1 = p ? p[c + 1] * scale : 0.f;
      split_pair(x0, x1, qh[ks][f], ql[ks][f]);
    }
  }
  float o[NDT][4];
#pragma unroll
  for (int i = 0; i < NDT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
  const bool active = qw < nq;

  if (sk.tree) {
    if (sk.n_chunks > 0) ring.load_tree(a);
  } else if (!early) {
    ring.start(a);
  }
  for (int ci = 0; ci < sk.n_chunks; ++ci) {
    const int c0 = sk.lo + ci * KC, st = sk.tree ? 0 : ci % KST;
    if (!sk.tree) {
      if (!ring.next(a, ci)) break;
    } else {
      __syncthreads();
    }
    if (active) {
      const unsigned char* kb = ring.kstage(st);  // tree chunk: lo halves one stage on
      const uint32_t vb32 = ring.vstage32(st);
      float s[NKT][4];
#pragma unroll
      for (int nt = 0; nt < NKT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < NKS; ++ks) {
        const int j = (ks & 3) * 2;  // 16-byte piece of dims ks*16 .. +7 within the half
#pragma unroll
        for (int nt = 0; nt < NKT; ++nt) {
          // key row n = nt * 8 + g, so n & 7 = g
          const unsigned char* kr = kb + (ks >> 2) * Ring::HB + (nt * 8 + g) * 128 + t4 * 4;
          const uint32_t b0 = *reinterpret_cast<const uint32_t*>(kr + ((j ^ g) << 4));
          const uint32_t b1 = *reinterpret_cast<const uint32_t*>(kr + (((j + 1) ^ g) << 4));
          mma_16816(s[nt], qh[ks], b0, b1);
          mma_16816(s[nt], ql[ks], b0, b1);
          if (sk.tree) {  // + q hi . k lo
            const uint32_t c0l = *reinterpret_cast<const uint32_t*>(kr + Ring::STB + ((j ^ g) << 4));
            const uint32_t c1l =
                *reinterpret_cast<const uint32_t*>(kr + Ring::STB + (((j + 1) ^ g) << 4));
            mma_16816(s[nt], qh[ks], c0l, c1l);
          }
        }
      }
      // keys past the split's end; in a tree chunk, slots off the query's path
#pragma unroll
      for (int nt = 0; nt < NKT; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = c0 + nt * 8 + t4 * 2 + (e & 1);
          bool ok = key < sk.hi;
          if (ok && sk.tree) {
            const uint32_t* mb = mrow_bits[e >> 1];
            ok = mb && ((mb[key >> 5] >> (key & 31)) & 1u);
          }
          if (!ok) s[nt][e] = -INFINITY;
        }
      }
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nt = 0; nt < NKT; ++nt) {
        mx[0] = fmaxf(mx[0], fmaxf(s[nt][0], s[nt][1]));
        mx[1] = fmaxf(mx[1], fmaxf(s[nt][2], s[nt][3]));
      }
      float alpha[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
        const float mn = fmaxf(mrow[h], mx[h]);
        alpha[h] = (mrow[h] == -INFINITY) ? 0.f : expf(mrow[h] - mn);
        mrow[h] = mn;
      }
      float ps[2] = {0.f, 0.f};
#pragma unroll
      for (int nt = 0; nt < NKT; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float m = mrow[e >> 1];
          const float p = (m == -INFINITY || s[nt][e] == -INFINITY) ? 0.f : expf(s[nt][e] - m);
          s[nt][e] = p;
          ps[e >> 1] += p;
        }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) lrow[h] = lrow[h] * alpha[h] + ps[h];
#pragma unroll
      for (int dt = 0; dt < NDT; ++dt) {
        o[dt][0] *= alpha[0];
        o[dt][1] *= alpha[0];
        o[dt][2] *= alpha[1];
        o[dt][3] *= alpha[1];
      }
      // O += P V over the chunk's keys, 16 at a time
#pragma unroll
      for (int kk = 0; kk < KC / 16; ++kk) {
        uint32_t ph[4], pl[4];
        split_pair(s[2 * kk][0], s[2 * kk][1], ph[0], pl[0]);
        split_pair(s[2 * kk][2], s[2 * kk][3], ph[1], pl[1]);
        split_pair(s[2 * kk + 1][0], s[2 * kk + 1][1], ph[2], pl[2]);
        split_pair(s[2 * kk + 1][2], s[2 * kk + 1][3], ph[3], pl[3]);
        const int mat = lane >> 3, r8 = lane & 7;
        // lane's row of matrix mat: key kk*16 + r8 (+8), dims d2*16 (+8); key & 7 = r8
        const uint32_t vrow = vb32 + (kk * 16 + r8 + (mat & 1) * 8) * 128;
#pragma unroll
        for (int d2 = 0; d2 < DH / 16; ++d2) {
          const uint32_t va = vrow + (d2 >> 2) * Ring::HB + ((((d2 & 3) * 2 + (mat >> 1)) ^ r8) << 4);
          uint32_t v0, v1, v2, v3;
          ldsm_x4_trans(v0, v1, v2, v3, va);
          mma_16816(o[2 * d2], ph, v0, v1);
          mma_16816(o[2 * d2], pl, v0, v1);
          mma_16816(o[2 * d2 + 1], ph, v2, v3);
          mma_16816(o[2 * d2 + 1], pl, v2, v3);
          if (sk.tree) {  // stage 1: the lo halves of the tree chunk's fp32 V
            ldsm_x4_trans(v0, v1, v2, v3, va + Ring::STB);
            mma_16816(o[2 * d2], ph, v0, v1);
            mma_16816(o[2 * d2 + 1], ph, v2, v3);
          }
        }
      }
    }
    __syncthreads();  // this stage is refilled at the next chunk
  }
  // partials: unnormalised o, running max, and the quad's sum of exp
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    lrow[h] += __shfl_xor_sync(0xffffffffu, lrow[h], 1);
    lrow[h] += __shfl_xor_sync(0xffffffffu, lrow[h], 2);
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if (qr[h] >= nq) continue;
    const int row = b * a.rows_per_req + qr[h] / G, head = kvh * G + qr[h] % G;
    const size_t base = ((size_t)split * R + row) * a.Hq + head;
    float* op = a.o_part + base * DH;
#pragma unroll
    for (int dt = 0; dt < NDT; ++dt) {
      op[dt * 8 + t4 * 2] = o[dt][2 * h];
      op[dt * 8 + t4 * 2 + 1] = o[dt][2 * h + 1];
    }
    if (t4 == 0) {
      a.ml_part[base * 2] = mrow[h];
      a.ml_part[base * 2 + 1] = lrow[h];
    }
  }
}

// Keys as the MMA's M dimension, for at most 16 queries per KV head (a batch
// of chains or of small trees): S^T = K Q^T and O^T += V^T P^T, with the
// queries as the 8-wide N dimension (NQT tiles of 8), so no MMA row is spent
// on an absent query.  Each warp takes 16 keys of every chunk and keeps its
// own softmax state per query; the four warps merge at the end.  P^T goes
// from the accumulator layout to the B operand by movmatrix (an in-register
// 8 x 8 transpose).  Q and P enter as bf16 hi + lo, as in the kernel above.
template <int DH, int NQT>
__global__ void __launch_bounds__(128) prefix_attention_kt_kernel(const __grid_constant__ AttnArgs a) {
  constexpr int NKS = DH / 16;  // k16 steps over dh; also the 16-dim tiles of O^T
  using Ring = KvRing<DH>;
  extern __shared__ __align__(16) unsigned char att_smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3, mat = lane >> 3, r8 = lane & 7;
  const int b = blockIdx.x / a.Hkv, kvh = blockIdx.x % a.Hkv, split = blockIdx.z;
  const int G = a.Hq / a.Hkv, nq = min(a.rows_per_req * G, 8 * NQT);
  const int R = a.B * a.rows_per_req;
  const SplitKeys sk = split_keys(a, b, split, tid == 0 && split == 0 && kvh == 0);
  Ring ring;
  ring.init(att_smem, b, kvh, sk);
  const bool early = a.prefix_stable && !sk.tree && sk.n_chunks > 0;  // as in the kernel above
  if (early) ring.start(a);
  pdl_begin();
  if (a.skip && *a.skip == 0) {
    if (early) ring.drain_start(a);
    return;
  }

  // B operand of S^T: query qt*8 + g, dims ks*16 + 2 t4 (+1) and + 8, scaled by 1/sqrt(dh)
  const float scale = rsqrtf((float)DH);
  uint32_t qb[NQT][NKS][2], qbl[NQT][NKS][2];
#pragma unroll
  for (int qt = 0; qt < NQT; ++qt) {
    const int q = qt * 8 + g;
    const float* qp = nullptr;
    if (q < nq) {
      const int row = b * a.rows_per_req + q / G, head = kvh * G + q % G;
      qp = a.q + (size_t)a.q_row[row] * a.Hq * DH + (size_t)head * DH;
    }
#pragma unroll
    for (int ks = 0; ks < NKS; ++ks) {
#pragma unroll
      for (int f = 0; f < 2; ++f) {
        const int c = ks * 16 + t4 * 2 + f * 8;
        const float x0 = qp ? qp[c] * scale : 0.f, x1 = qp ? qp[c + 1] * scale : 0.f;
        split_pair(x0, x1, qb[qt][ks][f], qbl[qt][ks][f]);
      }
    }
  }
  // this thread's accumulator columns: queries qt*8 + 2 t4 + e, and their mask rows
  const uint32_t* mrow_bits[NQT][2];
#pragma unroll
  for (int qt = 0; qt < NQT; ++qt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int q = qt * 8 + t4 * 2 + e;
      mrow_bits[qt][e] = q < nq ? a.mask + (size_t)(b * a.rows_per_req + q / G) * a.mask_words : nullptr;
    }
  float ot[NKS][NQT][4];  // O^T: dims dt*16 + g (+8) x queries qt*8 + 2 t4 (+1)
#pragma unroll
  for (int dt = 0; dt < NKS; ++dt)
#pragma unroll
    for (int qt = 0; qt < NQT; ++qt) ot[dt][qt][0] = ot[dt][qt][1] = ot[dt][qt][2] = ot[dt][qt][3] = 0.f;
  float mq[NQT][2], lq[NQT][2];
#pragma unroll
  for (int qt = 0; qt < NQT; ++qt) mq[qt][0] = mq[qt][1] = -INFINITY, lq[qt][0] = lq[qt][1] = 0.f;

  if (sk.tree) {
    if (sk.n_chunks > 0) ring.load_tree(a);
  } else if (!early) {
    ring.start(a);
  }
  const int kw = warp * 16;  // this warp's 16 keys of each chunk
  for (int ci = 0; ci < sk.n_chunks; ++ci) {
    const int c0 = sk.lo + ci * KC, st = sk.tree ? 0 : ci % KST;
    if (!sk.tree) {
      if (!ring.next(a, ci)) break;
    } else {
      __syncthreads();
    }
    // S^T over keys kw + g (+8): the A operand is a 16 x 16 tile of K, lane l
    // addressing row r8 of matrix mat (keys +8 if mat & 1, dims +8 if mat >> 1);
    // even and odd k steps accumulate apart, to shorten the dependent chains
    float sa[NQT][4], sz[NQT][4];
#pragma unroll
    for (int qt = 0; qt < NQT; ++qt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sa[qt][e] = sz[qt][e] = 0.f;
    const uint32_t krow = ring.kstage32(st) + (kw + r8 + (mat & 1) * 8) * 128;
#pragma unroll
    for (int ks = 0; ks < NKS; ++ks) {
      const uint32_t ka = krow + (ks >> 2) * Ring::HB + ((((ks & 3) * 2 + (mat >> 1)) ^ r8) << 4);
      uint32_t af[4];
      ldsm_x4(af, ka);
#pragma unroll
      for (int qt = 0; qt < NQT; ++qt) {
        float(&acc)[4] = (ks & 1) ? sz[qt] : sa[qt];
        mma_16816(acc, af, qb[qt][ks][0], qb[qt][ks][1]);
        mma_16816(acc, af, qbl[qt][ks][0], qbl[qt][ks][1]);
      }
      if (sk.tree) {  // + k lo . q hi (stage 1 holds the tree chunk's lo halves)
        ldsm_x4(af, ka + Ring::STB);
#pragma unroll
        for (int qt = 0; qt < NQT; ++qt) {
          float(&acc)[4] = (ks & 1) ? sz[qt] : sa[qt];
          mma_16816(acc, af, qb[qt][ks][0], qb[qt][ks][1]);
        }
      }
    }
    // element e: key kw + g + 8 (e >> 1), query qt*8 + 2 t4 + (e & 1)
    float s[NQT][4];
#pragma unroll
    for (int qt = 0; qt < NQT; ++qt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = c0 + kw + g + (e >> 1) * 8;
        const uint32_t* mb = mrow_bits[qt][e & 1];
        bool ok = key < sk.hi && mb;
        if (ok && sk.tree) ok = (mb[key >> 5] >> (key & 31)) & 1u;
        s[qt][e] = ok ? sa[qt][e] + sz[qt][e] : -INFINITY;
      }
    // online softmax per query column: max over the warp's 16 keys (lanes that
    // differ in g), rescale, exponentials; sums stay per lane until the end
    float alpha[NQT][2];
#pragma unroll
    for (int qt = 0; qt < NQT; ++qt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float mx = fmaxf(s[qt][e], s[qt][e + 2]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float mn = fmaxf(mq[qt][e], mx);
        alpha[qt][e] = (mq[qt][e] == -INFINITY) ? 0.f : expf(mq[qt][e] - mn);
        mq[qt][e] = mn;
        float ps = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float v = s[qt][e + 2 * h];
          const float p = (mn == -INFINITY || v == -INFINITY) ? 0.f : expf(v - mn);
          s[qt][e + 2 * h] = p;
          ps += p;
        }
        lq[qt][e] = lq[qt][e] * alpha[qt][e] + ps;
      }
    // P^T as the B operand: (keys g, queries 2 t4 .. +1) pairs, transposed to
    // (keys 2 t4 .. +1, query g); keys 0-7 give b0, keys 8-15 b1
    uint32_t pb[NQT][2], pbl[NQT][2];
#pragma unroll
    for (int qt = 0; qt < NQT; ++qt) {
      uint32_t h0, l0, h1, l1;
      split_pair(s[qt][0], s[qt][1], h0, l0);
      split_pair(s[qt][2], s[qt][3], h1, l1);
      pb[qt][0] = movmatrix_t(h0);
      pb[qt][1] = movmatrix_t(h1);
      pbl[qt][0] = movmatrix_t(l0);
      pbl[qt][1] = movmatrix_t(l1);
    }
    // O^T += V^T P^T: the A operand is V^T's 16 x 16 tile (dims x keys), read
    // transposed from V's rows -- matrix mat: keys +8 if mat >> 1, dims +8 if mat & 1
    const uint32_t vrow = ring.vstage32(st) + (kw + r8 + (mat >> 1) * 8) * 128;
#pragma unroll
    for (int dt = 0; dt < NKS; ++dt) {
      const uint32_t va = vrow + (dt >> 2) * Ring::HB + ((((dt & 3) * 2 + (mat & 1)) ^ r8) << 4);
      uint32_t av[4];
      ldsm_x4_trans(av[0], av[1], av[2], av[3], va);
#pragma unroll
      for (int qt = 0; qt < NQT; ++qt) {
        ot[dt][qt][0] *= alpha[qt][0];
        ot[dt][qt][1] *= alpha[qt][1];
        ot[dt][qt][2] *= alpha[qt][0];
        ot[dt][qt][3] *= alpha[qt][1];
        mma_16816(ot[dt][qt], av, pb[qt][0], pb[qt][1]);
        mma_16816(ot[dt][qt], av, pbl[qt][0], pbl[qt][1]);
      }
      if (sk.tree) {  // + v lo . p hi
        ldsm_x4_trans(av[0], av[1], av[2], av[3], va + Ring::STB);
#pragma unroll
        for (int qt = 0; qt < NQT; ++qt) mma_16816(ot[dt][qt], av, pb[qt][0], pb[qt][1]);
      }
    }
    __syncthreads();  // this stage is refilled at the next chunk
  }
  // sums over the warp's keys (lanes that differ in g)
#pragma unroll
  for (int qt = 0; qt < NQT; ++qt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      lq[qt][e] += __shfl_xor_sync(0xffffffffu, lq[qt][e], 4);
      lq[qt][e] += __shfl_xor_sync(0xffffffffu, lq[qt][e], 8);
      lq[qt][e] += __shfl_xor_sync(0xffffffffu, lq[qt][e], 16);
    }
  // the four warps' states meet in shared memory (the ring is free by now)
  constexpr int NQ = 8 * NQT;
  float* cm = reinterpret_cast<float*>(att_smem);  // [4 warps][NQ] max
  float* cl = cm + 4 * NQ;                          // [4][NQ] sum
  float* co = cl + 4 * NQ;                          // [4][NQ][DH] unnormalised o
#pragma unroll
  for (int qt = 0; qt < NQT; ++qt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int q = qt * 8 + t4 * 2 + e;
      if (g == 0) {
        cm[warp * NQ + q] = mq[qt][e];
        cl[warp * NQ + q] = lq[qt][e];
      }
#pragma unroll
      for (int dt = 0; dt < NKS; ++dt) {
        co[((size_t)warp * NQ + q) * DH + dt * 16 + g] = ot[dt][qt][e];
        co[((size_t)warp * NQ + q) * DH + dt * 16 + g + 8] = ot[dt][qt][e + 2];
      }
    }
  __syncthreads();
  for (int idx = tid; idx < nq * DH; idx += blockDim.x) {
    const int q = idx / DH, dim = idx % DH;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, cm[w * NQ + q]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float mw = cm[w * NQ + q];
      const float e = mw == -INFINITY ? 0.f : expf(mw - M);
      L += cl[w * NQ + q] * e;
      O += co[((size_t)w * NQ + q) * DH + dim] * e;
    }
    const int row = b * a.rows_per_req + q / G, head = kvh * G + q % G;
    const size_t base = ((size_t)split * R + row) * a.Hq + head;
    a.o_part[base * DH + dim] = O;
    if (dim == 0) {
      a.ml_part[base * 2] = M;
      a.ml_part[base * 2 + 1] = L;
    }
  }
}

// Wide query groups (more than 16 queries per KV head: tree frontiers, verify
// passes) on the tcgen05 tensor cores.  The 128 query rows of a group are the
// MMA's M dimension and TMEM's lanes; warps w and w + 4 share lane quarter
// w % 4 (rows 32 (w % 4) .. + 31), each taking half of a chunk's 64 keys and
// half of O's columns, so the softmax of a row is split over two threads that
// meet once per chunk (their row maxima, through shared memory).  Per chunk:
//   S = Q K^T: Q staged once as bf16 hi + lo, scaled by log2(e)/sqrt(dh) so S
//     is in base-2 units; K the ring's rows as a K-major B operand.
//   P = 2^(S - m) (one ex2.approx per element) with a lazy reference max m: O
//     and l are rescaled only when the row max has grown by more than kRescale
//     (P stays below 2^kRescale; O and l share m, so the result is exact).
//   O += P V: P written as bf16 hi + lo rows (K-major A operand), V read in
//     place as an MN-major B operand, one 64-dim half (N = 64) per MMA.
// One thread issues the MMAs; tcgen05.commit arrives on s_bar / o_bar.
template <int DH>
struct TcAttLayout {
  using Ring = KvRing<DH>;
  static constexpr int NH = DH / 64;
  static constexpr int QB = 128 * 128;  // bytes of a 64-dim half of the 128-row Q tile
  static constexpr int PB = 128 * 128;  // bytes of a P tile: 128 rows x 64 keys
  static constexpr int GAP = 2048;      // barriers, TMEM slot, abort word, the row maxima exchange
  static constexpr int SMEM = 1024 + KST * Ring::STB + GAP + 2 * NH * QB + 2 * PB;
  static constexpr uint32_t S_COL = 0, O_COL = 64, TM_COLS = DH == 128 ? 256 : 128;
};

__device__ __forceinline__ float ex2_approx(float x) {  // 2^x; 2^-inf = 0
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int DH>
__global__ void __launch_bounds__(256, 1) prefix_attention_tc_kernel(const __grid_constant__ AttnArgs a) {
  using L = TcAttLayout<DH>;
  using Ring = KvRing<DH>;
  constexpr int NH = L::NH;
  constexpr int OC = DH / 2;            // O columns of each of a row's two threads
  constexpr float kRescale = 12.f;      // base-2 units
  constexpr float kLn2 = 0.6931471805599453f, kLog2e = 1.4426950408889634f;
  constexpr uint32_t IDESC_S = att_idesc(64, false), IDESC_O = att_idesc(64, true);
  extern __shared__ __align__(16) unsigned char att_smem[];
  const int tid = threadIdx.x, warp = tid >> 5;
  const int rt = tid & 127, hv = tid >> 7;  // row of the group; which half of keys and of O
  const int b = blockIdx.x / a.Hkv, kvh = blockIdx.x % a.Hkv, split = blockIdx.z;
  const int G = a.Hq / a.Hkv, nq = a.rows_per_req * G;
  const int R = a.B * a.rows_per_req;
  const SplitKeys sk = split_keys(a, b, split, tid == 0 && split == 0 && kvh == 0 && blockIdx.y == 0);
  Ring ring;
  ring.init(att_smem, b, kvh, sk);
  unsigned char* gap = ring.sb + KST * Ring::STB;  // the ring's barriers take its first 8 KST bytes
  const uint32_t gap32 = ring.sb32 + KST * Ring::STB;
  const uint32_t s_bar = gap32 + 64, o_bar = gap32 + 72;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(gap + 80);
  volatile int* abort_f = reinterpret_cast<volatile int*>(gap + 84);
  float* xmax = reinterpret_cast<float*>(gap + 1024);  // [2 halves][128 rows]
  unsigned char* qs = gap + L::GAP;         // [hi, lo][NH][128 rows][128 B]
  unsigned char* ps = qs + 2 * NH * L::QB;  // [hi, lo][128 rows][128 B]
  const uint32_t qs32 = smem_u32(qs), ps32 = smem_u32(ps);

  if (warp == 0) utc_alloc(smem_u32(tslot), L::TM_COLS);
  if (tid == 0) {
    att_mbar_init(s_bar, 1);
    att_mbar_init(o_bar, 1);
    *abort_f = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  utc_fence_before();
  // as in the kernels above: with a stable prefix the first chunks are
  // requested before the wait for the previous kernel
  const bool early = a.prefix_stable && !sk.tree && sk.n_chunks > 0;
  if (early)
    ring.start(a);  // ends in a block barrier
  else
    __syncthreads();
  utc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);  // this warp's TMEM lanes
  pdl_begin();
  const bool live = !(a.skip && *a.skip == 0);

  // this thread's query row
  const int q = blockIdx.y * 128 + rt;
  const bool qv = live && q < nq;
  const float* qp = nullptr;
  const uint32_t* mrow = nullptr;
  int row = 0, head = 0;
  if (qv) {
    row = b * a.rows_per_req + q / G;
    head = kvh * G + q % G;
    qp = a.q + (size_t)a.q_row[row] * a.Hq * DH + (size_t)head * DH;
    mrow = a.mask + (size_t)row * a.mask_words;
  }
  if (live) {
    // the row of Q (this thread: half hv of its 16-byte pieces), scaled to base-2 units
    const float scale = rsqrtf((float)DH) * kLog2e;
#pragma unroll 1
    for (int p = hv * (DH / 16); p < (hv + 1) * (DH / 16); ++p) {
      float x[8];
      if (qp) {
        const float4 u0 = reinterpret_cast<const float4*>(qp)[2 * p];
        const float4 u1 = reinterpret_cast<const float4*>(qp)[2 * p + 1];
        x[0] = u0.x; x[1] = u0.y; x[2] = u0.z; x[3] = u0.w;
        x[4] = u1.x; x[5] = u1.y; x[6] = u1.z; x[7] = u1.w;
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = 0.f;
      }
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) split_pair(x[2 * e] * scale, x[2 * e + 1] * scale, hi[e], lo[e]);
      const int off = (p >> 3) * L::QB + rt * 128 + (((p & 7) ^ (rt & 7)) << 4);
      *reinterpret_cast<uint4*>(qs + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(qs + NH * L::QB + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    // O = 0 (this warp's half of the columns)
    float z[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) z[i] = 0.f;
#pragma unroll
    for (int c = 0; c < OC; c += 32) utc_st32(trow + L::O_COL + hv * OC + c, z);
    if (sk.tree) {
      if (sk.n_chunks > 0) ring.load_tree(a);
    } else if (!early) {
      ring.start(a);
    }
  } else if (early) {
    ring.drain_start(a);  // the requested chunks land before the shared memory is released
  }
  async_proxy_fence();  // Q, O's zeros and a tree chunk, before the tensor core reads them
  utc_fence_before();
  __syncthreads();

  float m = -INFINITY, l = 0.f;  // base-2 reference max of the row; this thread's share of the sum
  int done = 0;    // chunks whose P V was issued
  int landed = 0;  // prefix chunks awaited (those up to landed + KST - 2 were requested)
  bool drain = false;
  for (int ci = 0; live && ci < sk.n_chunks; ++ci) {
    const int c0 = sk.lo + ci * KC, st = sk.tree ? 0 : ci % KST;
    // the previous chunk's P V must be complete: its stage is refilled next and P rewritten
    bool ok = ci == 0 || att_wait_abort(o_bar, (uint32_t)(ci - 1) & 1u, a.flags, abort_f);
    if (!__syncthreads_and(ok)) {
      drain = !sk.tree;
      break;
    }
    if (!sk.tree) {
      if (!ring.next(a, ci)) break;  // it lets its own requests land
      landed = ci + 1;
    }
    if (tid == 0) {  // S = Q K^T
      utc_fence_after();
      const uint32_t kb = ring.kstage32(st);
#pragma unroll
      for (int h = 0; h < NH; ++h)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t bk = att_desc(kb + h * Ring::HB + kk * 32);
          const uint32_t qa = qs32 + h * L::QB + kk * 32;
          utc_mma(tmem + L::S_COL, att_desc(qa), bk, IDESC_S, (h | kk) ? 1u : 0u);
          utc_mma(tmem + L::S_COL, att_desc(qa + NH * L::QB), bk, IDESC_S, 1u);
          if (sk.tree)  // + q hi . k lo (stage 1 holds the tree chunk's lo halves)
            utc_mma(tmem + L::S_COL, att_desc(qa), att_desc(kb + Ring::STB + h * Ring::HB + kk * 32),
                    IDESC_S, 1u);
        }
      utc_commit(s_bar);
    }
    ok = att_wait_abort(s_bar, (uint32_t)ci & 1u, a.flags, abort_f);
    if (!__syncthreads_and(ok)) {
      drain = !sk.tree;
      break;
    }
    utc_fence_after();
    float sv[32];  // keys c0 + 32 hv + j
    utc_ld32(trow + L::S_COL + 32 * hv, sv);
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int key = c0 + 32 * hv + j;
      bool keep = qv && key < sk.hi;
      if (keep && sk.tree) keep = (mrow[key >> 5] >> (key & 31)) & 1u;
      if (!keep) sv[j] = -INFINITY;
      mx = fmaxf(mx, sv[j]);
    }
    // the two threads of the row meet: row max over the chunk's 64 keys
    xmax[hv * 128 + rt] = mx;
    asm volatile("bar.sync %0, 64;" ::"r"(1 + (warp & 3)) : "memory");
    mx = fmaxf(mx, xmax[(hv ^ 1) * 128 + rt]);
    // lazy reference max (the same decision in both threads of the row)
    float alpha = 1.f;
    if (mx > m + kRescale) {
      alpha = m == -INFINITY ? 0.f : ex2_approx(m - mx);
      m = mx;
    }
    if (__any_sync(0xffffffffu, alpha != 1.f)) {  // the TMEM row access is warp-wide
#pragma unroll
      for (int c = 0; c < OC; c += 32) {
        float o[32];
        utc_ld32(trow + L::O_COL + hv * OC + c, o);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] *= alpha;
        utc_st32(trow + L::O_COL + hv * OC + c, o);
      }
    }
    l *= alpha;
    // P: this thread's 4 pieces of 8 keys, hi and lo, swizzled like the other operands
#pragma unroll
    for (int pc = 0; pc < 4; ++pc) {
      float pv[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float v = sv[pc * 8 + e];
        pv[e] = (v == -INFINITY) ? 0.f : ex2_approx(v - m);
        l += pv[e];
      }
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) split_pair(pv[2 * e], pv[2 * e + 1], hi[e], lo[e]);
      const int piece = 4 * hv + pc;
      const int off = rt * 128 + ((piece ^ (rt & 7)) << 4);
      *reinterpret_cast<uint4*>(ps + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(ps + L::PB + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    async_proxy_fence();
    utc_fence_before();
    __syncthreads();
    if (tid == 0) {  // O += P V
      utc_fence_after();
      const uint32_t vb = ring.vstage32(st);
#pragma unroll
      for (int h = 0; h < NH; ++h)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {  // keys 16 kk .. + 15: rows 16 kk of V's half h
          const uint64_t bv = att_desc_mn(vb + h * Ring::HB + kk * 2048);
          const uint32_t od = tmem + L::O_COL + 64 * h;
          utc_mma(od, att_desc(ps32 + kk * 32), bv, IDESC_O, 1u);
          utc_mma(od, att_desc(ps32 + L::PB + kk * 32), bv, IDESC_O, 1u);
          if (sk.tree)  // + p hi . v lo
            utc_mma(od, att_desc(ps32 + kk * 32), att_desc_mn(vb + Ring::STB + h * Ring::HB + kk * 2048),
                    IDESC_O, 1u);
        }
      utc_commit(o_bar);
    }
    done = ci + 1;
  }
  if (drain)  // requested chunks land before the shared memory is released
    for (int c = landed; c < sk.n_chunks && c < landed + KST - 1; ++c)
      att_wait(ring.bar0 + 8u * (c % KST), (uint32_t)(c / KST) & 1u, a.flags);
  // the last P V, then the row's O, max (natural units) and sum
  bool ok = done == 0 || att_wait_abort(o_bar, (uint32_t)(done - 1) & 1u, a.flags, abort_f);
  ok = __syncthreads_and(ok) && live && !*abort_f;
  utc_fence_after();
  if (ok) {
    xmax[hv * 128 + rt] = l;
    const size_t base = ((size_t)split * R + row) * a.Hq + head;
#pragma unroll
    for (int c = 0; c < OC; c += 32) {
      float o[32];
      utc_ld32(trow + L::O_COL + hv * OC + c, o);  // warp-wide: every lane loads
      if (qv) {
        float4* op = reinterpret_cast<float4*>(a.o_part + base * DH + hv * OC + c);
#pragma unroll
        for (int i = 0; i < 8; ++i) op[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
      }
    }
    asm volatile("bar.sync %0, 64;" ::"r"(1 + (warp & 3)) : "memory");
    if (qv && hv == 0) {
      a.ml_part[base * 2] = m * kLn2;
      a.ml_part[base * 2 + 1] = l + xmax[128 + rt];
    }
  }
  utc_fence_before();
  __syncthreads();
  if (warp == 0) utc_dealloc(tmem, L::TM_COLS);
}

// merge the key splits of one (row, head): o = sum_s o_s e^{m_s - m} / sum_s l_s e^{m_s - m}
template <typename T>
__global__ void attention_combine_kernel(AttnArgs a) {
  pdl_begin();
  if (a.skip && *a.skip == 0) return;
  __shared__ float wts[256];  // per split: its weight e^{m_s - m} / l
  __shared__ float red[32];
  const int row = blockIdx.x, head = blockIdx.y, tid = threadIdx.x;
  const int R = a.B * a.rows_per_req;
  const int n_splits = a.n_prefix_splits + a.n_tree_splits;
  // every split's (max, sum) at once, then the global max and sum
  float m = -INFINITY;
  for (int s = tid; s < n_splits; s += blockDim.x) {
    const float ms = a.ml_part[(((size_t)s * R + row) * a.Hq + head) * 2];
    wts[s] = ms;
    m = fmaxf(m, ms);
  }
  m = warp_max(m);
  if ((tid & 31) == 0) red[tid >> 5] = m;
  __syncthreads();
  if (tid < 32) {
    float v = tid < (int)(blockDim.x >> 5) ? red[tid] : -INFINITY;
    v = warp_max(v);
    if (tid == 0) red[0] = v;
  }
  __syncthreads();
  m = red[0];
  __syncthreads();
  float l = 0.f;
  for (int s = tid; s < n_splits; s += blockDim.x) {
    const float ms = wts[s];
    const float w = ms == -INFINITY ? 0.f : expf(ms - m);
    l += w * a.ml_part[(((size_t)s * R + row) * a.Hq + head) * 2 + 1];
    wts[s] = w;
  }
  l = block_sum(l, red);
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const size_t sstride = (size_t)R * a.Hq * a.dh;  // one split's partials
  for (int dd = tid; dd < a.dh; dd += blockDim.x) {
    // eight splits' loads in flight at a time, each into its own accumulator
    const float* op = a.o_part + ((size_t)row * a.Hq + head) * a.dh + dd;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    int s = 0;
    for (; s + 8 <= n_splits; s += 8) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = op[(size_t)(s + u) * sstride];
#pragma unroll
      for (int u = 0; u < 8; ++u) acc[u] += v[u] * wts[s + u];
    }
    for (; s < n_splits; ++s) acc[0] += op[(size_t)s * sstride] * wts[s];
    float o = 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u) o += acc[u];
    st_act((T*)a.out + act_row(row, a.Hq * a.dh, a.split), a.Hq * a.dh, head * a.dh + dd, o * inv,
           a.split);
  }
}

template <typename T>
void launch_tree_attention(const AttnArgs& a, cudaStream_t st) {
  int R = a.B * a.rows_per_req;
  if (R <= 0) return;
  int n_splits = a.n_prefix_splits + a.n_tree_splits;
  const bool mma = attention_uses_mma((int)sizeof(T), a.dh, a.page_size);
  size_t smem = (size_t)(QG * (a.dh + 1) + KC * (a.dh + 1) + KC * a.dh + QG * KC + 3 * QG) *
                sizeof(float);
  // a refused limit shows as the launch's own error, which the caller reports
  smem_limit((const void*)tree_attention_kernel<T>, 160 * 1024);
  smem_limit((const void*)prefix_attention_mma_kernel<64>, KvRing<64>::SMEM);
  smem_limit((const void*)prefix_attention_mma_kernel<128>, KvRing<128>::SMEM);
  smem_limit((const void*)prefix_attention_tc_kernel<64>, TcAttLayout<64>::SMEM);
  smem_limit((const void*)prefix_attention_tc_kernel<128>, TcAttLayout<128>::SMEM);
  smem_limit((const void*)prefix_attention_kt_kernel<64, 1>, KvRing<64>::SMEM);
  smem_limit((const void*)prefix_attention_kt_kernel<64, 2>, KvRing<64>::SMEM);
  smem_limit((const void*)prefix_attention_kt_kernel<128, 1>, KvRing<128>::SMEM);
  smem_limit((const void*)prefix_attention_kt_kernel<128, 2>, KvRing<128>::SMEM);
  if (mma) {  // prefix and tree splits in one launch
    dim3 gp(a.B * a.Hkv, attention_qgroups(a.rows_per_req, a.Hq, a.Hkv, true), n_splits);
    const int nq = a.rows_per_req * (a.Hq / a.Hkv);
    const dim3 blk(128);
    if (a.dh == 128) {
      const size_t sm2 = KvRing<128>::SMEM;
      if (nq <= 8)
        launch_pdl(prefix_attention_kt_kernel<128, 1>, dim3(gp), blk, sm2, st, a);
      else if (nq <= QKT)
        launch_pdl(prefix_attention_kt_kernel<128, 2>, dim3(gp), blk, sm2, st, a);
      else if (nq <= QTC)
        launch_pdl(prefix_attention_mma_kernel<128>, dim3(gp), blk, sm2, st, a);
      else
        launch_pdl(prefix_attention_tc_kernel<128>, dim3(gp), dim3(256), (size_t)TcAttLayout<128>::SMEM, st, a);
    } else {
      const size_t sm2 = KvRing<64>::SMEM;
      if (nq <= 8)
        launch_pdl(prefix_attention_kt_kernel<64, 1>, dim3(gp), blk, sm2, st, a);
      else if (nq <= QKT)
        launch_pdl(prefix_attention_kt_kernel<64, 2>, dim3(gp), blk, sm2, st, a);
      else if (nq <= QTC)
        launch_pdl(prefix_attention_mma_kernel<64>, dim3(gp), blk, sm2, st, a);
      else
        launch_pdl(prefix_attention_tc_kernel<64>, dim3(gp), dim3(256), (size_t)TcAttLayout<64>::SMEM, st, a);
    }
  } else {
    dim3 grid(a.B * a.Hkv, attention_qgroups(a.rows_per_req, a.Hq, a.Hkv, false), n_splits);
    launch_pdl(tree_attention_kernel<T>, dim3(grid), dim3(NT), smem, st, a, 0);
  }
  dim3 g2(R, a.Hq);
  launch_pdl(attention_combine_kernel<T>, dim3(g2), dim3(a.dh), 0, st, a);
}

template void launch_tree_attention<float>(const AttnArgs&, cudaStream_t);
template void launch_tree_attention<bf16>(const AttnArgs&, cudaStream_t);

}  // namespace e3
