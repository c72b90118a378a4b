// Row plans, frontier expansion and the tree builder.
//
// EAGLE-2 confidence-value dynamic tree ("EAGLE-3 精读" 核心变化 and §2 last
// paragraph); a node's confidence is the product of draft probabilities along
// its path (EAGLE-4 blog, 几条技术路线正在收敛), kept here as a sum of log q.
// Reading of the expansion (the pages do not spell it out): depth 1 is the
// root's k children; each deeper level expands the k best-scoring nodes of the
// level above into k*k candidates; the tree kept for verification is the
// global top-M of every created node by (score desc, depth asc, creation id
// asc).  Because log q <= 0 and ties prefer the shallower node, the kept set is
// ancestor-closed.
//
// Pool layout per request (creation order): depth 1 at [0, k); depth t >= 2 at
// k + (t-2) k^2 + (parent's frontier rank) k + child rank.  Frontier slot of
// the rank-r node of depth t: (t-1) k + r.  State rows per request:
// 0 = root, 1 + slot = frontier node.
#include "common.cuh"
#include "kernels.h"

namespace e3 {

// ----------------------------------------------------------------------------- pass 0 plan
// Request b's new rows are rows r0 .. r1-1 of the round's packed rows: r0 =
// cu_new[b], r1 = cu_new[b+1] (or n_new rows each when cu_new is NULL); the
// last one is the tree's root.  A count outside [1, max_new] or past `total`
// raises FLAG_ROWS_RANGE and is clamped so that every index stays in range.
__global__ void plan_root_kernel(int B, int n_new, const int* cu_new, int total, int max_new,
                                 const int* tokens_new, const int* seq_lens, int n_slots,
                                 RowPlan rp, int* root_tok, int* root_pos, int* n_prefix,
                                 int* flags) {
  pdl_begin();
  int b = blockIdx.x;
  int L = seq_lens[b];
  int r0 = cu_new ? cu_new[b] : b * n_new;
  int r1 = cu_new ? cu_new[b + 1] : r0 + n_new;
  if (r0 < 0 || r1 > total || r1 - r0 < 1 || r1 - r0 > max_new) {
    if (threadIdx.x == 0) raise_flag(flags, FLAG_ROWS_RANGE);
    r0 = min(max(r0, 0), total - 1);
    r1 = min(max(r1, r0 + 1), min(total, r0 + max_new));
  }
  for (int j = threadIdx.x; j < r1 - r0; j += blockDim.x) {
    int r = r0 + j;
    rp.kv_b[r] = b;
    rp.kv_tok[r] = tokens_new[r];
    rp.kv_hid[r] = r;
    rp.kv_pos[r] = L + j;
    rp.kv_dst[r] = -1;
  }
  if (threadIdx.x == 0) {
    int rr = r1 - 1;
    rp.t_q[b] = rr;
    rp.t_b[b] = b;
    rp.t_hid[b] = rr;
    rp.t_sdst[b] = b * (1 + n_slots);
    rp.t_out[b] = b;
    root_tok[b] = tokens_new[rr];
    root_pos[b] = L + (r1 - r0) - 1;
    n_prefix[b] = L + (r1 - r0);
  }
  for (int w = threadIdx.x; w < rp.mask_words; w += blockDim.x) rp.t_mask[(size_t)b * rp.mask_words + w] = 0u;
}

void launch_plan_root(int B, int n_new, const int* cu_new, int total, int max_new,
                      const int* tokens_new, const int* seq_lens, int n_slots, const RowPlan& rp,
                      int* root_tok, int* root_pos, int* n_prefix, int* flags, cudaStream_t st) {
  launch_pdl(plan_root_kernel, dim3(B), dim3(64), 0, st, B, n_new, cu_new, total, max_new,
             tokens_new, seq_lens, n_slots, rp, root_tok, root_pos, n_prefix, flags);
}

// ----------------------------------------------------------------------------- next round's rows
// From a verification: request b's next rows are its accepted tokens and the
// bonus token, out_tokens[b][0 .. accept_len[b]], packed by request with
// offsets cu_new.  One block; the prefix sum over requests is serial.
__global__ void next_rows_kernel(int B, int D, const int* accept_len, const int* out_tokens,
                                 int* cu_new, int* tokens_new, int* flags) {
  pdl_begin();
  __shared__ int off[1025];
  if (threadIdx.x == 0) {
    int acc = 0;
    off[0] = 0;
    for (int b = 0; b < B; ++b) {
      int a = accept_len[b];
      if (a < 0 || a > D) {
        raise_flag(flags, FLAG_ROWS_RANGE);
        a = a < 0 ? 0 : D;
      }
      acc += a + 1;
      off[b + 1] = acc;
    }
  }
  __syncthreads();
  for (int b = threadIdx.x; b <= B; b += blockDim.x) cu_new[b] = off[b];
  for (int b = 0; b < B; ++b) {
    const int n = off[b + 1] - off[b];
    for (int i = threadIdx.x; i < n; i += blockDim.x)
      tokens_new[off[b] + i] = out_tokens[(size_t)b * (D + 1) + i];
  }
}

void launch_next_rows(int B, int D, const int* accept_len, const int* out_tokens, int* cu_new,
                      int* tokens_new, int* flags, cudaStream_t st) {
  launch_pdl(next_rows_kernel, dim3(1), dim3(256), 0, st, B, D, accept_len, out_tokens, cu_new,
             tokens_new, flags);
}

// ----------------------------------------------------------------------------- prefill plan
__global__ void plan_prefill_kernel(int rows, int r0, int B, const int* cu_rows, const int* tokens,
                                    const int* seq_lens, RowPlan rp) {
  pdl_begin();
  int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= rows) return;
  int r = r0 + i;
  int lo = 0, hi = B - 1;  // last b with cu_rows[b] <= r
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (cu_rows[mid] <= r) lo = mid; else hi = mid - 1;
  }
  rp.kv_b[i] = lo;
  rp.kv_tok[i] = tokens[r];
  rp.kv_hid[i] = i;
  rp.kv_pos[i] = seq_lens[lo] + (r - cu_rows[lo]);
  rp.kv_dst[i] = -1;
}

void launch_plan_prefill(int rows, int r0, int B, const int* cu_rows, const int* tokens,
                         const int* seq_lens, const RowPlan& rp, cudaStream_t st) {
  if (rows <= 0) return;
  launch_pdl(plan_prefill_kernel, dim3((rows + 255) / 256), dim3(256), 0, st, rows, r0, B, cu_rows, tokens, seq_lens, rp);
}

// ----------------------------------------------------------------------------- expansion (per pass)
// After the LM head of pass t (t = 0: the root, one row per request; t >= 1: the
// depth-t frontier, k rows per request): append the children to the pool,
// choose the depth-(t+1) frontier if another pass follows, and write that
// pass's row plan.
__global__ void expand_kernel(CtlDev ctl, int B, int t, int k, int D, const int* __restrict__ top_tok,
                              const float* __restrict__ top_logq, PoolDev pool, int* frontier,
                              uint32_t* slot_mask, int slot_words, const int* root_pos,
                              int n_slots, RowPlan rp) {
  pdl_begin();
  __shared__ float sc[256];
  __shared__ int nf[16];
  __shared__ int s_deff;
  int b = blockIdx.x, tid = threadIdx.x;
  int* ptok = pool.tok + (size_t)b * pool.n;
  int* ppar = pool.parent + (size_t)b * pool.n;
  int* pdep = pool.depth + (size_t)b * pool.n;
  int* pfwd = pool.fwd + (size_t)b * pool.n;
  float* psc = pool.score + (size_t)b * pool.n;
  float* plq = pool.logq + (size_t)b * pool.n;
  int* fr = frontier + b * k;
  // depth this request runs to, and its branch cap
  int kb = k;
  if (tid == 0) {
    int de = D;
    if (ctl.on) {
      if (t == 0) {
        if (ctl.depth_cap) de = max(1, min(D, ctl.depth_cap[b]));
        ctl.d_eff[b] = de;
      } else {
        de = ctl.d_eff[b];
      }
    }
    s_deff = de;
  }
  if (ctl.on) {
    kb = ctl.k_call;
    if (ctl.topk_cap) kb = max(1, min(kb, ctl.topk_cap[b]));
  }
  __syncthreads();
  const bool run = t < s_deff;  // this pass expands the request's frontier
  int n_new = (t == 0) ? k : k * k;
  int base = (t == 0) ? 0 : k + (t - 1) * k * k;
  if (tid < n_new) {
    int i = tid / k, j = tid % k;  // parent's frontier rank, child rank
    int row = (t == 0) ? b : b * k + i;
    int parent = (t == 0) ? -1 : fr[i];
    const bool real = run && j < kb && (t == 0 || psc[parent] != -INFINITY);
    int idx = base + tid;
    pdep[idx] = t + 1;
    pfwd[idx] = -1;
    if (real) {
      float lq = top_logq[(size_t)row * k + j];
      float lc = lq;
      if (ctl.clip) {  // sampled draft: min(log max q, log q of the earlier draws), never its own
        lc = ctl.lmax[row];
        for (int j2 = 0; j2 < j; ++j2) lc = fminf(lc, top_logq[(size_t)row * k + j2]);
      }
      float s = (parent < 0 ? 0.f : psc[parent]) + lc;
      ptok[idx] = top_tok[(size_t)row * k + j];
      ppar[idx] = parent;
      psc[idx] = s;
      plq[idx] = lq;
      sc[tid] = s;
    } else {  // not created: a cap, the depth rule or an empty frontier slot
      ptok[idx] = -1;
      ppar[idx] = -1;
      psc[idx] = -INFINITY;
      plq[idx] = -INFINITY;
      sc[tid] = -INFINITY;
    }
  }
  __syncthreads();
  if (t + 1 > D - 1) return;  // no further pass
  // frontier of depth t+1: rank of each candidate under (score desc, index asc)
  if (t == 0) {
    if (tid < k) nf[tid] = tid;
  } else if (tid < n_new) {
    float s = sc[tid];
    int rank = 0;
    for (int c = 0; c < n_new; ++c) rank += (sc[c] > s) || (sc[c] == s && c < tid);
    if (rank < k) nf[rank] = base + tid;
  }
  __syncthreads();
  if (tid == 0 && ctl.on) {
    // the depth rule: draft pass t+1 only while the frontier's confidence mass
    // pays for the pass; an empty frontier ends the request's drafting too
    int de = s_deff;
    float mass = 0.f;
    for (int r = 0; r < k; ++r) {
      const float s = psc[nf[r]];
      if (s != -INFINITY) mass += expf(s);
    }
    if (t + 1 < de) {
      if (mass == 0.f) de = t + 1;
      else if (ctl.tau_depth > 0.f &&
               !(mass >= ctl.tau_depth * powf(ctl.depth_growth, (float)(t + 1)) * ctl.pass_us[t + 1]))
        de = t + 1;
    }
    ctl.d_eff[b] = de;
    s_deff = de;
    if (t + 1 < de) atomicAdd(ctl.active + t + 1, 1);
  }
  __syncthreads();
  const bool next = t + 1 < s_deff;
  if (tid < k) {
    int r = tid;
    int node = nf[r];
    int slot = t * k + r;  // frontier slot of depth t+1, rank r
    const bool real = next && psc[node] != -INFINITY;
    int parent = real ? ppar[node] : -1;
    if (real) {
      pfwd[node] = slot;
      fr[r] = node;
    } else {
      fr[r] = node;  // an empty slot: its row runs on a placeholder and makes no children
    }
    int srow_base = b * (1 + n_slots);
    int hid = parent < 0 ? srow_base : srow_base + 1 + pfwd[parent];
    int row = b * k + r;
    rp.kv_b[row] = b;
    rp.kv_tok[row] = real ? ptok[node] : 0;
    rp.kv_hid[row] = hid;
    rp.kv_pos[row] = root_pos[b] + t + 1;
    rp.kv_dst[row] = slot;
    rp.t_q[row] = row;
    rp.t_b[row] = b;
    rp.t_hid[row] = hid;
    rp.t_sdst[row] = srow_base + 1 + slot;
    rp.t_out[row] = row;
    uint32_t* mine = slot_mask + ((size_t)b * n_slots + slot) * slot_words;
    const uint32_t* par = parent < 0 ? nullptr : slot_mask + ((size_t)b * n_slots + pfwd[parent]) * slot_words;
    for (int w = 0; w < rp.mask_words; ++w) {
      uint32_t m = 0u;
      if (w < slot_words) {
        m = par ? par[w] : 0u;
        if ((slot >> 5) == w) m |= 1u << (slot & 31);
        mine[w] = m;
      }
      rp.t_mask[(size_t)row * rp.mask_words + w] = m;
    }
  }
}

void launch_expand(const CtlDev& ctl, int B, int t, int k, int D, const int* top_tok, const float* top_logq,
                   const PoolDev& pool, int* frontier, uint32_t* slot_mask, int slot_words,
                   const int* root_pos, int n_slots, const RowPlan& rp, cudaStream_t st) {
  launch_pdl(expand_kernel, dim3(B), dim3(256), 0, st, ctl, B, t, k, D, top_tok, top_logq, pool,
             frontier, slot_mask, slot_words, root_pos, n_slots, rp);
}

// ----------------------------------------------------------------------------- tree builder
// One block per request.  Rank of node i = number of nodes ahead of it in
// (score desc, depth asc, index asc); the kept set is rank < M.  Canonical
// position among the kept nodes: (depth asc, rank asc).
__global__ void build_tree_kernel(CtlDev ctl, int pool_n, int M, const int* __restrict__ tok,
                                  const int* __restrict__ parent, const float* __restrict__ score,
                                  const int* __restrict__ depth, const int* root_tok,
                                  const int* root_pos, int* t_tok, int* t_parent, int* t_depth,
                                  int* t_pos, int* t_pidx, float* t_score, uint32_t* t_mask,
                                  int* flags) {
  pdl_begin();
  extern __shared__ int smi[];
  float* ssc = (float*)smi;             // [pool_n]
  int* sdep = smi + pool_n;             // [pool_n]
  int* tidx = sdep + pool_n;            // [pool_n] tree index of a kept node, else 0x7fffffff
  int* sel = tidx + pool_n;             // [M] pool index by rank
  int* tpar = sel + M;                  // [M+1] tree parent
  // [P2] sort keys, P2 = the power of two >= pool_n (8-byte aligned after tpar)
  unsigned long long* key =
      reinterpret_cast<unsigned long long*>(smi + ((3 * pool_n + 2 * M + 1 + 1) & ~1));
  int P2 = 1;
  while (P2 < pool_n) P2 <<= 1;
  int b = blockIdx.x, tid = threadIdx.x, nt = blockDim.x;
  const size_t pb = (size_t)b * pool_n;
  for (int i = tid; i < P2; i += nt) {
    if (i < pool_n) {
      const float sc = score[pb + i];
      const int dp = depth[pb + i];
      ssc[i] = sc;
      sdep[i] = dp;
      tidx[i] = 0x7fffffff;
      // larger key = earlier in (score desc, depth asc, index asc)
      const uint32_t u = __float_as_uint(sc == 0.f ? 0.f : sc);  // -0 ties with +0
      const uint32_t o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
      key[i] = ((unsigned long long)o << 32) |
               ((unsigned long long)(255 - min(max(dp, 0), 255)) << 24) |
               (unsigned long long)(0xFFFFFFu - (uint32_t)i);
    } else {
      key[i] = 0ull;  // padding sorts last
    }
  }
  __syncthreads();
  // bitonic sort, descending: rank r of the order is key[r]
  for (int k = 2; k <= P2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < P2; i += nt) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const unsigned long long a = key[i], c = key[ixj];
          if (((i & k) == 0) ? (a < c) : (a > c)) {
            key[i] = c;
            key[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int r = tid; r < M && r < pool_n; r += nt)
    sel[r] = (int)(0xFFFFFFu - (uint32_t)(key[r] & 0xFFFFFFull));
  __shared__ int s_mb;
  if (tid == 0) s_mb = M;
  __syncthreads();
  if (ctl.on && tid == 0) {
    // kept count: the request's verify cap, created nodes only, then the
    // verify rule over the selection order (at least one node)
    int mb = M;
    if (ctl.verify_cap) mb = max(1, min(mb, ctl.verify_cap[b]));
    int nfin = 0;
    for (int i = 0; i < pool_n; ++i) nfin += ssc[i] != -INFINITY;
    mb = max(1, min(mb, nfin));
    if (ctl.tau_verify > 0.f) {
      int m = 1;
      while (m < mb && expf(ssc[sel[m]]) >= ctl.tau_verify * (ctl.verify_us[m + 1] - ctl.verify_us[m]))
        ++m;
      mb = m;
    }
    s_mb = mb;
  }
  __syncthreads();
  const int Mb = s_mb;
  for (int q = tid; q < Mb; q += nt) {
    int node = sel[q], dd = sdep[node];
    int p = 0;
    for (int q2 = 0; q2 < Mb; ++q2) {
      int d2 = sdep[sel[q2]];
      p += (d2 < dd) || (d2 == dd && q2 < q);
    }
    tidx[node] = 1 + p;
  }
  __syncthreads();
  const int M1 = M + 1;
  const size_t tb = (size_t)b * M1;
  int rp = root_pos[b];
  for (int u = Mb + 1 + tid; u <= M; u += nt) {  // slots past the kept count
    tpar[u] = -1;
    t_tok[tb + u] = -1;
    t_parent[tb + u] = -1;
    t_depth[tb + u] = 0;
    t_pos[tb + u] = rp;
    t_pidx[tb + u] = -1;
    t_score[tb + u] = -INFINITY;
  }
  for (int q = tid; q < Mb; q += nt) {
    int node = sel[q];
    int u = tidx[node];
    int pp = parent[pb + node];
    int tp = 0;
    if (pp >= 0) {
      tp = (pp < pool_n) ? tidx[pp] : 0x7fffffff;
      if (tp == 0x7fffffff) {
        raise_flag(flags, FLAG_TREE_NOT_CLOSED);
        tp = 0;
      }
    }
    tpar[u] = tp;
    t_tok[tb + u] = tok[pb + node];
    t_parent[tb + u] = tp;
    t_depth[tb + u] = sdep[node];
    t_pos[tb + u] = rp + sdep[node];
    t_pidx[tb + u] = node;
    t_score[tb + u] = ssc[node];
  }
  if (tid == 0) {
    tpar[0] = -1;
    t_tok[tb] = root_tok[b];
    t_parent[tb] = -1;
    t_depth[tb] = 0;
    t_pos[tb] = rp;
    t_pidx[tb] = -1;
    t_score[tb] = 0.f;
  }
  __syncthreads();
  const int W = (M1 + 31) / 32;
  for (int u = tid; u < M1; u += nt) {
    uint32_t m[5] = {0u, 0u, 0u, 0u, 0u};
    int j = u, guard = 0;
    while (j >= 0 && guard++ <= M1) {
      m[j >> 5] |= 1u << (j & 31);
      j = tpar[j];
      if (j >= u) break;  // parents precede children; anything else is a broken tree
    }
    for (int w = 0; w < W; ++w) t_mask[(tb + u) * W + w] = m[w];
  }
}

void launch_build_tree(const CtlDev& ctl, int B, int pool_n, int M, const int* tok, const int* parent,
                       const float* score, const int* depth, const int* root_tok,
                       const int* root_pos, int* t_tok, int* t_parent, int* t_depth, int* t_pos,
                       int* t_pidx, float* t_score, uint32_t* t_mask, int* flags, cudaStream_t st) {
  int P2 = 1;
  while (P2 < pool_n) P2 <<= 1;
  size_t smem = (size_t)((3 * pool_n + 2 * M + 1 + 1) & ~1) * sizeof(int) + (size_t)P2 * 8;
  smem_limit((const void*)build_tree_kernel, 100 * 1024);  // refusal: the launch fails
  launch_pdl(build_tree_kernel, dim3(B), dim3(512), smem, st, ctl, pool_n, M, tok, parent, score, depth, root_tok, root_pos,
                                          t_tok, t_parent, t_depth, t_pos, t_pidx, t_score, t_mask,
                                          flags);
}

// ----------------------------------------------------------------------------- verify plan
// Rows b*M + (u-1) for tree nodes u = 1..M: hid = the parent's state (root:
// state row 0; else the parent's frontier slot), tree KV slot = u, mask = the
// node's mask row without bit 0 (the root's K/V live in the prefix cache).
// Also lists each node's children (canonical order) for the verify walk.
__global__ void plan_verify_kernel(int M, int kmax, const int* t_tok, const int* t_parent,
                                   const int* t_pos, const int* t_pidx, const uint32_t* t_mask,
                                   const int* pool_fwd, int pool_n, int n_slots, RowPlan rp,
                                   int* n_prefix, int* child_tok, int* child_node, int* n_child,
                                   int* flags) {
  pdl_begin();
  int b = blockIdx.x, tid = threadIdx.x;
  const int M1 = M + 1, W = (M1 + 31) / 32;
  const size_t tb = (size_t)b * M1;
  if (tid == 0) n_prefix[b] = t_pos[tb] + 1;
  for (int u = 1 + tid; u <= M; u += blockDim.x) {
    int row = b * M + (u - 1);
    int p = t_parent[tb + u];
    int hid = b * (1 + n_slots);
    if (p > 0) {
      int pi = t_pidx[tb + p];
      int f = (pi >= 0 && pi < pool_n) ? pool_fwd[(size_t)b * pool_n + pi] : -1;
      if (f < 0) {
        raise_flag(flags, FLAG_TREE_NOT_CLOSED);
        f = 0;
      }
      hid += 1 + f;
    }
    rp.kv_b[row] = b;
    rp.kv_tok[row] = max(t_tok[tb + u], 0);  // a padding slot (token -1) runs on a placeholder
    rp.kv_hid[row] = hid;
    rp.kv_pos[row] = t_pos[tb + u];
    rp.kv_dst[row] = u;
    rp.t_q[row] = row;
    rp.t_b[row] = b;
    rp.t_hid[row] = hid;
    rp.t_sdst[row] = -1;
    rp.t_out[row] = b * M1 + u;
    for (int w = 0; w < rp.mask_words; ++w) {
      uint32_t m = w < W ? t_mask[(tb + u) * W + w] : 0u;
      if (w == 0) m &= ~1u;
      rp.t_mask[(size_t)row * rp.mask_words + w] = m;
    }
  }
  for (int u = tid; u <= M; u += blockDim.x) {
    int c = 0;
    for (int v = u + 1; v <= M; ++v) {
      if (t_parent[tb + v] == u && c < kmax) {
        child_tok[(tb + u) * kmax + c] = t_tok[tb + v];
        child_node[(tb + u) * kmax + c] = v;
        ++c;
      }
    }
    n_child[tb + u] = c;
    for (int j = c; j < kmax; ++j) {
      child_tok[(tb + u) * kmax + j] = -1;
      child_node[(tb + u) * kmax + j] = -1;
    }
  }
}

void launch_plan_verify(int B, int M, int kmax, const int* t_tok, const int* t_parent,
                        const int* t_pos, const int* t_pidx, const uint32_t* t_mask,
                        const int* pool_fwd, int pool_n, int n_slots, const RowPlan& rp,
                        int* n_prefix, int* child_tok, int* child_node, int* n_child, int* flags,
                        cudaStream_t st) {
  launch_pdl(plan_verify_kernel, dim3(B), dim3(128), 0, st, M, kmax, t_tok, t_parent, t_pos, t_pidx, t_mask, pool_fwd,
                                        pool_n, n_slots, rp, n_prefix, child_tok, child_node,
                                        n_child, flags);
}

// ----------------------------------------------------------------------------- small copies
__global__ void copy_rows_kernel(int row_bytes, const char* src, size_t src_step, bool src_split,
                                 char* dst, size_t dst_step, bool dst_split) {
  pdl_begin();
  const int b = blockIdx.x;
  const char* sr = src + b * src_step;
  char* dr = dst + b * dst_step;
  if (row_bytes % 16 == 0) {  // rows of d * element-size bytes: 16-byte pieces
    const int n = row_bytes / 16;
    const uint4* s4 = reinterpret_cast<const uint4*>(sr);
    uint4* d4 = reinterpret_cast<uint4*>(dr);
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      d4[i] = s4[i];
      if (dst_split) d4[n + i] = src_split ? s4[n + i] : make_uint4(0u, 0u, 0u, 0u);
    }
    return;
  }
  for (int i = threadIdx.x; i < row_bytes; i += blockDim.x) {
    dr[i] = sr[i];
    if (dst_split) dr[row_bytes + i] = src_split ? sr[row_bytes + i] : 0;
  }
}

void launch_copy_rows(int B, int d, int elem_bytes, const void* src, int src_stride_rows,
                      bool src_split, void* dst, int dst_stride_rows, bool dst_split,
                      cudaStream_t st) {
  const size_t row = (size_t)d * elem_bytes;
  launch_pdl(copy_rows_kernel, dim3(B), dim3(256), 0, st, (int)row, (const char*)src,
                                      row * src_stride_rows * (src_split ? 2 : 1), src_split,
                                      (char*)dst, row * dst_stride_rows * (dst_split ? 2 : 1),
                                      dst_split);
}

__global__ void copy_pool_kernel(int n, PoolDev p, int* tok, int* parent, int* depth, int* fwd,
                                 float* score, float* logq) {
  pdl_begin();
  int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  if (tok) tok[i] = p.tok[i];
  if (parent) parent[i] = p.parent[i];
  if (depth) depth[i] = p.depth[i];
  if (fwd) fwd[i] = p.fwd[i];
  if (score) score[i] = p.score[i];
  if (logq) logq[i] = p.logq[i];
}

void launch_copy_pool(int B, const PoolDev& pool, int* tok, int* parent, int* depth, int* fwd,
                      float* score, float* logq, cudaStream_t st) {
  int n = B * pool.n;
  launch_pdl(copy_pool_kernel, dim3((n + 255) / 256), dim3(256), 0, st, n, pool, tok, parent, depth, fwd, score, logq);
}

}  // namespace e3
