// Host side of the C ABI: argument checks, the workspace arena, and the order
// of kernel launches of one EAGLE-3 round (prefill, draft passes, tree build,
// verification).  Everything runs on the caller's stream with no host
// synchronisation; the only allocation is the arena made at create time.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/eagle3.h"
#include "common.cuh"
#include "gemm_tc.h"
#include "kernels.h"
#include "lowrank.h"

using namespace e3;

namespace {
constexpr int kPrefillChunk = 2048;   // prefill rows per pass through the layer
constexpr int kTargetBlocks = 2 * 148;
// bf16 GEMM inputs of at most this many rows are stored split (hi, lo): the
// MMA then runs 2R columns, which is free while the weights bound the time.
constexpr int kSplitMaxRows = 128;
// largest logits buffer of the deferred bonus draw (see the workspace plan)
constexpr size_t kDeferMaxBytes = (size_t)4 << 30;

int cdiv(int a, int b) { return (a + b - 1) / b; }
size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
}  // namespace

struct eagle3_ctx {
  eagle3_config cfg;
  eagle3_weights w;
  bool bf;
  int esz;
  int M, M1, k, D, pool_n, n_slots, slot_words, tree_words, mask_words;
  int rows_cap, rows_pf, rope_rows, act_rows;
  // arena
  char* arena = nullptr;
  size_t arena_bytes = 0;
  // activations
  float *g, *part, *q, *r, *S, *o_part, *ml_part;
  void *x, *o, *z, *a, *h, *h_root, *h_ver;
  void *tk, *tv, *vk, *vv;
  size_t part_elems, attn_elems;
  float2* rope;
  // plans
  RowPlan rp;
  int *n_prefix, *root_tok, *root_pos;
  // draft head
  HeadParts hp;
  int* top_tok;
  float *top_logq, *top_lse;
  // pool
  PoolDev pool;
  int* frontier;
  uint32_t* slot_mask;
  // two-stage head
  bool lr = false;
  LowRankArgs la{};  // base pointers and sizes; per call: rows, inputs, outputs
  void* lr_t = nullptr;
  int* cand_all = nullptr;  // [B][n_exp][lr_cand] candidates of every expanded node
  int n_exp = 0;
  // verify
  int *child_tok, *child_node, *n_child, *z_arg, *g_arg;
  float *child_z, *vpart, *z_max, *lse, *g_max;
  float* vlogits = nullptr;  // [B*M1][V] target logits of a sampling pass (deferred bonus draw)
  unsigned long long* bonus_best = nullptr;  // [B] packed best (score, token) of the bonus draw
  int n_vparts;
  int* flags;
  // per-request caps and cost-aware rules (eagle3_set_control)
  CtlDev ctl{};
  eagle3_control ctl_host{};
  float *d_pass_us = nullptr, *d_verify_us = nullptr;
  int *d_deff = nullptr, *d_active = nullptr;
  const int* skip = nullptr;  // set while a draft pass t >= 1 is launched: &d_active[t]
  // sampled draft (EAGLE3_SAMPLED_DRAFT): logits [rows][V] and the walk's work rows
  bool sampled = false;
  unsigned long long draft_seed = 0;
  unsigned long long* d_draft_round = nullptr;
  float *lg = nullptr, *pqw = nullptr;
  // tcgen05 GEMM plans
  TcGemm* tc = nullptr;
  // tensor maps of the caller's K/V cache (tensor-core attention), re-encoded
  // when the cache pointers or sizes change
  const void *km_k = nullptr, *km_v = nullptr;
  int km_T = 0, km_rows = 0;
  CUtensorMap km_mk, km_mv;
  // CUDA graph of one step (draft round + verify), replayed by eagle3_graph_launch
  unsigned long long* d_round = nullptr;        // round id read by the captured verify kernels
  const unsigned long long* round_ptr = nullptr; // set while capturing
  cudaGraphExec_t gexec = nullptr;
  int graph_launches = 0;
  // bookkeeping
  cudaStream_t last = nullptr;
  std::string err;
  std::string host_err;  // a launch the host refused inside the current call
  int launches = 0;
  bool have_round = false;
  int last_B = 0;
};

namespace {

bool use_split(const eagle3_ctx* c, int R) { return c->bf && R <= kSplitMaxRows; }

// The control of one call: the context's setting plus the branch cap of this batch size.
CtlDev round_control(const eagle3_ctx* c, int B) {
  CtlDev d = c->ctl;
  d.clip = c->sampled ? 1 : 0;
  d.lmax = c->sampled ? c->top_lse : nullptr;  // written by the sampled head (largest log q)
  if (!d.on) return d;
  const eagle3_control& h = c->ctl_host;
  int kc = c->k;
  if (h.light_batch > 0) kc = std::min(kc, B <= h.light_batch ? h.k_light : h.k_heavy);
  d.k_call = std::max(1, kc);
  return d;
}

// position of x on an ascending grid: index i and weight w of g[i+1] (clamped)
void grid_pos(const int* g, int n, double x, int& i, double& w) {
  if (n <= 1 || x <= g[0]) { i = 0; w = 0.0; return; }
  if (x >= g[n - 1]) { i = n - 2; w = 1.0; return; }
  i = 0;
  while (g[i + 1] < x) ++i;
  w = (x - g[i]) / (double)(g[i + 1] - g[i]);
}

double table_at(const eagle3_latency_table* t, const float* v, int B, int P, int n) {
  int ib, ip, in;
  double wb, wp, wn;
  grid_pos(t->batch, t->n_batch, B, ib, wb);
  grid_pos(t->prefix, t->n_prefix, P, ip, wp);
  grid_pos(t->tokens, t->n_tokens, n, in, wn);
  double acc = 0.0;
  for (int a = 0; a < 2; ++a)
    for (int b = 0; b < 2; ++b)
      for (int e = 0; e < 2; ++e) {
        const int xb = std::min(ib + a, t->n_batch - 1), xp = std::min(ip + b, t->n_prefix - 1);
        const int xn = std::min(in + e, t->n_tokens - 1);
        const double w = (a ? wb : 1.0 - wb) * (b ? wp : 1.0 - wp) * (e ? wn : 1.0 - wn);
        if (w != 0.0) acc += w * v[((size_t)xb * t->n_prefix + xp) * t->n_tokens + xn];
      }
  return acc;
}

eagle3_status fail(eagle3_ctx* c, eagle3_status s, const std::string& msg) {
  if (c) c->err = msg;
  return s;
}

void tc_error(eagle3_ctx* c, const char* what) {
  if (c->host_err.empty()) c->host_err = what;
}

eagle3_status cuda_status(eagle3_ctx* c, const char* where) {
  if (!c->host_err.empty()) {
    std::string m = std::string(where) + ": " + c->host_err;
    c->host_err.clear();
    return fail(c, EAGLE3_ERR_CUDA, m);
  }
  cudaError_t e = cudaPeekAtLastError();
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(c, EAGLE3_ERR_CUDA, std::string(where) + ": " + cudaGetErrorString(e));
  }
  return EAGLE3_OK;
}

// K splits of a GEMM with output width N (the sum over its segments) on R rows.
int splits_for(const eagle3_ctx* c, int R, int N, int K) {
  if (c->bf) return tc_splits(R, cdiv(N, 128), K);
  int tiles = cdiv(N, 64) * cdiv(R, 64);
  int s = std::max(1, kTargetBlocks / std::max(1, tiles));
  s = std::min(s, std::max(1, K / 256));
  return std::min(s, 32);
}

// ---------------------------------------------------------------------------- dtype dispatch
#define DISPATCH(c, FN, ...) \
  do {                        \
    if ((c)->bf)              \
      FN<bf16>(__VA_ARGS__);  \
    else                      \
      FN<float>(__VA_ARGS__); \
  } while (0)

void tc_error(eagle3_ctx* c, const char* what);

// Y[s][r][seg.col0 + n] = X W_seg^T over K, split S ways: tcgen05 for bf16
// storage, the fp32 CUDA-core kernel for fp32 storage.
void gemm(eagle3_ctx* c, const GemmSeg* segs, int nseg, const void* X, int ldx, int K, float* Y,
          int ldy, int R, bool split, int S, size_t split_stride, cudaStream_t st) {
  if (c->bf) {
    if (!tc_gemm(c->tc, segs, nseg, X, ldx, K, Y, ldy, R, split, S, split_stride, c->flags, st,
                 c->skip))
      tc_error(c, "tcgen05 GEMM rejected its arguments");
    c->launches++;
    return;
  }
  for (int i = 0; i < nseg; ++i) {
    launch_gemm_simt<float>(X, ldx, segs[i].W, K, Y, ldy, segs[i].col0, R, segs[i].N, K, S,
                            split_stride, st);
    c->launches++;
  }
}

void gemm1(eagle3_ctx* c, int wid, const void* X, int ldx, const void* W, int N, int K, float* Y,
           int ldy, int R, bool split, int S, size_t split_stride, cudaStream_t st) {
  GemmSeg g{wid, W, N, 0};
  gemm(c, &g, 1, X, ldx, K, Y, ldy, R, split, S, split_stride, st);
}

struct KvTarget {  // where a pass writes K/V
  void *k, *v;
  int slots;  // tree slots per request (0: prefix cache)
};

// fusion + input build + QKV (or KV only) + RoPE + KV write, for rp.kv_* rows.
// hid_base rows for the input come from `g` when fuse_from != NULL.
void kv_rows(eagle3_ctx* c, int R, const void* feats, bool has_q, const float* hid_base,
             const eagle3_kv* kv, KvTarget tgt, bool split, cudaStream_t st) {
  const eagle3_config& f = c->cfg;
  const int d = f.d;
  if (feats) {  // the caller's features are exact storage values: never split
    int S = splits_for(c, R, d, 3 * d);
    gemm1(c, TCW_FC, feats, 3 * d, c->w.w_fc, d, 3 * d, c->part, d, R, false, S, (size_t)R * d, st);
    if (f.variant & EAGLE3_FC_NORM) {
      DISPATCH(c, launch_reduce_norm, R, d, S, f.rms_eps, c->part, c->w.g_fc, c->g, st);
    } else {
      launch_reduce_parts(R, d, S, c->part, c->g, st);
    }
    c->launches++;
    hid_base = c->g;
  }
  DISPATCH(c, launch_build_input, R, d, f.vocab, f.rms_eps, c->rp.kv_tok, hid_base, c->rp.kv_hid,
           c->w.embed, c->w.g_emb, c->w.g_hid, c->x, split, c->flags, st);
  c->launches++;
  const int qd = f.n_q_heads * f.head_dim, kvd = f.n_kv_heads * f.head_dim;
  const int ld = (has_q ? qd : 0) + 2 * kvd;
  int S = splits_for(c, R, ld, 2 * d);
  size_t ss = (size_t)R * ld;
  GemmSeg segs[3];
  int n = 0, col = 0;
  if (has_q) {
    segs[n++] = GemmSeg{TCW_Q, c->w.w_q, qd, 0};
    col = qd;
  }
  segs[n++] = GemmSeg{TCW_K, c->w.w_k, kvd, col};
  segs[n++] = GemmSeg{TCW_V, c->w.w_v, kvd, col + kvd};
  gemm(c, segs, n, c->x, 2 * d, 2 * d, c->part, ld, R, split, S, ss, st);
  QkvEpi p{};
  p.R = R;
  p.S = S;
  p.Hq = f.n_q_heads;
  p.Hkv = f.n_kv_heads;
  p.dh = f.head_dim;
  p.has_q = has_q;
  p.part = c->part;
  p.rope = c->rope;
  p.rope_rows = c->rope_rows;
  p.row_b = c->rp.kv_b;
  p.row_pos = c->rp.kv_pos;
  p.row_dst = c->rp.kv_dst;
  p.q_out = c->q;
  p.cache_k = kv->k;
  p.cache_v = kv->v;
  p.page_table = f.page_size ? kv->page_table : nullptr;
  p.page_size = f.page_size;
  p.max_pages = kv->max_pages;
  p.n_pages = kv->n_pages;
  p.max_prefix = f.max_prefix;
  p.tree_k = tgt.k;
  p.tree_v = tgt.v;
  p.tree_slots = tgt.slots;
  p.flags = c->flags;
  DISPATCH(c, launch_qkv_epilogue, p, st);
  c->launches++;
}

// Prefix key splits of the attention: about 4 blocks per SM in all (the
// tensor-core kernel holds 2-3 per SM), in multiples of 64 keys.  (Fewer,
// longer splits halved the merge but slowed the tensor-core kernel where the
// queries per KV head make it compute-bound, e.g. 240 verify queries.)
void attn_splits(const eagle3_ctx* c, int B, int rows_per_req, int& kps, int& nps) {
  const eagle3_config& f = c->cfg;
  const bool mma = attention_uses_mma(c->esz, f.head_dim, f.page_size);
  int blocks = B * f.n_kv_heads * attention_qgroups(rows_per_req, f.n_q_heads, f.n_kv_heads, mma);
  int maxp = f.max_prefix;
  // the tcgen05 kernel (groups of more than 128 queries) runs one CTA per SM
  // and stages its queries once per block: about two waves, 256+ keys a block
  const bool tc = mma && attention_uses_tc(rows_per_req, f.n_q_heads, f.n_kv_heads);
  const int target = tc ? 2 * 148 : mma ? 4 * 148 : kTargetBlocks;
  nps = std::max(1, std::min(cdiv(target, blocks), cdiv(maxp, tc ? 256 : 64)));
  nps = std::min(nps, 240);  // the merge keeps one weight per split (with the tree splits) in 256
  kps = cdiv(cdiv(maxp, nps), 64) * 64;
  nps = cdiv(maxp, kps);
}

// attention + O + FFN + final norm for rp.t_* rows (rows_per_req per request).
void tail_rows(eagle3_ctx* c, int B, int rows_per_req, const float* hid_base, const eagle3_kv* kv,
               KvTarget tree, void* h_base, bool split, cudaStream_t st) {
  const eagle3_config& f = c->cfg;
  const int d = f.d, R = B * rows_per_req;
  const int qd = f.n_q_heads * f.head_dim;
  AttnArgs a{};
  a.B = B;
  a.rows_per_req = rows_per_req;
  a.Hq = f.n_q_heads;
  a.Hkv = f.n_kv_heads;
  a.dh = f.head_dim;
  a.q = c->q;
  a.q_row = c->rp.t_q;
  a.n_prefix = c->n_prefix;
  a.cache_k = kv->k;
  a.cache_v = kv->v;
  a.page_table = f.page_size ? kv->page_table : nullptr;
  a.page_size = f.page_size;
  a.max_pages = kv->max_pages;
  a.n_pages = kv->n_pages;
  a.max_prefix = f.max_prefix;
  if (attention_uses_mma(c->esz, f.head_dim, f.page_size)) {
    const int rows = attention_box_rows(f.page_size);
    const long long T =
        f.page_size ? (long long)kv->n_pages * f.page_size : (long long)f.max_batch * f.max_prefix;
    if (T <= 0 || T > (long long)INT_MAX - 2 * 64) {
      tc_error(c, "K/V cache rows out of the attention's tensor-map range");
      return;
    }
    if (c->km_k != kv->k || c->km_v != kv->v || c->km_T != (int)T || c->km_rows != rows) {
      c->km_k = c->km_v = nullptr;
      if (!encode_kv_map(&c->km_mk, kv->k, (int)T, f.n_kv_heads, f.head_dim, rows) ||
          !encode_kv_map(&c->km_mv, kv->v, (int)T, f.n_kv_heads, f.head_dim, rows)) {
        tc_error(c, "cuTensorMapEncodeTiled refused the K/V cache");
        return;
      }
      c->km_k = kv->k;
      c->km_v = kv->v;
      c->km_T = (int)T;
      c->km_rows = rows;
    }
    a.tm_rows = rows;
    a.tm_T = (int)T;
    a.tm_k = c->km_mk;
    a.tm_v = c->km_mv;
  }
  a.tree_k = tree.k;
  a.tree_v = tree.v;
  a.tree_slots = tree.slots;
  a.mask = c->rp.t_mask;
  a.mask_words = c->mask_words;
  attn_splits(c, B, rows_per_req, a.keys_per_split, a.n_prefix_splits);
  a.n_tree_splits = cdiv(tree.slots, 64);
  a.o_part = c->o_part;
  a.ml_part = c->ml_part;
  a.out = c->o;
  a.split = split;
  a.flags = c->flags;
  a.skip = c->skip;
  // only the root pass writes prefix rows (its new rows) in the same pass
  a.prefix_stable = tree.slots > 0;
  DISPATCH(c, launch_tree_attention, a, st);
  c->launches += 2;
  // r = hid + W_o o ; z = rms(r)
  int S = splits_for(c, R, d, qd);
  gemm1(c, TCW_O, c->o, qd, c->w.w_o, d, qd, c->part, d, R, split, S, (size_t)R * d, st);
  const bool post = (f.variant & EAGLE3_POST_NORM) != 0;
  DISPATCH(c, launch_o_epilogue, R, d, S, f.rms_eps, c->part, hid_base, c->rp.t_hid, c->w.g_post,
           c->r, c->z, split, post, st);
  c->launches++;
  // a = silu(W_g z) * W_u z  (gate and up in one GEMM: columns [0, F) and [F, 2F))
  const int F = f.ffn;
  int Sf = splits_for(c, R, 2 * F, d);
  GemmSeg gu[2] = {GemmSeg{TCW_GATE, c->w.w_gate, F, 0}, GemmSeg{TCW_UP, c->w.w_up, F, F}};
  gemm(c, gu, 2, c->z, d, d, c->part, 2 * F, R, split, Sf, (size_t)R * 2 * F, st);
  DISPATCH(c, launch_swiglu, R, F, Sf, c->part, c->a, split, st);
  c->launches++;
  // s = r + W_down a ; h = rms(s)
  int Sd = splits_for(c, R, d, F);
  gemm1(c, TCW_DOWN, c->a, F, c->w.w_down, d, F, c->part, d, R, split, Sd, (size_t)R * d, st);
  DISPATCH(c, launch_down_epilogue, R, d, Sd, f.rms_eps, c->part, c->r, c->w.g_final, c->rp.t_sdst,
           c->S, c->rp.t_out, h_base, split, post, st);
  c->launches++;
}

// Two-stage head: t = V_lr h, low-rank sample and threshold, threshold append,
// then per row the sort, exact rescoring, log q over the candidates and top-k.
// slot0 >= 0 exports the candidates of rows b*rpr + j to node slot slot0 + j.
void draft_head_lowrank(eagle3_ctx* c, const void* H, int R, bool split, int* tok, float* logq,
                        float* lse, int slot0, int rpr, cudaStream_t st) {
  const eagle3_config& f = c->cfg;
  const int d = f.d, r = f.lr_rank;
  LowRankArgs la = c->la;
  la.R = R;
  la.H = H;
  la.h_split = split;
  // t only ranks the candidates (their log q comes from the exact head): one bf16
  la.t_split = false;
  la.tok = tok;
  la.logq = logq;
  la.lse = lse;
  la.cand_out = slot0 >= 0 ? c->cand_all : nullptr;
  la.cand_slot0 = slot0;
  la.cand_rpr = rpr;
  const int S = splits_for(c, R, r, d);
  gemm1(c, TCW_LRV, H, d, c->w.lr_v, r, d, c->part, r, R, split, S, (size_t)R * r, st);
  DISPATCH(c, launch_reduce_store, R, r, S, c->part, c->lr_t, la.t_split != 0, st);
  c->launches++;
  for (int mode = 0; mode < 2; ++mode) {
    if (c->bf) {
      if (!tc_lowrank(c->tc, mode, la, c->flags, st)) tc_error(c, "tcgen05 low-rank head rejected its arguments");
    } else {
      launch_lowrank_simt<float>(mode, la, st);
    }
    c->launches++;
    if (mode == 0) {
      launch_lowrank_threshold(la, st);
      c->launches++;
    }
  }
  DISPATCH(c, launch_lowrank_select, la, st);
  c->launches += 2;
}

void draft_head(eagle3_ctx* c, const void* H, int R, bool split, int* tok, float* logq, float* lse,
                cudaStream_t st, int slot0 = -1, int rpr = 1) {
  if (c->lr) {
    draft_head_lowrank(c, H, R, split, tok, logq, lse, slot0, rpr, st);
    return;
  }
  HeadParts hp = c->hp;
  hp.R = R;
  hp.skip = c->skip;
  if (c->bf) {
    if (!tc_lm_head(c->tc, H, R, split, hp, c->flags, st))
      tc_error(c, "tcgen05 LM head rejected its arguments");
  } else {
    launch_lm_head_simt<float>(H, c->w.w_lm, R, c->cfg.vocab, c->cfg.d, hp, st);
  }
  c->launches++;
  launch_topk_merge(hp, tok, logq, lse, 0, st);
  c->launches++;
}

// Sampled draft: the pass's logits by the tensor-core GEMM, then each row's k
// children drawn by Gumbel-top-k (rows b * rpr + j export to node slot slot0 + j).
void sampled_head(eagle3_ctx* c, const void* H, int R, bool split, int slot0, int rpr,
                  cudaStream_t st) {
  const int V = c->cfg.vocab, d = c->cfg.d;
  gemm1(c, TCW_LM, H, d, c->w.w_lm, V, d, c->lg, V, R, split, 1, 0, st);
  SampleArgs sa{};
  sa.V = V;
  sa.k = c->k;
  sa.rows_per_req = rpr;
  sa.slot0 = slot0;
  sa.seed = c->draft_seed;
  sa.round_ptr = c->d_draft_round;
  sa.logits = c->lg;
  sa.tok = c->top_tok;
  sa.logq = c->top_logq;
  sa.lmax = c->top_lse;
  launch_sample_children(sa, R, st);
  c->launches++;
}

bool kv_ok(const eagle3_ctx* c, const eagle3_kv* kv) {
  if (!kv || !kv->k || !kv->v || !kv->seq_lens) return false;
  if (c->cfg.page_size) {
    if (!kv->page_table || kv->max_pages <= 0 || kv->n_pages <= 0) return false;
  }
  return true;
}

bool tree_ok(const eagle3_tree* t) {
  return t && t->tokens && t->parent && t->depth && t->pos && t->pool_index && t->score && t->mask;
}

void* carve(char*& p, size_t bytes) {
  void* r = p;
  p += align_up(bytes, 256);
  return r;
}

}  // namespace

// ============================================================================ C ABI
extern "C" {

eagle3_status eagle3_create(const eagle3_config* cfg, const eagle3_weights* w, eagle3_ctx** out) {
  if (!cfg || !w || !out) return EAGLE3_ERR_INVALID_ARG;
  *out = nullptr;
  const eagle3_config& f = *cfg;
  if (f.d <= 0 || f.d % 8 || f.n_q_heads <= 0 || f.n_kv_heads <= 0 || f.n_q_heads % f.n_kv_heads ||
      f.head_dim <= 0 || f.head_dim % 16 || f.head_dim > 128 || f.ffn <= 0 || f.ffn % 8 ||
      f.vocab <= 0 || f.dtype < 0 || f.dtype > 1 || f.max_batch <= 0 || f.max_prefix <= 0 ||
      f.max_new <= 0 || f.page_size < 0 || !(f.rms_eps >= 0.f) || !(f.rope_theta > 0.f))
    return EAGLE3_ERR_INVALID_ARG;
  if (f.depth < 1 || f.depth > 16 || f.topk < 1 || f.topk > 16 || f.n_verify < 1 || f.n_verify > 128)
    return EAGLE3_ERR_UNSUPPORTED;
  const int pool_n = f.topk + (f.depth - 1) * f.topk * f.topk;
  if (f.n_verify > pool_n) return EAGLE3_ERR_SHAPE;
  if (f.lr_rank < 0 || (f.lr_rank > 0 && (f.lr_cand < f.topk || f.lr_cand > 128 || f.lr_cand > f.vocab ||
                                           f.lr_rank % 8 || f.lr_rank > 4096 || !w->lr_u || !w->lr_v)))
    return EAGLE3_ERR_INVALID_ARG;
  // bf16 streams U [V, r] in 64-column TMA boxes
  if (f.lr_rank > 0 && f.dtype == EAGLE3_BF16 && f.lr_rank % 64) return EAGLE3_ERR_UNSUPPORTED;
  if ((f.variant & ~(EAGLE3_FC_NORM | EAGLE3_POST_NORM | EAGLE3_SAMPLED_DRAFT)) ||
      ((f.variant & EAGLE3_FC_NORM) && !w->g_fc))
    return EAGLE3_ERR_INVALID_ARG;
  if ((f.variant & EAGLE3_SAMPLED_DRAFT) && f.lr_rank > 0) return EAGLE3_ERR_UNSUPPORTED;
  if (!w->w_fc || !w->embed || !w->w_q || !w->w_k || !w->w_v || !w->w_o || !w->w_gate || !w->w_up ||
      !w->w_down || !w->g_emb || !w->g_hid || !w->g_post || !w->g_final || !w->w_lm)
    return EAGLE3_ERR_INVALID_ARG;

  // bf16: the tcgen05 LM head takes at most 256 rows per launch
  if (f.dtype == EAGLE3_BF16 && f.max_batch * f.topk > 256) return EAGLE3_ERR_UNSUPPORTED;
  // Kernels request weight tiles before waiting for the preceding kernel on
  // their stream, so every write of the weights must be complete from here on.
  if (cudaDeviceSynchronize() != cudaSuccess) return EAGLE3_ERR_CUDA;
  eagle3_ctx* c = new eagle3_ctx();
  c->cfg = f;
  c->w = *w;
  c->bf = f.dtype == EAGLE3_BF16;
  c->esz = c->bf ? 2 : 4;
  if (c->bf) {
    char msg[256] = {0};
    c->tc = tc_create(f, *w, msg, sizeof(msg));
    if (!c->tc) {
      delete c;
      return EAGLE3_ERR_UNSUPPORTED;
    }
  }
  c->k = f.topk;
  c->D = f.depth;
  c->M = f.n_verify;
  c->M1 = f.n_verify + 1;
  c->pool_n = pool_n;
  c->n_slots = (f.depth - 1) * f.topk;
  c->slot_words = std::max(1, cdiv(c->n_slots, 32));
  c->tree_words = cdiv(c->M1, 32);
  c->mask_words = std::max(c->slot_words, c->tree_words);
  const int B = f.max_batch, d = f.d, k = f.topk;
  const int qd = f.n_q_heads * f.head_dim, kvd = f.n_kv_heads * f.head_dim;
  c->rows_pf = std::min(kPrefillChunk, std::max(1, B * f.max_prefix));
  c->rows_cap = std::max({c->rows_pf, B * f.max_new, B * k, B * c->M1});
  c->rope_rows = f.max_prefix + f.depth + 1;
  // rows of a GEMM-input activation buffer: split rows take two
  c->act_rows = c->bf ? std::max(c->rows_cap, 2 * std::min(c->rows_cap, kSplitMaxRows)) : c->rows_cap;
  const int sp = c->bf ? 2 : 1;  // row factor of the head inputs, which may be split

  // partial buffer: largest S * R * N over the GEMMs this context runs
  size_t part = 0;
  auto need = [&](int R, int N, int K) {
    part = std::max(part, (size_t)splits_for(c, R, N, K) * R * N);
  };
  // every row count a call can use: prefill chunks / new rows, and B' <= max_batch requests
  for (int R = 1; R <= std::max(c->rows_pf, B * f.max_new); ++R) {
    need(R, d, 3 * d);
    need(R, qd + 2 * kvd, 2 * d);
    need(R, 2 * kvd, 2 * d);
  }
  for (int b = 1; b <= B; ++b)
    for (int R : {b, b * k, b * c->M}) {
      need(R, qd + 2 * kvd, 2 * d);
      need(R, d, qd);
      need(R, 2 * f.ffn, d);
      need(R, d, f.ffn);
      if (f.lr_rank) need(R, f.lr_rank, d);
    }
  c->part_elems = part;
  size_t attn = 0;
  {
    struct P { int rpr, slots; };
    for (int b = 1; b <= B; ++b)
      for (P p : {P{1, 0}, P{k, c->n_slots}, P{c->M, c->M1}}) {
        int kps, nps;
        attn_splits(c, b, p.rpr, kps, nps);
        attn = std::max(attn, (size_t)(nps + cdiv(p.slots, 64)) * b * p.rpr * qd);
      }
  }
  c->attn_elems = attn;
  const int lm_parts = c->bf ? tc_head_parts(f.vocab) : lm_head_simt_parts(f.vocab);
  c->n_vparts = c->bf ? tc_head_parts(f.vocab) : verify_head_simt_parts(f.vocab);
  const int Rlm = B * k, Rv = B * c->M1;
  const int n_state = B * (1 + c->n_slots);

  // sizes
  std::vector<std::pair<void**, size_t>> plan;
  auto add = [&](void** p, size_t bytes) { plan.emplace_back(p, bytes); };
  add((void**)&c->g, (size_t)std::max(c->rows_pf, B * f.max_new) * d * 4);
  add(&c->x, (size_t)c->act_rows * 2 * d * c->esz);
  add((void**)&c->part, c->part_elems * 4);
  add((void**)&c->q, (size_t)c->rows_cap * qd * 4);
  add(&c->tk, (size_t)B * std::max(1, c->n_slots) * kvd * 4);  // tree K/V scratch: fp32
  add(&c->tv, (size_t)B * std::max(1, c->n_slots) * kvd * 4);
  add(&c->vk, (size_t)B * c->M1 * kvd * 4);
  add(&c->vv, (size_t)B * c->M1 * kvd * 4);
  add((void**)&c->o_part, c->attn_elems * 4);
  add((void**)&c->ml_part, c->attn_elems / f.head_dim * 2 * 4);
  add(&c->o, (size_t)c->act_rows * qd * c->esz);
  add((void**)&c->r, (size_t)c->rows_cap * d * 4);
  add(&c->z, (size_t)c->act_rows * d * c->esz);
  add(&c->a, (size_t)c->act_rows * f.ffn * c->esz);
  add((void**)&c->S, (size_t)n_state * d * 4);
  add(&c->h, (size_t)sp * Rlm * d * c->esz);
  add(&c->h_root, (size_t)sp * B * d * c->esz);
  add(&c->h_ver, (size_t)sp * Rv * d * c->esz);
  add((void**)&c->rope, (size_t)c->rope_rows * (f.head_dim / 2) * sizeof(float2));
  int* rp_int[10] = {};
  for (int i = 0; i < 10; ++i) add((void**)&rp_int[i], (size_t)c->rows_cap * 4);
  add((void**)&c->rp.t_mask, (size_t)c->rows_cap * c->mask_words * 4);
  add((void**)&c->n_prefix, (size_t)B * 4);
  add((void**)&c->root_tok, (size_t)B * 4);
  add((void**)&c->root_pos, (size_t)B * 4);
  add((void**)&c->hp.ms, (size_t)lm_parts * Rlm * 2 * 4);
  add((void**)&c->hp.val, (size_t)lm_parts * Rlm * k * 4);
  add((void**)&c->hp.idx, (size_t)lm_parts * Rlm * k * 4);
  add((void**)&c->top_tok, (size_t)Rlm * k * 4);
  add((void**)&c->top_logq, (size_t)Rlm * k * 4);
  add((void**)&c->top_lse, (size_t)Rlm * 4);
  add((void**)&c->pool.tok, (size_t)B * pool_n * 4);
  add((void**)&c->pool.parent, (size_t)B * pool_n * 4);
  add((void**)&c->pool.depth, (size_t)B * pool_n * 4);
  add((void**)&c->pool.fwd, (size_t)B * pool_n * 4);
  add((void**)&c->pool.score, (size_t)B * pool_n * 4);
  add((void**)&c->pool.logq, (size_t)B * pool_n * 4);
  add((void**)&c->frontier, (size_t)B * k * 4);
  add((void**)&c->slot_mask, (size_t)B * std::max(1, c->n_slots) * c->slot_words * 4);
  add((void**)&c->child_tok, (size_t)Rv * k * 4);
  add((void**)&c->child_node, (size_t)Rv * k * 4);
  add((void**)&c->n_child, (size_t)Rv * 4);
  add((void**)&c->child_z, (size_t)Rv * k * 4);
  add((void**)&c->vpart, (size_t)c->n_vparts * Rv * 6 * 4);
  add((void**)&c->z_max, (size_t)Rv * 4);
  add((void**)&c->z_arg, (size_t)Rv * 4);
  add((void**)&c->lse, (size_t)Rv * 4);
  add((void**)&c->g_arg, (size_t)Rv * 4);
  add((void**)&c->g_max, (size_t)Rv * 4);
  // The tensor-core verify head stores the target logits of a sampling pass
  // and leaves the Gumbel draw to the one node where each walk stops; past
  // kDeferMaxBytes of logits it draws in its epilogue instead.
  if (c->bf && (size_t)Rv * f.vocab * 4 <= kDeferMaxBytes) {
    add((void**)&c->vlogits, (size_t)Rv * f.vocab * 4);
    add((void**)&c->bonus_best, (size_t)B * 8);
  }
  c->lr = f.lr_rank > 0;
  c->n_exp = 1 + (f.depth - 1) * k;
  const int lr_groups = c->lr ? (c->bf ? lowrank_tc_groups(f.vocab) : lowrank_simt_groups(f.vocab)) : 0;
  if (c->lr) {
    add(&c->lr_t, (size_t)sp * Rlm * f.lr_rank * c->esz);
    add((void**)&c->la.gmax, (size_t)lr_groups * Rlm * 4);
    add((void**)&c->la.thr, (size_t)Rlm * 4);
    add((void**)&c->la.cnt, (size_t)Rlm * 4);
    add((void**)&c->la.cval, (size_t)Rlm * kLrCap * 4);
    add((void**)&c->la.ctok, (size_t)Rlm * kLrCap * 4);
    add((void**)&c->cand_all, (size_t)B * c->n_exp * f.lr_cand * 4);
    add((void**)&c->la.sel_tok, (size_t)Rlm * f.lr_cand * 4);
    add((void**)&c->la.sel_z, (size_t)Rlm * f.lr_cand * 4);
    add((void**)&c->la.sel_done, (size_t)Rlm * 4);
  }
  add((void**)&c->d_round, 8);
  add((void**)&c->flags, 64);
  add((void**)&c->d_pass_us, (size_t)f.depth * 4);
  add((void**)&c->d_verify_us, (size_t)(f.n_verify + 1) * 4);
  add((void**)&c->d_deff, (size_t)B * 4);
  add((void**)&c->d_active, (size_t)(f.depth + 1) * 4);
  c->sampled = (f.variant & EAGLE3_SAMPLED_DRAFT) != 0;
  if (c->sampled) {
    const size_t rows = std::max((size_t)B * k, (size_t)2 * B * (f.n_verify + 1));
    add((void**)&c->lg, rows * f.vocab * 4);
    add((void**)&c->pqw, (size_t)2 * B * f.vocab * 4);
    add((void**)&c->d_draft_round, 8);
  }
  size_t total = 0;
  for (auto& p : plan) total += align_up(p.second, 256);
  if (cudaMalloc(&c->arena, total) != cudaSuccess) {
    cudaGetLastError();
    tc_destroy(c->tc);
    delete c;
    return EAGLE3_ERR_OOM;
  }
  c->arena_bytes = total;
  char* p = c->arena;
  for (auto& e : plan) *e.first = carve(p, e.second);
  c->rp.kv_b = rp_int[0];
  c->rp.kv_tok = rp_int[1];
  c->rp.kv_hid = rp_int[2];
  c->rp.kv_pos = rp_int[3];
  c->rp.kv_dst = rp_int[4];
  c->rp.t_q = rp_int[5];
  c->rp.t_b = rp_int[6];
  c->rp.t_hid = rp_int[7];
  c->rp.t_sdst = rp_int[8];
  c->rp.t_out = rp_int[9];
  c->rp.mask_words = c->mask_words;
  c->hp.n_parts = lm_parts;
  c->hp.k = k;
  c->pool.n = pool_n;
  if (c->lr) {
    c->la.V = f.vocab;
    c->la.d = d;
    c->la.r = f.lr_rank;
    c->la.C = f.lr_cand;
    c->la.k = k;
    c->la.n_groups = lr_groups;
    c->la.t = c->lr_t;
    c->la.U = w->lr_u;
    c->la.W = w->w_lm;
    c->la.cand_n_exp = c->n_exp;
    c->la.flags = c->flags;
  }

  // RoPE table, rotate-half pairs: angle = pos * theta^(-2j/dh) in double
  {
    const int half = f.head_dim / 2;
    std::vector<float2> tab((size_t)c->rope_rows * half);
    for (int pos = 0; pos < c->rope_rows; ++pos)
      for (int j = 0; j < half; ++j) {
        double inv = std::pow((double)f.rope_theta, -2.0 * j / f.head_dim);
        double ang = pos * inv;
        tab[(size_t)pos * half + j] = make_float2((float)std::cos(ang), (float)std::sin(ang));
      }
    if (cudaMemset(c->arena, 0, total) != cudaSuccess ||
        cudaMemcpy(c->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice) != cudaSuccess) {
      cudaGetLastError();
      cudaFree(c->arena);
      tc_destroy(c->tc);
      delete c;
      return EAGLE3_ERR_CUDA;
    }
  }
  *out = c;
  return EAGLE3_OK;
}

void eagle3_destroy(eagle3_ctx* c) {
  if (!c) return;
  if (c->gexec) cudaGraphExecDestroy(c->gexec);
  if (c->tc) tc_destroy(c->tc);
  if (c->arena) cudaFree(c->arena);
  delete c;
}

eagle3_status eagle3_prefill(eagle3_ctx* c, int B, int total_rows, const int* cu_rows,
                             const void* feats, const int* tokens, const eagle3_kv* kv,
                             eagle3_stream stream) {
  if (!c) return EAGLE3_ERR_INVALID_ARG;
  c->err.clear();
  c->launches = 0;
  if (B < 1 || B > c->cfg.max_batch) return fail(c, EAGLE3_ERR_SHAPE, "B out of range");
  if (total_rows < 0) return fail(c, EAGLE3_ERR_SHAPE, "total_rows < 0");
  if (total_rows > 0 && (!cu_rows || !feats || !tokens))
    return fail(c, EAGLE3_ERR_INVALID_ARG, "null input");
  if (!kv_ok(c, kv)) return fail(c, EAGLE3_ERR_INVALID_ARG, "bad kv descriptor");
  cudaStream_t st = (cudaStream_t)stream;
  c->last = st;
  const int d = c->cfg.d;
  for (int r0 = 0; r0 < total_rows; r0 += c->rows_pf) {
    int R = std::min(c->rows_pf, total_rows - r0);
    launch_plan_prefill(R, r0, B, cu_rows, tokens, kv->seq_lens, c->rp, st);
    c->launches++;
    const char* f = (const char*)feats + (size_t)r0 * 3 * d * c->esz;
    kv_rows(c, R, f, false, nullptr, kv, KvTarget{nullptr, nullptr, 0}, use_split(c, R), st);
  }
  return cuda_status(c, "prefill");
}

}  // extern "C"

namespace {
// One draft round; the new rows are n_new per request (cu_new NULL) or ragged.
eagle3_status draft_round_impl(eagle3_ctx* c, int B, int n_new, const int* cu_new, int total_new,
                               const void* feats_new, const int* tokens_new, const eagle3_kv* kv,
                               eagle3_tree* out, eagle3_pool* pool_out, eagle3_stream stream) {
  cudaStream_t st = (cudaStream_t)stream;
  c->last = st;
  const int k = c->k, D = c->D;
  // pass 0: the new rows' K/V, then the root row through the whole layer
  launch_plan_root(B, n_new, cu_new, total_new, c->cfg.max_new, tokens_new, kv->seq_lens,
                   c->n_slots, c->rp, c->root_tok, c->root_pos, c->n_prefix, c->flags, st);
  c->launches++;
  const bool sp0 = use_split(c, B), spk = use_split(c, B * k);
  kv_rows(c, total_new, feats_new, true, nullptr, kv, KvTarget{nullptr, nullptr, 0},
          use_split(c, total_new), st);
  tail_rows(c, B, 1, c->g, kv, KvTarget{nullptr, nullptr, 0}, c->h_root, sp0, st);
  if (c->sampled)
    sampled_head(c, c->h_root, B, sp0, 0, 1, st);
  else
    draft_head(c, c->h_root, B, sp0, c->top_tok, c->top_logq, c->top_lse, st, 0, 1);
  CtlDev ctl = round_control(c, B);
  if (ctl.on) cudaMemsetAsync(c->d_active, 0, (size_t)(D + 1) * 4, st);
  launch_expand(ctl, B, 0, k, D, c->top_tok, c->top_logq, c->pool, c->frontier, c->slot_mask,
                c->slot_words, c->root_pos, c->n_slots, c->rp, st);
  c->launches++;
  // passes 1..D-1: the frontier of each depth with the parent's state as hid; with
  // control on, the heavy kernels of a pass that no request takes part in return at once
  KvTarget tree{c->tk, c->tv, c->n_slots};
  for (int t = 1; t < D; ++t) {
    c->skip = ctl.on ? c->d_active + t : nullptr;
    kv_rows(c, B * k, nullptr, true, c->S, kv, tree, spk, st);
    tail_rows(c, B, k, c->S, kv, tree, c->h, spk, st);
    if (c->sampled)
      sampled_head(c, c->h, B * k, spk, 1 + (t - 1) * k, k, st);
    else
      draft_head(c, c->h, B * k, spk, c->top_tok, c->top_logq, c->top_lse, st, 1 + (t - 1) * k, k);
    launch_expand(ctl, B, t, k, D, c->top_tok, c->top_logq, c->pool, c->frontier, c->slot_mask,
                  c->slot_words, c->root_pos, c->n_slots, c->rp, st);
    c->launches++;
  }
  c->skip = nullptr;
  launch_build_tree(ctl, B, c->pool_n, c->M, c->pool.tok, c->pool.parent, c->pool.score, c->pool.depth,
                    c->root_tok, c->root_pos, out->tokens, out->parent, out->depth, out->pos,
                    out->pool_index, out->score, out->mask, c->flags, st);
  c->launches++;
  if (pool_out) {
    launch_copy_pool(B, c->pool, pool_out->tok, pool_out->parent, pool_out->depth, pool_out->fwd,
                     pool_out->score, pool_out->logq, st);
    c->launches++;
    if (c->lr && pool_out->cand)
      cudaMemcpyAsync(pool_out->cand, c->cand_all, (size_t)B * c->n_exp * c->cfg.lr_cand * 4,
                      cudaMemcpyDeviceToDevice, st);
  }
  eagle3_status s = cuda_status(c, "draft_round");
  if (s == EAGLE3_OK) {
    c->have_round = true;
    c->last_B = B;
  }
  return s;
}
}  // namespace

extern "C" {

eagle3_status eagle3_draft_round(eagle3_ctx* c, int B, int n_new, const void* feats_new,
                                 const int* tokens_new, const eagle3_kv* kv, eagle3_tree* out,
                                 eagle3_pool* pool_out, eagle3_stream stream) {
  if (!c) return EAGLE3_ERR_INVALID_ARG;
  c->err.clear();
  c->launches = 0;
  if (B < 1 || B > c->cfg.max_batch) return fail(c, EAGLE3_ERR_SHAPE, "B out of range");
  if (n_new < 1 || n_new > c->cfg.max_new) return fail(c, EAGLE3_ERR_SHAPE, "n_new out of range");
  if (!feats_new || !tokens_new) return fail(c, EAGLE3_ERR_INVALID_ARG, "null input");
  if (!kv_ok(c, kv)) return fail(c, EAGLE3_ERR_INVALID_ARG, "bad kv descriptor");
  if (!tree_ok(out)) return fail(c, EAGLE3_ERR_INVALID_ARG, "bad tree output");
  return draft_round_impl(c, B, n_new, nullptr, B * n_new, feats_new, tokens_new, kv, out, pool_out,
                          stream);
}

eagle3_status eagle3_draft_round_ragged(eagle3_ctx* c, int B, int total_new, const int* cu_new,
                                        const void* feats_new, const int* tokens_new,
                                        const eagle3_kv* kv, eagle3_tree* out, eagle3_pool* pool_out,
                                        eagle3_stream stream) {
  if (!c) return EAGLE3_ERR_INVALID_ARG;
  c->err.clear();
  c->launches = 0;
  if (B < 1 || B > c->cfg.max_batch) return fail(c, EAGLE3_ERR_SHAPE, "B out of range");
  if (total_new < B || total_new > B * c->cfg.max_new)
    return fail(c, EAGLE3_ERR_SHAPE, "total_new must be in [B, B * max_new]");
  if (!cu_new || !feats_new || !tokens_new) return fail(c, EAGLE3_ERR_INVALID_ARG, "null input");
  if (!kv_ok(c, kv)) return fail(c, EAGLE3_ERR_INVALID_ARG, "bad kv descriptor");
  if (!tree_ok(out)) return fail(c, EAGLE3_ERR_INVALID_ARG, "bad tree output");
  return draft_round_impl(c, B, 0, cu_new, total_new, feats_new, tokens_new, kv, out, pool_out,
                          stream);
}

eagle3_status eagle3_next_rows(eagle3_ctx* c, int B, const int* accept_len, const int* out_tokens,
                               int* cu_new, int* tokens_new, eagle3_stream stream) {
  if (!c) return EAGLE3_ERR_INVALID_ARG;
  c->err.clear();
  c->launches = 0;
  if (B < 1 || B > c->cfg.max_batch || B > 1024) return fail(c, EAGLE3_ERR_SHAPE, "B out of range");
  if (!accept_len || !out_tokens || !cu_new || !tokens_new)
    return fail(c, EAGLE3_ERR_INVALID_ARG, "null pointer");
  cudaStream_t st = (cudaStream_t)stream;
  c->last = st;
  launch_next_rows(B, c->D, accept_len, out_tokens, cu_new, tokens_new, c->flags, st);
  c->launches++;
  return cuda_status(c, "next_rows");
}

eagle3_status eagle3_build_tree(eagle3_ctx* c, int B, int pool_n, const int* pool_tok,
                                const int* pool_parent, const float* pool_score,
                                const int* pool_depth, const int* root_tok, const int* root_pos,
                                eagle3_tree* out, eagle3_stream stream) {
  if (!c) return EAGLE3_ERR_INVALID_ARG;
  c->err.clear();
  c->launches = 0;
  if (B < 1 || B > c->cfg.max_batch) return fail(c, EAGLE3_ERR_SHAPE, "B out of range");
  if (pool_n < c->M || pool_n > 4096) return fail(c, EAGLE3_ERR_SHAPE, "pool_n must be in [M, 4096]");
  if (!pool_tok || !pool_parent || !pool_score || !pool_depth || !root_tok || !root_pos)
    return fail(c, EAGLE3_ERR_INVALID_ARG, "null input");
  if (!tree_ok(out)) return fail(c, EAGLE3_ERR_INVALID_ARG, "bad tree output");
  cudaStream_t st = (cudaStream_t)stream;
  c->last = st;
  launch_build_tree(round_control(c, B), B, pool_n, c->M, pool_tok, pool_parent, pool_score,
                    pool_depth, root_tok,
                    root_pos, out->tokens, out->parent, out->depth, out->pos, out->pool_index,
                    out->score, out->mask, c->flags, st);
  c->launches++;
  return cuda_status(c, "build_tree");
}

eagle3_status eagle3_verify(eagle3_ctx* c, int B, const eagle3_tree* tree, const eagle3_kv* kv,
                            int mode, float temperature, unsigned long long seed,
                            unsigned long long round_id, int* accept_len, int* path,
                            int* out_tokens, eagle3_verify_stats* stats, eagle3_stream stream) {
  if (!c) return EAGLE3_ERR_INVALID_ARG;
  c->err.clear();
  c->launches = 0;
  if (!c->have_round) return fail(c, EAGLE3_ERR_STATE, "verify needs a draft round on this context");
  if (B != c->last_B) return fail(c, EAGLE3_ERR_SHAPE, "B differs from the last draft round");
  if (mode < 0 || mode > 2) return fail(c, EAGLE3_ERR_INVALID_ARG, "mode must be 0, 1 or 2");
  if (mode == 2 && !c->sampled)
    return fail(c, EAGLE3_ERR_INVALID_ARG, "mode 2 needs the sampled-draft variant");
  if (mode >= 1 && !(temperature > 0.f)) return fail(c, EAGLE3_ERR_INVALID_ARG, "temperature must be > 0");
  if (!c->w.w_target) return fail(c, EAGLE3_ERR_INVALID_ARG, "no target head in the weights");
  if (!tree_ok((eagle3_tree*)tree) || !accept_len || !path || !out_tokens)
    return fail(c, EAGLE3_ERR_INVALID_ARG, "null output");
  if (!kv_ok(c, kv)) return fail(c, EAGLE3_ERR_INVALID_ARG, "bad kv descriptor");
  cudaStream_t st = (cudaStream_t)stream;
  c->last = st;
  const eagle3_config& f = c->cfg;
  const int M = c->M, M1 = c->M1, k = c->k, d = f.d;
  launch_plan_verify(B, M, k, tree->tokens, tree->parent, tree->pos, tree->pool_index, tree->mask,
                     c->pool.fwd, c->pool_n, c->n_slots, c->rp, c->n_prefix, c->child_tok,
                     c->child_node, c->n_child, c->flags, st);
  c->launches++;
  // one layout for the whole verify pass, chosen by the head's row count
  const bool spv = use_split(c, B * M1);
  launch_copy_rows(B, d, c->esz, c->h_root, 1, use_split(c, B), c->h_ver, M1, spv, st);
  c->launches++;
  KvTarget vt{c->vk, c->vv, M1};
  kv_rows(c, B * M, nullptr, true, c->S, kv, vt, spv, st);
  tail_rows(c, B, M, c->S, kv, vt, c->h_ver, spv, st);
  VerifyHeadArgs va{};
  va.R = B * M1;
  va.V = f.vocab;
  va.d = d;
  va.M1 = M1;
  va.kmax = k;
  va.sampling = mode == 1;
  va.inv_t = mode >= 1 ? 1.f / temperature : 1.f;
  va.seed = seed;
  va.round_id = round_id;
  va.round_ptr = c->round_ptr;
  va.child_tok = c->child_tok;
  va.child_z = c->child_z;
  va.n_parts = c->n_vparts;
  va.part = c->vpart;
  // per-node Gumbel-argmax asked for: draw it at every node, in the head
  va.logits = (mode == 1 && c->vlogits && !(stats && stats->g_argmax)) ? c->vlogits : nullptr;
  if (c->bf) {
    if (!tc_verify_head(c->tc, c->h_ver, spv, va, c->flags, st))
      tc_error(c, "tcgen05 verify head rejected its arguments");
  } else {
    launch_verify_head_simt<float>(c->h_ver, c->w.w_target, va, st);
  }
  c->launches++;
  launch_verify_merge(va, c->z_max, c->z_arg, c->lse, c->g_arg, c->g_max, st);
  c->launches++;
  if (mode == 2) {  // q-ratio walk over the draft and target logits of the kept nodes
    const int V = f.vocab;
    float* ell = c->lg;
    float* zl = c->lg + (size_t)B * M1 * V;
    gemm1(c, TCW_LM, c->h_ver, d, c->w.w_lm, V, d, ell, V, B * M1, spv, 1, 0, st);
    gemm1(c, TCW_T, c->h_ver, d, c->w.w_target, V, d, zl, V, B * M1, spv, 1, 0, st);
    QratioArgs qa{};
    qa.B = B;
    qa.M1 = M1;
    qa.kmax = k;
    qa.D = c->D;
    qa.V = V;
    qa.inv_t = 1.f / temperature;
    qa.seed = seed;
    qa.round_id = round_id;
    qa.round_ptr = c->round_ptr;
    qa.z = zl;
    qa.ell = ell;
    qa.pw = c->pqw;
    qa.qw = c->pqw + (size_t)B * V;
    qa.t_tok = tree->tokens;
    qa.pidx = tree->pool_index;
    qa.child_node = c->child_node;
    qa.n_child = c->n_child;
    qa.accept_len = accept_len;
    qa.path = path;
    qa.out_tokens = out_tokens;
    launch_qratio_walk(qa, st);
    c->launches++;
  } else {
  WalkArgs wa{};
  wa.B = B;
  wa.M1 = M1;
  wa.kmax = k;
  wa.D = c->D;
  wa.sampling = mode == 1;
  wa.inv_t = va.inv_t;
  wa.seed = seed;
  wa.round_id = round_id;
  wa.round_ptr = c->round_ptr;
  wa.t_tok = tree->tokens;
  wa.child_node = c->child_node;
  wa.n_child = c->n_child;
  wa.child_z = c->child_z;
  wa.lse = c->lse;
  wa.z_arg = c->z_arg;
  wa.g_arg = c->g_arg;
  wa.accept_len = accept_len;
  wa.path = path;
  wa.out_tokens = out_tokens;
  wa.bonus_best = va.logits ? c->bonus_best : nullptr;
  launch_walk(wa, st);
  c->launches++;
  if (va.logits) {
    BonusArgs ba{};
    ba.B = B;
    ba.M1 = M1;
    ba.kmax = k;
    ba.D = c->D;
    ba.V = f.vocab;
    ba.inv_t = va.inv_t;
    ba.seed = seed;
    ba.round_id = round_id;
    ba.round_ptr = c->round_ptr;
    ba.logits = va.logits;
    ba.child_tok = c->child_tok;
    ba.accept_len = accept_len;
    ba.path = path;
    ba.out_tokens = out_tokens;
    ba.g_arg = c->g_arg;
    ba.best = c->bonus_best;
    launch_bonus_gumbel(ba, st);
    c->launches += 2;
  }
  }
  if (stats) {
    size_t n = (size_t)B * M1;
    if (stats->z_max) cudaMemcpyAsync(stats->z_max, c->z_max, n * 4, cudaMemcpyDeviceToDevice, st);
    if (stats->lse) cudaMemcpyAsync(stats->lse, c->lse, n * 4, cudaMemcpyDeviceToDevice, st);
    if (stats->z_argmax) cudaMemcpyAsync(stats->z_argmax, c->z_arg, n * 4, cudaMemcpyDeviceToDevice, st);
    if (stats->g_argmax) cudaMemcpyAsync(stats->g_argmax, c->g_arg, n * 4, cudaMemcpyDeviceToDevice, st);
  }
  return cuda_status(c, "verify");
}

eagle3_status eagle3_verify_logits(eagle3_ctx* c, int B, const eagle3_tree* tree, const void* logits,
                                   int logits_dtype, long long ld, int mode, float temperature,
                                   unsigned long long seed, unsigned long long round_id,
                                   int* accept_len, int* path, int* out_tokens,
                                   eagle3_verify_stats* stats, eagle3_stream stream) {
  if (!c) return EAGLE3_ERR_INVALID_ARG;
  c->err.clear();
  c->launches = 0;
  const eagle3_config& f = c->cfg;
  if (B < 1 || B > f.max_batch) return fail(c, EAGLE3_ERR_SHAPE, "B out of range");
  if (mode == 2) return fail(c, EAGLE3_ERR_UNSUPPORTED, "q-ratio verification needs the draft logits");
  if (mode < 0 || mode > 1) return fail(c, EAGLE3_ERR_INVALID_ARG, "mode must be 0 or 1");
  if (mode == 1 && !(temperature > 0.f)) return fail(c, EAGLE3_ERR_INVALID_ARG, "temperature must be > 0");
  if (logits_dtype != EAGLE3_FP32 && logits_dtype != EAGLE3_BF16)
    return fail(c, EAGLE3_ERR_INVALID_ARG, "logits_dtype must be EAGLE3_FP32 or EAGLE3_BF16");
  if (!logits || !tree_ok((eagle3_tree*)tree) || !accept_len || !path || !out_tokens)
    return fail(c, EAGLE3_ERR_INVALID_ARG, "null pointer");
  const size_t esz = logits_dtype == EAGLE3_BF16 ? 2 : 4;
  if (ld < f.vocab) return fail(c, EAGLE3_ERR_SHAPE, "ld must be at least the vocabulary size");
  if (((uintptr_t)logits & 15) || ((size_t)ld * esz) % 16)
    return fail(c, EAGLE3_ERR_INVALID_ARG, "logits rows must start on 16-byte boundaries");
  cudaStream_t st = (cudaStream_t)stream;
  c->last = st;
  const int M1 = c->M1;
  LogitsVerifyArgs la{};
  la.B = B;
  la.M1 = M1;
  la.kmax = c->k;
  la.V = f.vocab;
  la.R = B * M1;
  la.ld = ld;
  la.logits = logits;
  la.t_tok = tree->tokens;
  la.t_parent = tree->parent;
  la.sampling = mode == 1;
  la.inv_t = mode == 1 ? 1.f / temperature : 1.f;
  la.seed = seed;
  la.round_id = round_id;
  la.round_ptr = c->round_ptr;
  la.child_tok = c->child_tok;
  la.child_node = c->child_node;
  la.n_child = c->n_child;
  la.child_z = c->child_z;
  la.n_chunks = logits_verify_chunks(la.R, f.vocab, c->n_vparts);
  la.part = c->vpart;
  la.flags = c->flags;
  launch_logits_verify(la, logits_dtype == EAGLE3_BF16, st);
  c->launches += 2;
  VerifyHeadArgs va{};
  va.R = la.R;
  va.n_parts = la.n_chunks;
  va.part = c->vpart;
  launch_verify_merge(va, c->z_max, c->z_arg, c->lse, c->g_arg, c->g_max, st);
  c->launches++;
  WalkArgs wa{};
  wa.B = B;
  wa.M1 = M1;
  wa.kmax = c->k;
  wa.D = c->D;
  wa.sampling = mode == 1;
  wa.inv_t = la.inv_t;
  wa.seed = seed;
  wa.round_id = round_id;
  wa.round_ptr = c->round_ptr;
  wa.t_tok = tree->tokens;
  wa.child_node = c->child_node;
  wa.n_child = c->n_child;
  wa.child_z = c->child_z;
  wa.lse = c->lse;
  wa.z_arg = c->z_arg;
  wa.g_arg = c->g_arg;
  wa.accept_len = accept_len;
  wa.path = path;
  wa.out_tokens = out_tokens;
  launch_walk(wa, st);
  c->launches++;
  if (stats) {
    const size_t n = (size_t)B * M1;
    if (stats->z_max) cudaMemcpyAsync(stats->z_max, c->z_max, n * 4, cudaMemcpyDeviceToDevice, st);
    if (stats->lse) cudaMemcpyAsync(stats->lse, c->lse, n * 4, cudaMemcpyDeviceToDevice, st);
    if (stats->z_argmax) cudaMemcpyAsync(stats->z_argmax, c->z_arg, n * 4, cudaMemcpyDeviceToDevice, st);
    if (stats->g_argmax) cudaMemcpyAsync(stats->g_argmax, c->g_arg, n * 4, cudaMemcpyDeviceToDevice, st);
  }
  return cuda_status(c, "verify_logits");
}

eagle3_status eagle3_graph_capture(eagle3_ctx* c, int B, int n_new, const void* feats_new,
                                   const int* tokens_new, const eagle3_kv* kv, eagle3_tree* out,
                                   int with_verify, int mode, float temperature,
                                   unsigned long long seed, int* accept_len, int* path,
                                   int* out_tokens, eagle3_stream stream) {
  if (!c) return EAGLE3_ERR_INVALID_ARG;
  if (!c->have_round)
    return fail(c, EAGLE3_ERR_STATE, "run one draft round and verify eagerly before capturing");
  if (!stream) return fail(c, EAGLE3_ERR_INVALID_ARG, "the legacy default stream cannot be captured");
  cudaStream_t st = (cudaStream_t)stream;
  if (c->gexec) {
    cudaGraphExecDestroy(c->gexec);
    c->gexec = nullptr;
  }
  if (cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaGetLastError();
    return fail(c, EAGLE3_ERR_CUDA, "cudaStreamBeginCapture failed");
  }
  c->round_ptr = c->d_round;
  eagle3_status s = eagle3_draft_round(c, B, n_new, feats_new, tokens_new, kv, out, nullptr, stream);
  const int n1 = c->launches;
  int n2 = 0;
  if (s == EAGLE3_OK && with_verify) {
    s = eagle3_verify(c, B, out, kv, mode, temperature, seed, 0, accept_len, path, out_tokens,
                      nullptr, stream);
    n2 = c->launches;
  }
  const std::string why = c->err;
  c->round_ptr = nullptr;
  cudaGraph_t g = nullptr;
  cudaError_t e = cudaStreamEndCapture(st, &g);
  if (s != EAGLE3_OK || e != cudaSuccess || !g) {
    if (g) cudaGraphDestroy(g);
    cudaGetLastError();
    return fail(c, s != EAGLE3_OK ? s : EAGLE3_ERR_CUDA,
                s != EAGLE3_OK ? "capture: " + why : "cudaStreamEndCapture failed");
  }
  e = cudaGraphInstantiate(&c->gexec, g, 0);
  cudaGraphDestroy(g);
  if (e != cudaSuccess) {
    cudaGetLastError();
    c->gexec = nullptr;
    return fail(c, EAGLE3_ERR_CUDA, std::string("cudaGraphInstantiate: ") + cudaGetErrorString(e));
  }
  c->graph_launches = n1 + n2;
  c->launches = 0;
  return EAGLE3_OK;
}

eagle3_status eagle3_graph_launch(eagle3_ctx* c, unsigned long long round_id, eagle3_stream stream) {
  if (!c) return EAGLE3_ERR_INVALID_ARG;
  c->err.clear();
  c->launches = 0;
  if (!c->gexec) return fail(c, EAGLE3_ERR_STATE, "no captured graph on this context");
  cudaStream_t st = (cudaStream_t)stream;
  c->last = st;
  launch_set_u64(c->d_round, round_id, st);
  if (c->sampled) launch_set_u64(c->d_draft_round, round_id, st);
  cudaError_t e = cudaGraphLaunch(c->gexec, st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(c, EAGLE3_ERR_CUDA, std::string("cudaGraphLaunch: ") + cudaGetErrorString(e));
  }
  c->launches = 1 + c->graph_launches;
  return cuda_status(c, "graph_launch");
}

eagle3_status eagle3_lm_head_topk(eagle3_ctx* c, int R, const void* h, int* tok, float* logq,
                                  float* lse, eagle3_stream stream) {
  if (!c) return EAGLE3_ERR_INVALID_ARG;
  c->err.clear();
  c->launches = 0;
  if (R < 1 || R > c->cfg.max_batch * c->k) return fail(c, EAGLE3_ERR_SHAPE, "R out of range");
  if (!h || !tok || !logq) return fail(c, EAGLE3_ERR_INVALID_ARG, "null pointer");
  cudaStream_t st = (cudaStream_t)stream;
  c->last = st;
  draft_head(c, h, R, false, tok, logq, lse, st);
  return cuda_status(c, "lm_head_topk");
}

eagle3_status eagle3_linear(eagle3_ctx* c, int which, int R, const void* X, float* Y,
                            eagle3_stream stream) {
  if (!c) return EAGLE3_ERR_INVALID_ARG;
  c->err.clear();
  c->launches = 0;
  const eagle3_config& f = c->cfg;
  const int d = f.d, qd = f.n_q_heads * f.head_dim, kvd = f.n_kv_heads * f.head_dim;
  struct Wd { int id; const void* p; int N, K; };
  const Wd defs[] = {{TCW_FC, c->w.w_fc, d, 3 * d},   {TCW_Q, c->w.w_q, qd, 2 * d},
                     {TCW_K, c->w.w_k, kvd, 2 * d},   {TCW_V, c->w.w_v, kvd, 2 * d},
                     {TCW_O, c->w.w_o, d, qd},        {TCW_GATE, c->w.w_gate, f.ffn, d},
                     {TCW_UP, c->w.w_up, f.ffn, d},   {TCW_DOWN, c->w.w_down, d, f.ffn},
                     {TCW_LM, c->w.w_lm, f.vocab, d}, {TCW_T, c->w.w_target, f.vocab, d}};
  if (which < 0 || which > 9) return fail(c, EAGLE3_ERR_INVALID_ARG, "which must be in 0..9");
  const Wd& e = defs[which];
  if (!e.p) return fail(c, EAGLE3_ERR_INVALID_ARG, "that weight is not set");
  if (R < 1 || R > c->rows_cap) return fail(c, EAGLE3_ERR_SHAPE, "R out of range");
  if (!X || !Y) return fail(c, EAGLE3_ERR_INVALID_ARG, "null pointer");
  cudaStream_t st = (cudaStream_t)stream;
  c->last = st;
  gemm1(c, e.id, X, e.K, e.p, e.N, e.K, Y, e.N, R, false, 1, (size_t)R * e.N, st);
  return cuda_status(c, "linear");
}

eagle3_status eagle3_check(eagle3_ctx* c) {
  if (!c) return EAGLE3_ERR_INVALID_ARG;
  cudaError_t e = cudaStreamSynchronize(c->last);
  if (e != cudaSuccess) return fail(c, EAGLE3_ERR_CUDA, std::string("sync: ") + cudaGetErrorString(e));
  int flags = 0;
  e = cudaMemcpy(&flags, c->flags, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(c, EAGLE3_ERR_CUDA, std::string("flag read: ") + cudaGetErrorString(e));
  if (!flags) return EAGLE3_OK;
  cudaMemset(c->flags, 0, sizeof(int));
  std::string m = "device check failed:";
  if (flags & FLAG_TREE_NOT_CLOSED) m += " kept set not ancestor-closed;";
  if (flags & FLAG_PAGE_RANGE) m += " page index out of range;";
  if (flags & FLAG_TOKEN_RANGE) m += " token id out of range;";
  if (flags & FLAG_POS_RANGE) m += " position beyond cache capacity;";
  if (flags & FLAG_ROWS_RANGE) m += " new-row count or accepted length out of range;";
  if (flags & FLAG_TIMEOUT) {
    m += " bounded wait timed out;";
    return fail(c, EAGLE3_ERR_TIMEOUT, m);
  }
  return fail(c, EAGLE3_ERR_DEVICE_ASSERT, m);
}

const char* eagle3_last_error(const eagle3_ctx* c) { return c ? c->err.c_str() : "null context"; }

size_t eagle3_workspace_bytes(const eagle3_ctx* c) { return c ? c->arena_bytes : 0; }

int eagle3_last_launch_count(const eagle3_ctx* c) { return c ? c->launches : 0; }

eagle3_status eagle3_draft_noise(eagle3_ctx* c, unsigned long long seed, unsigned long long round_id,
                                 eagle3_stream stream) {
  if (!c) return EAGLE3_ERR_INVALID_ARG;
  c->err.clear();
  if (!c->sampled) return fail(c, EAGLE3_ERR_STATE, "the context does not sample its draft");
  c->draft_seed = seed;
  launch_set_u64(c->d_draft_round, round_id, (cudaStream_t)stream);
  return cuda_status(c, "draft_noise");
}

eagle3_status eagle3_set_control(eagle3_ctx* c, const eagle3_control* ctl) {
  if (!c) return EAGLE3_ERR_INVALID_ARG;
  c->err.clear();
  if (!ctl) {
    c->ctl = CtlDev{};
    c->ctl_host = eagle3_control{};
    return EAGLE3_OK;
  }
  const eagle3_control& h = *ctl;
  auto ok_f = [](float x) { return x >= 0.f && x < 3.0e38f; };
  if (!ok_f(h.tau_depth) || !ok_f(h.tau_verify) || !(h.depth_growth > 0.f) || !ok_f(h.depth_growth) ||
      h.light_batch < 0 || (h.light_batch > 0 && (h.k_light < 1 || h.k_heavy < 1)) ||
      (h.tau_depth > 0.f && !h.pass_us) || (h.tau_verify > 0.f && !h.verify_us))
    return fail(c, EAGLE3_ERR_INVALID_ARG, "bad control");
  if (h.tau_depth > 0.f)
    for (int t = 0; t < c->D; ++t)
      if (!ok_f(h.pass_us[t])) return fail(c, EAGLE3_ERR_INVALID_ARG, "bad pass_us");
  if (h.tau_verify > 0.f)
    for (int m = 0; m <= c->M; ++m)
      if (!ok_f(h.verify_us[m])) return fail(c, EAGLE3_ERR_INVALID_ARG, "bad verify_us");
  if (h.tau_depth > 0.f &&
      cudaMemcpy(c->d_pass_us, h.pass_us, (size_t)c->D * 4, cudaMemcpyHostToDevice) != cudaSuccess)
    return fail(c, EAGLE3_ERR_CUDA, "control copy");
  if (h.tau_verify > 0.f &&
      cudaMemcpy(c->d_verify_us, h.verify_us, (size_t)(c->M + 1) * 4, cudaMemcpyHostToDevice) !=
          cudaSuccess)
    return fail(c, EAGLE3_ERR_CUDA, "control copy");
  CtlDev d{};
  d.on = 1;
  d.depth_cap = h.depth_cap;
  d.topk_cap = h.topk_cap;
  d.verify_cap = h.verify_cap;
  d.k_call = c->k;
  d.tau_depth = h.tau_depth;
  d.depth_growth = h.depth_growth;
  d.tau_verify = h.tau_verify;
  d.pass_us = c->d_pass_us;
  d.verify_us = c->d_verify_us;
  d.d_eff = c->d_deff;
  d.active = c->d_active;
  c->ctl = d;
  c->ctl_host = h;
  c->ctl_host.pass_us = nullptr;  // copied; the caller's arrays are not kept
  c->ctl_host.verify_us = nullptr;
  return EAGLE3_OK;
}

eagle3_status eagle3_latency_costs(const eagle3_latency_table* t, int B, int P, int depth,
                                   int topk, int n_verify, float* pass_us, float* verify_us) {
  if (!t || !pass_us || !verify_us || depth < 1 || topk < 1 || n_verify < 0 || t->n_batch < 1 ||
      t->n_prefix < 1 || t->n_tokens < 1 || !t->batch || !t->prefix || !t->tokens ||
      !t->draft_us || !t->verify_us)
    return EAGLE3_ERR_INVALID_ARG;
  auto ascending = [](const int* g, int n) {
    for (int i = 1; i < n; ++i)
      if (g[i] <= g[i - 1]) return false;
    return true;
  };
  if (!ascending(t->batch, t->n_batch) || !ascending(t->prefix, t->n_prefix) ||
      !ascending(t->tokens, t->n_tokens))
    return EAGLE3_ERR_INVALID_ARG;
  for (int i = 0; i < depth; ++i)
    pass_us[i] = (float)table_at(t, t->draft_us, B, P, i == 0 ? 1 : topk);
  verify_us[0] = 0.f;
  for (int m = 1; m <= n_verify; ++m) verify_us[m] = (float)table_at(t, t->verify_us, B, P, m);
  return EAGLE3_OK;
}

}  // extern "C"
