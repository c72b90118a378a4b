// Internal launch interface of the CUDA path (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace e3 {

// ----------------------------------------------------------------------------- decoder.cu
struct QkvEpi {
  int R, S, Hq, Hkv, dh, has_q;
  const float* part;        // [S][R][(has_q*Hq + 2Hkv) dh]
  const float2* rope;       // [rope_rows][dh/2] (cos, sin)
  int rope_rows;
  const int *row_b, *row_pos, *row_dst;
  float* q_out;             // [R][Hq dh]
  void *cache_k, *cache_v;  // prefix cache
  const int* page_table;    // NULL = contiguous
  int page_size, max_pages, n_pages, max_prefix;
  void *tree_k, *tree_v;    // tree scratch [B][tree_slots][Hkv][dh], fp32
  int tree_slots;
  int* flags;
};

template <typename T>
void launch_build_input(int R, int d, int V, float eps, const int* tok, const float* hid_base,
                        const int* hid_row, const void* E, const void* g_emb, const void* g_hid,
                        void* x, bool split, int* flags, cudaStream_t st);
void launch_reduce_parts(int R, int N, int S, const float* part, float* out, cudaStream_t st);
// g = rms(sum of fusion partials) * g_fc (the FC-norm variant), fp32 [R, N]
template <typename T>
void launch_reduce_norm(int R, int N, int S, float eps, const float* part, const void* g_fc,
                        float* out, cudaStream_t st);
template <typename T> void launch_qkv_epilogue(const QkvEpi& p, cudaStream_t st);
// post = false: r = hid + W_o o, z = rms(r) g_post; true (post-norm): r = z = rms(hid + W_o o) g_post
template <typename T>
void launch_o_epilogue(int R, int d, int S, float eps, const float* part, const float* hid_base,
                       const int* hid_row, const void* g_post, float* r_out, void* z_out,
                       bool split, bool post, cudaStream_t st);
// part: [S][R][2F] with the gate in columns [0, F) and up in [F, 2F)
template <typename T>
void launch_swiglu(int R, int F, int S, const float* part, void* a, bool split, cudaStream_t st);
// post = false: s = r + W_down a, h = rms(s) g_final; true (post-norm): s = h = rms(r + W_down a) g_final
template <typename T>
void launch_down_epilogue(int R, int d, int S, float eps, const float* part, const float* r_in,
                          const void* g_final, const int* s_dst, float* s_base, const int* h_dst,
                          void* h_base, bool split, bool post, cudaStream_t st);

// ----------------------------------------------------------------------------- gemm_simt.cu
// Y[s][r][col0 + n] = sum_{k in split s} X[r][k] W[n][k]  (fp32 accumulate)
template <typename T>
void launch_gemm_simt(const void* X, int ldx, const void* W, int ldw, float* Y, int ldy, int col0,
                      int R, int N, int K, int S, size_t split_stride, cudaStream_t st);

// ----------------------------------------------------------------------------- attention.cu
struct AttnArgs {
  int B, rows_per_req, Hq, Hkv, dh;
  const float* q;          // [*, Hq dh] fp32, row via q_row
  const int* q_row;        // [R] row of q for tail row r
  const int* n_prefix;     // [B] prefix keys 0..n_prefix-1
  const void *cache_k, *cache_v;
  const int* page_table;
  int page_size, max_pages, n_pages, max_prefix;
  const void *tree_k, *tree_v;  // [B][tree_slots][Hkv][dh], fp32
  int tree_slots;
  const uint32_t* mask;    // [R][mask_words] bits over tree slots
  int mask_words;
  int keys_per_split, n_prefix_splits, n_tree_splits;
  float* o_part;           // [n_splits][R][Hq][dh]
  float* ml_part;          // [n_splits][R][Hq][2]
  void* out;               // [R][Hq dh] storage type (split rows: see st_act)
  bool split;
  int* flags;
  const int* skip;  // if set and *skip == 0 (no request active in the pass), the kernels return
  bool prefix_stable;  // no kernel since the last completed one writes the prefix cache
  // tensor-core kernel: the caches as tensor maps (encode_kv_map), box_rows
  // tokens per box, tm_T tokens in the tensor (a box at row tm_T reads zeros)
  int tm_rows, tm_T;
  CUtensorMap tm_k, tm_v;
};
// Launches the key splits (prefix and tree) and their merge: 2 launches.
template <typename T> void launch_tree_attention(const AttnArgs& a, cudaStream_t st);
// query groups per (request, KV head) of the prefix-split kernel
int attention_qgroups(int rows_per_req, int Hq, int Hkv, bool mma);
// the tensor-core path takes the tcgen05 kernel (more than 128 queries per KV head)
bool attention_uses_tc(int rows_per_req, int Hq, int Hkv);
bool attention_uses_mma(int elem_bytes, int dh, int page_size);
// tokens per tensor-map box of the tensor-core kernel: 64, or the largest
// divisor of 64 that divides the page size (at least 8 when the kernel is used)
int attention_box_rows(int page_size);
// runtime.cu: the cache [T][Hkv][dh] (bf16) as a tensor map with boxes of
// 64 dims x 1 head x box_rows tokens, 128-byte swizzle; false if refused
bool encode_kv_map(CUtensorMap* m, const void* base, int T, int Hkv, int dh, int box_rows);

// ----------------------------------------------------------------------------- lmhead.cu
struct HeadParts {
  int n_parts, R, k;
  float* ms;     // [n_parts][R][2]    running max, sum exp
  float* val;    // [n_parts][R][k]
  int* idx;      // [n_parts][R][k]
  const int* skip;  // if set and *skip == 0 (no request active in the pass), the kernels return
};
template <typename T>
void launch_lm_head_simt(const void* H, const void* W, int R, int V, int d, const HeadParts& hp,
                         cudaStream_t st);
int lm_head_simt_parts(int V);
void launch_topk_merge(const HeadParts& hp, int* tok, float* logq, float* lse, int row_stride_tok,
                       cudaStream_t st);

struct VerifyHeadArgs {
  int R, V, d, M1, kmax;     // rows = B*(M+1); M1 = M+1
  float inv_t;               // 1/T (1 when greedy)
  int sampling;
  unsigned long long seed, round_id;
  const unsigned long long* round_ptr;  // if set, the round id is read here (graph replays)
  const int* child_tok;      // [R][kmax] (-1 padded)
  float* child_z;            // [R][kmax]  target logit at each child token
  int n_parts;
  float* part;               // [n_parts][R][6]
  // Deferred draw (sampling, tensor-core head): if set, the head stores z
  // here ([R][V], fp32) and draws no Gumbel noise; bonus_gumbel then draws
  // it over the one row where each request's walk stops.
  float* logits;
};
template <typename T>
void launch_verify_head_simt(const void* H, const void* W, const VerifyHeadArgs& a, cudaStream_t st);
int verify_head_simt_parts(int V);
void launch_verify_merge(const VerifyHeadArgs& a, float* z_max, int* z_arg, float* lse, int* g_arg,
                         float* g_max, cudaStream_t st);

// ----------------------------------------------------------------------------- tree.cu
struct RowPlan {
  // rows whose K/V are produced (input build + QKV)
  int *kv_b, *kv_tok, *kv_hid, *kv_pos, *kv_dst;
  // rows that run attention and the rest of the layer
  int *t_q, *t_b, *t_hid, *t_sdst, *t_out;
  uint32_t* t_mask;
  int mask_words;
};
struct PoolDev {
  int *tok, *parent, *depth, *fwd;
  float *score, *logq;
  int n;  // pool_n
};
// Per-request caps and cost-aware rules of a round (all off when `on` is 0).
struct CtlDev {
  int on;
  const int *depth_cap, *topk_cap, *verify_cap;  // [B] or NULL
  int k_call;           // branch cap of this call's batch size (the light/heavy rule), <= k
  float tau_depth, depth_growth, tau_verify;
  const float* pass_us;    // [D]
  const float* verify_us;  // [M+1]
  int* d_eff;           // [B] depth the request runs to (set at pass 0, lowered by the rule)
  int* active;          // [D + 1] requests active at pass t
  int clip;             // sampled draft: a draw's score from the earlier draws only (any `on`)
  const float* lmax;    // sampled draft: [rows] the row's largest log q (clip only)
};
// pass 0 rows: n_new rows per request, or the ragged rows given by cu_new [B+1]
void launch_plan_root(int B, int n_new, const int* cu_new, int total, int max_new,
                      const int* tokens_new, const int* seq_lens, int n_slots, const RowPlan& rp,
                      int* root_tok, int* root_pos, int* n_prefix, int* flags, cudaStream_t st);
// the next round's new rows from a verification (B <= 1024)
void launch_next_rows(int B, int D, const int* accept_len, const int* out_tokens, int* cu_new,
                      int* tokens_new, int* flags, cudaStream_t st);
void launch_plan_prefill(int rows, int r0, int B, const int* cu_rows, const int* tokens,
                         const int* seq_lens, const RowPlan& rp, cudaStream_t st);
void launch_expand(const CtlDev& ctl, int B, int t, int k, int D, const int* top_tok, const float* top_logq,
                   const PoolDev& pool, int* frontier, uint32_t* slot_mask, int slot_words,
                   const int* root_pos, int n_slots, const RowPlan& rp, cudaStream_t st);

void launch_build_tree(const CtlDev& ctl, int B, int pool_n, int M, const int* tok, const int* parent,
                       const float* score, const int* depth, const int* root_tok,
                       const int* root_pos, int* t_tok, int* t_parent, int* t_depth, int* t_pos,
                       int* t_pidx, float* t_score, uint32_t* t_mask, int* flags, cudaStream_t st);
void launch_plan_verify(int B, int M, int kmax, const int* t_tok, const int* t_parent,
                        const int* t_pos, const int* t_pidx, const uint32_t* t_mask,
                        const int* pool_fwd, int pool_n, int n_slots, const RowPlan& rp,
                        int* n_prefix, int* child_tok, int* child_node, int* n_child, int* flags,
                        cudaStream_t st);
// Copy B activation rows of d elements: row b of src (index b * src_stride_rows)
// to row b * dst_stride_rows of dst, each buffer split or plain (see st_act);
// a plain source gives a zero lo row in a split destination.
void launch_copy_rows(int B, int d, int elem_bytes, const void* src, int src_stride_rows,
                      bool src_split, void* dst, int dst_stride_rows, bool dst_split,
                      cudaStream_t st);
void launch_copy_pool(int B, const PoolDev& pool, int* tok, int* parent, int* depth, int* fwd,
                      float* score, float* logq, cudaStream_t st);

// ----------------------------------------------------------------------------- verify.cu
struct WalkArgs {
  int B, M1, kmax, D, sampling;
  float inv_t;
  unsigned long long seed, round_id;
  const unsigned long long* round_ptr;  // if set, the round id is read here (graph replays)
  const int* t_tok;       // [B][M1]
  const int* child_node;  // [B][M1][kmax] tree indices (-1 padded)
  const int* n_child;     // [B][M1]
  const float* child_z;   // [B*M1][kmax]
  const float* lse;       // [B*M1]
  const int* z_arg;       // [B*M1]
  const int* g_arg;       // [B*M1]
  int *accept_len, *path, *out_tokens;
  unsigned long long* bonus_best;  // if set: [B], zeroed here for the deferred bonus draw
};
void launch_walk(const WalkArgs& a, cudaStream_t st);
// The bonus token of a sampling walk whose head deferred the Gumbel draw: at
// the node where request b's walk stopped, the Gumbel-argmax of z / T over the
// node's non-children, from the stored logits row.  Blocks (n_blk per
// request) fold their best into best[b] by atomicMax of a packed key; a
// second launch writes the token.  2 launches.
struct BonusArgs {
  int B, M1, kmax, D, V;
  float inv_t;
  unsigned long long seed, round_id;
  const unsigned long long* round_ptr;  // if set, the round id is read here
  const float* logits;    // [B*M1][V]
  const int* child_tok;   // [B*M1][kmax] (-1 padded)
  const int *accept_len, *path;
  int* out_tokens;        // [B][D+1]: the slot at accept_len is written
  int* g_arg;             // [B*M1]: written at the stop node
  unsigned long long* best;  // [B] (score, token) keys, zeroed by the walk
};
void launch_bonus_gumbel(const BonusArgs& a, cudaStream_t st);

// ----------------------------------------------------------------------------- sampled.cu
struct SampleArgs {  // sampled children of a pass's rows (Gumbel-top-k over the logits)
  int V, k, rows_per_req, slot0;
  unsigned long long seed, round_id;
  const unsigned long long* round_ptr;  // if set, the round id is read here
  const float* logits;  // [R][V]
  int* tok;             // [R][k] in draw order
  float* logq;          // [R][k]
  float* lmax;          // [R] largest log q of the row
};
void launch_sample_children(const SampleArgs& a, int R, cudaStream_t st);
struct QratioArgs {  // q-ratio verification walk
  int B, M1, kmax, D, V;
  float inv_t;
  unsigned long long seed, round_id;
  const unsigned long long* round_ptr;
  const float *z, *ell;   // [B*M1][V] target and draft logits of the tree nodes
  float *pw, *qw;         // [B][V] work rows
  const int *t_tok, *pidx, *child_node, *n_child;
  int *accept_len, *path, *out_tokens;
};
void launch_qratio_walk(const QratioArgs& a, cudaStream_t st);
// ----------------------------------------------------------------------------- target_logits.cu
struct LogitsVerifyArgs {  // verification against caller-supplied target logits
  int B, M1, kmax, V, R;        // R = B * M1 rows
  long long ld;                 // elements between consecutive logits rows
  const void* logits;           // [R][ld], fp32 or bf16, 16-byte aligned rows
  const int *t_tok, *t_parent;  // [B][M1] the kept tree
  int sampling;
  float inv_t;
  unsigned long long seed, round_id;
  const unsigned long long* round_ptr;  // if set, the round id is read here
  int *child_tok, *child_node, *n_child;  // [R][kmax], [R][kmax], [R]
  float* child_z;                         // [R][kmax]
  int n_chunks, chunk;                    // vocabulary chunks per row, tokens per chunk
  float* part;                            // [n_chunks][R][6], the verify_merge layout
  int* flags;
};
// vocabulary chunks per row for R rows (at most max_parts)
int logits_verify_chunks(int R, int V, int max_parts);
// the children plan and the per-chunk scan (2 launches); verify_merge folds the chunks
void launch_logits_verify(LogitsVerifyArgs a, bool bf, cudaStream_t st);

// *p = v, in stream order (sets the round id a captured graph reads)
void launch_set_u64(unsigned long long* p, unsigned long long v, cudaStream_t st);

}  // namespace e3
