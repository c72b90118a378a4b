// Internal launch interface of the two-stage draft head (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace e3 {

// ----------------------------------------------------------------------------- lowrank.cu
// Two-stage draft head (EAGLE-4 blog, "Efficient LM Head": low-rank recall,
// exact rerank).  Per row: t = V_lr h; the low-rank scores l = U t are
// never stored -- a sample of the vocabulary gives, per 32-token group, its
// maximum; the C-th largest group maximum is a lower bound `thr` of the C-th
// best score (C groups each hold a score >= it), so every token with
// l >= thr is appended to a per-row buffer, and the buffer holds the top C.
// A per-row kernel sorts the buffer, keeps the top C (score desc, token asc),
// rescores them with the exact head and takes log q over C and its top k.
constexpr int kLrSampleTokens = 16384;  // tokens [0, 16384) form the sample
constexpr int kLrCap = 4096;            // buffer entries per row

struct LowRankArgs {
  int R, V, d, r, C, k;
  int n_groups;            // 32-token groups in the sample
  float* gmax;             // [n_groups][R] group maxima of the low-rank scores
  float* thr;              // [R]
  int* cnt;                // [R] entries appended (may exceed kLrCap)
  float* cval;             // [R][kLrCap]
  int* ctok;               // [R][kLrCap]
  const void* t;           // [R][r] low-rank activations (split rows when t_split)
  int t_split;
  const void* U;           // [V][r]
  const void* W;           // [V][d] exact head
  const void* H;           // [R][d] head input rows (split rows when h_split)
  int h_split;
  int* tok;                // [R][k]
  float* logq;             // [R][k]
  float* lse;              // [R] log-sum-exp over the C candidates (may be NULL)
  int* cand_out;           // optional [B][n_exp][C] candidates in low-rank order
  int cand_n_exp, cand_slot0, cand_rpr;
  int* sel_tok;            // [R][C] candidates of each row, low-rank order (workspace)
  float* sel_z;            // [R][C] their exact logits (workspace)
  int* sel_done;           // [R] rescoring blocks finished per row (workspace)
  int* flags;
};
// fp32 storage: low-rank scores of a 64x64 tile on CUDA cores; mode 0 writes
// the group maxima of the sample tokens, mode 1 appends tokens >= thr.
template <typename T> void launch_lowrank_simt(int mode, const LowRankArgs& a, cudaStream_t st);
int lowrank_simt_groups(int V);
int lowrank_tc_groups(int V);
// per row: thr = C-th largest group maximum (-inf when there are fewer than C
// groups), and the append counter reset to 0
void launch_lowrank_threshold(const LowRankArgs& a, cudaStream_t st);
// per row: the C candidates, then their exact logits, log q over C and top k (2 launches)
template <typename T> void launch_lowrank_select(const LowRankArgs& a, cudaStream_t st);
// Y rows from split-K partials: out row r (split or plain) = sum_s part[s][r]
template <typename T>
void launch_reduce_store(int R, int N, int S, const float* part, void* out, bool split,
                         cudaStream_t st);

}  // namespace e3
