// tcgen05 (5th-generation tensor core) GEMMs for bf16 storage.
//
// Y = X W^T with W [N, K] (weights, row-major) and X [R, K] (activation rows).
// The weights take the MMA's M side (128 output features per tile) and the
// activation rows its N side (16..256), so a round's few rows never pad the
// 128-wide M dimension ("swap AB").  Both operands stream through TMA into
// 128-byte-swizzled shared memory; the fp32 accumulator lives in tensor memory
// and is read back with tcgen05.ld for the epilogue.  Epilogues: split-K
// partial store, the draft LM head's online softmax + top-k, and the verify
// head's argmax / log-sum-exp / Gumbel-argmax.
#pragma once
#include <cuda_runtime.h>

#include "../../include/eagle3.h"
#include "kernels.h"
#include "lowrank.h"

namespace e3 {

enum TcWeight {
  TCW_FC, TCW_Q, TCW_K, TCW_V, TCW_O, TCW_GATE, TCW_UP, TCW_DOWN, TCW_LM, TCW_T, TCW_LRU, TCW_LRV, TCW_N
};

struct GemmSeg {  // one weight matrix whose output columns start at col0
  int wid;
  const void* W;
  int N;
  int col0;
};

struct TcGemm;
// Returns nullptr and fills `err` when the driver entry point for tensor maps is missing.
TcGemm* tc_create(const eagle3_config& cfg, const eagle3_weights& w, char* err, int errlen);
void tc_destroy(TcGemm* t);
int tc_splits(int R, int n_mtiles, int K);
int tc_head_parts(int V);
// Y[s][r][col0 + n] for each segment; all segments share X and K.  With
// `split`, X holds each row r as a (hi, lo) pair of bf16 rows 2r, 2r+1 (see
// st_act) and the product is taken on their sum.  Returns false (and nothing
// is launched) on an unusable argument.
// skip (may be NULL): the launch returns at once if *skip == 0 when it runs
bool tc_gemm(TcGemm* t, const GemmSeg* segs, int nseg, const void* X, int ldx, int K, float* Y,
             int ldy, int R, bool split, int S, size_t split_stride, int* flags, cudaStream_t st,
             const int* skip = nullptr);
// The vocabulary heads.  hp.n_parts / a.n_parts must hold at least
// tc_head_parts(V) partials; on return they give the number written, which
// the merge kernels read.
bool tc_lm_head(TcGemm* t, const void* H, int R, bool split, HeadParts& hp, int* flags,
                cudaStream_t st);
bool tc_verify_head(TcGemm* t, const void* H, bool split, VerifyHeadArgs& a, int* flags,
                    cudaStream_t st);
// Low-rank scores U t of the two-stage head: mode 0 writes the 32-token group
// maxima of the sample tokens, mode 1 appends the tokens that reach the
// row's threshold (see lowrank.h).
bool tc_lowrank(TcGemm* t, int mode, const LowRankArgs& la, int* flags, cudaStream_t st);
// The draft-head launch of tc_lm_head on a bare weight pointer W [V, d] (bf16),
// with no TcGemm object: the tensor maps are encoded on the host stack and
// nothing is allocated.  Returns 0 when launched, 1 for an unusable shape
// (nothing launched), 2 when the driver or runtime refused (the tensor-map
// entry point is missing, the driver rejected an encode, or a launch
// attribute could not be set; nothing launched).
int tc_lm_head_raw(const void* W, int V, int d, const void* H, int R, HeadParts& hp,
                   int* flags, cudaStream_t st);

}  // namespace e3
