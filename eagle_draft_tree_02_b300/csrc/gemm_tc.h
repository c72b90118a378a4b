// tcgen05 (5th-generation tensor core) GEMMs for bf16 storage: weights stream
// through TMA into shared memory, accumulators live in tensor memory.
#pragma once
#include <cuda_runtime.h>

#include "../../include/eagle3.h"
#include "kernels.h"

namespace e3 {

enum TcWeight { TCW_FC, TCW_Q, TCW_K, TCW_V, TCW_O, TCW_GATE, TCW_UP, TCW_DOWN, TCW_LM, TCW_T, TCW_N };

struct TcGemm;
TcGemm* tc_create(const eagle3_config& cfg, const eagle3_weights& w, eagle3_ctx* owner);
void tc_destroy(TcGemm* t);
bool tc_gemm(TcGemm* t, int wid, const void* X, int ldx, const void* W, int N, int K, float* Y,
             int ldy, int col0, int R, int S, size_t split_stride, cudaStream_t st);
bool tc_lm_head(TcGemm* t, const void* H, int R, const HeadParts& hp, cudaStream_t st);
bool tc_verify_head(TcGemm* t, const void* H, const VerifyHeadArgs& a, cudaStream_t st);

}  // namespace e3
