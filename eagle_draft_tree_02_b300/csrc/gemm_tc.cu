#include "gemm_tc.h"

namespace e3 {

struct TcGemm {};
TcGemm* tc_create(const eagle3_config&, const eagle3_weights&, eagle3_ctx*) { return nullptr; }
void tc_destroy(TcGemm* t) { delete t; }
bool tc_gemm(TcGemm*, int, const void*, int, const void*, int, int, float*, int, int, int, int,
             size_t, cudaStream_t) { return false; }
bool tc_lm_head(TcGemm*, const void*, int, const HeadParts&, cudaStream_t) { return false; }
bool tc_verify_head(TcGemm*, const void*, const VerifyHeadArgs&, cudaStream_t) { return false; }

}  // namespace e3
