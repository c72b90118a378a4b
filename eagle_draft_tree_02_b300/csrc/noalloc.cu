// eagle3_lm_head_topk_noalloc: the draft LM head with its fused softmax and
// top-k, for callers that must not allocate device memory.
//
// Who needs this: code that runs inside a host runtime which owns every byte of
// device memory (an inference server that reserves the whole HBM for its KV
// pool up front, a plugin that may only use its host framework's allocator),
// and latency-critical callers for which cudaMalloc's implicit device
// synchronisation is not acceptable.  Such a caller cannot create a context
// (eagle3_create allocates its workspace once), so this entry point takes the
// weights and sizes directly and keeps its scratch -- the per-tile partial
// (max, sum-exp) and top-k lists that the merge kernel reduces -- in one
// fixed-size array in the library's own device global memory.
//
// The array lives as long as the library is loaded, on every GPU that loads
// it.  Its address is looked up once per device (first call with that device
// current) and cached; later calls allocate nothing and call no allocating
// routine.  The first call on a device is special: under CUDA's default lazy
// module loading, the module holding this array is loaded onto the device
// when its address is first looked up, and that load places the 16 MiB array
// (and the module's code) in device memory, which may synchronise the device
// and fails if the device has no 16 MiB left.  So make the first call on each
// device early -- before the caller reserves its memory pools and before any
// stream capture -- and treat later calls as the allocation-free ones.  All
// calls share the array, so calls whose work overlaps on the GPU (two streams,
// or two host threads) race on it: the caller must order them.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/eagle3.h"
#include "common.cuh"
#include "gemm_tc.h"
#include "kernels.h"

// 16 MiB.  Word 0 is the device error flag the kernels raise; the partials
// follow at byte 256.
#define E3_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
static __device__ __align__(256) unsigned char g_noalloc_scratch[E3_NOALLOC_SCRATCH_BYTES];

namespace e3 {
namespace {

constexpr size_t kNoallocScratchBytes = E3_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Device address of the scratch array for the current device (nullptr on error).
void* scratch_address(eagle3_status* st) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    *st = EAGLE3_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      *st = EAGLE3_ERR_CUDA;
      return nullptr;
    }
    g_addr[dev] = p;
  }
  return g_addr[dev];
}

}  // namespace
}  // namespace e3

using namespace e3;

extern "C" eagle3_status eagle3_lm_head_topk_noalloc(int dtype, int vocab, int d, int topk,
                                                     const void* w_lm, int R, const void* h, int* tok,
                                                     float* logq, float* lse, int* dev_status,
                                                     eagle3_stream stream) {
  if (dtype != EAGLE3_FP32 && dtype != EAGLE3_BF16) return EAGLE3_ERR_INVALID_ARG;
  if (vocab <= 0 || d <= 0 || topk < 1 || topk > 16 || R < 1) return EAGLE3_ERR_INVALID_ARG;
  if (!w_lm || !h || !tok || !logq) return EAGLE3_ERR_INVALID_ARG;
  const bool bf = dtype == EAGLE3_BF16;
  // the tensor-core path reads W and h through TMA: 16-byte rows and bases, <= 256 rows
  if (bf && (d % 8 || ((uintptr_t)w_lm & 15) || ((uintptr_t)h & 15))) return EAGLE3_ERR_INVALID_ARG;
  if (bf && R > 256) return EAGLE3_ERR_SHAPE;
  const int n_parts = bf ? tc_head_parts(vocab) : lm_head_simt_parts(vocab);
  const size_t ms_b = align256((size_t)n_parts * R * 2 * sizeof(float));
  const size_t kv_b = align256((size_t)n_parts * R * topk * sizeof(float));
  const size_t need = 256 + ms_b + 2 * kv_b;
  if (need > kNoallocScratchBytes) return EAGLE3_ERR_SHAPE;

  eagle3_status s = EAGLE3_OK;
  char* base = static_cast<char*>(scratch_address(&s));
  if (!base) return s;
  cudaStream_t st = (cudaStream_t)stream;
  int* flags = reinterpret_cast<int*>(base);
  HeadParts hp{};
  hp.n_parts = n_parts;
  hp.R = R;
  hp.k = topk;
  hp.ms = reinterpret_cast<float*>(base + 256);
  hp.val = reinterpret_cast<float*>(base + 256 + ms_b);
  hp.idx = reinterpret_cast<int*>(base + 256 + ms_b + kv_b);
  // the flag word is the only scratch that must start at zero: every partial
  // is written by the head kernel before the merge reads it
  if (cudaMemsetAsync(flags, 0, sizeof(int), st) != cudaSuccess) {
    cudaGetLastError();
    return EAGLE3_ERR_CUDA;
  }
  if (bf) {
    const int rc = tc_lm_head_raw(w_lm, vocab, d, h, R, hp, flags, st);
    if (rc == 1) return EAGLE3_ERR_INVALID_ARG;
    if (rc != 0) return EAGLE3_ERR_CUDA;
  } else {
    launch_lm_head_simt<float>(h, w_lm, R, vocab, d, hp, st);
  }
  launch_topk_merge(hp, tok, logq, lse, 0, st);
  if (dev_status &&
      cudaMemcpyAsync(dev_status, flags, sizeof(int), cudaMemcpyDeviceToDevice, st) != cudaSuccess) {
    cudaGetLastError();
    return EAGLE3_ERR_CUDA;
  }
  cudaError_t e = cudaPeekAtLastError();
  if (e != cudaSuccess) {
    cudaGetLastError();
    return EAGLE3_ERR_CUDA;
  }
  return EAGLE3_OK;
}
