// Host-side runtime helpers shared by the launch code.
#include <cuda.h>
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"

namespace e3 {

// The dynamic shared-memory limit is an attribute of a kernel on one device,
// so it is raised once per (device, kernel) -- a process that drives several
// GPUs, or one whose host threads share the library, gets it on each device.
bool smem_limit(const void* kernel, int bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, int> done;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_pair(dev, kernel);
  auto it = done.find(key);
  if (it != done.end() && it->second >= bytes) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  done[key] = bytes;
  return true;
}

namespace {
typedef CUresult (*KvEncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                               const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                               CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                               CUtensorMapFloatOOBfill);

KvEncodeFn kv_encoder() {
  static std::once_flag once;
  static KvEncodeFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<KvEncodeFn>(p);
    else
      cudaGetLastError();
  });
  return fn;
}
}  // namespace

// The bf16 cache [T][Hkv][dh] as a three-dimensional tensor (dh innermost):
// one box is 64 dims (128 bytes, swizzled in 128-byte rows) of one KV head
// over box_rows consecutive tokens.
bool encode_kv_map(CUtensorMap* m, const void* base, int T, int Hkv, int dh, int box_rows) {
  KvEncodeFn enc = kv_encoder();
  if (!enc || !base || ((uintptr_t)base & 15) || T <= 0 || Hkv <= 0 || dh % 64 || box_rows <= 0 ||
      box_rows > 256)
    return false;
  cuuint64_t dims[3] = {(cuuint64_t)dh, (cuuint64_t)Hkv, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)dh * 2, (cuuint64_t)Hkv * dh * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace e3
