// Shared device helpers of the CUDA path: element loads/stores for the two
// storage types, warp reductions, the device error flag.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace e3 {

typedef __nv_bfloat16 bf16;

// device error flag bits (or-ed into ctx->d_flags[0])
enum : int {
  FLAG_TREE_NOT_CLOSED = 1,   // kept set of a supplied pool is not ancestor-closed
  FLAG_PAGE_RANGE = 2,        // page table entry outside [0, n_pages)
  FLAG_TOKEN_RANGE = 4,       // token id outside [0, V)
  FLAG_POS_RANGE = 8,         // row position beyond the cache capacity
  FLAG_TIMEOUT = 16,          // a bounded wait gave up
  FLAG_ROWS_RANGE = 32,       // a request's new-row count or accepted length out of range
};

template <typename T> __device__ __forceinline__ float ldf(const T* p);
template <> __device__ __forceinline__ float ldf<float>(const float* p) { return *p; }
template <> __device__ __forceinline__ float ldf<bf16>(const bf16* p) { return __bfloat162float(*p); }

template <typename T> __device__ __forceinline__ void stf(T* p, float v);
template <> __device__ __forceinline__ void stf<float>(float* p, float v) { *p = v; }
template <> __device__ __forceinline__ void stf<bf16>(bf16* p, float v) { *p = __float2bfloat16_rn(v); }

// Activation rows that feed a tcgen05 GEMM.  A "split" bf16 buffer stores row
// r as two rows of K: hi = bf16(v) at row 2r and lo = bf16(v - hi) at row
// 2r + 1, so the GEMM sees 2R rows and adds the two accumulator columns of a
// row: the activation then carries about 16 significant bits instead of 8,
// and the weights (the streamed operand) are still read once.  fp32 buffers
// are never split.
__device__ __forceinline__ size_t act_row(int r, int K, bool split) {
  return (size_t)r * K * (split ? 2 : 1);
}
template <typename T> __device__ __forceinline__ void st_act(T* row, int K, int j, float v, bool split);
template <> __device__ __forceinline__ void st_act<float>(float* row, int, int j, float v, bool) {
  row[j] = v;
}
template <> __device__ __forceinline__ void st_act<bf16>(bf16* row, int K, int j, float v, bool split) {
  const bf16 hi = __float2bfloat16_rn(v);
  row[j] = hi;
  if (split) row[K + j] = __float2bfloat16_rn(v - __bfloat162float(hi));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// (value desc, index asc) total order used by every top-k and argmax.
__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// Warp-wide best (value, index) under `better`; result in every lane.
__device__ __forceinline__ void warp_best(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float ov = __shfl_xor_sync(0xffffffffu, v, o);
    int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (better(ov, oi, v, i)) { v = ov; i = oi; }
  }
}

// Block-wide sum of a float for blockDim.x <= 1024; `red` holds >= 32 floats.
__device__ __forceinline__ float block_sum(float v, float* red) {
  int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  float t = (threadIdx.x < nw) ? red[threadIdx.x] : 0.f;
  if (wid == 0) t = warp_sum(t);
  if (threadIdx.x == 0) red[0] = t;
  __syncthreads();
  float r = red[0];
  __syncthreads();
  return r;
}

__device__ __forceinline__ void raise_flag(int* flags, int bit) { atomicOr(flags, bit); }

// Programmatic dependent launch.  Every kernel here is launched with
// launch_pdl, so it may start while the kernel before it on the stream is
// still finishing.  pdl_begin() first waits until that kernel has completed
// and its writes are visible (a no-op for a kernel launched the ordinary way),
// then lets the next kernel start launching.  It must run before the kernel
// reads anything a predecessor wrote, and before any thread returns: a kernel
// completes only after it has waited, which keeps the chain transitive.
__device__ __forceinline__ void pdl_begin() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Raise `kernel`'s dynamic shared-memory limit to `bytes` on the current device
// (once per device and kernel; thread-safe).  False if the runtime refused.
bool smem_limit(const void* kernel, int bytes);

// Launch `kernel` with programmatic stream serialization allowed (see pdl_begin).
template <typename... KArgs, typename... Args>
inline void launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, kernel, args...);
}

// launch_pdl with thread-block clusters of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
inline void launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               cudaStream_t st, int cluster_x, Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace e3
