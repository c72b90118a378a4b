// CUDA-core GEMM with fp32 accumulation: Y = X W^T, split along K.
//
// Used where the contraction must stay in fp32 (the fp32 storage config, whose
// logits are compared at 1e-4: TF32 tensor cores would round the operands to
// 10 mantissa bits).  64x64 output tile per block, 16-deep K slices staged in
// shared memory, 4x4 outputs per thread.
#include "common.cuh"
#include "kernels.h"

namespace e3 {

namespace {
constexpr int BM = 64, BN = 64, BK = 16;
}

template <typename T>
__global__ void __launch_bounds__(256) gemm_simt_kernel(const T* __restrict__ X, int ldx,
                                                        const T* __restrict__ W, int ldw,
                                                        float* __restrict__ Y, int ldy, int col0,
                                                        int R, int N, int K, int kps,
                                                        size_t split_stride) {
  pdl_begin();
  __shared__ float Xs[BK][BM + 4];
  __shared__ float Ws[BK][BN + 4];
  int tid = threadIdx.x;
  int tx = tid & 15, ty = tid >> 4;
  int r0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  int k_begin = blockIdx.z * kps;
  int k_end = min(K, k_begin + kps);
  float acc[4][4] = {};
  int lr = tid >> 2, lk = (tid & 3) * 4;  // loader: row lr, 4 consecutive k
  for (int k0 = k_begin; k0 < k_end; k0 += BK) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      int kk = k0 + lk + i;
      int xr = r0 + lr, wn = n0 + lr;
      Xs[lk + i][lr] = (xr < R && kk < k_end) ? ldf(X + (size_t)xr * ldx + kk) : 0.f;
      Ws[lk + i][lr] = (wn < N && kk < k_end) ? ldf(W + (size_t)wn * ldw + kk) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = Xs[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Ws[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
  float* Yz = Y + blockIdx.z * split_stride;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int r = r0 + ty * 4 + i;
    if (r >= R) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int n = n0 + tx * 4 + j;
      if (n < N) Yz[(size_t)r * ldy + col0 + n] = acc[i][j];
    }
  }
}

template <typename T>
void launch_gemm_simt(const void* X, int ldx, const void* W, int ldw, float* Y, int ldy, int col0,
                      int R, int N, int K, int S, size_t split_stride, cudaStream_t st) {
  if (R <= 0 || N <= 0) return;
  int kps = (K + S - 1) / S;
  kps = (kps + BK - 1) / BK * BK;
  dim3 grid((N + BN - 1) / BN, (R + BM - 1) / BM, S);
  launch_pdl(gemm_simt_kernel<T>, dim3(grid), dim3(256), 0, st, (const T*)X, ldx, (const T*)W, ldw, Y, ldy, col0, R, N,
                                            K, kps, split_stride);
}

template void launch_gemm_simt<float>(const void*, int, const void*, int, float*, int, int, int,
                                      int, int, int, size_t, cudaStream_t);

}  // namespace e3
