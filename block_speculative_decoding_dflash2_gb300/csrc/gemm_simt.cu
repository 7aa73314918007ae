// Exact fp32 contraction out[n][m] = sum_k W[m][k] * X[n][k] on the CUDA
// cores (FMA, k ascending) for the fp32 workload, whose tolerance (1e-4)
// rules out TF32 tensor cores.  Same contract as the tcgen05 path with one
// K split; the lm_head's top-k runs afterwards over the stored logits.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace df2 {

namespace {

constexpr int TM = 64, TN = 32, TK = 16;

__global__ void __launch_bounds__(256) simt_gemm_kernel(const float* __restrict__ W, int M, int K, int ldw,
                                                        const float* __restrict__ X, int N, int ldx,
                                                        float* __restrict__ out, int accumulate) {
  __shared__ float Ws[TK][TM + 1];
  __shared__ float Xs[TK][TN + 1];
  pdl_launch_next();
  pdl_wait();
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.x * TM, n0 = blockIdx.y * TN;
  float acc[4][2] = {};
  for (int k0 = 0; k0 < K; k0 += TK) {
    for (int i = threadIdx.x; i < TM * TK; i += 256) {
      const int mm = i / TK, kk = i % TK;
      const int m = m0 + mm, k = k0 + kk;
      Ws[kk][mm] = (m < M && k < K) ? W[(size_t)m * ldw + k] : 0.f;
    }
    for (int i = threadIdx.x; i < TN * TK; i += 256) {
      const int nn = i / TK, kk = i % TK;
      const int n = n0 + nn, k = k0 + kk;
      Xs[kk][nn] = (n < N && k < K) ? X[(size_t)n * ldx + k] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j) acc[i][j] = fmaf(Ws[kk][tx + 16 * i], Xs[kk][ty + 16 * j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int m = m0 + tx + 16 * i, n = n0 + ty + 16 * j;
      if (m < M && n < N) {
        float* p = out + (size_t)n * M + m;
        *p = accumulate ? *p + acc[i][j] : acc[i][j];
      }
    }
}

}  // namespace

int gemm_f32(const GemmOp& g, const Ctx& c) {
  if (g.M <= 0 || g.N <= 0 || g.K <= 0) return DFLASH2_ERR_SHAPE;
  dim3 grid((g.M + TM - 1) / TM, (g.N + TN - 1) / TN);
  return launch_k(simt_gemm_kernel, grid, dim3(256), 0, c, static_cast<const float*>(g.W), g.M, g.K, g.ldw,
                  static_cast<const float*>(g.X), g.N, g.ldx, g.out, g.accumulate ? 1 : 0);
}

}  // namespace df2
