// fp32 token-wise Linear on CUDA cores (fp32 models only).
//
// C[m, n] = sum_k A[m, k] W[n, k] over the flattened rows of the iteration,
// followed by the fused epilogue (bias, GeLU, residual Add, K/V Split).
// tcgen05's tf32 kind does not meet an fp32 tolerance, so fp32 models keep
// plain FMA accumulation; bf16 models use the tcgen05 kernel instead.
#include <stdint.h>

#include "epilogue.cuh"
#include "orca_internal.h"

namespace orca {
namespace {

constexpr int BM = 64, BN = 64, BK = 16;

__global__ void __launch_bounds__(256) gemm_simt_f32_kernel(const float *__restrict__ A,
                                                            const float *__restrict__ W, int M, int N,
                                                            int K, EpiParams epi) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Ws[BK][BN + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  float acc[4][4] = {};
  const int lr = threadIdx.x >> 2, lk = (threadIdx.x & 3) * 4;  // loader: row, k offset
  for (int k0 = 0; k0 < K; k0 += BK) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int k = k0 + lk + j;
      const int am = m0 + lr, wn = n0 + lr;
      As[lk + j][lr] = (am < M && k < K) ? A[(int64_t)am * K + k] : 0.f;
      Ws[lk + j][lr] = (wn < N && k < K) ? W[(int64_t)wn * K + k] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < BK; ++k) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) { a[i] = As[k][ty * 4 + i]; b[i] = Ws[k][tx * 4 + i]; }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
  const int col = n0 + tx * 4;
  if (col >= N) return;
  const int cnt = min(4, N - col);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = m0 + ty * 4 + i;
    if (row < M) epi_apply<float, 4>(epi, row, col, acc[i], cnt);
  }
}

}  // namespace

cudaError_t launch_gemm_simt_f32(const float *A, const float *W, int M, int N, int K, const EpiParams &epi,
                                 cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  dim3 grid((N + BN - 1) / BN, (M + BM - 1) / BM);
  gemm_simt_f32_kernel<<<grid, 256, 0, st>>>(A, W, M, N, K, epi);
  return cudaGetLastError();
}

}  // namespace orca
