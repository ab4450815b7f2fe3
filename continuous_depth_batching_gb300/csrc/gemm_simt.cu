// CUDA-core GEMM C = A . W^T with fp32 accumulation and fused epilogues.
//
// Used for fp32 models (no tensor-core kind meets an fp32 result at 1e-4) and
// for shapes the tensor-core path does not cover.  Every output element sums
// k = 0..K-1 in order in one thread, so a row's result does not depend on the
// number of rows in the batch.
#include "common.cuh"
#include "kernels.cuh"

namespace cdb {

namespace {
constexpr int BM = 64, BN = 64, BK = 16;
}

template <typename T, int EPI>
__global__ void __launch_bounds__(256)
    k_gemm_simt(const T* __restrict__ A, int lda, const T* __restrict__ W, const T* __restrict__ W2, int N,
                int K, int rows, float* __restrict__ Cf, T* __restrict__ Ct, int ldc) {
  pdl_wait();
  pdl_trigger();
  constexpr bool SW = EPI == kEpiSwiglu;
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  __shared__ float B2s[SW ? BK : 1][BN + 4];
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4], acc2[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = acc2[i][j] = 0.f;

  for (int k0 = 0; k0 < K; k0 += BK) {
    for (int u = threadIdx.x; u < BM * BK; u += 256) {
      const int r = u / BK, kk = u % BK;
      const int gr = m0 + r, gk = k0 + kk;
      As[kk][r] = (gr < rows && gk < K) ? to_f(A[(size_t)gr * lda + gk]) : 0.f;
      const int gn = n0 + r;
      Bs[kk][r] = (gn < N && gk < K) ? to_f(W[(size_t)gn * K + gk]) : 0.f;
      if (SW) B2s[kk][r] = (gn < N && gk < K) ? to_f(W2[(size_t)gn * K + gk]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4], b2[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        b[j] = Bs[kk][tx * 4 + j];
        if (SW) b2[j] = B2s[kk][tx * 4 + j];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
          if (SW) acc2[i][j] = fmaf(a[i], b2[j], acc2[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = m0 + ty * 4 + i;
    if (r >= rows) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = n0 + tx * 4 + j;
      if (c >= N) continue;
      const size_t o = (size_t)r * ldc + c;
      if (EPI == kEpiStore) Cf[o] = acc[i][j];
      else if (EPI == kEpiResid) Cf[o] = Cf[o] + acc[i][j];
      else {
        const float g = acc[i][j];
        Ct[o] = from_f<T>(g / (1.0f + expf(-g)) * acc2[i][j]);
      }
    }
  }
}

template <typename T>
void launch_gemm(cudaStream_t s, int epi, const T* A, int lda, const T* W, const T* W2, int N, int K, int rows,
                 float* Cf, T* Ct, int ldc) {
  if (rows <= 0) return;
  dim3 grid((N + BN - 1) / BN, (rows + BM - 1) / BM);
  count_launch();
  if (epi == kEpiStore) launch_pdl(k_gemm_simt<T, kEpiStore>, dim3(grid), dim3(256), 0, s, A, lda, W, W2, N, K, rows, Cf, Ct, ldc);
  else if (epi == kEpiResid)
    launch_pdl(k_gemm_simt<T, kEpiResid>, dim3(grid), dim3(256), 0, s, A, lda, W, W2, N, K, rows, Cf, Ct, ldc);
  else launch_pdl(k_gemm_simt<T, kEpiSwiglu>, dim3(grid), dim3(256), 0, s, A, lda, W, W2, N, K, rows, Cf, Ct, ldc);
}

template void launch_gemm<float>(cudaStream_t, int, const float*, int, const float*, const float*, int, int, int,
                                 float*, float*, int);
template void launch_gemm<__nv_bfloat16>(cudaStream_t, int, const __nv_bfloat16*, int, const __nv_bfloat16*,
                                         const __nv_bfloat16*, int, int, int, float*, __nv_bfloat16*, int);

}  // namespace cdb
