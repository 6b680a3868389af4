// SIMT kernels of the MLA draft layer (see simt.cuh).
#include "simt.cuh"

#include <math.h>

namespace mla {
namespace simt {

namespace {

constexpr int GB_M = 64, GB_N = 64, GB_K = 16, G_THREADS = 256;

template <typename TA, typename TC>
__global__ void __launch_bounds__(G_THREADS)
gemm_nt_kernel(int M, int N, int K, const TA* __restrict__ A, long lda, long sA,
               const TA* __restrict__ B, long ldb, long sB, TC* __restrict__ C, long ldc,
               long sC, const float* __restrict__ G, long ldg, long sG) {
  __shared__ float As[GB_K][GB_M + 4];
  __shared__ float Bs[GB_K][GB_N + 4];
  const int z = blockIdx.z;
  A += z * sA;
  B += z * sB;
  C += z * sC;
  const int m0 = blockIdx.y * GB_M, n0 = blockIdx.x * GB_N;
  const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
  const int lr = tid / 4, lk = (tid % 4) * 4;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += GB_K) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int k = k0 + lk + u;
      const int am = m0 + lr, bn = n0 + lr;
      As[lk + u][lr] = (am < M && k < K) ? to_f32(A[(long)am * lda + k]) : 0.f;
      Bs[lk + u][lr] = (bn < N && k < K) ? to_f32(B[(long)bn * ldb + k]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < GB_K; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= N) continue;
      float v = acc[i][j];
      if (G) {
        const float g = G[z * sG + (long)m * ldg + n];
        v = v / (1.f + expf(-g));
      }
      C[(long)m * ldc + n] = from_f32<TC>(v);
    }
  }
}

}  // namespace

template <typename TA, typename TC>
void gemm_nt(cudaStream_t st, int M, int N, int K, int batch, const TA* A, long lda, long sA,
             const TA* B, long ldb, long sB, TC* C, long ldc, long sC, const float* G, long ldg,
             long sG) {
  if (M <= 0 || N <= 0 || batch <= 0) return;
  dim3 grid((N + GB_N - 1) / GB_N, (M + GB_M - 1) / GB_M, batch);
  gemm_nt_kernel<TA, TC><<<grid, G_THREADS, 0, st>>>(M, N, K, A, lda, sA, B, ldb, sB, C, ldc,
                                                      sC, G, ldg, sG);
}

#define MLA_GEMM_INST(TA, TC)                                                              \
  template void gemm_nt<TA, TC>(cudaStream_t, int, int, int, int, const TA*, long, long,   \
                                const TA*, long, long, TC*, long, long, const float*, long, long);
MLA_GEMM_INST(float, float)
MLA_GEMM_INST(__nv_bfloat16, float)
MLA_GEMM_INST(__half, float)
MLA_GEMM_INST(__half, __half)
MLA_GEMM_INST(__half, __nv_bfloat16)
#undef MLA_GEMM_INST

}  // namespace simt
}  // namespace mla
