// gemm_f32.cu -- fp32 CUDA-core GEMM for the fp32 (precision-reference) path
// of the layer: C[M,N] = A[M,K]·B[K,N] with arbitrary element strides for A
// and B (so transposed operands need no copy), and the layer's epilogues.
#include "common.cuh"
#include "gemm.cuh"

namespace mtgr {

constexpr int F_BM = 64, F_BN = 64, F_BK = 16;

template <int EPI>
__global__ void __launch_bounds__(256) gemm_f32_kernel(int64_t M, int64_t N, int64_t K, const float* __restrict__ A,
                                                       int64_t sam, int64_t sak, const float* __restrict__ Bm,
                                                       int64_t sbk, int64_t sbn, float* __restrict__ C,
                                                       int64_t ldc, const float* __restrict__ R, int64_t ldr,
                                                       float* __restrict__ Z, int64_t ldz) {
  __shared__ float As[F_BK][F_BM + 1];
  __shared__ float Bs[F_BK][F_BN + 1];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int64_t m0 = (int64_t)blockIdx.y * F_BM, n0 = (int64_t)blockIdx.x * F_BN;
  float acc[4][4] = {};
  for (int64_t k0 = 0; k0 < K; k0 += F_BK) {
    for (int e = threadIdx.x; e < F_BM * F_BK; e += 256) {
      const int mm = e / F_BK, kk = e % F_BK;
      const int64_t gm = m0 + mm, gk = k0 + kk;
      As[kk][mm] = (gm < M && gk < K) ? A[gm * sam + gk * sak] : 0.f;
    }
    for (int e = threadIdx.x; e < F_BN * F_BK; e += 256) {
      const int nn = e % F_BN, kk = e / F_BN;
      const int64_t gn = n0 + nn, gk = k0 + kk;
      Bs[kk][nn] = (gn < N && gk < K) ? Bm[gk * sbk + gn * sbn] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < F_BK; ++kk) {
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
    const int64_t gm = m0 + ty * 4 + i;
    if (gm >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t gn = n0 + tx * 4 + j;
      if (gn >= N) continue;
      const float x = acc[i][j];
      if (EPI == EPI_SILU) {
        const float sg = 1.0f / (1.0f + expf(-x));  // C = silu(x), Z = silu'(x)
        Z[gm * ldz + gn] = sg * (1.0f + x * (1.0f - sg));
        C[gm * ldc + gn] = x * sg;
      } else if (EPI == EPI_RESIDUAL) {
        C[gm * ldc + gn] = R[gm * ldr + gn] + x;
      } else {
        C[gm * ldc + gn] = x;
      }
    }
  }
}

cudaError_t launch_gemm_f32(int epi, int64_t M, int64_t N, int64_t K, const float* A, int64_t sam, int64_t sak,
                            const float* B, int64_t sbk, int64_t sbn, float* C, int64_t ldc, const float* R,
                            int64_t ldr, float* Z, int64_t ldz, cudaStream_t s) {
  if (M == 0 || N == 0) return cudaSuccess;
  dim3 grid((unsigned)((N + F_BN - 1) / F_BN), (unsigned)((M + F_BM - 1) / F_BM));
  TraceScope tr("gemm_f32", s);
  switch (epi) {
    case EPI_SILU:
      gemm_f32_kernel<EPI_SILU><<<grid, 256, 0, s>>>(M, N, K, A, sam, sak, B, sbk, sbn, C, ldc, R, ldr, Z, ldz);
      break;
    case EPI_RESIDUAL:
      gemm_f32_kernel<EPI_RESIDUAL><<<grid, 256, 0, s>>>(M, N, K, A, sam, sak, B, sbk, sbn, C, ldc, R, ldr, Z, ldz);
      break;
    default:
      gemm_f32_kernel<EPI_PLAIN><<<grid, 256, 0, s>>>(M, N, K, A, sam, sak, B, sbk, sbn, C, ldc, R, ldr, Z, ldz);
  }
  return cudaGetLastError();
}

}  // namespace mtgr
