// gemm.cuh -- GEMM entry points used by the layer (internal).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mtgr {

enum GemmEpilogue : int {
  EPI_PLAIN = 0,     // C = acc
  EPI_SILU = 1,      // C = silu(acc), Z = silu'(acc)
  EPI_RESIDUAL = 2,  // C = R + acc
  EPI_F32 = 3,       // fp32 C = acc (split-K slices go to C + split*M*ldc)
};

// fp32 CUDA-core GEMM with element strides: A(m,k) = A[m*sam + k*sak], B(k,n) = B[k*sbk + n*sbn].
cudaError_t launch_gemm_f32(int epi, int64_t M, int64_t N, int64_t K, const float* A, int64_t sam, int64_t sak,
                            const float* B, int64_t sbk, int64_t sbn, float* C, int64_t ldc, const float* R,
                            int64_t ldr, float* Z, int64_t ldz, cudaStream_t s);

// bf16 tcgen05 GEMM.  A is [M,K] row-major (a_mn_major = false, lda >= K) or
// [K,M] row-major (a_mn_major = true, lda >= M); B is [N,K] row-major
// (b_mn_major = false) or [K,N] row-major (b_mn_major = true).  All leading
// dimensions and M/N/K multiples of 8; pointers 16-byte aligned.
struct GemmArgs {
  int64_t M, N, K;
  const __nv_bfloat16* A;
  int64_t lda;
  bool a_mn_major;
  const __nv_bfloat16* B;
  int64_t ldb;
  bool b_mn_major;
  int epi;
  void* C;  // bf16 (f16 when c_f16), or fp32 for EPI_F32
  bool c_f16;
  int64_t ldc;
  const __nv_bfloat16* R;  // residual (EPI_RESIDUAL)
  int64_t ldr;
  __nv_bfloat16* Z;  // silu'(acc) (EPI_SILU)
  int64_t ldz;
  bool ab_f16;  // A and B are f16 (else bf16)
  bool r_f16;   // the residual is f16 (else bf16)
  bool z_f16;   // silu'(acc) is written in f16 (else bf16)
  int splits;  // split-K slices (EPI_F32 only); slice s covers its own K range
  const float* out_scale;  // EPI_F32: device scalar the output is multiplied by (nullable)
  int32_t* status;
  const char* name;  // trace label
};
cudaError_t launch_gemm_bf16(const GemmArgs& a, cudaStream_t s);
// Split-K slices that launch_gemm_bf16 writes for a request of `splits` over K:
// every slice covers a whole number of 64-wide K blocks and at least one, so
// the count can come out below the request.  A caller that reduces the slices
// must size the reduction with this number.
inline int gemm_splits(int64_t K, int splits) {
  const int64_t nk = (K + 63) / 64;
  int64_t s = splits > 0 ? splits : 1;
  if (s > nk) s = nk > 0 ? nk : 1;
  const int64_t per = nk > 0 ? (nk + s - 1) / s : 1;
  s = nk > 0 ? (nk + per - 1) / per : 1;
  return (int)s;
}
// 16-bit out[i] = R[i] + sum_s parts[s*stride + i] for i < n (n and stride
// multiples of 8, 16-byte aligned; f16 or bf16 R and out)
cudaError_t launch_split_reduce_residual(const float* parts, int splits, int64_t stride, int64_t n, const void* R,
                                         void* out, bool f16, cudaStream_t s);
// fp32 out[i] = sum_s parts[s*stride + i] for i < n
cudaError_t launch_split_reduce(const float* parts, int splits, int64_t stride, int64_t n, float* out,
                                cudaStream_t s);

}  // namespace mtgr
