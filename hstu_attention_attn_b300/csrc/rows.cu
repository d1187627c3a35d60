// rows.cu -- row scatter for sparse upstream gradients: a loss on the
// candidate tokens only (fun-rec §7.3.1: each candidate is scored from its own
// position) leaves dx' zero on every other row, so a training step moves only
// the candidates' rows to the GPU and expands them here.
#include "common.cuh"

namespace mtgr {

// one warp per source row, 16-byte vectors; rows outside [0, T) are skipped
__global__ void __launch_bounds__(256) expand_rows_kernel(const uint4* __restrict__ src,
                                                          const int32_t* __restrict__ rows, int64_t n,
                                                          uint4* __restrict__ dst, int64_t T, int vec_per_row) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t k = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); k < n; k += nwarps) {
    const int64_t r = rows[k];
    if (r < 0 || r >= T) continue;
    for (int c = lane; c < vec_per_row; c += 32) dst[r * vec_per_row + c] = src[k * vec_per_row + c];
  }
}

cudaError_t launch_expand_rows(const void* src, const int32_t* rows, int64_t n, void* dst, int64_t T,
                               int64_t row_bytes, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(dst, 0, (size_t)(T * row_bytes), s);
  if (e != cudaSuccess || n == 0) return e;
  const int64_t want = (n + 7) / 8, cap = (int64_t)num_sms() * 8;
  TraceScope tr("expand_rows", s);
  expand_rows_kernel<<<(unsigned)(want < cap ? want : cap), 256, 0, s>>>(
      static_cast<const uint4*>(src), rows, n, static_cast<uint4*>(dst), T, (int)(row_bytes / 16));
  return cudaGetLastError();
}

}  // namespace mtgr
