// norm.cu -- the two row-normalisation steps of the HSTU layer, forward and
// backward.  Both are HBM-bound: one warp streams one row with 16-byte
// vector accesses, statistics are warp-reduced in fp32.
//
//  * Group LayerNorm (fun-rec chapter 7.3, §7.3.3; paper-daily "模型怎么搭"):
//      y = (x - μ)·rstd·γ_g + β_g, statistics per token over D features,
//      γ_g/β_g selected by the token's group id.
//  * Gate (paper-daily "模型怎么搭": normalise the aggregate, multiply by U):
//      Y = LayerNorm(O) ⊙ U over the H·d_h features of a token, no affine
//      (O is fp32 in the fp32 path and f16 in the bf16 path; statistics fp32).
#include <mutex>

#include "common.cuh"

namespace mtgr {

// 8 consecutive elements <-> 8 floats (one 16-byte vector for bf16, two for fp32)
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 r = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = bf16_lo(w[i]);
    v[2 * i + 1] = bf16_hi(w[i]);
  }
}
__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void load8(const __half* p, float (&v)[8]) {
  const uint4 r = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = f16_lo(w[i]);
    v[2 * i + 1] = f16_hi(w[i]);
  }
}
__device__ __forceinline__ void store8(__half* p, const float (&v)[8]) {
  uint4 r;
  r.x = pack_f16x2(v[0], v[1]);
  r.y = pack_f16x2(v[2], v[3]);
  r.z = pack_f16x2(v[4], v[5]);
  r.w = pack_f16x2(v[6], v[7]);
  *reinterpret_cast<uint4*>(p) = r;
}
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&v)[8]) {
  uint4 r;
  r.x = pack_bf16x2(v[0], v[1]);
  r.y = pack_bf16x2(v[2], v[3]);
  r.z = pack_bf16x2(v[4], v[5]);
  r.w = pack_bf16x2(v[6], v[7]);
  *reinterpret_cast<uint4*>(p) = r;
}
__device__ __forceinline__ void store8(float* p, const float (&v)[8]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}

// Lane `lane` owns 8-element chunks c = lane + 32*m (m < NCH) of a row of n features.
#define ROW_CHUNKS_FOR(m, c, lane, n) \
  _Pragma("unroll") for (int m = 0; m < NCH; ++m) if (const int c = (lane) + 32 * m; 8 * c < (n))

// ---------------------------------------------------------------------------
// Group LayerNorm
// ---------------------------------------------------------------------------
// 8 consecutive elements of a row kept in their stored form (one 16-byte
// vector for bf16, two for fp32) and widened to fp32 on use.
template <typename T>
struct Raw8;
template <>
struct Raw8<__nv_bfloat16> {
  uint4 w;
  __device__ __forceinline__ void load(const __nv_bfloat16* p) { w = *reinterpret_cast<const uint4*>(p); }
  __device__ __forceinline__ void get(float (&v)[8]) const {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = bf16_lo(u[i]);
      v[2 * i + 1] = bf16_hi(u[i]);
    }
  }
};
template <>
struct Raw8<__half> {
  uint4 w;
  __device__ __forceinline__ void load(const __half* p) { w = *reinterpret_cast<const uint4*>(p); }
  __device__ __forceinline__ void get(float (&v)[8]) const {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = f16_lo(u[i]);
      v[2 * i + 1] = f16_hi(u[i]);
    }
  }
};
template <>
struct Raw8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float* p) {
    a = *reinterpret_cast<const float4*>(p);
    b = *reinterpret_cast<const float4*>(p + 4);
  }
  __device__ __forceinline__ void get(float (&v)[8]) const {
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
};

// One warp per row, rows strided over the grid.  A row stays in its stored
// form (Raw8) and is widened on each of the three passes (mean, variance,
// output).  For 16-bit rows up to 1024 features the next row's chunks are
// requested before the current row is reduced and written, so each warp keeps
// a row of loads in flight through its whole loop, not only at the top of it.
template <typename T, typename TY, int NCH>
__global__ void __launch_bounds__(256) gln_fwd_kernel(const T* __restrict__ x, TY* __restrict__ y,
                                                      float* __restrict__ mean, float* __restrict__ rstd,
                                                      const uint8_t* __restrict__ gid,
                                                      const float* __restrict__ gamma,
                                                      const float* __restrict__ beta, int64_t rows, int D,
                                                      float eps) {
  constexpr bool PIPE = sizeof(T) == 2 && NCH <= 4;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  Raw8<T> nx[PIPE ? NCH : 1];
  if (PIPE && r < rows) {
    ROW_CHUNKS_FOR(m, c, lane, D) nx[PIPE ? m : 0].load(x + r * D + 8 * c);
  }
  for (; r < rows; r += nwarps) {
    Raw8<T> cur[NCH];
    if constexpr (PIPE) {
#pragma unroll
      for (int m = 0; m < NCH; ++m) cur[m] = nx[m];
      const int64_t rn = r + nwarps;
      if (rn < rows) {
        ROW_CHUNKS_FOR(m, c, lane, D) nx[m].load(x + rn * D + 8 * c);
      }
    } else {
      ROW_CHUNKS_FOR(m, c, lane, D) cur[m].load(x + r * D + 8 * c);
    }
    float s = 0.f;
    ROW_CHUNKS_FOR(m, c, lane, D) {
      float v[8];
      cur[m].get(v);
#pragma unroll
      for (int i = 0; i < 8; ++i) s += v[i];
    }
    const float mu = warp_sum(s) / (float)D;
    float q = 0.f;
    ROW_CHUNKS_FOR(m, c, lane, D) {
      float v[8];
      cur[m].get(v);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float d = v[i] - mu;
        q += d * d;
      }
    }
    const float rs = rsqrtf(warp_sum(q) / (float)D + eps);
    const int g = min((int)gid[r], 3);
    ROW_CHUNKS_FOR(m, c, lane, D) {
      float v[8], ga[8], be[8], o[8];
      cur[m].get(v);
      load8(gamma + (int64_t)g * D + 8 * c, ga);
      load8(beta + (int64_t)g * D + 8 * c, be);
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] = (v[i] - mu) * rs * ga[i] + be[i];
      store8(y + r * D + 8 * c, o);
    }
    if (lane == 0) {
      if (mean) mean[r] = mu;
      if (rstd) rstd[r] = rs;
    }
  }
}

// dx = rstd (dŷ - mean(dŷ) - x̂ mean(dŷ x̂)) (+ dres), dŷ = dy ⊙ γ_g, with dy
// read as stored times *dy_scale when dy_scale is given (an upstream gradient
// kept scaled by a power of two);
// per-block sums of dy ⊙ x̂ and dy per group go to `partial`
// ([gridDim.x][2][4][D] fp32), reduced by gln_param_reduce_kernel.
// Each warp takes a contiguous range of rows.  Tokens of a user are sorted by
// group, so the group id changes rarely along the range: for bf16 rows up to
// 1024 features (fp32 up to 512) every lane keeps the sums of its own columns
// in registers and adds them to the block's shared sums only when the group
// changes; for wider rows the registers do not suffice and every row adds
// into the shared sums directly.
template <typename TD, typename T, int NCH>
__global__ void __launch_bounds__(256, NCH * sizeof(T) <= 8 ? 2 : 1)
    gln_bwd_kernel(const TD* __restrict__ dy, const T* __restrict__ x, const float* __restrict__ mean,
                   const float* __restrict__ rstd, const uint8_t* __restrict__ gid, const float* __restrict__ gamma,
                   const T* __restrict__ dres, T* __restrict__ dx, float* __restrict__ partial, int64_t rows,
                   int D, int stage_dres, const float* __restrict__ dy_scale) {
  const float dsc = dy_scale ? *dy_scale : 1.f;
  constexpr bool REG = NCH * sizeof(T) <= 8;  // bf16 rows up to 1024, fp32 rows up to 512
  extern __shared__ float acc[];  // [2][4][D], then one dres row per warp
  for (int i = threadIdx.x; i < 8 * D; i += blockDim.x) acc[i] = 0.f;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  // the row's dres is requested with its x and dy (cp.async into the warp's
  // slot; each lane copies and later reads only its own chunks), so one HBM
  // round trip per row remains on the warp's path instead of two; without
  // room for the slots (fp32 rows above 2048) dres is loaded where it is used
  const bool staged = dres != nullptr && stage_dres != 0;
  uint8_t* dstage = reinterpret_cast<uint8_t*>(acc + 8 * D) + (threadIdx.x >> 5) * (D * (int)sizeof(T));
  const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t per = (rows + nw - 1) / nw;
  const int64_t r0 = w * per, r1 = r0 + per < rows ? r0 + per : rows;
  float sg[REG ? NCH : 1][8], sb[REG ? NCH : 1][8];  // Σ dy x̂, Σ dy of the current group
  if constexpr (REG) {
#pragma unroll
    for (int m = 0; m < NCH; ++m)
#pragma unroll
      for (int i = 0; i < 8; ++i) sg[m][i] = sb[m][i] = 0.f;
  }
  int gcur = -1;
  auto flush = [&]() {
    if constexpr (REG) {
      ROW_CHUNKS_FOR(m, c, lane, D) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          atomicAdd(&acc[gcur * D + 8 * c + i], sg[m][i]);
          atomicAdd(&acc[(4 + gcur) * D + 8 * c + i], sb[m][i]);
          sg[m][i] = sb[m][i] = 0.f;
        }
      }
    }
  };
  for (int64_t r = r0; r < r1; ++r) {
    const int g = min((int)gid[r], 3);
    if (g != gcur) {
      if (gcur >= 0) flush();
      gcur = g;
    }
    if (staged) {
      ROW_CHUNKS_FOR(m, c, lane, D) {
#pragma unroll
        for (int q = 0; q < (int)sizeof(T) / 2; ++q)
          cp_async16(smem_u32(dstage + 8 * c * sizeof(T) + 16 * q), dres + r * D + 8 * c + q * (16 / sizeof(T)));
      }
      cp_async_commit();
    }
    const float mu = mean[r], rs = rstd[r];
    Raw8<T> xr[NCH];
    Raw8<TD> dr[NCH];
    ROW_CHUNKS_FOR(m, c, lane, D) {
      xr[m].load(x + r * D + 8 * c);
      dr[m].load(dy + r * D + 8 * c);
    }
    float s1 = 0.f, s2 = 0.f;
    ROW_CHUNKS_FOR(m, c, lane, D) {
      float xv[8], dv[8], ga[8];
      xr[m].get(xv);
      dr[m].get(dv);
#pragma unroll
      for (int i = 0; i < 8; ++i) dv[i] *= dsc;
      load8(gamma + (int64_t)g * D + 8 * c, ga);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float xh = (xv[i] - mu) * rs, gy = dv[i] * ga[i];
        s1 += gy;
        s2 += gy * xh;
        if constexpr (REG) {
          sg[m][i] += dv[i] * xh;
          sb[m][i] += dv[i];
        } else {
          atomicAdd(&acc[g * D + 8 * c + i], dv[i] * xh);
          atomicAdd(&acc[(4 + g) * D + 8 * c + i], dv[i]);
        }
      }
    }
    const float m1 = warp_sum(s1) / (float)D, m2 = warp_sum(s2) / (float)D;
    if (staged) cp_async_wait<0>();
    ROW_CHUNKS_FOR(m, c, lane, D) {
      float xv[8], dv[8], ga[8], o[8];
      xr[m].get(xv);
      dr[m].get(dv);
#pragma unroll
      for (int i = 0; i < 8; ++i) dv[i] *= dsc;
      load8(gamma + (int64_t)g * D + 8 * c, ga);
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] = rs * (dv[i] * ga[i] - m1 - (xv[i] - mu) * rs * m2);
      if (dres) {
        float rv[8];
        if (staged)
          load8(reinterpret_cast<const T*>(dstage + 8 * c * sizeof(T)), rv);
        else
          load8(dres + r * D + 8 * c, rv);
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] += rv[i];
      }
      store8(dx + r * D + 8 * c, o);
    }
  }
  if (gcur >= 0) flush();
  __syncthreads();
  float* out = partial + (int64_t)blockIdx.x * 8 * D;
  for (int i = threadIdx.x; i < 8 * D; i += blockDim.x) out[i] = acc[i];
}

// dgamma[g][f] / dbeta[g][f] = sum over blocks of the partials (fixed order).
__global__ void gln_param_reduce_kernel(const float* __restrict__ partial, int nblocks, int D,
                                        float* __restrict__ dgamma, float* __restrict__ dbeta) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;  // over [2][4][D]
  if (i >= 8 * D) return;
  float s = 0.f;
  for (int b = 0; b < nblocks; ++b) s += partial[(int64_t)b * 8 * D + i];
  if (i < 4 * D)
    dgamma[i] = s;
  else
    dbeta[i - 4 * D] = s;
}

// ---------------------------------------------------------------------------
// Gate: Y = LayerNorm(O) ⊙ U
// ---------------------------------------------------------------------------
template <typename TOi, typename TU, typename TY, int NCH>
__global__ void __launch_bounds__(256) ln_gate_fwd_kernel(const TOi* __restrict__ O, const TU* __restrict__ U,
                                                          int64_t ldu, TY* __restrict__ Y,
                                                          float* __restrict__ mean, float* __restrict__ rstd,
                                                          int64_t rows, int n, float eps,
                                                          const float* __restrict__ opart, int64_t pstride,
                                                          TOi* __restrict__ o_out) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += nwarps) {
    float v[NCH][8];
    float s = 0.f;
    ROW_CHUNKS_FOR(m, c, lane, n) {
      if (opart) {
        // O = the two key halves' fp32 partial sums, rounded to O's stored type
        // (and stored) before the statistics, as an unsplit forward stores it
        const float4* pa = reinterpret_cast<const float4*>(opart + r * n + 8 * c);
        const float4* pb = reinterpret_cast<const float4*>(opart + pstride + r * n + 8 * c);
        const float4 a0 = pa[0], a1 = pa[1], b0 = pb[0], b1 = pb[1];
        const float t[8] = {a0.x + b0.x, a0.y + b0.y, a0.z + b0.z, a0.w + b0.w,
                            a1.x + b1.x, a1.y + b1.y, a1.z + b1.z, a1.w + b1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) v[m][i] = to_f32<TOi>(from_f32<TOi>(t[i]));
        store8(o_out + r * n + 8 * c, v[m]);
      } else {
        load8(O + r * n + 8 * c, v[m]);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) s += v[m][i];
    }
    const float mu = warp_sum(s) / (float)n;
    float q = 0.f;
    ROW_CHUNKS_FOR(m, c, lane, n) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float d = v[m][i] - mu;
        q += d * d;
      }
    }
    const float rs = rsqrtf(warp_sum(q) / (float)n + eps);
    ROW_CHUNKS_FOR(m, c, lane, n) {
      float u[8], o[8];
      load8(U + r * ldu + 8 * c, u);
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] = (v[m][i] - mu) * rs * u[i];
      store8(Y + r * n + 8 * c, o);
    }
    if (lane == 0) {
      mean[r] = mu;
      rstd[r] = rs;
    }
  }
}

// dO = rstd (g - mean(g) - ô mean(g ô)), g = dY ⊙ U;  dU = dY ⊙ ô (⊙ dsilu when given: silu'(z_u)).
template <typename TD, typename TG, typename TOi, typename TU, typename TO, int NCH>
__global__ void __launch_bounds__(256) ln_gate_bwd_kernel(const TD* __restrict__ dY, const TOi* __restrict__ O,
                                                          const TU* __restrict__ U, int64_t ldu,
                                                          const float* __restrict__ mean,
                                                          const float* __restrict__ rstd, TO* __restrict__ dO,
                                                          TG* __restrict__ dU, int64_t ldg,
                                                          const TG* __restrict__ dsilu, int64_t rows, int n) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += nwarps) {
    const float mu = mean[r], rs = rstd[r];
    float oh[NCH][8], g[NCH][8];
    float s1 = 0.f, s2 = 0.f;
    ROW_CHUNKS_FOR(m, c, lane, n) {
      float ov[8], dv[8], uv[8], du[8];
      load8(O + r * n + 8 * c, ov);
      load8(dY + r * n + 8 * c, dv);
      load8(U + r * ldu + 8 * c, uv);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        oh[m][i] = (ov[i] - mu) * rs;
        g[m][i] = dv[i] * uv[i];
        s1 += g[m][i];
        s2 += g[m][i] * oh[m][i];
        du[i] = dv[i] * oh[m][i];
      }
      if (dsilu) {
        float mv[8];
        load8(dsilu + r * ldg + 8 * c, mv);
#pragma unroll
        for (int i = 0; i < 8; ++i) du[i] *= mv[i];
      }
      store8(dU + r * ldg + 8 * c, du);
    }
    const float m1 = warp_sum(s1) / (float)n, m2 = warp_sum(s2) / (float)n;
    ROW_CHUNKS_FOR(m, c, lane, n) {
      float o[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] = rs * (g[m][i] - m1 - oh[m][i] * m2);
      store8(dO + r * n + 8 * c, o);
    }
  }
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------
static int row_blocks(int64_t rows) {
  const int64_t want = (rows + 7) / 8;
  const int64_t cap = (int64_t)num_sms() * 16;
  return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

#define NCH_DISPATCH(n, KERNEL_CALL)                   \
  do {                                                 \
    const int nch__ = ((n) + 255) / 256;               \
    if (nch__ <= 1) {                                  \
      constexpr int NCHV = 1;                          \
      KERNEL_CALL;                                     \
    } else if (nch__ <= 2) {                           \
      constexpr int NCHV = 2;                          \
      KERNEL_CALL;                                     \
    } else if (nch__ <= 4) {                           \
      constexpr int NCHV = 4;                          \
      KERNEL_CALL;                                     \
    } else if (nch__ <= 8) {                           \
      constexpr int NCHV = 8;                          \
      KERNEL_CALL;                                     \
    } else {                                           \
      constexpr int NCHV = 16;                         \
      KERNEL_CALL;                                     \
    }                                                  \
  } while (0)

template <typename T, typename TY>
cudaError_t launch_gln_fwd(const T* x, TY* y, float* mean, float* rstd, const uint8_t* gid, const float* gamma,
                           const float* beta, int64_t rows, int D, float eps, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  TraceScope tr("gln_fwd", s);
  NCH_DISPATCH(D, (gln_fwd_kernel<T, TY, NCHV><<<row_blocks(rows), 256, 0, s>>>(x, y, mean, rstd, gid, gamma, beta,
                                                                            rows, D, eps)));
  return cudaGetLastError();
}

int gln_bwd_blocks(int64_t rows) {
  const int64_t want = (rows + 7) / 8;
  const int64_t cap = (int64_t)num_sms() * 2;
  return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

template <typename TD, typename T>
cudaError_t launch_gln_bwd(const TD* dy, const T* x, const float* mean, const float* rstd, const uint8_t* gid,
                           const float* gamma, const T* dres, T* dx, float* dgamma, float* dbeta, float* partial,
                           int64_t rows, int D, const float* dy_scale, cudaStream_t s) {
  const int nb = gln_bwd_blocks(rows);
  const size_t stage_bytes = (size_t)8 * D * sizeof(T);  // 8 warps' dres rows
  const int stage = (size_t)8 * D * sizeof(float) + stage_bytes <= 232448 ? 1 : 0;
  const size_t smem = (size_t)8 * D * sizeof(float) + (stage ? stage_bytes : 0);
  {
  TraceScope tr("gln_bwd", s);
  NCH_DISPATCH(D, ({
                 auto k = gln_bwd_kernel<TD, T, NCHV>;
                 cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
                 k<<<nb, 256, smem, s>>>(dy, x, mean, rstd, gid, gamma, dres, dx, partial, rows, D, stage,
                                         dy_scale);
               }));
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  TraceScope tr("gln_param_reduce", s);
  gln_param_reduce_kernel<<<(8 * D + 255) / 256, 256, 0, s>>>(partial, nb, D, dgamma, dbeta);
  return cudaGetLastError();
}

template <typename TOi, typename TU, typename TY>
cudaError_t launch_ln_gate_fwd(const TOi* O, const TU* U, int64_t ldu, TY* Y, float* mean, float* rstd,
                               int64_t rows, int n, float eps, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  TraceScope tr("gate_fwd", s);
  NCH_DISPATCH(n, (ln_gate_fwd_kernel<TOi, TU, TY, NCHV><<<row_blocks(rows), 256, 0, s>>>(
                      O, U, ldu, Y, mean, rstd, rows, n, eps, nullptr, 0, nullptr)));
  return cudaGetLastError();
}

// The gate of a key-split forward: O = opart[0] + opart[1] ([rows, n] fp32 each,
// pstride apart), written to O in f16, then the gate as above.
template <typename TU, typename TY>
cudaError_t launch_ln_gate_fwd_parts(const float* opart, int64_t pstride, __half* O, const TU* U, int64_t ldu, TY* Y,
                                     float* mean, float* rstd, int64_t rows, int n, float eps, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  if (n % 8 != 0 || pstride % 8 != 0) return cudaErrorInvalidValue;
  TraceScope tr("gate_fwd", s);
  NCH_DISPATCH(n, (ln_gate_fwd_kernel<__half, TU, TY, NCHV><<<row_blocks(rows), 256, 0, s>>>(
                      O, U, ldu, Y, mean, rstd, rows, n, eps, opart, pstride, O)));
  return cudaGetLastError();
}

template <typename TD, typename TG, typename TOi, typename TU, typename TO>
cudaError_t launch_ln_gate_bwd(const TD* dY, const TOi* O, const TU* U, int64_t ldu, const float* mean,
                               const float* rstd, TO* dO, TG* dU, int64_t ldg, const TG* dsilu, int64_t rows, int n,
                               cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  TraceScope tr("gate_bwd", s);
  NCH_DISPATCH(n, (ln_gate_bwd_kernel<TD, TG, TOi, TU, TO, NCHV><<<row_blocks(rows), 256, 0, s>>>(
                      dY, O, U, ldu, mean, rstd, dO, dU, ldg, dsilu, rows, n)));
  return cudaGetLastError();
}

// 16-bit copy with a new row stride: dst[r, c] = src[r * lds + c] for c < n (exact
// for bf16 -> f16 when the value lies in the f16 normal range).
template <typename TS, typename TD>
__global__ void convert_rows_kernel(const TS* __restrict__ src, int64_t lds, TD* __restrict__ dst, int64_t ldd,
                                    int64_t rows, int n) {
  const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (i >= rows * n) return;
  const int64_t r = i / n;
  const int c = (int)(i - r * n);
  float v[8];
  load8(src + r * lds + c, v);
  store8(dst + r * ldd + c, v);
}

cudaError_t launch_bf16_to_f16(const __nv_bfloat16* src, int64_t lds, __half* dst, int64_t ldd, int64_t rows,
                               int n, cudaStream_t s) {
  const int64_t n8 = rows * n / 8;
  if (n8 == 0) return cudaSuccess;
  TraceScope tr("to_f16", s);
  convert_rows_kernel<<<(unsigned)((n8 + 255) / 256), 256, 0, s>>>(src, lds, dst, ldd, rows, n);
  return cudaGetLastError();
}

#define INSTANTIATE(T, TY)                                                                                    \
  template cudaError_t launch_gln_fwd<T, TY>(const T*, TY*, float*, float*, const uint8_t*, const float*,       \
                                             const float*, int64_t, int, float, cudaStream_t);                \
  template cudaError_t launch_gln_bwd<TY, T>(const TY*, const T*, const float*, const float*, const uint8_t*,   \
                                             const float*, const T*, T*, float*, float*, float*, int64_t, int,  \
                                             const float*, cudaStream_t);
INSTANTIATE(float, float)
INSTANTIATE(__nv_bfloat16, __nv_bfloat16)
INSTANTIATE(__half, __half)
// the bf16 layer: bf16 x and dx, f16 normalised activations and their gradient
INSTANTIATE(__nv_bfloat16, __half)

using bf16_t = __nv_bfloat16;
// O is fp32 in the fp32 path and f16 in the bf16 path
template cudaError_t launch_ln_gate_fwd<float, float, float>(const float*, const float*, int64_t, float*, float*,
                                                             float*, int64_t, int, float, cudaStream_t);
template cudaError_t launch_ln_gate_fwd<__half, bf16_t, bf16_t>(const __half*, const bf16_t*, int64_t, bf16_t*,
                                                                float*, float*, int64_t, int, float, cudaStream_t);
template cudaError_t launch_ln_gate_fwd<__half, __half, bf16_t>(const __half*, const __half*, int64_t, bf16_t*,
                                                                float*, float*, int64_t, int, float, cudaStream_t);
template cudaError_t launch_ln_gate_fwd<__half, __half, __half>(const __half*, const __half*, int64_t, __half*,
                                                               float*, float*, int64_t, int, float, cudaStream_t);
template cudaError_t launch_ln_gate_fwd_parts<bf16_t, bf16_t>(const float*, int64_t, __half*, const bf16_t*, int64_t,
                                                             bf16_t*, float*, float*, int64_t, int, float,
                                                             cudaStream_t);
template cudaError_t launch_ln_gate_fwd_parts<__half, bf16_t>(const float*, int64_t, __half*, const __half*, int64_t,
                                                             bf16_t*, float*, float*, int64_t, int, float,
                                                             cudaStream_t);
template cudaError_t launch_ln_gate_fwd_parts<__half, __half>(const float*, int64_t, __half*, const __half*, int64_t,
                                                             __half*, float*, float*, int64_t, int, float,
                                                             cudaStream_t);
template cudaError_t launch_ln_gate_bwd<float, float, float, float, float>(const float*, const float*,
                                                                           const float*, int64_t, const float*,
                                                                           const float*, float*, float*, int64_t,
                                                                           const float*, int64_t, int, cudaStream_t);
// standalone attention backward: bf16 dY and U from the caller
template cudaError_t launch_ln_gate_bwd<bf16_t, bf16_t, __half, bf16_t, __half>(
    const bf16_t*, const __half*, const bf16_t*, int64_t, const float*, const float*, __half*, bf16_t*, int64_t,
    const bf16_t*, int64_t, int, cudaStream_t);
// layer backward: f16 dY (the dY GEMM's output) and the f16 U of the UQKV projection
template cudaError_t launch_ln_gate_bwd<__half, __half, __half, __half, __half>(
    const __half*, const __half*, const __half*, int64_t, const float*, const float*, __half*, __half*, int64_t,
    const __half*, int64_t, int, cudaStream_t);

// ---------------------------------------------------------------------------
// f16 copy of an upstream gradient, scaled by a power of two
// ---------------------------------------------------------------------------
// The bf16 layer backward carries its gradients in f16 (11 significand bits);
// f16's range is narrower than bf16's, so the upstream gradient is first scaled
// by s = 2^-e, e = ceil(log2 max|g|), which puts its largest magnitude in
// (1/2, 1] whatever the loss scale (s = 1 for an all-zero or non-finite
// gradient).  The results that leave the layer are multiplied by 1/s.

// max |g| over n bf16 values (n a multiple of 8, 16-byte aligned), as the bit
// pattern of a non-negative bf16 (such patterns order like the values), into
// *out (cleared before).
__global__ void absmax_bf16_kernel(const __nv_bfloat16* __restrict__ g, int64_t n8, unsigned* __restrict__ out) {
  unsigned m = 0;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 w = reinterpret_cast<const uint4*>(g)[i];
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) m = max(m, max(u[k] & 0x7FFFu, (u[k] >> 16) & 0x7FFFu));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0 && m) atomicMax(out, m);
}

// s from the max bits (see above)
__device__ __forceinline__ float grad_scale_from_max(unsigned bits) {
  const float m = __uint_as_float(bits << 16);
  if (!(m > 0.f) || !isfinite(m)) return 1.f;
  int ex;
  const float f = frexpf(m, &ex);  // m = f 2^ex, f in [1/2, 1)
  const int c = f > 0.5f ? ex : ex - 1;  // ceil(log2 m)
  return ldexpf(1.f, -c);
}

// dst (f16) = src (bf16) * s; scale[0] = s, scale[1] = 1/s (written by thread 0).
__global__ void scale_to_f16_kernel(const __nv_bfloat16* __restrict__ src, __half* __restrict__ dst, int64_t n8,
                                    const unsigned* __restrict__ maxbits, float* __restrict__ scale) {
  const float sc = grad_scale_from_max(*maxbits);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    scale[0] = sc;
    scale[1] = 1.f / sc;
  }
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
    float v[8];
    load8(src + 8 * i, v);
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] *= sc;
    store8(dst + 8 * i, v);
  }
}

// n (a multiple of 8) elements; ws_max: one device word; scale: two device floats
cudaError_t launch_grad_to_f16(const __nv_bfloat16* src, __half* dst, int64_t n, unsigned* ws_max, float* scale,
                               cudaStream_t s) {
  TraceScope tr("grad_f16", s);
  cudaError_t e = cudaMemsetAsync(ws_max, 0, sizeof(unsigned), s);
  if (e != cudaSuccess) return e;
  const int64_t n8 = n / 8;
  const int blocks = (int)(n8 / 256 < (int64_t)num_sms() * 8 ? (n8 + 255) / 256 : (int64_t)num_sms() * 8);
  absmax_bf16_kernel<<<blocks > 0 ? blocks : 1, 256, 0, s>>>(src, n8, ws_max);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  scale_to_f16_kernel<<<blocks > 0 ? blocks : 1, 256, 0, s>>>(src, dst, n8, ws_max, scale);
  return cudaGetLastError();
}

}  // namespace mtgr

// ---------------------------------------------------------------------------
// Group LayerNorm backward for callers that cannot allocate device memory
// ---------------------------------------------------------------------------
// Some callers of this library cannot call cudaMalloc at the point where they
// run the backward: a host framework that owns every allocation through its own
// pool, a process whose device memory is fully reserved up front, or code that
// must not allocate inside a latency-critical step.  They also cannot size and
// pass the workspace that mtgr_group_layernorm_bwd needs for its per-block
// partial sums of dγ / dβ.  mtgr_group_layernorm_bwd_noalloc keeps those partial
// sums in the fixed array below instead.
namespace mtgr {

// 10 MiB of fp32 partial sums: 8*D floats per block, so the full grid of two
// blocks per SM of a 148-SM part (296 blocks) fits up to D = 1107
constexpr int64_t kGlnNoAllocFloats = int64_t(10) << 18;
static __device__ __align__(256) float g_gln_noalloc_partial[kGlnNoAllocFloats];

namespace {
// Device address of the array on the current device.  In host code the array's
// name is only a host-side stand-in, so the address is looked up once per device
// with that device current and cached (not valid across cudaDeviceReset).  On
// failure returns nullptr and writes the reason to the library's error message.
float* gln_noalloc_scratch() {
  static std::mutex mu;
  static float* cached[64] = {};
  int dev = 0;
  const cudaError_t eg = cudaGetDevice(&dev);
  if (eg != cudaSuccess) {
    set_error("mtgr_group_layernorm_bwd_noalloc: cudaGetDevice failed: %s", cudaGetErrorString(eg));
    return nullptr;
  }
  if (dev < 0 || dev >= 64) {
    set_error("mtgr_group_layernorm_bwd_noalloc: device index %d is outside the 64 devices it supports", dev);
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(mu);
  if (!cached[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_gln_noalloc_partial);
    if (e != cudaSuccess || p == nullptr) {
      set_error("mtgr_group_layernorm_bwd_noalloc: cudaGetSymbolAddress of the device scratch failed: %s",
                cudaGetErrorString(e));
      return nullptr;
    }
    cached[dev] = static_cast<float*>(p);
  }
  return cached[dev];
}

template <typename T>
cudaError_t launch_gln_bwd_noalloc(const T* dy, const T* x, const float* mean, const float* rstd, const uint8_t* gid,
                                   const float* gamma, const T* dres, T* dx, float* dgamma, float* dbeta,
                                   float* partial, int64_t rows, int D, cudaStream_t s) {
  // each block writes all 8*D of its partial sums, so fewer blocks than the
  // workspace variant may run, but nothing has to be cleared beforehand
  int nb = gln_bwd_blocks(rows);
  const int64_t fit = kGlnNoAllocFloats / (8 * (int64_t)D);
  if (nb > fit) nb = (int)fit;
  const size_t stage_bytes = (size_t)8 * D * sizeof(T);  // 8 warps' dres rows
  const int stage = (size_t)8 * D * sizeof(float) + stage_bytes <= 232448 ? 1 : 0;
  const size_t smem = (size_t)8 * D * sizeof(float) + (stage ? stage_bytes : 0);
  {
    TraceScope tr("gln_bwd", s);
    NCH_DISPATCH(D, ({
                   auto k = gln_bwd_kernel<T, T, NCHV>;
                   cudaError_t ea = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
                   if (ea != cudaSuccess) return ea;
                   k<<<nb, 256, smem, s>>>(dy, x, mean, rstd, gid, gamma, dres, dx, partial, rows, D, stage,
                                           nullptr);
                 }));
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  TraceScope tr("gln_param_reduce", s);
  gln_param_reduce_kernel<<<(8 * D + 255) / 256, 256, 0, s>>>(partial, nb, D, dgamma, dbeta);
  return cudaGetLastError();
}
}  // namespace
}  // namespace mtgr

extern "C" MTGR_API mtgr_status mtgr_group_layernorm_bwd_noalloc(const void* dy, const void* x, const float* mean,
                                                                 const float* rstd, const uint8_t* gid,
                                                                 const float* gamma, const void* dx_residual,
                                                                 void* dx, float* dgamma, float* dbeta, int64_t T,
                                                                 int32_t D, mtgr_dtype dtype, mtgr_stream_t stream) {
  using namespace mtgr;
  auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!(T >= 0 && D > 0 && D % 8 == 0)) {
    set_error("mtgr_group_layernorm_bwd_noalloc: D must be a positive multiple of 8 and T >= 0");
    return MTGR_ERR_UNSUPPORTED;
  }
  if (D > 4096) {
    set_error("mtgr_group_layernorm_bwd_noalloc: D = %d is above its maximum of 4096 (fixed 10 MiB device scratch)",
              (int)D);
    return MTGR_ERR_UNSUPPORTED;
  }
  if (dtype != MTGR_F32 && dtype != MTGR_BF16) {
    set_error("mtgr_group_layernorm_bwd_noalloc: %s", dtype == MTGR_F16 ? "MTGR_F16 is forward-only" : "bad dtype");
    return dtype == MTGR_F16 ? MTGR_ERR_UNSUPPORTED : MTGR_ERR_INVALID_ARG;
  }
  if (!dgamma || !dbeta || (T > 0 && !(dy && x && mean && rstd && gid && gamma && dx))) {
    set_error("mtgr_group_layernorm_bwd_noalloc: NULL pointer");
    return MTGR_ERR_INVALID_ARG;
  }
  if (!(a16(dy) && a16(x) && a16(dx) && a16(gamma) && a16(dx_residual))) {
    set_error("mtgr_group_layernorm_bwd_noalloc: tensors must be 16-byte aligned");
    return MTGR_ERR_INVALID_ARG;
  }
  float* partial = gln_noalloc_scratch();
  if (!partial) return MTGR_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e =
      dtype == MTGR_BF16
          ? launch_gln_bwd_noalloc(static_cast<const __nv_bfloat16*>(dy), static_cast<const __nv_bfloat16*>(x), mean,
                                   rstd, gid, gamma, static_cast<const __nv_bfloat16*>(dx_residual),
                                   static_cast<__nv_bfloat16*>(dx), dgamma, dbeta, partial, T, D, s)
          : launch_gln_bwd_noalloc(static_cast<const float*>(dy), static_cast<const float*>(x), mean, rstd, gid,
                                   gamma, static_cast<const float*>(dx_residual), static_cast<float*>(dx), dgamma,
                                   dbeta, partial, T, D, s);
  if (e != cudaSuccess) return cuda_status(e, "group_layernorm_bwd_noalloc");
  return MTGR_OK;
}
