// attn_f32.cu -- fp32 CUDA-core path of the HSTU attention core (the
// precision-reference path for small problems; the bf16 path runs on tcgen05).
//
//   s_ij = q_i·k_j / sqrt(d_h);  A_ij = M_ij silu(s_ij) / n_u;  O_i = Σ_j A_ij v_j
// (marovi.ai "Métodos" block formula; paper-daily "模型怎么搭": SiLU attention
// weights, no softmax).  M_ij is evaluated from the user's group boundaries
// and timestamps (fun-rec chapter 7.3, §7.3.4).  One warp owns one (row, head)
// pair; lane l holds features l, l+32, l+64, l+96 of the head.
#include "common.cuh"
#include "plan.cuh"

namespace mtgr {

// Which user owns absolute row t (binary search over the clamped segments).
__device__ __forceinline__ int find_user(const UserInfo* __restrict__ users, int B, int64_t t) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (users[mid].start <= t)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// Mask on segment-relative indices (group order User*, Seq*, RealTime*, Cand*).
__device__ __forceinline__ bool visible_rel(int ri, int rj, const UserInfo& u, int64_t ts_i, int64_t ts_j) {
  if (rj < u.eS) return true;                 // User/Seq key: visible to all
  if (rj < u.eR) {                            // RealTime key
    if (ri < u.eS) return false;              //   User/Seq rows precede the window
    return ri < u.eR ? (ts_j <= ts_i) : (ts_j < ts_i);
  }
  return ri == rj;                            // candidate key: itself only
}

__device__ __forceinline__ float silu_acc(float s) { return s / (1.0f + expf(-s)); }

template <int NV>
__global__ void __launch_bounds__(128) attn_f32_fwd_kernel(const float* __restrict__ q, const float* __restrict__ k,
                                                           const float* __restrict__ v, int64_t ld,
                                                           const UserInfo* __restrict__ users, int B,
                                                           const int64_t* __restrict__ ts, int64_t T, int H,
                                                           int dh, float* __restrict__ O) {
  const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= T * H) return;
  const int64_t i = w / H;
  const int h = (int)(w % H);
  const int b = find_user(users, B, i);
  const UserInfo u = users[b];
  if (i < u.start || i >= u.start + u.n) return;
  const int ri = (int)(i - u.start);
  const float c = rsqrtf((float)dh);
  float qv[NV], acc[NV];
#pragma unroll
  for (int m = 0; m < NV; ++m) {
    const int d = lane + 32 * m;
    qv[m] = d < dh ? q[i * ld + h * dh + d] : 0.f;
    acc[m] = 0.f;
  }
  const int64_t ts_i = ts[i];
  for (int rj = 0; rj < u.n; ++rj) {
    const int64_t j = u.start + rj;
    if (!visible_rel(ri, rj, u, ts_i, (rj >= u.eS && rj < u.eR) ? ts[j] : 0)) continue;
    float s = 0.f;
#pragma unroll
    for (int m = 0; m < NV; ++m) {
      const int d = lane + 32 * m;
      if (d < dh) s += qv[m] * k[j * ld + h * dh + d];
    }
    s = warp_sum(s) * c;
    const float p = silu_acc(s);
#pragma unroll
    for (int m = 0; m < NV; ++m) {
      const int d = lane + 32 * m;
      if (d < dh) acc[m] += p * v[j * ld + h * dh + d];
    }
  }
  const float inv_n = 1.0f / (float)u.nu;
#pragma unroll
  for (int m = 0; m < NV; ++m) {
    const int d = lane + 32 * m;
    if (d < dh) O[i * (int64_t)H * dh + h * dh + d] = acc[m] * inv_n;
  }
}

__device__ __forceinline__ float silu_grad_acc(float z) {
  const float sg = 1.0f / (1.0f + expf(-z));
  return sg * (1.0f + z * (1.0f - sg));
}

// dq_i = Σ_j ds_ij k_j / sqrt(d_h), ds_ij = (dO_i·v_j) silu'(s_ij) / n_u  (row-major pass)
template <int NV>
__global__ void __launch_bounds__(128) attn_f32_bwd_dq_kernel(
    const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v, int64_t ld,
    const float* __restrict__ dO, const UserInfo* __restrict__ users, int B, const int64_t* __restrict__ ts,
    int64_t T, int H, int dh, float* __restrict__ dq, int64_t ldg, const float* __restrict__ mq) {
  const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= T * H) return;
  const int64_t i = w / H;
  const int h = (int)(w % H);
  const int b = find_user(users, B, i);
  const UserInfo u = users[b];
  if (i < u.start || i >= u.start + u.n) return;
  const int ri = (int)(i - u.start);
  const float c = rsqrtf((float)dh);
  const float inv_n = 1.0f / (float)u.nu;
  float qv[NV], gv[NV], acc[NV];
#pragma unroll
  for (int m = 0; m < NV; ++m) {
    const int d = lane + 32 * m;
    qv[m] = d < dh ? q[i * ld + h * dh + d] : 0.f;
    gv[m] = d < dh ? dO[i * (int64_t)H * dh + h * dh + d] : 0.f;
    acc[m] = 0.f;
  }
  const int64_t ts_i = ts[i];
  for (int rj = 0; rj < u.n; ++rj) {
    const int64_t j = u.start + rj;
    if (!visible_rel(ri, rj, u, ts_i, (rj >= u.eS && rj < u.eR) ? ts[j] : 0)) continue;
    float s = 0.f, da = 0.f;
#pragma unroll
    for (int m = 0; m < NV; ++m) {
      const int d = lane + 32 * m;
      if (d < dh) {
        s += qv[m] * k[j * ld + h * dh + d];
        da += gv[m] * v[j * ld + h * dh + d];
      }
    }
    s = warp_sum(s) * c;
    da = warp_sum(da);
    const float ds = da * silu_grad_acc(s) * inv_n * c;
#pragma unroll
    for (int m = 0; m < NV; ++m) {
      const int d = lane + 32 * m;
      if (d < dh) acc[m] += ds * k[j * ld + h * dh + d];
    }
  }
#pragma unroll
  for (int m = 0; m < NV; ++m) {
    const int d = lane + 32 * m;
    if (d < dh) {
      float g = acc[m];
      if (mq) g *= mq[i * ldg + h * dh + d];
      dq[i * ldg + h * dh + d] = g;
    }
  }
}

// dk_j = Σ_i ds_ij q_i / sqrt(d_h);  dv_j = Σ_i A_ij dO_i  (key-major pass)
template <int NV>
__global__ void __launch_bounds__(128) attn_f32_bwd_dkdv_kernel(
    const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v, int64_t ld,
    const float* __restrict__ dO, const UserInfo* __restrict__ users, int B, const int64_t* __restrict__ ts,
    int64_t T, int H, int dh, float* __restrict__ dk, float* __restrict__ dv, int64_t ldg,
    const float* __restrict__ mk, const float* __restrict__ mv) {
  const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= T * H) return;
  const int64_t j = w / H;
  const int h = (int)(w % H);
  const int b = find_user(users, B, j);
  const UserInfo u = users[b];
  if (j < u.start || j >= u.start + u.n) return;
  const int rj = (int)(j - u.start);
  const float c = rsqrtf((float)dh);
  const float inv_n = 1.0f / (float)u.nu;
  float kv[NV], vv[NV], ak[NV], av[NV];
#pragma unroll
  for (int m = 0; m < NV; ++m) {
    const int d = lane + 32 * m;
    kv[m] = d < dh ? k[j * ld + h * dh + d] : 0.f;
    vv[m] = d < dh ? v[j * ld + h * dh + d] : 0.f;
    ak[m] = 0.f;
    av[m] = 0.f;
  }
  const int64_t ts_j = (rj >= u.eS && rj < u.eR) ? ts[j] : 0;
  for (int ri = 0; ri < u.n; ++ri) {
    const int64_t i = u.start + ri;
    if (!visible_rel(ri, rj, u, (rj >= u.eS && rj < u.eR) ? ts[i] : 0, ts_j)) continue;
    float s = 0.f, da = 0.f;
#pragma unroll
    for (int m = 0; m < NV; ++m) {
      const int d = lane + 32 * m;
      if (d < dh) {
        s += q[i * ld + h * dh + d] * kv[m];
        da += dO[i * (int64_t)H * dh + h * dh + d] * vv[m];
      }
    }
    s = warp_sum(s) * c;
    da = warp_sum(da);
    const float a = silu_acc(s) * inv_n;
    const float ds = da * silu_grad_acc(s) * inv_n * c;
#pragma unroll
    for (int m = 0; m < NV; ++m) {
      const int d = lane + 32 * m;
      if (d < dh) {
        ak[m] += ds * q[i * ld + h * dh + d];
        av[m] += a * dO[i * (int64_t)H * dh + h * dh + d];
      }
    }
  }
#pragma unroll
  for (int m = 0; m < NV; ++m) {
    const int d = lane + 32 * m;
    if (d < dh) {
      float gk = ak[m], gv = av[m];
      if (mk) gk *= mk[j * ldg + h * dh + d];
      if (mv) gv *= mv[j * ldg + h * dh + d];
      dk[j * ldg + h * dh + d] = gk;
      dv[j * ldg + h * dh + d] = gv;
    }
  }
}

cudaError_t launch_attn_f32_fwd(const float* q, const float* k, const float* v, int64_t ld, const UserInfo* users,
                                int B, const int64_t* ts, int64_t T, int H, int dh, float* O, cudaStream_t s) {
  if (T == 0 || B == 0) return cudaSuccess;
  const int64_t warps = T * H;
  const int blocks = (int)((warps * 32 + 127) / 128);
  TraceScope tr("attn_f32_fwd", s);
  if (dh <= 64)
    attn_f32_fwd_kernel<2><<<blocks, 128, 0, s>>>(q, k, v, ld, users, B, ts, T, H, dh, O);
  else
    attn_f32_fwd_kernel<4><<<blocks, 128, 0, s>>>(q, k, v, ld, users, B, ts, T, H, dh, O);
  return cudaGetLastError();
}

cudaError_t launch_attn_f32_bwd(const float* q, const float* k, const float* v, int64_t ld, const float* dO,
                                const UserInfo* users, int B, const int64_t* ts, int64_t T, int H, int dh,
                                float* dq, float* dk, float* dv, int64_t ldg, const float* mq, const float* mk,
                                const float* mv, cudaStream_t s) {
  if (T == 0 || B == 0) return cudaSuccess;
  const int64_t warps = T * H;
  const int blocks = (int)((warps * 32 + 127) / 128);
  TraceScope tr("attn_f32_bwd", s);
  if (dh <= 64) {
    attn_f32_bwd_dq_kernel<2><<<blocks, 128, 0, s>>>(q, k, v, ld, dO, users, B, ts, T, H, dh, dq, ldg, mq);
    attn_f32_bwd_dkdv_kernel<2><<<blocks, 128, 0, s>>>(q, k, v, ld, dO, users, B, ts, T, H, dh, dk, dv, ldg, mk, mv);
  } else {
    attn_f32_bwd_dq_kernel<4><<<blocks, 128, 0, s>>>(q, k, v, ld, dO, users, B, ts, T, H, dh, dq, ldg, mq);
    attn_f32_bwd_dkdv_kernel<4><<<blocks, 128, 0, s>>>(q, k, v, ld, dO, users, B, ts, T, H, dh, dk, dv, ldg, mk, mv);
  }
  return cudaGetLastError();
}

}  // namespace mtgr
