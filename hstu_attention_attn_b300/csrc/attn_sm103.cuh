// attn_sm103.cuh -- device helpers shared by the tcgen05 attention kernels
// (forward, dK/dV backward, dQ backward): shared-memory operand descriptors of
// the 128-row tiles, the persistent item order, SiLU in tanh form and its
// packed fp32-pair evaluation.
#pragma once
#include "common.cuh"
#include "plan.cuh"

namespace mtgr {
namespace attn {

constexpr int BT = 128;  // rows of every query / key tile

// Shared-memory descriptors of a [128 rows][D] 16-bit tile staged as D/64
// TMA boxes of [128][64] with 128-byte swizzle (16 KB per box), as 32-bit
// halves: K-major use (the reduction runs along the D columns, k-step kk of 16
// at byte offset (kk/4)*16384 + (kk%4)*32) and MN-major use (the reduction runs
// along the 128 rows, k-step kk at kk*2048, 64-element MN blocks 16 KB apart).
// An issue loop spends one add per operand per MMA (the MMA warp shares its
// sub-partition with epilogue warps, so every instruction of the issue loop
// competes for issue slots): the base of a tile, plus the low-half step of
// k-step kk.
__device__ __forceinline__ SmemDesc kmajor_base(uint32_t tile) { return smem_desc_sw128_h(tile, 16, 1024); }
__device__ __forceinline__ SmemDesc mnmajor_base(uint32_t tile) { return smem_desc_sw128_h(tile, 16384, 1024); }
__host__ __device__ constexpr uint32_t kmajor_step(int kk) { return (uint32_t)((kk >> 2) * 1024 + (kk & 3) * 2); }
__host__ __device__ constexpr uint32_t mnmajor_step(int kk) { return (uint32_t)(kk * 128); }

// 64-bit warp broadcast from lane src.
__device__ __forceinline__ int64_t shfl_i64(int64_t v, int src) {
  const int lo = __shfl_sync(0xffffffffu, (int)(uint32_t)(uint64_t)v, src);
  const int hi = __shfl_sync(0xffffffffu, (int)(uint32_t)((uint64_t)v >> 32), src);
  return (int64_t)(((uint64_t)(uint32_t)hi << 32) | (uint64_t)(uint32_t)lo);
}

// Stamps of 16 keys j0 .. j0+15 for the RealTime test, one per lane (lane & 15):
// the key's stamp when it is a RealTime key of the segment, else INT64_MAX
// (never visible through the stamp test).  Read back with shfl_i64(.., e).
__device__ __forceinline__ int64_t rt_key_stamp(const UserInfo& u, const int64_t* ts_u, int j0, int lane) {
  const int j = j0 + (lane & 15);
  return (j >= u.eS && j < u.eR) ? __ldg(ts_u + j) : INT64_MAX;
}

// Persistent item order of one CTA: rounds of gridDim.x items, serpentine so
// that a longest-first list is dealt out evenly.
__device__ __forceinline__ int item_at(int round) {
  const int G = gridDim.x, c = blockIdx.x;
  return round * G + ((round & 1) ? (G - 1 - c) : c);
}

// silu(x) with h = x/2: h + h tanh(h)  (σ(x) = (1 + tanh(x/2)) / 2)
__device__ __forceinline__ float silu_half(float h) { return fmaf(h, tanh_approx(h), h); }

// For h = x/2: silu(x) and silu'(x) = σ(x)(1 + x(1 - σ(x))) = σ + silu (1 - σ).
__device__ __forceinline__ void silu_and_grad_half(float h, float& silu, float& dsilu) {
  const float t = tanh_approx(h);
  const float sg = fmaf(0.5f, t, 0.5f);
  silu = fmaf(h, t, h);
  dsilu = fmaf(silu, 1.0f - sg, sg);
}

// ---------------------------------------------------------------------------
// Packed fp32 pairs (f32x2 arithmetic, sm_100+): two scores per instruction
// for everything but the transcendental, which stays one tanh.approx.f32 per
// score (its f16x2 form evaluates no faster).  A tcgen05.ld leaves the scores
// of consecutive columns in consecutive registers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t f2(uint32_t lo, uint32_t hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}
__device__ __forceinline__ void unf2(uint64_t v, uint32_t& lo, uint32_t& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint32_t pack_f16x2_2(uint64_t v) {
  uint32_t lo, hi;
  unf2(v, lo, hi);
  return pack_f16x2(__uint_as_float(lo), __uint_as_float(hi));
}
// In two steps, for an epilogue that has the scores before dP: from raw scores
// s0, s1 (fp32 bits) and hc2 = (c/2, c/2) the packed f16 pairs silu(c s) and
// silu'(c s) = σ + silu (1 - σ), σ = (1 + tanh(c s / 2)) / 2; later, with dp,
// the packed f16 pair silu' dp.
__device__ __forceinline__ void silu_pair_split(uint32_t s0, uint32_t s1, uint64_t hc2, uint32_t& p, uint32_t& dsl16) {
  const uint64_t h = mul2(f2(s0, s1), hc2);
  uint32_t h0, h1;
  unf2(h, h0, h1);
  const uint64_t t = f2(__float_as_uint(tanh_approx(__uint_as_float(h0))), __float_as_uint(tanh_approx(__uint_as_float(h1))));
  const uint64_t half = f2(0x3F000000u, 0x3F000000u), mhalf = f2(0xBF000000u, 0xBF000000u);
  const uint64_t sg = fma2(t, half, half);
  const uint64_t sl = fma2(h, t, h);
  const uint64_t omsg = fma2(t, mhalf, half);
  p = pack_f16x2_2(sl);
  dsl16 = pack_f16x2_2(fma2(sl, omsg, sg));
}
// silu'(c s) alone, as a packed f16 pair
__device__ __forceinline__ uint32_t dsilu_pair(uint32_t s0, uint32_t s1, uint64_t hc2) {
  const uint64_t h = mul2(f2(s0, s1), hc2);
  uint32_t h0, h1;
  unf2(h, h0, h1);
  const uint64_t t = f2(__float_as_uint(tanh_approx(__uint_as_float(h0))), __float_as_uint(tanh_approx(__uint_as_float(h1))));
  const uint64_t half = f2(0x3F000000u, 0x3F000000u), mhalf = f2(0xBF000000u, 0xBF000000u);
  const uint64_t sg = fma2(t, half, half);
  const uint64_t sl = fma2(h, t, h);
  const uint64_t omsg = fma2(t, mhalf, half);
  return pack_f16x2_2(fma2(sl, omsg, sg));
}
__device__ __forceinline__ uint32_t ds_pair(uint32_t dsl16, uint32_t dp0, uint32_t dp1) {
  const uint64_t d = f2(__float_as_uint(f16_lo(dsl16)), __float_as_uint(f16_hi(dsl16)));
  return pack_f16x2_2(mul2(d, f2(dp0, dp1)));
}
// 32-bit mask keeping element 0 (low half) and / or element 1 (high half) of a packed f16 pair
__device__ __forceinline__ uint32_t keep_mask(bool v0, bool v1) {
  return (v0 ? 0x0000FFFFu : 0u) | (v1 ? 0xFFFF0000u : 0u);
}

}  // namespace attn
}  // namespace mtgr
