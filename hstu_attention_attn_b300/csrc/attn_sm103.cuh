// attn_sm103.cuh -- device helpers shared by the tcgen05 attention kernels
// (forward, dK/dV backward, dQ backward): shared-memory operand descriptors of
// the 128-row tiles, the persistent item order, SiLU in tanh form and the
// coalesced bf16 row store through a small per-warp staging buffer.
#pragma once
#include "common.cuh"
#include "plan.cuh"

namespace mtgr {
namespace attn {

constexpr int BT = 128;  // rows of every query / key tile

// Shared-memory descriptors of a [128 rows][D] 16-bit tile staged as D/64
// TMA boxes of [128][64] with 128-byte swizzle (16 KB per box).
// K-major use (the reduction runs along the D columns), k-step kk of 16:
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile, int kk) {
  return smem_desc_sw128(tile + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
}
// MN-major use (the reduction runs along the 128 rows), k-step kk of 16 rows:
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t tile, int kk) {
  return smem_desc_sw128(tile + kk * 2048, 16384, 1024);
}

// TMEM column (relative to the 128-column region of a score tile) of the
// packed f16 operand for reduction step kk (rows/keys 16kk .. 16kk+15), when
// the epilogue writes the 8 packed words of every 16-column chunk into the
// first 8 columns of that chunk (so that no warp overwrites columns another
// warp has yet to read).
__device__ __forceinline__ uint32_t packed_col(int kk) { return (uint32_t)(16 * kk); }

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

// ---------------------------------------------------------------------------
// Packed arithmetic of the score epilogues: two scores per instruction.  A
// tcgen05.ld leaves the fp32 scores of consecutive columns in consecutive
// registers; f32x2 operations (sm_100+) scale a pair at once, the pair is
// rounded to one f16x2 word, and tanh.approx.f16x2 evaluates both hyperbolic
// tangents in one MUFU operation, so a pair of scores costs one transcendental
// instead of two.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t f32x2(uint32_t lo_bits, uint32_t hi_bits) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo_bits), "r"(hi_bits));
  return r;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// (a.lo, a.hi) -> one f16x2 word, element 0 in the low half
__device__ __forceinline__ uint32_t cvt_f16x2(uint64_t a) {
  uint32_t lo, hi, r;
  asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(a));
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(__uint_as_float(hi)), "f"(__uint_as_float(lo)));
  return r;
}
__device__ __forceinline__ uint32_t tanh_h2(uint32_t x) {
  uint32_t y;
  asm("tanh.approx.f16x2 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
constexpr uint32_t kH2Half = 0x38003800u;      // (0.5, 0.5) in f16x2
constexpr uint32_t kH2MinusHalf = 0xB800B800u; // (-0.5, -0.5)

// For two raw scores s (fp32 bits) and hs2 = (c/2, c/2) as f32x2 (c the score
// scale): h = c s / 2 as f16x2, and silu(c s) = h + h tanh(h) as f16x2.
__device__ __forceinline__ uint32_t silu_pair(uint32_t s0, uint32_t s1, uint64_t hs2, uint32_t& h, uint32_t& t) {
  h = cvt_f16x2(mul_f32x2(f32x2(s0, s1), hs2));
  t = tanh_h2(h);
  return hfma2(h, t, h);
}
// With t = tanh(h) and the pair's silu: silu' = σ + silu (1 - σ), σ = (1 + t)/2.
__device__ __forceinline__ uint32_t dsilu_pair(uint32_t silu, uint32_t t) {
  const uint32_t sg = hfma2(t, kH2Half, kH2Half);
  const uint32_t omsg = hfma2(t, kH2MinusHalf, kH2Half);
  return hfma2(silu, omsg, sg);
}
// 32-bit mask word keeping element 0 (low half) and/or element 1 (high half)
__device__ __forceinline__ uint32_t keep_mask(bool v0, bool v1) {
  return (v0 ? 0x0000FFFFu : 0u) | (v1 ? 0xFFFF0000u : 0u);
}

// For h = x/2: silu(x) and silu'(x) = σ(x)(1 + x(1 - σ(x))) = σ + silu (1 - σ).
__device__ __forceinline__ void silu_and_grad_half(float h, float& silu, float& dsilu) {
  const float t = tanh_approx(h);
  const float sg = fmaf(0.5f, t, 0.5f);
  silu = fmaf(h, t, h);
  dsilu = fmaf(silu, 1.0f - sg, sg);
}

// A warp holds 32 consecutive rows (lane = row) x 32 values; write them as
// the 16-bit type TG to rows row0 .. row0+31 of out (row stride ld elements),
// skipping rows >= nvalid, through a 2 KB staging buffer so that each store
// instruction writes 8 rows x 64 contiguous bytes.
template <typename TG>
__device__ __forceinline__ void store_rows16_32(const float (&x)[32], uint8_t* stg, TG* out, int64_t ld, int nvalid,
                                                int lane) {
  __syncwarp();
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    uint4 w;
    w.x = pack2<TG>(x[8 * v + 0], x[8 * v + 1]);
    w.y = pack2<TG>(x[8 * v + 2], x[8 * v + 3]);
    w.z = pack2<TG>(x[8 * v + 4], x[8 * v + 5]);
    w.w = pack2<TG>(x[8 * v + 6], x[8 * v + 7]);
    *reinterpret_cast<uint4*>(stg + lane * 64 + ((v ^ ((lane >> 1) & 3)) * 16)) = w;
  }
  __syncwarp();
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int r = it * 8 + (lane >> 2), c4 = lane & 3;
    const uint4 w = *reinterpret_cast<const uint4*>(stg + r * 64 + ((c4 ^ ((r >> 1) & 3)) * 16));
    if (r < nvalid) *reinterpret_cast<uint4*>(out + (int64_t)r * ld + c4 * 8) = w;
  }
}

// ---------------------------------------------------------------------------
// Multiplier chunks of an output warp, fetched ahead of use.  The output warps
// may multiply each [32 rows][32 columns] gradient chunk elementwise by the
// same block of a 16-bit multiplier (the layer passes silu'(z) of its UQKV
// projection); a plain per-chunk load would put one HBM round trip per chunk
// on the path that frees the TMEM accumulators, so the chunks go through a
// ring of MRING shared slots (2 KB each, rows of 64 bytes with the 16-byte
// pieces XOR-swizzled by (row >> 1) & 3, conflict-free for both the coalesced
// fill and the row-per-lane read) filled with cp.async.
// ---------------------------------------------------------------------------
constexpr int MRING = 3;
constexpr int MSLOT = 2048;

// Copy rows 0 .. nvalid-1 (at most 32) of a [32][32] 16-bit block (row stride
// ld elements) into a ring slot; one commit group per call is left to the caller.
__device__ __forceinline__ void mslot_fetch(uint8_t* slot, const uint16_t* src, int64_t ld, int nvalid, int lane) {
  const uint32_t s = smem_u32(slot);
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int r = it * 8 + (lane >> 2), c4 = lane & 3;
    if (r < nvalid) cp_async16(s + r * 64 + ((c4 ^ ((r >> 1) & 3)) * 16), src + (int64_t)r * ld + c4 * 8);
  }
}

// x[0..31] *= the 32 multipliers (16-bit type TG) of row `lane` in a ring slot.
template <typename TG>
__device__ __forceinline__ void mul_slot_32(float (&x)[32], const uint8_t* slot, int lane) {
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const uint4 mm = *reinterpret_cast<const uint4*>(slot + lane * 64 + ((v ^ ((lane >> 1) & 3)) * 16));
    const uint32_t w[4] = {mm.x, mm.y, mm.z, mm.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      x[8 * v + 2 * t] *= lo16<TG>(w[t]);
      x[8 * v + 2 * t + 1] *= hi16<TG>(w[t]);
    }
  }
}

}  // namespace attn
}  // namespace mtgr
