// gemm_sm103.cu -- bf16 GEMM on the 5th-generation tensor cores (tcgen05),
// used for the projections of the HSTU layer (UQKV + SiLU, output + residual)
// and their input / weight gradients.
//
// Persistent kernel, one CTA per SM, 128x256 output tiles, 64-deep K blocks:
//   warp 0      TMA producer: A/B tiles into a 4-stage shared-memory ring
//   warp 1      MMA issuer (one elected thread): tcgen05.mma 128x256x16,
//               fp32 accumulator in TMEM, double-buffered (2 x 256 columns)
//   warps 2..5  epilogue: tcgen05.ld -> fused epilogue -> global stores, which
//               overlaps the main loop of the next tile.
// Operands may be K-major or MN-major (a transposed operand needs no copy):
// the tensor-core reads both from the same 128-byte-swizzled staging layout.
#include "common.cuh"
#include "gemm.cuh"

namespace mtgr {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
static_assert(BK == 64, "gemm_splits counts K in blocks of 64");
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int B_BYTES = BN * BK * 2;  // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int ACC_COLS = BN;           // fp32 columns per accumulator
constexpr int TMEM_COLS = 2 * ACC_COLS;
// warp 0 TMA, warp 1 MMA, then 4 epilogue warps (EPI_RESIDUAL) or 8 (two per
// TMEM lane quarter, each draining half of the tile's columns)
constexpr int MAX_THREADS = 320;
// 32 KB of epilogue staging in 2 KB slots (each a [32][32] 16-bit TMA box).
// With 4 epilogue warps each has 8 KB: 2 residual slots + 2 output slots
// (EPI_RESIDUAL).  With 8 warps each has 4 KB: a ring of 2 output slots, or
// one fp32 box of 4 KB (EPI_F32).
constexpr int EP_TOTAL = 32768;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EP_TOTAL + 1024 /*align*/ + 256 /*barriers*/;

struct Smem {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint32_t tmem_base;
  int abort_flag;
};

struct Params {
  int64_t M, N, K;
  int m_tiles, n_tiles, splits, kb_per_split, nk;
  bool a_mn, b_mn;
  bool ab_f16, r_f16, z_f16;
  bool c_f16;
  int epi;
  void* C;
  int64_t ldc;
  const __nv_bfloat16* R;
  int64_t ldr;
  __nv_bfloat16* Z;
  int64_t ldz;
  const float* out_scale;  // EPI_F32: multiply by *out_scale when set
  int32_t* status;
};

// Stage 32 rows x 32 values (lane = row) as 16-bit T in the 64-byte-swizzled
// layout of a [32][32] TMA box and store the box at (x0, y0).
template <typename T>
__device__ __forceinline__ void stage_store16(const float (&x)[32], uint8_t* slot, const CUtensorMap* m, int x0,
                                              int y0, int lane) {
#pragma unroll
  for (int v = 0; v < 4; ++v)
    *reinterpret_cast<uint4*>(slot + lane * 64 + ((v ^ ((lane >> 1) & 3)) * 16)) = pack8<T>(x + 8 * v);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(m, slot, x0, y0);
    tma_store_commit();
  }
}
// fp32: 128-byte rows with the 128-byte swizzle, box [1][32][32] of a 3-D map.
__device__ __forceinline__ void stage_store32(const float (&x)[32], uint8_t* slot, const CUtensorMap* m, int x0,
                                              int y0, int z0, int lane) {
#pragma unroll
  for (int v = 0; v < 8; ++v)
    *reinterpret_cast<float4*>(slot + lane * 128 + ((v ^ (lane & 7)) * 16)) =
        make_float4(x[4 * v], x[4 * v + 1], x[4 * v + 2], x[4 * v + 3]);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_3d(m, slot, x0, y0, z0);
    tma_store_commit();
  }
}
// Before restaging a slot: at most N newer stores of this warp may still be reading theirs.
template <int N>
__device__ __forceinline__ void slot_free(int lane) {
  if (lane == 0) tma_store_wait_read_n<N>();
  __syncwarp();
}

__device__ __forceinline__ void tile_coords(const Params& p, int t, int& split, int& mt, int& nt) {
  const int per_split = p.m_tiles * p.n_tiles;
  split = t / per_split;
  const int r = t - split * per_split;
  mt = r / p.n_tiles;
  nt = r - mt * p.n_tiles;
}

__global__ void __launch_bounds__(MAX_THREADS, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmZ,
                     const Params p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned staging area (128-byte swizzle atoms), then the barriers
  uint8_t* stage_base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ep_base = stage_base + STAGES * STAGE_BYTES;
  Smem& S = *reinterpret_cast<Smem*>(ep_base + EP_TOTAL);
  const int n_epi = (int)(blockDim.x >> 5) - 2;  // 4 or 8
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_tiles = p.splits * p.m_tiles * p.n_tiles;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.acc_full[i], 1);
      mbar_init(&S.acc_empty[i], n_epi);  // one arrival per epilogue warp
    }
    S.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
    tma_prefetch_desc(&tmZ);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  volatile int* abort_flag = &S.abort_flag;
  bool ok = true;

  if (warp == 0) {
    // ---------------- TMA producer (whole warp polls, lane 0 issues) ----------------
    int stage = 0;
    uint32_t phase = 0;
    for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
      int split, mt, nt;
      tile_coords(p, t, split, mt, nt);
      const int kb0 = split * p.kb_per_split;
      const int kb1 = min(kb0 + p.kb_per_split, p.nk);
      const int m0 = mt * BM, n0 = nt * BN;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait_warp(&S.empty[stage], phase ^ 1, abort_flag)) { ok = false; break; }
        if (lane == 0) {
          uint8_t* sa = stage_base + stage * STAGE_BYTES;
          uint8_t* sb = sa + A_BYTES;
          mbar_arrive_expect_tx(&S.full[stage], STAGE_BYTES);
          const int k0 = kb * BK;
          if (!p.a_mn) {
            tma_load_2d(sa, &tmA, &S.full[stage], k0, m0);
          } else {
            tma_load_2d(sa, &tmA, &S.full[stage], m0, k0);
            tma_load_2d(sa + A_BYTES / 2, &tmA, &S.full[stage], m0 + 64, k0);
          }
          if (!p.b_mn) {
            tma_load_2d(sb, &tmB, &S.full[stage], k0, n0);
          } else {
#pragma unroll
            for (int i = 0; i < BN / 64; ++i)
              tma_load_2d(sb + i * (B_BYTES / 4), &tmB, &S.full[stage], n0 + 64 * i, k0);
          }
        }
        __syncwarp();
        if (++stage == STAGES) { stage = 0; phase ^= 1; }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (whole warp polls, lane 0 issues) ----------------
    const uint32_t idesc = p.ab_f16 ? idesc_f16_f32(BM, BN, p.a_mn, p.b_mn) : idesc_bf16_f32(BM, BN, p.a_mn, p.b_mn);
    int stage = 0;
    uint32_t phase = 0;
    int it = 0;
    for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++it) {
      int split, mt, nt;
      tile_coords(p, t, split, mt, nt);
      const int kb0 = split * p.kb_per_split;
      const int kb1 = min(kb0 + p.kb_per_split, p.nk);
      const int buf = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      if (!mbar_wait_warp(&S.acc_empty[buf], acc_phase ^ 1, abort_flag)) { ok = false; break; }
      tc_fence_after();
      const uint32_t d_tmem = tmem + buf * ACC_COLS;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait_warp(&S.full[stage], phase, abort_flag)) { ok = false; break; }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t sa = smem_u32(stage_base + stage * STAGE_BYTES);
          const uint32_t sb = sa + A_BYTES;
          const SmemDesc ad = p.a_mn ? smem_desc_sw128_h(sa, A_BYTES / 2, 1024) : smem_desc_sw128_h(sa, 16, 1024);
          const SmemDesc bd = p.b_mn ? smem_desc_sw128_h(sb, B_BYTES / 4, 1024) : smem_desc_sw128_h(sb, 16, 1024);
          const uint32_t a_step = p.a_mn ? 2048u >> 4 : 32u >> 4, b_step = p.b_mn ? 2048u >> 4 : 32u >> 4;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc_mma_ss_h(d_tmem, ad.lo + kk * a_step, ad.hi, bd.lo + kk * b_step, bd.hi, idesc,
                        (kb > kb0 || kk > 0) ? 1u : 0u);
          tc_commit(&S.empty[stage]);
        }
        __syncwarp();
        if (++stage == STAGES) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
      if (lane == 0) tc_commit(&S.acc_full[buf]);
      __syncwarp();
    }
  } else {
    // ---------------- epilogue (warps 2 .. 2 + n_epi - 1) ----------------
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    const uint32_t lane_sel = (uint32_t)(quarter * 32) << 16;
    const int e = warp - 2;
    const int cpw = (BN / 32) * 4 / n_epi;  // 32-column chunks per warp: 8 or 4
    const int c0 = (e >> 2) * cpw;          // this warp's first chunk of the tile
    // Outputs leave through TMA stores from the warp's staging slots, so the
    // warp never waits on global stores.  Residual chunks (EPI_RESIDUAL, 4
    // epilogue warps) come in through a 2-slot cp.async ring: chunks 0 and 1
    // are requested before the accumulator wait and the rest of the warp's
    // rows of the tile are prefetched into L2, so no chunk waits for a full
    // HBM round trip while the accumulator is held.
    uint8_t* wbuf = ep_base + e * (EP_TOTAL / n_epi);
    uint8_t* rres = wbuf;  // EPI_RESIDUAL: residual slots 0, 1; output slots 2, 3
    const bool wide = n_epi == 4;
    int ns = 0;            // stores issued by this warp
    // staging slot for the next 16-bit output box
    auto out_slot = [&]() -> uint8_t* {
      uint8_t* sl;
      if (p.epi == EPI_RESIDUAL) {
        slot_free<1>(lane);
        sl = wbuf + 4096 + (ns & 1) * 2048;
      } else if (wide) {
        slot_free<3>(lane);
        sl = wbuf + (ns & 3) * 2048;
      } else {
        slot_free<1>(lane);
        sl = wbuf + (ns & 1) * 2048;
      }
      ++ns;
      return sl;
    };
    int it = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++it) {
      int split, mt, nt;
      tile_coords(p, t, split, mt, nt);
      const int buf = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      const int64_t row0 = (int64_t)mt * BM + quarter * 32;
      const int nrows = (int)(p.M - row0 < 32 ? p.M - row0 : 32);
      if (p.epi == EPI_RESIDUAL && nrows > 0) {
        const int64_t n0 = (int64_t)nt * BN;
        const __nv_bfloat16* Rt = p.R + row0 * p.ldr + n0;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int64_t cq = n0 + 32 * q;
          if (cq < p.N) fetch_rows16_32(rres + q * 2048, Rt + 32 * q, p.ldr, nrows, (int)(p.N - cq < 32 ? p.N - cq : 32), lane);
          cp_async_commit();
        }
        const int64_t tcols = p.N - n0 < BN ? p.N - n0 : BN;
        if (lane < nrows && tcols > 64) prefetch_l2(Rt + (int64_t)lane * p.ldr + 64, (uint32_t)(tcols - 64) * 2u);
      }
      if (!mbar_wait(&S.acc_full[buf], acc_phase, abort_flag)) { ok = false; break; }
      tc_fence_after();
#pragma unroll 1
      for (int j = 0; j < cpw; ++j) {
        const int c = c0 + j;
        uint32_t r[32];
        tmem_ld32(tmem + buf * ACC_COLS + c * 32 + lane_sel, r);
        tmem_wait_ld();
        if (j == cpw - 1) {  // the accumulator is free once read
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.acc_empty[buf]);
        }
        const int64_t col0 = (int64_t)nt * BN + c * 32;
        const int ncols = (int)(p.N - col0 < 32 ? p.N - col0 : 32);
        if (ncols <= 0 || nrows <= 0) continue;
        float x[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(r[i]);
        if (p.epi == EPI_F32) {
          if (p.out_scale) {
            const float sc = *p.out_scale;
#pragma unroll
            for (int i = 0; i < 32; ++i) x[i] *= sc;
          }
          uint8_t* sl;
          if (wide) {
            slot_free<1>(lane);
            sl = wbuf + (ns & 1) * 4096;
          } else {
            slot_free<0>(lane);
            sl = wbuf;
          }
          ++ns;
          stage_store32(x, sl, &tmC, (int)col0, (int)row0, split, lane);
          continue;
        }
        if (p.epi == EPI_SILU) {
          // C = silu(z); Z = silu'(z) = σ(z)(1 + z(1 - σ(z))), the factor that
          // the backward applies to the gradient of silu(z) (not written when
          // Z is null: a forward that keeps nothing for a backward)
          float dz[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float sg = __fdividef(1.0f, 1.0f + __expf(-x[i]));
            dz[i] = sg * fmaf(x[i], 1.0f - sg, 1.0f);
            x[i] *= sg;
          }
          if (p.Z == nullptr) {
          } else if (p.z_f16) {
            stage_store16<__half>(dz, out_slot(), &tmZ, (int)col0, (int)row0, lane);
          } else {
            stage_store16<__nv_bfloat16>(dz, out_slot(), &tmZ, (int)col0, (int)row0, lane);
          }
        } else if (p.epi == EPI_RESIDUAL) {
          cp_async_wait<1>();
          __syncwarp();
          float res[32];
          if (p.r_f16)
            read_rows16_32<__half>(rres + (c & 1) * 2048, res, lane);
          else
            read_rows16_32<__nv_bfloat16>(rres + (c & 1) * 2048, res, lane);
          __syncwarp();
          const int64_t cx = col0 + 64;  // chunk c + 2 into the slot just read
          if (c + 2 < BN / 32 && cx < p.N)
            fetch_rows16_32(rres + (c & 1) * 2048, p.R + row0 * p.ldr + cx, p.ldr, nrows,
                            (int)(p.N - cx < 32 ? p.N - cx : 32), lane);
          cp_async_commit();
#pragma unroll
          for (int i = 0; i < 32; ++i) x[i] += res[i];
        }
        if (p.c_f16)
          stage_store16<__half>(x, out_slot(), &tmC, (int)col0, (int)row0, lane);
        else
          stage_store16<__nv_bfloat16>(x, out_slot(), &tmC, (int)col0, (int)row0, lane);
      }
    }
    if (lane == 0) tma_store_wait_all();
    __syncwarp();
    cp_async_wait<0>();
  }

  if (!ok) {
    *abort_flag = 1;
    if (p.status) atomicOr(p.status, DEV_ERR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

__global__ void split_reduce_kernel(const float* __restrict__ parts, int splits, int64_t stride, int64_t n,
                                    float* __restrict__ out) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float s = 0.f;
  for (int k = 0; k < splits; ++k) s += parts[k * stride + i];
  out[i] = s;
}

// out = R + sum over the split-K slices, 8 elements (16 bytes of 16-bit
// output) per thread: the residual epilogue of an output projection that ran
// split over K because its output tiles alone would leave most SMs idle.
template <typename T>
__global__ void split_reduce_residual_kernel(const float* __restrict__ parts, int splits, int64_t stride, int64_t n8,
                                             const T* __restrict__ R, T* __restrict__ out) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const uint4 r = *reinterpret_cast<const uint4*>(R + 8 * i);
  const uint32_t rw[4] = {r.x, r.y, r.z, r.w};
  float x[8];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    x[2 * t] = lo16<T>(rw[t]);
    x[2 * t + 1] = hi16<T>(rw[t]);
  }
  for (int k = 0; k < splits; ++k) {
    const float4* pk = reinterpret_cast<const float4*>(parts + k * stride + 8 * i);
    const float4 a = pk[0], b = pk[1];
    x[0] += a.x; x[1] += a.y; x[2] += a.z; x[3] += a.w;
    x[4] += b.x; x[5] += b.y; x[6] += b.z; x[7] += b.w;
  }
  *reinterpret_cast<uint4*>(out + 8 * i) = pack8<T>(x);
}

}  // namespace

cudaError_t launch_split_reduce_residual(const float* parts, int splits, int64_t stride, int64_t n, const void* R,
                                         void* out, bool f16, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  if (n % 8 != 0 || stride % 8 != 0) return cudaErrorInvalidValue;
  TraceScope tr("split_reduce_out", s);
  const int64_t n8 = n / 8;
  const unsigned blocks = (unsigned)((n8 + 255) / 256);
  if (f16)
    split_reduce_residual_kernel<__half><<<blocks, 256, 0, s>>>(parts, splits, stride, n8,
                                                                static_cast<const __half*>(R), static_cast<__half*>(out));
  else
    split_reduce_residual_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(
        parts, splits, stride, n8, static_cast<const __nv_bfloat16*>(R), static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

cudaError_t launch_split_reduce(const float* parts, int splits, int64_t stride, int64_t n, float* out,
                                cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  TraceScope tr("split_reduce", s);
  split_reduce_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(parts, splits, stride, n, out);
  return cudaGetLastError();
}

cudaError_t launch_gemm_bf16(const GemmArgs& a, cudaStream_t s) {
  if (a.M == 0 || a.N == 0) return cudaSuccess;
  CUtensorMap tmA, tmB;
  // A: K-major -> rows M, cols K, box 64 x 128;  MN-major -> rows K, cols M, box 64 x 64
  auto tmap16 = a.ab_f16 ? make_tmap_f16_2d : make_tmap_bf16_2d;
  bool okA = a.a_mn_major ? tmap16(&tmA, a.A, a.K, a.M, a.lda, 64, 64) : tmap16(&tmA, a.A, a.M, a.K, a.lda, 64, BM);
  bool okB = a.b_mn_major ? tmap16(&tmB, a.B, a.K, a.N, a.ldb, 64, 64) : tmap16(&tmB, a.B, a.N, a.K, a.ldb, 64, BN);
  if (!okA || !okB) return cudaErrorInvalidValue;
  Params p;
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.m_tiles = (int)((a.M + BM - 1) / BM);
  p.n_tiles = (int)((a.N + BN - 1) / BN);
  p.nk = (int)((a.K + BK - 1) / BK);
  const int splits = a.epi == EPI_F32 ? gemm_splits(a.K, a.splits) : 1;
  p.kb_per_split = (p.nk + splits - 1) / splits;
  p.splits = splits;
  // outputs: [32][32] boxes; fp32 split-K slices as a 3-D map
  CUtensorMap tmC, tmZ;
  const bool okC = a.epi == EPI_F32
                       ? make_tmap_out(&tmC, OUT_F32, a.C, a.M, a.N, a.ldc, splits, 32, 32)
                       : make_tmap_out(&tmC, a.c_f16 ? OUT_F16 : OUT_BF16, a.C, a.M, a.N, a.ldc, 0, 32, 32);
  const bool okZ =
      a.epi == EPI_SILU && a.Z ? make_tmap_out(&tmZ, a.z_f16 ? OUT_F16 : OUT_BF16, a.Z, a.M, a.N, a.ldz, 0, 32, 32)
                               : true;
  if (a.epi != EPI_SILU || !a.Z) tmZ = tmC;
  if (!okC || !okZ) return cudaErrorInvalidValue;
  p.a_mn = a.a_mn_major;
  p.b_mn = a.b_mn_major;
  p.ab_f16 = a.ab_f16;
  p.r_f16 = a.r_f16;
  p.z_f16 = a.z_f16;
  p.epi = a.epi;
  p.c_f16 = a.c_f16;
  p.C = a.C;
  p.ldc = a.ldc;
  p.R = a.R;
  p.ldr = a.ldr;
  p.Z = a.Z;
  p.ldz = a.ldz;
  p.out_scale = a.out_scale;
  p.status = a.status;
  cudaError_t e = cudaFuncSetAttribute(gemm_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int tiles = p.splits * p.m_tiles * p.n_tiles;
  const int grid = tiles < num_sms() ? tiles : num_sms();
  if (p.nk == 0) return cudaErrorInvalidValue;
  TraceScope tr(a.name ? a.name : "gemm", s);
  // the residual epilogue keeps 4 warps (its cp.async ring needs 8 KB each)
  const int threads = a.epi == EPI_RESIDUAL ? 192 : MAX_THREADS;
  gemm_bf16_kernel<<<grid, threads, SMEM_BYTES, s>>>(tmA, tmB, tmC, tmZ, p);
  return cudaGetLastError();
}

}  // namespace mtgr
