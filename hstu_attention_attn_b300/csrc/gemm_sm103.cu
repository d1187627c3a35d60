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
constexpr int NUM_THREADS = 192;
constexpr int STG_BYTES = 4096;  // per epilogue warp: 32 rows x 32 fp32
constexpr int RES_BYTES = 2 * 2048;  // per epilogue warp: 2 residual chunks of 32 rows x 32 bf16
constexpr int SMEM_BYTES =
    STAGES * STAGE_BYTES + 4 * STG_BYTES + 4 * RES_BYTES + 1024 /*align*/ + 256 /*barriers*/;

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
  bool c_f16;
  int epi;
  void* C;
  int64_t ldc;
  const __nv_bfloat16* R;
  int64_t ldr;
  __nv_bfloat16* Z;
  int64_t ldz;
  int32_t* status;
};

__device__ __forceinline__ void tile_coords(const Params& p, int t, int& split, int& mt, int& nt) {
  const int per_split = p.m_tiles * p.n_tiles;
  split = t / per_split;
  const int r = t - split * per_split;
  mt = r / p.n_tiles;
  nt = r - mt * p.n_tiles;
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const Params p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned staging area (128-byte swizzle atoms), then the barriers
  uint8_t* stage_base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stg_base = stage_base + STAGES * STAGE_BYTES;
  uint8_t* res_base = stg_base + 4 * STG_BYTES;
  Smem& S = *reinterpret_cast<Smem*>(res_base + 4 * RES_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_tiles = p.splits * p.m_tiles * p.n_tiles;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.acc_full[i], 1);
      mbar_init(&S.acc_empty[i], 4);  // one arrival per epilogue warp
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
    const uint32_t idesc = idesc_bf16_f32(BM, BN, p.a_mn, p.b_mn);
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
    // ---------------- epilogue (warps 2..5) ----------------
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    const uint32_t lane_sel = (uint32_t)(quarter * 32) << 16;
    uint8_t* stg = stg_base + (warp - 2) * STG_BYTES;
    // Residual chunks (EPI_RESIDUAL) go through a 2-slot cp.async ring: chunks
    // 0 and 1 are requested before the accumulator wait and the rest of the
    // warp's rows of the tile are prefetched into L2, so no chunk waits for a
    // full HBM round trip while the accumulator is held.
    uint8_t* rres = res_base + (warp - 2) * RES_BYTES;
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
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + buf * ACC_COLS + c * 32 + lane_sel, r);
        tmem_wait_ld();
        if (c == BN / 32 - 1) {  // the accumulator is free once read
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
          float* C = reinterpret_cast<float*>(p.C) + (int64_t)split * p.M * p.ldc + row0 * p.ldc + col0;
          store_rows32_32(x, stg, C, p.ldc, nrows, ncols, lane);
          continue;
        }
        if (p.epi == EPI_SILU) {
          // C = silu(z); Z = silu'(z) = σ(z)(1 + z(1 - σ(z))), the factor that
          // the backward applies to the gradient of silu(z)
          float dz[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float sg = __fdividef(1.0f, 1.0f + __expf(-x[i]));
            dz[i] = sg * fmaf(x[i], 1.0f - sg, 1.0f);
            x[i] *= sg;
          }
          store_rows16_32(dz, stg, p.Z + row0 * p.ldz + col0, p.ldz, nrows, ncols, lane);
        } else if (p.epi == EPI_RESIDUAL) {
          cp_async_wait<1>();
          __syncwarp();
          float res[32];
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
          store_rows16_32(x, stg, reinterpret_cast<__half*>(p.C) + row0 * p.ldc + col0, p.ldc, nrows, ncols, lane);
        else
          store_rows16_32(x, stg, reinterpret_cast<__nv_bfloat16*>(p.C) + row0 * p.ldc + col0, p.ldc, nrows, ncols,
                          lane);
      }
    }
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

}  // namespace

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
  bool okA = a.a_mn_major ? make_tmap_bf16_2d(&tmA, a.A, a.K, a.M, a.lda, 64, 64)
                    : make_tmap_bf16_2d(&tmA, a.A, a.M, a.K, a.lda, 64, BM);
  bool okB = a.b_mn_major ? make_tmap_bf16_2d(&tmB, a.B, a.K, a.N, a.ldb, 64, 64)
                          : make_tmap_bf16_2d(&tmB, a.B, a.N, a.K, a.ldb, 64, BN);
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
  p.a_mn = a.a_mn_major;
  p.b_mn = a.b_mn_major;
  p.epi = a.epi;
  p.c_f16 = a.c_f16;
  p.C = a.C;
  p.ldc = a.ldc;
  p.R = a.R;
  p.ldr = a.ldr;
  p.Z = a.Z;
  p.ldz = a.ldz;
  p.status = a.status;
  cudaError_t e = cudaFuncSetAttribute(gemm_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int tiles = p.splits * p.m_tiles * p.n_tiles;
  const int grid = tiles < num_sms() ? tiles : num_sms();
  if (p.nk == 0) return cudaErrorInvalidValue;
  TraceScope tr(a.name ? a.name : "gemm", s);
  gemm_bf16_kernel<<<grid, NUM_THREADS, SMEM_BYTES, s>>>(tmA, tmB, p);
  return cudaGetLastError();
}

}  // namespace mtgr
