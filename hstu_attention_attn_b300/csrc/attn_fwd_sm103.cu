// attn_fwd_sm103.cu -- jagged HSTU attention forward on the 5th-generation
// tensor cores (tcgen05 + TMEM + TMA): f16 operands (q, k, v and P), fp32
// accumulation, fp32 O.
//
// Computes, per head and per 128-row query tile of one user segment,
//   S = Q Kᵀ                       (tcgen05.mma, fp32 in TMEM)
//   P = M ⊙ silu(S / sqrt(d_h))    (epilogue warps, in registers; f16 into TMEM)
//   O += P V                       (tcgen05.mma with P read from TMEM)
// over the key tiles the dynamic mixed mask leaves visible, then O / n_u.
// Block formula: marovi.ai "Métodos" (Ṽ = silu(KᵀQ)/(N_U+N_S+N_R+N_I) · M · V);
// SiLU weights without softmax: paper-daily "模型怎么搭"; mask rules: fun-rec
// chapter 7.3, §7.3.4.  Without a softmax there is no running max and no
// rescaling: the accumulator simply sums, and 1/n_u is one per-row scale at
// the end (n_u is constant over a user's rows).
//
// CTA = one (user, query tile, head) work item from the longest-first list.
//   warp 0      TMA: Q once, then K_j / V_j (one buffer each)
//   warp 1      MMA issuer (one thread) + TMEM owner
//   warps 2..5  P epilogue (thread = query row = TMEM lane) and the O store
// TMEM: S at columns [0,128) (P aliases its first 64 columns as packed f16),
// O at [128, 128+d_h).  96 KB of shared memory and 256 TMEM columns per CTA,
// so two CTAs share an SM and interleave their MMA and epilogue phases.
#include "common.cuh"
#include "plan.cuh"

namespace mtgr {
namespace {

constexpr int BQ = 128, BKV = 128;
constexpr int NUM_THREADS = 192;

template <int D>
struct FwdCfg {
  static constexpr int TILE_BYTES = BQ * D * 2;  // one Q / K / V tile
  // at least ~100 KB so that no more than two CTAs (2 x 256 TMEM columns) share an SM
  static constexpr int SMEM = (3 * TILE_BYTES + 1152) > 102400 ? (3 * TILE_BYTES + 1152) : 102400;
  static constexpr uint32_t TMEM_COLS = 256;
  static constexpr uint32_t S_COL = 0, O_COL = 128;
};

struct FwdSmem {
  uint64_t q_full, k_full, k_empty, v_full, v_empty, s_full, p_full, o_full, pv_done;
  uint32_t tmem_base;
  int abort_flag;
};

struct FwdParams {
  const UserInfo* users;
  const WorkItem* items;
  const int32_t* counts;
  const int64_t* ts;
  float* O;  // [T, H*D] fp32
  int64_t ldo;
  int H;
  float scale;  // 1/sqrt(d_h)
  int32_t* status;
};

// Shared-memory descriptors of a [128 rows][D] 16-bit tile staged as D/64 boxes
// of [128][64] with 128-byte swizzle (16 KB per box).
template <int D>
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile, int kk) {  // K = d, step 16
  return smem_desc_sw128(tile + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t tile, int kk) {  // K = rows, step 16
  return smem_desc_sw128(tile + kk * 2048, 16384, 1024);
}

template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 2)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using Cfg = FwdCfg<D>;
  const int item_idx = blockIdx.x / p.H;
  const int h = blockIdx.x - item_idx * p.H;
  if (item_idx >= p.counts[0]) return;
  const WorkItem wi = p.items[item_idx];
  const UserInfo u = p.users[wi.b];
  const int qt = wi.t;
  const QTileKeys keys = qtile_keys(u, qt);
  const int nk = keys.count();

  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base;
  uint8_t* sK = base + Cfg::TILE_BYTES;
  uint8_t* sV = base + 2 * Cfg::TILE_BYTES;
  FwdSmem& S = *reinterpret_cast<FwdSmem*>(base + 3 * Cfg::TILE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&S.q_full, 1);
    mbar_init(&S.k_full, 1);
    mbar_init(&S.k_empty, 1);
    mbar_init(&S.v_full, 1);
    mbar_init(&S.v_empty, 1);
    mbar_init(&S.s_full, 1);
    mbar_init(&S.p_full, 4);
    mbar_init(&S.o_full, 1);
    mbar_init(&S.pv_done, 1);
    S.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  volatile int* abort_flag = &S.abort_flag;
  bool ok = true;
  const int col_h = h * D;  // column of this head inside q / k / v

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      mbar_arrive_expect_tx(&S.q_full, Cfg::TILE_BYTES);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_2d(sQ + c * 16384, &tmQ, &S.q_full, col_h + 64 * c, u.start + qt * BQ);
      for (int i = 0; i < nk && ok; ++i) {
        const int row = u.start + keys.kt(i, qt) * BKV;
        if (!mbar_wait(&S.k_empty, (i & 1) ^ 1, abort_flag)) { ok = false; break; }
        mbar_arrive_expect_tx(&S.k_full, Cfg::TILE_BYTES);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) tma_load_2d(sK + c * 16384, &tmK, &S.k_full, col_h + 64 * c, row);
        if (!mbar_wait(&S.v_empty, (i & 1) ^ 1, abort_flag)) { ok = false; break; }
        mbar_arrive_expect_tx(&S.v_full, Cfg::TILE_BYTES);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) tma_load_2d(sV + c * 16384, &tmV, &S.v_full, col_h + 64 * c, row);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t idesc_s = idesc_f16_f32(BQ, BKV, false, false);
      constexpr uint32_t idesc_o = idesc_f16_f32(BQ, D, false, true);
      const uint32_t q_addr = smem_u32(sQ), k_addr = smem_u32(sK), v_addr = smem_u32(sV);
      const uint32_t t_s = tmem + Cfg::S_COL, t_o = tmem + Cfg::O_COL;
      if (!mbar_wait(&S.q_full, 0, abort_flag)) ok = false;
      for (int i = 0; i < nk && ok; ++i) {
        const uint32_t par = i & 1;
        if (!mbar_wait(&S.k_full, par, abort_flag)) { ok = false; break; }
        // S_i overwrites the columns that hold P_{i-1}: wait until P_{i-1} V_{i-1} has read them
        if (i > 0 && !mbar_wait(&S.pv_done, par ^ 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc_mma_ss(t_s, kmajor_desc<D>(q_addr, kk), kmajor_desc<D>(k_addr, kk), idesc_s, kk > 0 ? 1u : 0u);
        tc_commit(&S.k_empty);
        tc_commit(&S.s_full);
        if (!mbar_wait(&S.p_full, par, abort_flag)) { ok = false; break; }
        if (!mbar_wait(&S.v_full, par, abort_flag)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BKV / 16; ++kk)
          tc_mma_ts(t_o, t_s + kk * 8, mnmajor_desc(v_addr, kk), idesc_o, (i > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&S.v_empty);
        tc_commit(&S.pv_done);
      }
      tc_commit(&S.o_full);
    }
  } else {
    // ---------------- P epilogue (warps 2..5) ----------------
    const int quarter = warp & 3;
    const uint32_t lane_sel = (uint32_t)(quarter * 32) << 16;
    const int ri = qt * BQ + quarter * 32 + lane;  // segment-relative query row
    const bool row_ok = ri < u.n;
    const int row_cls = ri < u.eS ? 0 : (ri < u.eR ? 1 : 2);  // 0 User/Seq, 1 RealTime, 2 Cand
    const int64_t ts_i = (row_ok && row_cls > 0) ? p.ts[u.start + ri] : 0;
    const float hs = 0.5f * p.scale;  // silu(x) = h + h tanh(h), h = x/2
    for (int i = 0; i < nk && ok; ++i) {
      const int kt = keys.kt(i, qt);
      if (!mbar_wait(&S.s_full, i & 1, abort_flag)) { ok = false; break; }
      tc_fence_after();
      const int k0 = kt * BKV;
      const bool all_static = k0 + BKV <= u.eS;
#pragma unroll
      for (int c = 0; c < BKV / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + Cfg::S_COL + c * 32 + lane_sel, r);
        tmem_wait_ld();
        uint32_t pk[16];
        if (all_static) {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float h0 = __uint_as_float(r[2 * e]) * hs, h1 = __uint_as_float(r[2 * e + 1]) * hs;
            pk[e] = pack_f16x2(fmaf(h0, tanh_approx(h0), h0), fmaf(h1, tanh_approx(h1), h1));
          }
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float pv[2];
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              const int rj = k0 + c * 32 + 2 * e + t;
              bool vis;
              if (rj < u.eS) {
                vis = true;
              } else if (rj < u.eR) {
                const int64_t ts_j = p.ts[u.start + rj];
                vis = row_cls == 1 ? (ts_j <= ts_i) : (row_cls == 2 && ts_j < ts_i);
              } else {
                vis = (rj == ri) && rj < u.n;
              }
              const float hh = __uint_as_float(r[2 * e + t]) * hs;
              pv[t] = vis ? fmaf(hh, tanh_approx(hh), hh) : 0.f;
            }
            pk[e] = pack_f16x2(pv[0], pv[1]);
          }
        }
        tmem_st16(tmem + Cfg::S_COL + c * 16 + lane_sel, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.p_full);
    }
    // ---------------- O = acc / n_u -> global ----------------
    if (ok && mbar_wait(&S.o_full, 0, abort_flag)) {
      tc_fence_after();
      const float inv_n = 1.0f / (float)u.n;
      float* orow = p.O + (int64_t)(u.start + ri) * p.ldo + col_h;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + Cfg::O_COL + c * 32 + lane_sel, r);
        tmem_wait_ld();
        if (row_ok) {
#pragma unroll
          for (int v = 0; v < 8; ++v)
            *reinterpret_cast<float4*>(orow + c * 32 + 4 * v) =
                make_float4(__uint_as_float(r[4 * v + 0]) * inv_n, __uint_as_float(r[4 * v + 1]) * inv_n,
                            __uint_as_float(r[4 * v + 2]) * inv_n, __uint_as_float(r[4 * v + 3]) * inv_n);
        }
      }
    } else {
      ok = false;
    }
  }

  if (!ok) {
    *abort_flag = 1;
    if (p.status) atomicOr(p.status, DEV_ERR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::TMEM_COLS);
  }
}

}  // namespace

// q, k, v: [T, *] f16 with row stride ld; O: [T, H*d] fp32.
cudaError_t launch_attn_fwd_f16(const __half* q, const __half* k, const __half* v,
                                 int64_t ld, int64_t T, int H, int d, const int32_t* plan, int32_t B,
                                 const int64_t* ts, float* O, int32_t* status, cudaStream_t s) {
  if (T == 0 || B == 0) return cudaSuccess;
  const PlanLayout L = plan_layout(B, T);
  const int HD = H * d;
  CUtensorMap tq, tk, tv;
  if (!make_tmap_f16_2d(&tq, q, T, HD, ld, 64, BQ) || !make_tmap_f16_2d(&tk, k, T, HD, ld, 64, BKV) ||
      !make_tmap_f16_2d(&tv, v, T, HD, ld, 64, BKV))
    return cudaErrorInvalidValue;
  FwdParams p;
  p.users = reinterpret_cast<const UserInfo*>(plan + L.users);
  p.items = reinterpret_cast<const WorkItem*>(plan + L.fwd_items);
  p.counts = plan + L.counts;
  p.ts = ts;
  p.O = O;
  p.ldo = HD;
  p.H = H;
  p.scale = 1.0f / sqrtf((float)d);
  p.status = status;
  const int64_t grid = L.max_items * H;
  if (grid > 0x7fffffff) return cudaErrorInvalidValue;
  TraceScope tr("attn_fwd", s);
  if (d == 128) {
    auto kern = attn_fwd_kernel<128>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, FwdCfg<128>::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)grid, NUM_THREADS, FwdCfg<128>::SMEM, s>>>(tq, tk, tv, p);
  } else if (d == 64) {
    auto kern = attn_fwd_kernel<64>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, FwdCfg<64>::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)grid, NUM_THREADS, FwdCfg<64>::SMEM, s>>>(tq, tk, tv, p);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace mtgr
