// attn_bwd_sm103.cu -- jagged HSTU attention backward on the 5th-generation
// tensor cores (tcgen05 + TMEM + TMA): f16 operands (q, k, v, dO, P, dS),
// fp32 accumulation, bf16 gradients.
//
// With s = q·k / sqrt(d_h), A = M ⊙ silu(s) / n_u and O = A V (marovi.ai
// "Métodos" block formula; paper-daily "模型怎么搭"), the gradients are
//   dV = Aᵀ dO,  dA = dO Vᵀ,  dS = M ⊙ dA ⊙ silu'(s) / (n_u sqrt(d_h)),
//   dQ = dS K,   dK = dSᵀ Q,   silu'(s) = σ(s)(1 + s(1 - σ(s))).
// There is no softmax, so no row statistics are needed: S is recomputed.
//
// CTA = one (user, key tile, head) work item from the longest-first list; it
// loops over the query tiles that see the key tile (dynamic mixed mask,
// fun-rec chapter 7.3, §7.3.4).  Per query tile:
//   Sᵀ  = K Qᵀ            -> TMEM [0,128)
//   dPᵀ = V dOᵀ           -> TMEM [128,256)
//   epilogue (thread = key row): Pᵀ (f16) into TMEM [0,64), dSᵀ (f16) into
//   shared memory (128-byte swizzled, written by threads)
//   dV += Pᵀ dO           (A from TMEM)            -> TMEM [256, 256+D)
//   dK += dSᵀ Q           (A K-major from smem)    -> TMEM [256+D, 256+2D)
//   dQ  = dS K            (A MN-major: same smem)  -> TMEM [128,128+D)
//   epilogue (thread = query row): dQ added into an fp32 accumulator in global
//   memory with vector atomics; a final pass applies silu'(z) and rounds to
//   bf16.  P is kept without the 1/n_u factor (dV is scaled once at the end).
// Warps: 0 TMA, 1 MMA issuer + TMEM owner, 2..5 epilogue.
#include "common.cuh"
#include "plan.cuh"

namespace mtgr {
namespace {

constexpr int BT = 128;  // key tile = query tile = 128 rows
constexpr int NUM_THREADS = 192;

template <int D>
struct BwdCfg {
  static constexpr int TILE = BT * D * 2;  // K / V / Q / dO tile bytes
  static constexpr int DS_BYTES = BT * BT * 2;
  static constexpr int SMEM = 4 * TILE + DS_BYTES + 1024 + 256;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t ST = 0, DPT = 128, DQ = 128, DV = 256, DK = 256 + D;
};

struct BwdSmem {
  uint64_t kv_full, q_full, q_empty, do_full, do_empty, sdp_full, p_ready, dq_full, dq_free, dkdv_full, dv_done;
  uint32_t tmem_base;
  int abort_flag;
};

struct BwdParams {
  const UserInfo* users;
  const WorkItem* items;
  const int32_t* counts;
  const int64_t* ts;
  float* dq_acc;  // [T, H*D] fp32 (row stride ldacc), zeroed before the launch
  int64_t ldacc;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int64_t ldg;
  const __nv_bfloat16* zk;  // optional pre-activations (row stride ldz)
  const __nv_bfloat16* zv;
  int64_t ldz;
  int H;
  float scale;
  int32_t* status;
};

template <int D>
__device__ __forceinline__ uint64_t kmaj(uint32_t tile, int kk) {
  return smem_desc_sw128(tile + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t mnmaj(uint32_t tile, int kk) {
  return smem_desc_sw128(tile + kk * 2048, 16384, 1024);
}

__device__ __forceinline__ float silu_grad_bf(float z) {
  const float sg = sigmoid_f(z);
  return sg * (1.f + z * (1.f - sg));
}

template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                    const BwdParams p) {
  using Cfg = BwdCfg<D>;
  const int item_idx = blockIdx.x / p.H;
  const int h = blockIdx.x - item_idx * p.H;
  if (item_idx >= p.counts[1]) return;
  const WorkItem wi = p.items[item_idx];
  const UserInfo u = p.users[wi.b];
  const int kt = wi.t;
  const KTileQueries qs = ktile_queries(u, kt);
  const int nq = qs.count();

  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = base;
  uint8_t* sV = base + Cfg::TILE;
  uint8_t* sQ = base + 2 * Cfg::TILE;
  uint8_t* sdO = base + 3 * Cfg::TILE;
  uint8_t* sdS = base + 4 * Cfg::TILE;
  BwdSmem& S = *reinterpret_cast<BwdSmem*>(base + 4 * Cfg::TILE + Cfg::DS_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&S.kv_full, 1);
    mbar_init(&S.q_full, 1);
    mbar_init(&S.q_empty, 1);
    mbar_init(&S.do_full, 1);
    mbar_init(&S.do_empty, 1);
    mbar_init(&S.sdp_full, 1);
    mbar_init(&S.p_ready, 4);
    mbar_init(&S.dq_full, 1);
    mbar_init(&S.dq_free, 4);
    mbar_init(&S.dkdv_full, 1);
    mbar_init(&S.dv_done, 1);
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
    tma_prefetch_desc(&tmdO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  volatile int* abort_flag = &S.abort_flag;
  bool ok = true;
  const int col_h = h * D;
  const int key_row0 = u.start + kt * BT;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      mbar_arrive_expect_tx(&S.kv_full, 2 * Cfg::TILE);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        tma_load_2d(sK + c * 16384, &tmK, &S.kv_full, col_h + 64 * c, key_row0);
        tma_load_2d(sV + c * 16384, &tmV, &S.kv_full, col_h + 64 * c, key_row0);
      }
      for (int i = 0; i < nq && ok; ++i) {
        const int qrow = u.start + qs.qt(i, kt) * BT;
        if (!mbar_wait(&S.q_empty, (i & 1) ^ 1, abort_flag)) { ok = false; break; }
        mbar_arrive_expect_tx(&S.q_full, Cfg::TILE);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) tma_load_2d(sQ + c * 16384, &tmQ, &S.q_full, col_h + 64 * c, qrow);
        if (!mbar_wait(&S.do_empty, (i & 1) ^ 1, abort_flag)) { ok = false; break; }
        mbar_arrive_expect_tx(&S.do_full, Cfg::TILE);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) tma_load_2d(sdO + c * 16384, &tmdO, &S.do_full, col_h + 64 * c, qrow);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t id_sq = idesc_f16_f32(BT, BT, false, false);  // Sᵀ, dPᵀ
      constexpr uint32_t id_dv = idesc_f16_f32(BT, D, false, true);    // dV (A tmem), dK (A K-major)
      constexpr uint32_t id_dq = idesc_f16_f32(BT, D, true, true);     // dQ: A = dS MN-major
      const uint32_t aK = smem_u32(sK), aV = smem_u32(sV), aQ = smem_u32(sQ), adO = smem_u32(sdO),
                     adS = smem_u32(sdS);
      if (!mbar_wait(&S.kv_full, 0, abort_flag)) ok = false;
      for (int i = 0; i < nq && ok; ++i) {
        const uint32_t par = i & 1;
        if (!mbar_wait(&S.q_full, par, abort_flag)) { ok = false; break; }
        // Sᵀ_i overwrites the columns holding Pᵀ_{i-1}: wait until dV_{i-1} has read them
        if (i > 0 && !mbar_wait(&S.dv_done, par ^ 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc_mma_ss(tmem + Cfg::ST, kmaj<D>(aK, kk), kmaj<D>(aQ, kk), id_sq, kk > 0 ? 1u : 0u);
        if (i > 0 && !mbar_wait(&S.dq_free, par ^ 1, abort_flag)) { ok = false; break; }
        if (!mbar_wait(&S.do_full, par, abort_flag)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc_mma_ss(tmem + Cfg::DPT, kmaj<D>(aV, kk), kmaj<D>(adO, kk), id_sq, kk > 0 ? 1u : 0u);
        tc_commit(&S.sdp_full);
        if (!mbar_wait(&S.p_ready, par, abort_flag)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BT / 16; ++kk)  // dV += Pᵀ dO, K = query rows
          tc_mma_ts(tmem + Cfg::DV, tmem + Cfg::ST + kk * 8, mnmaj(adO, kk), id_dv, (i > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&S.dv_done);
#pragma unroll
        for (int kk = 0; kk < BT / 16; ++kk)  // dK += dSᵀ Q
          tc_mma_ss(tmem + Cfg::DK, kmaj<BT>(adS, kk), mnmaj(aQ, kk), id_dv, (i > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < BT / 16; ++kk)  // dQ = dS K, K = key rows
          tc_mma_ss(tmem + Cfg::DQ, mnmaj(adS, kk), mnmaj(aK, kk), id_dq, kk > 0 ? 1u : 0u);
        tc_commit(&S.dq_full);
        tc_commit(&S.q_empty);
        tc_commit(&S.do_empty);
      }
      tc_commit(&S.dkdv_full);
    }
  } else {
    // ---------------- epilogue warps 2..5 ----------------
    const int quarter = warp & 3;
    const uint32_t lane_sel = (uint32_t)(quarter * 32) << 16;
    const int r_in = quarter * 32 + lane;  // TMEM lane
    const int rj = kt * BT + r_in;         // this thread's key row (segment-relative)
    const int key_cls = rj < u.eS ? 0 : (rj < u.eR ? 1 : 2);
    const int64_t ts_j = (key_cls == 1 && rj < u.n) ? p.ts[u.start + rj] : 0;
    const float c = p.scale, inv_n = 1.0f / (float)u.n;
    const float cds = c * inv_n;
    const bool all_static = kt * BT + BT <= u.eS;
    for (int i = 0; i < nq && ok; ++i) {
      const int qt = qs.qt(i, kt);
      const int q0 = qt * BT;
      if (!mbar_wait(&S.sdp_full, i & 1, abort_flag)) { ok = false; break; }
      tc_fence_after();
#pragma unroll 1
      for (int ch = 0; ch < BT / 32; ++ch) {
        uint32_t sr[32], dr[32];
        tmem_ld32(tmem + Cfg::ST + ch * 32 + lane_sel, sr);
        tmem_ld32(tmem + Cfg::DPT + ch * 32 + lane_sel, dr);
        tmem_wait_ld();
        uint32_t pk[16], dk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float pv[2], dsv[2];
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int col = ch * 32 + 2 * e + t;
            const int ri = q0 + col;
            bool vis;
            if (all_static || key_cls == 0) {
              vis = ri < u.n;
            } else if (key_cls == 1) {
              if (ri < u.eS || ri >= u.n) {
                vis = false;
              } else {
                const int64_t ts_i = p.ts[u.start + ri];
                vis = ri < u.eR ? (ts_j <= ts_i) : (ts_j < ts_i);
              }
            } else {
              vis = (ri == rj) && ri < u.n;
            }
            const float s = __uint_as_float(sr[2 * e + t]) * c;
            const float sg = fmaf(0.5f, tanh_approx(0.5f * s), 0.5f);
            const float silu = s * sg;
            const float dsil = sg * fmaf(s, 1.f - sg, 1.f);
            pv[t] = vis ? silu : 0.f;
            dsv[t] = vis ? __uint_as_float(dr[2 * e + t]) * dsil * cds : 0.f;
          }
          pk[e] = pack_f16x2(pv[0], pv[1]);
          dk[e] = pack_f16x2(dsv[0], dsv[1]);
        }
        tmem_st16(tmem + Cfg::ST + ch * 16 + lane_sel, pk);
        // dSᵀ row r_in, query columns ch*32 .. ch*32+31 -> 4 swizzled 16-byte chunks
        uint8_t* box = sdS + (ch >> 1) * 16384 + r_in * 128;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int chunk = ((ch & 1) * 4 + v) ^ (r_in & 7);
          *reinterpret_cast<uint4*>(box + chunk * 16) = make_uint4(dk[4 * v], dk[4 * v + 1], dk[4 * v + 2], dk[4 * v + 3]);
        }
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.p_ready);
      // ---- dQ partial of this key tile -> fp32 accumulator ----
      if (!mbar_wait(&S.dq_full, i & 1, abort_flag)) { ok = false; break; }
      tc_fence_after();
      const int ri = q0 + r_in;  // TMEM lane = query row for the dQ product
      float* dq_row = p.dq_acc + (int64_t)(u.start + ri) * p.ldacc + col_h;
#pragma unroll 1
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t r[32];
        tmem_ld32(tmem + Cfg::DQ + ch * 32 + lane_sel, r);
        tmem_wait_ld();
        if (ri < u.n) {
#pragma unroll
          for (int v = 0; v < 8; ++v)
            atomicAdd(reinterpret_cast<float4*>(dq_row + ch * 32 + 4 * v),
                      make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                  __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3])));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.dq_free);
    }
    // ---- dK, dV of this key tile -> global (bf16) ----
    if (ok && mbar_wait(&S.dkdv_full, 0, abort_flag)) {
      tc_fence_after();
      const bool row_ok = rj < u.n;
      const int64_t grow = (int64_t)(u.start + rj);
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        __nv_bfloat16* out = (which == 0 ? p.dk : p.dv) + grow * p.ldg + col_h;
        const __nv_bfloat16* z = which == 0 ? p.zk : p.zv;
        const uint32_t col = which == 0 ? Cfg::DK : Cfg::DV;
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t r[32];
          tmem_ld32(tmem + col + ch * 32 + lane_sel, r);
          tmem_wait_ld();
          if (!row_ok) continue;
          float x[32];
          const float sc = nq > 0 ? (which == 0 ? 1.f : inv_n) : 0.f;  // P carries no 1/n_u
#pragma unroll
          for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(r[e]) * sc;
          if (z) {
            const uint4* zp = reinterpret_cast<const uint4*>(z + grow * p.ldz + col_h + ch * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const uint4 zz = zp[v];
              const uint32_t w[4] = {zz.x, zz.y, zz.z, zz.w};
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                x[8 * v + 2 * t] *= silu_grad_bf(bf16_lo(w[t]));
                x[8 * v + 2 * t + 1] *= silu_grad_bf(bf16_hi(w[t]));
              }
            }
          }
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 o;
            o.x = pack_bf16x2(x[8 * v + 0], x[8 * v + 1]);
            o.y = pack_bf16x2(x[8 * v + 2], x[8 * v + 3]);
            o.z = pack_bf16x2(x[8 * v + 4], x[8 * v + 5]);
            o.w = pack_bf16x2(x[8 * v + 6], x[8 * v + 7]);
            *reinterpret_cast<uint4*>(out + ch * 32 + 8 * v) = o;
          }
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

// dq = bf16(dq_acc [* silu'(z)]) for every row that belongs to a segment.
__global__ void dq_finish_kernel(const float* __restrict__ acc, int64_t T, int HD, __nv_bfloat16* __restrict__ dq,
                                 int64_t ldg, const __nv_bfloat16* __restrict__ z, int64_t ldz) {
  const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (i >= T * HD) return;
  const int64_t row = i / HD;
  const int col = (int)(i - row * HD);
  const float4 a0 = *reinterpret_cast<const float4*>(acc + i);
  const float4 a1 = *reinterpret_cast<const float4*>(acc + i + 4);
  float x[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
  if (z) {
    const uint4 zz = *reinterpret_cast<const uint4*>(z + row * ldz + col);
    const uint32_t w[4] = {zz.x, zz.y, zz.z, zz.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      x[2 * t] *= silu_grad_bf(bf16_lo(w[t]));
      x[2 * t + 1] *= silu_grad_bf(bf16_hi(w[t]));
    }
  }
  uint4 o;
  o.x = pack_bf16x2(x[0], x[1]);
  o.y = pack_bf16x2(x[2], x[3]);
  o.z = pack_bf16x2(x[4], x[5]);
  o.w = pack_bf16x2(x[6], x[7]);
  *reinterpret_cast<uint4*>(dq + row * ldg + col) = o;
}

}  // namespace

cudaError_t launch_attn_bwd_f16(const __half* q, const __half* k, const __half* v,
                                 int64_t ld, const __half* dO, int64_t T, int H, int d, const int32_t* plan,
                                 int32_t B, const int64_t* ts, float* dq_acc, __nv_bfloat16* dq, __nv_bfloat16* dk,
                                 __nv_bfloat16* dv, int64_t ldg, const __nv_bfloat16* zq, const __nv_bfloat16* zk,
                                 const __nv_bfloat16* zv, int32_t* status, cudaStream_t s) {
  if (T == 0 || B == 0) return cudaSuccess;
  const PlanLayout L = plan_layout(B, T);
  const int HD = H * d;
  cudaError_t e;
  {
    TraceScope tr("dq_zero", s);
    e = cudaMemsetAsync(dq_acc, 0, sizeof(float) * (size_t)T * HD, s);
  }
  if (e != cudaSuccess) return e;
  CUtensorMap tq, tk, tv, tdo;
  if (!make_tmap_f16_2d(&tq, q, T, HD, ld, 64, BT) || !make_tmap_f16_2d(&tk, k, T, HD, ld, 64, BT) ||
      !make_tmap_f16_2d(&tv, v, T, HD, ld, 64, BT) || !make_tmap_f16_2d(&tdo, dO, T, HD, HD, 64, BT))
    return cudaErrorInvalidValue;
  BwdParams p;
  p.users = reinterpret_cast<const UserInfo*>(plan + L.users);
  p.items = reinterpret_cast<const WorkItem*>(plan + L.bwd_items);
  p.counts = plan + L.counts;
  p.ts = ts;
  p.dq_acc = dq_acc;
  p.dk = dk;
  p.dv = dv;
  p.ldg = ldg;
  p.zk = zk;
  p.zv = zv;
  p.ldz = 4 * (int64_t)HD;
  p.H = H;
  p.scale = 1.0f / sqrtf((float)d);
  p.status = status;
  p.ldacc = HD;
  const int64_t grid = L.max_items * H;
  if (grid > 0x7fffffff) return cudaErrorInvalidValue;
  {
  TraceScope tr("attn_bwd", s);
  if (d == 128) {
    auto kern = attn_bwd_kernel<128>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdCfg<128>::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)grid, NUM_THREADS, BwdCfg<128>::SMEM, s>>>(tq, tk, tv, tdo, p);
  } else if (d == 64) {
    auto kern = attn_bwd_kernel<64>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdCfg<64>::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)grid, NUM_THREADS, BwdCfg<64>::SMEM, s>>>(tq, tk, tv, tdo, p);
  } else {
    return cudaErrorInvalidValue;
  }
  e = cudaGetLastError();
  }
  if (e != cudaSuccess) return e;
  const int64_t n8 = (int64_t)T * HD / 8;
  TraceScope tr2("dq_finish", s);
  dq_finish_kernel<<<(unsigned)((n8 + 255) / 256), 256, 0, s>>>(dq_acc, T, HD, dq, ldg, zq, 4 * (int64_t)HD);
  return cudaGetLastError();
}

}  // namespace mtgr
