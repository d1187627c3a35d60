// attn_bwd_sm103.cu -- jagged HSTU attention backward on the 5th-generation
// tensor cores (tcgen05 + TMEM + TMA): f16 operands (q, k, v, dO, P, dS),
// fp32 accumulation, bf16 or f16 gradients.
//
// With s = q·k / sqrt(d_h), A = M ⊙ silu(s) / n_u and O = A V (marovi.ai
// "Métodos" block formula; paper-daily "模型怎么搭"), the gradients are
//   dV = Aᵀ dO,  dA = dO Vᵀ,  dS = M ⊙ dA ⊙ silu'(s) / (n_u sqrt(d_h)),
//   dQ = dS K,   dK = dSᵀ Q,   silu'(s) = σ(s)(1 + s(1 - σ(s))).
// There is no softmax, so no row statistics are needed: S is recomputed.
//
// Persistent kernels, none of which needs atomics:
//  * dK/dV (key-tile major): one item = (user, key tile, head), looping over
//    the query tiles that see the key tile (dynamic mixed mask, fun-rec
//    chapter 7.3, §7.3.4).  Per query tile: Sᵀ = K Qᵀ and dPᵀ = V dOᵀ in two
//    alternating TMEM regions; the epilogue writes Pᵀ (f16) over Sᵀ and dSᵀ
//    (f16) to shared memory; dV += Pᵀ dO reads Pᵀ from TMEM, dK += dSᵀ Q reads
//    dSᵀ from shared memory.
//  * dQ (query-tile major): one item = (user, query tile, head), looping over
//    the key tiles the query tile sees.  Per key tile: S = Q Kᵀ, dP = dO Vᵀ
//    (two alternating dP buffers); the epilogue writes dS (f16) over dP and
//    dQ += dS K reads it from TMEM.
// Recomputing S and dP in the dQ kernel costs 2 extra MMAs per tile pair but
// avoids accumulating dQ across CTAs through L2 reductions (64 KB of fp32
// read-modify-write per tile pair).  When the caller lends a store for them,
// the dK/dV kernel also copies each dSᵀ tile (32 KB) to HBM and a third
// kernel forms dQ = dS K from the stored tiles: one product per tile pair and
// 64 KB of HBM traffic (written once, read once) instead of two recomputed
// products; the plan decides on the device which dQ kernel runs.
//
// Warps of the dK/dV and recomputing dQ kernels: 0 TMA, 1 the first MMA
// issuer (the score products) + TMEM owner, 2..17 score epilogue (thread =
// TMEM lane = tile row; 4 lane quarters x 4 groups of 32 columns), 18..21
// output (TMEM -> 16-bit gradients), 22 the second MMA issuer (the gradient
// products); 23 in the dK/dV kernel's store instantiation copies the dSᵀ
// tiles to the store.  The dQ kernel that reads the stored tiles has its own
// warp layout (below).
#include "attn_sm103.cuh"

namespace mtgr {
namespace {
using attn::BT;
using attn::item_at;
using attn::silu_and_grad_half;


struct BwdParams {
  const UserInfo* users;
  const WorkItem* items;
  const int32_t* count;  // number of items in the list
  const int64_t* ts;
  uint16_t* g0;  // dkdv kernel: dk; dq kernel: dq (16-bit type TG of the kernel)
  uint16_t* g1;  // dkdv kernel: dv
  int64_t ldg;
  const uint16_t* m0;  // optional multipliers of g0 / g1 (type TG, row stride ldm)
  const uint16_t* m1;
  int64_t ldm;
  int H;
  float scale;  // 1/sqrt(d_h)
  int32_t* status;
  // stored dS tiles (plan.cuh): the dK/dV kernel writes each dS'ᵀ tile to its
  // slot and the dQ pass reads them back, when *ds_on (set by the plan) is 1
  uint8_t* ds_store;
  const int64_t* ds_base;
  const int32_t* ds_on;
};

// ---------------------------------------------------------------------------
// Mask helpers.  Rows / keys are segment-relative; eS, eR: first RealTime and
// first candidate token; n: tokens of the user.
// ---------------------------------------------------------------------------
// Query row ri sees key rj (dynamic mixed mask, fun-rec §7.3.4): User/Seq keys
// always; a RealTime key if ts_j < thr (thr = ts_i + 1 for a RealTime row,
// ts_i for a candidate row, INT64_MIN for a User/Seq row); a candidate key only
// on the diagonal.
struct RowMask {
  int ri;
  bool row_ok, cand;
  int64_t thr;
};
__device__ __forceinline__ RowMask row_mask(const UserInfo& u, const int64_t* ts, int ri) {
  RowMask m;
  m.ri = ri;
  m.row_ok = ri < u.n;
  m.cand = ri >= u.eR;
  m.thr = INT64_MIN;
  if (m.row_ok && ri >= u.eS) m.thr = ts[u.start + ri] + (m.cand ? 0 : 1);
  return m;
}

// =============================================================================
// dQ kernel
// =============================================================================
// Warps: 0 TMA, 1 first MMA issuer (S, dP) + TMEM owner, 2..17 score epilogue
// (thread = query row; 4 lane quarters x 4 groups of 32 key columns), 18..21
// output (TMEM -> 16-bit dQ, one warp per lane quarter), 22 second MMA issuer
// (dQ), so that each issuer waits only for its own operands.
constexpr int DQ_THREADS = 736;  // + the second MMA issuer (warp 22)
constexpr int DQ_EPI = 16;
constexpr int DQ_OUT = 4;

template <int D>
struct DqCfg {
  static constexpr int TILE = BT * D * 2;
  static constexpr int RING = D == 128 ? 5 : 8;  // K / V tiles in flight
  static constexpr int KR = D == 128 ? 3 : 4, VR = RING - KR;  // K stages (held until dQ), V stages
  static constexpr int Q_OFF = 0, DO_OFF = TILE, RING_OFF = 2 * TILE;
  static constexpr int BAR_OFF = RING_OFF + RING * TILE;
  static constexpr int SMEM = BAR_OFF + 512 + 1024;
  // S in columns [0, 128), two dP / dS' buffers in [128, 384), the dQ
  // accumulators after them (one for d_h = 128, two for d_h = 64)
  static constexpr int NQB = 384 + 2 * D <= 512 ? 2 : 1;
  static constexpr uint32_t S_COL = 0;
  __device__ static constexpr uint32_t dp_col(int b) { return 128u + 128u * (uint32_t)b; }
  __device__ static constexpr uint32_t dq_col(int b) { return 384u + (uint32_t)b * D; }
};

struct DqBars {
  uint64_t qdo_full, qdo_empty;
  uint64_t ring_full[8], ring_empty[8];
  uint64_t s_full, s_read, dp_full[2], ds_ready[2], dq_done[2], dq_full[2], dq_free[2];
  uint32_t tmem_base;
  int abort_flag;
};

struct DqItem {
  UserInfo u;
  QTileKeys keys;
  int qt, h, b;
};
__device__ __forceinline__ DqItem dq_item(const BwdParams& p, int idx) {
  DqItem c;
  const WorkItem wi = p.items[idx];
  c.b = wi.b;
  c.h = wi.h();
  c.u = p.users[wi.b];
  c.qt = wi.t();
  c.keys = qtile_keys(c.u, c.qt);
  return c;
}

// 16 scores of one query row, keys j0 .. j0+15 -> 8 packed f16 values of
// M ⊙ silu'(s c) (the factor dS' = M ⊙ silu' ⊙ dP takes once dP is there; dS'
// leaves out c / n_u, which the dQ output applies).  The chunk class depends
// only on j0, so it is uniform across the warp.
__device__ __forceinline__ void dsl_chunk_q(const uint32_t (&sr)[16], int j0, const UserInfo& u, const RowMask& m,
                                            int64_t tk, float hc, uint64_t hc2, uint32_t (&dsl)[8]) {
  if (j0 + 16 <= u.eS) {
#pragma unroll
    for (int e = 0; e < 8; ++e) dsl[e] = attn::dsilu_pair(sr[2 * e], sr[2 * e + 1], hc2);
  } else if (j0 >= u.eR) {
    // candidate keys (or keys past the segment): only the diagonal is visible
    const int ed = m.ri - j0;
    const bool diag = m.cand && m.row_ok && ed >= 0 && ed < 16;
    float s_d = 0.f;
#pragma unroll
    for (int e = 0; e < 16; ++e) s_d = (e == ed) ? __uint_as_float(sr[e]) : s_d;
    float sl, ds;
    silu_and_grad_half(s_d * hc, sl, ds);
    const float vd = diag ? ds : 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) dsl[e] = pack_f16x2((2 * e == ed) ? vd : 0.f, (2 * e + 1 == ed) ? vd : 0.f);
  } else {
    // the chunk overlaps the RealTime keys: branch-free predicate; tk holds the
    // stamp of key j0 + (lane & 15) (attn::rt_key_stamp), broadcast
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      bool vis[2];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int jj = j0 + 2 * e + t;
        vis[t] = (jj < u.eS) | (attn::shfl_i64(tk, 2 * e + t) < m.thr) | (m.cand & (jj == m.ri));
      }
      dsl[e] = attn::dsilu_pair(sr[2 * e], sr[2 * e + 1], hc2) & attn::keep_mask(vis[0], vis[1]);
    }
  }
}

// One item = (user, query tile, head): Q and dO stay in shared memory while
// the key tiles the query tile sees stream through a ring (K_j, then V_j).
// Per key tile j: S = Q K_jᵀ (SS) and dP = dO V_jᵀ (SS) in TMEM; the epilogue
// turns S into M ⊙ silu' (kept in registers) and signals that S may be
// overwritten, then, with dP, writes dS' = M ⊙ silu' ⊙ dP (f16) over dP;
// dQ += dS' K_j accumulates in TMEM with dS' read from TMEM (TS).  dP
// alternates between two buffers, so dP(j+1) runs while the epilogue and
// dQ(j) still use dP(j); the issue order S(j+1), dP(j+1), dQ(j) keeps the
// epilogue, which the transcendental paces, busy.  Q and dO are released after
// the last dP of an item, so the next item's load overlaps its last dQ.
template <int D, typename TG>
__global__ void __launch_bounds__(DQ_THREADS, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                       const BwdParams p) {
  using Cfg = DqCfg<D>;
  constexpr int RING = Cfg::RING;
  constexpr int NQB = Cfg::NQB;
  if (p.ds_on != nullptr && *p.ds_on != 0) return;  // dQ comes from the stored dS tiles instead
  const int total = p.count[0];
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base + Cfg::Q_OFF;
  uint8_t* sdO = base + Cfg::DO_OFF;
  uint8_t* sRing = base + Cfg::RING_OFF;
  DqBars& S = *reinterpret_cast<DqBars*>(base + Cfg::BAR_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&S.qdo_full, 1);
    mbar_init(&S.qdo_empty, 1);
    for (int i = 0; i < RING; ++i) {
      mbar_init(&S.ring_full[i], 1);
      // a K stage is read by S (first issuer) and dQ (second issuer), a V stage by dP
      mbar_init(&S.ring_empty[i], i < Cfg::KR ? 2 : 1);
    }
    mbar_init(&S.s_full, 1);
    mbar_init(&S.s_read, DQ_EPI);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.dp_full[i], 1);
      mbar_init(&S.ds_ready[i], DQ_EPI);
      mbar_init(&S.dq_full[i], 1);
      mbar_init(&S.dq_free[i], DQ_OUT);
      mbar_init(&S.dq_done[i], 1);
    }
    S.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, 512);
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

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer: Q, dO per item; K_j, V_j per key tile ----------------
      // K tiles through a ring of KR stages, V tiles through one of VR stages
      int st[2] = {0, 0};
      uint32_t ph[2] = {0, 0};
      int n_items = 0;
      for (int r = 0; ok; ++r) {
        const int idx = item_at(r);
        if (idx >= total) break;
        const DqItem c = dq_item(p, idx);
        const int col_h = c.h * D;
        if (!mbar_wait_sleepy(&S.qdo_empty, (n_items & 1) ^ 1, abort_flag)) { ok = false; break; }
        ++n_items;
        mbar_arrive_expect_tx(&S.qdo_full, 2 * Cfg::TILE);
#pragma unroll
        for (int cc = 0; cc < D / 64; ++cc) {
          tma_load_2d(sQ + cc * 16384, &tmQ, &S.qdo_full, col_h + 64 * cc, c.u.start + c.qt * BT);
          tma_load_2d(sdO + cc * 16384, &tmdO, &S.qdo_full, col_h + 64 * cc, c.u.start + c.qt * BT);
        }
        const int nk = c.keys.count();
        for (int i = 0; i < nk && ok; ++i) {
          const int row = c.u.start + c.keys.kt(i, c.qt) * BT;
#pragma unroll
          for (int kv = 0; kv < 2; ++kv) {  // K_j, then V_j
            const int slot = (kv ? Cfg::KR : 0) + st[kv];
            if (!mbar_wait_sleepy(&S.ring_empty[slot], ph[kv] ^ 1, abort_flag)) { ok = false; break; }
            uint8_t* dst = sRing + slot * Cfg::TILE;
            mbar_arrive_expect_tx(&S.ring_full[slot], Cfg::TILE);
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc)
              tma_load_2d(dst + cc * 16384, kv == 0 ? &tmK : &tmV, &S.ring_full[slot], col_h + 64 * cc, row);
            if (++st[kv] == (kv ? Cfg::VR : Cfg::KR)) { st[kv] = 0; ph[kv] ^= 1; }
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- first issuer: S(j) = Q K_jᵀ and dP(j) = dO V_jᵀ ----------------
      constexpr uint32_t idesc_s = idesc_f16_f32(BT, BT, false, false);
      const uint32_t q_addr = smem_u32(sQ), do_addr = smem_u32(sdO);
      const uint32_t ring_addr = smem_u32(sRing);
      int ks = 0, vs = 0, n_items = 0;
      uint32_t kph = 0, vph = 0;
      int g = 0;  // global key-tile count of this CTA
      for (int r = 0; ok; ++r) {
        const int idx = item_at(r);
        if (idx >= total) break;
        const DqItem c = dq_item(p, idx);
        if (!mbar_wait(&S.qdo_full, n_items & 1, abort_flag)) { ok = false; break; }
        ++n_items;
        const int nk = c.keys.count();
        for (int i = 0; i < nk; ++i) {
          const int gt = g + i;
          // S(gt) once the epilogue has read S(gt - 1) (one S buffer)
          if (gt >= 1 && !mbar_wait(&S.s_read, (gt - 1) & 1, abort_flag)) { ok = false; break; }
          if (!mbar_wait(&S.ring_full[ks], kph, abort_flag)) { ok = false; break; }
          tc_fence_after();
          {
            const SmemDesc qd = attn::kmajor_base(q_addr), kd = attn::kmajor_base(ring_addr + ks * Cfg::TILE);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              tc_mma_ss_h(tmem + Cfg::S_COL, qd.lo + attn::kmajor_step(kk), qd.hi, kd.lo + attn::kmajor_step(kk),
                          kd.hi, idesc_s, kk > 0 ? 1u : 0u);
          }
          tc_commit(&S.s_full);
          tc_commit(&S.ring_empty[ks]);  // first of the K stage's two readers
          if (++ks == Cfg::KR) { ks = 0; kph ^= 1; }
          // dP(gt) into buffer gt & 1 once dQ(gt - 2) has read dS'(gt - 2) there
          if (gt >= 2 && !mbar_wait(&S.dq_done[gt & 1], ((gt - 2) >> 1) & 1, abort_flag)) { ok = false; break; }
          const int vslot = Cfg::KR + vs;
          if (!mbar_wait(&S.ring_full[vslot], vph, abort_flag)) { ok = false; break; }
          tc_fence_after();
          {
            const SmemDesc od = attn::kmajor_base(do_addr), vd = attn::kmajor_base(ring_addr + vslot * Cfg::TILE);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              tc_mma_ss_h(tmem + Cfg::dp_col(gt & 1), od.lo + attn::kmajor_step(kk), od.hi,
                          vd.lo + attn::kmajor_step(kk), vd.hi, idesc_s, kk > 0 ? 1u : 0u);
          }
          tc_commit(&S.dp_full[gt & 1]);
          tc_commit(&S.ring_empty[vslot]);
          if (++vs == Cfg::VR) { vs = 0; vph ^= 1; }
        }
        if (!ok) break;
        tc_commit(&S.qdo_empty);  // Q and dO are free once the item's S and dP complete
        g += nk;
      }
    }
  } else if (warp == 2 + DQ_EPI + DQ_OUT) {
    if (lane == 0) {
      // ---------------- second issuer: dQ += dS'(j) K_j (dS' read from TMEM) ----------------
      constexpr uint32_t idesc_dq = idesc_f16_f32(BT, D, false, true);
      const uint32_t ring_addr = smem_u32(sRing);
      int ks = 0, n_items = 0;
      int g = 0;
      for (int r = 0; ok; ++r) {
        const int idx = item_at(r);
        if (idx >= total) break;
        const DqItem c = dq_item(p, idx);
        const int it = n_items, qb = it % NQB;
        ++n_items;
        // the accumulator still holds item it - NQB until the output warps have read it
        if (it >= NQB && !mbar_wait(&S.dq_free[qb], ((it - NQB) / NQB) & 1, abort_flag)) { ok = false; break; }
        const int nk = c.keys.count();
        for (int i = 0; i < nk; ++i) {
          const int gi = g + i;
          // dS'(gi) is in TMEM (and S(gi), hence K_gi's load, completed before it)
          if (!mbar_wait(&S.ds_ready[gi & 1], (gi >> 1) & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          {  // keys 16kk..16kk+15: column group kk/2, packed half kk&1
            const SmemDesc kd = attn::mnmajor_base(ring_addr + ks * Cfg::TILE);
            const uint32_t a_t = tmem + Cfg::dp_col(gi & 1);
#pragma unroll
            for (int kk = 0; kk < BT / 16; ++kk)
              tc_mma_ts_h(tmem + Cfg::dq_col(qb), a_t + 32 * (kk >> 1) + 8 * (kk & 1), kd.lo + attn::mnmajor_step(kk),
                          kd.hi, idesc_dq, (i > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(&S.dq_done[gi & 1]);
          tc_commit(&S.ring_empty[ks]);  // second reader of the K stage
          if (++ks == Cfg::KR) ks = 0;
        }
        if (!ok) break;
        tc_commit(&S.dq_full[qb]);
        g += nk;
      }
    }
  } else if (warp < 2 + DQ_EPI) {
    // ---------------- dS' epilogue (thread = query row) ----------------
    const int ew = warp - 2;
    const int kg = ew >> 2;  // group of 32 key columns
    const int quarter = warp & 3;
    const uint32_t lane_sel = (uint32_t)(quarter * 32) << 16;
    const int qr = quarter * 32 + lane;  // query row inside the tile
    const float hc = 0.5f * p.scale;
    const uint64_t hc2 = attn::f2(__float_as_uint(hc), __float_as_uint(hc));
    int g = 0;
    for (int r = 0; ok; ++r) {
      const int idx = item_at(r);
      if (idx >= total) break;
      const DqItem c = dq_item(p, idx);
      const UserInfo& u = c.u;
      const RowMask m = row_mask(u, p.ts, c.qt * BT + qr);
      const int64_t* ts_u = p.ts + u.start;
      const int nk = c.keys.count();
      for (int i = 0; i < nk && ok; ++i) {
        const int gi = g + i, b = gi & 1;
        const int j0 = c.keys.kt(i, c.qt) * BT + kg * 32;  // first key of this warp's group
        // stamps of the keys this lane broadcasts, loaded before the wait
        const int64_t tk0 = attn::rt_key_stamp(u, ts_u, j0, lane), tk1 = attn::rt_key_stamp(u, ts_u, j0 + 16, lane);
        // phase 1: M ⊙ silu' from S
        if (!mbar_wait(&S.s_full, gi & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        uint32_t buf[2][16], dsl[2][8];
        tmem_ld16(tmem + Cfg::S_COL + kg * 32 + lane_sel, buf[0]);
        tmem_ld16(tmem + Cfg::S_COL + kg * 32 + 16 + lane_sel, buf[1]);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.s_read);  // the tensor core may overwrite S
        dsl_chunk_q(buf[0], j0, u, m, tk0, hc, hc2, dsl[0]);
        dsl_chunk_q(buf[1], j0 + 16, u, m, tk1, hc, hc2, dsl[1]);
        // phase 2: dS' = (M ⊙ silu') ⊙ dP, packed f16 over the first 16 columns
        // of this warp's 32 (which only this warp reads)
        if (!mbar_wait(&S.dp_full[b], (gi >> 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t t_dp = tmem + Cfg::dp_col(b) + kg * 32 + lane_sel;
        tmem_ld16(t_dp, buf[0]);
        tmem_ld16(t_dp + 16, buf[1]);
        tmem_wait_ld();
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          uint32_t pd[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) pd[e] = attn::ds_pair(dsl[ch][e], buf[ch][2 * e], buf[ch][2 * e + 1]);
          tmem_st8(t_dp + 8 * ch, pd);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.ds_ready[b]);
      }
      g += nk;
    }
  } else {
    // ---------------- dQ output (thread = query row) ----------------
    const int quarter = warp & 3;
    const uint32_t lane_sel = (uint32_t)(quarter * 32) << 16;
    const bool has_m = p.m0 != nullptr;
    constexpr int NC = D / 32;
    int n_items = 0;
    for (int r = 0; ok; ++r) {
      const int idx = item_at(r);
      if (idx >= total) break;
      const DqItem c = dq_item(p, idx);
      const int qb = n_items % NQB;
      const uint32_t par = (n_items / NQB) & 1;
      ++n_items;
      const int rl = c.qt * BT + quarter * 32 + lane;  // this lane's query row, segment-relative
      const bool row_ok = rl < c.u.n;
      const bool any = c.keys.count() > 0;
      const int64_t grow = (int64_t)c.u.start + rl;
      const float cn = p.scale / (float)c.u.nu;  // the factor c / n_u left out of dS'
      const uint16_t* mrow = has_m ? p.m0 + grow * p.ldm + c.h * D : nullptr;
      if (has_m && row_ok) prefetch_l2(mrow, D * 2);
      if (!mbar_wait_sleepy(&S.dq_full[qb], par, abort_flag)) { ok = false; break; }
      tc_fence_after();
      uint16_t* orow = p.g0 + grow * p.ldg + c.h * D;
#pragma unroll 1
      for (int cc = 0; cc < NC; ++cc) {
        uint32_t rr[32];
        tmem_ld32(tmem + Cfg::dq_col(qb) + cc * 32 + lane_sel, rr);
        uint4 mm[4];  // the multipliers of this chunk load while the TMEM read completes
        if (has_m && row_ok) {
#pragma unroll
          for (int v = 0; v < 4; ++v) mm[v] = *reinterpret_cast<const uint4*>(mrow + cc * 32 + 8 * v);
        }
        tmem_wait_ld();
        if (cc == NC - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.dq_free[qb]);
        }
        if (!row_ok) continue;
        float x[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] = any ? __uint_as_float(rr[e]) * cn : 0.f;
        if (has_m) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const uint32_t w[4] = {mm[v].x, mm[v].y, mm[v].z, mm[v].w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              x[8 * v + 2 * t] *= lo16<TG>(w[t]);
              x[8 * v + 2 * t + 1] *= hi16<TG>(w[t]);
            }
          }
        }
#pragma unroll
        for (int v = 0; v < 4; ++v) *reinterpret_cast<uint4*>(orow + cc * 32 + 8 * v) = pack8<TG>(x + 8 * v);
      }
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
    tmem_dealloc(tmem, 512);
  }
}

// =============================================================================
// dQ from the stored dS tiles
// =============================================================================
// When the dK/dV kernel has kept its dS'ᵀ tiles, dQ needs one product per
// tile pair instead of three: dQ += dS' K_j, with dS' read straight from the
// stored [128 keys][128 queries] tile (the MN-major form of the A operand) and
// K_j MN-major as in the recomputing kernel.  The kernel streams 32 KB of dS'
// per tile pair from HBM, so memory, not the tensor core, sets its pace.
// Warps: 0 loads (bulk copy of the dS'ᵀ tile, TMA of K_j), 1 MMA issuer +
// TMEM owner, 2..9 output (TMEM -> 16-bit dQ; 4 lane quarters x 2 column
// halves).  Two dQ accumulators of d_h columns alternate between items.
constexpr int DQS_THREADS = 320;
constexpr int DQS_OUT = 8;

template <int D>
struct DqsCfg {
  static constexpr int KTILE = BT * D * 2;
  static constexpr int STAGE = kDsTileBytes + KTILE;  // [dS'ᵀ tile][K_j], both 1024-byte aligned
  static constexpr int STAGES = D == 128 ? 3 : 4;
  static constexpr int BAR_OFF = STAGES * STAGE;
  static constexpr int SMEM = BAR_OFF + 256 + 1024;
  static constexpr int TMEM_COLS = 2 * D;  // 256 or 128
};

struct DqsBars {
  uint64_t full[4], empty[4], acc_full[2], acc_free[2];
  uint32_t tmem_base;
  int abort_flag;
};

template <int D, typename TG>
__global__ void __launch_bounds__(DQS_THREADS, 1)
    attn_bwd_dq_ds_kernel(const __grid_constant__ CUtensorMap tmK, const BwdParams p) {
  using Cfg = DqsCfg<D>;
  constexpr int ST = Cfg::STAGES;
  if (p.ds_on == nullptr || *p.ds_on == 0) return;  // the tiles were not kept: the recomputing kernel runs
  const int total = p.count[0];
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  DqsBars& S = *reinterpret_cast<DqsBars*>(base + Cfg::BAR_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < ST; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.acc_full[i], 1);
      mbar_init(&S.acc_free[i], DQS_OUT);
    }
    S.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) tma_prefetch_desc(&tmK);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  volatile int* abort_flag = &S.abort_flag;
  bool ok = true;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- loads: per key tile j, the stored dS'ᵀ(qt, j) and K_j ----------------
      int st = 0;
      uint32_t ph = 0;
      for (int r = 0; ok; ++r) {
        const int idx = item_at(r);
        if (idx >= total) break;
        const DqItem c = dq_item(p, idx);
        const int nt = ceil_div(c.u.n, BT);
        const int64_t b0 = p.ds_base[c.b];
        const int nk = c.keys.count();
        for (int j = 0; j < nk; ++j) {
          const int kt = c.keys.kt(j, c.qt);
          if (!mbar_wait_sleepy(&S.empty[st], ph ^ 1, abort_flag)) { ok = false; break; }
          uint8_t* dst = base + st * Cfg::STAGE;
          mbar_arrive_expect_tx(&S.full[st], Cfg::STAGE);
          bulk_load(dst, p.ds_store + ds_slot(b0, nt, c.h, kt, c.qt) * kDsTileBytes, kDsTileBytes, &S.full[st]);
#pragma unroll
          for (int cc = 0; cc < D / 64; ++cc)
            tma_load_2d(dst + kDsTileBytes + cc * 16384, &tmK, &S.full[st], c.h * D + 64 * cc, c.u.start + kt * BT);
          if (++st == ST) { st = 0; ph ^= 1; }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer: dQ(item) += dS'(j) K_j into accumulator it & 1 ----------------
      constexpr uint32_t idesc = idesc_f16_f32(BT, D, true, true);
      const uint32_t sbase = smem_u32(base);
      int st = 0;
      uint32_t ph = 0;
      int it = 0;
      for (int r = 0; ok; ++r, ++it) {
        const int idx = item_at(r);
        if (idx >= total) break;
        const DqItem c = dq_item(p, idx);
        const int ab = it & 1;
        // the accumulator holds item it - 2 until the output warps have read it
        if (it >= 2 && !mbar_wait(&S.acc_free[ab], ((it - 2) >> 1) & 1, abort_flag)) { ok = false; break; }
        const int nk = c.keys.count();
        for (int j = 0; j < nk; ++j) {
          if (!mbar_wait(&S.full[st], ph, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = sbase + st * Cfg::STAGE;
          const SmemDesc ad = attn::mnmajor_base(sa), bd = attn::mnmajor_base(sa + kDsTileBytes);
#pragma unroll
          for (int kk = 0; kk < BT / 16; ++kk)  // keys 16kk .. 16kk+15
            tc_mma_ss_h(tmem + ab * D, ad.lo + attn::mnmajor_step(kk), ad.hi, bd.lo + attn::mnmajor_step(kk), bd.hi,
                        idesc, (j > 0 || kk > 0) ? 1u : 0u);
          tc_commit(&S.empty[st]);
          if (++st == ST) { st = 0; ph ^= 1; }
        }
        if (!ok) break;
        tc_commit(&S.acc_full[ab]);
      }
    }
  } else {
    // ---------------- dQ output (thread = query row; this warp's half of the columns) ----------------
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const uint32_t lane_sel = (uint32_t)(quarter * 32) << 16;
    const bool has_m = p.m0 != nullptr;
    constexpr int NC = D / 64;  // 32-column chunks per half
    int it = 0;
    for (int r = 0; ok; ++r, ++it) {
      const int idx = item_at(r);
      if (idx >= total) break;
      const DqItem c = dq_item(p, idx);
      const int ab = it & 1;
      const int rl = c.qt * BT + quarter * 32 + lane;  // this lane's query row, segment-relative
      const bool row_ok = rl < c.u.n;
      const bool any = c.keys.count() > 0;
      const int64_t grow = (int64_t)c.u.start + rl;
      const float cn = p.scale / (float)c.u.nu;  // the factor c / n_u left out of dS'
      const int col0 = half * (D / 2);
      const uint16_t* mrow = has_m ? p.m0 + grow * p.ldm + c.h * D + col0 : nullptr;
      if (has_m && row_ok) prefetch_l2(mrow, D);
      if (!mbar_wait_sleepy(&S.acc_full[ab], (it >> 1) & 1, abort_flag)) { ok = false; break; }
      tc_fence_after();
      uint16_t* orow = p.g0 + grow * p.ldg + c.h * D + col0;
#pragma unroll 1
      for (int cc = 0; cc < NC; ++cc) {
        uint32_t rr[32];
        tmem_ld32(tmem + ab * D + col0 + cc * 32 + lane_sel, rr);
        uint4 mm[4];  // the multipliers of this chunk load while the TMEM read completes
        if (has_m && row_ok) {
#pragma unroll
          for (int v = 0; v < 4; ++v) mm[v] = *reinterpret_cast<const uint4*>(mrow + cc * 32 + 8 * v);
        }
        tmem_wait_ld();
        if (cc == NC - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.acc_free[ab]);
        }
        if (!row_ok) continue;
        float x[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] = any ? __uint_as_float(rr[e]) * cn : 0.f;
        if (has_m) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const uint32_t w[4] = {mm[v].x, mm[v].y, mm[v].z, mm[v].w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              x[8 * v + 2 * t] *= lo16<TG>(w[t]);
              x[8 * v + 2 * t + 1] *= hi16<TG>(w[t]);
            }
          }
        }
#pragma unroll
        for (int v = 0; v < 4; ++v) *reinterpret_cast<uint4*>(orow + cc * 32 + 8 * v) = pack8<TG>(x + 8 * v);
      }
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

// =============================================================================
// dK/dV kernel
// =============================================================================
// Warps: 0 TMA, 1 first MMA issuer (Sᵀ, dPᵀ) + TMEM owner, 2..17 score
// epilogue (thread = key row; 4 lane quarters x 4 groups of 32 query columns),
// 18..21 output (TMEM -> 16-bit dV then dK, one warp per lane quarter), 22
// second MMA issuer (dV, dK), and in the STORE instantiation 23, the dS'ᵀ tile
// store (launched when the caller lends a store for the dQ pass).  Both
// instantiations are compiled for 24 warps (80 registers a thread): with the
// budget of 23 warps the compiler spills more in the epilogue.
constexpr int dkv_threads(bool store) { return store ? 768 : 736; }
constexpr int DKV_EPI = 16;
constexpr int DKV_OUT = 4;

template <int D>
struct DkvCfg {
  static constexpr int TILE = BT * D * 2;
  static constexpr int RING = D == 128 ? 4 : 8;  // Q / dO tiles in flight
  static constexpr int K_OFF = 0, V_OFF = TILE, DS_OFF = 2 * TILE;
  static constexpr int RING_OFF = DS_OFF + BT * BT * 2;  // dSᵀ: [128 keys][128 queries] f16
  static constexpr int BAR_OFF = RING_OFF + RING * TILE;
  static constexpr int SMEM = BAR_OFF + 512 + 1024;
  // two 128-column score regions: Sᵀ (then Pᵀ) of query tile g in region g & 1,
  // dPᵀ of tile g in the other one
  __device__ static constexpr uint32_t r_col(int b) { return (uint32_t)b * 128u; }
  static constexpr uint32_t DV_COL = 256, DK_COL = 256 + D;
};

struct DkvBars {
  uint64_t kv_full, kv_empty;
  uint64_t ring_full[8], ring_empty[8];
  uint64_t s_full, dp_full, p_ready[2], dp_read, ds_ready, pv_done[2], dk_done, dkdv_full, dv_free, dk_free;
  uint64_t ds_copied;  // the store has read dS'ᵀ(g) out of shared memory
  uint32_t tmem_base;
  int abort_flag;
};

struct DkvItem {
  UserInfo u;
  KTileQueries qs;
  int kt, h, b;
};
__device__ __forceinline__ DkvItem dkv_item(const BwdParams& p, int idx) {
  DkvItem c;
  const WorkItem wi = p.items[idx];
  c.b = wi.b;
  c.h = wi.h();
  c.u = p.users[wi.b];
  c.kt = wi.t();
  c.qs = ktile_queries(c.u, c.kt);
  return c;
}

// Key row rj as seen by query rows (the transposed mask): User/Seq keys by
// every row of the segment; a RealTime key by RealTime rows stamped at or after
// it and candidate rows stamped after it; a candidate key only by itself.
struct KeyMask {
  int rj;
  int cls;  // 0 User/Seq, 1 RealTime, 2 candidate, 3 past the segment
  int64_t ts_j;
};

// Stamp threshold of query row rq for the RealTime test of the transposed mask:
// ts_i + 1 for a RealTime row, ts_i for a candidate row, INT64_MIN for a
// User/Seq row or a row past the segment.
__device__ __forceinline__ int64_t query_adj(const UserInfo& u, const int64_t* ts_u, int rq) {
  return (rq >= u.eS && rq < u.n) ? __ldg(ts_u + rq) + (rq < u.eR ? 1 : 0) : INT64_MIN;
}

// 16 scores sᵀ of one key row, query rows q0 .. q0+15 -> 8 packed f16 Pᵀ
// values (silu, without 1/n_u) and 8 packed f16 values of M ⊙ silu' (the
// factor that dS'ᵀ = M ⊙ silu' ⊙ dPᵀ takes once dPᵀ is there; dS' leaves out
// c / n_u, which the dK output applies).  warp_us: every key of the warp is
// User/Seq (warp-uniform).  hc2: (c/2, c/2) as an f32 pair.
__device__ __forceinline__ void p_chunk_k(const uint32_t (&sr)[16], int q0, const UserInfo& u, const KeyMask& k,
                                          bool warp_us, int64_t adj, uint64_t hc2, uint32_t (&pp)[8],
                                          uint32_t (&dsl)[8]) {
  if (warp_us && q0 + 16 <= u.n) {
    // every key of the warp is User/Seq and every query row lies in the segment
#pragma unroll
    for (int e = 0; e < 8; ++e) attn::silu_pair_split(sr[2 * e], sr[2 * e + 1], hc2, pp[e], dsl[e]);
  } else {
    // Query row ri sees a RealTime key stamped ts_j iff ts_j < adj_i (see
    // query_adj); adj holds adj_{q0 + (lane & 15)} and is broadcast.
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      bool vis[2];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int ri = q0 + 2 * e + t;
        const int64_t adj_i = attn::shfl_i64(adj, 2 * e + t);
        vis[t] = ((k.cls == 0) & (ri < u.n)) | ((k.cls == 1) & (k.ts_j < adj_i)) | ((k.cls == 2) & (ri == k.rj));
      }
      attn::silu_pair_split(sr[2 * e], sr[2 * e + 1], hc2, pp[e], dsl[e]);
      const uint32_t mk = attn::keep_mask(vis[0], vis[1]);
      pp[e] &= mk;
      dsl[e] &= mk;
    }
  }
}

// One item = (user, key tile, head): K and V stay in shared memory while the
// query tiles that see the key tile stream through a ring (Q_i, then dO_i).
// Per query tile g (counted over the CTA's items) the tensor core computes
//   Sᵀ = K Q_gᵀ into TMEM region g & 1,  dPᵀ = V dO_gᵀ into region (g+1) & 1;
// the epilogue writes Pᵀ = M ⊙ silu(Sᵀ c) (f16) over Sᵀ as soon as Sᵀ is there
// (keeping M ⊙ silu' in registers), then, once dPᵀ is there, dS'ᵀ = M ⊙ silu'
// ⊙ dPᵀ (f16) to shared memory; the tensor core adds
//   dV += Pᵀ dO_g  (A from TMEM),  dK += dS'ᵀ Q_g  (A from shared memory).
// The epilogue signals three points of tile g: Pᵀ(g) written (dV(g) may
// start), dPᵀ(g) read into registers (Sᵀ(g+1) may take its region) and dS'ᵀ(g)
// stored (dK(g) may start).  Two warps issue the products, each waiting only
// for its own operands: the first Sᵀ(g+1) then dPᵀ(g+1) (into the region Pᵀ(g)
// leaves once dV(g) has read it), the second dV(g) then dK(g); a Q or dO stage
// of the ring is free once both have read it.
template <int D, typename TG, bool STORE>
__global__ void __launch_bounds__(768, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                         const BwdParams p) {
  using Cfg = DkvCfg<D>;
  constexpr int RING = Cfg::RING;
  const int total = p.count[0];
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = base + Cfg::K_OFF;
  uint8_t* sV = base + Cfg::V_OFF;
  uint8_t* sDS = base + Cfg::DS_OFF;
  uint8_t* sRing = base + Cfg::RING_OFF;
  DkvBars& S = *reinterpret_cast<DkvBars*>(base + Cfg::BAR_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&S.kv_full, 1);
    mbar_init(&S.kv_empty, 1);
    for (int i = 0; i < RING; ++i) {
      mbar_init(&S.ring_full[i], 1);
      mbar_init(&S.ring_empty[i], 2);  // read by both issuers (Q: Sᵀ and dK; dO: dPᵀ and dV)
    }
    mbar_init(&S.s_full, 1);
    mbar_init(&S.dp_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.p_ready[i], DKV_EPI);
      mbar_init(&S.pv_done[i], 1);
    }
    mbar_init(&S.dp_read, DKV_EPI);
    mbar_init(&S.ds_ready, DKV_EPI);
    mbar_init(&S.dk_done, 1);
    mbar_init(&S.dkdv_full, 1);
    mbar_init(&S.dv_free, DKV_OUT);
    mbar_init(&S.dk_free, DKV_OUT);
    mbar_init(&S.ds_copied, 1);
    S.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, 512);
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
  const bool store_on = STORE && p.ds_on != nullptr && *p.ds_on != 0;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer: K, V per item; Q_i, dO_i per query tile ----------------
      int stage = 0, n_items = 0;
      uint32_t ph = 0;
      for (int r = 0; ok; ++r) {
        const int idx = item_at(r);
        if (idx >= total) break;
        const DkvItem c = dkv_item(p, idx);
        const int col_h = c.h * D;
        if (!mbar_wait_sleepy(&S.kv_empty, (n_items & 1) ^ 1, abort_flag)) { ok = false; break; }
        ++n_items;
        mbar_arrive_expect_tx(&S.kv_full, 2 * Cfg::TILE);
#pragma unroll
        for (int cc = 0; cc < D / 64; ++cc) {
          tma_load_2d(sK + cc * 16384, &tmK, &S.kv_full, col_h + 64 * cc, c.u.start + c.kt * BT);
          tma_load_2d(sV + cc * 16384, &tmV, &S.kv_full, col_h + 64 * cc, c.u.start + c.kt * BT);
        }
        const int nq = c.qs.count();
        for (int i = 0; i < nq && ok; ++i) {
          const int row = c.u.start + c.qs.qt(i, c.kt) * BT;
#pragma unroll
          for (int which = 0; which < 2; ++which) {  // Q_i, then dO_i
            if (!mbar_wait_sleepy(&S.ring_empty[stage], ph ^ 1, abort_flag)) { ok = false; break; }
            uint8_t* dst = sRing + stage * Cfg::TILE;
            mbar_arrive_expect_tx(&S.ring_full[stage], Cfg::TILE);
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc)
              tma_load_2d(dst + cc * 16384, which == 0 ? &tmQ : &tmdO, &S.ring_full[stage], col_h + 64 * cc, row);
            if (++stage == RING) { stage = 0; ph ^= 1; }
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- first issuer: Sᵀ(g) = K Q_gᵀ and dPᵀ(g) = V dO_gᵀ ----------------
      constexpr uint32_t idesc_s = idesc_f16_f32(BT, BT, false, false);
      const uint32_t k_addr = smem_u32(sK), v_addr = smem_u32(sV);
      const uint32_t ring_addr = smem_u32(sRing);
      int stage = 0, n_items = 0;
      uint32_t ph = 0;
      int g = 0;  // global query-tile count of this CTA
      auto next_stage = [&](int& st) -> bool {
        if (!mbar_wait(&S.ring_full[stage], ph, abort_flag)) return false;
        st = stage;
        if (++stage == RING) { stage = 0; ph ^= 1; }
        return true;
      };
      for (int r = 0; ok; ++r) {
        const int idx = item_at(r);
        if (idx >= total) break;
        const DkvItem c = dkv_item(p, idx);
        if (!mbar_wait(&S.kv_full, n_items & 1, abort_flag)) { ok = false; break; }
        ++n_items;
        const int nq = c.qs.count();
        for (int i = 0; i < nq; ++i) {
          const int gt = g + i;
          int q_s = 0, do_s = 0;
          // Sᵀ(gt) into region gt & 1 once the epilogue has read dPᵀ(gt - 1) there
          if (gt >= 1 && !mbar_wait(&S.dp_read, (gt - 1) & 1, abort_flag)) { ok = false; break; }
          if (!next_stage(q_s)) { ok = false; break; }
          tc_fence_after();
          {
            const SmemDesc kd = attn::kmajor_base(k_addr), qd = attn::kmajor_base(ring_addr + q_s * Cfg::TILE);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              tc_mma_ss_h(tmem + Cfg::r_col(gt & 1), kd.lo + attn::kmajor_step(kk), kd.hi, qd.lo + attn::kmajor_step(kk),
                          qd.hi, idesc_s, kk > 0 ? 1u : 0u);
          }
          tc_commit(&S.s_full);
          tc_commit(&S.ring_empty[q_s]);
          // dPᵀ(gt) into region (gt + 1) & 1 once dV(gt - 1) has read Pᵀ(gt - 1) there
          if (gt >= 1 && !mbar_wait(&S.pv_done[(gt - 1) & 1], ((gt - 1) >> 1) & 1, abort_flag)) { ok = false; break; }
          if (!next_stage(do_s)) { ok = false; break; }
          tc_fence_after();
          {
            const SmemDesc vd = attn::kmajor_base(v_addr), od = attn::kmajor_base(ring_addr + do_s * Cfg::TILE);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              tc_mma_ss_h(tmem + Cfg::r_col((gt + 1) & 1), vd.lo + attn::kmajor_step(kk), vd.hi,
                          od.lo + attn::kmajor_step(kk), od.hi, idesc_s, kk > 0 ? 1u : 0u);
          }
          tc_commit(&S.dp_full);
          tc_commit(&S.ring_empty[do_s]);
        }
        if (!ok) break;
        tc_commit(&S.kv_empty);  // K and V are free once the item's Sᵀ and dPᵀ complete
        g += nq;
      }
    }
  } else if (warp == 2 + DKV_EPI + DKV_OUT) {
    if (lane == 0) {
      // ---------------- second issuer: dV += Pᵀ dO_g (Pᵀ from TMEM), dK += dS'ᵀ Q_g ----------------
      constexpr uint32_t idesc_g = idesc_f16_f32(BT, D, false, true);
      const uint32_t ds_addr = smem_u32(sDS);
      const uint32_t ring_addr = smem_u32(sRing);
      int stage = 0, n_items = 0;
      uint32_t ph = 0;
      int g = 0;
      for (int r = 0; ok; ++r) {
        const int idx = item_at(r);
        if (idx >= total) break;
        const DkvItem c = dkv_item(p, idx);
        const int it = n_items;
        ++n_items;
        // dV and dK of item it - 1 stay in TMEM until the output warps have read them
        bool dv_ok = it == 0, dk_ok = it == 0;
        auto wait_free = [&](bool& flag, uint64_t* bar) -> bool {
          if (flag) return true;
          flag = true;
          return mbar_wait(bar, (it - 1) & 1, abort_flag);
        };
        const int nq = c.qs.count();
        for (int i = 0; i < nq; ++i) {
          const int gi = g + i;
          const int q_s = stage, do_s = (stage + 1) % RING;  // the ring holds Q_g, then dO_g
          const uint32_t ph_q = ph, ph_do = (stage + 1 == RING) ? ph ^ 1 : ph;
          if ((stage += 2) >= RING) { stage -= RING; ph ^= 1; }
          if (!mbar_wait(&S.p_ready[gi & 1], (gi >> 1) & 1, abort_flag) || !wait_free(dv_ok, &S.dv_free) ||
              !mbar_wait(&S.ring_full[do_s], ph_do, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          {  // dV += Pᵀ dO_g: Pᵀ packed in region g & 1 (query rows 16kk..: column 32(kk/2) + 8(kk%2))
            const SmemDesc od = attn::mnmajor_base(ring_addr + do_s * Cfg::TILE);
#pragma unroll
            for (int kk = 0; kk < BT / 16; ++kk)
              tc_mma_ts_h(tmem + Cfg::DV_COL, tmem + Cfg::r_col(gi & 1) + 32 * (kk >> 1) + 8 * (kk & 1),
                          od.lo + attn::mnmajor_step(kk), od.hi, idesc_g, (i > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(&S.pv_done[gi & 1]);
          tc_commit(&S.ring_empty[do_s]);
          if (!mbar_wait(&S.ds_ready, gi & 1, abort_flag) || !wait_free(dk_ok, &S.dk_free) ||
              !mbar_wait(&S.ring_full[q_s], ph_q, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          {  // dK += dS'ᵀ Q_g
            const SmemDesc sd = attn::kmajor_base(ds_addr), qd = attn::mnmajor_base(ring_addr + q_s * Cfg::TILE);
#pragma unroll
            for (int kk = 0; kk < BT / 16; ++kk)
              tc_mma_ss_h(tmem + Cfg::DK_COL, sd.lo + attn::kmajor_step(kk), sd.hi, qd.lo + attn::mnmajor_step(kk),
                          qd.hi, idesc_g, (i > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(&S.dk_done);
          tc_commit(&S.ring_empty[q_s]);
        }
        // (an item without query tiles has not waited for the accumulators yet)
        if (!ok || !wait_free(dv_ok, &S.dv_free) || !wait_free(dk_ok, &S.dk_free)) {
          ok = false;
          break;
        }
        g += nq;
        tc_commit(&S.dkdv_full);
      }
    }
  } else if (STORE && warp == 3 + DKV_EPI + DKV_OUT) {
    // ---------------- dS'ᵀ store: each tile the epilogue leaves in shared memory
    // also goes, by one bulk copy, to its slot of the caller's store ----------------
    if (store_on && lane == 0) {
      const uint64_t pol = l2_evict_first();  // written once, read once by the dQ pass
      int g = 0;
      for (int r = 0; ok; ++r) {
        const int idx = item_at(r);
        if (idx >= total) break;
        const DkvItem c = dkv_item(p, idx);
        const int nt = ceil_div(c.u.n, BT);
        const int64_t b0 = p.ds_base[c.b];
        const int nq = c.qs.count();
        for (int i = 0; i < nq; ++i) {
          const int gi = g + i;
          if (!mbar_wait(&S.ds_ready, gi & 1, abort_flag)) { ok = false; break; }
          const int64_t slot = ds_slot(b0, nt, c.h, c.kt, c.qs.qt(i, c.kt));
          bulk_store(p.ds_store + slot * kDsTileBytes, sDS, kDsTileBytes, pol);
          tma_store_commit();
          tma_store_wait_read_n<0>();  // the epilogue may write dS'ᵀ(gi + 1) once the copy has read the tile
          mbar_arrive(&S.ds_copied);
        }
        if (!ok) break;
        g += nq;
      }
      tma_store_wait_all();
    }
  } else if (warp < 2 + DKV_EPI) {
    // ---------------- Pᵀ / dS'ᵀ epilogue (thread = key row) ----------------
    const int ew = warp - 2;
    const int qg = ew >> 2;  // group of 32 query columns
    const int quarter = warp & 3;
    const uint32_t lane_sel = (uint32_t)(quarter * 32) << 16;
    const int kr = quarter * 32 + lane;  // key row inside the tile
    const float hc = 0.5f * p.scale;
    const uint64_t hc2 = attn::f2(__float_as_uint(hc), __float_as_uint(hc));
    // this thread's row of dS'ᵀ in the query box of this group; its 16-byte
    // pieces 4 (qg & 1) .. +3 at their 128-byte-swizzle positions
    uint8_t* ds_row = sDS + (qg >> 1) * 16384 + kr * 128;
    const int jb = 4 * (qg & 1);
    int g = 0;
    for (int r = 0; ok; ++r) {
      const int idx = item_at(r);
      if (idx >= total) break;
      const DkvItem c = dkv_item(p, idx);
      const UserInfo& u = c.u;
      KeyMask km;
      km.rj = c.kt * BT + kr;
      km.cls = km.rj < u.eS ? 0 : (km.rj < u.eR ? 1 : (km.rj < u.n ? 2 : 3));
      km.ts_j = km.cls == 1 ? p.ts[u.start + km.rj] : 0;
      const bool warp_us = __all_sync(0xffffffffu, km.cls == 0);
      const bool any_rt = __any_sync(0xffffffffu, km.cls == 1);
      const int64_t* ts_u = p.ts + u.start;
      const int nq = c.qs.count();
      for (int i = 0; i < nq && ok; ++i) {
        const int gi = g + i;
        const int q0 = c.qs.qt(i, c.kt) * BT + qg * 32;  // first query row of this warp's group
        // stamps of the query rows this lane broadcasts in the masked chunks,
        // loaded before the wait so that their latency is hidden
        const int64_t adj0 = any_rt ? query_adj(u, ts_u, q0 + (lane & 15)) : INT64_MIN;
        const int64_t adj1 = any_rt ? query_adj(u, ts_u, q0 + 16 + (lane & 15)) : INT64_MIN;
        // phase 1: Pᵀ and M ⊙ silu' from Sᵀ
        if (!mbar_wait(&S.s_full, gi & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t t_s = tmem + Cfg::r_col(gi & 1) + qg * 32 + lane_sel;
        const uint32_t t_d = tmem + Cfg::r_col((gi + 1) & 1) + qg * 32 + lane_sel;
        uint32_t buf[2][16], pp[8], dsl[2][8];
        tmem_ld16(t_s, buf[0]);
        tmem_ld16(t_s + 16, buf[1]);
        tmem_wait_ld();
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          p_chunk_k(buf[ch], q0 + 16 * ch, u, km, warp_us, ch ? adj1 : adj0, hc2, pp, dsl[ch]);
          tmem_st8(t_s + 8 * ch, pp);  // Pᵀ over Sᵀ columns this warp has read
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.p_ready[gi & 1]);  // dV(gi) may read Pᵀ
        // phase 2: dS'ᵀ = (M ⊙ silu') ⊙ dPᵀ, once dPᵀ is there and dK(gi - 1)
        // has finished reading the shared dS'ᵀ tile
        if (!mbar_wait(&S.dp_full, gi & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        tmem_ld16(t_d, buf[0]);
        tmem_ld16(t_d + 16, buf[1]);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.dp_read);  // Sᵀ(gi + 1) may overwrite dPᵀ
        uint4 pd[4];  // the row's 32 values of dS'ᵀ as four 16-byte pieces
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          uint32_t w[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) w[e] = attn::ds_pair(dsl[ch][e], buf[ch][2 * e], buf[ch][2 * e + 1]);
          pd[2 * ch] = make_uint4(w[0], w[1], w[2], w[3]);
          pd[2 * ch + 1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
        // the shared tile is free once dK(gi - 1) and (with the store) its copy have read it
        if (gi >= 1 && !mbar_wait(&S.dk_done, (gi - 1) & 1, abort_flag)) { ok = false; break; }
        if (store_on && gi >= 1 && !mbar_wait(&S.ds_copied, (gi - 1) & 1, abort_flag)) { ok = false; break; }
#pragma unroll
        for (int v = 0; v < 4; ++v) *reinterpret_cast<uint4*>(ds_row + (((jb + v) ^ (kr & 7)) * 16)) = pd[v];
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.ds_ready);
      }
      g += nq;
    }
  } else {
    // ---------------- dV / dK output (thread = key row) ----------------
    const int quarter = warp & 3;
    const uint32_t lane_sel = (uint32_t)(quarter * 32) << 16;
    const bool has_m = p.m0 != nullptr && p.m1 != nullptr;
    constexpr int NC = D / 32;
    int n_items = 0;
    for (int r = 0; ok; ++r) {
      const int idx = item_at(r);
      if (idx >= total) break;
      const DkvItem c = dkv_item(p, idx);
      const int rl = c.kt * BT + quarter * 32 + lane;  // this lane's key row, segment-relative
      const bool row_ok = rl < c.u.n;
      const bool any = c.qs.count() > 0;
      const int64_t grow = (int64_t)c.u.start + rl;
      const float inv_n = 1.0f / (float)c.u.nu;
      if (has_m && row_ok) {
        prefetch_l2(p.m1 + grow * p.ldm + c.h * D, D * 2);
        prefetch_l2(p.m0 + grow * p.ldm + c.h * D, D * 2);
      }
      if (!mbar_wait_sleepy(&S.dkdv_full, n_items & 1, abort_flag)) { ok = false; break; }
      ++n_items;
      tc_fence_after();
#pragma unroll 1
      for (int ch = 0; ch < 2 * NC; ++ch) {  // dV chunks, then dK chunks
        const bool is_k = ch >= NC;
        const int cc = is_k ? ch - NC : ch;
        uint32_t rr[32];
        tmem_ld32(tmem + (is_k ? Cfg::DK_COL : Cfg::DV_COL) + cc * 32 + lane_sel, rr);
        // the multipliers of this chunk load while the TMEM read completes
        uint4 mm[4];
        if (has_m && row_ok) {
          const uint16_t* mrow = (is_k ? p.m0 : p.m1) + grow * p.ldm + c.h * D + cc * 32;
#pragma unroll
          for (int v = 0; v < 4; ++v) mm[v] = *reinterpret_cast<const uint4*>(mrow + 8 * v);
        }
        tmem_wait_ld();
        if (ch == NC - 1 || ch == 2 * NC - 1) {  // dV (then dK) may be overwritten by the next item
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(is_k ? &S.dk_free : &S.dv_free);
        }
        if (!row_ok) continue;
        // dV: Pᵀ carries no 1/n_u; dK: dS'ᵀ carries neither c nor 1/n_u
        const float sc = is_k ? p.scale * inv_n : inv_n;
        float x[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] = any ? __uint_as_float(rr[e]) * sc : 0.f;
        if (has_m) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const uint32_t w[4] = {mm[v].x, mm[v].y, mm[v].z, mm[v].w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              x[8 * v + 2 * t] *= lo16<TG>(w[t]);
              x[8 * v + 2 * t + 1] *= hi16<TG>(w[t]);
            }
          }
        }
        uint16_t* orow = (is_k ? p.g0 : p.g1) + grow * p.ldg + c.h * D + cc * 32;
#pragma unroll
        for (int v = 0; v < 4; ++v) *reinterpret_cast<uint4*>(orow + 8 * v) = pack8<TG>(x + 8 * v);
      }
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
    tmem_dealloc(tmem, 512);
  }
}

template <int D, typename TG>
cudaError_t launch_bwd_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                         BwdParams pa, BwdParams pq, int grid, cudaStream_t s) {
  cudaError_t e;
  {
    TraceScope tr("attn_bwd", s);
    const bool store = pa.ds_on != nullptr;
    auto kern = store ? attn_bwd_dkdv_kernel<D, TG, true> : attn_bwd_dkdv_kernel<D, TG, false>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, DkvCfg<D>::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<grid, dkv_threads(store), DkvCfg<D>::SMEM, s>>>(tq, tk, tv, tdo, pa);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return e;
  if (pq.ds_on != nullptr) {
    // dQ from the kept dS tiles; the recomputing kernel below then returns at once
    // (which of the two works is decided on the device, by the plan)
    TraceScope tr("attn_bwd_dq", s);
    auto kern = attn_bwd_dq_ds_kernel<D, TG>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, DqsCfg<D>::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<grid, DQS_THREADS, DqsCfg<D>::SMEM, s>>>(tk, pq);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  TraceScope tr("attn_bwd_dq", s);
  auto kern = attn_bwd_dq_kernel<D, TG>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, DqCfg<D>::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<grid, DQ_THREADS, DqCfg<D>::SMEM, s>>>(tq, tk, tv, tdo, pq);
  return cudaGetLastError();
}

}  // namespace

// q, k, v: [T, *] f16 with row stride ld; dO: [T, H*d] f16.  dq, dk, dv: f16
// (g_f16) or bf16 with row stride ldg, each multiplied elementwise by the
// multiplier block mq / mk / mv of the same type when given (row stride
// 4*H*d; the layer passes silu'(z) of its UQKV projection).  Every row of
// every segment is written.  ds_store, ds_cap: the caller's store of dS tiles
// (1024-byte aligned, ds_cap tiles; the plan was built with the same ds_cap),
// or nullptr / 0 for the dQ pass that recomputes S and dP.
cudaError_t launch_attn_bwd_f16(const __half* q, const __half* k, const __half* v, int64_t ld, const __half* dO,
                                int64_t T, int H, int d, const int32_t* plan, int32_t B, const int64_t* ts, void* dq,
                                void* dk, void* dv, int64_t ldg, const void* mq, const void* mk, const void* mv,
                                bool g_f16, int32_t* status, cudaStream_t s, uint8_t* ds_store, int64_t ds_cap) {
  if (T == 0 || B == 0) return cudaSuccess;
  const PlanLayout L = plan_layout(B, T, H);
  const int HD = H * d;
  CUtensorMap tq, tk, tv, tdo;
  if (!make_tmap_f16_2d(&tq, q, T, HD, ld, 64, BT) || !make_tmap_f16_2d(&tk, k, T, HD, ld, 64, BT) ||
      !make_tmap_f16_2d(&tv, v, T, HD, ld, 64, BT) || !make_tmap_f16_2d(&tdo, dO, T, HD, HD, 64, BT))
    return cudaErrorInvalidValue;
  BwdParams pa{};
  pa.users = reinterpret_cast<const UserInfo*>(plan + L.users);
  pa.ts = ts;
  pa.ldg = ldg;
  pa.ldm = 4 * (int64_t)HD;
  pa.H = H;
  pa.scale = 1.0f / sqrtf((float)d);
  pa.status = status;
  if (ds_store != nullptr && ds_cap > 0) {
    pa.ds_store = ds_store;
    pa.ds_base = reinterpret_cast<const int64_t*>(plan + L.ds_base);
    pa.ds_on = plan + L.counts + 3;
  }
  BwdParams pq = pa;
  pa.items = reinterpret_cast<const WorkItem*>(plan + L.bwd_items);
  pa.count = plan + L.counts + 1;
  pa.g0 = static_cast<uint16_t*>(dk);
  pa.g1 = static_cast<uint16_t*>(dv);
  pa.m0 = static_cast<const uint16_t*>(mk);
  pa.m1 = static_cast<const uint16_t*>(mv);
  pq.items = reinterpret_cast<const WorkItem*>(plan + L.dq_items);
  pq.count = plan + L.counts + 2;
  pq.g0 = static_cast<uint16_t*>(dq);
  pq.g1 = nullptr;
  pq.m0 = static_cast<const uint16_t*>(mq);
  pq.m1 = nullptr;
  const int64_t max_items = L.max_items;
  const int grid = (int)(max_items < num_sms() ? max_items : num_sms());
  if (d == 128)
    return g_f16 ? launch_bwd_d<128, __half>(tq, tk, tv, tdo, pa, pq, grid, s)
                 : launch_bwd_d<128, __nv_bfloat16>(tq, tk, tv, tdo, pa, pq, grid, s);
  if (d == 64)
    return g_f16 ? launch_bwd_d<64, __half>(tq, tk, tv, tdo, pa, pq, grid, s)
                 : launch_bwd_d<64, __nv_bfloat16>(tq, tk, tv, tdo, pa, pq, grid, s);
  return cudaErrorInvalidValue;
}

}  // namespace mtgr
