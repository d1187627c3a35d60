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
// Persistent kernel, one CTA per SM.  A work item is a pair of consecutive
// query tiles (slots a and b) of one (user, head); both slots share one stream
// of K/V tiles (the union of their key lists) through a TMA ring, and the two
// slots ping-pong: while the epilogue of one slot turns S into P, the tensor
// core works on the other slot.
//   warp 0       TMA: Q_a/Q_b per item, then K_j, V_j into a 4-stage ring
//   warp 1       MMA issuer (one thread) + TMEM owner
//   warps 2..9   slot a epilogue: two warpgroups, one per half of the 128 key
//                columns (thread = query row = TMEM lane), then the O store
//   warps 10..17 slot b epilogue
// TMEM (512 columns): S_a [0,128), S_b [128,256), O_a [256, 256+d_h),
// O_b [256+d_h, 256+2 d_h).  P overwrites S as packed f16: the keys of column
// half g go to columns 64g .. 64g+31 of the slot's S region, so each
// warpgroup only ever writes the columns it has already read.
// The fp32 O rows leave through a per-warp shared-memory transpose so that the
// global stores are coalesced.
#include "attn_sm103.cuh"

namespace mtgr {
namespace {
using attn::item_at;
using attn::kmajor_desc;
using attn::mnmajor_desc;
using attn::silu_half;

constexpr int BQ = 128, BKV = 128;
constexpr int NUM_THREADS = 576;  // 18 warps
constexpr int EPI_WARPS = 8;      // per slot
constexpr int RING = 4;
constexpr int STG_FLOATS = 32 * 16;  // per-warp O staging, 2 KB: one [32][32] f16 box

template <int D>
struct FwdCfg {
  static constexpr int TILE = BQ * D * 2;  // one Q / K / V tile (f16)
  static constexpr int RING_OFF = 2 * TILE;
  static constexpr int STG_OFF = RING_OFF + RING * TILE;  // O staging, one buffer per epilogue warp
  static constexpr int BAR_OFF = STG_OFF + 2 * EPI_WARPS * STG_FLOATS * 4;
  static constexpr int SMEM = BAR_OFF + 256 + 1024;  // + barriers + alignment slack
  // TMEM columns of slot sl: S (and P) at s_col, the O accumulator at o_col
  __device__ static constexpr uint32_t s_col(int sl) { return (uint32_t)sl * 128u; }
  __device__ static constexpr uint32_t o_col(int sl) { return 256u + (uint32_t)sl * D; }
};

struct FwdBars {
  uint64_t q_full, q_empty;
  uint64_t ring_full[RING], ring_empty[RING];
  uint64_t s_full[2], p_full[2], pv_done[2], o_full[2], o_free[2];
  uint32_t tmem_base;
  int abort_flag;
};

struct FwdParams {
  const UserInfo* users;
  const WorkItem* items;  // (user, first query tile of the pair), longest first
  const int32_t* counts;
  const int64_t* ts;
  __half* O;  // [T, H*D] f16
  int64_t ldo;
  int H;
  float scale;  // 1/sqrt(d_h)
  int32_t* status;
};

struct ItemCtx {
  UserInfo u;
  PairKeys pk;
  int h;
};
__device__ __forceinline__ ItemCtx item_ctx(const FwdParams& p, int idx) {
  ItemCtx c;
  const WorkItem wi = p.items[idx];
  c.h = wi.h();
  c.u = p.users[wi.b];
  c.pk = pair_keys(c.u, wi.t() & (kSingleItem - 1), (wi.t() & kSingleItem) != 0);
  return c;
}

// N scores of one query row (keys j0 .. j0+N-1 of the segment) -> N/2 packed
// f16 P values under the dynamic mixed mask.  The chunk class depends only on
// j0, so it is uniform across the warp.  Pairs of scores go through the packed
// path (attn::silu_pair: one f16x2 tanh per pair).
template <int N>
__device__ __forceinline__ void p_chunk(const uint32_t (&r)[N], int j0, const UserInfo& u, int ri, bool row_ok,
                                        bool cand, int64_t thr, int64_t tk, float hs, uint64_t hs2,
                                        uint32_t (&pk)[N / 2]) {
  if (j0 + N <= u.eS) {
    // every key is User/Seq: visible to every row
#pragma unroll
    for (int e = 0; e < N / 2; ++e) {
      uint32_t h, t;
      pk[e] = attn::silu_pair(r[2 * e], r[2 * e + 1], hs2, h, t);
    }
  } else if (j0 >= u.eR) {
    // candidate keys (or keys past the segment): only the diagonal is visible
    const int ed = ri - j0;
    const bool diag = cand && row_ok && ed >= 0 && ed < N;
    float sd = 0.f;
#pragma unroll
    for (int e = 0; e < N; ++e) sd = (e == ed) ? __uint_as_float(r[e]) : sd;
    const float pd = diag ? silu_half(sd * hs) : 0.f;
#pragma unroll
    for (int e = 0; e < N / 2; ++e) pk[e] = pack_f16x2((2 * e == ed) ? pd : 0.f, (2 * e + 1 == ed) ? pd : 0.f);
  } else {
    // the chunk overlaps the RealTime keys: full predicate, branch-free; tk
    // holds the stamp of key j0 + (lane & 15) (attn::rt_key_stamp), broadcast
    static_assert(N == 16, "stamp broadcast covers 16 keys");
#pragma unroll
    for (int e = 0; e < N / 2; ++e) {
      bool vis[2];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int jj = j0 + 2 * e + t;
        vis[t] = (jj < u.eS) | (attn::shfl_i64(tk, 2 * e + t) < thr) | (cand & (jj == ri));
      }
      uint32_t h, t;
      pk[e] = attn::silu_pair(r[2 * e], r[2 * e + 1], hs2, h, t) & attn::keep_mask(vis[0], vis[1]);
    }
  }
}

template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1)  // 18 warps: 96 registers each (5 warps on some SMSPs)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    const FwdParams p) {
  using Cfg = FwdCfg<D>;
  const int total = p.counts[0];

  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base;  // Q_a, Q_b
  uint8_t* sRing = base + Cfg::RING_OFF;
  float* sStg = reinterpret_cast<float*>(base + Cfg::STG_OFF);
  FwdBars& S = *reinterpret_cast<FwdBars*>(base + Cfg::BAR_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&S.q_full, 1);
    mbar_init(&S.q_empty, 1);
    for (int i = 0; i < RING; ++i) {
      mbar_init(&S.ring_full[i], 1);
      mbar_init(&S.ring_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.s_full[i], 1);
      mbar_init(&S.p_full[i], EPI_WARPS);
      mbar_init(&S.pv_done[i], 1);
      mbar_init(&S.o_full[i], 1);
      mbar_init(&S.o_free[i], EPI_WARPS);
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
    tma_prefetch_desc(&tmO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  volatile int* abort_flag = &S.abort_flag;
  bool ok = true;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      int stage = 0;
      uint32_t ph = 0;
      int n_items = 0;
      for (int r = 0; ok; ++r) {
        const int idx = item_at(r);
        if (idx >= total) break;
        const ItemCtx c = item_ctx(p, idx);
        const int col_h = c.h * D;
        if (!mbar_wait(&S.q_empty, (n_items & 1) ^ 1, abort_flag)) { ok = false; break; }
        ++n_items;
        const bool two = c.pk.qb >= 0;
        mbar_arrive_expect_tx(&S.q_full, (two ? 2 : 1) * Cfg::TILE);
#pragma unroll
        for (int cc = 0; cc < D / 64; ++cc) {
          tma_load_2d(sQ + cc * 16384, &tmQ, &S.q_full, col_h + 64 * cc, c.u.start + c.pk.qa * BQ);
          if (two) tma_load_2d(sQ + Cfg::TILE + cc * 16384, &tmQ, &S.q_full, col_h + 64 * cc,
                               c.u.start + c.pk.qb * BQ);
        }
        const int nk = c.pk.count();
        for (int i = 0; i < nk && ok; ++i) {
          const int row = c.u.start + c.pk.kt(i) * BKV;
#pragma unroll
          for (int kv = 0; kv < 2; ++kv) {
            if (!mbar_wait(&S.ring_empty[stage], ph ^ 1, abort_flag)) { ok = false; break; }
            uint8_t* dst = sRing + stage * Cfg::TILE;
            mbar_arrive_expect_tx(&S.ring_full[stage], Cfg::TILE);
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc)
              tma_load_2d(dst + cc * 16384, kv == 0 ? &tmK : &tmV, &S.ring_full[stage], col_h + 64 * cc, row);
            if (++stage == RING) { stage = 0; ph ^= 1; }
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t idesc_s = idesc_f16_f32(BQ, BKV, false, false);
      constexpr uint32_t idesc_o = idesc_f16_f32(BQ, D, false, true);
      const uint32_t q_addr[2] = {smem_u32(sQ), smem_u32(sQ + Cfg::TILE)};
      const uint32_t ring_addr = smem_u32(sRing);
      int stage = 0;
      uint32_t ph = 0;
      int n_items = 0;
      bool pv_pending[2] = {false, false}, o_pending[2] = {false, false};
      uint32_t pv_waits[2] = {0, 0}, p_waits[2] = {0, 0}, o_waits[2] = {0, 0};
      for (int r = 0; ok; ++r) {
        const int idx = item_at(r);
        if (idx >= total) break;
        const ItemCtx c = item_ctx(p, idx);
        if (!mbar_wait(&S.q_full, n_items & 1, abort_flag)) { ok = false; break; }
        ++n_items;
        bool first[2] = {true, true};
        const int nk = c.pk.count();
        // Issue order per key tile i: PV_a(i), S_a(i+1), PV_b(i), S_b(i+1), so the
        // two epilogues alternate: slot a's P(i+1) is computed while the tensor
        // core runs PV_b(i) and S_b(i+1), and the other way round.  S_slot(i+1)
        // overwrites the columns P_slot(i) is read from, so it waits for PV_slot(i).
        auto issue_s = [&](int sl, uint32_t k_addr) -> bool {
          if (pv_pending[sl]) {
            if (!mbar_wait(&S.pv_done[sl], pv_waits[sl] & 1, abort_flag)) return false;
            ++pv_waits[sl];
            pv_pending[sl] = false;
            tc_fence_after();
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            tc_mma_ss(tmem + Cfg::s_col(sl), kmajor_desc(q_addr[sl], kk), kmajor_desc(k_addr, kk), idesc_s,
                      kk > 0 ? 1u : 0u);
          tc_commit(&S.s_full[sl]);
          return true;
        };
        auto issue_pv = [&](int sl, uint32_t v_addr) -> bool {
          if (!mbar_wait(&S.p_full[sl], p_waits[sl] & 1, abort_flag)) return false;
          ++p_waits[sl];
          if (first[sl] && o_pending[sl]) {  // O_slot still holds the previous item's result
            if (!mbar_wait(&S.o_free[sl], o_waits[sl] & 1, abort_flag)) return false;
            ++o_waits[sl];
            o_pending[sl] = false;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BKV / 16; ++kk)  // keys 16kk..16kk+15: column half kk/4, packed columns
            tc_mma_ts(tmem + Cfg::o_col(sl), tmem + Cfg::s_col(sl) + (kk >> 2) * 64 + (kk & 3) * 8,
                      mnmajor_desc(v_addr, kk), idesc_o, (!first[sl] || kk > 0) ? 1u : 0u);
          tc_commit(&S.pv_done[sl]);
          pv_pending[sl] = true;
          first[sl] = false;
          return true;
        };
        // prologue: S of the first key tile
        {
          const int kt = c.pk.kt(0);
          if (!mbar_wait(&S.ring_full[stage], ph, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t k_addr = ring_addr + stage * Cfg::TILE;
          if (c.pk.in_a(kt) && !issue_s(0, k_addr)) { ok = false; break; }
          if (c.pk.in_b(kt) && !issue_s(1, k_addr)) { ok = false; break; }
          tc_commit(&S.ring_empty[stage]);
          if (nk == 1) tc_commit(&S.q_empty);
          if (++stage == RING) { stage = 0; ph ^= 1; }
        }
        for (int i = 0; i < nk && ok; ++i) {
          const int kt = c.pk.kt(i);
          const bool in[2] = {c.pk.in_a(kt), c.pk.in_b(kt)};
          const bool more = i + 1 < nk;
          const int kt1 = more ? c.pk.kt(i + 1) : 0;
          const bool in1[2] = {more && c.pk.in_a(kt1), more && c.pk.in_b(kt1)};
          // V_i, then K_{i+1} (ring order)
          if (!mbar_wait(&S.ring_full[stage], ph, abort_flag)) { ok = false; break; }
          const int v_stage = stage;
          const uint32_t v_addr = ring_addr + stage * Cfg::TILE;
          if (++stage == RING) { stage = 0; ph ^= 1; }
          int k_stage = -1;
          uint32_t k_addr = 0;
          if (more) {
            if (!mbar_wait(&S.ring_full[stage], ph, abort_flag)) { ok = false; break; }
            k_stage = stage;
            k_addr = ring_addr + stage * Cfg::TILE;
            if (++stage == RING) { stage = 0; ph ^= 1; }
          }
          tc_fence_after();
#pragma unroll
          for (int sl = 0; sl < 2; ++sl) {
            if (in[sl] && !issue_pv(sl, v_addr)) { ok = false; break; }
            if (in1[sl] && !issue_s(sl, k_addr)) { ok = false; break; }
          }
          if (!ok) break;
          tc_commit(&S.ring_empty[v_stage]);
          if (more) {
            tc_commit(&S.ring_empty[k_stage]);
            if (i + 2 == nk) tc_commit(&S.q_empty);  // the item's last S has been issued
          }
        }
        if (!ok) break;
        for (int sl = 0; sl < 2; ++sl) {
          if (!first[sl]) {
            tc_commit(&S.o_full[sl]);
            o_pending[sl] = true;
          }
        }
      }
    }
  } else {
    // ---------------- epilogue warpgroups ----------------
    const int ew = warp - 2;             // 0..15
    const int sl = ew >> 3;              // slot
    const int g = (ew >> 2) & 1;         // column half of S (and of O)
    const int quarter = warp & 3;        // TMEM lane quarter this warp may access
    const uint32_t lane_sel = (uint32_t)(quarter * 32) << 16;
    const int r_in = quarter * 32 + lane;
    const float hs = 0.5f * p.scale;
    const uint64_t hs2 = attn::f32x2(__float_as_uint(hs), __float_as_uint(hs));
    float* stg = sStg + ew * STG_FLOATS;
    uint32_t s_waits = 0, o_waits = 0;
    for (int r = 0; ok; ++r) {
      const int idx = item_at(r);
      if (idx >= total) break;
      const ItemCtx c = item_ctx(p, idx);
      const int qt = sl == 0 ? c.pk.qa : c.pk.qb;
      if (qt < 0) continue;
      const UserInfo& u = c.u;
      const int ri = qt * BQ + r_in;  // segment-relative query row
      const bool row_ok = ri < u.n;
      const bool cand = ri >= u.eR;
      // RealTime key j is visible to this row iff ts_j < thr (User/Seq rows: never)
      int64_t thr = INT64_MIN;
      if (row_ok && ri >= u.eS) thr = p.ts[u.start + ri] + (cand ? 0 : 1);
      const int64_t* ts_u = p.ts + u.start;
      bool any = false;
      const int nk = c.pk.count();
      for (int i = 0; i < nk && ok; ++i) {
        const int kt = c.pk.kt(i);
        if (!(sl == 0 ? c.pk.in_a(kt) : c.pk.in_b(kt))) continue;
        any = true;
        const int jg = kt * BKV + g * 64;  // first key of this warp's column half
        // stamps of the keys this lane broadcasts in masked chunks, loaded before the wait
        int64_t tk[4];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) tk[ch] = attn::rt_key_stamp(u, ts_u, jg + 16 * ch, lane);
        if (!mbar_wait(&S.s_full[sl], s_waits & 1, abort_flag)) { ok = false; break; }
        ++s_waits;
        tc_fence_after();
        const uint32_t t_s = tmem + Cfg::s_col(sl) + g * 64 + lane_sel;
        // 4 chunks of 16 keys; the load of chunk c+1 is in flight while chunk c
        // is computed.  P of chunk c goes to columns 8c..8c+7 of this half,
        // which chunk c/2 has already read.
        uint32_t rc[2][16], pk[8];
        tmem_ld16(t_s, rc[0]);
        tmem_wait_ld();
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          if (ch < 3) tmem_ld16(t_s + 16 * (ch + 1), rc[(ch + 1) & 1]);
          p_chunk<16>(rc[ch & 1], jg + 16 * ch, u, ri, row_ok, cand, thr, tk[ch], hs, hs2, pk);
          tmem_st8(t_s + 8 * ch, pk);
          if (ch < 3) tmem_wait_ld();
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.p_full[sl]);
      }
      if (!ok || !any) {
        if (!any) continue;
        break;
      }
      // ---------------- O = acc / n_u -> global (columns g*D/2 .. of this head) ----------------
      if (!mbar_wait(&S.o_full[sl], o_waits & 1, abort_flag)) { ok = false; break; }
      ++o_waits;
      tc_fence_after();
      const float inv_n = 1.0f / (float)u.n;
      const int row0 = qt * BQ + quarter * 32;  // segment-relative first row of this warp
      __half* obase = p.O + (int64_t)(u.start + row0) * p.ldo + c.h * D + g * (D / 2);
      uint8_t* box_buf = reinterpret_cast<uint8_t*>(stg);
      // A box of 32 rows inside the segment leaves by TMA store; the warp that
      // holds the segment's end stores its valid rows one by one (a box would
      // also write the next user's rows).
      const bool box = row0 + 32 <= u.n;
#pragma unroll 1
      for (int cc = 0; cc < D / 64; ++cc) {
        uint32_t rr[32];
        tmem_ld32(tmem + Cfg::o_col(sl) + g * (D / 2) + cc * 32 + lane_sel, rr);
        tmem_wait_ld();
        // row r_in's 32 values as f16 -> box_buf[lane][64 bytes], 16-byte pieces
        // XOR-swizzled by row (the 64-byte swizzle of a [32][32] f16 TMA box);
        // the previous box store must have finished reading the buffer
        if (lane == 0) tma_store_wait_read_n<0>();
        __syncwarp();
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint4 w;
          w.x = pack_f16x2(__uint_as_float(rr[8 * v + 0]) * inv_n, __uint_as_float(rr[8 * v + 1]) * inv_n);
          w.y = pack_f16x2(__uint_as_float(rr[8 * v + 2]) * inv_n, __uint_as_float(rr[8 * v + 3]) * inv_n);
          w.z = pack_f16x2(__uint_as_float(rr[8 * v + 4]) * inv_n, __uint_as_float(rr[8 * v + 5]) * inv_n);
          w.w = pack_f16x2(__uint_as_float(rr[8 * v + 6]) * inv_n, __uint_as_float(rr[8 * v + 7]) * inv_n);
          *reinterpret_cast<uint4*>(box_buf + lane * 64 + ((v ^ ((lane >> 1) & 3)) * 16)) = w;
        }
        if (box) {
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmO, box_buf, c.h * D + g * (D / 2) + cc * 32, u.start + row0);
            tma_store_commit();
          }
          continue;
        }
        __syncwarp();
        // 8 rows x 64 bytes per store instruction
#pragma unroll
        for (int it = 0; it < 4; ++it) {
          const int rw = it * 8 + (lane >> 2), c4 = lane & 3;
          const uint4 val = *reinterpret_cast<const uint4*>(box_buf + rw * 64 + ((c4 ^ ((rw >> 1) & 3)) * 16));
          if (row0 + rw < u.n) *reinterpret_cast<uint4*>(obase + (int64_t)rw * p.ldo + cc * 32 + c4 * 8) = val;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.o_free[sl]);
    }
    if (lane == 0) tma_store_wait_all();
    __syncwarp();
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

}  // namespace

// q, k, v: [T, *] f16 with row stride ld; O: [T, H*d] f16 (scaled by 1/n_u).
cudaError_t launch_attn_fwd_f16(const __half* q, const __half* k, const __half* v, int64_t ld, int64_t T, int H,
                                int d, const int32_t* plan, int32_t B, const int64_t* ts, __half* O, int32_t* status,
                                cudaStream_t s) {
  if (T == 0 || B == 0) return cudaSuccess;
  const PlanLayout L = plan_layout(B, T, H);
  const int HD = H * d;
  CUtensorMap tq, tk, tv, to;
  if (!make_tmap_f16_2d(&tq, q, T, HD, ld, 64, BQ) || !make_tmap_f16_2d(&tk, k, T, HD, ld, 64, BKV) ||
      !make_tmap_f16_2d(&tv, v, T, HD, ld, 64, BKV) || !make_tmap_out(&to, OUT_F16, O, T, HD, HD, 0, 32, 32))
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
  // persistent: one CTA per SM (the item count lives on the device; CTAs without an item exit at once)
  const int64_t max_items = L.max_items;
  const int grid = (int)(max_items < num_sms() ? max_items : num_sms());
  TraceScope tr("attn_fwd", s);
  if (d == 128) {
    auto kern = attn_fwd_kernel<128>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, FwdCfg<128>::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<grid, NUM_THREADS, FwdCfg<128>::SMEM, s>>>(tq, tk, tv, to, p);
  } else if (d == 64) {
    auto kern = attn_fwd_kernel<64>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, FwdCfg<64>::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<grid, NUM_THREADS, FwdCfg<64>::SMEM, s>>>(tq, tk, tv, to, p);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace mtgr
