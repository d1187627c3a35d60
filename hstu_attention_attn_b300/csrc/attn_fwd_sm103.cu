// attn_fwd_sm103.cu -- jagged HSTU attention forward on the 5th-generation
// tensor cores (tcgen05 + TMEM + TMA): f16 operands (q, k, v and P), fp32
// accumulation, f16 O.
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
// Persistent kernel, one CTA per SM; a work item is one query tile of one
// (user, head).  The score tiles are double-buffered in TMEM, so the tensor
// core computes S of key tile j+1 while the epilogue turns S_j into P_j:
//   warp 0       TMA: Q per item (one buffer, released once the item's last S
//                completes), then K tiles through a 3-stage ring and V tiles
//                through a 2-stage ring
//   warp 1       S issuer (one thread) + TMEM owner
//   warp 2       PV issuer (one thread)
//   warps 3..18  epilogue: 4 lane quarters x 4 groups of 32 key columns
//                (thread = query row = TMEM lane), then the O store
// Key tiles are counted over the CTA's items (g); tile g uses score buffer
// g & 1.  The S issuer writes S(g) once PV(g - 2) has read the P that buffer
// held, so S(g + 1) is computed while the epilogue turns S(g) into P(g) and
// PV(g) runs.  Each issuer waits only on its own operands: a thread that
// issues blocks while the tensor core drains its queue, and two issuers keep
// one product queued behind the other.
// TMEM (512 columns): S/P buffers [0,128) and [128,256); two O accumulators
// of d_h columns from 256 (items alternate, so one item's O store overlaps the
// next item's products).  P overwrites S as packed f16: the 32 keys of column
// group g go to columns 32g .. 32g+15, which only that group's warps read.
#include "attn_sm103.cuh"

namespace mtgr {
namespace {
using attn::item_at;
using attn::silu_half;

constexpr int BQ = 128, BKV = 128;
constexpr int NUM_THREADS = 608;  // 19 warps
constexpr int EPI_WARPS = 16;
// shared memory: QB buffers of Q, then the K ring (KR stages) and the V ring (VR)
constexpr int QB = 1, KR = 3, VR = 2, RING = KR + VR;
constexpr int STG_BYTES = 2048;  // per-warp O staging: one [32][32] f16 box

template <int D>
struct FwdCfg {
  static constexpr int TILE = BQ * D * 2;  // one Q / K / V tile (f16)
  static constexpr int RING_OFF = QB * TILE;
  static constexpr int STG_OFF = RING_OFF + RING * TILE;  // O staging, one buffer per epilogue warp
  static constexpr int BAR_OFF = STG_OFF + EPI_WARPS * STG_BYTES;
  static constexpr int SMEM = BAR_OFF + 256 + 1024;  // + barriers + alignment slack
  __device__ static constexpr uint32_t s_col(int b) { return (uint32_t)b * 128u; }
  __device__ static constexpr uint32_t o_col(int b) { return 256u + (uint32_t)b * D; }
};

struct FwdBars {
  uint64_t q_full[QB], q_empty[QB];
  uint64_t ring_full[RING], ring_empty[RING];
  uint64_t s_full[2], p_full[2], pv_done[2], o_full[2], o_free[2];
  uint32_t tmem_base;
  int abort_flag;
};

struct FwdParams {
  const UserInfo* users;
  const WorkItem* items;  // (user, query tile, head), longest users first
  const int32_t* counts;  // item count at counts[0]
  const int64_t* ts;
  __half* O;  // [T, H*D] f16
  int64_t ldo;
  // key split (2 when the items alone would leave most SMs idle, else 1):
  // item v of the kernel is part v % split of list item v / split, taking its
  // share of the key tiles; each part then writes its O (already / n_u) in
  // fp32 to Opart + part * pstride ([T, H*D]) instead of O, and the gate adds them
  int split;
  float* Opart;
  int64_t pstride;
  int H;
  float scale;  // 1/sqrt(d_h)
  int32_t* status;
};

struct ItemCtx {
  UserInfo u;
  QTileKeys keys;
  int qt, h;
  int part, k0, n;  // key split part; its key tiles are keys.kt(k0 .. k0 + n - 1)
  __device__ __forceinline__ int kt(int j) const { return keys.kt(k0 + j, qt); }
};
__device__ __forceinline__ ItemCtx item_ctx(const FwdParams& p, int v) {
  ItemCtx c;
  const int idx = p.split == 2 ? v >> 1 : v;
  c.part = v - idx * p.split;
  const WorkItem wi = p.items[idx];
  c.h = wi.h();
  c.u = p.users[wi.b];
  c.qt = wi.t();
  c.keys = qtile_keys(c.u, c.qt);
  const int nk = c.keys.count(), h0 = p.split == 2 ? (nk + 1) >> 1 : nk;
  c.k0 = c.part ? h0 : 0;
  c.n = c.part ? nk - h0 : h0;
  return c;
}

// N scores of one query row (keys j0 .. j0+N-1 of the segment) -> N/2 packed
// f16 P values under the dynamic mixed mask.  The chunk class depends only on
// j0, so it is uniform across the warp.
template <int N>
__device__ __forceinline__ void p_chunk(const uint32_t (&r)[N], int j0, const UserInfo& u, int ri, bool row_ok,
                                        bool cand, int64_t thr, int64_t tk, float hs, uint32_t (&pk)[N / 2]) {
  if (j0 + N <= u.eS) {
    // every key is User/Seq: visible to every row
#pragma unroll
    for (int e = 0; e < N / 2; ++e)
      pk[e] = pack_f16x2(silu_half(__uint_as_float(r[2 * e]) * hs), silu_half(__uint_as_float(r[2 * e + 1]) * hs));
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
      float pv[2];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int jj = j0 + 2 * e + t;
        const bool vis = (jj < u.eS) | (attn::shfl_i64(tk, 2 * e + t) < thr) | (cand & (jj == ri));
        const float v = silu_half(__uint_as_float(r[2 * e + t]) * hs);
        pv[t] = vis ? v : 0.f;
      }
      pk[e] = pack_f16x2(pv[0], pv[1]);
    }
  }
}

template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1)  // 19 warps
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    const __grid_constant__ CUtensorMap tmP,
                    const FwdParams p) {
  using Cfg = FwdCfg<D>;
  const int total = p.counts[0] * p.split;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base;  // two Q buffers
  uint8_t* sRing = base + Cfg::RING_OFF;
  uint8_t* sStg = base + Cfg::STG_OFF;
  FwdBars& S = *reinterpret_cast<FwdBars*>(base + Cfg::BAR_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      if (i < QB) {
        mbar_init(&S.q_full[i], 1);
        mbar_init(&S.q_empty[i], 1);
      }
      mbar_init(&S.s_full[i], 1);
      mbar_init(&S.p_full[i], EPI_WARPS);
      mbar_init(&S.pv_done[i], 1);
      mbar_init(&S.o_full[i], 1);
      mbar_init(&S.o_free[i], EPI_WARPS);
    }
    for (int i = 0; i < RING; ++i) {
      mbar_init(&S.ring_full[i], 1);
      mbar_init(&S.ring_empty[i], 1);
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
    if (p.split > 1) tma_prefetch_desc(&tmP);
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
      // K tiles through a 2-stage ring (read by the S issuer), V tiles through
      // another (read by the PV issuer); order per item: Q; K_0, K_1; then
      // V_j, K_{j+2} for j = 0 .. n-1
      int st[2] = {0, 0};
      uint32_t ph[2] = {0, 0};
      auto load_kv = [&](int which, int row, int col_h) -> bool {  // which: 0 K, 1 V
        const int slot = (which ? KR : 0) + st[which];
        if (!mbar_wait(&S.ring_empty[slot], ph[which] ^ 1, abort_flag)) return false;
        uint8_t* dst = sRing + slot * Cfg::TILE;
        mbar_arrive_expect_tx(&S.ring_full[slot], Cfg::TILE);
        const CUtensorMap* m = which ? &tmV : &tmK;
#pragma unroll
        for (int cc = 0; cc < D / 64; ++cc) tma_load_2d(dst + cc * 16384, m, &S.ring_full[slot], col_h + 64 * cc, row);
        if (++st[which] == (which ? VR : KR)) { st[which] = 0; ph[which] ^= 1; }
        return true;
      };
      int it = 0;
      for (int r = 0; ok; ++r, ++it) {
        const int idx = item_at(r);
        if (idx >= total) break;
        const ItemCtx c = item_ctx(p, idx);
        const int col_h = c.h * D;
        const int qb = it % QB;
        if (!mbar_wait(&S.q_empty[qb], ((it / QB) & 1) ^ 1, abort_flag)) { ok = false; break; }
        mbar_arrive_expect_tx(&S.q_full[qb], Cfg::TILE);
#pragma unroll
        for (int cc = 0; cc < D / 64; ++cc)
          tma_load_2d(sQ + qb * Cfg::TILE + cc * 16384, &tmQ, &S.q_full[qb], col_h + 64 * cc, c.u.start + c.qt * BQ);
        const int n = c.n;
        const int row0 = c.u.start;
        for (int t = 0; t < 2 && t < n && ok; ++t) ok = load_kv(0, row0 + c.kt(t) * BKV, col_h);
        for (int j = 0; j < n && ok; ++j) {
          ok = load_kv(1, row0 + c.kt(j) * BKV, col_h);
          if (ok && j + 2 < n) ok = load_kv(0, row0 + c.kt(j + 2) * BKV, col_h);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- S issuer: S(gs) = Q · K_gsᵀ into buffer gs & 1, once
      // PV(gs - 2) has finished reading the P that buffer held ----------------
      constexpr uint32_t idesc_s = idesc_f16_f32(BQ, BKV, false, false);
      const uint32_t ring_addr = smem_u32(sRing);
      int ks = 0;
      uint32_t kph = 0;
      int g = 0, it = 0;
      for (int r = 0; ok; ++r, ++it) {
        const int idx = item_at(r);
        if (idx >= total) break;
        const ItemCtx c = item_ctx(p, idx);
        const int qb = it % QB;
        const uint32_t q_addr = smem_u32(sQ + qb * Cfg::TILE);
        if (!mbar_wait(&S.q_full[qb], (it / QB) & 1, abort_flag)) { ok = false; break; }
        const int n = c.n;
        for (int t = 0; t < n; ++t) {
          const int gs = g + t, sb = gs & 1;
          if (gs >= 2 && !mbar_wait(&S.pv_done[sb], ((gs - 2) >> 1) & 1, abort_flag)) { ok = false; break; }
          if (!mbar_wait(&S.ring_full[ks], kph, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const SmemDesc qd = attn::kmajor_base(q_addr), kd = attn::kmajor_base(ring_addr + ks * Cfg::TILE);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            tc_mma_ss_h(tmem + Cfg::s_col(sb), qd.lo + attn::kmajor_step(kk), qd.hi, kd.lo + attn::kmajor_step(kk),
                        kd.hi, idesc_s, kk > 0 ? 1u : 0u);
          tc_commit(&S.s_full[sb]);
          tc_commit(&S.ring_empty[ks]);
          if (++ks == KR) { ks = 0; kph ^= 1; }
        }
        if (!ok) break;
        tc_commit(&S.q_empty[qb]);  // once the item's products of Q complete
        g += n;
      }
    }
  } else if (warp == 2) {
    if (lane == 0) {
      // ---------------- PV issuer: O += P(j) V_j once the epilogue has written P(j) ----------------
      constexpr uint32_t idesc_o = idesc_f16_f32(BQ, D, false, true);
      const uint32_t ring_addr = smem_u32(sRing);
      int vs = 0;
      uint32_t vph = 0;
      int g = 0, it = 0;
      for (int r = 0; ok; ++r, ++it) {
        const int idx = item_at(r);
        if (idx >= total) break;
        const ItemCtx c = item_ctx(p, idx);
        const int ob = it & 1;
        const int n = c.n;
        // the accumulator still holds item it - 2 until the epilogue has read it
        // (waited also by a part without keys, which writes zeros)
        if (it >= 2 && !mbar_wait(&S.o_free[ob], ((it - 2) >> 1) & 1, abort_flag)) { ok = false; break; }
        for (int j = 0; j < n; ++j) {
          const int gj = g + j, sb = gj & 1;
          if (!mbar_wait(&S.p_full[sb], (gj >> 1) & 1, abort_flag)) { ok = false; break; }
          if (!mbar_wait(&S.ring_full[KR + vs], vph, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const SmemDesc vd = attn::mnmajor_base(ring_addr + (KR + vs) * Cfg::TILE);
#pragma unroll
          for (int kk = 0; kk < BKV / 16; ++kk)  // keys 16kk..16kk+15: column group kk/2, packed half kk&1
            tc_mma_ts_h(tmem + Cfg::o_col(ob), tmem + Cfg::s_col(sb) + 32 * (kk >> 1) + 8 * (kk & 1),
                        vd.lo + attn::mnmajor_step(kk), vd.hi, idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
          tc_commit(&S.pv_done[sb]);
          tc_commit(&S.ring_empty[KR + vs]);
          if (++vs == VR) { vs = 0; vph ^= 1; }
        }
        if (!ok) break;
        tc_commit(&S.o_full[ob]);
        g += n;
      }
    }
  } else {
    // ---------------- epilogue warps ----------------
    const int ew = warp - 3;             // 0..15
    const int grp = ew >> 2;             // group of 32 key columns of S (and of O)
    const int quarter = warp & 3;        // TMEM lane quarter this warp may access
    const uint32_t lane_sel = (uint32_t)(quarter * 32) << 16;
    const int r_in = quarter * 32 + lane;
    const float hs = 0.5f * p.scale;
    uint8_t* box_buf = sStg + ew * STG_BYTES;
    int g = 0, it = 0;
    for (int r = 0; ok; ++r, ++it) {
      const int idx = item_at(r);
      if (idx >= total) break;
      const ItemCtx c = item_ctx(p, idx);
      const UserInfo& u = c.u;
      const int ri = c.qt * BQ + r_in;  // segment-relative query row
      const bool row_ok = ri < u.n;
      const bool cand = ri >= u.eR;
      // RealTime key j is visible to this row iff ts_j < thr (User/Seq rows: never)
      int64_t thr = INT64_MIN;
      if (row_ok && ri >= u.eS) thr = p.ts[u.start + ri] + (cand ? 0 : 1);
      const int64_t* ts_u = p.ts + u.start;
      const int n = c.n;
      for (int j = 0; j < n && ok; ++j) {
        const int gj = g + j, sb = gj & 1;
        const int jg = c.kt(j) * BKV + grp * 32;  // first key of this warp's column group
        // stamps of the keys this lane broadcasts in masked chunks, loaded before the wait
        const int64_t tk0 = attn::rt_key_stamp(u, ts_u, jg, lane), tk1 = attn::rt_key_stamp(u, ts_u, jg + 16, lane);
        if (!mbar_wait(&S.s_full[sb], (gj >> 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t t_s = tmem + Cfg::s_col(sb) + grp * 32 + lane_sel;
        uint32_t rc[2][16], pk[8];
        tmem_ld16(t_s, rc[0]);
        tmem_ld16(t_s + 16, rc[1]);
        tmem_wait_ld();
        p_chunk<16>(rc[0], jg, u, ri, row_ok, cand, thr, tk0, hs, pk);
        tmem_st8(t_s, pk);
        p_chunk<16>(rc[1], jg + 16, u, ri, row_ok, cand, thr, tk1, hs, pk);
        tmem_st8(t_s + 8, pk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.p_full[sb]);
      }
      if (!ok) break;
      g += n;
      // ---------------- O = acc / n_u -> global (columns 32 grp .. of this head) ----------------
      const int ob = it & 1;
      if (!mbar_wait(&S.o_full[ob], (it >> 1) & 1, abort_flag)) { ok = false; break; }
      tc_fence_after();
      if (grp * 32 < D) {
        const float inv_n = 1.0f / (float)u.nu;
        const int row0 = c.qt * BQ + quarter * 32;  // segment-relative first row of this warp
        uint32_t rr[32];
        tmem_ld32(tmem + Cfg::o_col(ob) + grp * 32 + lane_sel, rr);
        tmem_wait_ld();
        if (p.split > 1) {
          // key-split part: fp32 partial O (zeros for a part without keys, whose
          // accumulator holds stale values: select, not scale), in two [32][16]
          // fp32 boxes through the same 64-byte-swizzled staging as the f16 box
          const bool any = c.n > 0;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            if (lane == 0) tma_store_wait_read_n<0>();
            __syncwarp();
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              float4 w;
              w.x = any ? __uint_as_float(rr[16 * hh + 4 * v + 0]) * inv_n : 0.f;
              w.y = any ? __uint_as_float(rr[16 * hh + 4 * v + 1]) * inv_n : 0.f;
              w.z = any ? __uint_as_float(rr[16 * hh + 4 * v + 2]) * inv_n : 0.f;
              w.w = any ? __uint_as_float(rr[16 * hh + 4 * v + 3]) * inv_n : 0.f;
              *reinterpret_cast<float4*>(box_buf + lane * 64 + ((v ^ ((lane >> 1) & 3)) * 16)) = w;
            }
            if (row0 + 32 <= u.n) {
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_3d(&tmP, box_buf, c.h * D + grp * 32 + 16 * hh, u.start + row0, c.part);
                tma_store_commit();
              }
            } else {
              __syncwarp();
              float* pbase = p.Opart + c.part * p.pstride + (int64_t)(u.start + row0) * p.ldo + c.h * D + grp * 32 +
                             16 * hh;
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const int rw = k * 8 + (lane >> 2), c4 = lane & 3;
                const uint4 val = *reinterpret_cast<const uint4*>(box_buf + rw * 64 + ((c4 ^ ((rw >> 1) & 3)) * 16));
                if (row0 + rw < u.n) *reinterpret_cast<uint4*>(pbase + (int64_t)rw * p.ldo + c4 * 4) = val;
              }
            }
          }
        } else {
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
        // A box of 32 rows inside the segment leaves by TMA store; the warp that
        // holds the segment's end stores its valid rows one by one (a box would
        // also write the next user's rows).
        if (row0 + 32 <= u.n) {
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmO, box_buf, c.h * D + grp * 32, u.start + row0);
            tma_store_commit();
          }
        } else {
          __syncwarp();
          __half* obase = p.O + (int64_t)(u.start + row0) * p.ldo + c.h * D + grp * 32;
          // 8 rows x 64 bytes per store instruction
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int rw = k * 8 + (lane >> 2), c4 = lane & 3;
            const uint4 val = *reinterpret_cast<const uint4*>(box_buf + rw * 64 + ((c4 ^ ((rw >> 1) & 3)) * 16));
            if (row0 + rw < u.n) *reinterpret_cast<uint4*>(obase + (int64_t)rw * p.ldo + c4 * 8) = val;
          }
        }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.o_free[ob]);
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
// opart: nullptr, or [2][T, H*d] fp32 for a key-split launch (each query tile's
// keys in two halves on two CTAs; O is then not written, the gate adds the halves).
cudaError_t launch_attn_fwd_f16(const __half* q, const __half* k, const __half* v, int64_t ld, int64_t T, int H,
                                int d, const int32_t* plan, int32_t B, const int64_t* ts, __half* O, int32_t* status,
                                cudaStream_t s, float* opart) {
  if (T == 0 || B == 0) return cudaSuccess;
  const PlanLayout L = plan_layout(B, T, H);
  const int HD = H * d;
  CUtensorMap tq, tk, tv, to, tp;
  if (!make_tmap_f16_2d(&tq, q, T, HD, ld, 64, BQ) || !make_tmap_f16_2d(&tk, k, T, HD, ld, 64, BKV) ||
      !make_tmap_f16_2d(&tv, v, T, HD, ld, 64, BKV) || !make_tmap_out(&to, OUT_F16, O, T, HD, HD, 0, 32, 32))
    return cudaErrorInvalidValue;
  // the two key halves' fp32 partial O: [2][T][H*d], [32 rows][16 fp32] boxes
  tp = to;  // unused without the split
  if (opart && !make_tmap_out(&tp, OUT_F32, opart, T, HD, HD, 2, 16, 32)) return cudaErrorInvalidValue;
  FwdParams p;
  p.users = reinterpret_cast<const UserInfo*>(plan + L.users);
  p.items = reinterpret_cast<const WorkItem*>(plan + L.dq_items);  // one item per (user, query tile, head)
  p.counts = plan + L.counts + 2;
  p.split = opart ? 2 : 1;
  p.Opart = opart;
  p.pstride = T * HD;
  p.ts = ts;
  p.O = O;
  p.ldo = HD;
  p.H = H;
  p.scale = 1.0f / sqrtf((float)d);
  p.status = status;
  // persistent: one CTA per SM (the item count lives on the device; CTAs without an item exit at once)
  const int64_t max_items = L.max_items;
  const int64_t units = max_items * p.split;
  const int grid = (int)(units < num_sms() ? units : num_sms());
  TraceScope tr("attn_fwd", s);
  if (d == 128) {
    auto kern = attn_fwd_kernel<128>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, FwdCfg<128>::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<grid, NUM_THREADS, FwdCfg<128>::SMEM, s>>>(tq, tk, tv, to, tp, p);
  } else if (d == 64) {
    auto kern = attn_fwd_kernel<64>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, FwdCfg<64>::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<grid, NUM_THREADS, FwdCfg<64>::SMEM, s>>>(tq, tk, tv, to, tp, p);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace mtgr
