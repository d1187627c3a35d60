// plan.cuh -- jagged tile schedule of the HSTU attention kernels.
//
// Every user segment [U* S* R* C*] is cut into 128-row tiles starting at the
// segment's first token.  The dynamic mixed mask (fun-rec chapter 7.3,
// §7.3.4) makes the (query tile, key tile) grid block-structured:
//   * key tiles holding User/Seq keys are visible to every query tile;
//   * key tiles that start inside RealTime are visible only to query tiles
//     holding a RealTime or candidate row;
//   * candidate keys are visible only on the diagonal, i.e. to key tile == query tile.
// So query tile qt needs the key tiles [0, hi) plus, when it holds candidate
// rows and qt >= hi, key tile qt itself; hi = ceil(eS/128) for a tile of
// User/Seq rows only and ceil(eR/128) otherwise (eS, eR: segment-relative
// index of the first RealTime / first candidate token).  The transposed rule
// gives the query tiles of a key tile for the backward pass.
#pragma once
#include <stdint.h>

namespace mtgr {

constexpr int kTile = 128;

struct UserInfo {
  int32_t start;  // first token (absolute)
  int32_t n;      // tokens in the segment
  int32_t eS;     // first RealTime token, segment-relative (== n if none after)
  int32_t eR;     // first candidate token, segment-relative
  int32_t nu;     // n_u of the 1/n_u factor: n, unless the caller gives it
  int32_t q0;     // first query row the forward computes (segment-relative; 0 unless given)
};

struct WorkItem {
  int32_t b;   // user
  int32_t th;  // tile index inside the user (low 16 bits) | head << 16
  __host__ __device__ __forceinline__ int t() const { return th & 0xFFFF; }
  __host__ __device__ __forceinline__ int h() const { return th >> 16; }
};

__host__ __device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Key tiles visited by query tile qt: the first `hi` tiles then (if extra) tile qt.
struct QTileKeys {
  int hi;
  int extra;  // 1 when the diagonal tile qt must be appended
  __host__ __device__ __forceinline__ int count() const { return hi + extra; }
  __host__ __device__ __forceinline__ int kt(int i, int qt) const { return i < hi ? i : qt; }
};

__host__ __device__ __forceinline__ QTileKeys qtile_keys(const UserInfo& u, int qt) {
  const int r1 = min((qt + 1) * kTile, u.n);
  QTileKeys k;
  k.hi = (r1 > u.eS) ? ceil_div(u.eR, kTile) : ceil_div(u.eS, kTile);
  k.extra = (r1 > u.eR && qt >= k.hi) ? 1 : 0;
  return k;
}

// Key tiles of a pair of consecutive query tiles (qa, qb = qa + 1, or qb = -1
// when qa is the user's last tile) processed together by the forward kernel:
// the union of both key lists, in increasing order, with per-tile membership.
// Rows of qa precede rows of qb, so hi_a <= hi_b and the union is [0, hi_b)
// plus the diagonal tiles that lie at or beyond it.
struct PairKeys {
  int qa, qb;
  int hi_a, ea, hi_b, eb;  // key list of each tile: [0, hi) plus the diagonal when e
  int hi;                  // max(hi_a, hi_b)
  __host__ __device__ __forceinline__ bool xa() const { return ea && qa >= hi; }
  __host__ __device__ __forceinline__ bool xb() const { return eb && qb >= hi; }
  __host__ __device__ __forceinline__ int count() const { return hi + (xa() ? 1 : 0) + (xb() ? 1 : 0); }
  __host__ __device__ __forceinline__ int kt(int i) const {
    if (i < hi) return i;
    return (i == hi && xa()) ? qa : qb;
  }
  __host__ __device__ __forceinline__ bool in_a(int k) const { return k < hi_a || (ea && k == qa); }
  __host__ __device__ __forceinline__ bool in_b(int k) const { return qb >= 0 && (k < hi_b || (eb && k == qb)); }
};

// A forward work item names qa in the low 15 bits of its tile field; bit 15
// marks an item of qa alone (used when pairs would leave SMs idle).
constexpr int kSingleItem = 0x8000;
__host__ __device__ __forceinline__ PairKeys pair_keys(const UserInfo& u, int qa, bool single = false) {
  PairKeys p;
  const int nt = ceil_div(u.n, kTile);
  p.qa = qa;
  p.qb = (!single && qa + 1 < nt) ? qa + 1 : -1;
  const QTileKeys a = qtile_keys(u, qa);
  p.hi_a = a.hi;
  p.ea = a.extra;
  if (p.qb >= 0) {
    const QTileKeys b = qtile_keys(u, p.qb);
    p.hi_b = b.hi;
    p.eb = b.extra;
  } else {
    p.hi_b = 0;
    p.eb = 0;
  }
  p.hi = p.hi_a > p.hi_b ? p.hi_a : p.hi_b;
  return p;
}

// Query tiles visiting key tile kt: tiles [lo, nq) then (if extra) tile kt.
struct KTileQueries {
  int lo, nq;
  int extra;
  __host__ __device__ __forceinline__ int count() const { return (nq - lo) + extra; }
  __host__ __device__ __forceinline__ int qt(int i, int kt) const { return i < nq - lo ? lo + i : kt; }
};

__host__ __device__ __forceinline__ KTileQueries ktile_queries(const UserInfo& u, int kt) {
  KTileQueries q;
  q.nq = ceil_div(u.n, kTile);
  const int ktA = ceil_div(u.eS, kTile), ktB = ceil_div(u.eR, kTile);
  if (kt < ktA)
    q.lo = 0;
  else if (kt < ktB)
    q.lo = (u.eS < u.n) ? (u.eS / kTile) : q.nq;
  else
    q.lo = q.nq;
  const int r1 = min((kt + 1) * kTile, u.n);
  q.extra = (r1 > u.eR && kt < q.lo) ? 1 : 0;
  return q;
}

// Workspace layout of a plan (all int32), offsets in elements.  Each list
// holds one item per (tile, head), grouped by user (users in decreasing order
// of work, a user's items for one head consecutive) so that concurrently
// running CTAs share the user's streamed operands through L2.
struct PlanLayout {
  int64_t users;      // UserInfo[B]
  int64_t counts;     // [4]: items of the fwd / bwd key-tile / bwd query-tile lists; 1 when the
                      // backward keeps its dS tiles (the batch's tiles fit the caller's store), else 0
  int64_t ds_base;    // int64[B] (8-byte aligned): first dS tile slot of each user
  int64_t fwd_items;  // WorkItem[max_items]: (user, first query tile of a pair, head)
  int64_t bwd_items;  // WorkItem[max_items]: (user, key tile, head)
  int64_t dq_items;   // WorkItem[max_items]: (user, query tile, head)
  int64_t total;      // int32 count
  int64_t max_items;
};
constexpr int kBuckets = 1024;

// The backward's stored dS tiles: one [128 key rows][128 query columns] f16
// tile, in the 128-byte-swizzled layout of two [128][64] boxes, per (user,
// head, key tile, query tile) of the user's full tile grid, at slot
//   ds_base[b] + (h * nt + kt) * nt + qt,   nt = ceil(n_b / 128),
// with ds_base[b] = H * sum over users b' < b of nt_b'^2.
constexpr int kDsTileBytes = kTile * kTile * 2;
__host__ __device__ __forceinline__ int64_t ds_slot(int64_t base, int nt, int h, int kt, int qt) {
  return base + ((int64_t)h * nt + kt) * nt + qt;
}

__host__ __device__ inline PlanLayout plan_layout(int32_t B, int64_t T, int32_t H) {
  PlanLayout L;
  L.max_items = (T / kTile + (int64_t)B + 1) * (H > 0 ? H : 1);
  int64_t o = 0;
  L.users = o;
  o += 6 * (int64_t)B;
  L.counts = o;
  o += 4;
  o = (o + 1) & ~int64_t(1);  // 8-byte alignment (the plan itself starts 256-byte aligned)
  L.ds_base = o;
  o += 2 * (int64_t)B;
  L.fwd_items = o;
  o += 2 * L.max_items;
  L.bwd_items = o;
  o += 2 * L.max_items;
  L.dq_items = o;
  o += 2 * L.max_items;
  L.total = o;
  return L;
}

}  // namespace mtgr
