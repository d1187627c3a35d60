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
  int32_t n;      // tokens in the segment (n_u)
  int32_t eS;     // first RealTime token, segment-relative (== n if none after)
  int32_t eR;     // first candidate token, segment-relative
};

struct WorkItem {
  int32_t b;  // user
  int32_t t;  // tile index inside the user (query tile fwd, key tile bwd)
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

// Workspace layout of a plan (all int32), offsets in elements.
struct PlanLayout {
  int64_t users;      // UserInfo[B]
  int64_t counts;     // [4]: fwd items, bwd items, (reserved)
  int64_t fwd_items;  // WorkItem[max_items]
  int64_t bwd_items;  // WorkItem[max_items]
  int64_t hist;       // [2][kBuckets] histograms / cursors
  int64_t total;      // int32 count
  int64_t max_items;
};
constexpr int kBuckets = 1024;

__host__ __device__ inline PlanLayout plan_layout(int32_t B, int64_t T) {
  PlanLayout L;
  L.max_items = T / kTile + (int64_t)B + 1;
  int64_t o = 0;
  L.users = o;
  o += 4 * (int64_t)B;
  L.counts = o;
  o += 4;
  L.fwd_items = o;
  o += 2 * L.max_items;
  L.bwd_items = o;
  o += 2 * L.max_items;
  L.hist = o;
  o += 4 * kBuckets;
  L.total = o;
  return L;
}

}  // namespace mtgr
