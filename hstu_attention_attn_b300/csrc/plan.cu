// plan.cu -- batch metadata on the device: validation, per-user group
// boundaries, integer visible-pair counts, and the work lists of the jagged
// attention kernels (see plan.cuh for the tile rule).
#include "common.cuh"
#include "plan.cuh"

namespace mtgr {

// One warp per user: clamp the segment to [0, T], find the first RealTime and
// first candidate token, and (optionally) check the metadata.
__global__ void user_info_kernel(const int32_t* __restrict__ offsets, int32_t B, const uint8_t* __restrict__ gid,
                                 int64_t T, UserInfo* __restrict__ users, int32_t* __restrict__ status,
                                 const int32_t* __restrict__ n_norm, const int32_t* __restrict__ q_begin) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= B) return;
  const int b = warp;
  int64_t s0 = offsets[b], s1 = offsets[b + 1];
  int32_t bits = 0;
  if (b == 0 && s0 != 0) bits |= DEV_ERR_OFFSETS;
  if (b == B - 1 && s1 != T) bits |= DEV_ERR_OFFSETS;
  if (s1 < s0) bits |= DEV_ERR_OFFSETS;
  s0 = s0 < 0 ? 0 : (s0 > T ? T : s0);
  s1 = s1 < s0 ? s0 : (s1 > T ? T : s1);
  const int n = (int)(s1 - s0);
  int eS = n, eR = n;
  int prev_last = 0;  // group of the last token of the previous chunk
  for (int base = 0; base < n; base += 32) {
    const int i = base + lane;
    const int g = (i < n) ? (int)gid[s0 + i] : 3;
    if (g > 3) bits |= DEV_ERR_GROUP_ID;
    const int gp = __shfl_up_sync(0xffffffffu, g, 1);
    const int prev = lane == 0 ? prev_last : gp;
    if (i < n && g < prev) bits |= DEV_ERR_GROUP_ORDER;
    const unsigned rt = __ballot_sync(0xffffffffu, i < n && g >= 2);
    const unsigned cd = __ballot_sync(0xffffffffu, i < n && g >= 3);
    if (rt && eS == n) eS = base + __ffs(rt) - 1;
    if (cd && eR == n) eR = base + __ffs(cd) - 1;
    prev_last = __shfl_sync(0xffffffffu, g, 31);
  }
  if (eR < eS) eR = eS;  // only with a bad group order; keeps eS <= eR <= n
  bits = __reduce_or_sync(0xffffffffu, bits);
  if (lane == 0) {
    const int nu = n_norm ? max(n_norm[b], 1) : n;
    const int q0 = q_begin ? min(max(q_begin[b], 0), n) : 0;
    if (users) users[b] = UserInfo{(int32_t)s0, n, eS, eR, nu, q0};
    if (status && bits) atomicOr(status, bits);
  }
}

// Users whose records (and tile costs) the plan kernel stages in shared memory
// first, so that its warps, which walk the users one after another, do not
// wait on a global load per user; larger batches read them from global memory.
constexpr int kPlanSmemUsers = 4096;
static size_t plan_smem_bytes(int32_t B) { return B <= kPlanSmemUsers ? (size_t)B * (sizeof(UserInfo) + 4) : 0; }

// One block: order users by their work (tile products), largest first, then
// write each list user by user, head by head, tile by tile.  A user's items
// for one head are consecutive, so the persistent kernels (which deal items
// out to CTAs in order) work on one user's tiles at the same time and its
// streamed operands are read from HBM about once.  One warp per user: the
// lanes sum the user's tile costs, lane 0 takes the user's place in each
// list, and the lanes write its items to consecutive addresses.
__global__ void __launch_bounds__(1024) plan_items_kernel(const UserInfo* __restrict__ users, int32_t B, int32_t H,
                                                          int32_t singles, int32_t* __restrict__ counts,
                                                          WorkItem* __restrict__ fwd_items,
                                                          WorkItem* __restrict__ bwd_items,
                                                          WorkItem* __restrict__ dq_items, int64_t max_items,
                                                          int64_t* __restrict__ ds_base, int64_t ds_cap,
                                                          int32_t* __restrict__ status) {
  __shared__ int32_t hist[3][kBuckets];  // items of each list per cost bucket, then cursors
  __shared__ int32_t tot[3];
  __shared__ long long wsum[32];
  __shared__ long long ds_run;
  extern __shared__ __align__(16) uint8_t plan_dyn[];  // plan_smem_bytes(B): user records, then tile costs
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = (int)(blockDim.x >> 5);
  const bool staged = B <= kPlanSmemUsers;
  UserInfo* s_users = reinterpret_cast<UserInfo*>(plan_dyn);
  int32_t* s_cost = reinterpret_cast<int32_t*>(plan_dyn + (size_t)(staged ? B : 0) * sizeof(UserInfo));
  if (staged)
    for (int i = tid; i < B; i += blockDim.x) s_users[i] = users[i];
  for (int i = tid; i < 3 * kBuckets; i += blockDim.x) (&hist[0][0])[i] = 0;
  __syncthreads();
  auto user_at = [&](int b) { return staged ? s_users[b] : users[b]; };
  auto user_cost = [&](const UserInfo& u) {  // whole warp; the same value on every lane
    const int nt = ceil_div(u.n, kTile);
    int c = 0;
    for (int t = lane; t < nt; t += 32) c += qtile_keys(u, t).count();
    c = __reduce_add_sync(0xffffffffu, c);
    return min(c, kBuckets - 1);
  };
  for (int b = warp; b < B; b += nw) {
    const UserInfo u = user_at(b);
    const int nt = ceil_div(u.n, kTile);
    const int c = user_cost(u);
    if (lane == 0) {
      if (staged) s_cost[b] = c;
      atomicAdd(&hist[0][c], (singles ? nt : (nt + 1) / 2) * H);
      atomicAdd(&hist[1][c], nt * H);
      atomicAdd(&hist[2][c], (nt - u.q0 / kTile) * H);
    }
  }
  __syncthreads();
  // exclusive scan from the most expensive bucket down (one warp per list)
  if (tid < 96) {
    const int list = tid >> 5;
    int running = 0;
    for (int base = kBuckets - 1; base >= 0; base -= 32) {
      const int c = base - lane;
      const int v = c >= 0 ? hist[list][c] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (c >= 0) hist[list][c] = running + incl - v;
      running += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) tot[list] = running;
  }
  __syncthreads();
  for (int b = warp; b < B; b += nw) {
    const UserInfo u = user_at(b);
    const int nt = ceil_div(u.n, kTile);
    const int np = singles ? nt : (nt + 1) / 2;  // forward items per head
    const int c = staged ? s_cost[b] : user_cost(u);
    int pf = 0, pb = 0, pq = 0;
    const int t0 = u.q0 / kTile, nq = nt - t0;  // query tiles of the per-tile list
    if (lane == 0) {
      pf = atomicAdd(&hist[0][c], np * H);
      pb = atomicAdd(&hist[1][c], nt * H);
      pq = atomicAdd(&hist[2][c], nq * H);
    }
    pf = __shfl_sync(0xffffffffu, pf, 0);
    pb = __shfl_sync(0xffffffffu, pb, 0);
    pq = __shfl_sync(0xffffffffu, pq, 0);
    for (int e = lane; e < np * H; e += 32) {  // head e / np, pair e % np
      const int h = e / np, i = e - h * np;
      const int64_t o = (int64_t)pf + e;
      if (o < max_items) fwd_items[o] = WorkItem{b, (singles ? (i | kSingleItem) : 2 * i) | (h << 16)};
    }
    for (int e = lane; e < nt * H; e += 32) {  // head e / nt, tile e % nt
      const int h = e / nt, t = e - h * nt;
      const int64_t ob = (int64_t)pb + e;
      if (ob < max_items) bwd_items[ob] = WorkItem{b, t | (h << 16)};
    }
    for (int e = lane; e < nq * H; e += 32) {  // head e / nq, tile t0 + e % nq
      const int h = e / nq, t = t0 + (e - h * nq);
      const int64_t oq = (int64_t)pq + e;
      if (oq < max_items) dq_items[oq] = WorkItem{b, t | (h << 16)};
    }
  }
  // dS tile slots (plan.cuh): exclusive prefix over the users, in user order,
  // of H * nt^2; the backward keeps its dS tiles only when all of them fit
  if (tid == 0) ds_run = 0;
  __syncthreads();
  if (ds_base != nullptr) {
    for (int c0 = 0; c0 < B; c0 += (int)blockDim.x) {
      const int b = c0 + tid;
      long long v = 0;
      if (b < B) {
        const long long nt = ceil_div(user_at(b).n, kTile);
        v = (long long)H * nt * nt;
      }
      long long x = v;  // inclusive scan in the warp
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (lane == 31) wsum[warp] = x;
      __syncthreads();
      if (warp == 0) {  // inclusive scan of the warp sums
        long long w = lane < nw ? wsum[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const long long y = __shfl_up_sync(0xffffffffu, w, o);
          if (lane >= o) w += y;
        }
        wsum[lane] = w;
      }
      __syncthreads();
      if (b < B) ds_base[b] = ds_run + (warp > 0 ? wsum[warp - 1] : 0) + x - v;
      __syncthreads();
      if (tid == 0) ds_run += wsum[31];
      __syncthreads();
    }
  }
  if (tid == 0) {
    counts[0] = tot[0];
    counts[1] = tot[1];
    counts[2] = tot[2];
    counts[3] = (ds_base != nullptr && ds_cap > 0 && ds_run <= ds_cap) ? 1 : 0;
    if ((tot[0] > max_items || tot[1] > max_items || tot[2] > max_items) && status) atomicOr(status, DEV_ERR_PLAN);
  }
}

// Visible keys per row: User/Seq keys (eS of them) for everyone, plus the
// RealTime keys allowed by the timestamp rule, plus itself for a candidate.
// One block per user; the block finds its own group boundaries.
__global__ void visible_counts_kernel(const int32_t* __restrict__ offsets, const uint8_t* __restrict__ gid,
                                      const int64_t* __restrict__ ts, int64_t T, int32_t* __restrict__ cnt,
                                      unsigned long long* __restrict__ total) {
  __shared__ int eS_s, eR_s;
  __shared__ unsigned long long part[32];
  int64_t s0 = offsets[blockIdx.x], s1 = offsets[blockIdx.x + 1];
  s0 = s0 < 0 ? 0 : (s0 > T ? T : s0);
  s1 = s1 < s0 ? s0 : (s1 > T ? T : s1);
  const int n = (int)(s1 - s0);
  if (threadIdx.x == 0) {
    eS_s = n;
    eR_s = n;
  }
  __syncthreads();
  for (int r = threadIdx.x; r < n; r += blockDim.x) {
    const int g = gid[s0 + r];
    if (g >= 2) atomicMin(&eS_s, r);
    if (g >= 3) atomicMin(&eR_s, r);
  }
  __syncthreads();
  const int eS = eS_s, eR = max(eR_s, eS_s);
  unsigned long long local = 0;
  for (int r = threadIdx.x; r < n; r += blockDim.x) {
    int c;
    if (r < eS) {
      c = eS;
    } else {
      const int64_t ti = ts[s0 + r];
      const bool cand = r >= eR;
      c = eS + (cand ? 1 : 0);
      for (int j = eS; j < eR; ++j) {
        const int64_t tj = ts[s0 + j];
        c += cand ? (tj < ti) : (tj <= ti);
      }
    }
    cnt[s0 + r] = c;
    local += (unsigned long long)c;
  }
  for (int o = 16; o > 0; o >>= 1) local += __shfl_xor_sync(0xffffffffu, local, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = local;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long sum = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) sum += part[w];
    atomicAdd(total, sum);
  }
}

// ---------------------------------------------------------------------------
// Host wrappers (internal)
// ---------------------------------------------------------------------------
cudaError_t launch_user_info(const int32_t* offsets, int32_t B, const uint8_t* gid, int64_t T, UserInfo* users,
                             int32_t* status, cudaStream_t s, const int32_t* n_norm, const int32_t* q_begin) {
  if (B <= 0) return cudaSuccess;
  const int threads = 256;
  const int blocks = (int)(((int64_t)B * 32 + threads - 1) / threads);
  TraceScope tr("plan_users", s);
  user_info_kernel<<<blocks, threads, 0, s>>>(offsets, B, gid, T, users, status, n_norm, q_begin);
  return cudaGetLastError();
}

// ds_cap: dS tile slots the caller's store holds (0: the backward recomputes S
// and dP for dQ; the plan then skips the slot prefix)
cudaError_t launch_plan(const int32_t* offsets, int32_t B, const uint8_t* gid, int64_t T, int32_t H, int32_t* ws,
                        int32_t* status, cudaStream_t s, const int32_t* n_norm, const int32_t* q_begin,
                        int64_t ds_cap) {
  const PlanLayout L = plan_layout(B, T, H);
  UserInfo* users = reinterpret_cast<UserInfo*>(ws + L.users);
  cudaError_t e = launch_user_info(offsets, B, gid, T, users, status, s, n_norm, q_begin);
  if (e != cudaSuccess) return e;
  // single query tiles per forward item when even (T/128 + B) / 2 pairs per
  // head would not fill the SMs twice (short requests): twice the items
  const int singles = (T / kTile + B) * (int64_t)H <= 4 * (int64_t)num_sms() ? 1 : 0;
  TraceScope tr("plan_items", s);
  const size_t dyn = plan_smem_bytes(B);
  if (dyn > 48 * 1024) {
    cudaError_t e2 = cudaFuncSetAttribute(plan_items_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
    if (e2 != cudaSuccess) return e2;
  }
  plan_items_kernel<<<1, 1024, dyn, s>>>(users, B, H, singles, ws + L.counts, reinterpret_cast<WorkItem*>(ws + L.fwd_items),
                                       reinterpret_cast<WorkItem*>(ws + L.bwd_items),
                                       reinterpret_cast<WorkItem*>(ws + L.dq_items), L.max_items,
                                       ds_cap > 0 ? reinterpret_cast<int64_t*>(ws + L.ds_base) : nullptr, ds_cap,
                                       status);
  return cudaGetLastError();
}

cudaError_t launch_visible_counts(const int32_t* offsets, int32_t B, const uint8_t* gid, const int64_t* ts,
                                  int64_t T, int32_t* cnt, int64_t* total, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(total, 0, sizeof(int64_t), s);
  if (e != cudaSuccess) return e;
  if (B <= 0) return cudaSuccess;
  TraceScope tr("visible_counts", s);
  visible_counts_kernel<<<B, 256, 0, s>>>(offsets, gid, ts, T, cnt, reinterpret_cast<unsigned long long*>(total));
  return cudaGetLastError();
}

}  // namespace mtgr
