// batching.cpp -- host-side construction of training batches: stochastic-length
// selection of long behaviour histories, and token-balanced per-GPU batches.
// Plain C++ on host arrays (no CUDA); the caller gathers the kept rows and
// copies each rank's batch to its device.
#include <stdint.h>

#include "mtgr.h"

namespace mtgr {
void set_error(const char* fmt, ...);
}
using mtgr::set_error;

// Stochastic length (paper-daily "MTGR：美团外卖生成式推荐Scaling Law落地实践",
// "计算量涨了 65 倍…": training shortens long user sequences by sampling a
// piece of them; scoring keeps the whole sequence).  Per user: the User
// tokens, RealTime tokens and candidates are kept; a Seq run longer than
// max_seq is cut to the window of max_seq consecutive Seq tokens starting at
// draws[u] mod (n_S - max_seq + 1).
extern "C" MTGR_API mtgr_status mtgr_stochastic_length(const int32_t* offsets, int32_t B, const uint8_t* gid,
                                                       int64_t T, int32_t max_seq, const uint64_t* draws,
                                                       int32_t* keep, int32_t* new_offsets, int64_t* new_T) {
  if (B < 0 || T < 0 || max_seq < 0 || !offsets || !new_offsets || !new_T || (T > 0 && (!gid || !keep)) ||
      (B > 0 && !draws)) {
    set_error("mtgr_stochastic_length: bad argument (B=%d, T=%lld, max_seq=%d, or a NULL pointer)", (int)B,
              (long long)T, (int)max_seq);
    return MTGR_ERR_INVALID_ARG;
  }
  if (offsets[0] != 0 || offsets[B] != T) {
    set_error("mtgr_stochastic_length: offsets must start at 0 and end at T");
    return MTGR_ERR_BAD_OFFSETS;
  }
  for (int32_t u = 0; u < B; ++u)
    if (offsets[u + 1] < offsets[u]) {
      set_error("mtgr_stochastic_length: offsets decrease at user %d", (int)u);
      return MTGR_ERR_BAD_OFFSETS;
    }
  for (int32_t u = 0; u < B; ++u) {
    const int64_t s0 = offsets[u], s1 = offsets[u + 1];
    for (int64_t i = s0; i < s1; ++i)
      if (gid[i] > 3 || (i > s0 && gid[i] < gid[i - 1])) {
        set_error("mtgr_stochastic_length: user %d: group ids must be 0..3 in the order User, Seq, RealTime, "
                  "candidate (token %lld)", (int)u, (long long)i);
        return MTGR_ERR_BAD_GROUP_ORDER;
      }
  }
  int64_t w = 0;
  new_offsets[0] = 0;
  for (int32_t u = 0; u < B; ++u) {
    const int64_t s0 = offsets[u], s1 = offsets[u + 1];
    int64_t sS = s0;
    while (sS < s1 && gid[sS] == 0) ++sS;  // first Seq token
    int64_t eS = sS;
    while (eS < s1 && gid[eS] == 1) ++eS;  // one past the last Seq token
    int64_t k0 = sS, k1 = eS;              // kept Seq tokens
    const int64_t nS = eS - sS;
    if (nS > max_seq) {
      k0 = sS + (int64_t)(draws[u] % (uint64_t)(nS - max_seq + 1));
      k1 = k0 + max_seq;
    }
    for (int64_t i = s0; i < sS; ++i) keep[w++] = (int32_t)i;
    for (int64_t i = k0; i < k1; ++i) keep[w++] = (int32_t)i;
    for (int64_t i = eS; i < s1; ++i) keep[w++] = (int32_t)i;
    new_offsets[u + 1] = (int32_t)w;
  }
  *new_T = w;
  return MTGR_OK;
}

// Token-balanced batches (zzxanthony.github.io "MTGR：工业级生成式推荐框架",
// §11.3 "Dynamic batch size 做负载均衡"; paper-daily "计算量涨了 65 倍…"):
// users, in arrival order, are cut into n_ranks contiguous groups whose
// largest token count is as small as possible; the gradient of rank r is
// weighted by its share of the users.
extern "C" MTGR_API mtgr_status mtgr_token_balanced_split(const int64_t* tokens, int32_t B, int32_t n_ranks,
                                                          int32_t* rank_first, int64_t* rank_tokens,
                                                          double* grad_weight) {
  if (B < 0 || n_ranks < 1 || (B > 0 && !tokens) || !rank_first || !rank_tokens || !grad_weight) {
    set_error("mtgr_token_balanced_split: bad argument (B=%d, n_ranks=%d, or a NULL pointer)", (int)B,
              (int)n_ranks);
    return MTGR_ERR_INVALID_ARG;
  }
  int64_t lo = 0, hi = 0;
  for (int32_t i = 0; i < B; ++i) {
    if (tokens[i] < 0) {
      set_error("mtgr_token_balanced_split: tokens[%d] is negative", (int)i);
      return MTGR_ERR_INVALID_ARG;
    }
    lo = tokens[i] > lo ? tokens[i] : lo;
    hi += tokens[i];
  }
  // groups a left-to-right cut needs when no group may exceed M (M >= every user's tokens)
  auto groups_needed = [&](int64_t M) {
    int32_t g = 1;
    int64_t s = 0;
    for (int32_t i = 0; i < B; ++i) {
      if (s + tokens[i] > M) {
        ++g;
        s = tokens[i];
      } else {
        s += tokens[i];
      }
    }
    return g;
  };
  while (lo < hi) {  // smallest feasible maximum
    const int64_t mid = lo + (hi - lo) / 2;
    if (groups_needed(mid) <= n_ranks)
      hi = mid;
    else
      lo = mid + 1;
  }
  const int64_t M = lo;
  // cut: each rank takes users while it stays within M, leaving at least one
  // user for every later rank when there are users enough
  int32_t i = 0;
  for (int32_t r = 0; r < n_ranks; ++r) {
    rank_first[r] = i;
    const int32_t later = n_ranks - 1 - r;
    const int32_t reserve = B >= n_ranks ? later : 0;
    int64_t s = 0;
    while (i < B && s + tokens[i] <= M && B - (i + 1) >= reserve) s += tokens[i++];
    rank_tokens[r] = s;
    grad_weight[r] = B > 0 ? (double)(i - rank_first[r]) / (double)B : 0.0;
  }
  rank_first[n_ranks] = i;
  if (i != B) {  // cannot happen for M from the search above
    set_error("mtgr_token_balanced_split: internal error, %d of %d users placed", (int)i, (int)B);
    return MTGR_ERR_INVALID_ARG;
  }
  return MTGR_OK;
}
