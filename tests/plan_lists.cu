// Host-side dump of the attention kernels' tile lists (compiled by
// tests/test_plan_tiles.py; test infrastructure, not part of the library).
// Reads users as "n eS eR" lines and prints, per user, the key tiles of each
// query tile (dQ kernel), the query tiles of each key tile (dK/dV kernel), the
// dS tile slots each side uses, and the forward work items in pair and single
// mode with their membership flags.
#include <cstdio>

#include "plan.cuh"

int main() {
  int n, eS, eR;
  while (std::scanf("%d %d %d", &n, &eS, &eR) == 3) {
    const mtgr::UserInfo u{0, n, eS, eR, n, 0};
    const int nt = mtgr::ceil_div(n, mtgr::kTile);
    std::printf("U %d %d %d %d\n", n, eS, eR, nt);
    for (int qt = 0; qt < nt; ++qt) {
      const mtgr::QTileKeys k = mtgr::qtile_keys(u, qt);
      std::printf("Q %d", qt);
      for (int i = 0; i < k.count(); ++i) std::printf(" %d", k.kt(i, qt));
      std::printf("\n");
    }
    for (int kt = 0; kt < nt; ++kt) {
      const mtgr::KTileQueries q = mtgr::ktile_queries(u, kt);
      std::printf("K %d", kt);
      for (int i = 0; i < q.count(); ++i) std::printf(" %d", q.qt(i, kt));
      std::printf("\n");
    }
    // dS tile slots (user base 0, 3 heads): as the dQ pass reads them (per query
    // tile, its key tiles) and as the dK/dV pass writes them (per key tile, its query tiles)
    std::printf("SR");
    for (int h = 0; h < 3; ++h)
      for (int qt = 0; qt < nt; ++qt) {
        const mtgr::QTileKeys k = mtgr::qtile_keys(u, qt);
        for (int i = 0; i < k.count(); ++i) std::printf(" %lld", (long long)mtgr::ds_slot(0, nt, h, k.kt(i, qt), qt));
      }
    std::printf("\nSW");
    for (int h = 0; h < 3; ++h)
      for (int kt = 0; kt < nt; ++kt) {
        const mtgr::KTileQueries q = mtgr::ktile_queries(u, kt);
        for (int i = 0; i < q.count(); ++i) std::printf(" %lld", (long long)mtgr::ds_slot(0, nt, h, kt, q.qt(i, kt)));
      }
    std::printf("\n");
    for (int single = 0; single < 2; ++single) {
      for (int qa = 0; qa < nt; qa += single ? 1 : 2) {
        const mtgr::PairKeys p = mtgr::pair_keys(u, qa, single != 0);
        std::printf("P %d %d %d", single, p.qa, p.qb);
        for (int i = 0; i < p.count(); ++i) {
          const int kt = p.kt(i);
          std::printf(" %d:%d%d", kt, p.in_a(kt) ? 1 : 0, p.in_b(kt) ? 1 : 0);
        }
        std::printf("\n");
      }
    }
  }
  return 0;
}
