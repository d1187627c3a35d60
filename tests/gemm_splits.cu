// Host-side dump of the split-K slice count of the tcgen05 GEMM (compiled by
// tests/test_host_logic.py; test infrastructure, not part of the library).
// Prints "K request slices" for K = 8 .. 8*kmax in steps of 8 and requests 0 .. 20.
#include <cstdio>
#include <cstdlib>

#include "gemm.cuh"

int main(int argc, char** argv) {
  const int kmax = argc > 1 ? std::atoi(argv[1]) : 512;
  for (int k8 = 1; k8 <= kmax; ++k8)
    for (int req = 0; req <= 20; ++req) std::printf("%d %d %d\n", 8 * k8, req, mtgr::gemm_splits(8 * k8, req));
  return 0;
}
