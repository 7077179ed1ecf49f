// Host driver for the main kernel's longest-first sequence order (common.cuh: sched_fill): reads lines
// "n k_0 .. k_{n-1}" (k_q = KV tiles of sequence q) from stdin and prints the order perm[0 .. n) that
// one host thread fills, on one line.
#include <cstdio>
#include <vector>
#include "common.cuh"

int main() {
  int n;
  while (std::scanf("%d", &n) == 1) {
    std::vector<int> key(n), perm(n > 0 ? n : 1, -1);
    for (int q = 0; q < n; ++q)
      if (std::scanf("%d", &key[q]) != 1) return 1;
    gqa::sched_fill(perm.data(), key.data(), n, 0, 1);
    for (int q = 0; q < n; ++q) std::printf("%d ", perm[q]);
    std::printf("\n");
  }
  return 0;
}
