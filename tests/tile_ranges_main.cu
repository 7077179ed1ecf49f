// Host driver for the tile-range bookkeeping of the CUDA path (common.cuh, fwd_tiles.cuh): reads lines
// "kind tile len_q len_k rows right window" from stdin and prints the range "first end" that
//   kind q: q_tiles_for_kv_tile -- query tiles of `rows` rows that may see the 128-key tile `tile`
//   kind k: kv_tiles_for_q_tile -- key tiles of `rows` keys that the 128-row query tile `tile` may see
//   kind f: fwd_pair_tiles -- for the pair `tile` of 128-row query tiles, "k0 n jlo0 jhi0 jlo1 jhi1":
//           the union of key tiles the forward's CTA loads and each query tile's own part of it
// The kernels visit only these tiles, so a range that misses a visible tile drops gradient terms.
#include <cstdio>
#include "common.cuh"
#include "fwd_tiles.cuh"

int main() {
  char kind;
  int tile, len_q, len_k, rows, right, window;
  while (std::scanf(" %c %d %d %d %d %d %d", &kind, &tile, &len_q, &len_k, &rows, &right, &window) == 7) {
    int a = 0, b = 0;
    if (kind == 'f') {
      int k0, n, jlo0, jhi0, jlo1, jhi1;
      gqa::fwd_pair_tiles(tile, len_q, len_k, rows, right, window, &k0, &n, &jlo0, &jhi0, &jlo1, &jhi1);
      std::printf("%d %d %d %d %d %d\n", k0, n, jlo0, jhi0, jlo1, jhi1);
      continue;
    }
    if (kind == 'q')
      gqa::q_tiles_for_kv_tile(tile, len_q, len_k, rows, right, window, &a, &b);
    else
      gqa::kv_tiles_for_q_tile(tile, len_q, len_k, rows, right, window, &a, &b);
    std::printf("%d %d\n", a, b);
  }
  return 0;
}
