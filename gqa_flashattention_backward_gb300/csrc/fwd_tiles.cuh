// Key-tile ranges of the forward's CTA, which owns a pair of 128-row query tiles (host and device, so
// that the host checks them against brute-force visibility).
#pragma once
#include "common.cuh"

namespace gqa {

// The forward's key tiles for the pair tp of 128-row query tiles (2 tp, and 2 tp + 1 if the sequence
// has it), `bk` keys a tile: the union [*k0, *k0 + *n) of the two tiles' own ranges, which the CTA
// loads, and each tile's own range as local indices [*jlo_w, *jhi_w) of the union (0, 0: no key
// visible to that tile, or no such tile).
__host__ __device__ __forceinline__ void fwd_pair_tiles(int tp, int len_q, int len_k, int bk, int right, int window,
                                                        int* k0, int* n, int* jlo0, int* jhi0, int* jlo1,
                                                        int* jhi1) {
  int lo0, hi0, lo1 = 0, hi1 = 0;
  kv_tiles_for_q_tile(2 * tp, len_q, len_k, bk, right, window, &lo0, &hi0);
  if (2 * tp + 1 < (len_q + 127) / 128) kv_tiles_for_q_tile(2 * tp + 1, len_q, len_k, bk, right, window, &lo1, &hi1);
  const bool e0 = hi0 > lo0, e1 = hi1 > lo1;
  const int a = e0 && e1 ? (lo0 < lo1 ? lo0 : lo1) : e0 ? lo0 : e1 ? lo1 : 0;
  const int b = e0 && e1 ? (hi0 > hi1 ? hi0 : hi1) : e0 ? hi0 : e1 ? hi1 : 0;
  *k0 = a;
  *n = b - a;
  *jlo0 = e0 ? lo0 - a : 0;
  *jhi0 = e0 ? hi0 - a : 0;
  *jlo1 = e1 ? lo1 - a : 0;
  *jhi1 = e1 ? hi1 - a : 0;
}

}  // namespace gqa
