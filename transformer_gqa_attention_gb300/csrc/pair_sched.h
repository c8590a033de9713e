// pair_sched.h — work schedule of the CTA-pair projection GEMM (gemm_tc_pair_kernel), shared
// by the kernel (device) and the host code that sizes its grid and tensor maps.
//
// The output is m_tiles x n_tiles tiles of 256 x 256 (n tile fastest), handed round-robin to
// n_pairs co-resident CTA pairs.  When the last round is partial, its tiles are cut along N
// into narrower pieces so that every pair gets about the same share of it.
#pragma once

#include "params.h"

namespace gqa {

// Host side: fill p.full_rounds / p.tail_w for n_pairs co-resident pairs and return the grid
// size in CTAs.  Whole tiles go round-robin; when the last round is partial, each of its m
// rows has its remaining columns cut into pieces of tail_w columns, one piece per pair,
// tail_w the smallest multiple of 32 (the epilogue's chunk width) for which the pieces of
// all those rows fit the pairs.  No such width below 256: whole tiles throughout (tail_w 0).
inline int plan_pair_grid(GemmParams& p, int n_pairs) {
  const int total = p.m_tiles * p.n_tiles;
  const int ncols = p.n_tiles * 256;
  p.full_rounds = total / n_pairs;
  p.tail_w = 0;
  const int base = p.full_rounds * n_pairs;
  if (base == total) return 2 * n_pairs;
  auto pieces = [&](int w) {
    int n = 0;
    for (int r = base / p.n_tiles, c = (base % p.n_tiles) * 256; r < p.m_tiles; ++r, c = 0)
      n += (ncols - c + w - 1) / w;
    return n;
  };
  for (int w = 32; w < 256; w += 32) {
    if (pieces(w) <= n_pairs) {
      p.tail_w = w;
      break;
    }
  }
  if (p.tail_w == 0) return 2 * (total < n_pairs ? total : n_pairs);
  return 2 * (p.full_rounds > 0 ? n_pairs : pieces(p.tail_w));
}

// Work item idx of a CTA pair: m tile mt, output columns n0 .. n0 + w - 1.  First the whole
// 256x256 tiles pair + j * n_pairs (n tile fastest), j < full_rounds; then, with tail_w > 0,
// one piece of the last, partial round: each m row of that round has its remaining columns
// cut into pieces of tail_w columns (a multiple of 32; the last piece of a row may be
// narrower), numbered row by row, piece `pair` going to this pair.  So the partial round
// costs about tail_w / 256 of a tile instead of a whole one, and no pair streams a row band
// of A twice.  Returns false past the pair's last item.
__host__ __device__ __forceinline__ bool pair_item(const GemmParams& p, int pair, int n_pairs, int idx, int& mt,
                                                   int& n0, int& w) {
  const int total = p.m_tiles * p.n_tiles;
  if (p.tail_w == 0 || idx < p.full_rounds) {
    const int u = pair + idx * n_pairs;
    mt = u / p.n_tiles;
    n0 = (u - mt * p.n_tiles) * 256;
    w = 256;
    return u < total;
  }
  if (idx > p.full_rounds) return false;
  const int ncols = p.n_tiles * 256;
  const int base = p.full_rounds * n_pairs;  // first tile of the partial round
  int r = base / p.n_tiles;
  int c = (base - r * p.n_tiles) * 256;
  int q = pair;
  for (; r < p.m_tiles; ++r, c = 0) {
    const int k = (ncols - c + p.tail_w - 1) / p.tail_w;
    if (q < k) {
      mt = r;
      n0 = c + q * p.tail_w;
      w = ncols - n0 < p.tail_w ? ncols - n0 : p.tail_w;
      return true;
    }
    q -= k;
  }
  return false;
}

}  // namespace gqa
