// Device side of the stream-K plan (see internal.h, struct SKPlan).
#pragma once
#include "common.cuh"
#include "internal.h"

namespace spec {

// The host guarantees T * (G + 1) < 2^32, so plan arithmetic runs in 32 bits.
SPEC_DEV long long sk_begin(const SKPlan& p, int c) { return (long long)((uint32_t)c * (uint32_t)p.T / (uint32_t)p.G); }
// CTA whose iteration range holds iteration x
SPEC_DEV int sk_cta_of(const SKPlan& p, long long x) {
  return (int)(((uint32_t)(x + 1) * (uint32_t)p.G - 1u) / (uint32_t)p.T);
}

// Tile index and row offset of stacked matrix i holding tile t.
SPEC_DEV void sk_tile_map(const SKPlan& p, int t, int& mat, int& row0) {
  int i = 0;
  while (i + 1 < p.nmat && t >= p.tbase[i + 1]) ++i;
  mat = i;
  row0 = (t - p.tbase[i]) * 128;
}

SPEC_DEV size_t sk_slot(const SKPlan& p, int c, int j) { return ((size_t)c * p.maxseg + j) * p.mpad * 128; }

// Where the partials of one tile live: CTAs c0..c1, segment j0 inside CTA c0
// (segment 0 inside every later CTA).
struct SKTileSegs {
  int c0, c1, j0;
};
SPEC_DEV SKTileSegs sk_tile_segs(const SKPlan& p, int tile) {
  const uint32_t it0 = (uint32_t)tile * (uint32_t)p.kc;
  SKTileSegs s;
  s.c0 = sk_cta_of(p, it0);
  s.c1 = sk_cta_of(p, it0 + p.kc - 1);
  s.j0 = tile - (int)((uint32_t)sk_begin(p, s.c0) / (uint32_t)p.kc);
  return s;
}
// Stacked-feature n -> (tile, lane)
SPEC_DEV void sk_feature(const SKPlan& p, int n, int& tile, int& lane) {
  int i = 0;
  while (i + 1 < p.nmat && n >= p.obase[i + 1]) ++i;
  const int local = n - p.obase[i];
  tile = p.tbase[i] + (local >> 7);
  lane = local & 127;
}
SPEC_DEV float sk_sum_segs(const float* __restrict__ part, const SKPlan& p, const SKTileSegs& s, int m, int lane) {
  float acc = part[sk_slot(p, s.c0, s.j0) + (size_t)m * 128 + lane];
  for (int c = s.c0 + 1; c <= s.c1; ++c) acc += part[sk_slot(p, c, 0) + (size_t)m * 128 + lane];
  return acc;
}

// Sum over the segments of the fp32 partials of output (row m, feature n),
// n in the stacked feature space; CTAs in ascending order (deterministic).
SPEC_DEV float sk_sum(const float* __restrict__ part, const SKPlan& p, int m, int n) {
  int tile, lane;
  sk_feature(p, n, tile, lane);
  return sk_sum_segs(part, p, sk_tile_segs(p, tile), m, lane);
}

}  // namespace spec
