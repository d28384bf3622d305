// Device side of the stream-K plan (see internal.h, struct SKPlan).
#pragma once
#include "common.cuh"
#include "internal.h"

namespace spec {

SPEC_DEV long long sk_begin(const SKPlan& p, int c) { return (long long)c * p.T / p.G; }
// CTA whose iteration range holds iteration x
SPEC_DEV int sk_cta_of(const SKPlan& p, long long x) { return (int)(((x + 1) * p.G - 1) / p.T); }

// Tile index and row offset of stacked matrix i holding tile t.
SPEC_DEV void sk_tile_map(const SKPlan& p, int t, int& mat, int& row0) {
  int i = 0;
  while (i + 1 < p.nmat && t >= p.tbase[i + 1]) ++i;
  mat = i;
  row0 = (t - p.tbase[i]) * 128;
}

SPEC_DEV size_t sk_slot(const SKPlan& p, int c, int j) { return ((size_t)c * p.maxseg + j) * p.mpad * 128; }

// Sum over the segments of the fp32 partials of output (row m, feature n),
// n in the stacked feature space; CTAs in ascending order (deterministic).
SPEC_DEV float sk_sum(const float* __restrict__ part, const SKPlan& p, int m, int n) {
  int i = 0;
  while (i + 1 < p.nmat && n >= p.obase[i + 1]) ++i;
  const int local = n - p.obase[i];
  const int tile = p.tbase[i] + local / 128, lane = local % 128;
  const long long it0 = (long long)tile * p.kc;
  const int c0 = sk_cta_of(p, it0), c1 = sk_cta_of(p, it0 + p.kc - 1);
  float s = 0.f;
  for (int c = c0; c <= c1; ++c) {
    const int j = tile - (int)(sk_begin(p, c) / p.kc);
    s += part[sk_slot(p, c, j) + (size_t)m * 128 + lane];
  }
  return s;
}

}  // namespace spec
