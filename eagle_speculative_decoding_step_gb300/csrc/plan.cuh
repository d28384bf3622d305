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
// (constant indices only: the plan stays in parameter space)
SPEC_DEV void sk_feature(const SKPlan& p, int n, int& tile, int& lane) {
  int ob = p.obase[0], tb = p.tbase[0];
#pragma unroll
  for (int k = 1; k < 4; ++k)
    if (k < p.nmat && n >= p.obase[k]) {
      ob = p.obase[k];
      tb = p.tbase[k];
    }
  const int local = n - ob;
  tile = tb + (local >> 7);
  lane = local & 127;
}
// Sum over the segments of the fp32 partials of outputs (row m, features n[f]),
// n in the stacked feature space; CTAs in ascending order (deterministic).  The
// loads of up to 1 + SB segments of every feature are issued before the
// first add, so a feature costs one round trip to L2 rather than one per
// segment; a tile spread over more CTAs takes the rest one by one.  Features
// with on[f] false read nothing and give 0.
constexpr int kSegBatch = 8;
template <int NF, int SB = kSegBatch>
struct SKGather {
  SKTileSegs s[NF];
  const float* q[NF];
  float first[NF], v[NF][SB];
  bool on[NF];
};
// Issue the loads (sk_gather), do other work, then add them up (sk_reduce).
// sk_gather_segs takes each feature's tile segments and lane from the caller
// (e.g. a block-wide table in shared memory), sk_gather works them out.
template <int NF, int SB>
SPEC_DEV void sk_gather_segs(const float* __restrict__ part, const SKPlan& p, int m, const SKTileSegs (&seg)[NF],
                             const int (&lane)[NF], const bool (&on)[NF], SKGather<NF, SB>& g) {
#pragma unroll
  for (int f = 0; f < NF; ++f) {
    g.s[f] = seg[f];
    g.q[f] = part + (size_t)m * 128 + lane[f];
    g.on[f] = on[f];
  }
#pragma unroll
  for (int f = 0; f < NF; ++f) {
    g.first[f] = on[f] ? g.q[f][sk_slot(p, g.s[f].c0, g.s[f].j0)] : 0.f;
#pragma unroll
    for (int k = 0; k < SB; ++k)
      g.v[f][k] = on[f] && g.s[f].c0 + 1 + k <= g.s[f].c1 ? g.q[f][sk_slot(p, g.s[f].c0 + 1 + k, 0)] : 0.f;
  }
}
template <int NF, int SB>
SPEC_DEV void sk_gather(const float* __restrict__ part, const SKPlan& p, int m, const int (&n)[NF],
                        const bool (&on)[NF], SKGather<NF, SB>& g) {
  SKTileSegs seg[NF];
  int lane[NF];
#pragma unroll
  for (int f = 0; f < NF; ++f) {
    int tile;
    sk_feature(p, n[f], tile, lane[f]);
    seg[f] = sk_tile_segs(p, tile);
  }
  sk_gather_segs<NF, SB>(part, p, m, seg, lane, on, g);
}
template <int NF, int SB>
SPEC_DEV void sk_reduce(const SKPlan& p, const SKGather<NF, SB>& g, float (&out)[NF]) {
#pragma unroll
  for (int f = 0; f < NF; ++f) {
    float acc = g.first[f];
#pragma unroll
    for (int k = 0; k < SB; ++k)
      if (g.s[f].c0 + 1 + k <= g.s[f].c1) acc += g.v[f][k];
    if (g.on[f])
      for (int c = g.s[f].c0 + 1 + SB; c <= g.s[f].c1; ++c) acc += g.q[f][sk_slot(p, c, 0)];
    out[f] = g.on[f] ? acc : 0.f;
  }
}
template <int NF, int SB = kSegBatch>
SPEC_DEV void sk_sum_n(const float* __restrict__ part, const SKPlan& p, int m, const int (&n)[NF],
                       const bool (&on)[NF], float (&out)[NF]) {
  SKGather<NF, SB> g;
  sk_gather<NF, SB>(part, p, m, n, on, g);
  sk_reduce<NF, SB>(p, g, out);
}

SPEC_DEV float sk_sum(const float* __restrict__ part, const SKPlan& p, int m, int n) {
  const int nn[1] = {n};
  const bool on[1] = {true};
  float out[1];
  sk_sum_n<1>(part, p, m, nn, on, out);
  return out[0];
}

}  // namespace spec
