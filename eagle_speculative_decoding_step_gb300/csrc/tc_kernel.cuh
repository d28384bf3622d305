// Warp-specialised tcgen05 GEMM kernel template: schedules (which weight
// tiles and K chunks a CTA processes) and epilogues (what happens to each
// finished TMEM accumulator) are policies.
#pragma once
#include "tc_core.cuh"
#include "plan.cuh"

namespace spec {
namespace tc {

// ---------------------------------------------------------------- schedules
// A schedule hands each role of a CTA the same sequence of segments: a 128-row
// weight tile (matrix `mat`, first row `row0`) and a K-chunk range [k0, k1).
struct Seg {
  int mat, row0, k0, k1, idx;
  int lo, hi;   // weight rows [lo, hi) of the tile this segment is responsible for
  int keep;     // the next segment re-reads part of this tile: keep it in L2
};

// stream-K over tiles x chunks (see SKPlan)
struct SchedSK {
  using Params = SKPlan;
  const SKPlan& p;
  long long it, end;
  int idx;
  SPEC_DEV SchedSK(const SKPlan& pp, int c) : p(pp), it(sk_begin(pp, c)), end(sk_begin(pp, c + 1)), idx(0) {}
  SPEC_DEV bool next(Seg& s) {
    if (it >= end) return false;
    const int tile = (int)(it / p.kc);
    const long long se = min(end, (long long)(tile + 1) * p.kc);
    sk_tile_map(p, tile, s.mat, s.row0);
    s.k0 = (int)(it - (long long)tile * p.kc);
    s.k1 = s.k0 + (int)(se - it);
    s.idx = idx++;
    s.lo = s.row0;
    s.hi = s.row0 + 128;
    s.keep = 0;
    it = se;
    return true;
  }
};

// contiguous weight-row ranges, one per CTA, all K chunks per tile; the last
// tile of a range is shifted back to end at the range end (its overlap with the
// previous tile is re-read from L2 and masked)
struct RowsParams {
  int N, G, kc;
};
struct SchedRows {
  using Params = RowsParams;
  int v0, v1, t, nt, kc;
  SPEC_DEV SchedRows(const RowsParams& rp, int c) {
    v0 = (int)((long long)c * rp.N / rp.G);
    v1 = (int)((long long)(c + 1) * rp.N / rp.G);
    nt = (v1 - v0 + 127) / 128;
    t = 0;
    kc = rp.kc;
  }
  SPEC_DEV bool next(Seg& s) {
    if (t >= nt) return false;
    const int st = v0 + 128 * t;
    s.mat = 0;
    s.row0 = min(st, max(v0, v1 - 128));
    s.k0 = 0;
    s.k1 = kc;
    s.idx = t;
    s.lo = st;
    s.hi = min(st + 128, v1);
    // the last tile is shifted back to end at v1 and overlaps this one
    s.keep = (t == nt - 2) && ((v1 - v0) % 128 != 0);
    ++t;
    return true;
  }
};

// ---------------------------------------------------------------- epilogues
// fp32 partial sums of each segment into slot (CTA, segment) of a stream-K plan
template <int MPAD>
struct EpiPartial {
  struct Params {
    SKPlan p;
    int M;
    float* part;
  };
  const Params& P;
  int c;
  static constexpr int kScratch = 0;
  static SPEC_DEV void init(uint8_t*) {}
  SPEC_DEV EpiPartial(const Params& pp, int cc, uint8_t*, volatile int*) : P(pp), c(cc) {}
  SPEC_DEV bool after(const Seg&, int, int) { return true; }
  SPEC_DEV bool segment(const Seg& s, uint32_t tb, int warp, int lane) {
    float* dst = P.part + sk_slot(P.p, c, s.idx) + warp * 32 + lane;
    // the partials stay in L2 (evict-last) for the epilogue kernel that reduces them,
    // through the weights streaming past (evict-first)
    const uint64_t keep = policy_evict_last();
    // up to 64 accumulator columns in flight before one wait
    constexpr int CB = MPAD < 64 ? MPAD : 64;
#pragma unroll
    for (int cb = 0; cb < MPAD; cb += CB) {
      if (cb >= P.M) break;
      uint32_t r[CB];
#pragma unroll
      for (int c16 = 0; c16 < CB / 16; ++c16)
        if (cb + c16 * 16 < P.M) tmem_ld16(tb + (uint32_t)(cb + c16 * 16), r + 16 * c16);
      tmem_ld_wait();
#pragma unroll
      for (int q = 0; q < CB; ++q) {
        const int m = cb + q;
        if (m < P.M)
          asm volatile("st.global.L2::cache_hint.b32 [%0], %1, %2;" ::"l"(dst + (size_t)m * 128), "r"(r[q]), "l"(keep)
                       : "memory");
      }
    }
    return true;
  }
  SPEC_DEV void finish(int, int) {}
};

// fp32 outputs written straight from TMEM: out[m * ld + n] for the segment's
// rows [lo, hi) (row-range schedule: every tile is complete within one CTA)
template <int MPAD>
struct EpiStore {
  struct Params {
    int M;
    int ld;
    float* out;
  };
  const Params& P;
  static constexpr int kScratch = 0;
  static SPEC_DEV void init(uint8_t*) {}
  SPEC_DEV EpiStore(const Params& pp, int, uint8_t*, volatile int*) : P(pp) {}
  SPEC_DEV bool after(const Seg&, int, int) { return true; }
  SPEC_DEV bool segment(const Seg& s, uint32_t tb, int warp, int lane) {
    const int n = s.row0 + warp * 32 + lane;
    const bool valid = n >= s.lo && n < s.hi;
    // up to 64 accumulator columns in flight before one wait
    constexpr int CB = MPAD < 64 ? MPAD : 64;
#pragma unroll
    for (int cb = 0; cb < MPAD; cb += CB) {
      if (cb >= P.M) break;
      uint32_t r[CB];
#pragma unroll
      for (int c16 = 0; c16 < CB / 16; ++c16)
        if (cb + c16 * 16 < P.M) tmem_ld16(tb + (uint32_t)(cb + c16 * 16), r + 16 * c16);
      tmem_ld_wait();
      if (valid) {
#pragma unroll
        for (int q = 0; q < CB; ++q) {
          const int m = cb + q;
          if (m < P.M) P.out[(size_t)m * P.ld + n] = __uint_as_float(r[q]);
        }
      }
    }
    return true;
  }
  SPEC_DEV void finish(int, int) {}
};

// ---------------------------------------------------------------- kernel
template <int MPAD, class Sched, class Epi>
__global__ void __launch_bounds__(kThreads, 1)
    tc_kernel(const __grid_constant__ CUtensorMap tA0, const __grid_constant__ CUtensorMap tA1,
              const __grid_constant__ CUtensorMap tA2, const __grid_constant__ CUtensorMap tB,
              const __grid_constant__ typename Sched::Params sp, const __grid_constant__ typename Epi::Params ep,
              void* ws) {
  SPEC_TL(spec::kTLTc);
  using C = Cfg<MPAD, Epi::kScratch>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)S * C::kStage);
  // bars: full[S], empty[S], afull[2], aempty[2], drain
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t full0 = su32(bars), empty0 = su32(bars + S), afull0 = su32(bars + 2 * S),
                 aempty0 = su32(bars + 2 * S + 2), drain = su32(bars + 2 * S + 4);

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(afull0 + 8 * s, 1);
      mbar_init(aempty0 + 8 * s, 4);
    }
    mbar_init(drain, 1);
    Epi::init(smem + (size_t)S * C::kStage + 256);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    tmem_alloc(su32(&s_tmem), C::kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  volatile int* abort = &s_abort;
  const int c = blockIdx.x;

  if (warp == 4) {
    if (lane == 0) {
      // ---------------- TMA producer
      const uint64_t pw = policy_evict_first(), px = policy_evict_last();
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tA0)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tB)) : "memory");
      int stage = 0;
      uint32_t phase = 0;
      int pending[16];
      for (int s = 0; s < S; ++s) pending[s] = -1;
      Sched sch(sp, c);
      Seg sg;
      bool have = sch.next(sg);
      int kk = have ? sg.k0 : 0;
      // Weights do not depend on the previous kernel: fill the ring with weight
      // tiles before waiting for it, then add the activation tiles.
      int primed = 0;
      int pk[16];
      while (have && primed < S) {
        const CUtensorMap* ta = sg.mat == 0 ? &tA0 : (sg.mat == 1 ? &tA1 : &tA2);
        const uint32_t sa = su32(smem + (size_t)primed * C::kStage);
        const uint32_t fb = full0 + 8 * primed;
        mbar_expect_tx(fb, C::kStage);
        tma_load_2d(sa, ta, fb, kk * kBK, sg.row0, sg.keep ? px : pw);
        pending[primed] = 0;
        pk[primed] = kk;
        ++primed;
        if (++kk >= sg.k1) {
          have = sch.next(sg);
          if (have) kk = sg.k0;
        }
      }
      pdl_wait();
      pdl_trigger();
      for (int i = 0; i < primed; ++i)
#pragma unroll
        for (int j = 0; j < C::kBLoads; ++j)
          tma_load_2d(su32(smem + (size_t)i * C::kStage) + kABytes + j * C::kBBox * 128, &tB, full0 + 8 * i,
                      pk[i] * kBK, j * C::kBBox, px);
      stage = primed % S;
      phase = (primed == S) ? 1u : 0u;
      bool ok = true;
      while (ok && have) {
        const CUtensorMap* ta = sg.mat == 0 ? &tA0 : (sg.mat == 1 ? &tA1 : &tA2);
        for (; kk < sg.k1; ++kk) {
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, abort)) { ok = false; break; }
          const uint32_t sa = su32(smem + (size_t)stage * C::kStage);
          const uint32_t fb = full0 + 8 * stage;
          mbar_expect_tx(fb, C::kStage);
          tma_load_2d(sa, ta, fb, kk * kBK, sg.row0, sg.keep ? px : pw);
#pragma unroll
          for (int j = 0; j < C::kBLoads; ++j)
            tma_load_2d(sa + kABytes + j * C::kBBox * 128, &tB, fb, kk * kBK, j * C::kBBox, px);
          pending[stage] = (int)phase;
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        have = sch.next(sg);
        if (have) kk = sg.k0;
      }
      if (*abort) {
        // let copies in flight land before the CTA exits
        for (int s = 0; s < S; ++s)
          if (pending[s] >= 0) mbar_wait(full0 + 8 * s, (uint32_t)pending[s], abort, false);
      }
    } else {
      pdl_wait();
      pdl_trigger();
    }
  } else if (warp == 5) {
    pdl_wait();
    pdl_trigger();
    if (lane == 0) {
      // ---------------- MMA issuer
      constexpr uint32_t idesc0 = idesc_bf16(128, C::kN0);
      constexpr uint32_t idesc1 = idesc_bf16(128, C::kN1 > 0 ? C::kN1 : 16);
      int stage = 0;
      uint32_t phase = 0;
      int abuf = 0;
      uint32_t aphase = 0;
      Sched sch(sp, c);
      Seg sg;
      bool ok = true;
      while (ok && sch.next(sg)) {
        if (!mbar_wait(aempty0 + 8 * abuf, aphase ^ 1u, abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(abuf * MPAD);
        for (int kk = sg.k0; kk < sg.k1; ++kk) {
          if (!mbar_wait(full0 + 8 * stage, phase, abort)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = su32(smem + (size_t)stage * C::kStage);
          const uint64_t da = desc_sw128(sa), db = desc_sw128(sa + kABytes);
#pragma unroll
          for (int k16 = 0; k16 < kBK / 16; ++k16)
          {
            const uint32_t acc = (kk == sg.k0 && k16 == 0) ? 0u : 1u;
            tc_mma(d, da + (uint64_t)(2 * k16), db + (uint64_t)(2 * k16), idesc0, acc);
            if (C::kN1 > 0)   // rows 256.. of the activation tile: 256 * 128 B further, TMEM columns 256..
              tc_mma(d + 256u, da + (uint64_t)(2 * k16), db + (uint64_t)(2 * k16) + (uint64_t)((256 * 128) >> 4),
                     idesc1, acc);
          }
          tc_commit(empty0 + 8 * stage);
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit(afull0 + 8 * abuf);
        if (++abuf == C::kBufs) { abuf = 0; aphase ^= 1u; }
      }
      // all MMAs issued by this thread complete before TMEM is released
      tc_commit(drain);
      mbar_wait(drain, 0, abort, false);
    }
  } else {
    // ---------------- epilogue warps 0-3: TMEM lanes 32*warp .. 32*warp+31
    pdl_wait();
    pdl_trigger();
    Epi epi(ep, c, smem + (size_t)S * C::kStage + 256, abort);
    int abuf = 0;
    uint32_t aphase = 0;
    Sched sch(sp, c);
    Seg sg;
    bool ok = true;
    while (ok && sch.next(sg)) {
      if (!mbar_wait(afull0 + 8 * abuf, aphase, abort)) { ok = false; break; }
      tc_fence_after();
      ok = epi.segment(sg, tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(abuf * MPAD), warp, lane);
      if (!ok) break;
      // the accumulator goes back to the MMA warp before the work that no longer needs it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(aempty0 + 8 * abuf);
      if (++abuf == C::kBufs) { abuf = 0; aphase ^= 1u; }
      ok = epi.after(sg, warp, lane);
    }
    if (ok) epi.finish(warp, lane);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kCols);
  }
  if (threadIdx.x == 0 && s_abort) report(ws, SPEC_ERR_TIMEOUT, c, 0);
}

// 2-D bf16 tensor [rows, cols] row-major, box 64 (cols) x box_rows, 128-byte swizzle
bool make_map(CUtensorMap* tm, const void* ptr, int rows, int cols, int box_rows);

template <int MPAD, class Sched, class Epi>
spec_status launch_tc(const CUtensorMap* a, const CUtensorMap& b, const typename Sched::Params& sp,
                      const typename Epi::Params& ep, int G, size_t extra_static, void* ws, cudaStream_t st) {
  using C = Cfg<MPAD, Epi::kScratch>;
  static int attr_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  auto kern = tc_kernel<MPAD, Sched, Epi>;
  if (attr_dev != dev) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem) != cudaSuccess)
      return SPEC_ERR_CUDA;
    attr_dev = dev;
  }
  (void)extra_static;
  launch_pdl(kern, dim3(G), dim3(kThreads), C::kSmem, st, a[0], a[1], a[2], b, sp, ep, ws);
  return last_launch();
}

}  // namespace tc
}  // namespace spec
