// Full-vocabulary LM head with a fused top-k / log-softmax epilogue.
//
// [NEURON] "Speculative Decoding (EAGLE3) in the vLLM Neuron Framework",
// section "Eagle3 Draft Model Architecture" (LM head after the final norm) and
// "Design Choices" (greedy draft: top-1); top-k per tree node from [EAGLET]
// draft_top_k.
//
// logits = hn @ lm_head^T is never written: each CTA of the tensor-core
// kernel owns a contiguous vocabulary range (one CTA per SM) and its four
// epilogue warps fold every 128-row tile out of TMEM into running per-row
// statistics: online max / sum of exp (log-sum-exp) and the top-KT.  A tile is
// first transposed through shared memory ([m][128]), so that row m belongs to
// one warp (m = 4 j + warp) and each lane folds four consecutive vocabulary ids
// of it: the running max / sum-exp and, for k = 1, the best (value, id) are
// per lane and need no cross-lane work until the CTA's last tile.  For k > 1
// the row's sorted list lives in lanes 0..KT-1 of the owning warp (lane q holds
// entry q), every lane caches entry KT-1, and cross-lane work happens only for
// a value that beats it -- one list per row and CTA, so few values do.  At the
// end each warp writes one record per (CTA, row) it owns; a small kernel
// merges the records of all CTAs.
#include "tc_kernel.cuh"

namespace spec {
namespace tc {

constexpr int kLmMaxMpad = 64;

template <int MPAD, int KT>
struct EpiStats {
  static_assert(KT >= 1 && KT <= 32, "list spread over the lanes of one warp");
  static constexpr int R = MPAD / 4;              // rows per warp: m = 4 j + warp
  static constexpr int REC = 2 + 2 * KT;          // floats per (CTA, row) record
  // two mbarriers (tile written, tile read), then the transposed tile [MPAD][128]
  static constexpr int kScratch = 128 + MPAD * 128 * 4;
  struct Params {
    int M;
    float* out;      // [G][MPAD][REC]
  };
  const Params& P;
  int c;
  uint32_t bar_w, bar_r;
  float* S;
  volatile int* abort;
  int t = 0;                  // tiles folded so far
  float RM[R], RS[R];         // this lane's running max / sum of exp(x - max)
  float LV[R];                // k = 1: this lane's best; k > 1: list entry `lane`
  int LI[R];
  float TV[R];                // k > 1: list entry KT-1 (admission threshold)
  int TI[R];

  static SPEC_DEV void init(uint8_t* scratch) {
    mbar_init(su32(scratch), 4);
    mbar_init(su32(scratch + 8), 4);
  }
  SPEC_DEV EpiStats(const Params& pp, int cc, uint8_t* scratch, volatile int* ab) : P(pp), c(cc), abort(ab) {
    bar_w = su32(scratch);
    bar_r = su32(scratch + 8);
    S = reinterpret_cast<float*>(scratch + 128);
#pragma unroll
    for (int j = 0; j < R; ++j) {
      RM[j] = -INFINITY;
      RS[j] = 0.f;
      LV[j] = -INFINITY;
      LI[j] = 0x7fffffff;
      TV[j] = -INFINITY;
      TI[j] = 0x7fffffff;
    }
  }

  // TMEM -> shared memory, transposed; invalid vocabulary rows become -inf
  SPEC_DEV bool segment(const Seg& sg, uint32_t tb, int warp, int lane) {
    const int r = warp * 32 + lane;
    const int vid = sg.row0 + r;
    const bool valid = vid >= sg.lo && vid < sg.hi;
#pragma unroll
    for (int c16 = 0; c16 < MPAD / 16; ++c16) {
      if (c16 * 16 >= P.M) break;
      uint32_t x[16];
      tmem_ld16(tb + (uint32_t)(c16 * 16), x);
      tmem_ld_wait();
      // every warp has read the previous tile
      if (c16 == 0 && t > 0 && !mbar_wait(bar_r, (uint32_t)((t - 1) & 1), abort)) return false;
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const int m = c16 * 16 + q;
        if (m < P.M) S[m * 128 + r] = valid ? __uint_as_float(x[q]) : -INFINITY;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_w);
    return true;
  }

  SPEC_DEV float comp(const float4& x, int q) { return q == 0 ? x.x : (q == 1 ? x.y : (q == 2 ? x.z : x.w)); }

  SPEC_DEV bool after(const Seg& sg, int warp, int lane) {
    if (!mbar_wait(bar_w, (uint32_t)(t & 1), abort)) return false;
    const int id0 = sg.row0 + 4 * lane;
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const int m = 4 * j + warp;
      if (m >= P.M) break;
      const float4 x = *reinterpret_cast<const float4*>(S + m * 128 + 4 * lane);
      const float mx = fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w));
      if (mx > -INFINITY) {
        const float nm = fmaxf(RM[j], mx);
        RS[j] = RS[j] * expf(RM[j] - nm) + (expf(x.x - nm) + expf(x.y - nm)) + (expf(x.z - nm) + expf(x.w - nm));
        RM[j] = nm;
      }
      if constexpr (KT == 1) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (better(comp(x, q), id0 + q, LV[j], LI[j])) { LV[j] = comp(x, q); LI[j] = id0 + q; }
      } else {
        unsigned cm = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (comp(x, q) > -INFINITY && better(comp(x, q), id0 + q, TV[j], TI[j])) cm |= 1u << q;
        while (__any_sync(0xffffffffu, cm != 0)) {
          // this lane's best candidate, then the warp's
          float bv = -INFINITY;
          int bi = 0x7fffffff, bq = -1;
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (((cm >> q) & 1u) && better(comp(x, q), id0 + q, bv, bi)) { bv = comp(x, q); bi = id0 + q; bq = q; }
          float wv = bv;
          int wi = bi;
          warp_argmax(wv, wi);
          if (bq >= 0 && bi == wi) cm &= ~(1u << bq);
          // sorted insert into the list held by lanes 0..KT-1
          const bool ahead = lane < KT && better(LV[j], LI[j], wv, wi);
          const int pos = __popc(__ballot_sync(0xffffffffu, ahead));
          const float uv = __shfl_up_sync(0xffffffffu, LV[j], 1);
          const int ui = __shfl_up_sync(0xffffffffu, LI[j], 1);
          if (lane == pos) {
            LV[j] = wv;
            LI[j] = wi;
          } else if (lane > pos && lane < KT) {
            LV[j] = uv;
            LI[j] = ui;
          }
          TV[j] = __shfl_sync(0xffffffffu, LV[j], KT - 1);
          TI[j] = __shfl_sync(0xffffffffu, LI[j], KT - 1);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (((cm >> q) & 1u) && !better(comp(x, q), id0 + q, TV[j], TI[j])) cm &= ~(1u << q);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_r);
    ++t;
    return true;
  }

  SPEC_DEV void finish(int warp, int lane) {
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const int m = 4 * j + warp;
      if (m >= P.M) break;
      const float M_ = warp_max(RM[j]);
      const float S_ = warp_sum(RM[j] > -INFINITY ? RS[j] * expf(RM[j] - M_) : 0.f);
      float* o = P.out + ((size_t)c * MPAD + m) * REC;
      if constexpr (KT == 1) {
        float v = LV[j];
        int i = LI[j];
        warp_argmax(v, i);
        if (lane == 0) {
          o[0] = M_;
          o[1] = S_;
          o[2] = v;
          o[3] = __int_as_float(i);
        }
      } else {
        if (lane == 0) {
          o[0] = M_;
          o[1] = S_;
        }
        if (lane < KT) {
          o[2 + lane] = LV[j];
          o[2 + KT + lane] = __int_as_float(LI[j]);
        }
      }
    }
  }
};

}  // namespace tc

// Merge the per-CTA records of row m: lse (whole block) and the k best (every
// thread loads its CTA's (max, sum) head and its share of the list entries at
// once, keeps a sorted top-KT of those entries; every warp takes its k best by k
// rounds of a warp argmax over the lanes' heads, and warp 0 does the same over
// the warps' lists).  256 threads.
constexpr int kLmMaxCtas = 256;

template <int KT>
__global__ void __launch_bounds__(256) lm_merge_kernel(const float* __restrict__ part, int G, int mpad, int k,
                                                       int32_t* __restrict__ ids, int ld_ids,
                                                       float* __restrict__ lp, float* __restrict__ lse_out,
                                                       const int32_t* __restrict__ d2t) {
  SPEC_TL(spec::kTLLmMerge);
  pdl_wait();
  pdl_trigger();
  constexpr int REC = 2 + 2 * KT;
  constexpr int PER = (kLmMaxCtas * KT + 255) / 256;     // list entries a thread scans
  __shared__ float red[32];
  const int m = blockIdx.x;
  float hm = -INFINITY, hs = 0.f;
  if ((int)threadIdx.x < G) {
    const float* r = part + ((size_t)threadIdx.x * mpad + m) * REC;
    hm = r[0];
    hs = r[1];
  }
  float ev[PER];
  int ei[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int e = threadIdx.x + 256 * j;
    ev[j] = -INFINITY;
    ei[j] = 0x7fffffff;
    if (e < G * KT) {
      const float* r = part + ((size_t)(e / KT) * mpad + m) * REC;
      ev[j] = r[2 + e % KT];
      ei[j] = __float_as_int(r[2 + KT + e % KT]);
    }
  }
  const float mx = block_max(hm, red);
  const float s = block_sum(hm > -INFINITY ? hs * expf(hm - mx) : 0.f, red);
  const float lse = mx + logf(s);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // every thread: a sorted top-KT of the entries it scans; every warp: its best k
  // by k rounds of a warp argmax over the lanes' heads; warp 0: the best k of those
  __shared__ float wv[8][KT];
  __shared__ int wi[8][KT];
  float tv[KT];
  int ti[KT];
#pragma unroll
  for (int q = 0; q < KT; ++q) { tv[q] = -INFINITY; ti[q] = 0x7fffffff; }
  auto insert = [&](float v, int i) {
    if (!better(v, i, tv[KT - 1], ti[KT - 1])) return;
#pragma unroll
    for (int q = KT - 1; q >= 0; --q) {
      if (better(v, i, tv[q], ti[q])) {
        if (q > 0 && better(v, i, tv[q - 1], ti[q - 1])) {
          tv[q] = tv[q - 1];
          ti[q] = ti[q - 1];
        } else {
          tv[q] = v;
          ti[q] = i;
        }
      }
    }
  };
  auto pop_rounds = [&](float* ov, int* oi) {     // k rounds; lane 0 receives the winners
#pragma unroll
    for (int rr = 0; rr < KT; ++rr) {
      if (rr >= k) break;
      float bv = tv[0];
      int bi = ti[0];
      warp_argmax_redux(bv, bi);
      if (ti[0] == bi && bv == tv[0]) {           // the lane whose head won pops it
#pragma unroll
        for (int q = 0; q < KT - 1; ++q) { tv[q] = tv[q + 1]; ti[q] = ti[q + 1]; }
        tv[KT - 1] = -INFINITY;
        ti[KT - 1] = 0x7fffffff;
      }
      if (lane == 0) { ov[rr] = bv; oi[rr] = bi; }
    }
  };
#pragma unroll
  for (int j = 0; j < PER; ++j)
    if (threadIdx.x + 256 * j < G * KT) insert(ev[j], ei[j]);
  pop_rounds(wv[warp], wi[warp]);
  __syncthreads();
  if (warp != 0) return;
#pragma unroll
  for (int q = 0; q < KT; ++q) { tv[q] = -INFINITY; ti[q] = 0x7fffffff; }
  const int nw = blockDim.x >> 5;
  for (int e = lane; e < nw * k; e += 32) insert(wv[e / k][e % k], wi[e / k][e % k]);
  float fv[KT];
  int fi[KT];
  pop_rounds(fv, fi);
  if (lane == 0) {
#pragma unroll
    for (int rr = 0; rr < KT; ++rr) {
      if (rr >= k) break;
      ids[(size_t)m * ld_ids + rr] = d2t ? d2t[fi[rr]] : fi[rr];
      lp[(size_t)m * ld_ids + rr] = fv[rr] - lse;
    }
  }
  if (lane == 0 && lse_out) lse_out[m] = lse;
}

size_t lm_fused_ws_bytes(int /*M*/, int sms) {
  return (size_t)sms * tc::kLmMaxMpad * (2 + 2 * 8) * 4;
}

int tc_mpad(int M);

template <int MPAD, int KT>
static spec_status lm_launch(const CUtensorMap* a, const CUtensorMap& b, int V, int H, int M, float* part, int G,
                             void* ws, cudaStream_t st) {
  using namespace tc;
  RowsParams rp{V, G, (H + kBK - 1) / kBK};
  typename EpiStats<MPAD, KT>::Params ep{M, part};
  return launch_tc<MPAD, SchedRows, EpiStats<MPAD, KT>>(a, b, rp, ep, G, 0, ws, st);
}

spec_status launch_lm_head_fused(const spec_model_desc& d, const void* hn, const void* lm_head, int M, int k,
                                 int32_t* ids, int ld_ids, float* lp, float* lse, const int32_t* d2t, void* ws,
                                 size_t part_off, cudaStream_t st) {
  using namespace tc;
  const int V = d.draft_vocab > 0 ? d.draft_vocab : d.vocab, H = d.hidden;
  if (M > kLmMaxMpad) return SPEC_ERR_UNSUPPORTED;
  if (!aligned(hn, 16) || !aligned(lm_head, 16)) return SPEC_ERR_ALIGN;
  const int mpad = tc_mpad(M);
  int G = sm_count();
  if (G > (V + 127) / 128) G = (V + 127) / 128;
  if (G > kLmMaxCtas) G = kLmMaxCtas;
  float* part = reinterpret_cast<float*>(static_cast<char*>(ws) + part_off);
  CUtensorMap a[3];
  if (!make_map(&a[0], lm_head, V, H, 128)) return SPEC_ERR_CUDA;
  a[1] = a[0];
  a[2] = a[0];
  CUtensorMap b;
  if (!make_map(&b, hn, M, H, mpad)) return SPEC_ERR_CUDA;
  spec_status s;
  if (k == 1) {
    switch (mpad) {
      case 16: s = lm_launch<16, 1>(a, b, V, H, M, part, G, ws, st); break;
      case 32: s = lm_launch<32, 1>(a, b, V, H, M, part, G, ws, st); break;
      default: s = lm_launch<64, 1>(a, b, V, H, M, part, G, ws, st); break;
    }
    if (s != SPEC_OK) return s;
    launch_pdl(lm_merge_kernel<1>, dim3(M), dim3(256), 0, st, part, G, mpad, k, ids, ld_ids, lp, lse, d2t);
  } else {
    switch (mpad) {
      case 16: s = lm_launch<16, 8>(a, b, V, H, M, part, G, ws, st); break;
      case 32: s = lm_launch<32, 8>(a, b, V, H, M, part, G, ws, st); break;
      default: s = lm_launch<64, 8>(a, b, V, H, M, part, G, ws, st); break;
    }
    if (s != SPEC_OK) return s;
    launch_pdl(lm_merge_kernel<8>, dim3(M), dim3(256), 0, st, part, G, mpad, k, ids, ld_ids, lp, lse, d2t);
  }
  return last_launch();
}

}  // namespace spec

// per-unit log setter of the instrumented build (no-op otherwise)
SPEC_TL_SETTER(lmhead)
