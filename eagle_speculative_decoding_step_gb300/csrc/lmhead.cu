// Full-vocabulary LM head with a fused top-k / log-softmax epilogue.
//
// [NEURON] "Speculative Decoding (EAGLE3) in the vLLM Neuron Framework",
// section "Eagle3 Draft Model Architecture" (LM head after the final norm) and
// "Design Choices" (greedy draft: top-1); top-k per tree node from [EAGLET]
// draft_top_k.
//
// logits = hn @ lm_head^T is never written: each CTA of the tensor-core
// kernel owns a contiguous vocabulary range (one CTA per SM), and its epilogue
// warps fold every 128-row tile straight out of TMEM into per-row running
// statistics -- online max / sum of exp (log-sum-exp) and a sorted top-KT list
// -- held in registers by the lane that owns the row (row m -> lane m % 32).
// A candidate only enters a list if it beats the list's current last entry, so
// after the first tiles a tile costs two warp reductions per row.  At the end
// the four epilogue warps merge through shared memory and write one partial
// per (CTA, row); a small kernel merges the partials of all CTAs.
#include "tc_kernel.cuh"

namespace spec {
namespace tc {

constexpr int kLmMaxMpad = 64;

template <int MPAD, int KT>
struct EpiStats {
  static constexpr int NS = (MPAD + 31) / 32;     // rows owned per lane
  static constexpr int REC = 2 + 2 * KT;          // floats per (CTA, row) record
  struct Params {
    int M;
    float* out;      // [G][MPAD][REC]
  };
  const Params& P;
  int c;
  float RM[NS], RS[NS], TV[NS][KT];
  int TI[NS][KT];

  SPEC_DEV EpiStats(const Params& pp, int cc) : P(pp), c(cc) {
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      RM[s] = -INFINITY;
      RS[s] = 0.f;
#pragma unroll
      for (int q = 0; q < KT; ++q) { TV[s][q] = -INFINITY; TI[s][q] = 0x7fffffff; }
    }
  }

  // sorted insert (descending value, ascending id) into list s of this lane
  template <int s> SPEC_DEV void insert(float v, int i) {
#pragma unroll
    for (int q = KT - 1; q >= 0; --q) {
      if (better(v, i, TV[s][q], TI[s][q])) {
        if (q > 0 && better(v, i, TV[s][q - 1], TI[s][q - 1])) {
          TV[s][q] = TV[s][q - 1];
          TI[s][q] = TI[s][q - 1];
        } else {
          TV[s][q] = v;
          TI[s][q] = i;
        }
      }
    }
  }

  template <int m> SPEC_DEV void column(float x, bool valid, int vid, int lane) {
    constexpr int s = m >> 5;
    constexpr int owner = m & 31;
    const float xv = valid ? x : -INFINITY;
    const float wm = warp_max(xv);
    if (wm > -INFINITY) {
      const float e = valid ? expf(xv - wm) : 0.f;
      const float se = warp_sum(e);
      if (lane == owner) {
        const float nm = fmaxf(RM[s], wm);
        RS[s] = RS[s] * expf(RM[s] - nm) + se * expf(wm - nm);
        RM[s] = nm;
      }
    }
    float thr = __shfl_sync(0xffffffffu, TV[s][KT - 1], owner);
    int thri = __shfl_sync(0xffffffffu, TI[s][KT - 1], owner);
    bool cand = valid && better(xv, vid, thr, thri);
    while (__any_sync(0xffffffffu, cand)) {
      float bv = cand ? xv : -INFINITY;
      int bi = cand ? vid : 0x7fffffff;
      warp_argmax(bv, bi);
      if (lane == owner) insert<s>(bv, bi);
      if (vid == bi) cand = false;
      thr = __shfl_sync(0xffffffffu, TV[s][KT - 1], owner);
      thri = __shfl_sync(0xffffffffu, TI[s][KT - 1], owner);
      cand = cand && better(xv, vid, thr, thri);
    }
  }

  template <int c16> SPEC_DEV void chunk(uint32_t tb, bool valid, int vid, int lane) {
    if (c16 * 16 >= P.M) return;
    uint32_t r[16];
    tmem_ld16(tb + (uint32_t)(c16 * 16), r);
    tmem_ld_wait();
    unroll_cols<c16 * 16>(r, valid, vid, lane);
  }
  template <int m0> SPEC_DEV void unroll_cols(const uint32_t* r, bool valid, int vid, int lane) {
    if constexpr (m0 < MPAD) {
      if (m0 < P.M) {
        column<m0>(__uint_as_float(r[m0 & 15]), valid, vid, lane);
        if constexpr (((m0 + 1) & 15) != 0) unroll_cols<m0 + 1>(r, valid, vid, lane);
      }
    }
  }
  template <int c16> SPEC_DEV void chunks(uint32_t tb, bool valid, int vid, int lane) {
    if constexpr (c16 * 16 < MPAD) {
      chunk<c16>(tb, valid, vid, lane);
      chunks<c16 + 1>(tb, valid, vid, lane);
    }
  }

  SPEC_DEV void segment(const Seg& sg, uint32_t tb, int warp, int lane) {
    const int vid = sg.row0 + warp * 32 + lane;
    const bool valid = vid >= sg.lo && vid < sg.hi;
    chunks<0>(tb, valid, vid, lane);
  }

  SPEC_DEV void finish(int warp, int lane) {
    __shared__ float sh[4][MPAD][REC];
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      const int m = 32 * s + lane;
      if (m < MPAD) {
        sh[warp][m][0] = RM[s];
        sh[warp][m][1] = RS[s];
#pragma unroll
        for (int q = 0; q < KT; ++q) {
          sh[warp][m][2 + q] = TV[s][q];
          sh[warp][m][2 + KT + q] = __int_as_float(TI[s][q]);
        }
      }
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (warp != 0) return;
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      const int m = 32 * s + lane;
      if (m >= P.M) continue;
      float M_ = -INFINITY;
      for (int w = 0; w < 4; ++w) M_ = fmaxf(M_, sh[w][m][0]);
      float S_ = 0.f;
      for (int w = 0; w < 4; ++w)
        if (sh[w][m][0] > -INFINITY) S_ += sh[w][m][1] * expf(sh[w][m][0] - M_);
      for (int w = 1; w < 4; ++w)
        for (int q = 0; q < KT; ++q) {
          const float v = sh[w][m][2 + q];
          const int i = __float_as_int(sh[w][m][2 + KT + q]);
          if (better(v, i, TV[s][KT - 1], TI[s][KT - 1])) insert_rt(s, v, i);
        }
      float* o = P.out + ((size_t)c * MPAD + m) * REC;
      o[0] = M_;
      o[1] = S_;
      for (int q = 0; q < KT; ++q) {
        o[2 + q] = TV[s][q];
        o[2 + KT + q] = __int_as_float(TI[s][q]);
      }
    }
  }
  SPEC_DEV void insert_rt(int s, float v, int i) {
#pragma unroll
    for (int ss = 0; ss < NS; ++ss)
      if (ss == s) {
#pragma unroll
        for (int q = KT - 1; q >= 0; --q) {
          if (better(v, i, TV[ss][q], TI[ss][q])) {
            if (q > 0 && better(v, i, TV[ss][q - 1], TI[ss][q - 1])) {
              TV[ss][q] = TV[ss][q - 1];
              TI[ss][q] = TI[ss][q - 1];
            } else {
              TV[ss][q] = v;
              TI[ss][q] = i;
            }
          }
        }
      }
  }
};

}  // namespace tc

// Merge the per-CTA records of row m: lse (whole block) and the k best (warp 0:
// every lane keeps a sorted top-KT of the records it scans, then k rounds of a
// warp argmax over the lanes' heads).
template <int KT>
__global__ void __launch_bounds__(256) lm_merge_kernel(const float* __restrict__ part, int G, int mpad, int k,
                                                       int32_t* __restrict__ ids, int ld_ids,
                                                       float* __restrict__ lp, float* __restrict__ lse_out,
                                                       const int32_t* __restrict__ d2t) {
  pdl_wait();
  pdl_trigger();
  constexpr int REC = 2 + 2 * KT;
  __shared__ float red[32];
  __shared__ float s_lse;
  const int m = blockIdx.x;
  float mx = -INFINITY;
  for (int c = threadIdx.x; c < G; c += blockDim.x) mx = fmaxf(mx, part[((size_t)c * mpad + m) * REC]);
  mx = block_max(mx, red);
  float s = 0.f;
  for (int c = threadIdx.x; c < G; c += blockDim.x) {
    const float* r = part + ((size_t)c * mpad + m) * REC;
    if (r[0] > -INFINITY) s += r[1] * expf(r[0] - mx);
  }
  s = block_sum(s, red);
  const float lse = mx + logf(s);
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  float tv[KT];
  int ti[KT];
#pragma unroll
  for (int q = 0; q < KT; ++q) { tv[q] = -INFINITY; ti[q] = 0x7fffffff; }
  for (int e = lane; e < G * KT; e += 32) {
    const float* r = part + ((size_t)(e / KT) * mpad + m) * REC;
    const float v = r[2 + e % KT];
    const int i = __float_as_int(r[2 + KT + e % KT]);
    if (!better(v, i, tv[KT - 1], ti[KT - 1])) continue;
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
  }
  for (int rr = 0; rr < k; ++rr) {
    float bv = tv[0];
    int bi = ti[0];
    warp_argmax(bv, bi);
    if (ti[0] == bi) {          // the lane whose head won pops it (ids are distinct)
#pragma unroll
      for (int q = 0; q < KT - 1; ++q) { tv[q] = tv[q + 1]; ti[q] = ti[q + 1]; }
      tv[KT - 1] = -INFINITY;
      ti[KT - 1] = 0x7fffffff;
    }
    if (lane == 0) {
      ids[(size_t)m * ld_ids + rr] = d2t ? d2t[bi] : bi;
      lp[(size_t)m * ld_ids + rr] = bv - lse;
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
