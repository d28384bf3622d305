// Draft decoder layer: prologue (embedding gather + the two input norms),
// stream-K GEMM epilogues (RoPE + paged K/V write, residual + norms, SwiGLU),
// split-KV masked decode attention, and the unfused LM-head statistics.
//
// [NEURON] "Speculative Decoding (EAGLE3) in the vLLM Neuron Framework",
// section "Eagle3 Draft Model Architecture": embeds = input_layernorm(embed),
// hidden = hidden_norm(target hidden), concat [embeds, hidden] (2H), attention
// with QKV sized for 2H input, residual, post_attention_layernorm + MLP +
// residual, final norm; "EagleProposer" and "KV Cache Sharing": slot mapping
// block_table[pos // block_size] * block_size + pos % block_size.
// [EAGLE4] Eagle4Config.sliding_window: keys a draft query attends to, itself
// and its chain included.
//
// Storage precision (bf16 models): the concatenated normalised input x, q/k/v,
// the attention output, the post-attention-norm output, the MLP activation,
// hidden_prenorm and the normed output are stored in bf16; the residual stream
// stays fp32 inside the workspace; all accumulation is fp32.
#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"
#include "plan.cuh"
#include "tc_core.cuh"

namespace cg = cooperative_groups;

namespace spec {

// ---------------------------------------------------------------- row metadata
struct RowInfo {
  int M, B, R, step;
  const int32_t* ctx_len;
  const int32_t* tok;
  int tok_stride;
  const int32_t* pos;
  const int32_t* kv_idx;
  const uint64_t* mask;
  const int32_t* hid_src;
};
SPEC_DEV int row_req(const RowInfo& r, int m) { return m / r.R; }
SPEC_DEV int row_pos(const RowInfo& r, int m) { return r.pos ? r.pos[m] : r.ctx_len[m / r.R] + r.step; }
SPEC_DEV int row_kvidx(const RowInfo& r, int m) { return r.kv_idx ? r.kv_idx[m] : r.step; }
SPEC_DEV unsigned long long row_mask(const RowInfo& r, int m) {
  if (r.mask) return r.mask[m];
  return (r.step >= 63) ? ~0ull : ((2ull << r.step) - 1ull);
}
SPEC_DEV int row_src(const RowInfo& r, int m) { return r.hid_src ? r.hid_src[m] : m; }

RowInfo to_rowinfo(const spec_rows& r) {
  return RowInfo{r.M, r.B, r.rows_per_req, r.step, r.ctx_len, r.tok, r.tok_stride > 0 ? r.tok_stride : 1,
                 r.pos, r.kv_idx, r.mask, r.hid_src};
}

// ---------------------------------------------------------------- cluster helpers
// Row-wide reductions (RMSNorm over H) run on a thread-block cluster of CL
// CTAs per row, 2048 threads a row: each CTA owns H / CL features, the per-CTA
// sums meet in distributed shared memory, summed in rank order
// (deterministic).  Few rows spread over many SMs (CL = 8 CTAs of 256);
// from 32 rows on, a row takes two CTAs of 1024 (fewer cluster barriers;
// measured: 32 rows 384 -> 389 steps/s, 4 rows 686 -> 676 with CL = 2).
template <int CL> struct NormCL {
  static constexpr int kThreads = 2048 / CL < 1024 ? 2048 / CL : 1024;
};
inline int norm_cl(int M) { return M >= 32 ? 2 : 8; }
// Features a thread of the row-norm kernels keeps in registers (rows up to
// 2 x 2048 = 4096 features); wider rows take the looping form.
constexpr int kNormKeep = 2;

// Sum of v over the kCL CTAs of the cluster (each CTA: a block sum of both
// components in one pass, then its total pushed into slot[rank] of every CTA of
// the cluster; one cluster barrier; each CTA adds the slots in rank order).
// red: 64 floats of shared memory, slot: kCL float2 of shared memory.
template <int kCL>
SPEC_DEV float2 cluster_sum2(float2 v, float* red, float2* slot) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v.x = warp_sum(v.x);
  v.y = warp_sum(v.y);
  __syncthreads();
  if (lane == 0) reinterpret_cast<float2*>(red)[wid] = v;
  __syncthreads();
  float2 w = lane < nw ? reinterpret_cast<float2*>(red)[lane] : make_float2(0.f, 0.f);
  w.x = warp_sum(w.x);
  w.y = warp_sum(w.y);
  cg::cluster_group cl = cg::this_cluster();
  const int me = (int)cl.block_rank();
  if (threadIdx.x < kCL) cl.map_shared_rank(slot, (int)threadIdx.x)[me] = w;
  cl.sync();     // the pushes land before any CTA reads its slots; none is touched after
  float2 t = make_float2(0.f, 0.f);
#pragma unroll
  for (int r = 0; r < kCL; ++r) {
    const float2 o = slot[r];
    t.x += o.x;
    t.y += o.y;
  }
  return t;
}

struct RopeFreq {
  double inv[128];   // theta^(-2i/hd), i < hd/2 (hd <= 256)
};

// ---------------------------------------------------------------- prologue
// x[m] = [ input_layernorm(embed[tok_m]) , hidden_norm(hid_in[src_m]) ] and the
// row's rotary cos/sin table.  The angle pos * theta^(-2i/hd) is formed in fp64,
// reduced modulo 2*pi in fp64 (Cody-Waite, two-part 2*pi), then sin/cos are
// taken in fp32 on the reduced argument.
template <typename T, int kCL>
__global__ void __cluster_dims__(kCL, 1, 1) __launch_bounds__(NormCL<kCL>::kThreads)
    prologue_kernel(RowInfo ri, int H, int V, int hd, float eps, const __grid_constant__ RopeFreq rf,
                    const T* __restrict__ embed, const T* __restrict__ g_in, const T* __restrict__ g_hid,
                    const T* __restrict__ hid_in, T* __restrict__ x, float2* __restrict__ cs, void* ws) {
  SPEC_TL(spec::kTLPrologue);
  pdl_wait();
  pdl_trigger();
  __shared__ float red[64];
  __shared__ float2 slot[kCL];
  const int m = blockIdx.x / kCL, rk = blockIdx.x % kCL;
  int tok = ri.tok[(size_t)m * ri.tok_stride];
  if (tok < 0 || tok >= V) {
    if (threadIdx.x == 0 && rk == 0) report(ws, SPEC_ERR_DEVICE, m, tok);
    tok = 0;
  }
  const T* e = embed + (size_t)tok * H;
  const T* h = hid_in + (size_t)row_src(ri, m) * H;
  const int n0 = rk * H / kCL, n1 = (rk + 1) * H / kCL;
  T* xo = x + (size_t)m * 2 * H;
  float2 ss = make_float2(0.f, 0.f);
  if (n1 - n0 <= kNormKeep * (int)blockDim.x) {
    // at most kNormKeep features a thread: rows, gains and all loads at once, kept
    // in registers across the cluster reduction
    float a[kNormKeep], c[kNormKeep], ga[kNormKeep], gh[kNormKeep];
#pragma unroll
    for (int u = 0; u < kNormKeep; ++u) {
      const int n = n0 + threadIdx.x + u * blockDim.x;
      const bool on = n < n1;
      a[u] = on ? ld(e + n) : 0.f;
      c[u] = on ? ld(h + n) : 0.f;
      ga[u] = on ? ld(g_in + n) : 0.f;
      gh[u] = on ? ld(g_hid + n) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kNormKeep; ++u) {
      ss.x += a[u] * a[u];
      ss.y += c[u] * c[u];
    }
    const float2 tot = cluster_sum2<kCL>(ss, red, slot);
    const float re = 1.f / sqrtf(tot.x / H + eps), rh = 1.f / sqrtf(tot.y / H + eps);
#pragma unroll
    for (int u = 0; u < kNormKeep; ++u) {
      const int n = n0 + threadIdx.x + u * blockDim.x;
      if (n < n1) {
        st(xo + n, a[u] * re * ga[u]);
        st(xo + H + n, c[u] * rh * gh[u]);
      }
    }
  } else {
    for (int n = n0 + threadIdx.x; n < n1; n += blockDim.x) {
      const float a = ld(e + n), c = ld(h + n);
      ss.x += a * a;
      ss.y += c * c;
    }
    const float2 tot = cluster_sum2<kCL>(ss, red, slot);
    const float re = 1.f / sqrtf(tot.x / H + eps), rh = 1.f / sqrtf(tot.y / H + eps);
    for (int n = n0 + threadIdx.x; n < n1; n += blockDim.x) {
      st(xo + n, ld(e + n) * re * ld(g_in + n));
      st(xo + H + n, ld(h + n) * rh * ld(g_hid + n));
    }
  }
  if (rk == 0) {
    const int pos = row_pos(ri, m);
    const double two_pi_hi = 6.283185307179586, two_pi_lo = 2.4492935982947064e-16;
    for (int i = threadIdx.x; i < hd / 2; i += blockDim.x) {
      const double ang = (double)pos * rf.inv[i];
      const double k = rint(ang * (1.0 / 6.283185307179586));
      double r = fma(-k, two_pi_hi, ang);
      r = fma(-k, two_pi_lo, r);
      float sn, cn;
      sincosf((float)r, &sn, &cn);
      cs[(size_t)m * (hd / 2) + i] = make_float2(cn, sn);
    }
  }
}

// ---------------------------------------------------------------- epilogues
// plain: out[m, n] = sum of partials (stored in T or fp32)
template <typename TO>
__global__ void epi_store_kernel(const float* __restrict__ part, SKPlan p, int M, int N, TO* __restrict__ out,
                                 int ld_out) {
  SPEC_TL(spec::kTLEpiStore);
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const bool live = idx < (long long)M * N;
  const int m = live ? (int)(idx / N) : 0, n = live ? (int)(idx % N) : 0;
  // the feature's tile segments from the plan before the dependency wait
  SKTileSegs seg[1];
  int lane[1], tile;
  sk_feature(p, n, tile, lane[0]);
  seg[0] = sk_tile_segs(p, tile);
  pdl_wait();
  pdl_trigger();
  if (!live) return;
  const bool on[1] = {true};
  SKGather<1, 16> gat;                        // up to 17 segments (one-tile GEMMs with a long K) at once
  sk_gather_segs<1, 16>(part, p, m, seg, lane, on, gat);
  float v[1];
  sk_reduce<1, 16>(p, gat, v);
  st(out + (size_t)m * ld_out + n, v[0]);
}

// q / k get the rotary embedding (pairs i, i + hd/2), v is copied; q goes to
// qbuf [M, nq*hd], k and v to the paged cache at entry ctx + kv_idx.
template <typename T>
__global__ void epi_qkv_kernel(const float* __restrict__ part, SKPlan p, RowInfo ri, int nq, int nkv, int hd,
                               const float2* __restrict__ cs, T* __restrict__ qbuf, spec_kv kv, int* __restrict__ work,
                               void* ws) {
  SPEC_TL(spec::kTLEpiQkv);
  const int half = hd / 2;
  const int nh = nq + 2 * nkv;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const bool live = idx < (long long)ri.M * nh * half;
  const int m = live ? (int)(idx / (nh * half)) : 0;
  const int rem = live ? (int)(idx % (nh * half)) : 0;
  const int hh = rem / half, i = rem % half;
  const int n1 = hh * hd + i, n2 = n1 + half;
  // Before the dependency wait: the pair's tile segments (both features lie in
  // one tile -- heads do not straddle tiles -- so worked out once), and for a K / V
  // head the row's cache slot.  Context lengths, cache indices and the block table
  // are inputs of the call that no kernel of it writes, and this kernel starts only
  // once every block of the QKV GEMM has passed its own wait, i.e. after the
  // prologue (and all earlier launches) finished; they are read through L2.
  SKTileSegs seg[2];
  int lane[2], t1, t2;
  sk_feature(p, n1, t1, lane[0]);
  sk_feature(p, n2, t2, lane[1]);
  seg[0] = sk_tile_segs(p, t1);
  seg[1] = t2 == t1 ? seg[0] : sk_tile_segs(p, t2);
  int b = 0, ci = 0;
  long long slot = 0;
  if (live && hh >= nq) {
    b = row_req(ri, m);
    ci = __ldcg(ri.ctx_len + b) + (ri.kv_idx ? __ldcg(ri.kv_idx + m) : ri.step);
    const int blk = ci / kv.block_size;
    slot = -1;
    if (ci >= 0 && blk < kv.max_blocks) {
      const long long s0 = (long long)__ldcg(kv.block_table + (long long)b * kv.max_blocks + blk) * kv.block_size +
                           ci % kv.block_size;
      if (s0 >= 0 && s0 < kv.num_slots) slot = s0;
    }
  }
  pdl_wait();
  pdl_trigger();
  if (work != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *work = 0;   // the attention's item counter
  if (!live) return;
  // the rotary pair (written by the prologue) is read while the partials load
  float2 c = make_float2(1.f, 0.f);
  if (hh < nq + nkv) c = cs[(size_t)m * half + i];
  const bool on[2] = {true, true};
  SKGather<2, kSegBatch> gat;
  sk_gather_segs<2, kSegBatch>(part, p, m, seg, lane, on, gat);
  float xv[2];
  sk_reduce<2, kSegBatch>(p, gat, xv);
  float x1 = xv[0], x2 = xv[1];
  if (hh < nq + nkv) {
    const float y1 = x1 * c.x - x2 * c.y;
    const float y2 = x2 * c.x + x1 * c.y;
    x1 = y1;
    x2 = y2;
  }
  if (hh < nq) {
    T* q = qbuf + (size_t)m * nq * hd + (size_t)hh * hd;
    st(q + i, x1);
    st(q + i + half, x2);
    return;
  }
  if (slot < 0) {
    report(ws, SPEC_ERR_DEVICE, m, ci);
    return;
  }
  const bool isk = hh < nq + nkv;
  const int g = isk ? hh - nq : hh - nq - nkv;
  T* base = reinterpret_cast<T*>(isk ? kv.k : kv.v) + ((size_t)slot * nkv + g) * hd;
  st(base + i, x1);
  st(base + i + half, x2);
}

// MODE 0 (after o_proj):  r = hid_in[src] + o;   out_b = post_attention_layernorm(r)
// MODE 1 (after down):    r = r + down; out_a = r (hidden_prenorm); out_b = final_norm(r)
// MODE 2 (after the FC, EAGLE-3.1 fc_norm): r = fc output; out_b = fc_norm(r)
// One cluster of kCL CTAs per row.
template <typename T, int MODE, int kCL>
__global__ void __cluster_dims__(kCL, 1, 1) __launch_bounds__(NormCL<kCL>::kThreads)
    resnorm_kernel(const float* __restrict__ part, SKPlan p, RowInfo ri, int H, float eps,
                   const T* __restrict__ hid_in, const T* __restrict__ gain, float* __restrict__ r,
                   T* __restrict__ out_a, T* __restrict__ out_b) {
  SPEC_TL(spec::kTLResnorm);
  // the next launch (a GEMM) may start and fill its ring with weight tiles once every
  // block of this one has started, instead of after this kernel's dependency wait
  pdl_trigger();
  __shared__ float red[64];
  __shared__ float2 slot[kCL];
  __shared__ SKTileSegs s_seg[kNormKeep * 1024 / 128 + 2];
  const int m = blockIdx.x / kCL, rk = blockIdx.x % kCL;
  const int n0 = rk * H / kCL, n1 = (rk + 1) * H / kCL;
  const T* h = (MODE == 0) ? hid_in + (size_t)row_src(ri, m) * H : nullptr;
  float* rr = r + (size_t)m * H;
  float ss = 0.f;
  if (n1 - n0 <= kNormKeep * (int)blockDim.x && p.nmat == 1) {
    // at most kNormKeep features a thread: bases, partials and gains loaded at once,
    // the row kept in registers across the cluster reduction.  The segments of the
    // block's tiles (from the plan) and the gains (weights) before the dependency wait.
    const int tb = n0 >> 7;
    for (int t = threadIdx.x; t <= ((n1 - 1) >> 7) - tb; t += blockDim.x) s_seg[t] = sk_tile_segs(p, tb + t);
    int nn[kNormKeep], lane[kNormKeep];
    bool on[kNormKeep];
    float base[kNormKeep], sv[kNormKeep], gv[kNormKeep];
#pragma unroll
    for (int u = 0; u < kNormKeep; ++u) {
      nn[u] = n0 + threadIdx.x + u * blockDim.x;
      on[u] = nn[u] < n1;
      lane[u] = nn[u] & 127;
      gv[u] = on[u] ? ld(gain + nn[u]) : 0.f;
    }
    pdl_wait();
      __syncthreads();
    SKTileSegs seg[kNormKeep];
#pragma unroll
    for (int u = 0; u < kNormKeep; ++u) {
      seg[u] = s_seg[on[u] ? (nn[u] >> 7) - tb : 0];
      base[u] = !on[u] ? 0.f : (MODE == 0) ? ld(h + nn[u]) : (MODE == 1 ? rr[nn[u]] : 0.f);
    }
    SKGather<kNormKeep, kSegBatch> gat;
    sk_gather_segs<kNormKeep, kSegBatch>(part, p, m, seg, lane, on, gat);
    sk_reduce<kNormKeep, kSegBatch>(p, gat, sv);
#pragma unroll
    for (int u = 0; u < kNormKeep; ++u) {
      sv[u] += base[u];
      if (!on[u]) continue;
      rr[nn[u]] = sv[u];
      if (MODE == 1) st(out_a + (size_t)m * H + nn[u], sv[u]);
      ss += sv[u] * sv[u];
    }
    const float2 tot = cluster_sum2<kCL>(make_float2(ss, 0.f), red, slot);
    const float rs = 1.f / sqrtf(tot.x / H + eps);
#pragma unroll
    for (int u = 0; u < kNormKeep; ++u)
      if (on[u]) st(out_b + (size_t)m * H + nn[u], sv[u] * rs * gv[u]);
    return;
  }
  pdl_wait();
  // two features a thread per round, their partials' loads in flight together
  for (int n = n0 + threadIdx.x; n < n1; n += 2 * blockDim.x) {
    const int nn[2] = {n, n + (int)blockDim.x};
    const bool on[2] = {true, nn[1] < n1};
    float base[2], sv[2];
#pragma unroll
    for (int u = 0; u < 2; ++u)
      base[u] = !on[u] ? 0.f : (MODE == 0) ? ld(h + nn[u]) : (MODE == 1 ? rr[nn[u]] : 0.f);
    sk_sum_n<2>(part, p, m, nn, on, sv);
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (!on[u]) continue;
      const int k = nn[u];
      const float v = base[u] + sv[u];
      rr[k] = v;
      if (MODE == 1) st(out_a + (size_t)m * H + k, v);
      ss += v * v;
    }
  }
  const float2 tot = cluster_sum2<kCL>(make_float2(ss, 0.f), red, slot);
  const float rs = 1.f / sqrtf(tot.x / H + eps);
  for (int n = n0 + threadIdx.x; n < n1; n += blockDim.x) st(out_b + (size_t)m * H + n, rr[n] * rs * ld(gain + n));
}

// act = silu(gate) * up  (gate rows [0, I), up rows [I, 2I) of the stacked output).
// Block (x, m): features x * 256 U + u * 256 + threadIdx.x of row m, u < U (U = 4
// when the batch gives enough blocks, else 1); every partial of a thread's
// features is loaded before the first add (a gate / up tile spans few CTAs:
// three segments are loaded at once, more one by one).
template <typename T, int U>
__global__ void __launch_bounds__(256) epi_swiglu_kernel(const float* __restrict__ part, SKPlan p, int M, int I,
                                                         T* __restrict__ act) {
  SPEC_TL(spec::kTLSwiglu);
  // one feature a thread (small batches): the down projection may start and fill its
  // ring once every block has started (measured better there, worse at four)
  if (U == 1) pdl_trigger();
  // the block's 2U gate tiles and 2U up tiles: their segments once, into shared
  // memory, from the plan alone (before the dependency wait)
  __shared__ SKTileSegs s_seg[4 * U];
  const int ib = blockIdx.x * U * 256;
  if (threadIdx.x < 4 * U) {
    const int k = threadIdx.x, half = k / (2 * U);
    int tile, lane;
    sk_feature(p, half * I + min(ib + 128 * (k % (2 * U)), I - 1), tile, lane);
    s_seg[k] = sk_tile_segs(p, tile);
  }
  pdl_wait();
  if (U != 1) pdl_trigger();
  __syncthreads();
  const int m = blockIdx.y;
  SKTileSegs seg[2 * U];
  int lane[2 * U];
  bool on[2 * U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int i = ib + threadIdx.x + u * 256;
    on[2 * u] = on[2 * u + 1] = i < I;
    lane[2 * u] = lane[2 * u + 1] = i & 127;
    seg[2 * u] = s_seg[(threadIdx.x >> 7) + 2 * u];
    seg[2 * u + 1] = s_seg[2 * U + (threadIdx.x >> 7) + 2 * u];
  }
  SKGather<2 * U, 2> gat;
  sk_gather_segs<2 * U, 2>(part, p, m, seg, lane, on, gat);
  float gu[2 * U];
  sk_reduce<2 * U, 2>(p, gat, gu);
#pragma unroll
  for (int u = 0; u < U; ++u) {
    if (!on[2 * u]) continue;
    const float g = gu[2 * u], v = gu[2 * u + 1];
    st(act + (size_t)m * I + ib + threadIdx.x + u * 256, g / (1.f + expf(-g)) * v);
  }
}

// ---------------------------------------------------------------- SIMT GEMM
// Stream-K GEMM on CUDA cores (fp32 models, and M <= 32): partial sums of
// X[M, K] @ W^T for the CTA's iteration range, same partial layout as the
// tensor-core kernel.
template <typename T>
__global__ void __launch_bounds__(256) simt_gemm_kernel(const T* __restrict__ A0, const T* __restrict__ A1,
                                                        const T* __restrict__ A2, int K, const T* __restrict__ X,
                                                        int M, SKPlan p, float* __restrict__ part) {
  SPEC_TL(spec::kTLSimt);
  pdl_wait();
  pdl_trigger();
  __shared__ float sW[128][65];
  __shared__ float sX[32][65];
  const int c = blockIdx.x;
  long long it = sk_begin(p, c);
  const long long end = sk_begin(p, c + 1);
  const int r = threadIdx.x & 127, mh = threadIdx.x >> 7;
  int j = 0;
  while (it < end) {
    const int tile = (int)(it / p.kc);
    const long long seg_end = min(end, (long long)(tile + 1) * p.kc);
    int mat, row0;
    sk_tile_map(p, tile, mat, row0);
    const T* A = mat == 0 ? A0 : (mat == 1 ? A1 : A2);
    const int rows = p.obase[mat + 1] - p.obase[mat];
    float acc[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) acc[q] = 0.f;
    for (; it < seg_end; ++it) {
      const int k0 = (int)(it % p.kc) * 64;
      __syncthreads();
      for (int e = threadIdx.x; e < 128 * 64; e += blockDim.x) {
        const int rr = e >> 6, kk = e & 63;
        sW[rr][kk] = (row0 + rr < rows && k0 + kk < K) ? ld(A + (size_t)(row0 + rr) * K + k0 + kk) : 0.f;
      }
      for (int e = threadIdx.x; e < 32 * 64; e += blockDim.x) {
        const int mm = e >> 6, kk = e & 63;
        sX[mm][kk] = (mm < M && k0 + kk < K) ? ld(X + (size_t)mm * K + k0 + kk) : 0.f;
      }
      __syncthreads();
#pragma unroll 4
      for (int kk = 0; kk < 64; ++kk) {
        const float w = sW[r][kk];
#pragma unroll
        for (int q = 0; q < 16; ++q) acc[q] += w * sX[mh + 2 * q][kk];
      }
    }
    float* dst = part + sk_slot(p, c, j);
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const int m = mh + 2 * q;
      if (m < M) dst[(size_t)m * 128 + r] = acc[q];
    }
    ++j;
  }
}

// ---------------------------------------------------------------- attention
SPEC_DEV void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem_dst)),
               "l"(gmem_src)
               : "memory");
}
SPEC_DEV void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

template <typename T> SPEC_DEV void unpack16(const uint4& r, float* o);
template <> SPEC_DEV void unpack16<float>(const uint4& r, float* o) {
  o[0] = __uint_as_float(r.x); o[1] = __uint_as_float(r.y); o[2] = __uint_as_float(r.z); o[3] = __uint_as_float(r.w);
}
template <> SPEC_DEV void unpack16<__nv_bfloat16>(const uint4& r, float* o) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    o[2 * i] = __uint_as_float(w[i] << 16);
    o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// Split-KV decode attention with the row masks of spec_rows.
//
// Work item = (request b, query group qg, kv head g, split s): up to QMAX
// queries (rows of one request x the q heads of kv head g) over one slice of
// that request's keys -- context keys [klo, ctx) then draft-region keys
// [ctx, ctx + nd).  The grid is persistent (as many CTAs as fit at once); CTA c
// takes items c, c + grid, ...  Keys stream through shared memory in tiles of
// 64 with cp.async, NST tiles in flight, so the copies of the next tiles
// overlap the arithmetic on the current one.  Per tile: scores (thread = key x
// half of the queries, packed fp32 FMAs), an online softmax per query (warp w:
// queries w, w + 4, ...), then P.V with warp w taking keys 16w .. 16w+15 for
// every query and lane l the head dims of l.  The four warps' partial outputs
// are summed once per item.
constexpr int kAttnTK = 64;
constexpr int kAttnNST = 2;

template <typename T, int HD> struct AttnShape {
  static constexpr int KP = HD + 16 / (int)sizeof(T);          // padded K row (elements)
  static constexpr int CH = HD * (int)sizeof(T) / 16;          // 16-byte chunks per row
  static constexpr int STAGE = kAttnTK * KP * (int)sizeof(T) + kAttnTK * HD * (int)sizeof(T);
  static constexpr int DPL = HD / 32;                          // head dims per lane in P.V
};

template <typename T, int HD, int QMAX>
constexpr size_t attn_smem_for() {
  using A = AttnShape<T, HD>;
  const size_t stages = (size_t)kAttnNST * A::STAGE;
  const size_t red = (size_t)4 * QMAX * HD * 4;                // the warps' partial outputs (aliases the stages)
  return (stages > red ? stages : red) + (size_t)QMAX * HD * 4 + (size_t)QMAX * kAttnTK * 4;
}

template <typename T> SPEC_DEV void unpack_pair(uint32_t w, float2& o);
template <> SPEC_DEV void unpack_pair<__nv_bfloat16>(uint32_t w, float2& o) {
  o.x = __uint_as_float(w << 16);
  o.y = __uint_as_float(w & 0xffff0000u);
}

template <typename T, int HD, int QMAX>
__global__ void __launch_bounds__(128) attn_split_kernel(const T* __restrict__ qbuf, spec_kv kv, RowInfo ri,
                                                         int nq, int nkv, int window, int nsplit, int nqg,
                                                         int n_items, float scale, float* __restrict__ opart,
                                                         float2* __restrict__ mlpart, void* ws) {
  SPEC_TL(spec::kTLAttnSplit);
  pdl_wait();
  pdl_trigger();
  using A = AttnShape<T, HD>;
  constexpr int TK = kAttnTK, NST = kAttnNST, KP = A::KP, CH = A::CH, DPL = A::DPL;
  constexpr int QH = QMAX / 2;                  // queries per thread in the scores
  constexpr int QW = QMAX / 4;                  // queries per warp in the softmax
  extern __shared__ __align__(16) uint8_t attn_smem[];
  constexpr size_t kStages = attn_smem_for<T, HD, QMAX>() - (size_t)QMAX * HD * 4 - (size_t)QMAX * TK * 4;
  float* sQ = reinterpret_cast<float*>(attn_smem + kStages);          // [QMAX][HD], scaled
  float* sS = sQ + QMAX * HD;                                         // [QMAX][TK]
  float* red = reinterpret_cast<float*>(attn_smem);                   // [4][QMAX][HD] after the last tile
  __shared__ float sM[QMAX], sL[QMAX], sA[QMAX];
  __shared__ int s_lo[QMAX];
  __shared__ unsigned long long s_mask[QMAX];
  __shared__ int s_klo, s_nd;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = nq / nkv;
  const int nQall = ri.R * G;

  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int s = item % nsplit;
    const int g = (item / nsplit) % nkv;
    const int bq = item / (nsplit * nkv);
    const int b = bq / nqg, qg = bq % nqg;
    const int q0 = qg * QMAX;
    const int nQ = min(QMAX, nQall - q0);
    const int ctx = ri.ctx_len[b];

    if (tid < 32) {
      int lo = 0x7fffffff;
      unsigned long long mk = 0;
      if (tid < nQ) {
        const int m = b * ri.R + (q0 + tid) / G;
        const int pos = row_pos(ri, m);
        lo = window > 0 ? max(0, pos - window + 1) : 0;
        if (lo > ctx) lo = ctx;
        mk = row_mask(ri, m);
      }
      if (tid < QMAX) {
        s_lo[tid] = lo;
        s_mask[tid] = mk;
        sM[tid] = -INFINITY;
        sL[tid] = 0.f;
      }
      int mlo = lo;
      unsigned long long om = mk;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        mlo = min(mlo, __shfl_xor_sync(0xffffffffu, mlo, o));
        om |= __shfl_xor_sync(0xffffffffu, om, o);
      }
      if (tid == 0) {
        s_klo = mlo;
        s_nd = om ? 64 - __clzll((long long)om) : 0;
      }
    }
    for (int e = tid; e < QMAX * HD; e += blockDim.x) {
      const int qi = e / HD, d = e % HD;
      float v = 0.f;
      if (qi < nQ) {
        const int q = q0 + qi;
        const int m = b * ri.R + q / G, h = g * G + q % G;
        v = ld(qbuf + ((size_t)m * nq + h) * HD + d) * scale;
      }
      sQ[e] = v;
    }
    __syncthreads();
    const int klo = s_klo, nd = s_nd;
    const int nctx = ctx - klo;
    const int total = nctx + nd;
    const int chunk = ((total + nsplit - 1) / nsplit + TK - 1) / TK * TK;   // whole tiles per split
    const int kbeg = min(total, s * chunk), kend = min(total, kbeg + chunk);
    const int ntiles = (kend - kbeg + TK - 1) / TK;

    // stage tile j (keys kbeg + j*TK ...) into ring slot j % NST: thread t copies
    // chunk t % CH of keys t / CH, t / CH + 128 / CH, ...
    auto issue = [&](int j) {
      if (j < ntiles) {
        uint8_t* st = attn_smem + (size_t)(j % NST) * A::STAGE;
        T* sK = reinterpret_cast<T*>(st);
        T* sV = reinterpret_cast<T*>(st + TK * KP * sizeof(T));
        const int t0 = kbeg + j * TK;
        const int nk = min(TK, kend - t0);
        const int ch = tid % CH;
        for (int kt = tid / CH; kt < nk; kt += 128 / CH) {
          const int kidx = t0 + kt;
          const int ci = kidx < nctx ? klo + kidx : ctx + (kidx - nctx);
          const long long slot = slot_of(kv, b, ci);
          uint4* dk = reinterpret_cast<uint4*>(sK + kt * KP) + ch;
          uint4* dv = reinterpret_cast<uint4*>(sV + kt * HD) + ch;
          if (slot >= 0) {
            const size_t off = ((size_t)slot * nkv + g) * HD;
            cp_async16(dk, reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(kv.k) + off) + ch);
            cp_async16(dv, reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(kv.v) + off) + ch);
          } else {
            *dk = make_uint4(0, 0, 0, 0);
            *dv = make_uint4(0, 0, 0, 0);
          }
        }
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    };

    float2 acc[QMAX][DPL / 2];
#pragma unroll
    for (int q = 0; q < QMAX; ++q)
#pragma unroll
      for (int u = 0; u < DPL / 2; ++u) acc[q][u] = make_float2(0.f, 0.f);

#pragma unroll
    for (int j = 0; j < NST - 1; ++j) issue(j);
    for (int j = 0; j < ntiles; ++j) {
      issue(j + NST - 1);
      asm volatile("cp.async.wait_group %0;" ::"n"(NST - 1) : "memory");
      __syncthreads();
      const uint8_t* st = attn_smem + (size_t)(j % NST) * A::STAGE;
      const T* sK = reinterpret_cast<const T*>(st);
      const T* sV = reinterpret_cast<const T*>(st + TK * KP * sizeof(T));
      const int t0 = kbeg + j * TK;
      const int nk = min(TK, kend - t0);
      // scores: thread = (key kt, query half qh)
      {
        const int kt = tid % TK, qh = tid / TK;
        if (kt < nk) {
          const int kidx = t0 + kt;
          const int ci = kidx < nctx ? klo + kidx : ctx + (kidx - nctx);
          const bool valid = slot_of(kv, b, ci) >= 0;
          float2 sc[QH];
#pragma unroll
          for (int q = 0; q < QH; ++q) sc[q] = make_float2(0.f, 0.f);
          const uint4* kr = reinterpret_cast<const uint4*>(sK + kt * KP);
#pragma unroll 4
          for (int c = 0; c < CH; ++c) {
            const uint4 raw = kr[c];
            float2 k2[4];
            if constexpr (sizeof(T) == 2) {
              unpack_pair<T>(raw.x, k2[0]);
              unpack_pair<T>(raw.y, k2[1]);
              unpack_pair<T>(raw.z, k2[2]);
              unpack_pair<T>(raw.w, k2[3]);
            } else {
              k2[0] = make_float2(__uint_as_float(raw.x), __uint_as_float(raw.y));
              k2[1] = make_float2(__uint_as_float(raw.z), __uint_as_float(raw.w));
            }
            constexpr int NP = sizeof(T) == 2 ? 4 : 2;            // float pairs in 16 bytes
            const int d0 = c * 2 * NP;
#pragma unroll
            for (int q = 0; q < QH; ++q) {
              const float2* qr = reinterpret_cast<const float2*>(sQ + (qh * QH + q) * HD + d0);
#pragma unroll
              for (int u = 0; u < NP; ++u) sc[q] = __ffma2_rn(qr[u], k2[u], sc[q]);
            }
          }
#pragma unroll
          for (int q = 0; q < QH; ++q) {
            const int qi = qh * QH + q;
            bool ok = valid && qi < nQ;
            if (ok) {
              if (ci < ctx) ok = ci >= s_lo[qi];
              else ok = (s_mask[qi] >> (ci - ctx)) & 1ull;
            }
            sS[qi * TK + kt] = ok ? sc[q].x + sc[q].y : -INFINITY;
          }
        } else {
#pragma unroll
          for (int q = 0; q < QH; ++q) sS[(qh * QH + q) * TK + kt] = -INFINITY;
        }
      }
      __syncthreads();
      // online softmax: warp w handles queries w, w + 4, ...
#pragma unroll
      for (int a = 0; a < QW; ++a) {
        const int qi = warp + 4 * a;
        const float v0 = sS[qi * TK + lane], v1 = sS[qi * TK + lane + 32];
        const float mx = warp_max(fmaxf(v0, v1));
        const float mold = sM[qi];
        const float mnew = fmaxf(mold, mx);
        const float e0 = mnew == -INFINITY ? 0.f : expf(v0 - mnew);
        const float e1 = mnew == -INFINITY ? 0.f : expf(v1 - mnew);
        sS[qi * TK + lane] = e0;
        sS[qi * TK + lane + 32] = e1;
        const float sum = warp_sum(e0 + e1);
        if (lane == 0) {
          const float al = mold == -INFINITY ? 0.f : expf(mold - mnew);
          sA[qi] = al;
          sL[qi] = sL[qi] * al + sum;
          sM[qi] = mnew;
        }
      }
      __syncthreads();
      // P.V: warp w takes keys 16w .. 16w+15, all queries; lane l head dims DPL*l ..
#pragma unroll
      for (int q = 0; q < QMAX; ++q) {
        const float al = sA[q];
#pragma unroll
        for (int u = 0; u < DPL / 2; ++u) acc[q][u] = __fmul2_rn(acc[q][u], make_float2(al, al));
      }
      const int kb = warp * (TK / 4), ke = min(nk, kb + TK / 4);
      for (int kt = kb; kt < ke; ++kt) {
        float2 v2[DPL / 2];
        if constexpr (sizeof(T) == 2) {
          if constexpr (DPL == 4) {
            const uint2 raw = *reinterpret_cast<const uint2*>(sV + kt * HD + DPL * lane);
            unpack_pair<T>(raw.x, v2[0]);
            unpack_pair<T>(raw.y, v2[1]);
          } else {
            const uint32_t raw = *reinterpret_cast<const uint32_t*>(sV + kt * HD + DPL * lane);
            unpack_pair<T>(raw, v2[0]);
          }
        } else {
#pragma unroll
          for (int u = 0; u < DPL / 2; ++u)
            v2[u] = *reinterpret_cast<const float2*>(reinterpret_cast<const float*>(sV) + kt * HD + DPL * lane + 2 * u);
        }
#pragma unroll
        for (int q = 0; q < QMAX; ++q) {
          const float pw = sS[q * TK + kt];
#pragma unroll
          for (int u = 0; u < DPL / 2; ++u) acc[q][u] = __ffma2_rn(make_float2(pw, pw), v2[u], acc[q][u]);
        }
      }
      __syncthreads();     // ring slot j % NST is refilled by the next iteration's copies
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    // sum the warps' partial outputs, write this split's partials
#pragma unroll
    for (int q = 0; q < QMAX; ++q)
#pragma unroll
      for (int u = 0; u < DPL / 2; ++u)
        *reinterpret_cast<float2*>(red + ((size_t)warp * QMAX + q) * HD + DPL * lane + 2 * u) = acc[q][u];
    __syncthreads();
    for (int e = tid; e < QMAX * HD; e += blockDim.x) {
      const int qi = e / HD, d = e % HD;
      if (qi >= nQ) continue;
      const float o = red[e] + red[QMAX * HD + e] + red[2 * QMAX * HD + e] + red[3 * QMAX * HD + e];
      const int q = q0 + qi;
      const int m = b * ri.R + q / G, h = g * G + q % G;
      const size_t base = ((size_t)m * nq + h) * nsplit + s;
      opart[base * HD + d] = o;
      if (d == 0) mlpart[base] = make_float2(sM[qi], sL[qi]);
    }
    __syncthreads();     // red / sQ / sM reused by the next item
  }
}

// ---------------------------------------------------------------- attention on tensor cores (bf16)
// Same work items, persistent grid and two-stage cp.async ring of 64-key tiles
// as attn_split_kernel, but the two products run as warp-level bf16 MMAs
// (m16n8k16, fp32 accumulate): the item's up to 16*MT queries are the MMA rows
// (padded with zero rows), warp w owns keys 16w .. 16w+15 of every tile and
// keeps its own running max / sum / output for them (no cross-warp exchange
// per tile); the four warps' results merge once per item.  Scores:
// S[q, key] = Q[q, :] . K[key, :] with K rows as the "col" operand; the
// probabilities P (bf16) go straight from the score accumulators into the
// P.V product's A operand; V tiles are read transposed by ldmatrix.
constexpr int kMmaTK = 64;
// K/V ring slots.  Two (one tile in flight ahead of the one in use) with three
// CTAs per SM measured faster than three slots with two CTAs per SM.
constexpr int mma_stages(int) { return 2; }

template <int HD> struct MmaShape {
  static constexpr int KP = HD + 8;                         // padded bf16 row: ldmatrix rows on distinct banks
  static constexpr int STAGE = 2 * kMmaTK * KP * 2;          // K and V tiles
};

template <int HD, int MT>
constexpr size_t attn_mma_smem() {
  using S = MmaShape<HD>;
  const size_t ring = (size_t)mma_stages(MT) * S::STAGE;
  const size_t red = (size_t)4 * 16 * MT * (HD + 8) * 4;      // the warps' outputs after the last tile (aliases the ring)
  return (ring > red ? ring : red) + (size_t)16 * MT * S::KP * 2 + (size_t)mma_stages(MT) * kMmaTK * 4;
}

SPEC_DEV uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
SPEC_DEV void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
SPEC_DEV void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
SPEC_DEV void mma_bf16(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
               "{%0,%1,%2,%3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
SPEC_DEV uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

template <int HD, int MT>
__global__ void __launch_bounds__(128) attn_mma_kernel(const __nv_bfloat16* __restrict__ qbuf, spec_kv kv, RowInfo ri,
                                                       int nq, int nkv, int window, int nsplit, int nqg,
                                                       int n_items, float scale_log2, float* __restrict__ opart,
                                                       float2* __restrict__ mlpart, int* __restrict__ work,
                                                       void* ws) {
  SPEC_TL(spec::kTLAttnMma);
  pdl_wait();
  pdl_trigger();
  using Sh = MmaShape<HD>;
  constexpr int TK = kMmaTK, KP = Sh::KP, CH = HD / 8, QM = 16 * MT, NT = HD / 8, KS = HD / 16;
  extern __shared__ __align__(16) uint8_t mma_smem[];
  constexpr int NS = mma_stages(MT);
  constexpr size_t kRing = attn_mma_smem<HD, MT>() - (size_t)QM * KP * 2 - (size_t)NS * TK * 4;
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(mma_smem + kRing);   // [QM][KP]
  int* sCi = reinterpret_cast<int*>(sQ + QM * KP);                          // [NS][TK] cache index, -1 = no slot
  float* red = reinterpret_cast<float*>(mma_smem);                           // [4][QM][HD + 8]
  __shared__ float sMw[4][QM], sLw[4][QM];
  __shared__ int s_lo[QM];
  __shared__ unsigned long long s_mask[QM];
  __shared__ int s_klo, s_nd;
  __shared__ __align__(8) uint64_t full_bar[NS];    // a ring slot's rows have landed
  __shared__ int s_abort, s_next;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int grp = lane >> 2, tig = lane & 3;
  const int G = nq / nkv;
  const int nQall = ri.R * G;
  const uint32_t bar0 = smem_u32(&full_bar[0]);
  if (tid == 0) {
    s_abort = 0;
    for (int i = 0; i < NS; ++i) tc::mbar_init(bar0 + 8u * i, 128);   // every thread arrives once per fill
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  volatile int* abort = &s_abort;
  uint64_t kv_policy;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(kv_policy));
  uint32_t fills = 0;                                 // ring fills consumed by this CTA before this item
  uint32_t issued = 0, cons = 0;                      // fills issued; the fill a timed-out wait was for
  bool ok_all = true;

  // items: blockIdx.x first, then the next unclaimed one from a shared counter (ragged
  // requests make items of very different lengths; claiming balances them)
  for (int item = blockIdx.x; item < n_items;) {
    const int s = item % nsplit;
    const int g = (item / nsplit) % nkv;
    const int bq = item / (nsplit * nkv);
    const int b = bq / nqg, qg = bq % nqg;
    const int q0 = qg * QM;
    const int nQ = min(QM, nQall - q0);
    const int ctx = ri.ctx_len[b];

    if (tid < 32) {
      int lo = 0x7fffffff;
      unsigned long long mk = 0;
      if (tid < nQ) {
        const int m = b * ri.R + (q0 + tid) / G;
        const int pos = row_pos(ri, m);
        lo = window > 0 ? max(0, pos - window + 1) : 0;
        if (lo > ctx) lo = ctx;
        mk = row_mask(ri, m);
      }
      if (tid < QM) {
        s_lo[tid] = lo;
        s_mask[tid] = mk;
      }
      int mlo = lo;
      unsigned long long om = mk;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        mlo = min(mlo, __shfl_xor_sync(0xffffffffu, mlo, o));
        om |= __shfl_xor_sync(0xffffffffu, om, o);
      }
      if (tid == 0) {
        s_klo = mlo;
        s_nd = om ? 64 - __clzll((long long)om) : 0;
      }
    }
    __syncthreads();
    const int klo = s_klo, nd = s_nd;
    const int nctx = ctx - klo;
    const int total = nctx + nd;
    const int chunk = ((total + nsplit - 1) / nsplit + TK - 1) / TK * TK;
    const int kbeg = min(total, s * chunk), kend = min(total, kbeg + chunk);
    const int ntiles = (kend - kbeg + TK - 1) / TK;
    if (ntiles > 0) {
      // queries of the item (bf16, unscaled), zero rows past nQ
      for (int e = tid; e < QM * CH; e += blockDim.x) {
        const int qi = e / CH, c = e % CH;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (qi < nQ) {
          const int q = q0 + qi;
          const int m = b * ri.R + q / G, h = g * G + q % G;
          v = *reinterpret_cast<const uint4*>(qbuf + ((size_t)m * nq + h) * HD + c * 8);
        }
        *reinterpret_cast<uint4*>(sQ + qi * KP + c * 8) = v;
      }
    } else {
      // an empty split (a short request): its partials say "no keys"
      for (int e = tid; e < nQ * HD; e += blockDim.x) {
        const int qi = e / HD, d = e % HD;
        const int q = q0 + qi;
        const size_t base = ((size_t)(b * ri.R + q / G) * nq + g * G + q % G) * nsplit + s;
        opart[base * HD + d] = 0.f;
        if (d == 0) mlpart[base] = make_float2(-INFINITY, 0.f);
      }
    }
    __syncthreads();

    if (ntiles > 0) {
      // stage tile j into ring slot (fills + j) % NS: thread t moves one row, the K
      // row (t < 64) or the V row (t >= 64) of key t & 63, with one bulk
      // asynchronous copy whose bytes complete on the slot's mbarrier; keys
      // without a slot get a zero row
      auto issue = [&](int j) {
        if (j >= ntiles) return;
        const uint32_t fi = fills + (uint32_t)j;
        issued = fi + 1;
        uint8_t* st = mma_smem + (size_t)(fi % NS) * Sh::STAGE;
        const int t0 = kbeg + j * TK;
        const int nk = min(TK, kend - t0);
        const int kt = tid & (TK - 1);
        const bool isv = tid >= TK;
        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(st) + (isv ? TK * KP : 0) + kt * KP;
        int ci = -1;
        long long slot = -1;
        if (kt < nk) {
          const int kidx = t0 + kt;
          ci = kidx < nctx ? klo + kidx : ctx + (kidx - nctx);
          slot = slot_of(kv, b, ci);
        }
        if (!isv) sCi[(fi % NS) * TK + kt] = slot >= 0 ? ci : -1;
        const uint32_t bar = bar0 + 8u * (fi % NS);
        if (slot >= 0) {
          // the row was last touched by ordinary loads (the previous tile, the merge
          // buffer): order them before the copy engine's write
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          tc::mbar_expect_tx(bar, (uint32_t)(HD * 2));
          const __nv_bfloat16* src = reinterpret_cast<const __nv_bfloat16*>(isv ? kv.v : kv.k) + ((size_t)slot * nkv + g) * HD;
          asm volatile(
              "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
              ::"r"(smem_u32(dst)), "l"(src), "r"(HD * 2), "r"(bar), "l"(kv_policy)
              : "memory");
        } else {
          uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
          for (int c = 0; c < CH; ++c) d4[c] = make_uint4(0, 0, 0, 0);
          tc::mbar_arrive(bar);
        }
      };

      float acc[MT][NT][4];
      float mrun[MT][2], lrun[MT][2];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[mt][n][e] = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) { mrun[mt][h] = -INFINITY; lrun[mt][h] = 0.f; }
      }
      const uint32_t qbase = smem_u32(sQ);
      // per-row constants of this thread's rows (m-tile mt, half h: row mt*16 + grp + 8h)
      int rlo[MT][2];
      unsigned long long rmask[MT][2];
      bool rok[MT][2];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int qi = mt * 16 + grp + 8 * h;
          rok[mt][h] = qi < nQ;
          rlo[mt][h] = s_lo[qi];
          rmask[mt][h] = s_mask[qi];
        }

#pragma unroll
      for (int j = 0; j < NS - 1; ++j) issue(j);
      for (int j = 0; j < ntiles; ++j) {
        issue(j + NS - 1);
        const uint32_t fi = fills + (uint32_t)j;
        const bool ok = tc::mbar_wait(bar0 + 8u * (fi % NS), (fi / NS) & 1u, abort);
        if (__syncthreads_or(!ok)) { ok_all = false; cons = fi; break; }
        const uint8_t* st = mma_smem + (size_t)(fi % NS) * Sh::STAGE;
        const uint32_t kbase = smem_u32(st), vbase = kbase + TK * KP * 2;
        const int* ci_t = sCi + (fi % NS) * TK;
        // scores for this warp's 16 keys: S[mt][nt] (16 queries x 8 keys)
        float sc[MT][2][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) sc[mt][nt][e] = 0.f;
        const uint32_t krow = kbase + (uint32_t)((warp * 16 + 8 * (lane >> 4) + (lane & 7)) * KP +
                                                 8 * ((lane >> 3) & 1)) * 2;
        const uint32_t qrow = qbase + (uint32_t)((8 * ((lane >> 3) & 1) + (lane & 7)) * KP + 8 * (lane >> 4)) * 2;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          uint32_t b0, b1, b2, b3;   // keys 16w + {0..7, 8..15} x dims ks*16 + {0..7, 8..15}
          ldsm_x4(krow + (uint32_t)(ks * 16 * 2), b0, b1, b2, b3);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(qrow + (uint32_t)((mt * 16 * KP + ks * 16) * 2), a0, a1, a2, a3);
            mma_bf16(sc[mt][0], a0, a1, a2, a3, b0, b1);
            mma_bf16(sc[mt][1], a0, a1, a2, a3, b2, b3);
          }
        }
        // mask, scale to log2 units, warp-local online softmax
        int kci[4];                 // cache index of this thread's four keys (-1: no slot)
#pragma unroll
        for (int u = 0; u < 4; ++u) kci[u] = ci_t[warp * 16 + (u >> 1) * 8 + 2 * tig + (u & 1)];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (mt * 16 + 8 * h >= nQ) continue;     // rows of zero queries only (uniform in the warp)
            const bool qok = rok[mt][h];
            const int qlo = rlo[mt][h];
            const unsigned long long qmask = rmask[mt][h];
            float mx = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int ci = kci[2 * nt + e];
                bool ok = qok && ci >= 0;
                if (ok) ok = ci < ctx ? ci >= qlo : ((qmask >> (ci - ctx)) & 1ull) != 0;
                const float v = ok ? sc[mt][nt][2 * h + e] * scale_log2 : -INFINITY;
                sc[mt][nt][2 * h + e] = v;
                mx = fmaxf(mx, v);
              }
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float mnew = fmaxf(mrun[mt][h], mx);
            const float al = mnew == -INFINITY ? 1.f : exp2f(mrun[mt][h] - mnew);
            float ps = 0.f;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const float p = mnew == -INFINITY ? 0.f : exp2f(sc[mt][nt][2 * h + e] - mnew);
                sc[mt][nt][2 * h + e] = p;
                ps += p;
              }
            lrun[mt][h] = lrun[mt][h] * al + ps;
            mrun[mt][h] = mnew;
            if (al != 1.f) {
#pragma unroll
              for (int n = 0; n < NT; ++n) {
                acc[mt][n][2 * h] *= al;
                acc[mt][n][2 * h + 1] *= al;
              }
            }
          }
        }
        // P.V: A = P (queries x this warp's 16 keys), B = V^T via transposed ldmatrix
        uint32_t pa[MT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          pa[mt][0] = pack_bf16(sc[mt][0][0], sc[mt][0][1]);
          pa[mt][1] = pack_bf16(sc[mt][0][2], sc[mt][0][3]);
          pa[mt][2] = pack_bf16(sc[mt][1][0], sc[mt][1][1]);
          pa[mt][3] = pack_bf16(sc[mt][1][2], sc[mt][1][3]);
        }
        const uint32_t vrow = vbase + (uint32_t)((warp * 16 + 8 * ((lane >> 3) & 1) + (lane & 7)) * KP +
                                                 8 * (lane >> 4)) * 2;
#pragma unroll
        for (int n2 = 0; n2 < NT / 2; ++n2) {
          uint32_t v0, v1, v2, v3;   // keys 16w + {0..7, 8..15} x dims 16*n2 + {0..7, 8..15}
          ldsm_x4_t(vrow + (uint32_t)(n2 * 16 * 2), v0, v1, v2, v3);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            mma_bf16(acc[mt][2 * n2], pa[mt][0], pa[mt][1], pa[mt][2], pa[mt][3], v0, v1);
            mma_bf16(acc[mt][2 * n2 + 1], pa[mt][0], pa[mt][1], pa[mt][2], pa[mt][3], v2, v3);
          }
        }
        __syncthreads();     // this ring slot is refilled by the next iteration's copies
      }
      if (!ok_all) break;
      fills += (uint32_t)ntiles;
      __syncthreads();
      // merge the four warps: row sums over the quad, then max / rescale through shared memory
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float l = lrun[mt][h];
          l += __shfl_xor_sync(0xffffffffu, l, 1);
          l += __shfl_xor_sync(0xffffffffu, l, 2);
          if (tig == 0) {
            sMw[warp][mt * 16 + grp + 8 * h] = mrun[mt][h];
            sLw[warp][mt * 16 + grp + 8 * h] = l;
          }
        }
      constexpr int RS = HD + 8;      // padded row of the merge buffer (fewer bank conflicts)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int h = 0; h < 2; ++h)
          if (rok[mt][h]) {
            const int row = mt * 16 + grp + 8 * h;
#pragma unroll
            for (int n = 0; n < NT; ++n)
              *reinterpret_cast<float2*>(red + ((size_t)warp * QM + row) * RS + n * 8 + 2 * tig) =
                  make_float2(acc[mt][n][2 * h], acc[mt][n][2 * h + 1]);
          }
      __syncthreads();
      for (int e = tid; e < nQ * HD; e += blockDim.x) {
        const int qi = e / HD, d = e % HD;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) M = fmaxf(M, sMw[w][qi]);
        float o = 0.f, L = 0.f;
        if (M > -INFINITY) {
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const float f = exp2f(sMw[w][qi] - M);
            o += red[((size_t)w * QM + qi) * RS + d] * f;
            L += sLw[w][qi] * f;
          }
        }
        const int q = q0 + qi;
        const int m = b * ri.R + q / G, h = g * G + q % G;
        const size_t base = ((size_t)m * nq + h) * nsplit + s;
        opart[base * HD + d] = o;
        // the combine kernel takes natural-log maxima of the scaled scores
        if (d == 0) mlpart[base] = make_float2(M == -INFINITY ? -INFINITY : M * 0.69314718055994531f, L);
      }
    }
    __syncthreads();     // red / sQ / sMw reused by the next item
    if (work != nullptr) {
      if (tid == 0) s_next = (int)gridDim.x + atomicAdd(work, 1);
      __syncthreads();
      item = s_next;
    } else {
      item += gridDim.x;
    }
  }
  if (!ok_all) {
    // let the copies still in flight land before the CTA's shared memory goes away
    for (uint32_t f = cons; f < issued; ++f) tc::mbar_wait(bar0 + 8u * (f % NS), (f / NS) & 1u, abort, false);
    if (tid == 0) report(ws, SPEC_ERR_TIMEOUT, blockIdx.x, 0);
  }
}

// ---------------------------------------------------------------- warp-specialised attention (bf16, TMA)
// The same work items and partial results as attn_mma_kernel (up to 16 queries
// of one request and kv head, one split of its keys), for caches whose block
// size is a multiple of 8.  A split's keys are the cache indices [klo, ctx+nd)
// cut into 64-key tiles aligned to multiples of 64; warp 4 produces, warps 0-3
// consume:
//  * the producer claims items, reads each tile's block-table entries and loads
//    K and V by 3-D tensor copies (head dim x kv head x slot; one box is one
//    8- or 16-slot run of a cache block and one 64-column half of the head, 128-B
//    swizzled) and, with an item's first tile, its query rows, all completing on
//    the ring slot's "full" barrier; runs without a valid key are not loaded;
//  * consumer warp w owns keys 16w .. 16w+15 of every tile (scores and P.V as
//    m16n8k16 bf16 MMAs with an online softmax, as in attn_mma_kernel), skips a
//    tile none of whose keys is valid, zeroes the V rows of its invalid keys
//    when some are valid (masked keys then add exact zeros), and releases the
//    slot with one arrive per warp on its "empty" barrier;
//  * after an item's last tile the four warps merge through that tile's slot.
// No CTA-wide barrier runs per tile or per item; every wait is bounded.
// What it computes is the draft layer's attention of the file header ([NEURON]
// "Eagle3 Draft Model Architecture"; slots from the block table as in "KV Cache
// Sharing"; the window of [EAGLE4] Eagle4Config.sliding_window): per query,
// softmax(q . k / sqrt(hd)) over the allowed keys, times V.
struct AttnTileMeta {
  int b, g, q0, nQ, s, ctx, ci0, flags;
  unsigned long long valid;         // bit k: key ci0 + k is attended to by some query row
};
constexpr int kTileFirst = 1, kTileLast = 2, kTileEnd = 4, kTileQBuf = 8;

// MT query m-tiles of 16 per item: the four consumer warps split an item's 64
// keys into 4 / MT blocks of 16 * MT keys; warp w serves m-tile w / (4 / MT)
// with key block w % (4 / MT), so every K / V row is read from shared memory
// once per m-tile and the merge combines the 4 / MT warps of an m-tile.
template <int HD, int MT = 1> struct WsShape {
  static constexpr int TK = 64, QM = 16 * MT, NS = 2, NH = HD / 64, KP = HD + 8;
  static constexpr int HALF = TK * 128;                  // 64 keys x one 64-column half, 128-B rows
  static constexpr int KVB = NH * HALF;                  // a K (or V) tile
  static constexpr int STG = 2 * KVB;
  static constexpr size_t kQ = (size_t)NS * STG;                      // [2][QM][KP] bf16 queries
  static constexpr size_t kMeta = kQ + (size_t)2 * QM * KP * 2;      // [NS] AttnTileMeta
  static constexpr size_t kLo = kMeta + (size_t)NS * 64;             // [2][QM] int
  static constexpr size_t kMask = kLo + (size_t)2 * QM * 4;          // [2][QM] u64
  static constexpr size_t kMw = kMask + (size_t)2 * QM * 8;          // [4][QM] float, then [4][QM] float
  static constexpr size_t kBar = kMw + (size_t)2 * 4 * QM * 4;       // full[NS], empty[NS], merge
  static constexpr size_t kMisc = kBar + (size_t)(2 * NS + 1) * 8;   // abort, consumed[4], issued
  static constexpr size_t kBytes = kMisc + 32;
  static constexpr size_t kSmem = kBytes + 1024;                     // + alignment of the ring to 1024 B
  static_assert((size_t)4 * 16 * HD * 4 <= (size_t)STG, "the merge reuses one ring slot");
  static_assert(MT == 1 || MT == 2, "one or two m-tiles");
};

SPEC_DEV void tma_load_3d(uint32_t dst, const CUtensorMap* tm, uint32_t bar, int x, int y, int z, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(pol)
      : "memory");
}

template <int HD, int MT>
__global__ void __launch_bounds__(160, MT == 1 ? 3 : 2) attn_ws_kernel(const __grid_constant__ CUtensorMap tmk,
                                                         const __grid_constant__ CUtensorMap tmv,
                                                         const __nv_bfloat16* __restrict__ qbuf, spec_kv kv,
                                                         RowInfo ri, int nq, int nkv, int window, int nsplit,
                                                         int nqg, int n_items, int bh, float scale_log2,
                                                         float* __restrict__ opart, float2* __restrict__ mlpart,
                                                         int* __restrict__ work, void* ws) {
  SPEC_TL(spec::kTLAttnWs);
  using S = WsShape<HD, MT>;
  constexpr int TK = S::TK, QM = S::QM, NS = S::NS, NH = S::NH, KP = S::KP, NT = HD / 8, KS = HD / 16;
  constexpr int WPM = 4 / MT, KPW = TK / WPM;   // warps per m-tile, keys per warp
  extern __shared__ __align__(1024) uint8_t wsm_raw[];
  uint8_t* sm = wsm_raw + ((1024u - (smem_u32(wsm_raw) & 1023u)) & 1023u);
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(sm + S::kQ);
  AttnTileMeta* meta = reinterpret_cast<AttnTileMeta*>(sm + S::kMeta);
  int* s_lo = reinterpret_cast<int*>(sm + S::kLo);
  unsigned long long* s_mask = reinterpret_cast<unsigned long long*>(sm + S::kMask);
  float* sMw = reinterpret_cast<float*>(sm + S::kMw);
  float* sLw = sMw + 4 * QM;
  const uint32_t full0 = smem_u32(sm + S::kBar), empty0 = full0 + 8u * NS, mbar = full0 + 16u * NS;
  int* misc = reinterpret_cast<int*>(sm + S::kMisc);
  volatile int* abort = misc;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = nq / nkv;
  const int nQall = ri.R * G;
  if (tid == 0) {
    misc[0] = 0;
    for (int i = 0; i < NS; ++i) {
      tc::mbar_init(full0 + 8u * i, 1);      // the producer's arrive (+ the copies' bytes)
      tc::mbar_init(empty0 + 8u * i, 4);     // one arrive per consumer warp
    }
    tc::mbar_init(mbar, 4);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
    }
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    uint32_t fill = 0;
    int qbuf_sel = 0;
    int it = blockIdx.x;
    bool ok = true;
    const int ng = TK / bh;                    // block-table runs per tile
    // An item's keys and the block-table entries of its tiles.  Context lengths,
    // row positions and masks and the block table are inputs of the call that no
    // kernel of it writes, and this kernel starts only once every block of the
    // launch before it has passed its own dependency wait, i.e. once all earlier
    // launches (this call's prologue and QKV GEMM among them) have finished: so
    // the first item is described before the wait, reading through L2.
    struct Item {
      int s, g, b, q0, nQ, ctx, lo, klo, kend, cb, t0, ntiles;
      unsigned long long mk;
    };
    auto describe = [&](int i) {
      Item d;
      d.s = i % nsplit;
      d.g = (i / nsplit) % nkv;
      const int bq = i / (nsplit * nkv);
      d.b = bq / nqg;
      d.q0 = (bq % nqg) * QM;
      d.nQ = min(QM, nQall - d.q0);
      d.ctx = __ldcg(ri.ctx_len + d.b);
      d.lo = 0x7fffffff;
      d.mk = 0;
      if (lane < d.nQ) {
        const int m = d.b * ri.R + (d.q0 + lane) / G;
        const int pos = ri.pos ? __ldcg(ri.pos + m) : d.ctx + ri.step;
        d.lo = window > 0 ? max(0, pos - window + 1) : 0;
        if (d.lo > d.ctx) d.lo = d.ctx;
        d.mk = ri.mask ? __ldcg(reinterpret_cast<const unsigned long long*>(ri.mask) + m) : row_mask(ri, m);
      }
      int klo = d.lo;
      unsigned long long om = d.mk;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        klo = min(klo, __shfl_xor_sync(0xffffffffu, klo, o));
        om |= __shfl_xor_sync(0xffffffffu, om, o);
      }
      d.klo = klo;
      d.kend = d.ctx + (om ? 64 - __clzll((long long)om) : 0);   // keys: cache indices [klo, kend)
      d.cb = klo & ~(TK - 1);
      const int T = d.kend > klo ? (d.kend - d.cb + TK - 1) / TK : 0;
      const int ct = (T + nsplit - 1) / nsplit;
      d.t0 = d.s * ct;
      d.ntiles = max(0, min(T, d.t0 + ct) - d.t0);
      return d;
    };
    auto table_entry = [&](const Item& d, int j) {   // lane r < ng: block-table entry of run r of tile j
      int ent = -1;
      if (lane < ng) {
        const int ci = d.cb + (d.t0 + j) * TK + lane * bh;
        const int blk = ci / kv.block_size;
        if (ci < d.kend && blk < kv.max_blocks) ent = __ldcg(kv.block_table + (size_t)d.b * kv.max_blocks + blk);
      }
      return ent;
    };
    Item cur = describe(it);
    int ent0 = table_entry(cur, 0);
    pdl_wait();
    pdl_trigger();
    while (ok && it < n_items) {
      int nxt = it;
      if (lane == 0) nxt = work != nullptr ? (int)gridDim.x + atomicAdd(work, 1) : it + (int)gridDim.x;
      const int s = cur.s, g = cur.g, b = cur.b, q0 = cur.q0, nQ = cur.nQ, ctx = cur.ctx, lo = cur.lo;
      const unsigned long long mk = cur.mk;
      const int klo = cur.klo, kend = cur.kend, cb = cur.cb, t0 = cur.t0, ntiles = cur.ntiles;
      if (ntiles == 0) {
        // an empty split: its partials say "no keys"
        for (int e = lane; e < nQ * HD; e += 32) {
          const int qi = e / HD, d = e % HD;
          const int q = q0 + qi;
          const size_t base = ((size_t)(b * ri.R + q / G) * nq + g * G + q % G) * nsplit + s;
          opart[base * HD + d] = 0.f;
          if (d == 0) mlpart[base] = make_float2(-INFINITY, 0.f);
        }
      } else {
        // the item's row constants and queries go to buffer qbuf_sel: its previous
        // user finished at least two fills ago (every item has a tile), and the wait
        // for this item's first slot covers those
        for (int j = 0; j < ntiles; ++j) {
          const int slot = (int)(fill % NS);
          const int ci0 = cb + (t0 + j) * TK;
          const int ent = j == 0 ? ent0 : table_entry(cur, j);
          if (fill >= (uint32_t)NS) {
            const bool w = tc::mbar_wait(empty0 + 8u * slot, ((fill / NS) - 1u) & 1u, abort);
            if (__any_sync(0xffffffffu, !w)) { ok = false; break; }
          }
          unsigned long long valid = 0;
#pragma unroll
          for (int hk = 0; hk < 2; ++hk) {
            const int kt = lane + 32 * hk;
            const int ci = ci0 + kt;
            const int e = __shfl_sync(0xffffffffu, ent, kt / bh);
            bool v = ci >= klo && ci < kend && e >= 0;
            if (v) v = (long long)e * kv.block_size + ci % kv.block_size < (long long)kv.num_slots;
            valid |= (unsigned long long)__ballot_sync(0xffffffffu, v) << (32 * hk);
          }
          // lane -> one box: run r = lane / (2 NH), K or V, column half
          const int r = lane / (2 * NH), isv = (lane / NH) & 1, hh = lane % NH;
          const unsigned long long rmask = bh == 16 ? 0xffffull : 0xffull;
          const int er = __shfl_sync(0xffffffffu, ent, r < ng ? r : 0);
          const bool box = r < ng && ((valid >> (r * bh)) & rmask) != 0;
          const uint32_t nbox = __popc(__ballot_sync(0xffffffffu, box));
          uint32_t bytes = nbox * (uint32_t)(bh * 128);
          if (j == 0) bytes += (uint32_t)(nQ * HD * 2);
          if (j == 0 && lane < QM) {
            s_lo[qbuf_sel * QM + lane] = lo;
            s_mask[qbuf_sel * QM + lane] = mk;
          }
          if (lane == 0) {
            AttnTileMeta mt;
            mt.b = b; mt.g = g; mt.q0 = q0; mt.nQ = nQ; mt.s = s; mt.ctx = ctx; mt.ci0 = ci0;
            mt.flags = (j == 0 ? kTileFirst : 0) | (j == ntiles - 1 ? kTileLast : 0) | (qbuf_sel ? kTileQBuf : 0);
            mt.valid = valid;
            meta[slot] = mt;
          }
          __syncwarp();
          if (lane == 0) tc::mbar_expect_tx(full0 + 8u * slot, bytes);
          __syncwarp();
          const uint32_t bar = full0 + 8u * slot;
          if (box) {
            const int ci = ci0 + r * bh;
            const int slot0 = er * kv.block_size + ci % kv.block_size;
            const uint32_t dst = smem_u32(sm + (size_t)slot * S::STG + (size_t)isv * S::KVB + (size_t)hh * S::HALF +
                                          (size_t)r * bh * 128);
            tma_load_3d(dst, isv ? &tmv : &tmk, bar, hh * 64, g, slot0, pol);
          }
          if (j == 0 && lane < nQ) {
            const int q = q0 + lane;
            const __nv_bfloat16* src = qbuf + ((size_t)(b * ri.R + q / G) * nq + g * G + q % G) * HD;
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                ::"r"(smem_u32(sQ + ((size_t)qbuf_sel * QM + lane) * KP)), "l"(src), "r"(HD * 2), "r"(bar)
                : "memory");
          }
          ++fill;
        }
        qbuf_sel ^= 1;
      }
      it = __shfl_sync(0xffffffffu, nxt, 0);
      if (it < n_items) {
        cur = describe(it);
        ent0 = table_entry(cur, 0);
      }
    }
    // end of the sequence: one more slot, without copies
    if (ok) {
      const int slot = (int)(fill % NS);
      bool w = true;
      if (fill >= (uint32_t)NS) w = tc::mbar_wait(empty0 + 8u * slot, ((fill / NS) - 1u) & 1u, abort);
      if (!__any_sync(0xffffffffu, !w) && lane == 0) {
        meta[slot].flags = kTileEnd;
        tc::mbar_arrive(full0 + 8u * slot);
      }
    }
    if (lane == 0) misc[5] = (int)fill;
  } else {
    // ------------------------------------------------------------ consumers
    pdl_wait();
    pdl_trigger();
    const int grp = lane >> 2, tig = lane & 3;
    const int mtile = MT == 1 ? 0 : warp / WPM, kbase = (warp % WPM) * KPW;   // this warp's m-tile and keys
    uint32_t fill = 0, mph = 0;
    float acc[NT][4];
    float mrun[2], lrun[2];
    int rlo[2], nQ = 0, qsel = 0, lo_max = 0;   // lo_max: the latest window start of the warp's rows
    unsigned long long rmask[2];
    bool rok[2];
    // this lane's ldmatrix rows (relative to the warp's first key): K (scores' "col"
    // operand) and V (transposed)
    const int key_k = 8 * (lane >> 4) + (lane & 7), sel_k = (lane >> 3) & 1;
    const int key_v = 8 * ((lane >> 3) & 1) + (lane & 7), sel_v = lane >> 4;
    const uint32_t x7 = (uint32_t)(lane & 7);
    constexpr uint32_t kFull = KPW == 32 ? 0xffffffffu : ((1u << KPW) - 1u);
    for (;; ++fill) {
      const int slot = (int)(fill % NS);
      if (!tc::mbar_wait(full0 + 8u * slot, (fill / NS) & 1u, abort)) break;
      const AttnTileMeta mt = meta[slot];
      if (mt.flags & kTileEnd) break;
      if (mt.flags & kTileFirst) {
        nQ = mt.nQ;
        qsel = (mt.flags & kTileQBuf) ? 1 : 0;
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[n][e] = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          mrun[h] = -INFINITY;
          lrun[h] = 0.f;
          const int qi = 16 * mtile + grp + 8 * h;
          rok[h] = qi < nQ;
          rlo[h] = s_lo[qsel * QM + qi];
          rmask[h] = s_mask[qsel * QM + qi];
        }
        lo_max = max(rok[0] ? rlo[0] : 0, rok[1] ? rlo[1] : 0);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lo_max = max(lo_max, __shfl_xor_sync(0xffffffffu, lo_max, o));
      }
      uint8_t* st = sm + (size_t)slot * S::STG;
      const uint32_t vm = (uint32_t)(mt.valid >> kbase) & kFull;
      bool wrote = false;
      if (vm != 0 && 16 * mtile < nQ) {
        if (vm != kFull) {
          // V rows of this warp's invalid keys: zeros (stale or unloaded rows may hold
          // anything); a warp of the other m-tile may write the same zeros
          for (int e = lane; e < KPW * NH * 8; e += 32) {
            const int kr = e / (NH * 8), c = e % (NH * 8);
            if (!((vm >> kr) & 1u)) {
              const int key = kbase + kr;
              *reinterpret_cast<uint4*>(st + S::KVB + (size_t)(c >> 3) * S::HALF + (size_t)key * 128 + (c & 7) * 16) =
                  make_uint4(0, 0, 0, 0);
            }
          }
          wrote = true;
          __syncwarp();
        }
        const uint32_t kst = smem_u32(st), vst = kst + S::KVB;
        const uint32_t qb = smem_u32(sQ + (size_t)qsel * QM * KP + (size_t)mtile * 16 * KP);
        const uint32_t qrow = qb + (uint32_t)((8 * ((lane >> 3) & 1) + (lane & 7)) * KP + 8 * (lane >> 4)) * 2;
        float sc[2 * MT][4];
#pragma unroll
        for (int nt = 0; nt < 2 * MT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) sc[nt][e] = 0.f;
        const uint32_t krow = kst + (uint32_t)((kbase + key_k) * 128);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          const uint32_t c = (uint32_t)(((ks & 3) << 1) | sel_k);
          uint32_t b[MT][4];         // keys kbase + 16j + {0..7, 8..15} x dims ks*16 + {0..7, 8..15}
#pragma unroll
          for (int j = 0; j < MT; ++j)
            ldsm_x4(krow + (uint32_t)((ks >> 2) * S::HALF + 16 * j * 128) + ((c ^ x7) << 4), b[j][0], b[j][1],
                    b[j][2], b[j][3]);
          uint32_t a0, a1, a2, a3;
          ldsm_x4(qrow + (uint32_t)(ks * 16 * 2), a0, a1, a2, a3);
#pragma unroll
          for (int j = 0; j < MT; ++j) {
            mma_bf16(sc[2 * j], a0, a1, a2, a3, b[j][0], b[j][1]);
            mma_bf16(sc[2 * j + 1], a0, a1, a2, a3, b[j][2], b[j][3]);
          }
        }
        // mask, scale to log2 units, warp-local online softmax; a tile of valid context
        // keys at or past every row's window start needs no per-key test
        const bool open = vm == kFull && mt.ci0 + TK <= mt.ctx && mt.ci0 >= lo_max;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (16 * mtile + 8 * h >= nQ) continue;     // rows of absent queries only (uniform in the warp)
          float mx = -INFINITY;
#pragma unroll
          for (int nt = 0; nt < 2 * MT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int kr = nt * 8 + 2 * tig + e;
              const int ci = mt.ci0 + kbase + kr;
              bool ok = rok[h];
              if (!open) {
                ok = ok && ((vm >> kr) & 1u);
                if (ok) ok = ci < mt.ctx ? ci >= rlo[h] : ((rmask[h] >> (ci - mt.ctx)) & 1ull) != 0;
              }
              const float v = ok ? sc[nt][2 * h + e] * scale_log2 : -INFINITY;
              sc[nt][2 * h + e] = v;
              mx = fmaxf(mx, v);
            }
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
          const float mnew = fmaxf(mrun[h], mx);
          const float al = mnew == -INFINITY ? 1.f : exp2f(mrun[h] - mnew);
          float ps = 0.f;
#pragma unroll
          for (int nt = 0; nt < 2 * MT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float p = mnew == -INFINITY ? 0.f : exp2f(sc[nt][2 * h + e] - mnew);
              sc[nt][2 * h + e] = p;
              ps += p;
            }
          lrun[h] = lrun[h] * al + ps;
          mrun[h] = mnew;
          if (al != 1.f) {
#pragma unroll
            for (int n = 0; n < NT; ++n) {
              acc[n][2 * h] *= al;
              acc[n][2 * h + 1] *= al;
            }
          }
        }
        const uint32_t vrow = vst + (uint32_t)((kbase + key_v) * 128);
#pragma unroll
        for (int j = 0; j < MT; ++j) {
          // P of keys kbase + 16j .. + 15 as the A operand (bf16)
          const uint32_t pa0 = pack_bf16(sc[2 * j][0], sc[2 * j][1]), pa1 = pack_bf16(sc[2 * j][2], sc[2 * j][3]);
          const uint32_t pa2 = pack_bf16(sc[2 * j + 1][0], sc[2 * j + 1][1]);
          const uint32_t pa3 = pack_bf16(sc[2 * j + 1][2], sc[2 * j + 1][3]);
#pragma unroll
          for (int n2 = 0; n2 < NT / 2; ++n2) {
            uint32_t v0, v1, v2, v3;   // keys kbase + 16j + {0..7, 8..15} x dims 16*n2 + {0..7, 8..15}
            const uint32_t c = (uint32_t)(((n2 & 3) << 1) | sel_v);
            ldsm_x4_t(vrow + (uint32_t)((n2 >> 2) * S::HALF + 16 * j * 128) + ((c ^ x7) << 4), v0, v1, v2, v3);
            mma_bf16(acc[2 * n2], pa0, pa1, pa2, pa3, v0, v1);
            mma_bf16(acc[2 * n2 + 1], pa0, pa1, pa2, pa3, v2, v3);
          }
        }
      }
      if (mt.flags & kTileLast) {
        // merge the warps of each m-tile through this slot (every warp is done with its K and V)
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(mbar);
        bool okm = tc::mbar_wait(mbar, mph, abort);
        mph ^= 1u;
        if (!okm) break;
        float* red = reinterpret_cast<float*>(st);     // [4 warps][16][HD], 8-float blocks swizzled by row
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float l = lrun[h];
          l += __shfl_xor_sync(0xffffffffu, l, 1);
          l += __shfl_xor_sync(0xffffffffu, l, 2);
          const int row = grp + 8 * h;
          if (tig == 0) {
            sMw[warp * 16 + row] = mrun[h];
            sLw[warp * 16 + row] = l;
          }
          if (rok[h]) {
#pragma unroll
            for (int n = 0; n < NT; ++n)
              *reinterpret_cast<float2*>(red + ((size_t)warp * 16 + row) * HD + ((n ^ (row & 7)) << 3) + 2 * tig) =
                  make_float2(acc[n][2 * h], acc[n][2 * h + 1]);
          }
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(mbar);
        okm = tc::mbar_wait(mbar, mph, abort);
        mph ^= 1u;
        if (!okm) break;
        // thread -> one query row (TPR threads a row) and every TPR-th 4-float chunk of
        // it: the row's weights once, then independent 16-byte loads and stores
        constexpr int TPR = 128 / QM, NCH = HD / 4 / TPR;
        const int qi = tid / TPR, cq = tid % TPR;
        if (qi < nQ) {
          const int r = qi & 15, w0 = (qi >> 4) * WPM;
          float mw[WPM], f[WPM];
          float M = -INFINITY, L = 0.f;
#pragma unroll
          for (int w = 0; w < WPM; ++w) {
            mw[w] = sMw[(w0 + w) * 16 + r];
            M = fmaxf(M, mw[w]);
          }
#pragma unroll
          for (int w = 0; w < WPM; ++w) {
            f[w] = M == -INFINITY ? 0.f : exp2f(mw[w] - M);
            L += sLw[(w0 + w) * 16 + r] * f[w];
          }
          const int q = mt.q0 + qi;
          const size_t base = ((size_t)(mt.b * ri.R + q / G) * nq + mt.g * G + q % G) * nsplit + mt.s;
          float4* dst = reinterpret_cast<float4*>(opart + base * HD);
#pragma unroll
          for (int k = 0; k < NCH; ++k) {
            const int c = k * TPR + cq;                                   // dims 4c .. 4c + 3
            const int col = (((c >> 1) ^ (r & 7)) << 3) + ((c & 1) << 2);
            float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w = 0; w < WPM; ++w) {
              const float4 v = *reinterpret_cast<const float4*>(red + ((size_t)(w0 + w) * 16 + r) * HD + col);
              o.x += v.x * f[w];
              o.y += v.y * f[w];
              o.z += v.z * f[w];
              o.w += v.w * f[w];
            }
            dst[c] = o;
          }
          // the combine kernel takes natural-log maxima of the scaled scores
          if (cq == 0) mlpart[base] = make_float2(M == -INFINITY ? -INFINITY : M * 0.69314718055994531f, L);
        }
        wrote = true;
      }
      // generic writes to the slot come before the copy engine's next fill of it
      if (wrote) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(empty0 + 8u * slot);
    }
    if (lane == 0) misc[1 + warp] = (int)fill;
  }
  __syncthreads();
  if (*abort) {
    // let the copies still in flight land before the CTA's shared memory goes away
    if (tid == 0) {
      int c = misc[1];
      for (int w = 2; w <= 4; ++w) c = min(c, misc[w]);
      for (uint32_t f = (uint32_t)c; f < (uint32_t)misc[5]; ++f)
        tc::mbar_wait(full0 + 8u * (f % NS), (f / NS) & 1u, abort, false);
      report(ws, SPEC_ERR_TIMEOUT, blockIdx.x, 0);
    }
  }
}

template <typename T, int HD, int NSM>
__global__ void __launch_bounds__(HD) attn_combine_kernel(const float* __restrict__ opart,
                                                          const float2* __restrict__ mlpart, int nq, int nsplit,
                                                          T* __restrict__ out) {
  SPEC_TL(spec::kTLCombine);
  pdl_wait();
  pdl_trigger();
  const int mh = blockIdx.x;          // m * nq + h
  const int d = threadIdx.x;
  // every split's value of this dimension (nsplit <= NSM <= 64) is loaded together
  // with the splits' (max, sum) pairs, which go to shared memory (nsplit <= 64 <= HD)
  // with the splits' weights; the weighted sum then takes the splits in order
  const float* op = opart + (size_t)mh * nsplit * HD + d;
  float v[NSM];
#pragma unroll
  for (int u = 0; u < NSM; ++u) v[u] = u < nsplit ? op[(size_t)u * HD] : 0.f;
  __shared__ float sm_[64], sl_[64], sw[64];
  if (d < nsplit) {
    const float2 ml = mlpart[(size_t)mh * nsplit + d];
    sm_[d] = ml.x;
    sl_[d] = ml.y;
  }
  __syncthreads();
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, sm_[s]);
  if (d < nsplit) sw[d] = (M > -INFINITY && sm_[d] > -INFINITY) ? expf(sm_[d] - M) : 0.f;
  __syncthreads();
  float L = 0.f;
  for (int s = 0; s < nsplit; ++s) L += sl_[s] * sw[s];
  float o4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int u = 0; u < NSM; ++u)
    if (u < nsplit) o4[u & 3] += v[u] * sw[u];
  const float o = (o4[0] + o4[1]) + (o4[2] + o4[3]);
  st(out + (size_t)mh * HD + d, L > 0.f ? o / L : 0.f);
}

// The combine with a register batch sized to the split count (16, 32 or 64).
template <typename T, int HD>
static void launch_combine(const float* opart, const float2* mlpart, int M, int nq, int nsplit, void* out,
                           cudaStream_t st) {
  const dim3 grid(M * nq), block(HD);
  if (nsplit <= 16)
    launch_pdl(attn_combine_kernel<T, HD, 16>, grid, block, 0, st, opart, mlpart, nq, nsplit, (T*)out);
  else if (nsplit <= 32)
    launch_pdl(attn_combine_kernel<T, HD, 32>, grid, block, 0, st, opart, mlpart, nq, nsplit, (T*)out);
  else
    launch_pdl(attn_combine_kernel<T, HD, 64>, grid, block, 0, st, opart, mlpart, nq, nsplit, (T*)out);
}

// ---------------------------------------------------------------- row statistics
// From full fp32 logits [M, V]: lse and the k largest (ties to smaller id).
__global__ void __launch_bounds__(256) row_stats_kernel(const float* __restrict__ logits, int V, int k,
                                                        int32_t* __restrict__ ids, int ld_ids, float* __restrict__ lp,
                                                        float* __restrict__ lse_out, const int32_t* __restrict__ d2t) {
  SPEC_TL(spec::kTLRowStats);
  pdl_wait();
  pdl_trigger();
  __shared__ float red[32];
  __shared__ int redi[32];
  __shared__ int chosen[8];
  const int m = blockIdx.x;
  const float* x = logits + (size_t)m * V;
  float mx = -INFINITY;
  for (int v = threadIdx.x; v < V; v += blockDim.x) mx = fmaxf(mx, x[v]);
  mx = block_max(mx, red);
  float s = 0.f;
  for (int v = threadIdx.x; v < V; v += blockDim.x) s += expf(x[v] - mx);
  s = block_sum(s, red);
  const float lse = mx + logf(s);
  for (int r = 0; r < k; ++r) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int v = threadIdx.x; v < V; v += blockDim.x) {
      bool used = false;
      for (int q = 0; q < r; ++q) used |= (chosen[q] == v);
      if (!used && better(x[v], v, bv, bi)) { bv = x[v]; bi = v; }
    }
    block_argmax(bv, bi, red, redi);
    if (threadIdx.x == 0) {
      chosen[r] = bi;
      ids[(size_t)m * ld_ids + r] = d2t ? d2t[bi] : bi;
      lp[(size_t)m * ld_ids + r] = bv - lse;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0 && lse_out) lse_out[m] = lse;
}

// ---------------------------------------------------------------- top-K selection
SPEC_DEV uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The Kc largest of each row of s [M, V] (ties to the smaller id), in
// descending order.  A cluster of kTkCL CTAs (1024 threads each) per row, on
// order-preserving 32-bit keys; CTA r owns a contiguous part of the row:
//  1. every thread takes the largest key among its elements; the Kc-th largest
//     of its CTA's 1024 maxima is a lower bound of the row's Kc-th largest key
//     (the Kc largest maxima are Kc distinct elements at least that large), and
//     so is the lower edge of its 16-bit bucket and the largest of the cluster's
//     bounds, T0 (exchanged in distributed shared memory);
//  2. a second pass copies the CTA's elements >= T0 -- a few hundred in the
//     whole row -- to its shared memory;
//  3. rank 0 gathers the copies, one per thread, and each copy's rank among them
//     (larger key first, then smaller id) is its place in the output.  With more
//     copies than threads an exact radix selection gives the Kc-th key and how
//     many elements equal to it are taken (smallest ids first), and a bitonic
//     sort orders the Kc selected.
// Both passes over the row are plain streaming reads (16-byte loads, one
// shared-counter update per warp and round).  If more elements pass step 2
// than shared memory takes (long runs of equal values), rank 0 selects with
// radix passes over the whole row, ties collected in id order.
constexpr int kTkCL = 2;            // one wave at 64 rows: 128 CTAs of 1024 threads
constexpr int kTkCap = 6144;          // copies rank 0 gathers
constexpr int kTkCapCta = 2048;       // copies one CTA keeps

size_t topk_select_smem() { return (size_t)kTkCap * 8 + (size_t)kTkCapCta * 8 + 1024 * 8 + 256 * 4; }

SPEC_DEV int block_excl_scan(int v, int* wsum, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) wsum[w] = x;
  __syncthreads();
  if (w == 0) {
    int t = lane < nw ? wsum[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < nw) wsum[lane] = t;     // inclusive prefix of the warp totals
    if (lane == 31) *total = t;
  }
  __syncthreads();
  return x - v + (w > 0 ? wsum[w - 1] : 0);
}

// radix select over n keys (shared memory, or the float row x): the key of the
// need-th largest, digit by digit (8 bits) from the top, and in *tie_need how
// many elements equal to it belong to the need largest.  Lanes of a warp that
// fall in the same digit add to the histogram once; warp 0 finds the digit.
// With fewer than four rounds the result is the lower edge of the need-th
// largest key's bucket (its top 8 * rounds bits): at least `need` keys are >= it.
template <bool SMEM_KEYS>
SPEC_DEV uint32_t radix_select(const float* x, const uint32_t* keys, int n, int need, int* hist, uint32_t* s_prefix,
                               int* s_need, int* tie_need, int rounds = 4) {
  const int tid = threadIdx.x, lane = tid & 31;
  if (tid == 0) { *s_prefix = 0u; *s_need = need; }
  for (int lo = 24; lo >= 32 - 8 * rounds; lo -= 8) {
    if (tid < 256) hist[tid] = 0;
    __syncthreads();
    const uint32_t pf = *s_prefix;
    const uint32_t pmask = lo == 24 ? 0u : (0xffffffffu << (lo + 8));
    for (int base = 0; base < n; base += blockDim.x) {
      const int i = base + tid;
      uint32_t k = 0;
      bool ok = i < n;
      if (ok) {
        k = SMEM_KEYS ? keys[i] : order_key(x[i]);
        ok = (k & pmask) == (pf & pmask);
      }
      const unsigned act = __ballot_sync(0xffffffffu, ok);
      if (ok) {
        const uint32_t dg = (k >> lo) & 0xffu;
        const unsigned peers = __match_any_sync(act, dg);
        if (lane == __ffs(peers) - 1) atomicAdd(&hist[dg], __popc(peers));
      }
    }
    __syncthreads();
    if (tid < 32) {
      // lane l owns digits 255-8l .. 248-8l; count above the lane's digits =
      // prefix over the lanes before it
      const int nn = *s_need;
      int hv[8], c = 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        hv[u] = hist[255 - 8 * lane - u];
        c += hv[u];
      }
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int before = incl - c;
      if (before < nn && incl >= nn) {
        int acc = before, dsel = 0;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (acc + hv[u] >= nn) { dsel = 255 - 8 * lane - u; break; }
          acc += hv[u];
        }
        *s_need = nn - acc;
        *s_prefix = pf | ((uint32_t)dsel << lo);
      }
    }
    __syncthreads();
  }
  *tie_need = *s_need;
  return *s_prefix;
}

// Bitonic sort of the Kc selected (key descending, index ascending) and store.
SPEC_DEV void sort_selected(uint32_t* skey, int* sidx, int Kc, int32_t* out) {
  const int tid = threadIdx.x;
  int n2 = 1;
  while (n2 < Kc) n2 <<= 1;
  if (tid >= Kc && tid < n2) { skey[tid] = 0; sidx[tid] = 0x7fffffff; }
  __syncthreads();
  for (int size = 2; size <= n2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (tid < n2) {
        const int o = tid ^ stride;
        if (o > tid) {
          const bool up = (tid & size) == 0;   // first half: descending order
          const uint32_t ka = skey[tid], kb = skey[o];
          const int ia = sidx[tid], ib = sidx[o];
          const bool a_first = ka > kb || (ka == kb && ia < ib);
          if (up != a_first) {
            skey[tid] = kb; skey[o] = ka;
            sidx[tid] = ib; sidx[o] = ia;
          }
        }
      }
      __syncthreads();
    }
  }
  if (tid < Kc) out[tid] = sidx[tid];
}

// The Kc largest of a float row x[0..V) (ties to the smaller id) into skey / sidx
// (unordered; *s_nsel counts them): radix selection of the Kc-th key over the
// row, then an ordered pass that takes every larger element and the ties in id
// order.  Block-wide; skey / sidx hold at least Kc entries; *s_nsel starts at 0.
SPEC_DEV void select_row_exact(const float* x, int V, int Kc, uint32_t* skey, int* sidx, int* hist, int* wsum,
                               uint32_t* s_prefix, int* s_need, int* s_tie, int* s_total, int* s_nsel) {
  const int tid = threadIdx.x, lane = tid & 31;
  int tie_need;
  const uint32_t kth = radix_select<false>(x, nullptr, V, Kc, hist, s_prefix, s_need, &tie_need);
  if (tid == 0) *s_tie = 0;
  __syncthreads();
  for (int base = 0; base < V; base += blockDim.x) {
    const int v = base + tid;
    uint32_t k = 0;
    bool gt = false, eq = false;
    if (v < V) {
      k = order_key(x[v]);
      gt = k > kth;
      eq = k == kth;
    }
    if (gt) {
      const int p = atomicAdd(s_nsel, 1);
      skey[p] = k;
      sidx[p] = v;
    }
    // rank of this tie in id order: ties of earlier chunks, earlier warps, earlier lanes
    const unsigned bal = __ballot_sync(0xffffffffu, eq);
    const int before = block_excl_scan(lane == 0 ? __popc(bal) : 0, wsum, s_total);
    const int taken = *s_tie;
    const int o = __shfl_sync(0xffffffffu, before, 0);
    if (eq && taken + o + __popc(bal & ((1u << lane) - 1u)) < tie_need) {
      const int p = atomicAdd(s_nsel, 1);
      skey[p] = k;
      sidx[p] = v;
    }
    __syncthreads();
    if (tid == 0) *s_tie = taken + *s_total;
    __syncthreads();
  }
}

__global__ void __cluster_dims__(kTkCL, 1, 1) __launch_bounds__(1024)
    topk_select_kernel(const float* __restrict__ s, int V, int Kc, int32_t* __restrict__ out_ids) {
  SPEC_TL(spec::kTLTopk);
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) uint8_t tk_smem[];
  uint32_t* gkey = reinterpret_cast<uint32_t*>(tk_smem);              // [kTkCap] gathered copies (rank 0)
  int* gidx = reinterpret_cast<int*>(gkey + kTkCap);
  uint32_t* ckey = reinterpret_cast<uint32_t*>(gidx + kTkCap);        // [kTkCapCta] this CTA's copies
  int* cidx = reinterpret_cast<int*>(ckey + kTkCapCta);
  uint32_t* skey = reinterpret_cast<uint32_t*>(cidx + kTkCapCta);     // [1024] maxima, then the selected
  int* sidx = reinterpret_cast<int*>(skey + 1024);
  int* hist = sidx + 1024;                                            // [256]
  __shared__ int wsum[32];
  __shared__ int s_total, s_nsel, s_nc, s_need, s_tie;
  __shared__ uint32_t s_prefix, s_bound;
  cg::cluster_group cl = cg::this_cluster();
  const int rank = (int)cl.block_rank();
  const int m = blockIdx.x / kTkCL;
  const float* x = s + (size_t)m * V;
  const int tid = threadIdx.x, lane = tid & 31;
  if (tid == 0) { s_nsel = 0; s_nc = 0; }
  // this CTA's groups of four consecutive elements (16-byte loads), UNR groups
  // (4 * UNR loads) in flight per thread
  constexpr int UNR = 4;
  const bool vec = (V % 4 == 0) && ((reinterpret_cast<uintptr_t>(x) & 15u) == 0);
  const int ng = (V + 3) / 4;
  const int g0 = (int)((long long)rank * ng / kTkCL), g1 = (int)((long long)(rank + 1) * ng / kTkCL);
  auto load4 = [&](int gi, float* v) {
    if (gi >= g1) {
      v[0] = v[1] = v[2] = v[3] = -INFINITY;
    } else if (vec) {
      const float4 q = __ldg(reinterpret_cast<const float4*>(x) + gi);
      v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) v[e] = 4 * gi + e < V ? x[4 * gi + e] : -INFINITY;
    }
  };
  // 1. per-thread maxima, the CTA's bound, the cluster's bound T0
  uint32_t tmax = 0;
  for (int base = g0; base < g1; base += UNR * blockDim.x) {
    float v[UNR][4];
#pragma unroll
    for (int u = 0; u < UNR; ++u) load4(base + u * blockDim.x + tid, v[u]);
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int gi = base + u * blockDim.x + tid;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (gi < g1 && 4 * gi + e < V) tmax = max(tmax, order_key(v[u][e]));
    }
  }
  skey[tid] = tmax;           // 0 for a thread without elements: below every key
  __syncthreads();
  int tie_need;
  // the bound needs no more than the top 16 bits: the lower edge of the Kc-th
  // largest maximum's bucket still has Kc maxima at or above it
  const uint32_t tb = radix_select<true>(nullptr, skey, blockDim.x, Kc, hist, &s_prefix, &s_need, &tie_need, 2);
  if (tid == 0) s_bound = tb;
  cl.sync();
  uint32_t t0 = 0;
#pragma unroll
  for (int r = 0; r < kTkCL; ++r) t0 = max(t0, *cl.map_shared_rank(&s_bound, r));
  // 2. copy this CTA's elements >= T0
  for (int base = g0; base < g1; base += UNR * blockDim.x) {
    float v[UNR][4];
#pragma unroll
    for (int u = 0; u < UNR; ++u) load4(base + u * blockDim.x + tid, v[u]);
    uint32_t takem = 0;
    int cnt = 0;
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int gi = base + u * blockDim.x + tid;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (gi < g1 && 4 * gi + e < V && order_key(v[u][e]) >= t0) {
          takem |= 1u << (4 * u + e);
          ++cnt;
        }
    }
    if (__ballot_sync(0xffffffffu, cnt > 0)) {
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      int slot0 = 0;
      if (lane == 31) slot0 = atomicAdd(&s_nc, incl);
      slot0 = __shfl_sync(0xffffffffu, slot0, 31);
      int p = slot0 + incl - cnt;
#pragma unroll
      for (int u = 0; u < UNR; ++u)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if ((takem >> (4 * u + e)) & 1u) {
            if (p < kTkCapCta) {
              ckey[p] = order_key(v[u][e]);
              cidx[p] = 4 * (base + u * blockDim.x + tid) + e;
            }
            ++p;
          }
    }
  }
  cl.sync();                  // every CTA's copies and count are final
  if (rank == 0) {
    int cnt[kTkCL], total = 0;
    bool over = false;
#pragma unroll
    for (int r = 0; r < kTkCL; ++r) {
      cnt[r] = *cl.map_shared_rank(&s_nc, r);
      over = over || cnt[r] > kTkCapCta;
      total += cnt[r];
    }
    over = over || total > kTkCap;
    uint32_t kth;
    if (!over && total <= (int)blockDim.x) {
      // 3. gather one copy per thread; its rank among the copies (larger key first,
      // then smaller id) is its place in the output, and only the Kc first are kept
      uint32_t k = 0;
      int id = 0x7fffffff;
      int off = 0;
#pragma unroll
      for (int r = 0; r < kTkCL; ++r) {
        if (tid >= off && tid < off + cnt[r]) {
          k = cl.map_shared_rank(ckey, r)[tid - off];
          id = cl.map_shared_rank(cidx, r)[tid - off];
        }
        off += cnt[r];
      }
      // pad to a multiple of 8 with entries that never rank above a copy (key 0, id max)
      const int tpad = (total + 7) & ~7;
      if (tid < tpad) {
        gkey[tid] = tid < total ? k : 0u;
        gidx[tid] = tid < total ? id : 0x7fffffff;
      }
      __syncthreads();
      if (tid < total) {
        // four candidates per 16-byte load, two independent counts
        const uint4* k4 = reinterpret_cast<const uint4*>(gkey);
        const int4* i4 = reinterpret_cast<const int4*>(gidx);
        int r0 = 0, r1 = 0;
        for (int j = 0; j < tpad / 4; j += 2) {
          const uint4 ka = k4[j], kb = k4[j + 1];
          const int4 ia = i4[j], ib = i4[j + 1];
          r0 += (ka.x > k || (ka.x == k && ia.x < id)) + (ka.y > k || (ka.y == k && ia.y < id)) +
                (ka.z > k || (ka.z == k && ia.z < id)) + (ka.w > k || (ka.w == k && ia.w < id));
          r1 += (kb.x > k || (kb.x == k && ib.x < id)) + (kb.y > k || (kb.y == k && ib.y < id)) +
                (kb.z > k || (kb.z == k && ib.z < id)) + (kb.w > k || (kb.w == k && ib.w < id));
        }
        const int rnk = r0 + r1;
        if (rnk < Kc) out_ids[(size_t)m * Kc + rnk] = id;
      }
    } else if (!over) {
      // 3. gather, select, sort
      int off = 0;
#pragma unroll
      for (int r = 0; r < kTkCL; ++r) {
        const uint32_t* rk = cl.map_shared_rank(ckey, r);
        const int* ri = cl.map_shared_rank(cidx, r);
        for (int i = tid; i < cnt[r]; i += blockDim.x) {
          gkey[off + i] = rk[i];
          gidx[off + i] = ri[i];
        }
        off += cnt[r];
      }
      __syncthreads();
      kth = radix_select<true>(nullptr, gkey, total, Kc, hist, &s_prefix, &s_need, &tie_need);
      for (int i = tid; i < total; i += blockDim.x) {
        const uint32_t k = gkey[i];
        bool take = k > kth;
        if (k == kth) {
          const int id = gidx[i];
          int rnk = 0;
          for (int j = 0; j < total; ++j) rnk += (gkey[j] == kth && gidx[j] < id);
          take = rnk < tie_need;
        }
        if (take) {
          const int p = atomicAdd(&s_nsel, 1);
          skey[p] = k;
          sidx[p] = gidx[i];
        }
      }
    } else {
      select_row_exact(x, V, Kc, skey, sidx, hist, wsum, &s_prefix, &s_need, &s_tie, &s_total, &s_nsel);
    }
    if (over || total > (int)blockDim.x) {
      __syncthreads();
      sort_selected(skey, sidx, Kc, out_ids + (size_t)m * Kc);
    }
  }
  cl.sync();                  // no CTA leaves while rank 0 may still read its copies
}

// exact logits of the candidates: lm_head[cand] . hn[m]; one warp per candidate
template <typename T>
__global__ void __launch_bounds__(256) rescore_kernel(const T* __restrict__ hn, const T* __restrict__ lm_head,
                                                      int H, int V, const int32_t* __restrict__ cand, int Kc,
                                                      float* __restrict__ exact, void* ws) {
  SPEC_TL(spec::kTLRescore);
  pdl_wait();
  pdl_trigger();
  const int m = blockIdx.y;
  const int j = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (j >= Kc) return;
  int c = cand[(size_t)m * Kc + j];
  if (c < 0 || c >= V) {
    if (lane == 0) report(ws, SPEC_ERR_DEVICE, m, c);
    c = 0;
  }
  const T* w = lm_head + (size_t)c * H;
  const T* h = hn + (size_t)m * H;
  float s = 0.f;
  constexpr int EPV = 16 / sizeof(T);          // elements per 16-byte load
  if (H % EPV == 0 && ((reinterpret_cast<uintptr_t>(w) | reinterpret_cast<uintptr_t>(h)) & 15u) == 0) {
    // 16-byte loads, four in flight per lane (the row of h is shared by the CTA's warps: L1)
    const uint4* w4 = reinterpret_cast<const uint4*>(w);
    const uint4* h4 = reinterpret_cast<const uint4*>(h);
    const int nch = H / EPV;
    for (int c0 = lane; c0 < nch; c0 += 4 * 32) {
      uint4 a[4], b[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (c0 + u * 32 < nch) {
          a[u] = __ldg(w4 + c0 + u * 32);
          b[u] = __ldg(h4 + c0 + u * 32);
        }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (c0 + u * 32 < nch) {
          float fa[EPV], fb[EPV];
          unpack16<T>(a[u], fa);
          unpack16<T>(b[u], fb);
#pragma unroll
          for (int e = 0; e < EPV; ++e) s += fa[e] * fb[e];
        }
    }
  } else {
    for (int n = lane; n < H; n += 32) s += ld(w + n) * ld(h + n);
  }
  s = warp_sum(s);
  if (lane == 0) exact[(size_t)m * Kc + j] = s;
}

// best k_out exact logits among the candidates (ties to the smaller token id)
// (with out_lp: log-probs of the chosen ids under the softmax over the candidates'
// exact logits)
__global__ void __launch_bounds__(128) cand_best_kernel(const float* __restrict__ exact,
                                                        const int32_t* __restrict__ cand, int Kc, int k_out,
                                                        int32_t* __restrict__ out, int ld_out,
                                                        float* __restrict__ out_lp) {
  SPEC_TL(spec::kTLCandBest);
  pdl_wait();
  pdl_trigger();
  __shared__ float red[32];
  __shared__ int redi[32];
  __shared__ int chosen[8];
  const int m = blockIdx.x;
  float lse = 0.f;
  if (out_lp) {
    float mx = -INFINITY;
    for (int j = threadIdx.x; j < Kc; j += blockDim.x) mx = fmaxf(mx, exact[(size_t)m * Kc + j]);
    mx = block_max(mx, red);
    float sm = 0.f;
    for (int j = threadIdx.x; j < Kc; j += blockDim.x) sm += expf(exact[(size_t)m * Kc + j] - mx);
    sm = block_sum(sm, red);
    lse = mx + logf(sm);
  }
  for (int r = 0; r < k_out; ++r) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int j = threadIdx.x; j < Kc; j += blockDim.x) {
      const int t = cand[(size_t)m * Kc + j];
      bool used = false;
      for (int q = 0; q < r; ++q) used |= chosen[q] == t;
      const float v = exact[(size_t)m * Kc + j];
      if (!used && better(v, t, bv, bi)) { bv = v; bi = t; }
    }
    block_argmax(bv, bi, red, redi);
    if (threadIdx.x == 0) {
      chosen[r] = bi;
      out[(size_t)m * ld_out + r] = bi;
      if (out_lp) out_lp[(size_t)m * ld_out + r] = bv - lse;
    }
    __syncthreads();
  }
}

// ================================================================ launchers
static inline unsigned blocks_for(long long n, int bs) { return (unsigned)((n + bs - 1) / bs); }

#define DISPATCH_T(dtype, ...)                                  \
  do {                                                          \
    if ((dtype) == SPEC_DTYPE_BF16) {                           \
      using T = __nv_bfloat16;                                  \
      __VA_ARGS__;                                              \
    } else {                                                    \
      using T = float;                                          \
      __VA_ARGS__;                                              \
    }                                                           \
  } while (0)

void launch_prologue(const spec_model_desc& d, const spec_rows& rows, const spec_weights& w, const void* hid_in,
                     void* x, float2* cs, void* ws, cudaStream_t st) {
  RowInfo ri = to_rowinfo(rows);
  RopeFreq rf;
  for (int i = 0; i < d.head_dim / 2 && i < 128; ++i)
    rf.inv[i] = pow((double)d.rope_theta, -2.0 * (double)i / (double)d.head_dim);
#define PROLOGUE_CL(CL)                                                                                   \
  DISPATCH_T(d.dtype, launch_pdl(prologue_kernel<T, CL>, dim3(rows.M * CL), dim3(NormCL<CL>::kThreads), 0, st, \
                                 ri, d.hidden, d.vocab, d.head_dim, d.rms_eps, rf, (const T*)w.embed,          \
                                 (const T*)w.in_norm, (const T*)w.hidden_norm, (const T*)hid_in, (T*)x, cs, ws))
  if (norm_cl(rows.M) == 2)
    PROLOGUE_CL(2);
  else
    PROLOGUE_CL(8);
#undef PROLOGUE_CL
}

// residual + RMSNorm epilogue of MODE over M rows, cluster size by the row count
template <int MODE>
static void launch_resnorm(int dtype, int M, const float* part, const SKPlan& p, const RowInfo& ri, int H, float eps,
                           const void* hid_in, const void* gain, float* r, void* out_a, void* out_b, cudaStream_t st) {
#define RESNORM_CL(CL)                                                                                     \
  DISPATCH_T(dtype, (launch_pdl(resnorm_kernel<T, MODE, CL>, dim3(M * CL), dim3(NormCL<CL>::kThreads), 0, st, \
                                part, p, ri, H, eps, (const T*)hid_in, (const T*)gain, r, (T*)out_a, (T*)out_b)))
  if (norm_cl(M) == 2)
    RESNORM_CL(2);
  else
    RESNORM_CL(8);
#undef RESNORM_CL
}

void launch_epi_store(int dtype_out, const float* part, const SKPlan& p, int M, int N, void* out, int ld_out,
                      cudaStream_t st) {
  const long long n = (long long)M * N;
  if (dtype_out == SPEC_DTYPE_BF16)
    launch_pdl(epi_store_kernel<__nv_bfloat16>, dim3(blocks_for(n, 256)), dim3(256), 0, st, part, p, M, N, (__nv_bfloat16*)out, ld_out);
  else
    launch_pdl(epi_store_kernel<float>, dim3(blocks_for(n, 256)), dim3(256), 0, st, part, p, M, N, (float*)out, ld_out);
}

void launch_epi_qkv(const spec_model_desc& d, const float* part, const SKPlan& p, const spec_rows& rows,
                    const float2* cs, void* qbuf, const spec_kv& kv, int* work, void* ws, cudaStream_t st) {
  RowInfo ri = to_rowinfo(rows);
  const long long n = (long long)rows.M * (d.n_q_heads + 2 * d.n_kv_heads) * (d.head_dim / 2);
  DISPATCH_T(d.dtype, launch_pdl(epi_qkv_kernel<T>, dim3(blocks_for(n, 256)), dim3(256), 0, st, 
                          part, p, ri, d.n_q_heads, d.n_kv_heads, d.head_dim, cs, (T*)qbuf, kv, work, ws));
}

void launch_epi_oproj(const spec_model_desc& d, const float* part, const SKPlan& p, const spec_rows& rows,
                      const void* hid_in, const spec_weights& w, float* r1, void* nout, cudaStream_t st) {
  RowInfo ri = to_rowinfo(rows);
  launch_resnorm<0>(d.dtype, rows.M, part, p, ri, d.hidden, d.rms_eps, hid_in, w.post_norm, r1, nullptr, nout, st);
}

void launch_epi_fcnorm(const spec_model_desc& d, const float* part, const SKPlan& p, int M, float* r,
                       const void* gain, void* h0, cudaStream_t st) {
  RowInfo ri{};
  launch_resnorm<2>(d.dtype, M, part, p, ri, d.hidden, d.rms_eps, nullptr, gain, r, nullptr, h0, st);
}

void launch_epi_swiglu(const spec_model_desc& d, const float* part, const SKPlan& p, int M, void* act,
                       cudaStream_t st) {
  // four features a thread once that still gives two blocks per SM
  const int I = d.intermediate;
  if ((long long)((I + 1023) / 1024) * M >= 2LL * sm_count()) {
    const dim3 grid((I + 1023) / 1024, M);
    DISPATCH_T(d.dtype, launch_pdl(epi_swiglu_kernel<T, 4>, grid, dim3(256), 0, st, part, p, M, I, (T*)act));
  } else {
    const dim3 grid((I + 255) / 256, M);
    DISPATCH_T(d.dtype, launch_pdl(epi_swiglu_kernel<T, 1>, grid, dim3(256), 0, st, part, p, M, I, (T*)act));
  }
}

void launch_epi_down(const spec_model_desc& d, const float* part, const SKPlan& p, int M, float* r1,
                     const spec_weights& w, void* prenorm, void* normed, cudaStream_t st) {
  RowInfo ri{};
  launch_resnorm<1>(d.dtype, M, part, p, ri, d.hidden, d.rms_eps, nullptr, w.final_norm, r1, prenorm, normed, st);
}

void launch_simt_gemm(int dtype, const void* A0, const void* A1, const void* A2, int K, const void* X, int M,
                      const SKPlan& p, float* part, cudaStream_t st) {
  DISPATCH_T(dtype, launch_pdl(simt_gemm_kernel<T>, dim3(p.G), dim3(256), 0, st, (const T*)A0, (const T*)A1, (const T*)A2, K,
                                                              (const T*)X, M, p, part));
}

int attn_qmax(int rows_per_req, int G) {
  const int n = rows_per_req * G;
  if (n <= 4) return 4;
  if (n <= 8) return 8;
  if (n <= 16) return 16;
  return 32;
}

// Splits per (request, kv head, query group): about four work items per
// resident CTA of the persistent grid (at most three CTAs per SM), but no split
// shorter than two 64-key tiles when an upper bound of the context is known.
constexpr int kAttnItemsPerSm = 12;

int attn_splits(int B, int nkv, int nqg, int sms, int max_keys) {
  const int pairs = B * nkv * nqg;
  int s = (kAttnItemsPerSm * sms + pairs - 1) / pairs;
  if (max_keys > 0) {
    const int by_len = (max_keys + 127) / 128;
    if (s > by_len) s = by_len;
  }
  if (s < 1) s = 1;
  if (s > 64) s = 64;
  return s;
}

// Upper bound of the split count for any call with M rows: a work item serves
// at most 32 query slots, so a pass has at least nkv * ceil(M * G / 32) pairs.
int attn_splits_max(const spec_model_desc& d, int M, int sms) {
  const int G = d.n_q_heads / d.n_kv_heads;
  const int min_pairs = d.n_kv_heads * ((M * G + 31) / 32);
  int s = (kAttnItemsPerSm * sms + min_pairs - 1) / min_pairs;
  if (s < 1) s = 1;
  if (s > 64) s = 64;
  return s;
}

template <typename TT, int HDV, int QM>
static spec_status attn_launch(const spec_model_desc& d, const RowInfo& ri, const spec_rows& rows, const void* qbuf,
                               const spec_kv& kv, float* opart, float2* mlpart, void* attn_out, int nsplit, int nqg,
                               void* ws, cudaStream_t st) {
  static int attr_dev = -1, occ = 1;
  int dev = 0;
  cudaGetDevice(&dev);
  constexpr size_t smem = attn_smem_for<TT, HDV, QM>();
  auto kern = attn_split_kernel<TT, HDV, QM>;
  if (attr_dev != dev) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return SPEC_ERR_CUDA;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, 128, smem) != cudaSuccess || occ < 1) occ = 1;
    attr_dev = dev;
  }
  const int n_items = nsplit * d.n_kv_heads * rows.B * nqg;
  const int grid = std::min(n_items, occ * sm_count());
  const float scale = 1.f / sqrtf((float)d.head_dim);
  launch_pdl(kern, dim3(grid), dim3(128), smem, st, (const TT*)qbuf, kv, ri, d.n_q_heads, d.n_kv_heads, d.window,
             nsplit, nqg, n_items, scale, opart, mlpart, ws);
  launch_combine<TT, HDV>(opart, mlpart, rows.M, d.n_q_heads, nsplit, attn_out, st);
  return SPEC_OK;
}

template <int HDV, int MT>
static spec_status attn_mma_launch(const spec_model_desc& d, const RowInfo& ri, const spec_rows& rows,
                                   const void* qbuf, const spec_kv& kv, float* opart, float2* mlpart, void* attn_out,
                                   int nsplit, int nqg, int* work, void* ws, cudaStream_t st) {
  static int attr_dev = -1, occ = 1;
  int dev = 0;
  cudaGetDevice(&dev);
  constexpr size_t smem = attn_mma_smem<HDV, MT>();
  auto kern = attn_mma_kernel<HDV, MT>;
  if (attr_dev != dev) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return SPEC_ERR_CUDA;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, 128, smem) != cudaSuccess || occ < 1) occ = 1;
    attr_dev = dev;
  }
  const int n_items = nsplit * d.n_kv_heads * rows.B * nqg;
  const int grid = std::min(n_items, occ * sm_count());
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)d.head_dim);
  launch_pdl(kern, dim3(grid), dim3(128), smem, st, (const __nv_bfloat16*)qbuf, kv, ri, d.n_q_heads, d.n_kv_heads,
             d.window, nsplit, nqg, n_items, scale_log2, opart, mlpart, n_items > grid ? work : nullptr, ws);
  launch_combine<__nv_bfloat16, HDV>(opart, mlpart, rows.M, d.n_q_heads, nsplit, attn_out, st);
  return SPEC_OK;
}

// K / V tensor maps of a cache, reused while the cache and its shape stay the same
static bool kv_maps(const spec_kv& kv, int nkv, int hd, int bh, CUtensorMap* tk, CUtensorMap* tv) {
  struct Entry {
    const void* k;
    const void* v;
    int slots, nkv, hd, bh, dev;
    CUtensorMap mk, mv;
  };
  static Entry e{};
  static bool have = false;
  int dev = 0;
  cudaGetDevice(&dev);
  if (!have || e.k != kv.k || e.v != kv.v || e.slots != kv.num_slots || e.nkv != nkv || e.hd != hd || e.bh != bh ||
      e.dev != dev) {
    have = false;
    if (!tc::make_kv_map(&e.mk, kv.k, kv.num_slots, nkv, hd, bh) ||
        !tc::make_kv_map(&e.mv, kv.v, kv.num_slots, nkv, hd, bh))
      return false;
    e.k = kv.k; e.v = kv.v; e.slots = kv.num_slots; e.nkv = nkv; e.hd = hd; e.bh = bh; e.dev = dev;
    have = true;
  }
  *tk = e.mk;
  *tv = e.mv;
  return true;
}

template <int HDV, int MT>
static spec_status attn_ws_launch(const spec_model_desc& d, const RowInfo& ri, const spec_rows& rows,
                                  const void* qbuf, const spec_kv& kv, float* opart, float2* mlpart, void* attn_out,
                                  int nsplit, int nqg, int* work, void* ws, cudaStream_t st) {
  static int attr_dev = -1, occ = 1;
  int dev = 0;
  cudaGetDevice(&dev);
  constexpr size_t smem = WsShape<HDV, MT>::kSmem;
  auto kern = attn_ws_kernel<HDV, MT>;
  if (attr_dev != dev) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return SPEC_ERR_CUDA;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, 160, smem) != cudaSuccess || occ < 1) occ = 1;
    attr_dev = dev;
  }
  const int bh = kv.block_size % 16 == 0 ? 16 : 8;
  CUtensorMap tk, tv;
  if (!kv_maps(kv, d.n_kv_heads, HDV, bh, &tk, &tv)) return SPEC_ERR_CUDA;
  const int n_items = nsplit * d.n_kv_heads * rows.B * nqg;
  const int grid = std::min(n_items, occ * sm_count());
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)d.head_dim);
  launch_pdl(kern, dim3(grid), dim3(160), smem, st, tk, tv, (const __nv_bfloat16*)qbuf, kv, ri, d.n_q_heads,
             d.n_kv_heads, d.window, nsplit, nqg, n_items, bh, scale_log2, opart, mlpart,
             n_items > grid ? work : nullptr, ws);
  launch_combine<__nv_bfloat16, HDV>(opart, mlpart, rows.M, d.n_q_heads, nsplit, attn_out, st);
  return SPEC_OK;
}

template <typename TT, int HDV>
static spec_status attn_qdispatch(int qmax, const spec_model_desc& d, const RowInfo& ri, const spec_rows& rows,
                                  const void* qbuf, const spec_kv& kv, float* opart, float2* mlpart, void* out,
                                  int nsplit, int nqg, void* ws, cudaStream_t st) {
  switch (qmax) {
    case 4: return attn_launch<TT, HDV, 4>(d, ri, rows, qbuf, kv, opart, mlpart, out, nsplit, nqg, ws, st);
    case 8: return attn_launch<TT, HDV, 8>(d, ri, rows, qbuf, kv, opart, mlpart, out, nsplit, nqg, ws, st);
    case 16: return attn_launch<TT, HDV, 16>(d, ri, rows, qbuf, kv, opart, mlpart, out, nsplit, nqg, ws, st);
    default: return attn_launch<TT, HDV, 32>(d, ri, rows, qbuf, kv, opart, mlpart, out, nsplit, nqg, ws, st);
  }
}

spec_status launch_attention(const spec_model_desc& d, const spec_rows& rows, const void* qbuf, const spec_kv& kv,
                             float* opart, float2* mlpart, void* attn_out, int nsplit, int* work, void* ws,
                             cudaStream_t st) {
  RowInfo ri = to_rowinfo(rows);
  const int G = d.n_q_heads / d.n_kv_heads;
  const int qmax = attn_qmax(rows.rows_per_req, G);
  const int nqg = (rows.rows_per_req * G + qmax - 1) / qmax;
  spec_status s;
  if (d.dtype == SPEC_DTYPE_BF16) {
    // tensor-core path: 16 or 32 query rows per item (the same groups as qmax <= 16 / 32)
    const bool two = qmax > 16;
    // warp-specialised kernel with tensor copies: one or two m-tiles, cache blocks of a
    // multiple of 8 slots, 16-byte aligned caches
    const bool tma = kv.block_size % 8 == 0 && ((reinterpret_cast<uintptr_t>(kv.k) |
                                                 reinterpret_cast<uintptr_t>(kv.v)) & 15u) == 0;
    if (tma && d.head_dim == 128)
      return two ? attn_ws_launch<128, 2>(d, ri, rows, qbuf, kv, opart, mlpart, attn_out, nsplit, nqg, work, ws, st)
                 : attn_ws_launch<128, 1>(d, ri, rows, qbuf, kv, opart, mlpart, attn_out, nsplit, nqg, work, ws, st);
    if (tma && d.head_dim == 64)
      return two ? attn_ws_launch<64, 2>(d, ri, rows, qbuf, kv, opart, mlpart, attn_out, nsplit, nqg, work, ws, st)
                 : attn_ws_launch<64, 1>(d, ri, rows, qbuf, kv, opart, mlpart, attn_out, nsplit, nqg, work, ws, st);
    if (d.head_dim == 128)
      s = two ? attn_mma_launch<128, 2>(d, ri, rows, qbuf, kv, opart, mlpart, attn_out, nsplit, nqg, work, ws, st)
              : attn_mma_launch<128, 1>(d, ri, rows, qbuf, kv, opart, mlpart, attn_out, nsplit, nqg, work, ws, st);
    else if (d.head_dim == 64)
      s = two ? attn_mma_launch<64, 2>(d, ri, rows, qbuf, kv, opart, mlpart, attn_out, nsplit, nqg, work, ws, st)
              : attn_mma_launch<64, 1>(d, ri, rows, qbuf, kv, opart, mlpart, attn_out, nsplit, nqg, work, ws, st);
    else
      return SPEC_ERR_UNSUPPORTED;
  } else {
    if (d.head_dim == 128)
      s = attn_qdispatch<float, 128>(qmax, d, ri, rows, qbuf, kv, opart, mlpart, attn_out, nsplit, nqg, ws, st);
    else if (d.head_dim == 64)
      s = attn_qdispatch<float, 64>(qmax, d, ri, rows, qbuf, kv, opart, mlpart, attn_out, nsplit, nqg, ws, st);
    else
      return SPEC_ERR_UNSUPPORTED;
  }
  return s;
}

void launch_row_stats(const float* logits, int M, int V, int k, int32_t* ids, int ld_ids, float* lp, float* lse,
                      const int32_t* d2t, cudaStream_t st) {
  launch_pdl(row_stats_kernel, dim3(M), dim3(256), 0, st, logits, V, k, ids, ld_ids, lp, lse, d2t);
}

void launch_topk_select(const float* s, int M, int V, int Kc, int32_t* out_ids, cudaStream_t st) {
  static int attr_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_dev != dev) {
    cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)topk_select_smem());
    attr_dev = dev;
  }
  launch_pdl(topk_select_kernel, dim3(M * kTkCL), dim3(1024), topk_select_smem(), st, s, V, Kc, out_ids);
}

void launch_rescore(int dtype, const void* hn, const void* lm_head, int H, int V, const int32_t* cand, int M, int Kc,
                    float* exact, void* ws, cudaStream_t st) {
  dim3 grid((Kc + 7) / 8, M);
  DISPATCH_T(dtype, launch_pdl(rescore_kernel<T>, dim3(grid), dim3(256), 0, st, (const T*)hn, (const T*)lm_head, H, V, cand, Kc, exact,
                                                             ws));
}

void launch_cand_best(const float* exact, const int32_t* cand, int M, int Kc, int k_out, int32_t* out, int ld_out,
                      float* out_lp, cudaStream_t st) {
  launch_pdl(cand_best_kernel, dim3(M), dim3(128), 0, st, exact, cand, Kc, k_out, out, ld_out, out_lp);
}

}  // namespace spec

// per-unit log setter of the instrumented build (no-op otherwise)
SPEC_TL_SETTER(layer)
