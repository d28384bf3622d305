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
// Row-wide reductions (RMSNorm over H) run on a thread-block cluster of kCL
// CTAs per row: each CTA owns H / kCL features, the per-CTA sums meet in
// distributed shared memory, summed in rank order (deterministic).
constexpr int kCL = 8;

SPEC_DEV float2 cluster_sum2(float2 v, float* red, float2* slot) {
  v.x = block_sum(v.x, red);
  v.y = block_sum(v.y, red);
  if (threadIdx.x == 0) *slot = v;
  cg::cluster_group cl = cg::this_cluster();
  cl.sync();
  float2 t = make_float2(0.f, 0.f);
#pragma unroll
  for (int r = 0; r < kCL; ++r) {
    const float2 o = *cl.map_shared_rank(slot, r);
    t.x += o.x;
    t.y += o.y;
  }
  cl.sync();     // no CTA leaves while another still reads its slot
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
template <typename T>
__global__ void __cluster_dims__(kCL, 1, 1) __launch_bounds__(256)
    prologue_kernel(RowInfo ri, int H, int V, int hd, float eps, const __grid_constant__ RopeFreq rf,
                    const T* __restrict__ embed, const T* __restrict__ g_in, const T* __restrict__ g_hid,
                    const T* __restrict__ hid_in, T* __restrict__ x, float2* __restrict__ cs, void* ws) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[32];
  __shared__ float2 slot;
  const int m = blockIdx.x / kCL, rk = blockIdx.x % kCL;
  int tok = ri.tok[(size_t)m * ri.tok_stride];
  if (tok < 0 || tok >= V) {
    if (threadIdx.x == 0 && rk == 0) report(ws, SPEC_ERR_DEVICE, m, tok);
    tok = 0;
  }
  const T* e = embed + (size_t)tok * H;
  const T* h = hid_in + (size_t)row_src(ri, m) * H;
  const int n0 = rk * H / kCL, n1 = (rk + 1) * H / kCL;
  float2 ss = make_float2(0.f, 0.f);
  for (int n = n0 + threadIdx.x; n < n1; n += blockDim.x) {
    const float a = ld(e + n), c = ld(h + n);
    ss.x += a * a;
    ss.y += c * c;
  }
  const float2 tot = cluster_sum2(ss, red, &slot);
  const float re = 1.f / sqrtf(tot.x / H + eps), rh = 1.f / sqrtf(tot.y / H + eps);
  T* xo = x + (size_t)m * 2 * H;
  for (int n = n0 + threadIdx.x; n < n1; n += blockDim.x) {
    st(xo + n, ld(e + n) * re * ld(g_in + n));
    st(xo + H + n, ld(h + n) * rh * ld(g_hid + n));
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
  pdl_wait();
  pdl_trigger();
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)M * N) return;
  const int m = (int)(idx / N), n = (int)(idx % N);
  st(out + (size_t)m * ld_out + n, sk_sum(part, p, m, n));
}

// q / k get the rotary embedding (pairs i, i + hd/2), v is copied; q goes to
// qbuf [M, nq*hd], k and v to the paged cache at entry ctx + kv_idx.
template <typename T>
__global__ void epi_qkv_kernel(const float* __restrict__ part, SKPlan p, RowInfo ri, int nq, int nkv, int hd,
                               const float2* __restrict__ cs, T* __restrict__ qbuf, spec_kv kv, void* ws) {
  pdl_wait();
  pdl_trigger();
  const int half = hd / 2;
  const int nh = nq + 2 * nkv;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)ri.M * nh * half) return;
  const int m = (int)(idx / (nh * half));
  const int rem = (int)(idx % (nh * half));
  const int hh = rem / half, i = rem % half;
  const int n1 = hh * hd + i, n2 = n1 + half;
  float x1 = sk_sum(part, p, m, n1), x2 = sk_sum(part, p, m, n2);
  if (hh < nq + nkv) {
    const float2 c = cs[(size_t)m * half + i];
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
  const int b = row_req(ri, m);
  const int ci = ri.ctx_len[b] + row_kvidx(ri, m);
  const long long slot = slot_of(kv, b, ci);
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
// One cluster of kCL CTAs per row.
template <typename T, int MODE>
__global__ void __cluster_dims__(kCL, 1, 1) __launch_bounds__(256)
    resnorm_kernel(const float* __restrict__ part, SKPlan p, RowInfo ri, int H, float eps,
                   const T* __restrict__ hid_in, const T* __restrict__ gain, float* __restrict__ r,
                   T* __restrict__ out_a, T* __restrict__ out_b) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[32];
  __shared__ float2 slot;
  const int m = blockIdx.x / kCL, rk = blockIdx.x % kCL;
  const int n0 = rk * H / kCL, n1 = (rk + 1) * H / kCL;
  const T* h = (MODE == 0) ? hid_in + (size_t)row_src(ri, m) * H : nullptr;
  float* rr = r + (size_t)m * H;
  float ss = 0.f;
  for (int n = n0 + threadIdx.x; n < n1; n += blockDim.x) {
    const float base = (MODE == 0) ? ld(h + n) : rr[n];
    const float v = base + sk_sum(part, p, m, n);
    rr[n] = v;
    if (MODE == 1) st(out_a + (size_t)m * H + n, v);
    ss += v * v;
  }
  const float2 tot = cluster_sum2(make_float2(ss, 0.f), red, &slot);
  const float rs = 1.f / sqrtf(tot.x / H + eps);
  for (int n = n0 + threadIdx.x; n < n1; n += blockDim.x) st(out_b + (size_t)m * H + n, rr[n] * rs * ld(gain + n));
}

// act = silu(gate) * up  (gate rows [0, I), up rows [I, 2I) of the stacked output)
template <typename T>
__global__ void epi_swiglu_kernel(const float* __restrict__ part, SKPlan p, int M, int I, T* __restrict__ act) {
  pdl_wait();
  pdl_trigger();
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)M * I) return;
  const int m = (int)(idx / I), i = (int)(idx % I);
  const float g = sk_sum(part, p, m, i);
  const float u = sk_sum(part, p, m, I + i);
  st(act + (size_t)m * I + i, g / (1.f + expf(-g)) * u);
}

// ---------------------------------------------------------------- SIMT GEMM
// Stream-K GEMM on CUDA cores (fp32 models, and M <= 32): partial sums of
// X[M, K] @ W^T for the CTA's iteration range, same partial layout as the
// tensor-core kernel.
template <typename T>
__global__ void __launch_bounds__(256) simt_gemm_kernel(const T* __restrict__ A0, const T* __restrict__ A1,
                                                        const T* __restrict__ A2, int K, const T* __restrict__ X,
                                                        int M, SKPlan p, float* __restrict__ part) {
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

// Split-KV decode attention with the row masks of spec_rows.  grid = (nsplit,
// nkv, B * nqg); a CTA serves up to QMAX queries (rows of one request x the q
// heads of one kv head) over one slice of that request's key range: context
// keys [klo, ctx) then draft-region keys [ctx, ctx + nd).  Keys are processed
// 128 at a time (one per thread for the scores), K and V staged through shared
// memory with 16-byte copies.
template <typename T, int HD, int QMAX>
__global__ void __launch_bounds__(128) attn_split_kernel(const T* __restrict__ qbuf, spec_kv kv, RowInfo ri,
                                                         int nq, int nkv, int window, int nsplit, int nqg,
                                                         float scale, float* __restrict__ opart,
                                                         float2* __restrict__ mlpart, void* ws) {
  pdl_wait();
  pdl_trigger();
  constexpr int TK = 128;                      // keys per tile (one per thread)
  constexpr int KP = HD + (16 / sizeof(T));    // padded smem row (elements)
  constexpr int QW = QMAX / 4;                 // queries per warp in softmax / PV
  extern __shared__ __align__(16) uint8_t attn_smem[];
  float* sQ = reinterpret_cast<float*>(attn_smem);                       // [QMAX][HD]
  float* sS = sQ + QMAX * HD;                                           // [QMAX][TK]
  T* sK = reinterpret_cast<T*>(sS + QMAX * TK);                         // [TK][KP]
  T* sV = sK + TK * KP;                                                 // [TK][HD]
  __shared__ float sM[QMAX], sL[QMAX], sA[QMAX];
  __shared__ int s_lo[QMAX];
  __shared__ unsigned long long s_mask[QMAX];
  __shared__ int s_klo, s_nd;

  const int s = blockIdx.x, g = blockIdx.y;
  const int b = blockIdx.z / nqg, qg = blockIdx.z % nqg;
  const int G = nq / nkv;
  const int nQall = ri.R * G;
  const int q0 = qg * QMAX;
  const int nQ = min(QMAX, nQall - q0);
  const int ctx = ri.ctx_len[b];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (tid < 32) {
    int lo = 0x7fffffff;
    unsigned long long mk = 0;
    if (tid < nQ) {
      const int m = b * ri.R + (q0 + tid) / G;
      const int pos = row_pos(ri, m);
      lo = window > 0 ? max(0, pos - window + 1) : 0;
      if (lo > ctx) lo = ctx;
      mk = row_mask(ri, m);
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
    if (tid < QMAX) {
      sM[tid] = -INFINITY;
      sL[tid] = 0.f;
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
  const int kbeg = s * chunk, kend = min(total, kbeg + chunk);

  constexpr int DJ = HD / 32;
  float acc[QW][DJ];
#pragma unroll
  for (int a = 0; a < QW; ++a)
#pragma unroll
    for (int jj = 0; jj < DJ; ++jj) acc[a][jj] = 0.f;

  for (int t0 = kbeg; t0 < kend; t0 += TK) {
    const int nk = min(TK, kend - t0);
    // stage K / V rows of this tile: asynchronous 16-byte copies, all in flight
    // together (a key's row of one kv head is HD contiguous elements)
    constexpr int CH = HD * sizeof(T) / 16;        // 16-byte chunks per row
    for (int e = tid; e < nk * CH; e += blockDim.x) {
      const int kt = e / CH, ch = e % CH;
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
    cp_async_wait_all();
    __syncthreads();
    // scores: thread tid owns key tid of the tile
    if (tid < nk) {
      const int kidx = t0 + tid;
      const int ci = kidx < nctx ? klo + kidx : ctx + (kidx - nctx);
      const bool valid = slot_of(kv, b, ci) >= 0;
      float sc[QMAX];
#pragma unroll
      for (int qi = 0; qi < QMAX; ++qi) sc[qi] = 0.f;
      constexpr int EPV = 16 / sizeof(T);
      const uint4* kr = reinterpret_cast<const uint4*>(sK + tid * KP);
#pragma unroll 2
      for (int d0 = 0; d0 < HD; d0 += EPV) {
        float kd[EPV];
        unpack16<T>(kr[d0 / EPV], kd);
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
#pragma unroll
          for (int qi = 0; qi < QMAX; ++qi) sc[qi] += sQ[qi * HD + d0 + e] * kd[e];
        }
      }
#pragma unroll
      for (int qi = 0; qi < QMAX; ++qi) {
        bool ok = valid && qi < nQ;
        if (ok) {
          if (ci < ctx) ok = ci >= s_lo[qi];
          else ok = (s_mask[qi] >> (ci - ctx)) & 1ull;
        }
        sS[qi * TK + tid] = ok ? sc[qi] : -INFINITY;
      }
    } else {
#pragma unroll
      for (int qi = 0; qi < QMAX; ++qi) sS[qi * TK + tid] = -INFINITY;
    }
    __syncthreads();
    // online softmax: warp w handles queries w, w+4, ...
#pragma unroll
    for (int a = 0; a < QW; ++a) {
      const int qi = warp + 4 * a;
      float v[TK / 32];
      float mx = -INFINITY;
#pragma unroll
      for (int u = 0; u < TK / 32; ++u) {
        v[u] = sS[qi * TK + lane + 32 * u];
        mx = fmaxf(mx, v[u]);
      }
      mx = warp_max(mx);
      const float mold = sM[qi];
      const float mnew = fmaxf(mold, mx);
      float sum = 0.f;
#pragma unroll
      for (int u = 0; u < TK / 32; ++u) {
        const float e = (mnew == -INFINITY) ? 0.f : expf(v[u] - mnew);
        sS[qi * TK + lane + 32 * u] = e;
        sum += e;
      }
      sum = warp_sum(sum);
      const float alpha = (mold == -INFINITY) ? 0.f : expf(mold - mnew);
      __syncwarp();
      if (lane == 0) {
        sA[qi] = alpha;
        sL[qi] = sL[qi] * alpha + sum;
        sM[qi] = mnew;
      }
#pragma unroll
      for (int jj = 0; jj < DJ; ++jj) acc[a][jj] *= alpha;
    }
    __syncwarp();
    // P @ V (each warp reads only the probabilities of its own queries)
    for (int kt = 0; kt < nk; ++kt) {
      float vv[DJ];
#pragma unroll
      for (int jj = 0; jj < DJ; ++jj) vv[jj] = ld(sV + kt * HD + lane + 32 * jj);
#pragma unroll
      for (int a = 0; a < QW; ++a) {
        const float pw = sS[(warp + 4 * a) * TK + kt];
#pragma unroll
        for (int jj = 0; jj < DJ; ++jj) acc[a][jj] += pw * vv[jj];
      }
    }
    __syncthreads();
  }
  // write this split's partials
#pragma unroll
  for (int a = 0; a < QW; ++a) {
    const int qi = warp + 4 * a;
    if (qi >= nQ) continue;
    const int q = q0 + qi;
    const int m = b * ri.R + q / G, h = g * G + q % G;
    const size_t base = ((size_t)m * nq + h) * nsplit + s;
    float* o = opart + base * HD;
#pragma unroll
    for (int jj = 0; jj < DJ; ++jj) o[lane + 32 * jj] = acc[a][jj];
    if (lane == 0) mlpart[base] = make_float2(sM[qi], sL[qi]);
  }
}

template <typename T, int HD>
__global__ void __launch_bounds__(HD) attn_combine_kernel(const float* __restrict__ opart,
                                                          const float2* __restrict__ mlpart, int nq, int nsplit,
                                                          T* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int mh = blockIdx.x;          // m * nq + h
  const int d = threadIdx.x;
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, mlpart[(size_t)mh * nsplit + s].x);
  float L = 0.f, o = 0.f;
  if (M > -INFINITY) {
    for (int s = 0; s < nsplit; ++s) {
      const float2 ml = mlpart[(size_t)mh * nsplit + s];
      if (ml.x == -INFINITY) continue;
      const float w = expf(ml.x - M);
      L += ml.y * w;
      o += opart[((size_t)mh * nsplit + s) * HD + d] * w;
    }
  }
  st(out + (size_t)mh * HD + d, L > 0.f ? o / L : 0.f);
}

// ---------------------------------------------------------------- row statistics
// From full fp32 logits [M, V]: lse and the k largest (ties to smaller id).
__global__ void __launch_bounds__(256) row_stats_kernel(const float* __restrict__ logits, int V, int k,
                                                        int32_t* __restrict__ ids, int ld_ids, float* __restrict__ lp,
                                                        float* __restrict__ lse_out, const int32_t* __restrict__ d2t) {
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
// descending order: exact radix selection of the Kc-th key, ordered collection
// of the ties, bitonic sort of the selected.  One CTA of 1024 threads per row.
__global__ void __launch_bounds__(1024) topk_select_kernel(const float* __restrict__ s, int V, int Kc,
                                                           int32_t* __restrict__ out_ids) {
  pdl_wait();
  pdl_trigger();
  __shared__ int hist[256];
  __shared__ uint32_t s_prefix;
  __shared__ int s_need;
  __shared__ uint32_t skey[1024];
  __shared__ int sidx[1024];
  __shared__ int s_cnt, s_tie_taken;
  __shared__ int wcount[32];
  const int m = blockIdx.x;
  const float* x = s + (size_t)m * V;
  const int tid = threadIdx.x;
  if (tid == 0) { s_prefix = 0; s_need = Kc; }
  __syncthreads();
  // radix select: find the key value of the Kc-th largest and how many of the
  // elements equal to it are needed
  for (int shift = 24; shift >= 0; shift -= 8) {
    if (tid < 256) hist[tid] = 0;
    __syncthreads();
    const uint32_t prefix = s_prefix;
    const uint32_t pmask = (shift == 24) ? 0u : (0xffffffffu << (shift + 8));
    for (int v = tid; v < V; v += blockDim.x) {
      const uint32_t k = order_key(x[v]);
      if ((k & pmask) == (prefix & pmask)) atomicAdd(&hist[(k >> shift) & 0xff], 1);
    }
    __syncthreads();
    if (tid == 0) {
      int need = s_need, acc = 0, dsel = 0;
      for (int dgt = 255; dgt >= 0; --dgt) {
        if (acc + hist[dgt] >= need) { dsel = dgt; break; }
        acc += hist[dgt];
      }
      s_need = need - acc;
      s_prefix = prefix | ((uint32_t)dsel << shift);
    }
    __syncthreads();
  }
  const uint32_t kth = s_prefix;
  const int tie_need = s_need;      // elements equal to kth to take (smallest ids)
  if (tid == 0) { s_cnt = 0; s_tie_taken = 0; }
  __syncthreads();
  // collect in index order (ties keep the smallest ids)
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
      const int p = atomicAdd(&s_cnt, 1);
      skey[p] = k;
      sidx[p] = v;
    }
    // ordered ranks of the ties within this chunk
    const unsigned bal = __ballot_sync(0xffffffffu, eq);
    if ((tid & 31) == 0) wcount[tid >> 5] = __popc(bal);
    __syncthreads();
    int before = 0;
    for (int w = 0; w < (tid >> 5); ++w) before += wcount[w];
    before += __popc(bal & ((1u << (tid & 31)) - 1u));
    const int taken = s_tie_taken;
    if (eq && taken + before < tie_need) {
      const int p = atomicAdd(&s_cnt, 1);
      skey[p] = k;
      sidx[p] = v;
    }
    __syncthreads();
    if (tid == 0) {
      int tot = 0;
      for (int w = 0; w < 32; ++w) tot += wcount[w];
      s_tie_taken = taken + tot;
    }
    __syncthreads();
  }
  // bitonic sort of the Kc selected: key descending, index ascending
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
  if (tid < Kc) out_ids[(size_t)m * Kc + tid] = sidx[tid];
}

// exact logits of the candidates: lm_head[cand] . hn[m]; one warp per candidate
template <typename T>
__global__ void __launch_bounds__(256) rescore_kernel(const T* __restrict__ hn, const T* __restrict__ lm_head,
                                                      int H, int V, const int32_t* __restrict__ cand, int Kc,
                                                      float* __restrict__ exact, void* ws) {
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
  for (int n = lane; n < H; n += 32) s += ld(w + n) * ld(h + n);
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
  DISPATCH_T(d.dtype, launch_pdl(prologue_kernel<T>, dim3(rows.M * kCL), dim3(256), 0, st, 
                          ri, d.hidden, d.vocab, d.head_dim, d.rms_eps, rf,
                          (const T*)w.embed, (const T*)w.in_norm, (const T*)w.hidden_norm, (const T*)hid_in,
                          (T*)x, cs, ws));
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
                    const float2* cs, void* qbuf, const spec_kv& kv, void* ws, cudaStream_t st) {
  RowInfo ri = to_rowinfo(rows);
  const long long n = (long long)rows.M * (d.n_q_heads + 2 * d.n_kv_heads) * (d.head_dim / 2);
  DISPATCH_T(d.dtype, launch_pdl(epi_qkv_kernel<T>, dim3(blocks_for(n, 256)), dim3(256), 0, st, 
                          part, p, ri, d.n_q_heads, d.n_kv_heads, d.head_dim, cs, (T*)qbuf, kv, ws));
}

void launch_epi_oproj(const spec_model_desc& d, const float* part, const SKPlan& p, const spec_rows& rows,
                      const void* hid_in, const spec_weights& w, float* r1, void* nout, cudaStream_t st) {
  RowInfo ri = to_rowinfo(rows);
  DISPATCH_T(d.dtype, (launch_pdl(resnorm_kernel<T, 0>, dim3(rows.M * kCL), dim3(256), 0, st, 
                          part, p, ri, d.hidden, d.rms_eps, (const T*)hid_in, (const T*)w.post_norm, r1, nullptr,
                          (T*)nout)));
}

void launch_epi_swiglu(const spec_model_desc& d, const float* part, const SKPlan& p, int M, void* act,
                       cudaStream_t st) {
  const long long n = (long long)M * d.intermediate;
  DISPATCH_T(d.dtype,
             launch_pdl(epi_swiglu_kernel<T>, dim3(blocks_for(n, 256)), dim3(256), 0, st, part, p, M, d.intermediate, (T*)act));
}

void launch_epi_down(const spec_model_desc& d, const float* part, const SKPlan& p, int M, float* r1,
                     const spec_weights& w, void* prenorm, void* normed, cudaStream_t st) {
  RowInfo ri{};
  DISPATCH_T(d.dtype, (launch_pdl(resnorm_kernel<T, 1>, dim3(M * kCL), dim3(256), 0, st, part, p, ri, d.hidden, d.rms_eps, nullptr,
                                                                     (const T*)w.final_norm, r1, (T*)prenorm,
                                                                     (T*)normed)));
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

// Splits per (request, kv head, query group): enough CTAs for ~2 per SM, but no
// split shorter than one 128-key tile when an upper bound of the context is known.
int attn_splits(int B, int nkv, int nqg, int sms, int max_keys) {
  const int ctas = B * nkv * nqg;
  int s = (2 * sms + ctas - 1) / ctas;
  if (max_keys > 0) {
    const int by_len = (max_keys + 127) / 128;
    if (s > by_len) s = by_len;
  }
  if (s < 1) s = 1;
  if (s > 64) s = 64;
  return s;
}

// Upper bound of the split count for any call with M rows: every CTA serves at
// most 32 query slots, so a pass has at least nkv * ceil(M * G / 32) CTAs.
int attn_splits_max(const spec_model_desc& d, int M, int sms) {
  const int G = d.n_q_heads / d.n_kv_heads;
  const int min_ctas = d.n_kv_heads * ((M * G + 31) / 32);
  int s = (2 * sms + min_ctas - 1) / min_ctas;
  if (s < 1) s = 1;
  if (s > 64) s = 64;
  return s;
}

size_t attn_smem_bytes(int dtype, int hd, int qmax) {
  const size_t es = dtype == SPEC_DTYPE_BF16 ? 2 : 4;
  const size_t kp = hd + 16 / es;
  return (size_t)qmax * hd * 4 + (size_t)qmax * 128 * 4 + 128 * kp * es + 128 * hd * es;
}

template <typename TT, int HDV, int QM>
static spec_status attn_launch(const spec_model_desc& d, const RowInfo& ri, const spec_rows& rows, const void* qbuf,
                               const spec_kv& kv, float* opart, float2* mlpart, void* attn_out, int nsplit, int nqg,
                               void* ws, cudaStream_t st) {
  static int attr_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  const size_t smem = attn_smem_bytes(d.dtype, HDV, QM);
  if (attr_dev != dev) {
    if (cudaFuncSetAttribute(attn_split_kernel<TT, HDV, QM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return SPEC_ERR_CUDA;
    attr_dev = dev;
  }
  dim3 grid(nsplit, d.n_kv_heads, rows.B * nqg);
  const float scale = 1.f / sqrtf((float)d.head_dim);
  launch_pdl(attn_split_kernel<TT, HDV, QM>, dim3(grid), dim3(128), smem, st, (const TT*)qbuf, kv, ri, d.n_q_heads, d.n_kv_heads,
                                                          d.window, nsplit, nqg, scale, opart, mlpart, ws);
  launch_pdl(attn_combine_kernel<TT, HDV>, dim3(rows.M * d.n_q_heads), dim3(HDV), 0, st, opart, mlpart, d.n_q_heads, nsplit,
                                                                     (TT*)attn_out);
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
                             float* opart, float2* mlpart, void* attn_out, int nsplit, void* ws, cudaStream_t st) {
  RowInfo ri = to_rowinfo(rows);
  const int G = d.n_q_heads / d.n_kv_heads;
  const int qmax = attn_qmax(rows.rows_per_req, G);
  const int nqg = (rows.rows_per_req * G + qmax - 1) / qmax;
  spec_status s;
  if (d.dtype == SPEC_DTYPE_BF16) {
    if (d.head_dim == 128)
      s = attn_qdispatch<__nv_bfloat16, 128>(qmax, d, ri, rows, qbuf, kv, opart, mlpart, attn_out, nsplit, nqg, ws, st);
    else if (d.head_dim == 64)
      s = attn_qdispatch<__nv_bfloat16, 64>(qmax, d, ri, rows, qbuf, kv, opart, mlpart, attn_out, nsplit, nqg, ws, st);
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
  launch_pdl(topk_select_kernel, dim3(M), dim3(1024), 0, st, s, V, Kc, out_ids);
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
