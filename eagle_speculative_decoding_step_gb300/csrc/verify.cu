// Verification of drafts against target logits.
//
// [NEURON] "Speculative Decoding (EAGLE3) in the vLLM Neuron Framework",
// section "Rejection Sampling": the on-device greedy sampler (match mask,
// first mismatch, accept through the mismatch emitting the target token, bonus
// token when all match, -1 padding) and the CPU probabilistic sampler
// (arXiv:2211.17192: accept when u <= p(draft) with draft prob 1; recovered
// token by Gumbel-max over the target distribution with the draft token
// removed; bonus token sampled from the target at the last position).
// Tree verification ([EAGLET] introduction: the target verifies the tree in one
// pass): a node is accepted when its parent is and its token equals the
// target's argmax at the parent; the deepest accepted node's path is emitted,
// then its K/V is compacted to contiguous cache indices.
//
// Both verifiers are one streaming read of the fp32 target logits (HBM-bound):
// kernel 1 splits every row into chunks and reduces each chunk (argmax, or
// max / sum-exp / Gumbel key for the stochastic sampler); kernel 2 runs one
// CTA per request over the chunk partials and makes the sequential accept
// decisions, writes the outputs and moves the accepted K/V.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace spec {

struct ArgPart { float v; int i; };
struct RejPart { float m, s, key; int idx; };

static int verify_chunks(int rows, int V) {
  int want = (640 + rows - 1) / rows;
  int cap = V / 4096;
  if (cap < 1) cap = 1;
  if (want > cap) want = cap;
  if (want > 64) want = 64;
  return want < 1 ? 1 : want;
}
static int chunk_len(int V, int nch) { int L = (V + nch - 1) / nch; return (L + 3) & ~3; }

// ---------------------------------------------------------------- greedy argmax
template <bool VEC>
__global__ void __launch_bounds__(256) argmax_chunks_kernel(const float* __restrict__ logits, int V,
                                                           int nch, int L, ArgPart* __restrict__ part) {
  pdl_wait();
  pdl_trigger();
  __shared__ float rv[32];
  __shared__ int ri[32];
  const int row = blockIdx.y, c = blockIdx.x;
  const float* x = logits + (size_t)row * V;
  const int lo = c * L, hi = min(V, lo + L);
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  if (VEC) {
    // four 16-byte loads in flight per thread
    for (int j0 = lo + 4 * threadIdx.x; j0 < hi; j0 += 16 * blockDim.x) {
      float4 q[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + 4 * u * blockDim.x;
        if (j < hi) q[u] = *reinterpret_cast<const float4*>(x + j);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + 4 * u * blockDim.x;
        if (j >= hi) break;
        if (better(q[u].x, j, bv, bi)) { bv = q[u].x; bi = j; }
        if (j + 1 < hi && better(q[u].y, j + 1, bv, bi)) { bv = q[u].y; bi = j + 1; }
        if (j + 2 < hi && better(q[u].z, j + 2, bv, bi)) { bv = q[u].z; bi = j + 2; }
        if (j + 3 < hi && better(q[u].w, j + 3, bv, bi)) { bv = q[u].w; bi = j + 3; }
      }
    }
  } else {
    for (int j = lo + threadIdx.x; j < hi; j += blockDim.x) {
      float q = x[j];
      if (better(q, j, bv, bi)) { bv = q; bi = j; }
    }
  }
  block_argmax(bv, bi, rv, ri);
  if (threadIdx.x == 0) part[(size_t)row * nch + c] = ArgPart{bv, bi};
}

__device__ int merged_argmax(const ArgPart* part, int row, int nch) {
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int c = 0; c < nch; ++c) {
    ArgPart p = part[(size_t)row * nch + c];
    if (better(p.v, p.i, bv, bi)) { bv = p.v; bi = p.i; }
  }
  return bi;
}

// Moves the accepted path's K/V from cache index ctx + src[d] to ctx + d,
// d = 1 .. a, in increasing d (a source index is never below its destination
// and sources increase along the path, so no source is overwritten first).
template <typename T>
__device__ void compact_path(const spec_kv& kv, int b, int ctx, const int* src, int a, int row_elems,
                             void* ws) {
  for (int d = 1; d <= a; ++d) {
    long long s = slot_of(kv, b, ctx + src[d]);
    long long t = slot_of(kv, b, ctx + d);
    if (s < 0 || t < 0) {
      if (threadIdx.x == 0) report(ws, SPEC_ERR_DEVICE, b, d);
    } else if (s != t) {
      T* K = reinterpret_cast<T*>(kv.k);
      T* Vv = reinterpret_cast<T*>(kv.v);
      for (int e = threadIdx.x; e < row_elems; e += blockDim.x) {
        K[t * row_elems + e] = K[s * row_elems + e];
        Vv[t * row_elems + e] = Vv[s * row_elems + e];
      }
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(128) verify_greedy_finalize_kernel(
    int R, int nch, const ArgPart* __restrict__ part, const int32_t* __restrict__ draft,
    const int32_t* __restrict__ parent, int max_depth, int32_t* __restrict__ out,
    int32_t* __restrict__ acc_out, int32_t* __restrict__ kv_src, spec_kv kv, int has_kv,
    int row_elems, int elem_bytes, const int32_t* __restrict__ ctx_len, void* ws) {
  pdl_wait();
  pdl_trigger();
  __shared__ int t[64];
  __shared__ int path[65];
  __shared__ int s_a;
  const int b = blockIdx.x;
  for (int n = threadIdx.x; n < R; n += blockDim.x) t[n] = merged_argmax(part, b * R + n, nch);
  __syncthreads();
  const int W = (parent == nullptr) ? R : max_depth + 1;
  if (threadIdx.x == 0) {
    int a = 0;
    if (parent == nullptr) {
      const int K = R - 1;
      const int32_t* d = draft + (size_t)b * K;
      while (a < K && d[a] == t[a]) ++a;
      for (int i = 0; i < W; ++i) {
        out[(size_t)b * W + i] = i < a ? d[i] : (i == a ? t[a] : -1);
        if (kv_src) kv_src[(size_t)b * W + i] = i <= a ? i : -1;
      }
      path[0] = 0;
    } else {
      const int32_t* tok = draft + (size_t)b * R;
      const int32_t* par = parent + (size_t)b * R;
      unsigned long long accepted = 1ull;   // R <= 64
      int depth[64];
      depth[0] = 0;
      int best = 0;
      for (int n = 1; n < R; ++n) {
        int p = par[n];
        if (p < 0 || p >= n) {
          report(ws, SPEC_ERR_DEVICE, b, n);
          depth[n] = 0;
          continue;
        }
        depth[n] = depth[p] + 1;
        if (((accepted >> p) & 1ull) && tok[n] == t[p]) {
          accepted |= 1ull << n;
          if (depth[n] > depth[best]) best = n;
        }
      }
      a = depth[best];
      if (a > max_depth) {
        report(ws, SPEC_ERR_DEVICE, b, a);
        a = max_depth;
      }
      int n = best;
      for (int dd = depth[best]; dd > 0; --dd) {
        if (dd <= a) path[dd] = n;
        n = par[n];
      }
      path[0] = 0;
      for (int i = 0; i < W; ++i) {
        int o = -1;
        if (i < a) o = tok[path[i + 1]];
        else if (i == a) o = t[best];
        out[(size_t)b * W + i] = o;
        if (kv_src) kv_src[(size_t)b * W + i] = i <= a ? path[i] : -1;
      }
    }
    acc_out[b] = a;
    s_a = a;
  }
  __syncthreads();
  if (parent != nullptr && has_kv) {
    const int ctx = ctx_len[b];
    if (elem_bytes == 2)
      compact_path<__nv_bfloat16>(kv, b, ctx, path, s_a, row_elems, ws);
    else
      compact_path<float>(kv, b, ctx, path, s_a, row_elems, ws);
  }
}

// ---------------------------------------------------------------- top-k / top-p
// Per-row kept set of a filtered target distribution, as a threshold in the
// order (value desc, id asc): token x is kept iff key(x) > key or (key(x) == key
// and x <= id), key() being an order-preserving map of logit / T.
struct Thr { uint32_t key; int id; };

SPEC_DEV uint32_t okey(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
SPEC_DEV bool kept_by(const Thr& t, uint32_t k, int x) { return k > t.key || (k == t.key && x <= t.id); }

// id of the `need`-th (1-based) smallest index x with key(x) == kk that `inside`
// accepts; block-wide ordered scan (ballots per 1024-wide chunk)
template <typename F>
__device__ int nth_tie_id(const float* x, float T, int V, uint32_t kk, int need, F inside, int* wcount, int* s_taken,
                          int* s_id) {
  const int tid = threadIdx.x;
  if (tid == 0) { *s_taken = 0; *s_id = 0x7fffffff; }
  __syncthreads();
  for (int base = 0; base < V; base += blockDim.x) {
    const int v = base + tid;
    bool eq = false;
    if (v < V) {
      const uint32_t k = okey(x[v] / T);
      eq = (k == kk) && inside(k, v);
    }
    const unsigned bal = __ballot_sync(0xffffffffu, eq);
    if ((tid & 31) == 0) wcount[tid >> 5] = __popc(bal);
    __syncthreads();
    int before = 0;
    for (int w = 0; w < (tid >> 5); ++w) before += wcount[w];
    before += __popc(bal & ((1u << (tid & 31)) - 1u));
    const int taken = *s_taken;
    if (eq && taken + before + 1 == need) *s_id = v;
    __syncthreads();
    if (tid == 0) {
      int tot = 0;
      for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += wcount[w];
      *s_taken = taken + tot;
    }
    __syncthreads();
    if (*s_taken >= need) break;
  }
  return *s_id;
}

// One CTA (1024 threads) per row.  top-k: exact radix selection of the k-th key
// and the id of the last tie kept.  top-p (within the top-k set): radix search
// of the shortest prefix whose probability mass reaches top_p, masses
// exp(y - max) in 2^-40 fixed point so the sums do not depend on thread order.
__global__ void __launch_bounds__(1024) reject_threshold_kernel(const float* __restrict__ logits, int K, int V,
                                                                const float* __restrict__ temperature,
                                                                const int32_t* __restrict__ top_k,
                                                                const float* __restrict__ top_p, Thr* __restrict__ thr) {
  pdl_wait();
  pdl_trigger();
  __shared__ unsigned long long hist[256];
  __shared__ uint32_t s_prefix;
  __shared__ unsigned long long s_need;
  __shared__ int wcount[32];
  __shared__ int s_taken, s_id;
  __shared__ float red[32];
  __shared__ unsigned long long s_tot;
  const int row = blockIdx.x;
  const int b = row / (K + 1);
  const int tid = threadIdx.x;
  const float T = temperature[b];
  const int kk_req = top_k ? top_k[b] : 0;
  const float pp = top_p ? top_p[b] : 1.f;
  Thr t{0u, 0x7fffffff};                       // keep everything
  const bool do_k = T > 0.f && kk_req > 0 && kk_req < V;
  const bool do_p = T > 0.f && pp < 1.f;
  if (!do_k && !do_p) {
    if (tid == 0) thr[row] = t;
    return;
  }
  const float* x = logits + (size_t)row * V;
  if (do_k) {
    if (tid == 0) { s_prefix = 0; s_need = (unsigned long long)kk_req; }
    __syncthreads();
    for (int shift = 24; shift >= 0; shift -= 8) {
      if (tid < 256) hist[tid] = 0;
      __syncthreads();
      const uint32_t prefix = s_prefix;
      const uint32_t pmask = (shift == 24) ? 0u : (0xffffffffu << (shift + 8));
      for (int v = tid; v < V; v += blockDim.x) {
        const uint32_t k = okey(x[v] / T);
        if ((k & pmask) == (prefix & pmask)) atomicAdd(&hist[(k >> shift) & 0xff], 1ull);
      }
      __syncthreads();
      if (tid == 0) {
        unsigned long long need = s_need, acc = 0;
        int dsel = 0;
        for (int d = 255; d >= 0; --d) {
          if (acc + hist[d] >= need) { dsel = d; break; }
          acc += hist[d];
        }
        s_need = need - acc;
        s_prefix = prefix | ((uint32_t)dsel << shift);
      }
      __syncthreads();
    }
    t.key = s_prefix;
    const int need = (int)s_need;
    t.id = nth_tie_id(x, T, V, t.key, need, [](uint32_t, int) { return true; }, wcount, &s_taken, &s_id);
  }
  if (do_p) {
    const Thr tk = t;
    float mx = -INFINITY;
    for (int v = tid; v < V; v += blockDim.x) mx = fmaxf(mx, x[v] / T);
    mx = block_max(mx, red);
    const double scale = 1099511627776.0;     // 2^40
    if (tid == 0) s_tot = 0;
    __syncthreads();
    unsigned long long z = 0;
    for (int v = tid; v < V; v += blockDim.x) {
      const float y = x[v] / T;
      if (kept_by(tk, okey(y), v)) z += (unsigned long long)((double)expf(y - mx) * scale + 0.5);
    }
    atomicAdd(&s_tot, z);
    __syncthreads();
    if (tid == 0) {
      s_prefix = 0;
      s_need = (unsigned long long)ceil((double)pp * (double)s_tot);
      if (s_need == 0) s_need = 1;
    }
    __syncthreads();
    for (int shift = 24; shift >= 0; shift -= 8) {
      if (tid < 256) hist[tid] = 0;
      __syncthreads();
      const uint32_t prefix = s_prefix;
      const uint32_t pmask = (shift == 24) ? 0u : (0xffffffffu << (shift + 8));
      for (int v = tid; v < V; v += blockDim.x) {
        const float y = x[v] / T;
        const uint32_t k = okey(y);
        if ((k & pmask) == (prefix & pmask) && kept_by(tk, k, v))
          atomicAdd(&hist[(k >> shift) & 0xff], (unsigned long long)((double)expf(y - mx) * scale + 0.5));
      }
      __syncthreads();
      if (tid == 0) {
        unsigned long long need = s_need, acc = 0;
        int dsel = 0;
        for (int d = 255; d >= 0; --d) {
          if (hist[d] && acc + hist[d] >= need) { dsel = d; break; }
          acc += hist[d];
          dsel = d;
        }
        s_need = need > acc ? need - acc : 1;
        s_prefix = prefix | ((uint32_t)dsel << shift);
      }
      __syncthreads();
    }
    const uint32_t vkey = s_prefix;
    // every tie at vkey has the same mass; take as many (smallest ids first) as the
    // remaining mass needs
    float yv = 0.f;
    {
      const uint32_t u = (vkey & 0x80000000u) ? (vkey & 0x7fffffffu) : ~vkey;
      yv = __uint_as_float(u);
    }
    const unsigned long long each = (unsigned long long)((double)expf(yv - mx) * scale + 0.5);
    int need = each ? (int)((s_need + each - 1) / each) : 1;
    if (need < 1) need = 1;
    t.key = vkey;
    t.id = nth_tie_id(x, T, V, vkey, need, [tk](uint32_t k, int v) { return kept_by(tk, k, v); }, wcount,
                      &s_taken, &s_id);
  }
  if (tid == 0) thr[row] = t;
}

// ---------------------------------------------------------------- rejection
// Two streaming passes instead of one heavy one.  The accept tests need, per
// row, only the log-sum-exp of the (filtered, tempered) target distribution;
// the Gumbel sample is needed on one row per request: the first rejected
// position, or row K for the bonus token.  So:
//  1. rej_stats_kernel: every row, chunked -- max / sum-exp over the kept
//     tokens (greedy rows: argmax);
//  2. rej_decide_kernel: one warp per request -- merges the chunks row by row
//     and makes the sequential accept decisions (greedy: draft == argmax),
//     writes accept_len, the accepted drafts, -1 padding, kv_src, and for
//     greedy requests the emitted token;
//  3. rej_sample_kernel: the sampled row of every stochastic request, chunked
//     -- Philox noise and the Gumbel-max key over the kept tokens, the draft
//     token excluded on a rejected row (its records go where that request's
//     row statistics were, no longer needed);
//  4. rej_emit_kernel: merges the chunk keys, writes the emitted token.
template <bool VEC>
__global__ void __launch_bounds__(256) rej_stats_kernel(const float* __restrict__ logits, int K, int V, int nch,
                                                        int L, const float* __restrict__ temperature,
                                                        RejPart* __restrict__ part, const Thr* __restrict__ thr) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[32];
  __shared__ int redi[32];
  const int row = blockIdx.y, c = blockIdx.x;
  const Thr tr = thr ? thr[row] : Thr{0u, 0x7fffffff};
  const int b = row / (K + 1);
  const float T = temperature[b];
  const bool greedy = !(T > 0.f);
  const bool unit = T == 1.f;                 // y = l / 1 exactly: skip the division
  const bool filt = thr != nullptr;
  const float* x = logits + (size_t)row * V;
  const int lo = c * L, hi = min(V, lo + L);
  float m = -INFINITY, s = 0.f, bk = -INFINITY;
  int bi = 0x7fffffff;
  constexpr int UNR = 4;                      // 16-byte loads in flight per thread
  for (int j0 = lo + 4 * threadIdx.x; j0 < hi; j0 += 4 * UNR * blockDim.x) {
    float vv[UNR][4];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int j = j0 + 4 * u * blockDim.x;
      if (VEC) {
        if (j < hi) {
          const float4 q = *reinterpret_cast<const float4*>(x + j);
          vv[u][0] = q.x; vv[u][1] = q.y; vv[u][2] = q.z; vv[u][3] = q.w;
        }
      } else {
#pragma unroll
        for (int l = 0; l < 4; ++l) vv[u][l] = (j + l < hi) ? x[j + l] : -INFINITY;
      }
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int j = j0 + 4 * u * blockDim.x;
      if (j >= hi) break;
      const float* v = vv[u];
      if (greedy) {
#pragma unroll
        for (int l = 0; l < 4; ++l)
          if (j + l < hi && better(v[l], j + l, bk, bi)) { bk = v[l]; bi = j + l; }
        continue;
      }
      // the group's kept values, -inf for the rest (ids past hi, filtered by top-k / top-p)
      float y[4];
#pragma unroll
      for (int l = 0; l < 4; ++l) {
        y[l] = (j + l < hi) ? (unit ? v[l] : v[l] / T) : -INFINITY;
        if (filt && y[l] > -INFINITY && !kept_by(tr, okey(y[l]), j + l)) y[l] = -INFINITY;
      }
      // online sum of exp: one max update per group of four
      const float gm = fmaxf(fmaxf(y[0], y[1]), fmaxf(y[2], y[3]));
      if (gm > m) {
        s *= __expf(m - gm);
        m = gm;
      }
      if (m > -INFINITY) s += (__expf(y[0] - m) + __expf(y[1] - m)) + (__expf(y[2] - m) + __expf(y[3] - m));
    }
  }
  const float bm = block_max(m, red);
  const float contrib = (m == -INFINITY) ? 0.f : s * expf(m - bm);
  const float bs = block_sum(contrib, red);
  block_argmax(bk, bi, red, redi);
  if (threadIdx.x == 0) part[(size_t)row * nch + c] = RejPart{bm, bs, bk, bi};
}

__global__ void __launch_bounds__(32) rej_decide_kernel(
    const float* __restrict__ logits, int K, int V, int nch, const RejPart* __restrict__ part,
    const int32_t* __restrict__ draft, const float* __restrict__ temperature, uint2 key, uint32_t ctr_w0,
    int32_t* __restrict__ out, int32_t* __restrict__ acc_out, int32_t* __restrict__ kv_src,
    const Thr* __restrict__ thr) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x, lane = threadIdx.x;
  const float T = temperature[b];
  const bool greedy = !(T > 0.f);
  int a = 0, emitted = -1;
  for (int i = 0; i <= K; ++i) {
    const size_t row = (size_t)b * (K + 1) + i;
    // merge the row's chunk records (lane c takes chunks c, c + 32, ...)
    float M = -INFINITY, bk = -INFINITY;
    int bi = 0x7fffffff;
    for (int c = lane; c < nch; c += 32) {
      const RejPart p = part[row * nch + c];
      M = fmaxf(M, p.m);
      if (better(p.key, p.idx, bk, bi)) { bk = p.key; bi = p.idx; }
    }
    M = warp_max(M);
    warp_argmax(bk, bi);
    float S = 0.f;
    for (int c = lane; c < nch; c += 32) {
      const RejPart p = part[row * nch + c];
      if (p.m > -INFINITY) S += p.s * expf(p.m - M);
    }
    S = warp_sum(S);
    if (i == K) {
      if (greedy) emitted = bi;
      break;
    }
    const int d = draft[(size_t)b * K + i];
    bool ok;
    if (greedy) {
      ok = (d == bi);
    } else {
      const float lse = M + logf(S);
      float pd = 0.f;
      if (d >= 0 && d < V) {
        const float yd = logits[row * V + d] / T;
        const Thr tr = thr ? thr[row] : Thr{0u, 0x7fffffff};
        if (kept_by(tr, okey(yd), d)) pd = expf(yd - lse);
      }
      const uint4 r = philox4x32_10(make_uint4(0u, (uint32_t)i, (uint32_t)b, ctr_w0), key);
      ok = word_to_uniform(r.x) <= pd;
    }
    if (!ok) {
      if (greedy) emitted = bi;
      break;
    }
    ++a;
  }
  for (int i = lane; i <= K; i += 32) {
    if (i != a || greedy) out[(size_t)b * (K + 1) + i] = i < a ? draft[(size_t)b * K + i] : (i == a ? emitted : -1);
    if (kv_src) kv_src[(size_t)b * (K + 1) + i] = i <= a ? i : -1;
  }
  if (lane == 0) acc_out[b] = a;
}

template <bool VEC>
__global__ void __launch_bounds__(256) rej_sample_kernel(const float* __restrict__ logits, int K, int V, int nchs,
                                                         int L, int region, const int32_t* __restrict__ draft,
                                                         const float* __restrict__ temperature, uint2 key,
                                                         uint32_t ctr_w, const int32_t* __restrict__ acc_in,
                                                         RejPart* __restrict__ part, const Thr* __restrict__ thr) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[32];
  __shared__ int redi[32];
  const int b = blockIdx.y, c = blockIdx.x;
  const float T = temperature[b];
  if (!(T > 0.f)) return;                     // greedy requests were settled by the decision kernel
  const int i = acc_in[b];
  const int row = b * (K + 1) + i;
  const Thr tr = thr ? thr[row] : Thr{0u, 0x7fffffff};
  const bool unit = T == 1.f;
  const int excl = i < K ? draft[(size_t)b * K + i] : -1;
  const float* x = logits + (size_t)row * V;
  const int lo = c * L, hi = min(V, lo + L);
  float bk = -INFINITY;
  int bi = 0x7fffffff;
  // every thread handles aligned groups of 4 vocabulary ids = one Philox block
  for (int j = lo + 4 * threadIdx.x; j < hi; j += 4 * blockDim.x) {
    float v[4];
    if (VEC) {
      float4 q = *reinterpret_cast<const float4*>(x + j);
      v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
    } else {
#pragma unroll
      for (int l = 0; l < 4; ++l) v[l] = (j + l < hi) ? x[j + l] : -INFINITY;
    }
    const uint4 r = philox4x32_10(make_uint4((uint32_t)(j >> 2), (uint32_t)i, (uint32_t)b, ctr_w), key);
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int l = 0; l < 4; ++l) {
      if (j + l >= hi) break;
      const float y = unit ? v[l] : v[l] / T;
      if (j + l == excl || !kept_by(tr, okey(y), j + l)) continue;
      const float g = y - logf(-logf(word_to_uniform(w[l])));
      if (better(g, j + l, bk, bi)) { bk = g; bi = j + l; }
    }
  }
  block_argmax(bk, bi, red, redi);
  if (threadIdx.x == 0) part[(size_t)b * region + c] = RejPart{0.f, 0.f, bk, bi};
}

__global__ void __launch_bounds__(32) rej_emit_kernel(int K, int nchs, int region, const RejPart* __restrict__ part,
                                                      const float* __restrict__ temperature,
                                                      const int32_t* __restrict__ acc_in, int32_t* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x, lane = threadIdx.x;
  if (!(temperature[b] > 0.f)) return;
  float bk = -INFINITY;
  int bi = 0x7fffffff;
  for (int c = lane; c < nchs; c += 32) {
    const RejPart p = part[(size_t)b * region + c];
    if (better(p.key, p.idx, bk, bi)) { bk = p.key; bi = p.idx; }
  }
  warp_argmax(bk, bi);
  if (lane == 0) out[(size_t)b * (K + 1) + acc_in[b]] = bi;
}

}  // namespace spec

using namespace spec;

extern "C" size_t spec_verify_workspace_bytes(int32_t B, int32_t R, int32_t V) {
  if (B <= 0 || R <= 0 || V <= 0) return 0;
  int rows = B * R;
  int nch = verify_chunks(rows, V);
  return kWsHeader + align_up((size_t)rows * nch * sizeof(RejPart), 256) + align_up((size_t)rows * sizeof(Thr), 256);
}

extern "C" spec_status spec_verify_greedy(int32_t B, int32_t R, int32_t V, const float* target_logits,
                                          const int32_t* draft_tok, const int32_t* parent,
                                          int32_t max_depth, int32_t* out_tok, int32_t* accept_len,
                                          int32_t* kv_src, const spec_model_desc* desc,
                                          const spec_kv* kv, const int32_t* ctx_len, void* ws,
                                          size_t ws_bytes, spec_stream_t stream) {
  if (B <= 0 || R <= 0 || V <= 0) return SPEC_ERR_SHAPE;
  if (!target_logits || !draft_tok || !out_tok || !accept_len) return SPEC_ERR_ARG;
  if (R > 64) return SPEC_ERR_CAPACITY;
  if (parent == nullptr && R < 2) return SPEC_ERR_SHAPE;
  if (parent != nullptr && (max_depth < 0 || max_depth >= 64)) return SPEC_ERR_SHAPE;
  if (!ws || !aligned(ws, 256) || ws_bytes < spec_verify_workspace_bytes(B, R, V)) return SPEC_ERR_WORKSPACE;
  int has_kv = 0, row_elems = 0, elem_bytes = 4;
  spec_kv kvv{};
  if (parent != nullptr && kv != nullptr) {
    if (!desc || !ctx_len || !kv->k || !kv->v || !kv->block_table) return SPEC_ERR_ARG;
    if (kv->block_size <= 0 || kv->max_blocks <= 0 || kv->num_slots <= 0) return SPEC_ERR_SHAPE;
    has_kv = 1;
    kvv = *kv;
    row_elems = desc->n_kv_heads * desc->head_dim;
    elem_bytes = desc->dtype == SPEC_DTYPE_BF16 ? 2 : 4;
  }
  const int rows = B * R;
  const int nch = verify_chunks(rows, V);
  const int L = chunk_len(V, nch);
  ArgPart* part = reinterpret_cast<ArgPart*>(static_cast<char*>(ws) + kWsHeader);
  dim3 grid(nch, rows);
  const bool vec = (V % 4 == 0) && aligned(target_logits, 16);
  if (vec)
    launch_pdl(argmax_chunks_kernel<true>, dim3(grid), dim3(256), 0, stream, target_logits, V, nch, L, part);
  else
    launch_pdl(argmax_chunks_kernel<false>, dim3(grid), dim3(256), 0, stream, target_logits, V, nch, L, part);
  launch_pdl(verify_greedy_finalize_kernel, dim3(B), dim3(128), 0, stream, R, nch, part, draft_tok, parent, max_depth, out_tok,
                                                       accept_len, kv_src, kvv, has_kv, row_elems, elem_bytes,
                                                       ctx_len, ws);
  return last_launch();
}

extern "C" spec_status spec_verify_rejection(int32_t B, int32_t K, int32_t V, const float* target_logits,
                                             const int32_t* draft_tok, const float* temperature,
                                             const int32_t* top_k, const float* top_p,
                                             uint64_t seed, uint64_t step_offset, int32_t* out_tok,
                                             int32_t* accept_len, int32_t* kv_src, void* ws,
                                             size_t ws_bytes, spec_stream_t stream) {
  if (B <= 0 || K <= 0 || V <= 0) return SPEC_ERR_SHAPE;
  if (!target_logits || !draft_tok || !temperature || !out_tok || !accept_len) return SPEC_ERR_ARG;
  const int R = K + 1;
  if (!ws || !aligned(ws, 256) || ws_bytes < spec_verify_workspace_bytes(B, R, V)) return SPEC_ERR_WORKSPACE;
  const int rows = B * R;
  const int nch = verify_chunks(rows, V);
  const int L = chunk_len(V, nch);
  RejPart* part = reinterpret_cast<RejPart*>(static_cast<char*>(ws) + kWsHeader);
  uint2 key = make_uint2((uint32_t)(seed & 0xffffffffull), (uint32_t)(seed >> 32));
  uint32_t w0 = (uint32_t)((2ull * step_offset) & 0xffffffffull);
  Thr* thr = nullptr;
  if (top_k || top_p) {
    thr = reinterpret_cast<Thr*>(reinterpret_cast<char*>(part) + align_up((size_t)rows * nch * sizeof(RejPart), 256));
    launch_pdl(reject_threshold_kernel, dim3(rows), dim3(1024), 0, stream, target_logits, K, V, temperature, top_k,
               top_p, thr);
  }
  const bool vec = (V % 4 == 0) && aligned(target_logits, 16);
  if (vec)
    launch_pdl(rej_stats_kernel<true>, dim3(nch, rows), dim3(256), 0, stream, target_logits, K, V, nch, L, temperature,
               part, (const Thr*)thr);
  else
    launch_pdl(rej_stats_kernel<false>, dim3(nch, rows), dim3(256), 0, stream, target_logits, K, V, nch, L,
               temperature, part, (const Thr*)thr);
  launch_pdl(rej_decide_kernel, dim3(B), dim3(32), 0, stream, target_logits, K, V, nch, (const RejPart*)part,
             draft_tok, temperature, key, w0, out_tok, accept_len, kv_src, (const Thr*)thr);
  // the sampled rows: one per request, chunked over the CTAs; each request's records
  // take the slots of its (now consumed) row statistics
  const int region = R * nch;
  int nchs = std::min(region, std::max(1, (640 + B - 1) / B));
  nchs = std::min(nchs, std::max(1, V / 2048));
  const int Ls = chunk_len(V, nchs);
  if (vec)
    launch_pdl(rej_sample_kernel<true>, dim3(nchs, B), dim3(256), 0, stream, target_logits, K, V, nchs, Ls, region,
               draft_tok, temperature, key, w0 + 1u, (const int32_t*)accept_len, part, (const Thr*)thr);
  else
    launch_pdl(rej_sample_kernel<false>, dim3(nchs, B), dim3(256), 0, stream, target_logits, K, V, nchs, Ls, region,
               draft_tok, temperature, key, w0 + 1u, (const int32_t*)accept_len, part, (const Thr*)thr);
  launch_pdl(rej_emit_kernel, dim3(B), dim3(32), 0, stream, K, nchs, region, (const RejPart*)part, temperature,
             (const int32_t*)accept_len, out_tok);
  return last_launch();
}

// ---------------------------------------------------------------- no-allocation variant
// Some callers cannot allocate device memory at all: a host framework that owns
// every device buffer and hands the verifier only its inputs and outputs, code
// that runs where cudaMalloc is forbidden because it synchronises the device
// (latency-critical serving loops), or plugins that see no allocator.  For them
// spec_verify_greedy_static keeps its scratch in a fixed array in device memory
// that is part of the loaded library (every GPU that loads the library holds it
// until the process exits).
namespace spec {
constexpr size_t kStaticVerifyScratch = 256 * 1024;     // header + chunk partials
static __device__ __align__(256) unsigned char g_verify_scratch[kStaticVerifyScratch];
constexpr int kStaticMaxDevices = 64;
static void* g_verify_scratch_addr[kStaticMaxDevices];
static std::mutex g_verify_scratch_mu;

// Device address of the scratch array on the current device (looked up once per
// device, with that device current).  nullptr if the lookup fails.
static void* static_verify_scratch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kStaticMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_verify_scratch_mu);
  if (g_verify_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_verify_scratch) != cudaSuccess) return nullptr;
    g_verify_scratch_addr[dev] = p;
  }
  return g_verify_scratch_addr[dev];
}
}  // namespace spec

extern "C" spec_status spec_verify_greedy_static(int32_t B, int32_t R, int32_t V, const float* target_logits,
                                                 const int32_t* draft_tok, const int32_t* parent,
                                                 int32_t max_depth, int32_t* out_tok, int32_t* accept_len,
                                                 int32_t* kv_src, const spec_model_desc* desc, const spec_kv* kv,
                                                 const int32_t* ctx_len, spec_stream_t stream) {
  if (B <= 0 || R <= 0 || V <= 0) return SPEC_ERR_SHAPE;
  if (!target_logits || !draft_tok || !out_tok || !accept_len) return SPEC_ERR_ARG;
  if (R > 64) return SPEC_ERR_CAPACITY;
  if (parent == nullptr && R < 2) return SPEC_ERR_SHAPE;
  if (parent != nullptr && (max_depth < 0 || max_depth >= 64)) return SPEC_ERR_SHAPE;
  // the same scratch layout as the workspace version must fit the fixed array
  if (spec_verify_workspace_bytes(B, R, V) > kStaticVerifyScratch) return SPEC_ERR_CAPACITY;
  int has_kv = 0, row_elems = 0, elem_bytes = 4;
  spec_kv kvv{};
  if (parent != nullptr && kv != nullptr) {
    if (!desc || !ctx_len || !kv->k || !kv->v || !kv->block_table) return SPEC_ERR_ARG;
    if (kv->block_size <= 0 || kv->max_blocks <= 0 || kv->num_slots <= 0) return SPEC_ERR_SHAPE;
    has_kv = 1;
    kvv = *kv;
    row_elems = desc->n_kv_heads * desc->head_dim;
    elem_bytes = desc->dtype == SPEC_DTYPE_BF16 ? 2 : 4;
  }
  void* ws = static_verify_scratch();
  if (ws == nullptr) return SPEC_ERR_CUDA;
  // the array keeps the previous call's contents: the error header starts at zero;
  // every chunk partial is rewritten before it is read
  if (cudaMemsetAsync(ws, 0, kWsHeader, stream) != cudaSuccess) return SPEC_ERR_CUDA;
  const int rows = B * R;
  const int nch = verify_chunks(rows, V);
  const int L = chunk_len(V, nch);
  ArgPart* part = reinterpret_cast<ArgPart*>(static_cast<char*>(ws) + kWsHeader);
  dim3 grid(nch, rows);
  const bool vec = (V % 4 == 0) && aligned(target_logits, 16);
  if (vec)
    launch_pdl(argmax_chunks_kernel<true>, dim3(grid), dim3(256), 0, stream, target_logits, V, nch, L, part);
  else
    launch_pdl(argmax_chunks_kernel<false>, dim3(grid), dim3(256), 0, stream, target_logits, V, nch, L, part);
  launch_pdl(verify_greedy_finalize_kernel, dim3(B), dim3(128), 0, stream, R, nch, part, draft_tok, parent, max_depth, out_tok,
                                                       accept_len, kv_src, kvv, has_kv, row_elems, elem_bytes,
                                                       ctx_len, ws);
  return last_launch();
}
