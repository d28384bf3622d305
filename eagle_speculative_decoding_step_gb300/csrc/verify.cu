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
#include "tc_core.cuh"

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

// ---------------------------------------------------------------- control words
// After the header, a verifier workspace holds its completion counters (zero
// when idle; every kernel that raises one sets it back to zero before it
// finishes, so a zero-filled workspace stays ready for the next call):
//   ticket, finished  -- rejection: start-order tickets / finished CTAs;
//   cnt[B]            -- chunk CTAs of request b that finished their statistics;
//   scnt[B]           -- sampling CTAs of request b that finished;
//   decided[B]        -- rejection: request b's decision is published.
// Header bytes 64..71 are two knobs a caller may set (zero = default): the
// bound on a sampling CTA's wait in microseconds, and a test hook that keeps
// request (value - 1)'s decision unpublished so its waits run out.
struct VerifyCtl { int ticket, finished; };
constexpr size_t kKnobWait = 64, kKnobWithhold = 68;
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;     // 2 s

static size_t ctl_bytes(int B) { return align_up(sizeof(VerifyCtl) + (size_t)B * 3 * sizeof(int), 256); }

SPEC_DEV int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
SPEC_DEV void st_release(int* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Thread 0 of a CTA that finished its share of request b: true for the last of
// `total` CTAs of that request (the counter is reset by the caller of this when
// it is done).  Every earlier CTA's writes are visible to the last one.
__device__ bool last_arrival(int* counter, int total, int* s_flag) {
  if (threadIdx.x == 0) {
    __threadfence();
    const int n = atomicAdd(counter, 1);
    *s_flag = (n == total - 1);
    if (*s_flag) __threadfence();
  }
  __syncthreads();
  return *s_flag != 0;
}

// ---------------------------------------------------------------- chunk streaming
// A chunk [lo, hi) of a 16-byte aligned fp32 row (lo and hi - lo multiples of 4)
// passes through a ring of kVStages shared-memory stages of kVStage floats that
// thread 0 fills with bulk copies (cp.async.bulk) kVStages ahead, so the
// copies in flight do not depend on registers.  Thread t calls f(j, v) for the
// 4-float group at offset 4t + 1024u (u < 4) of every stage: the same
// thread-to-element order as a loop of four 16-byte loads per thread over the
// chunk.  256 threads.  Every wait is bounded (2 s); the block leaves the loop
// together (a vote per stage), waits for the copies it issued and returns false.
constexpr int kVStages = 4, kVStage = 4096;
constexpr int kVStreamMin = 4 * kVStage;     // shorter chunks keep the register loop
constexpr size_t kVRingBytes = (size_t)kVStages * kVStage * 4 + 8 * kVStages;

template <class F>
__device__ bool stream_chunk(const float* __restrict__ x, int lo, int hi, uint8_t* ring, F&& f) {
  float* buf = reinterpret_cast<float*>(ring);
  const uint32_t bar0 = tc::su32(ring + (size_t)kVStages * kVStage * 4);
  __shared__ int s_abort;
  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int i = 0; i < kVStages; ++i) tc::mbar_init(bar0 + 8u * i, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int nst = (hi - lo + kVStage - 1) / kVStage;
  auto issue = [&](int k) {
    const int base = lo + k * kVStage;
    const uint32_t bytes = (uint32_t)min(kVStage, hi - base) * 4u;
    const uint32_t bar = bar0 + 8u * (uint32_t)(k % kVStages);
    tc::mbar_expect_tx(bar, bytes);
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(tc::su32(buf + (size_t)(k % kVStages) * kVStage)), "l"(x + base), "r"(bytes), "r"(bar)
                 : "memory");
  };
  if (threadIdx.x == 0)
    for (int k = 0; k < min(kVStages, nst); ++k) issue(k);
  int k = 0;
  for (; k < nst; ++k) {
    const int slot = k % kVStages;
    const bool w = tc::mbar_wait(bar0 + 8u * slot, (uint32_t)(k / kVStages) & 1u, &s_abort);
    if (w) {
      const int base = lo + k * kVStage, n = min(kVStage, hi - base);
      const float* sb = buf + (size_t)slot * kVStage;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int o = 4 * threadIdx.x + 1024 * u;
        if (o >= n) break;
        const float4 q = *reinterpret_cast<const float4*>(sb + o);
        const float v[4] = {q.x, q.y, q.z, q.w};
        f(base + o, v);
      }
    }
    if (!__syncthreads_and(w)) break;          // every thread is done with the slot
    if (threadIdx.x == 0 && k + kVStages < nst) issue(k + kVStages);
  }
  if (k == nst) return true;
  // the copies issued for stages k .. min(k + kVStages, nst) - 1 land before the
  // shared memory is given up
  if (threadIdx.x == 0)
    for (int q = k; q < min(k + kVStages, nst); ++q)
      tc::mbar_wait(bar0 + 8u * (uint32_t)(q % kVStages), (uint32_t)(q / kVStages) & 1u, &s_abort, false);
  __syncthreads();
  return false;
}

// ---------------------------------------------------------------- greedy
// One launch: CTA (c, row) reduces chunk c of a logits row to its argmax; the
// last CTA of a request to finish (completion counter, no waiting) merges the
// request's chunk records, makes the sequential accept decisions, writes the
// outputs and moves the accepted K/V.
__device__ int merged_argmax(const ArgPart* part, int row, int nch) {
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int c = 0; c < nch; ++c) {
    const float v = __ldcg(&part[(size_t)row * nch + c].v);
    const int i = __ldcg(&part[(size_t)row * nch + c].i);
    if (better(v, i, bv, bi)) { bv = v; bi = i; }
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

// Chunk records of one request the deciding CTA stages in shared memory at once
// (more are read row by row).
constexpr int kStageRecs = 1024;

struct GreedyArgs {
  const float* logits;
  int V, R, nch, L;
  ArgPart* part;
  long long part_cap;        // chunk records the scratch holds (a larger index is not written)
  int* cnt;
  const int32_t* draft;
  const int32_t* parent;
  int max_depth;
  int32_t* out;
  int32_t* acc_out;
  int32_t* kv_src;
  spec_kv kv;
  int has_kv, row_elems, elem_bytes;
  const int32_t* ctx_len;
  void* ws;
};

template <bool VEC>
__global__ void __launch_bounds__(256) verify_greedy_kernel(GreedyArgs g) {
  SPEC_TL(spec::kTLGreedy);
  pdl_wait();
  pdl_trigger();
  __shared__ float rv[32];
  __shared__ int ri[32];
  __shared__ int t[64];
  __shared__ int path[65];
  __shared__ int s_a, s_last;
  const int row = blockIdx.y, c = blockIdx.x;
  const int V = g.V, R = g.R;
  const float* x = g.logits + (size_t)row * V;
  const int lo = c * g.L, hi = min(V, lo + g.L);
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  if (VEC && g.L >= kVStreamMin) {
    extern __shared__ __align__(128) uint8_t vring[];   // chunk ring (kVRingBytes)
    const bool ok = stream_chunk(x, lo, hi, vring, [&](int j, const float* v) {
#pragma unroll
      for (int l = 0; l < 4; ++l)
        if (better(v[l], j + l, bv, bi)) { bv = v[l]; bi = j + l; }
    });
    if (!ok && threadIdx.x == 0) report(g.ws, SPEC_ERR_TIMEOUT, row, c);
  } else if (VEC) {
    // short chunks: four 16-byte loads in flight per thread
    for (int j0 = lo + 4 * threadIdx.x; j0 < hi; j0 += 16 * blockDim.x) {
      float4 q[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + 4 * u * blockDim.x;
        if (j < hi) q[u] = __ldcs(reinterpret_cast<const float4*>(x + j));
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + 4 * u * blockDim.x;
        if (j >= hi) break;
        if (better(q[u].x, j, bv, bi)) { bv = q[u].x; bi = j; }
        if (better(q[u].y, j + 1, bv, bi)) { bv = q[u].y; bi = j + 1; }
        if (better(q[u].z, j + 2, bv, bi)) { bv = q[u].z; bi = j + 2; }
        if (better(q[u].w, j + 3, bv, bi)) { bv = q[u].w; bi = j + 3; }
      }
    }
  } else {
    for (int j = lo + threadIdx.x; j < hi; j += blockDim.x) {
      float q = x[j];
      if (better(q, j, bv, bi)) { bv = q; bi = j; }
    }
  }
  block_argmax(bv, bi, rv, ri);
  if (threadIdx.x == 0) {
    const long long at = (long long)row * g.nch + c;
    if (at < g.part_cap) g.part[at] = ArgPart{bv, bi};
    else report(g.ws, SPEC_ERR_CAPACITY, row, c);
  }
  const int b = row / R;
  if (!last_arrival(&g.cnt[b], R * g.nch, &s_last)) return;

  // ---- the request's last CTA: decisions, outputs, K/V compaction
  if (R * g.nch <= kStageRecs) {
    // every chunk record of the request loaded at once, then each row merged from
    // shared memory in chunk order
    __shared__ ArgPart s_rec[kStageRecs];
    const ArgPart* src = g.part + (size_t)b * R * g.nch;
    ArgPart rec[kStageRecs / 256];
#pragma unroll
    for (int u = 0; u < kStageRecs / 256; ++u) {
      const int e = threadIdx.x + 256 * u;
      if (e < R * g.nch) rec[u] = ArgPart{__ldcg(&src[e].v), __ldcg(&src[e].i)};
    }
#pragma unroll
    for (int u = 0; u < kStageRecs / 256; ++u) {
      const int e = threadIdx.x + 256 * u;
      if (e < R * g.nch) s_rec[e] = rec[u];
    }
    __syncthreads();
    for (int n = threadIdx.x; n < R; n += blockDim.x) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
      for (int c = 0; c < g.nch; ++c) {
        const ArgPart q = s_rec[n * g.nch + c];
        if (better(q.v, q.i, bv, bi)) { bv = q.v; bi = q.i; }
      }
      t[n] = bi;
    }
  } else {
    for (int n = threadIdx.x; n < R; n += blockDim.x) t[n] = merged_argmax(g.part, b * R + n, g.nch);
  }
  __syncthreads();
  const int W = (g.parent == nullptr) ? R : g.max_depth + 1;
  if (threadIdx.x == 0) {
    int a = 0;
    if (g.parent == nullptr) {
      const int K = R - 1;
      const int32_t* d = g.draft + (size_t)b * K;
      while (a < K && d[a] == t[a]) ++a;
      for (int i = 0; i < W; ++i) {
        g.out[(size_t)b * W + i] = i < a ? d[i] : (i == a ? t[a] : -1);
        if (g.kv_src) g.kv_src[(size_t)b * W + i] = i <= a ? i : -1;
      }
      path[0] = 0;
    } else {
      const int32_t* tok = g.draft + (size_t)b * R;
      const int32_t* par = g.parent + (size_t)b * R;
      unsigned long long accepted = 1ull;   // R <= 64
      int depth[64];
      depth[0] = 0;
      int best = 0;
      for (int n = 1; n < R; ++n) {
        int p = par[n];
        if (p < 0 || p >= n) {
          report(g.ws, SPEC_ERR_DEVICE, b, n);
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
      if (a > g.max_depth) {
        report(g.ws, SPEC_ERR_DEVICE, b, a);
        a = g.max_depth;
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
        g.out[(size_t)b * W + i] = o;
        if (g.kv_src) g.kv_src[(size_t)b * W + i] = i <= a ? path[i] : -1;
      }
    }
    g.acc_out[b] = a;
    s_a = a;
    g.cnt[b] = 0;                              // ready for the next call
  }
  __syncthreads();
  if (g.parent != nullptr && g.has_kv) {
    const int ctx = g.ctx_len[b];
    if (g.elem_bytes == 2)
      compact_path<__nv_bfloat16>(g.kv, b, ctx, path, s_a, g.row_elems, g.ws);
    else
      compact_path<float>(g.kv, b, ctx, path, s_a, g.row_elems, g.ws);
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
  SPEC_TL(spec::kTLThreshold);
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
// One launch, two roles, in start order.  The accept tests need, per row, only
// the log-sum-exp of the (filtered, tempered) target distribution; the Gumbel
// sample is needed on one row per request: the first rejected position, or
// row K for the bonus token.  So:
//  * statistics CTAs (the first rows*nch tickets): chunk c of a row -- max /
//    sum-exp over the kept tokens (greedy rows: argmax); the last of a
//    request's statistics CTAs merges the chunks row by row, makes the
//    sequential accept decisions, writes accept_len, the accepted drafts, -1
//    padding, kv_src (greedy requests: also the emitted token) and publishes
//    the decision;
//  * sampling CTAs (the next B*nchs tickets): chunk c of request b's sampled
//    row -- they wait (bounded) for the decision, then Philox noise and the
//    Gumbel-max key over the kept tokens, the draft token excluded on a
//    rejected row; the last of them writes the emitted token.
// Tickets are taken when a CTA starts, so every statistics CTA had started
// before any sampling CTA waits, and none of them waits on anything: the waits
// end.  They are bounded all the same (SPEC_ERR_TIMEOUT).
// a chunk record written by another CTA of this launch (read past L1)
SPEC_DEV RejPart ld_rejpart(const RejPart* p) {
  const float4 q = __ldcg(reinterpret_cast<const float4*>(p));
  return RejPart{q.x, q.y, q.z, __float_as_int(q.w)};
}

struct RejArgs {
  const float* logits;
  int K, V, nch, L, nchs, Ls, nstat, ncta;
  const float* temperature;
  const Thr* thr;
  const int32_t* draft;
  uint2 key;
  uint32_t w0;
  RejPart* part;      // [rows, nch] statistics records
  RejPart* spart;     // [B, nchs] sampling records
  VerifyCtl* ctl;
  int* cnt;
  int* scnt;
  int* decided;
  int32_t* out;
  int32_t* acc_out;
  int32_t* kv_src;
  void* ws;
};

template <bool VEC>
__device__ void rej_stats(const RejArgs& g, int row, int c, float* red, int* redi, uint8_t* ring) {
  const int K = g.K, V = g.V;
  const Thr tr = g.thr ? g.thr[row] : Thr{0u, 0x7fffffff};
  const int b = row / (K + 1);
  const float T = g.temperature[b];
  const bool greedy = !(T > 0.f);
  const bool unit = T == 1.f;                 // y = l / 1 exactly: skip the division
  const bool filt = g.thr != nullptr;
  const float* x = g.logits + (size_t)row * V;
  const int lo = c * g.L, hi = min(V, lo + g.L);
  float m = -INFINITY, s = 0.f, bk = -INFINITY;
  int bi = 0x7fffffff;
  // one group of four ids j .. j + 3 (ids past hi are ignored)
  auto group = [&](int j, const float* v) {
    if (greedy) {
#pragma unroll
      for (int l = 0; l < 4; ++l)
        if (j + l < hi && better(v[l], j + l, bk, bi)) { bk = v[l]; bi = j + l; }
      return;
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
  };
  if (VEC && g.L >= kVStreamMin) {
    if (!stream_chunk(x, lo, hi, ring, group) && threadIdx.x == 0) report(g.ws, SPEC_ERR_TIMEOUT, row, c);
  } else {
    constexpr int UNR = 4;                    // 16-byte loads in flight per thread
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
        group(j, vv[u]);
      }
    }
  }
  const float bm = block_max(m, red);
  const float contrib = (m == -INFINITY) ? 0.f : s * expf(m - bm);
  const float bs = block_sum(contrib, red);
  block_argmax(bk, bi, red, redi);
  if (threadIdx.x == 0) g.part[(size_t)row * g.nch + c] = RejPart{bm, bs, bk, bi};
}

// The request's sequential accept decisions, by one warp, from the chunk records.
__device__ void rej_decide(const RejArgs& g, int b) {
  const int K = g.K, V = g.V, nch = g.nch, lane = threadIdx.x & 31;
  const float T = g.temperature[b];
  const bool greedy = !(T > 0.f);
  int a = 0, emitted = -1;
  for (int i = 0; i <= K; ++i) {
    const size_t row = (size_t)b * (K + 1) + i;
    // merge the row's chunk records (lane c takes chunks c, c + 32, ...)
    float M = -INFINITY, bk = -INFINITY;
    int bi = 0x7fffffff;
    for (int c = lane; c < nch; c += 32) {
      const RejPart p = ld_rejpart(&g.part[row * nch + c]);
      M = fmaxf(M, p.m);
      if (better(p.key, p.idx, bk, bi)) { bk = p.key; bi = p.idx; }
    }
    M = warp_max(M);
    warp_argmax(bk, bi);
    float S = 0.f;
    for (int c = lane; c < nch; c += 32) {
      const RejPart p = ld_rejpart(&g.part[row * nch + c]);
      if (p.m > -INFINITY) S += p.s * expf(p.m - M);
    }
    S = warp_sum(S);
    if (i == K) {
      if (greedy) emitted = bi;
      break;
    }
    const int d = g.draft[(size_t)b * K + i];
    bool ok;
    if (greedy) {
      ok = (d == bi);
    } else {
      const float lse = M + logf(S);
      float pd = 0.f;
      if (d >= 0 && d < V) {
        const float yd = g.logits[row * V + d] / T;
        const Thr tr = g.thr ? g.thr[row] : Thr{0u, 0x7fffffff};
        if (kept_by(tr, okey(yd), d)) pd = expf(yd - lse);
      }
      const uint4 r = philox4x32_10(make_uint4(0u, (uint32_t)i, (uint32_t)b, g.w0), g.key);
      ok = word_to_uniform(r.x) <= pd;
    }
    if (!ok) {
      if (greedy) emitted = bi;
      break;
    }
    ++a;
  }
  for (int i = lane; i <= K; i += 32) {
    if (i != a || greedy) g.out[(size_t)b * (K + 1) + i] = i < a ? g.draft[(size_t)b * K + i] : (i == a ? emitted : -1);
    if (g.kv_src) g.kv_src[(size_t)b * (K + 1) + i] = i <= a ? i : -1;
  }
  if (lane == 0) g.acc_out[b] = a;
}

template <bool VEC>
__device__ void rej_sample(const RejArgs& g, int b, int c, int i, float* red, int* redi) {
  const int K = g.K, V = g.V;
  const float T = g.temperature[b];
  const int row = b * (K + 1) + i;
  const Thr tr = g.thr ? g.thr[row] : Thr{0u, 0x7fffffff};
  const bool unit = T == 1.f;
  const int excl = i < K ? g.draft[(size_t)b * K + i] : -1;
  const float* x = g.logits + (size_t)row * V;
  const int lo = c * g.Ls, hi = min(V, lo + g.Ls);
  float bk = -INFINITY;
  int bi = 0x7fffffff;
  // every thread handles aligned groups of 4 vocabulary ids = one Philox block;
  // the logits of two groups are loaded before the first one's noise is drawn
  constexpr int SB = 2;
  for (int j0 = lo + 4 * threadIdx.x; j0 < hi; j0 += 4 * SB * blockDim.x) {
    float v[SB][4];
#pragma unroll
    for (int u = 0; u < SB; ++u) {
      const int j = j0 + 4 * u * blockDim.x;
      if (VEC) {
        if (j < hi) {
          const float4 q = *reinterpret_cast<const float4*>(x + j);
          v[u][0] = q.x; v[u][1] = q.y; v[u][2] = q.z; v[u][3] = q.w;
        }
      } else {
#pragma unroll
        for (int l = 0; l < 4; ++l) v[u][l] = (j + l < hi) ? x[j + l] : -INFINITY;
      }
    }
#pragma unroll
    for (int u = 0; u < SB; ++u) {
      const int j = j0 + 4 * u * blockDim.x;
      if (j >= hi) break;
      const uint4 r = philox4x32_10(make_uint4((uint32_t)(j >> 2), (uint32_t)i, (uint32_t)b, g.w0 + 1u), g.key);
      const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int l = 0; l < 4; ++l) {
        if (j + l >= hi) break;
        const float y = unit ? v[u][l] : v[u][l] / T;
        if (j + l == excl || !kept_by(tr, okey(y), j + l)) continue;
        const float gk = y - logf(-logf(word_to_uniform(w[l])));
        if (better(gk, j + l, bk, bi)) { bk = gk; bi = j + l; }
      }
    }
  }
  block_argmax(bk, bi, red, redi);
  if (threadIdx.x == 0) g.spart[(size_t)b * g.nchs + c] = RejPart{0.f, 0.f, bk, bi};
}

template <bool VEC>
__global__ void __launch_bounds__(256, 3) verify_rejection_kernel(RejArgs g) {
  SPEC_TL(spec::kTLRejection);
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(128) uint8_t vring[];   // chunk ring (VEC: kVRingBytes)
  __shared__ float red[32];
  __shared__ int redi[32];
  __shared__ int s_t, s_flag, s_ok, s_i;
  const int nstat = g.nstat;
  if (threadIdx.x == 0) s_t = atomicAdd(&g.ctl->ticket, 1);
  __syncthreads();
  const int t = s_t;
  const int K = g.K;
  if (t < nstat) {
    const int row = t / g.nch, c = t % g.nch, b = row / (K + 1);
    rej_stats<VEC>(g, row, c, red, redi, vring);
    if (last_arrival(&g.cnt[b], (K + 1) * g.nch, &s_flag)) {
      if (threadIdx.x < 32) rej_decide(g, b);
      if (threadIdx.x == 0) {
        g.cnt[b] = 0;
        const int hold = *reinterpret_cast<const int*>(static_cast<const char*>(g.ws) + kKnobWithhold);
        if (g.temperature[b] > 0.f && hold != b + 1) {
          __threadfence();
          st_release(&g.decided[b], 1);
        }
      }
    }
  } else {
    const int sidx = t - nstat, b = sidx / g.nchs, c = sidx % g.nchs;
    if (g.temperature[b] > 0.f) {              // greedy requests were settled by their decision
      if (threadIdx.x == 0) {
        const int lim_us = *reinterpret_cast<const int*>(static_cast<const char*>(g.ws) + kKnobWait);
        const unsigned long long lim = lim_us > 0 ? (unsigned long long)lim_us * 1000ull : kDefaultWaitNs;
        const unsigned long long t0 = globaltimer_ns();
        int ok = 0;
        for (unsigned it = 0; it < (1u << 24); ++it) {      // the timer ends it; the count bounds it too
          if (ld_acquire(&g.decided[b]) != 0) { ok = 1; break; }
          if ((it & 15u) == 0 && globaltimer_ns() - t0 > lim) break;
          __nanosleep(256);
        }
        if (!ok) report(g.ws, SPEC_ERR_TIMEOUT, b, c);
        const int i = ok ? __ldcg(&g.acc_out[b]) : 0;
        s_ok = ok && i >= 0 && i <= g.K;
        s_i = i;
      }
      __syncthreads();
      if (s_ok) {
        rej_sample<VEC>(g, b, c, s_i, red, redi);
      } else if (threadIdx.x == 0) {
        g.spart[(size_t)b * g.nchs + c] = RejPart{0.f, 0.f, -INFINITY, 0x7fffffff};
      }
      if (last_arrival(&g.scnt[b], g.nchs, &s_flag)) {
        if (threadIdx.x < 32) {
          const int lane = threadIdx.x;
          float bk = -INFINITY;
          int bi = 0x7fffffff;
          for (int cc = lane; cc < g.nchs; cc += 32) {
            const RejPart p = ld_rejpart(&g.spart[(size_t)b * g.nchs + cc]);
            if (better(p.key, p.idx, bk, bi)) { bk = p.key; bi = p.idx; }
          }
          warp_argmax(bk, bi);
          if (lane == 0) {
            const int i = __ldcg(&g.acc_out[b]);
            if (i >= 0 && i <= K) g.out[(size_t)b * (K + 1) + i] = (bi == 0x7fffffff) ? -1 : bi;
            else report(g.ws, SPEC_ERR_DEVICE, b, i);
            g.scnt[b] = 0;
            g.decided[b] = 0;
          }
        }
      }
    }
  }
  // the last CTA of the grid rewinds the ticket counter for the next call
  if (threadIdx.x == 0) {
    __threadfence();
    const int n = atomicAdd(&g.ctl->finished, 1);
    if (n == g.ncta - 1) {
      g.ctl->ticket = 0;
      g.ctl->finished = 0;
    }
  }
}

}  // namespace spec

namespace spec {
// Verifier workspace: header | control words | chunk records | sampling records
// | top-k / top-p thresholds.  The greedy verifier uses the first three regions
// only (8-byte records).
struct VLayout {
  size_t ctl, part, spart, thr, total, greedy_total;
  int nch, nchs;
};
static int sample_chunks(int B, int V) {
  int n = std::max(1, (640 + B - 1) / B);
  return std::min(n, std::max(1, V / 2048));
}
static VLayout vlayout(int B, int R, int V) {
  VLayout L{};
  const int rows = B * R;
  L.nch = verify_chunks(rows, V);
  L.nchs = sample_chunks(B, V);
  L.ctl = kWsHeader;
  L.part = L.ctl + ctl_bytes(B);
  L.greedy_total = L.part + align_up((size_t)rows * L.nch * sizeof(ArgPart), 256);
  L.spart = L.part + align_up((size_t)rows * L.nch * sizeof(RejPart), 256);
  L.thr = L.spart + align_up((size_t)B * L.nchs * sizeof(RejPart), 256);
  L.total = L.thr + align_up((size_t)rows * sizeof(Thr), 256);
  return L;
}

static spec_status greedy_args(int32_t B, int32_t R, int32_t V, const float* target_logits, const int32_t* draft_tok,
                               const int32_t* parent, int32_t max_depth, int32_t* out_tok, int32_t* accept_len,
                               int32_t* kv_src, const spec_model_desc* desc, const spec_kv* kv,
                               const int32_t* ctx_len, GreedyArgs* g) {
  if (B <= 0 || R <= 0 || V <= 0) return SPEC_ERR_SHAPE;
  if (!target_logits || !draft_tok || !out_tok || !accept_len) return SPEC_ERR_ARG;
  if (R > 64) return SPEC_ERR_CAPACITY;
  if (parent == nullptr && R < 2) return SPEC_ERR_SHAPE;
  if (parent != nullptr && (max_depth < 0 || max_depth >= 64)) return SPEC_ERR_SHAPE;
  *g = GreedyArgs{};
  if (parent != nullptr && kv != nullptr) {
    if (!desc || !ctx_len || !kv->k || !kv->v || !kv->block_table) return SPEC_ERR_ARG;
    if (kv->block_size <= 0 || kv->max_blocks <= 0 || kv->num_slots <= 0) return SPEC_ERR_SHAPE;
    g->has_kv = 1;
    g->kv = *kv;
    g->row_elems = desc->n_kv_heads * desc->head_dim;
    g->elem_bytes = desc->dtype == SPEC_DTYPE_BF16 ? 2 : 4;
  }
  g->logits = target_logits;
  g->V = V;
  g->R = R;
  g->draft = draft_tok;
  g->parent = parent;
  g->max_depth = max_depth;
  g->out = out_tok;
  g->acc_out = accept_len;
  g->kv_src = kv_src;
  g->ctx_len = ctx_len;
  return SPEC_OK;
}

// The chunk ring's dynamic shared memory, allowed once per device and kernel.
template <class K>
static bool ring_attr(K* kern) {
  static int done_dev = -1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (done_dev == dev) return true;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kVRingBytes) != cudaSuccess)
    return false;
  done_dev = dev;
  return true;
}

static spec_status launch_greedy(GreedyArgs g, int B, void* ws, const VLayout& L, cudaStream_t stream) {
  g.nch = L.nch;
  g.L = chunk_len(g.V, L.nch);
  g.part = reinterpret_cast<ArgPart*>(static_cast<char*>(ws) + L.part);
  g.part_cap = (long long)B * g.R * L.nch;
  g.cnt = reinterpret_cast<int*>(static_cast<char*>(ws) + L.ctl + sizeof(VerifyCtl));
  g.ws = ws;
  const dim3 grid(L.nch, B * g.R);
  const bool vec = (g.V % 4 == 0) && aligned(g.logits, 16);
  if (vec) {
    const bool ring = g.L >= kVStreamMin;
    if (ring && !ring_attr(verify_greedy_kernel<true>)) return SPEC_ERR_CUDA;
    launch_pdl(verify_greedy_kernel<true>, grid, dim3(256), ring ? kVRingBytes : 0, stream, g);
  }
  else
    launch_pdl(verify_greedy_kernel<false>, grid, dim3(256), 0, stream, g);
  return last_launch();
}
}  // namespace spec

using namespace spec;

extern "C" size_t spec_verify_workspace_bytes(int32_t B, int32_t R, int32_t V) {
  if (B <= 0 || R <= 0 || V <= 0) return 0;
  return vlayout(B, R, V).total;
}

extern "C" spec_status spec_verify_greedy(int32_t B, int32_t R, int32_t V, const float* target_logits,
                                          const int32_t* draft_tok, const int32_t* parent,
                                          int32_t max_depth, int32_t* out_tok, int32_t* accept_len,
                                          int32_t* kv_src, const spec_model_desc* desc,
                                          const spec_kv* kv, const int32_t* ctx_len, void* ws,
                                          size_t ws_bytes, spec_stream_t stream) {
  GreedyArgs g;
  spec_status s = greedy_args(B, R, V, target_logits, draft_tok, parent, max_depth, out_tok, accept_len, kv_src,
                              desc, kv, ctx_len, &g);
  if (s != SPEC_OK) return s;
  if (!ws || !aligned(ws, 256) || ws_bytes < spec_verify_workspace_bytes(B, R, V)) return SPEC_ERR_WORKSPACE;
  return launch_greedy(g, B, ws, vlayout(B, R, V), stream);
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
  const VLayout L = vlayout(B, R, V);
  const int rows = B * R;
  char* base = static_cast<char*>(ws);
  RejArgs g{};
  g.logits = target_logits;
  g.K = K;
  g.V = V;
  g.nch = L.nch;
  g.L = chunk_len(V, L.nch);
  g.nchs = L.nchs;
  g.Ls = chunk_len(V, L.nchs);
  g.nstat = rows * L.nch;
  g.ncta = g.nstat + B * L.nchs;
  g.temperature = temperature;
  g.draft = draft_tok;
  g.key = make_uint2((uint32_t)(seed & 0xffffffffull), (uint32_t)(seed >> 32));
  g.w0 = (uint32_t)((2ull * step_offset) & 0xffffffffull);
  g.part = reinterpret_cast<RejPart*>(base + L.part);
  g.spart = reinterpret_cast<RejPart*>(base + L.spart);
  g.ctl = reinterpret_cast<VerifyCtl*>(base + L.ctl);
  g.cnt = reinterpret_cast<int*>(base + L.ctl + sizeof(VerifyCtl));
  g.scnt = g.cnt + B;
  g.decided = g.cnt + 2 * B;
  g.out = out_tok;
  g.acc_out = accept_len;
  g.kv_src = kv_src;
  g.ws = ws;
  if (top_k || top_p) {
    Thr* thr = reinterpret_cast<Thr*>(base + L.thr);
    launch_pdl(reject_threshold_kernel, dim3(rows), dim3(1024), 0, stream, target_logits, K, V, temperature, top_k,
               top_p, thr);
    g.thr = thr;
  }
  const bool vec = (V % 4 == 0) && aligned(target_logits, 16);
  if (vec) {
    const bool ring = g.L >= kVStreamMin;
    if (ring && !ring_attr(verify_rejection_kernel<true>)) return SPEC_ERR_CUDA;
    launch_pdl(verify_rejection_kernel<true>, dim3(g.ncta), dim3(256), ring ? kVRingBytes : 0, stream, g);
  }
  else
    launch_pdl(verify_rejection_kernel<false>, dim3(g.ncta), dim3(256), 0, stream, g);
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
constexpr size_t kStaticVerifyScratch = 256 * 1024;     // header + control words + chunk records
static __device__ __align__(256) unsigned char g_verify_scratch[kStaticVerifyScratch];
constexpr int kStaticMaxDevices = 64;
static void* g_verify_scratch_addr[kStaticMaxDevices];
static std::mutex g_verify_scratch_mu;

// Device address of the scratch array on the current device (looked up once per
// device, with that device current; the cached address does not survive a
// cudaDeviceReset of that device).  nullptr if the lookup fails.
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

extern "C" size_t spec_verify_greedy_static_capacity(void) { return kStaticVerifyScratch; }

extern "C" size_t spec_verify_greedy_static_bytes(int32_t B, int32_t R, int32_t V) {
  if (B <= 0 || R <= 0 || V <= 0) return 0;
  return vlayout(B, R, V).greedy_total;
}

extern "C" spec_status spec_verify_greedy_static(int32_t B, int32_t R, int32_t V, const float* target_logits,
                                                 const int32_t* draft_tok, const int32_t* parent,
                                                 int32_t max_depth, int32_t* out_tok, int32_t* accept_len,
                                                 int32_t* kv_src, const spec_model_desc* desc, const spec_kv* kv,
                                                 const int32_t* ctx_len, spec_stream_t stream) {
  GreedyArgs g;
  spec_status s = greedy_args(B, R, V, target_logits, draft_tok, parent, max_depth, out_tok, accept_len, kv_src,
                              desc, kv, ctx_len, &g);
  if (s != SPEC_OK) return s;
  // the greedy layout (header, control words, 8-byte chunk records) must fit the array
  const VLayout L = vlayout(B, R, V);
  if (L.greedy_total > kStaticVerifyScratch) return SPEC_ERR_CAPACITY;
  void* ws = static_verify_scratch();
  if (ws == nullptr) return SPEC_ERR_CUDA;
  // the array keeps the previous call's contents: the error header and the
  // completion counters start at zero; every chunk record is rewritten before it
  // is read
  if (cudaMemsetAsync(ws, 0, L.part, stream) != cudaSuccess) return SPEC_ERR_CUDA;
  return launch_greedy(g, B, ws, L, stream);
}

extern "C" spec_status spec_verify_greedy_static_error(int32_t* code_out, spec_stream_t stream) {
  if (!code_out) return SPEC_ERR_ARG;
  void* ws = static_verify_scratch();
  if (ws == nullptr) return SPEC_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, stream) != cudaSuccess) return SPEC_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return SPEC_ERR_CUDA;
  *code_out = v;
  return SPEC_OK;
}

// per-unit log setter of the instrumented build (no-op otherwise)
SPEC_TL_SETTER(verify)
