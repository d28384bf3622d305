// Top-k draft-tree expansion ranked by cumulative log-probability.
//
// [EAGLET] "Eaglet": draft_top_k, draft_depth, total_draft_tokens (the draft
// model proposes a token tree that the target verifies in one pass).  The
// expansion rule (EAGLE-2 style; the pages give only the three parameters):
// depth 1 takes the root's top-k; at depth d >= 2 every frontier node's top-k
// children, scored parent score + log-prob in fp32, join a candidate pool and
// the k best of them form the next frontier; after the last depth the
// `total` best pool nodes are the tree, numbered by (depth, score, creation).
//
// One CTA per request.  Pool sizes are small (k + (D-1) k^2 <= a few hundred),
// so ranks are computed by counting (each thread compares its candidate with
// all others), which gives exact, deterministic orders with the stated ties.
#include "common.cuh"
#include "internal.h"

namespace spec {

struct TreeDims {
  int k, D, N, P;
};

// per-request state layout (bytes, each array 8-byte aligned)
struct TreeView {
  int* count;
  int* tok;
  int* parent;
  int* depth;
  float* score;
  int* srcrow;
  unsigned long long* mask;
  int* frontier;
};

__host__ __device__ inline size_t tree_req_bytes(int k, int P) {
  size_t b = 16;                       // count, root token, pad
  b += (size_t)P * 4 * 5;              // tok, parent, depth, score, srcrow
  b = (b + 7) & ~size_t(7);
  b += (size_t)P * 8;                  // mask
  b += (size_t)k * 4;                  // frontier
  return (b + 255) & ~size_t(255);
}

__device__ TreeView tree_view(void* base, int k, int P) {
  char* p = static_cast<char*>(base);
  TreeView v;
  v.count = reinterpret_cast<int*>(p);
  p += 16;
  v.tok = reinterpret_cast<int*>(p); p += (size_t)P * 4;
  v.parent = reinterpret_cast<int*>(p); p += (size_t)P * 4;
  v.depth = reinterpret_cast<int*>(p); p += (size_t)P * 4;
  v.score = reinterpret_cast<float*>(p); p += (size_t)P * 4;
  v.srcrow = reinterpret_cast<int*>(p); p += (size_t)P * 4;
  p = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(p) + 7) & ~uintptr_t(7));
  v.mask = reinterpret_cast<unsigned long long*>(p); p += (size_t)P * 8;
  v.frontier = reinterpret_cast<int*>(p);
  return v;
}

// candidate a ranks before candidate b: larger score, then smaller creation index
__device__ __forceinline__ bool ranks_before(float sa, int ia, float sb, int ib) {
  return sa > sb || (sa == sb && ia < ib);
}

__global__ void __launch_bounds__(1024) tree_expand_kernel(TreeDims td, int d, const int32_t* __restrict__ ctx_len,
                                                          const int32_t* __restrict__ root_tok,
                                                          const int32_t* __restrict__ ids,
                                                          const float* __restrict__ lp, void* state,
                                                          spec_tree_io io) {
  SPEC_TL(spec::kTLTree);
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x;
  const int k = td.k, P = td.P;
  TreeView tv = tree_view(static_cast<char*>(state) + (size_t)b * tree_req_bytes(k, P), k, P);
  __shared__ int s_map[1024];
  __shared__ int s_order[64];
  const int c0 = (d == 1) ? 0 : *tv.count;
  if (d == 1 && threadIdx.x == 0) {
    tv.count[0] = 0;
    tv.count[1] = root_tok[b];      // kept for the final call
  }
  const int nc = (d == 1) ? k : k * k;
  // 1. append the new candidates (creation order f*k + j)
  for (int t = threadIdx.x; t < nc; t += blockDim.x) {
    int p = c0 + t;
    if (d == 1) {
      const int row = b;
      tv.tok[p] = ids[(size_t)row * k + t];
      tv.parent[p] = -1;
      tv.score[p] = 0.f + lp[(size_t)row * k + t];
      tv.srcrow[p] = row;
    } else {
      const int f = t / k, j = t % k;
      const int row = b * k + f;
      const int par = tv.frontier[f];
      tv.tok[p] = ids[(size_t)row * k + j];
      tv.parent[p] = par;
      tv.score[p] = tv.score[par] + lp[(size_t)row * k + j];
      tv.srcrow[p] = row;
    }
    tv.depth[p] = d;
    tv.mask[p] = 0ull;
  }
  __syncthreads();
  // pool scores / depths staged in shared memory for the rank counting below
  __shared__ float s_score[1024];
  __shared__ unsigned char s_depth[1024];
  const int cnt = c0 + nc;
  for (int p = threadIdx.x; p < cnt; p += blockDim.x) {
    s_score[p] = tv.score[p];
    s_depth[p] = (unsigned char)tv.depth[p];
  }
  __syncthreads();
  // 2. next frontier = the k best new candidates
  for (int t = threadIdx.x; t < nc; t += blockDim.x) {
    const int p = c0 + t;
    const float sp = s_score[p];
    int r = 0;
    for (int u = 0; u < nc; ++u) r += ranks_before(s_score[c0 + u], c0 + u, sp, p) ? 1 : 0;
    if (r < k) s_order[r] = p;
  }
  __syncthreads();
  if (threadIdx.x < k) tv.frontier[threadIdx.x] = s_order[threadIdx.x];
  if (threadIdx.x == 0) *tv.count = c0 + nc;
  __syncthreads();
  if (d < td.D) {
    // 3a. rows of the next draft pass
    if (threadIdx.x < k) {
      const int f = threadIdx.x;
      const int node = s_order[f];
      const int par = tv.parent[node];
      const int idx = 1 + (d - 1) * k + f;
      const unsigned long long pm = (par < 0) ? 1ull : tv.mask[par];
      const unsigned long long m = pm | (1ull << idx);
      tv.mask[node] = m;
      const int row = b * k + f;
      io.frontier_tok[row] = tv.tok[node];
      io.frontier_pos[row] = ctx_len[b] + d;
      io.frontier_kv_idx[row] = idx;
      io.frontier_mask[row] = m;
      io.frontier_hid_src[row] = tv.srcrow[node];
    }
    return;
  }
  // 3b. final selection: the N best of the pool, numbered by (depth, score, creation).
  // A candidate's rank is counted by four threads (every fourth pool entry each);
  // the order of the N selected by a warp each (every 32nd entry a lane).
  const int N = td.N;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
  for (int base = 0; base < cnt; base += blockDim.x / 4) {
    const int p = base + (int)threadIdx.x / 4, q = threadIdx.x & 3;
    int r = 0;
    if (p < cnt) {
      const float sp = s_score[p];
      for (int u = q; u < cnt; u += 4) r += ranks_before(s_score[u], u, sp, p) ? 1 : 0;
    }
    r += __shfl_xor_sync(0xffffffffu, r, 1);
    r += __shfl_xor_sync(0xffffffffu, r, 2);
    if (p < cnt && q == 0) s_map[p] = (r < N) ? 0 : -1;
  }
  __syncthreads();
  for (int p = warp; p < cnt; p += nwarp) {
    if (s_map[p] < 0) continue;                 // uniform in the warp
    const int dp = s_depth[p];
    const float sp = s_score[p];
    int r = 0;
    for (int u = lane; u < cnt; u += 32) {
      if (s_map[u] < 0) continue;
      const int du = s_depth[u];
      r += (du < dp || (du == dp && ranks_before(s_score[u], u, sp, p))) ? 1 : 0;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
    if (lane == 0) s_order[r] = p;    // final index r + 1
  }
  __syncthreads();
  // final index of every selected node; then one thread per node writes its
  // outputs, and its mask is the OR of its ancestors' bits (final parents come
  // first in the numbering, so the chain ends at the root)
  for (int n = threadIdx.x; n < N; n += blockDim.x) s_map[s_order[n]] = n + 1;
  __syncthreads();
  __shared__ int s_pf[64];
  const size_t o = (size_t)b * (N + 1);
  const int ctx = ctx_len[b];
  for (int n = 1 + threadIdx.x; n <= N; n += blockDim.x) {
    const int p = s_order[n - 1];
    const int par = tv.parent[p];
    int pf = (par < 0) ? 0 : s_map[par];
    if (pf < 0 || pf >= n) pf = 0;   // cannot happen: the selection is ancestor-closed
    s_pf[n] = pf;
    io.tree_tok[o + n] = tv.tok[p];
    io.tree_parent[o + n] = pf;
    io.tree_depth[o + n] = s_depth[p];
    io.tree_pos[o + n] = ctx + s_depth[p];
    io.tree_score[o + n] = s_score[p];
  }
  if (threadIdx.x == 0) {
    io.tree_tok[o] = tv.count[1];
    io.tree_parent[o] = -1;
    io.tree_depth[o] = 0;
    io.tree_pos[o] = ctx;
    io.tree_score[o] = 0.f;
    io.tree_mask[o] = 1ull;
  }
  __syncthreads();
  for (int n = 1 + threadIdx.x; n <= N; n += blockDim.x) {
    unsigned long long msk = 1ull;
    for (int a = n; a > 0; a = s_pf[a]) msk |= 1ull << a;
    io.tree_mask[o + n] = msk;
  }
}

}  // namespace spec

using namespace spec;

extern "C" size_t spec_tree_state_bytes(int32_t B, int32_t top_k, int32_t draft_depth, int32_t total) {
  if (B <= 0 || top_k <= 0 || draft_depth <= 0 || total <= 0) return 0;
  const int P = top_k + (draft_depth - 1) * top_k * top_k;
  return (size_t)B * tree_req_bytes(top_k, P);
}

extern "C" spec_status spec_tree_expand(int32_t B, int32_t top_k, int32_t depth_idx, int32_t draft_depth,
                                        int32_t total, const int32_t* ctx_len, const int32_t* root_tok,
                                        const int32_t* topk_ids, const float* topk_logprob, void* tree_state,
                                        const spec_tree_io* io, spec_stream_t stream) {
  if (B <= 0 || top_k <= 0 || draft_depth <= 0 || total <= 0) return SPEC_ERR_SHAPE;
  if (depth_idx < 1 || depth_idx > draft_depth) return SPEC_ERR_ARG;
  if (!ctx_len || !topk_ids || !topk_logprob || !tree_state || !io) return SPEC_ERR_ARG;
  if (depth_idx == 1 && !root_tok) return SPEC_ERR_ARG;
  if (top_k > 16) return SPEC_ERR_UNSUPPORTED;
  const int P = top_k + (draft_depth - 1) * top_k * top_k;
  if (P > 1024) return SPEC_ERR_CAPACITY;
  if (total + 1 > 64 || 1 + (draft_depth - 1) * top_k > 64 || total > P) return SPEC_ERR_CAPACITY;
  if (!aligned(tree_state, 256)) return SPEC_ERR_ALIGN;
  if (depth_idx < draft_depth) {
    if (!io->frontier_tok || !io->frontier_pos || !io->frontier_kv_idx || !io->frontier_mask ||
        !io->frontier_hid_src)
      return SPEC_ERR_ARG;
  } else {
    if (!io->tree_tok || !io->tree_parent || !io->tree_depth || !io->tree_pos || !io->tree_score ||
        !io->tree_mask)
      return SPEC_ERR_ARG;
  }
  TreeDims td{top_k, draft_depth, total, P};
  launch_pdl(tree_expand_kernel, dim3(B), dim3(1024), 0, stream, td, depth_idx, ctx_len, root_tok, topk_ids, topk_logprob, tree_state,
                                            *io);
  return last_launch();
}

// per-unit log setter of the instrumented build (no-op otherwise)
SPEC_TL_SETTER(tree)
