// Shared device helpers of libeaglespec (sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <utility>

#include "../../include/eaglespec.h"

#define SPEC_DEV __device__ __forceinline__

namespace spec {

// Workspace header: the first 256 bytes of every workspace.
struct WsHeader {
  int32_t error;      // 0 = ok, else a spec_status code
  int32_t detail[7];  // first failing index information (debug)
};
constexpr size_t kWsHeader = 256;

// ---------------------------------------------------------------- timeline (instrumented build)
// Compiled only with SPEC_TIMELINE (libeaglespec_timeline.so): thread 0 of every
// block of every kernel takes a slot of the log set by spec_timeline_set_<unit>
// (one per translation unit) and writes the global timer at its start and at
// its exit, with kernel id | grid size << 8 | block index << 32.  Log layout
// (u64): [0] slot counter, then 4 words a slot from index 8.  The product
// build has none of this (SPEC_TL expands to nothing).
enum TLKernel : unsigned {
  kTLTc = 1, kTLAttnWs, kTLAttnMma, kTLAttnSplit, kTLCombine, kTLPrologue, kTLEpiStore, kTLEpiQkv,
  kTLResnorm, kTLSwiglu, kTLSimt, kTLRowStats, kTLTopk, kTLRescore, kTLCandBest, kTLLmMerge, kTLTree,
  kTLGreedy, kTLRejection, kTLThreshold, kTLPrefill, kTLMetadata, kTLGather
};
#ifdef SPEC_TIMELINE
static __device__ unsigned long long* g_spec_tl;
constexpr unsigned kTLSlots = 1u << 20;
SPEC_DEV unsigned long long tl_now() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
struct TLRec {
  unsigned idx = 0xffffffffu;
  SPEC_DEV bool first() const { return threadIdx.x == 0 && threadIdx.y == 0 && threadIdx.z == 0; }
  SPEC_DEV explicit TLRec(unsigned id) {
    if (first() && g_spec_tl != nullptr) {
      const unsigned i = atomicAdd(reinterpret_cast<unsigned*>(g_spec_tl), 1u);
      if (i < kTLSlots) {
        idx = i;
        unsigned long long* e = g_spec_tl + 8 + 4ull * i;
        e[0] = tl_now();
        e[3] = (unsigned long long)id | ((unsigned long long)(gridDim.x * gridDim.y) << 8) |
               ((unsigned long long)(blockIdx.x + gridDim.x * blockIdx.y) << 32);
      }
    }
  }
  SPEC_DEV ~TLRec() {
    if (idx != 0xffffffffu) g_spec_tl[8 + 4ull * idx + 2] = tl_now();
  }
};
#define SPEC_TL(id) ::spec::TLRec spec_tl_rec_(id)
#define SPEC_TL_SETTER(unit)                                                   \
  extern "C" int spec_timeline_set_##unit(void* p) {                          \
    return (int)cudaMemcpyToSymbol(::spec::g_spec_tl, &p, sizeof(p));          \
  }
#else
#define SPEC_TL(id) ((void)0)
#define SPEC_TL_SETTER(unit)
#endif

SPEC_DEV void report(void* ws, int code, int a = 0, int b = 0) {
  if (ws == nullptr) return;
  WsHeader* h = reinterpret_cast<WsHeader*>(ws);
  if (atomicCAS(&h->error, 0, code) == 0) {
    h->detail[0] = a;
    h->detail[1] = b;
  }
}

// ---------------------------------------------------------------- element I/O
template <typename T> SPEC_DEV float ld(const T* p);
template <> SPEC_DEV float ld<float>(const float* p) { return *p; }
template <> SPEC_DEV float ld<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }

template <typename T> SPEC_DEV void st(T* p, float v);
template <> SPEC_DEV void st<float>(float* p, float v) { *p = v; }
template <> SPEC_DEV void st<__nv_bfloat16>(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// value as stored (rounded to T), returned as float
template <typename T> SPEC_DEV float rnd(float v);
template <> SPEC_DEV float rnd<float>(float v) { return v; }
template <> SPEC_DEV float rnd<__nv_bfloat16>(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

// ---------------------------------------------------------------- reductions
SPEC_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
SPEC_DEV float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
// (value, index) better: larger value, then smaller index
SPEC_DEV bool better(float v, int i, float bv, int bi) { return v > bv || (v == bv && i < bi); }
SPEC_DEV void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float ov = __shfl_xor_sync(0xffffffffu, v, o);
    int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (better(ov, oi, v, i)) { v = ov; i = oi; }
  }
}

// The same winner as warp_argmax for non-NaN values (largest value, then smallest
// index; -0 equals +0) from two warp-wide reductions on an order-preserving key
// instead of five shuffle rounds; a NaN never wins here.
SPEC_DEV void warp_argmax_redux(float& v, int& i) {
  const uint32_t u = __float_as_uint(v == 0.f ? 0.f : v);
  const uint32_t k = v != v ? 0u : ((u & 0x80000000u) ? ~u : (u | 0x80000000u));
  const uint32_t km = __reduce_max_sync(0xffffffffu, k);
  const int im = __reduce_min_sync(0xffffffffu, k == km ? i : 0x7fffffff);
  const unsigned who = __ballot_sync(0xffffffffu, k == km && i == im);
  v = __shfl_sync(0xffffffffu, v, __ffs(who) - 1);
  i = im;
}

// block-wide sum for blockDim.x a multiple of 32 (<= 1024); all threads get the result
SPEC_DEV float block_sum(float v, float* red) {
  int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  float r = (lane < nw) ? red[lane] : 0.f;
  r = warp_sum(r);
  return r;
}
SPEC_DEV float block_max(float v, float* red) {
  int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_max(v);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  float r = (lane < nw) ? red[lane] : -INFINITY;
  return warp_max(r);
}
SPEC_DEV void block_argmax(float& v, int& i, float* redv, int* redi) {
  int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  warp_argmax(v, i);
  __syncthreads();
  if (lane == 0) { redv[wid] = v; redi[wid] = i; }
  __syncthreads();
  v = (lane < nw) ? redv[lane] : -INFINITY;
  i = (lane < nw) ? redi[lane] : 0x7fffffff;
  warp_argmax(v, i);
}

// ---------------------------------------------------------------- paged cache
SPEC_DEV long long slot_of(const spec_kv& kv, int b, int cache_idx) {
  int blk = cache_idx / kv.block_size;
  if (cache_idx < 0 || blk >= kv.max_blocks) return -1;
  long long s = (long long)kv.block_table[(long long)b * kv.max_blocks + blk] * kv.block_size +
                cache_idx % kv.block_size;
  if (s < 0 || s >= kv.num_slots) return -1;
  return s;
}

// ---------------------------------------------------------------- Philox4x32-10
// Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3"
// (SC'11): per round two 32x32 -> 64-bit products of counter words 0 and 2 by
// the round multipliers; the high halves are XORed with counter words 1 / 3 and
// the round key and the words permuted; the key advances by the Weyl constants.
SPEC_DEV uint4 philox4x32_10(uint4 c, uint2 k) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) { k.x += W0; k.y += W1; }
    uint32_t lo0 = M0 * c.x, hi0 = __umulhi(M0, c.x);
    uint32_t lo1 = M1 * c.z, hi1 = __umulhi(M1, c.z);
    c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
  }
  return c;
}
// 32-bit word -> u = ((x >> 8) + 0.5) * 2^-24 in (0, 1), exact in fp32
SPEC_DEV float word_to_uniform(uint32_t x) { return ((float)(x >> 8) + 0.5f) * 5.9604644775390625e-8f; }

// ---------------------------------------------------------------- dependent launch
// Kernels of a step are launched with programmatic stream serialisation: a
// kernel may start while its predecessor finishes; griddepcontrol.wait blocks
// until the predecessor grid has completed and its writes are visible, so every
// kernel calls pdl_wait() before touching data another kernel produced or
// consumes, then pdl_trigger() to let its own successor launch.  Both are no-ops
// when the kernel was launched without the attribute.
SPEC_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
SPEC_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------- misc
SPEC_DEV uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

}  // namespace spec
