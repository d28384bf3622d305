// tcgen05 / TMA / mbarrier primitives for sm_103a and the warp-specialised
// mainloop shared by the tensor-core GEMM kernels (tc_gemm.cu, lmhead.cu).
//
// Layout: the A operand (weight tile, 128 rows x 64 K of bf16) and the B
// operand (activation tile, MPAD rows x 64 K) are loaded by TMA with 128-byte
// swizzle into a ring of shared-memory stages; one thread issues
// tcgen05.mma (M = 128, N = MPAD, K = 16 per instruction) into one of two TMEM
// accumulators; four warps drain TMEM with tcgen05.ld.
#pragma once
#include <cuda.h>

#include "common.cuh"
#include "internal.h"

namespace spec {
namespace tc {

constexpr int kThreads = 192;
constexpr int kBK = 64;                          // K elements per chunk (128 B of bf16)
constexpr int kABytes = 128 * kBK * 2;           // A stage: 128 rows x 128 B
constexpr uint64_t kWaitNs = 2000000000ull;      // bounded waits: 2 s

// EXTRA: bytes of dynamic shared memory the epilogue claims after the stage ring
template <int MPAD, int EXTRA = 0> struct Cfg {
  static_assert(MPAD % 16 == 0 && MPAD <= 384, "activation tile rows");
  static constexpr int kBBytes = MPAD * kBK * 2;
  static constexpr int kStage = kABytes + kBBytes;
  static constexpr int kBudget = (MPAD > 256 ? 212 * 1024 : 196 * 1024) - EXTRA;
  static constexpr int kStages = kBudget / kStage > 10 ? 10 : kBudget / kStage;
  // two TMEM accumulators (MMA of the next segment overlaps the drain of the
  // previous one) when they fit in TMEM's 512 columns, else one
  static constexpr int kBufs = 2 * MPAD <= 512 ? 2 : 1;
  static constexpr int kCols = kBufs * MPAD <= 32 ? 32 : (kBufs * MPAD <= 64 ? 64 : (kBufs * MPAD <= 128 ? 128 :
                               (kBufs * MPAD <= 256 ? 256 : 512)));
  // B (activation) tile: one TMA box of MPAD rows, or 128-row boxes above 256
  static constexpr int kBBox = MPAD <= 256 ? MPAD : 128;
  static constexpr int kBLoads = MPAD / kBBox;
  // MMA N per instruction: MPAD, or 256 + the remainder above 256
  static constexpr int kN0 = MPAD <= 256 ? MPAD : 256;
  static constexpr int kN1 = MPAD - kN0;
  static constexpr size_t kSmem = (size_t)kStages * kStage + 1024 + 256 + EXTRA;
};

// 3-D tensor map of a bf16 paged K or V cache [slots][nkv][hd] (defined in tc_gemm.cu)
bool make_kv_map(CUtensorMap* tm, const void* ptr, int slots, int nkv, int hd, int box_keys);

SPEC_DEV uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

SPEC_DEV void mbar_init(uint32_t a, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(n) : "memory");
}
SPEC_DEV void mbar_expect_tx(uint32_t a, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a), "r"(bytes) : "memory");
}
SPEC_DEV void mbar_arrive(uint32_t a) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(a) : "memory");
}
SPEC_DEV bool mbar_try(uint32_t a, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(a), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait.  Returns false on timeout (sets *abort) or when another role aborted.
SPEC_DEV bool mbar_wait(uint32_t a, uint32_t parity, volatile int* abort, bool honour_abort = true) {
  if (mbar_try(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1; it < (1u << 30); ++it) {
    if (mbar_try(a, parity)) return true;
    if ((it & 255u) == 0) {
      if (honour_abort && *abort) return false;
      if (globaltimer_ns() - t0 > kWaitNs) break;
    }
  }
  *abort = 1;
  return false;
}

SPEC_DEV void tma_load_2d(uint32_t dst, const CUtensorMap* tm, uint32_t mbar, int x, int y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(mbar), "l"(policy)
      : "memory");
}
SPEC_DEV uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
SPEC_DEV uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

SPEC_DEV void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
SPEC_DEV void tmem_relinquish() { asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory"); }
SPEC_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
SPEC_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
SPEC_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
SPEC_DEV void tc_commit(uint32_t mbar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar) : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 in, fp32 accumulate)
SPEC_DEV void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns
SPEC_DEV void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
SPEC_DEV void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 B in 8-row (1024 B) swizzle atoms: stride byte offset 1024; the leading
// byte offset is unused for this layout; descriptor version 1; swizzle code 2.
SPEC_DEV uint64_t desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major,
// N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

}  // namespace tc
}  // namespace spec
