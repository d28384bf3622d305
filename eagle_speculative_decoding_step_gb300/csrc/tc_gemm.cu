// bf16 tensor-core GEMM for the draft step's contractions (FC, QKV, O,
// gate/up, down, low-rank projections), written for sm_103a's 5th-generation
// tensor cores: tcgen05.mma with the accumulator in tensor memory (TMEM),
// operands staged in shared memory by TMA (cp.async.bulk.tensor, 128-byte
// swizzle), mbarrier pipelines, one elected thread issuing the MMAs.
//
// Shape: out[m, n] = sum_k X[m, k] * W[n, k] with few rows m (the draft
// batch, 1..256) and many weight rows n.  The weight is the MMA's A operand
// (M = 128 weight rows per tile) and the activation its B operand
// (N = MPAD >= M rows), so every byte of the weight is read from HBM exactly
// once and the tensor core never waits on a padded activation tile.
// Work is split stream-K: tiles x 64-wide K chunks spread evenly over the CTAs
// (one per SM); each CTA emits fp32 partial sums per tile segment that the
// epilogue kernels reduce in a fixed order.
//
// Warp roles (192 threads): warps 0-3 drain TMEM (tcgen05.ld, one 32-lane
// quarter each), warp 4 lane 0 issues TMA loads, warp 5 lane 0 issues MMAs.
// Two TMEM accumulators let the MMA of the next segment overlap the drain of
// the previous one.  Every mbarrier wait is bounded (2 s); on expiry the CTA
// records SPEC_ERR_TIMEOUT in the workspace error word, drains its copies in
// flight, frees its TMEM and exits.
#include "tc_kernel.cuh"

namespace spec {
namespace tc {

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

// 2-D bf16 tensor [rows, cols] row-major, box 64 (cols) x box_rows, 128-byte swizzle.
bool make_map(CUtensorMap* tm, const void* ptr, int rows, int cols, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 paged cache [slots][nkv][hd]: box 64 columns x 1 head x box_keys slots, 128-byte swizzle
// (rows past the last slot read as zeros).
bool make_kv_map(CUtensorMap* tm, const void* ptr, int slots, int nkv, int hd, int box_keys) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)hd, (cuuint64_t)nkv, (cuuint64_t)slots};
  cuuint64_t strides[2] = {(cuuint64_t)hd * 2, (cuuint64_t)nkv * hd * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)box_keys};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MPAD>
static spec_status launch_mpad(const CUtensorMap* a, const CUtensorMap& b, const SKPlan& p, int M, float* part,
                               void* ws, cudaStream_t st) {
  typename EpiPartial<MPAD>::Params ep{p, M, part};
  return launch_tc<MPAD, SchedSK, EpiPartial<MPAD>>(a, b, p, ep, p.G, 0, ws, st);
}

}  // namespace tc

int tc_mpad(int M) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  if (M <= 128) return 128;
  if (M <= 256) return 256;
  return 384;
}
static int bbox_rows(int mpad) { return mpad <= 256 ? mpad : 128; }

// Partial sums of X[M, K] @ [W0; W1; W2]^T into `part` (plan p), bf16 operands.
spec_status launch_tc_gemm(const void* const* W, const int* rows, int nmat, int K, const void* X, int M,
                           const SKPlan& p, float* part, void* ws, cudaStream_t st) {
  using namespace tc;
  if (M < 1 || M > 384 || K % 8 != 0) return SPEC_ERR_SHAPE;
  for (int i = 0; i < nmat; ++i)
    if (!aligned(W[i], 16)) return SPEC_ERR_ALIGN;
  if (!aligned(X, 16)) return SPEC_ERR_ALIGN;
  const int mpad = p.mpad;
  CUtensorMap a[3];
  for (int i = 0; i < 3; ++i) {
    const int src = i < nmat ? i : 0;
    if (!make_map(&a[i], W[src], rows[src], K, 128)) return SPEC_ERR_CUDA;
  }
  CUtensorMap b;
  if (!make_map(&b, X, M, K, bbox_rows(mpad))) return SPEC_ERR_CUDA;
  switch (mpad) {
    case 384: return launch_mpad<384>(a, b, p, M, part, ws, st);
    case 16: return launch_mpad<16>(a, b, p, M, part, ws, st);
    case 32: return launch_mpad<32>(a, b, p, M, part, ws, st);
    case 64: return launch_mpad<64>(a, b, p, M, part, ws, st);
    case 128: return launch_mpad<128>(a, b, p, M, part, ws, st);
    case 256: return launch_mpad<256>(a, b, p, M, part, ws, st);
    default: return SPEC_ERR_SHAPE;
  }
}

}  // namespace spec

namespace spec {

// out[M, N] (fp32, row stride ld) = X[M, K] @ W[N, K]^T with every 128-row tile
// finished by one CTA (contiguous row ranges per CTA): no partial sums.
spec_status launch_tc_gemm_store(const void* W, int N, int K, const void* X, int M, float* out, int ld, void* ws,
                                 cudaStream_t st) {
  using namespace tc;
  if (M < 1 || M > 384 || K % 8 != 0) return SPEC_ERR_SHAPE;
  if (!aligned(W, 16) || !aligned(X, 16)) return SPEC_ERR_ALIGN;
  const int mpad = tc_mpad(M);
  int G = sm_count();
  if (G > (N + 127) / 128) G = (N + 127) / 128;
  CUtensorMap a[3];
  if (!make_map(&a[0], W, N, K, 128)) return SPEC_ERR_CUDA;
  a[1] = a[0];
  a[2] = a[0];
  CUtensorMap b;
  if (!make_map(&b, X, M, K, bbox_rows(mpad))) return SPEC_ERR_CUDA;
  RowsParams rp{N, G, (K + kBK - 1) / kBK};
  switch (mpad) {
#define STORE_CASE(MP)                                                                          \
  case MP: {                                                                                    \
    typename EpiStore<MP>::Params ep{M, ld, out};                                               \
    return launch_tc<MP, SchedRows, EpiStore<MP>>(a, b, rp, ep, G, 0, ws, st);                  \
  }
    STORE_CASE(16)
    STORE_CASE(32)
    STORE_CASE(64)
    STORE_CASE(128)
    STORE_CASE(256)
    STORE_CASE(384)
#undef STORE_CASE
    default: return SPEC_ERR_SHAPE;
  }
}

}  // namespace spec

// per-unit log setter of the instrumented build (no-op otherwise)
SPEC_TL_SETTER(tc_gemm)
