// Inputs of the batched initial draft pass over the verified tokens, and a row
// gather.
//
// [NEURON] "Speculative Decoding (EAGLE3) in the vLLM Neuron Framework",
// section "EagleProposer: Draft Model Management", propose() prefill phase: the
// draft processes all target tokens of the step; its input ids are the target's
// ids shifted by one, with the newly sampled token scattered at each request's
// last token position; the first draft token and the recurrent state come from
// that last position.  The pages do not fix the row layout; the one taken here:
// request b's R verified tokens sit at positions ctx_b .. ctx_b + R - 1, write
// their K/V at draft-region entries 0 .. R-1 and attend causally (row j sees the
// context and entries 0..j); rows after the last accepted one carry shifted
// ids of rejected drafts and are ignored by the caller.
#include "common.cuh"
#include "internal.h"

namespace spec {

__global__ void __launch_bounds__(256) prefill_inputs_kernel(int B, int R, const int32_t* __restrict__ input_ids,
                                                             const int32_t* __restrict__ next_token,
                                                             const int32_t* __restrict__ last_idx,
                                                             const int32_t* __restrict__ ctx_len,
                                                             int32_t* __restrict__ tok, int32_t* __restrict__ pos,
                                                             int32_t* __restrict__ kv_idx,
                                                             uint64_t* __restrict__ mask, int32_t* __restrict__ last_row,
                                                             int32_t* __restrict__ ctx_next, void* ws) {
  SPEC_TL(spec::kTLPrefill);
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= B * R) return;
  const int b = i / R, j = i % R;
  int li = last_idx[b];
  if (li < 0 || li >= R) {
    report(ws, SPEC_ERR_DEVICE, b, li);
    li = R - 1;
  }
  tok[i] = (j == li) ? next_token[b] : (j + 1 < R ? input_ids[(size_t)b * R + j + 1] : 0);
  pos[i] = ctx_len[b] + j;
  kv_idx[i] = j;
  mask[i] = (j >= 63) ? ~0ull : ((2ull << j) - 1ull);
  if (j == 0) {
    last_row[b] = b * R + li;
    if (ctx_next) ctx_next[b] = ctx_len[b] + li + 1;
  }
}

__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ src, const int32_t* __restrict__ rows,
                                                          int n_src, int chunks, uint4* __restrict__ dst, void* ws) {
  SPEC_TL(spec::kTLGather);
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.y;
  int s = rows[r];
  if (s < 0 || s >= n_src) {
    if (threadIdx.x == 0 && blockIdx.x == 0) report(ws, SPEC_ERR_DEVICE, r, s);
    return;
  }
  for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < chunks; c += gridDim.x * blockDim.x)
    dst[(size_t)r * chunks + c] = src[(size_t)s * chunks + c];
}

}  // namespace spec

using namespace spec;

extern "C" spec_status spec_prefill_inputs(int32_t B, int32_t R, const int32_t* input_ids, const int32_t* next_token,
                                           const int32_t* last_idx, const int32_t* ctx_len, int32_t* tok,
                                           int32_t* pos, int32_t* kv_idx, uint64_t* mask, int32_t* last_row,
                                           int32_t* ctx_next, void* ws, spec_stream_t stream) {
  if (B <= 0 || R <= 0 || R > 64) return SPEC_ERR_SHAPE;
  if (!input_ids || !next_token || !last_idx || !ctx_len || !tok || !pos || !kv_idx || !mask || !last_row)
    return SPEC_ERR_ARG;
  const int n = B * R;
  launch_pdl(prefill_inputs_kernel, dim3((n + 255) / 256), dim3(256), 0, stream, B, R, input_ids, next_token,
             last_idx, ctx_len, tok, pos, kv_idx, mask, last_row, ctx_next, ws);
  return last_launch();
}

extern "C" spec_status spec_gather_rows(const void* src, int32_t n_src, int32_t row_bytes, const int32_t* rows,
                                        int32_t n, void* dst, void* ws, spec_stream_t stream) {
  if (n <= 0 || n_src <= 0 || row_bytes <= 0) return SPEC_ERR_SHAPE;
  if (!src || !rows || !dst) return SPEC_ERR_ARG;
  if (row_bytes % 16 || !aligned(src, 16) || !aligned(dst, 16)) return SPEC_ERR_ALIGN;
  const int chunks = row_bytes / 16;
  const int bx = (chunks + 255) / 256;
  launch_pdl(gather_rows_kernel, dim3(bx, n), dim3(256), 0, stream, reinterpret_cast<const uint4*>(src), rows, n_src,
             chunks, reinterpret_cast<uint4*>(dst), ws);
  return last_launch();
}

// per-unit log setter of the instrumented build (no-op otherwise)
SPEC_TL_SETTER(prefill)
