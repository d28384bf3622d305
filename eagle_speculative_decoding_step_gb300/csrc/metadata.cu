// SpecDecodeMetadata index bookkeeping for ragged per-request draft counts.
//
// [NEURON] "Speculative Decoding (EAGLE3) in the vLLM Neuron Framework",
// section "SpecDecodeMetadata: Index Bookkeeping": from the cumulative
// scheduled-token counts and the per-request draft counts, the positions whose
// logits are needed (each request's last num_draft + 1 scheduled positions),
// which of them verify drafts, which one is the bonus position, the cumulative
// draft counts, and the draft token ids (the token scheduled after each
// verified position).  One CTA; requests in chunks of 1024 with a block-wide
// prefix sum, so the indices are built on the device without a host round trip.
#include "common.cuh"
#include "internal.h"

namespace spec {

__global__ void __launch_bounds__(1024) spec_metadata_kernel(int R, const int32_t* __restrict__ cu_sched,
                                                             const int32_t* __restrict__ nd,
                                                             const int32_t* __restrict__ ids,
                                                             int32_t* __restrict__ cu_nd, int32_t* __restrict__ logits,
                                                             int32_t* __restrict__ target, int32_t* __restrict__ bonus,
                                                             int32_t* __restrict__ draft_ids, void* ws) {
  SPEC_TL(spec::kTLMetadata);
  pdl_wait();
  pdl_trigger();
  __shared__ int wsum[32];
  __shared__ int s_carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) s_carry = 0;
  __syncthreads();
  for (int base = 0; base < R; base += blockDim.x) {
    const int r = base + tid;
    int v = (r < R) ? nd[r] : 0;
    if (v < 0) {
      report(ws, SPEC_ERR_DEVICE, r, v);
      v = 0;
    }
    // inclusive scan of v over the block
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int t = (lane < (int)(blockDim.x >> 5)) ? wsum[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, t, o);
        if (lane >= o) t += y;
      }
      wsum[lane] = t;
    }
    __syncthreads();
    const int incl = x + (warp > 0 ? wsum[warp - 1] : 0);
    const int carry = s_carry;
    if (r < R) {
      const int excl = carry + incl - v;            // drafts of earlier requests
      const int off = excl + r;                      // logits entries of earlier requests
      const int start = (r > 0) ? cu_sched[r - 1] : 0;
      int first = cu_sched[r] - (v + 1);
      if (first < start) {
        report(ws, SPEC_ERR_DEVICE, r, first);
        first = start;
      }
      cu_nd[r] = carry + incl;
      for (int j = 0; j <= v; ++j) logits[off + j] = first + j;
      for (int j = 0; j < v; ++j) {
        target[excl + j] = off + j;
        if (draft_ids) draft_ids[excl + j] = ids[first + j + 1];
      }
      bonus[r] = off + v;
    }
    __syncthreads();
    if (tid == blockDim.x - 1) s_carry = carry + incl;
    __syncthreads();
  }
}

}  // namespace spec

using namespace spec;

extern "C" spec_status spec_decode_metadata(int32_t R, const int32_t* cu_num_scheduled, const int32_t* num_draft,
                                            const int32_t* input_ids, int32_t* cu_num_draft,
                                            int32_t* logits_indices, int32_t* target_logits_indices,
                                            int32_t* bonus_logits_indices, int32_t* draft_token_ids, void* ws,
                                            spec_stream_t stream) {
  if (R <= 0) return SPEC_ERR_SHAPE;
  if (!cu_num_scheduled || !num_draft || !cu_num_draft || !logits_indices || !target_logits_indices ||
      !bonus_logits_indices)
    return SPEC_ERR_ARG;
  if (draft_token_ids && !input_ids) return SPEC_ERR_ARG;
  if (ws && !aligned(ws, 256)) return SPEC_ERR_WORKSPACE;
  launch_pdl(spec_metadata_kernel, dim3(1), dim3(1024), 0, stream, R, cu_num_scheduled, num_draft, input_ids,
             cu_num_draft, logits_indices, target_logits_indices, bonus_logits_indices, draft_token_ids, ws);
  return last_launch();
}

// per-unit log setter of the instrumented build (no-op otherwise)
SPEC_TL_SETTER(metadata)
