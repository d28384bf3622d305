// Host-side internals shared by the translation units of libeaglespec.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/eaglespec.h"

namespace spec {

int sm_count();                 // SMs of the current device (cached per device)
inline spec_status cuda_status(cudaError_t e) { return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA; }
inline spec_status last_launch() { return cuda_status(cudaGetLastError()); }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ---------------------------------------------------------------- stream-K plan
// The weight matrix (rows = output features, up to three stacked matrices) is
// cut into 128-row tiles and K into 64-wide chunks; the tiles x chunks
// iteration space is split evenly over G CTAs.  CTA c owns iterations
// [c*T/G, (c+1)*T/G); each maximal run inside one tile is a "segment" whose
// fp32 partial sums go to slot (c, j) (j-th segment of CTA c).
struct SKPlan {
  int ntiles;      // 128-row tiles over all stacked matrices
  int kc;          // 64-wide K chunks
  int G;           // CTAs
  int maxseg;      // segments per CTA (slot stride)
  int mpad;        // padded rows of the activation operand (columns of a partial)
  long long T;     // ntiles * kc
  // stacked matrices: output row n in [obase[i], obase[i+1]) belongs to matrix i,
  // whose tiles are [tbase[i], tbase[i+1])
  int nmat;
  int obase[4];
  int tbase[4];
};

SKPlan make_plan(const int* rows_per_mat, int nmat, int K, int M, int G);
size_t plan_partial_bytes(const SKPlan& p);

// Bytes of the workspace regions of the draft-layer / head entry points.
struct WsLayout {
  size_t err, x, q, attn_part, attn_work, attn, r1, n, act, part, lm_part, logits, z, cand, total;
  int attn_splits;
};
WsLayout ws_layout(const spec_model_desc& d, int max_rows, int max_ctx, int sms);

}  // namespace spec
