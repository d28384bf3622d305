// C-ABI entry points of the draft step: argument checks, workspace layout,
// kernel sequencing.  The kernels live in layer.cu (prologue, epilogues,
// attention, statistics), tc_gemm.cu (tensor-core GEMM) and lmhead.cu (fused
// LM-head GEMM + top-k / log-softmax epilogue).
#include <algorithm>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace spec {

// launchers (layer.cu, tc_gemm.cu, lmhead.cu)
void launch_prologue(const spec_model_desc&, const spec_rows&, const spec_weights&, const void*, void*, float2*,
                     void*, cudaStream_t);
void launch_epi_store(int, const float*, const SKPlan&, int, int, void*, int, cudaStream_t);
void launch_epi_qkv(const spec_model_desc&, const float*, const SKPlan&, const spec_rows&, const float2*, void*,
                    const spec_kv&, int*, void*, cudaStream_t);
void launch_epi_oproj(const spec_model_desc&, const float*, const SKPlan&, const spec_rows&, const void*,
                      const spec_weights&, float*, void*, cudaStream_t);
void launch_epi_swiglu(const spec_model_desc&, const float*, const SKPlan&, int, void*, cudaStream_t);
void launch_epi_fcnorm(const spec_model_desc&, const float*, const SKPlan&, int, float*, const void*, void*,
                       cudaStream_t);
void launch_epi_down(const spec_model_desc&, const float*, const SKPlan&, int, float*, const spec_weights&, void*,
                     void*, cudaStream_t);
void launch_simt_gemm(int, const void*, const void*, const void*, int, const void*, int, const SKPlan&, float*,
                      cudaStream_t);
spec_status launch_tc_gemm(const void* const*, const int*, int, int, const void*, int, const SKPlan&, float*, void*,
                           cudaStream_t);
int tc_mpad(int M);
int attn_splits(int B, int nkv, int nqg, int sms, int max_keys);
int attn_splits_max(const spec_model_desc& d, int M, int sms);
int attn_qmax(int rows_per_req, int G);
spec_status launch_attention(const spec_model_desc&, const spec_rows&, const void*, const spec_kv&, float*, float2*,
                             void*, int, int*, void*, cudaStream_t);
void launch_row_stats(const float*, int, int, int, int32_t*, int, float*, float*, const int32_t*, cudaStream_t);
void launch_topk_select(const float*, int, int, int, int32_t*, cudaStream_t);
void launch_rescore(int, const void*, const void*, int, int, const int32_t*, int, int, float*, void*, cudaStream_t);
void launch_cand_best(const float*, const int32_t*, int, int, int, int32_t*, int, float*, cudaStream_t);
spec_status launch_lm_head_fused(const spec_model_desc&, const void*, const void*, int, int, int32_t*, int, float*,
                                 float*, const int32_t*, void*, size_t, cudaStream_t);
size_t lm_fused_ws_bytes(int M, int sms);
spec_status launch_tc_gemm_store(const void* W, int N, int K, const void* X, int M, float* out, int ld, void* ws,
                                 cudaStream_t st);

int sm_count() {
  static int cached_dev = -1, cached = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev != cached_dev) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached = n;
    cached_dev = dev;
  }
  return cached;
}

SKPlan make_plan(const int* rows, int nmat, int K, int M, int G) {
  SKPlan p{};
  p.nmat = nmat;
  p.obase[0] = 0;
  p.tbase[0] = 0;
  for (int i = 0; i < nmat; ++i) {
    p.obase[i + 1] = p.obase[i] + rows[i];
    p.tbase[i + 1] = p.tbase[i] + (rows[i] + 127) / 128;
  }
  for (int i = nmat + 1; i < 4; ++i) {
    p.obase[i] = p.obase[nmat];
    p.tbase[i] = p.tbase[nmat];
  }
  p.ntiles = p.tbase[nmat];
  p.kc = (K + 63) / 64;
  p.T = (long long)p.ntiles * p.kc;
  // at least kMinIters iterations per CTA (a tiny GEMM -- one tile, long K -- would
  // otherwise leave one partial per CTA for its epilogue to add up), but every tile
  // keeps a CTA of its own
  constexpr long long kMinIters = 4;
  p.G = (int)std::min<long long>(G, std::max<long long>(p.ntiles, (p.T + kMinIters - 1) / kMinIters));
  if (p.G < 1) p.G = 1;
  p.mpad = tc_mpad(M);
  int ms = 1;
  for (int c = 0; c < p.G; ++c) {
    const long long b = (long long)c * p.T / p.G, e = (long long)(c + 1) * p.T / p.G;
    if (e <= b) continue;
    const int segs = (int)((e - 1) / p.kc - b / p.kc + 1);
    ms = std::max(ms, segs);
  }
  p.maxseg = ms;
  // device-side plan arithmetic is 32-bit
  if ((unsigned long long)p.T * (unsigned long long)(p.G + 1) >= (1ull << 32)) p.G = 0;
  return p;
}

size_t plan_partial_bytes(const SKPlan& p) { return (size_t)p.G * p.maxseg * p.mpad * 128 * 4; }

static int es_of(const spec_model_desc& d) { return d.dtype == SPEC_DTYPE_BF16 ? 2 : 4; }

WsLayout ws_layout(const spec_model_desc& d, int M, int /*max_ctx*/, int sms) {
  WsLayout L{};
  const size_t es = es_of(d);
  const int H = d.hidden, nq = d.n_q_heads, nkv = d.n_kv_heads, hd = d.head_dim, I = d.intermediate, V = d.vocab;
  const int r = d.rank > 0 ? d.rank : 0;
  size_t o = kWsHeader;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align_up(o + bytes, 256);
    return at;
  };
  L.err = 0;
  L.x = take((size_t)M * 2 * H * es);
  L.q = take((size_t)M * nq * hd * es + (size_t)M * (hd / 2) * 8);     // q + rotary table
  const int smax = attn_splits_max(d, M, sms);
  L.attn_splits = smax;
  L.attn_part = take((size_t)M * nq * smax * hd * 4 + (size_t)M * nq * smax * 8);
  L.attn_work = take(4);                       // the attention's item counter
  L.attn = take((size_t)M * nq * hd * es);
  L.r1 = take((size_t)M * H * 4);
  L.n = take((size_t)M * H * es);
  L.act = take((size_t)M * I * es);
  const int G = sms;
  size_t pb = 0;
  auto upd = [&](std::initializer_list<int> rows, int K) {
    std::vector<int> v(rows);
    pb = std::max(pb, plan_partial_bytes(make_plan(v.data(), (int)v.size(), K, M, G)));
  };
  upd({H}, 3 * H);
  upd({nq * hd, nkv * hd, nkv * hd}, 2 * H);
  upd({H}, nq * hd);
  upd({I, I}, H);
  upd({H}, I);
  upd({V}, H);
  if (r > 0) {
    upd({r}, H);
    upd({V}, r);
  }
  L.part = take(pb);
  L.lm_part = take(lm_fused_ws_bytes(M, sms));
  L.logits = take((size_t)M * V * 4);
  L.z = take((size_t)M * (r > 0 ? r : 1) * es);
  const int Kc = d.num_candidates > 0 ? d.num_candidates : 1;
  L.cand = take((size_t)M * Kc * 8);
  L.total = o;
  return L;
}

static spec_status check_desc(const spec_model_desc* d) {
  if (!d) return SPEC_ERR_ARG;
  if (d->hidden <= 0 || d->n_q_heads <= 0 || d->n_kv_heads <= 0 || d->head_dim <= 0 || d->intermediate <= 0 ||
      d->vocab <= 0)
    return SPEC_ERR_SHAPE;
  if (d->n_q_heads % d->n_kv_heads != 0 || d->head_dim % 2 != 0) return SPEC_ERR_SHAPE;
  if (d->dtype != SPEC_DTYPE_BF16 && d->dtype != SPEC_DTYPE_F32) return SPEC_ERR_UNSUPPORTED;
  if (d->window < 0 || (d->window > 0 && d->window < 64)) return SPEC_ERR_SHAPE;
  if (d->rank < 0 || (d->rank > 0 && (d->num_candidates <= 0 || d->num_candidates > 1024 ||
                                      d->num_candidates > d->vocab)))
    return SPEC_ERR_SHAPE;
  if (d->draft_vocab < 0 || d->draft_vocab > d->vocab || (d->draft_vocab > 0 && d->rank > 0)) return SPEC_ERR_SHAPE;
  if (d->dtype == SPEC_DTYPE_BF16) {
    // TMA rows must be multiples of 16 bytes
    if (d->hidden % 8 || d->intermediate % 8 || (d->n_q_heads * d->head_dim) % 8 || (d->rank > 0 && d->rank % 8))
      return SPEC_ERR_SHAPE;
  }
  return SPEC_OK;
}

static spec_status check_ws(const spec_model_desc& d, int M, void* ws, size_t bytes, WsLayout* L) {
  if (!ws) return SPEC_ERR_WORKSPACE;
  if (!aligned(ws, 256)) return SPEC_ERR_WORKSPACE;
  *L = ws_layout(d, M, 0, sm_count());
  if (bytes < L->total) return SPEC_ERR_WORKSPACE;
  return SPEC_OK;
}

static int max_rows_for(const spec_model_desc& d) { return d.dtype == SPEC_DTYPE_BF16 ? 384 : 32; }

// Partial sums of X[M, K] @ [W...]^T with the model dtype's GEMM.
static spec_status gemm(const spec_model_desc& d, std::initializer_list<const void*> Wl,
                        std::initializer_list<int> rowsl, int K, const void* X, int M, float* part, void* ws,
                        cudaStream_t st, SKPlan* plan_out) {
  const void* W[3] = {nullptr, nullptr, nullptr};
  int rows[3] = {0, 0, 0};
  int n = 0;
  for (const void* w : Wl) W[n++] = w;
  n = 0;
  for (int r : rowsl) rows[n++] = r;
  const int nmat = n;
  for (int i = 0; i < nmat; ++i)
    if (!W[i]) return SPEC_ERR_ARG;
  SKPlan p = make_plan(rows, nmat, K, M, sm_count());
  if (p.G <= 0) return SPEC_ERR_SHAPE;
  *plan_out = p;
  if (d.dtype == SPEC_DTYPE_BF16) return launch_tc_gemm(W, rows, nmat, K, X, M, p, part, ws, st);
  launch_simt_gemm(d.dtype, W[0], W[1] ? W[1] : W[0], W[2] ? W[2] : W[0], K, X, M, p, part, st);
  return last_launch();
}

template <typename Tp> static inline Tp* at(void* ws, size_t off) {
  return reinterpret_cast<Tp*>(static_cast<char*>(ws) + off);
}

}  // namespace spec

using namespace spec;

extern "C" const char* spec_status_string(int s) {
  switch (s) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_ARG: return "invalid argument";
    case SPEC_ERR_SHAPE: return "invalid or unsupported shape";
    case SPEC_ERR_UNSUPPORTED: return "unsupported";
    case SPEC_ERR_CAPACITY: return "capacity exceeded";
    case SPEC_ERR_CUDA: return "CUDA error";
    case SPEC_ERR_DEVICE: return "device-side index check failed";
    case SPEC_ERR_TIMEOUT: return "device-side wait timed out";
    case SPEC_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case SPEC_ERR_ALIGN: return "pointer misaligned";
    default: return "unknown status";
  }
}

extern "C" int spec_version(void) { return 1; }

extern "C" size_t spec_workspace_bytes(const spec_model_desc* desc, int32_t max_rows, int32_t max_ctx) {
  if (check_desc(desc) != SPEC_OK || max_rows <= 0) return 0;
  // the layout of a call depends on its own row count (not monotonically):
  // size for the largest over every row count up to max_rows
  size_t best = 0;
  const int sms = sm_count();
  for (int m = 1; m <= max_rows; ++m) best = std::max(best, ws_layout(*desc, m, max_ctx, sms).total);
  return best;
}

extern "C" spec_status spec_get_device_error(const void* ws, int32_t* code_out, spec_stream_t stream) {
  if (!ws || !code_out) return SPEC_ERR_ARG;
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, stream) != cudaSuccess) return SPEC_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return SPEC_ERR_CUDA;
  *code_out = v;
  return SPEC_OK;
}

extern "C" spec_status spec_clear_device_error(void* ws, spec_stream_t stream) {
  if (!ws) return SPEC_ERR_ARG;
  return cuda_status(cudaMemsetAsync(ws, 0, kWsHeader, stream));
}

extern "C" spec_status spec_fc_fuse(const spec_model_desc* desc, const spec_weights* w, const void* aux, void* h0,
                                    int32_t M, void* ws, size_t ws_bytes, spec_stream_t stream) {
  spec_status s = check_desc(desc);
  if (s != SPEC_OK) return s;
  if (!w || !w->fc || !aux || !h0) return SPEC_ERR_ARG;
  const spec_model_desc& d = *desc;
  if (d.fc_norm && !w->fc_norm) return SPEC_ERR_ARG;
  if (M <= 0 || M > max_rows_for(d)) return SPEC_ERR_SHAPE;
  if (!aligned(aux, 16) || !aligned(h0, 16) || !aligned(w->fc, 16)) return SPEC_ERR_ALIGN;
  WsLayout L;
  if ((s = check_ws(d, M, ws, ws_bytes, &L)) != SPEC_OK) return s;
  float* part = at<float>(ws, L.part);
  SKPlan p;
  if ((s = gemm(d, {w->fc}, {d.hidden}, 3 * d.hidden, aux, M, part, ws, stream, &p)) != SPEC_OK) return s;
  if (d.fc_norm)
    launch_epi_fcnorm(d, part, p, M, at<float>(ws, L.r1), w->fc_norm, h0, stream);
  else
    launch_epi_store(d.dtype, part, p, M, d.hidden, h0, d.hidden, stream);
  return last_launch();
}

extern "C" spec_status spec_draft_layer(const spec_model_desc* desc, const spec_weights* w, const spec_rows* rows,
                                        const void* hid_in, void* hid_prenorm, void* hid_normed, const spec_kv* kv,
                                        void* ws, size_t ws_bytes, spec_stream_t stream) {
  spec_status s = check_desc(desc);
  if (s != SPEC_OK) return s;
  if (!w || !rows || !hid_in || !hid_prenorm || !hid_normed || !kv) return SPEC_ERR_ARG;
  const spec_model_desc& d = *desc;
  const spec_rows& r = *rows;
  if (r.M <= 0 || r.M > max_rows_for(d) || r.B <= 0 || r.rows_per_req <= 0 || r.B * r.rows_per_req != r.M)
    return SPEC_ERR_SHAPE;
  if (r.step < 0 || r.step >= 64) return SPEC_ERR_SHAPE;
  if (!r.ctx_len || !r.tok) return SPEC_ERR_ARG;
  if (!w->embed || !w->hidden_norm || !w->in_norm || !w->post_norm || !w->final_norm || !w->wq || !w->wk ||
      !w->wv || !w->wo || !w->wgate || !w->wup || !w->wdown)
    return SPEC_ERR_ARG;
  if (!kv->k || !kv->v || !kv->block_table || kv->block_size <= 0 || kv->max_blocks <= 0 || kv->num_slots <= 0)
    return SPEC_ERR_ARG;
  if (d.head_dim != 64 && d.head_dim != 128) return SPEC_ERR_UNSUPPORTED;
  if (!aligned(kv->k, 16) || !aligned(kv->v, 16) || !aligned(hid_in, 16) || !aligned(hid_prenorm, 16) ||
      !aligned(hid_normed, 16))
    return SPEC_ERR_ALIGN;
  WsLayout L;
  if ((s = check_ws(d, r.M, ws, ws_bytes, &L)) != SPEC_OK) return s;
  const int M = r.M, H = d.hidden, nq = d.n_q_heads, nkv = d.n_kv_heads, hd = d.head_dim, I = d.intermediate;
  const size_t es = es_of(d);
  void* x = at<void>(ws, L.x);
  void* qbuf = at<void>(ws, L.q);
  float2* cs = reinterpret_cast<float2*>(static_cast<char*>(qbuf) + align_up((size_t)M * nq * hd * es, 16));
  float* opart = at<float>(ws, L.attn_part);
  float2* mlpart = reinterpret_cast<float2*>(opart + (size_t)M * nq * L.attn_splits * hd);
  void* attn = at<void>(ws, L.attn);
  float* r1 = at<float>(ws, L.r1);
  void* nbuf = at<void>(ws, L.n);
  void* act = at<void>(ws, L.act);
  float* part = at<float>(ws, L.part);
  SKPlan p;

  launch_prologue(d, r, *w, hid_in, x, cs, ws, stream);
  if ((s = gemm(d, {w->wq, w->wk, w->wv}, {nq * hd, nkv * hd, nkv * hd}, 2 * H, x, M, part, ws, stream, &p)) !=
      SPEC_OK)
    return s;
  int* work = at<int>(ws, L.attn_work);
  launch_epi_qkv(d, part, p, r, cs, qbuf, *kv, work, ws, stream);
  const int G = nq / nkv;
  const int qmax = attn_qmax(r.rows_per_req, G);
  const int nqg = (r.rows_per_req * G + qmax - 1) / qmax;
  int max_keys = 0;
  if (r.max_ctx > 0) max_keys = (d.window > 0 ? std::min(r.max_ctx, d.window) : r.max_ctx) + 64;
  const int nsplit = std::min(attn_splits(r.B, nkv, nqg, sm_count(), max_keys), L.attn_splits);
  if ((s = launch_attention(d, r, qbuf, *kv, opart, mlpart, attn, nsplit, work, ws, stream)) != SPEC_OK) return s;
  if ((s = gemm(d, {w->wo}, {H}, nq * hd, attn, M, part, ws, stream, &p)) != SPEC_OK) return s;
  launch_epi_oproj(d, part, p, r, hid_in, *w, r1, nbuf, stream);
  if ((s = gemm(d, {w->wgate, w->wup}, {I, I}, H, nbuf, M, part, ws, stream, &p)) != SPEC_OK) return s;
  launch_epi_swiglu(d, part, p, M, act, stream);
  if ((s = gemm(d, {w->wdown}, {H}, I, act, M, part, ws, stream, &p)) != SPEC_OK) return s;
  launch_epi_down(d, part, p, M, r1, *w, hid_prenorm, hid_normed, stream);
  return last_launch();
}

extern "C" spec_status spec_lm_head(const spec_model_desc* desc, const spec_weights* w, const void* hn, int32_t M,
                                    int32_t k, int32_t* topk_ids, int32_t ids_ld, float* topk_logprob, float* lse,
                                    float* logits_or_null, void* ws, size_t ws_bytes, spec_stream_t stream) {
  spec_status s = check_desc(desc);
  if (s != SPEC_OK) return s;
  if (!w || !w->lm_head || !hn || !topk_ids || !topk_logprob) return SPEC_ERR_ARG;
  const spec_model_desc& d = *desc;
  if (M <= 0 || M > max_rows_for(d)) return SPEC_ERR_SHAPE;
  // a reduced draft vocabulary: lm_head has draft_vocab rows, ids map through d2t
  const int dv = d.draft_vocab > 0 ? d.draft_vocab : d.vocab;
  const int32_t* d2t = d.draft_vocab > 0 ? w->d2t : nullptr;
  if (d.draft_vocab > 0 && !d2t) return SPEC_ERR_ARG;
  if (k < 1 || k > 8 || k > dv) return SPEC_ERR_SHAPE;
  if (ids_ld == 0) ids_ld = k;
  if (ids_ld < k) return SPEC_ERR_SHAPE;
  if (!aligned(hn, 16) || !aligned(w->lm_head, 16)) return SPEC_ERR_ALIGN;
  WsLayout L;
  if ((s = check_ws(d, M, ws, ws_bytes, &L)) != SPEC_OK) return s;
  if (d.dtype == SPEC_DTYPE_BF16 && logits_or_null == nullptr && M <= 64)
    return launch_lm_head_fused(d, hn, w->lm_head, M, k, topk_ids, ids_ld, topk_logprob, lse, d2t, ws, L.lm_part,
                                stream);
  float* part = at<float>(ws, L.part);
  float* logits = logits_or_null ? logits_or_null : at<float>(ws, L.logits);
  if (d.dtype == SPEC_DTYPE_BF16) {
    if ((s = launch_tc_gemm_store(w->lm_head, dv, d.hidden, hn, M, logits, dv, ws, stream)) != SPEC_OK) return s;
  } else {
    SKPlan p;
    if ((s = gemm(d, {w->lm_head}, {dv}, d.hidden, hn, M, part, ws, stream, &p)) != SPEC_OK) return s;
    launch_epi_store(SPEC_DTYPE_F32, part, p, M, dv, logits, dv, stream);
  }
  launch_row_stats(logits, M, dv, k, topk_ids, ids_ld, topk_logprob, lse, d2t, stream);
  return last_launch();
}

extern "C" spec_status spec_lowrank_candidates(const spec_model_desc* desc, const spec_weights* w, const void* hn,
                                               int32_t M, int32_t k_out, int32_t* cand_ids, float* cand_logits,
                                               int32_t* out_ids, float* out_logprob, int32_t out_ld, void* ws,
                                               size_t ws_bytes, spec_stream_t stream) {
  spec_status s = check_desc(desc);
  if (s != SPEC_OK) return s;
  const spec_model_desc& d = *desc;
  if (d.rank <= 0) return SPEC_ERR_UNSUPPORTED;
  if (!w || !w->lr_down || !w->lr_up || !w->lm_head || !hn || !out_ids) return SPEC_ERR_ARG;
  if (M <= 0 || M > max_rows_for(d)) return SPEC_ERR_SHAPE;
  const int Kc = d.num_candidates;
  if (k_out < 1 || k_out > 8 || k_out > Kc) return SPEC_ERR_SHAPE;
  if (out_ld == 0) out_ld = k_out;
  if (out_ld < k_out) return SPEC_ERR_SHAPE;
  if (!aligned(hn, 16)) return SPEC_ERR_ALIGN;
  WsLayout L;
  if ((s = check_ws(d, M, ws, ws_bytes, &L)) != SPEC_OK) return s;
  float* part = at<float>(ws, L.part);
  void* z = at<void>(ws, L.z);
  float* sc = at<float>(ws, L.logits);
  int32_t* cand = cand_ids ? cand_ids : at<int32_t>(ws, L.cand);
  float* exact = cand_logits ? cand_logits : reinterpret_cast<float*>(at<int32_t>(ws, L.cand) + (size_t)M * Kc);
  SKPlan p;
  if ((s = gemm(d, {w->lr_down}, {d.rank}, d.hidden, hn, M, part, ws, stream, &p)) != SPEC_OK) return s;
  launch_epi_store(d.dtype, part, p, M, d.rank, z, d.rank, stream);
  if (d.dtype == SPEC_DTYPE_BF16) {
    if ((s = launch_tc_gemm_store(w->lr_up, d.vocab, d.rank, z, M, sc, d.vocab, ws, stream)) != SPEC_OK) return s;
  } else {
    if ((s = gemm(d, {w->lr_up}, {d.vocab}, d.rank, z, M, part, ws, stream, &p)) != SPEC_OK) return s;
    launch_epi_store(SPEC_DTYPE_F32, part, p, M, d.vocab, sc, d.vocab, stream);
  }
  launch_topk_select(sc, M, d.vocab, Kc, cand, stream);
  launch_rescore(d.dtype, hn, w->lm_head, d.hidden, d.vocab, cand, M, Kc, exact, ws, stream);
  launch_cand_best(exact, cand, M, Kc, k_out, out_ids, out_ld, out_logprob, stream);
  return last_launch();
}
