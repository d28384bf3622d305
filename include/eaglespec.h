/*
 * libeaglespec -- the data-parallel hot path of EAGLE-3 / EAGLE-4 speculative
 * decoding on one NVIDIA GB300 (sm_103a): draft step, top-k tree expansion,
 * verification.
 *
 * Sources the operations follow (cited per entry point below):
 *   [NEURON] "Speculative Decoding (EAGLE3) in the vLLM Neuron Framework"
 *            (AWS Neuron vLLM plugin design document).
 *   [EAGLET] "Eaglet" (Qualcomm QAIRT documentation).
 *   [EAGLE4] "nemo_automodel.components.speculative.eagle.eagle4" (NVIDIA NeMo
 *            AutoModel API page).
 *   [QUARK]  "EAGLE-3" (AMD Quark documentation).
 *
 * Conventions for every entry point:
 *   - Every tensor pointer is a DEVICE pointer owned by the caller, except the
 *     descriptor structs themselves (host memory, read during the call only).
 *     The library allocates no device memory: scratch space comes from a
 *     caller-provided workspace (``ws``, ``ws_bytes``) sized by the matching
 *     ``*_workspace_bytes`` query, 256-byte aligned.
 *   - Calls are asynchronous on ``stream`` (a cudaStream_t; NULL = the legacy
 *     default stream).  They do no host synchronisation and no host<->device
 *     copies, so a sequence of calls can be captured into a CUDA graph.
 *   - Shapes, alignment and capacities are checked on the host before any
 *     launch; a violation returns an error status and launches nothing.
 *   - A launch failure returns SPEC_ERR_CUDA.  Violations that can only be seen
 *     on the device (a token id outside the vocabulary, a cache index outside
 *     the block table, a parent index that does not precede its node, a
 *     bounded wait that ran out) set an error word at the start of the
 *     workspace and the kernel skips the offending access; read it with
 *     spec_get_device_error.  No kernel traps.
 *   - Matrices are row-major.  Weights use the nn.Linear layout [out, in].
 *     Token ids are int32; -1 marks rejected output positions.
 *   - dtype SPEC_DTYPE_BF16: weights, activations and the K/V cache are bf16
 *     with fp32 accumulation; SPEC_DTYPE_F32: everything fp32.
 */
#ifndef EAGLESPEC_H
#define EAGLESPEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *spec_stream_t; /* == cudaStream_t */

typedef enum {
  SPEC_OK = 0,
  SPEC_ERR_ARG = -1,          /* NULL pointer or invalid scalar argument */
  SPEC_ERR_SHAPE = -2,        /* inconsistent or unsupported sizes */
  SPEC_ERR_UNSUPPORTED = -3,  /* valid request this build does not implement */
  SPEC_ERR_CAPACITY = -4,     /* cache / tree / workspace capacity exceeded */
  SPEC_ERR_CUDA = -5,         /* a CUDA runtime call or launch failed */
  SPEC_ERR_DEVICE = -6,       /* device-side index check failed (error word) */
  SPEC_ERR_TIMEOUT = -7,      /* a bounded device-side wait ran out */
  SPEC_ERR_WORKSPACE = -8,    /* workspace missing, too small or misaligned */
  SPEC_ERR_ALIGN = -9         /* a pointer lacks the alignment the kernels need */
} spec_status;

enum { SPEC_DTYPE_F32 = 0, SPEC_DTYPE_BF16 = 1 };

/* Shape of the single-layer EAGLE-3 draft model ([NEURON] "Eagle3 Draft Model
 * Architecture"; window, rank and num_candidates from [EAGLE4]
 * Eagle4Config.sliding_window and Eagle4CandidateHeadConfig). */
typedef struct {
  int32_t hidden;         /* H */
  int32_t n_q_heads;      /* query heads; a multiple of n_kv_heads */
  int32_t n_kv_heads;     /* key/value heads (grouped-query attention) */
  int32_t head_dim;       /* even */
  int32_t intermediate;   /* SwiGLU MLP width I */
  int32_t vocab;          /* V */
  int32_t dtype;          /* SPEC_DTYPE_* */
  float rms_eps;          /* RMSNorm epsilon */
  float rope_theta;       /* rotary base */
  int32_t window;         /* sliding window W in keys (itself included); 0 = full
                             causal.  When > 0 it must be >= 64 so every
                             draft-region key of a row is inside the window. */
  int32_t rank;           /* rank r of the EAGLE-4 candidate head; 0 = none */
  int32_t num_candidates; /* candidates kept from the low-rank scores (Kc) */
  int32_t draft_vocab;    /* rows of lm_head when the draft predicts over a
                             reduced vocabulary ([QUARK] calibrate_draft_vocab,
                             draft_vocab_size; [EAGLE4] selected_token_ids);
                             0 = the full vocabulary.  Needs weights.d2t. */
  int32_t fc_norm;        /* EAGLE-3.1 ([QUARK] "Background: EAGLE-3 and
                             EAGLE-3.1", eagle_architecture_config.fc_norm):
                             nonzero = spec_fc_fuse ends with an RMSNorm of the
                             fused feature, gain weights.fc_norm.  The page names
                             the flag only; this is the reading implemented. */
  int32_t norm_output;    /* EAGLE-3.1 norm_output: nonzero = the caller feeds the
                             normalised output (hid_normed) of a draft pass, not
                             hidden_prenorm, to the next pass.  No library call
                             changes with it; the step sequences built on the
                             library (the Python engine) read it. */
} spec_model_desc;

/* Draft weights, device pointers, dtype of the descriptor.  [NEURON] "Eagle3
 * Draft Model Architecture" (fc, embed_tokens, the decoder layer's norms and
 * projections with QKV sized for 2H input, final norm, LM head); [EAGLE4]
 * CANDIDATE_HEAD_KEYS (efficient_lm_head_down_proj, efficient_lm_head). */
typedef struct {
  const void *fc;          /* [H, 3H] */
  const void *embed;       /* [V, H] */
  const void *hidden_norm; /* [H] gain of the norm on the incoming hidden state */
  const void *in_norm;     /* [H] input_layernorm gain (on the token embedding) */
  const void *post_norm;   /* [H] post_attention_layernorm gain */
  const void *final_norm;  /* [H] final norm gain */
  const void *wq;          /* [nq*hd, 2H] */
  const void *wk;          /* [nkv*hd, 2H] */
  const void *wv;          /* [nkv*hd, 2H] */
  const void *wo;          /* [H, nq*hd] */
  const void *wgate;       /* [I, H] */
  const void *wup;         /* [I, H] */
  const void *wdown;       /* [H, I] */
  const void *lm_head;     /* [V, H] */
  const void *lr_down;     /* [r, H]  efficient_lm_head_down_proj (rank > 0) */
  const void *lr_up;       /* [V, r]  efficient_lm_head (rank > 0) */
  const int32_t *d2t;      /* [draft_vocab] target token id of each draft-vocabulary
                              entry (draft_vocab > 0); lm_head is then
                              [draft_vocab, H] */
  const void *fc_norm;     /* [H] gain of the RMSNorm after the FC (desc.fc_norm) */
} spec_weights;

/* Paged K/V cache of the draft layer ([NEURON] "KV Cache Sharing" and
 * "EagleProposer", recurrent phase).  Logical cache index j of request b lives
 * in slot block_table[b * max_blocks + j / block_size] * block_size
 * + j % block_size.  k and v are [num_slots, n_kv_heads, head_dim] in the
 * model dtype; keys are stored after the rotary embedding. */
typedef struct {
  void *k;
  void *v;
  const int32_t *block_table; /* [B, max_blocks] */
  int32_t block_size;
  int32_t max_blocks;
  int32_t num_slots;
} spec_kv;

/* The rows of one draft pass.  Rows of request b are [b*rows_per_req,
 * (b+1)*rows_per_req); M = B * rows_per_req.  Request b's context occupies
 * cache indices [0, ctx_len[b]); the draft region that follows holds up to 64
 * draft / tree entries, entry i at cache index ctx_len[b] + i.
 *
 * A row writes its K/V at draft-region entry kv_idx, sits at rotary position
 * pos, and attends to the context (with a window: positions > pos - W only)
 * plus every draft-region entry whose bit is set in mask (its own included).
 * A NULL array takes the chain value for draft step ``step`` ([NEURON]
 * "EagleProposer": positions advance by one per recurrent pass):
 *   pos = ctx_len[b] + step, kv_idx = step, mask = bits 0..step,
 *   hid_src = the row itself. */
typedef struct {
  int32_t M;
  int32_t B;
  int32_t rows_per_req;
  int32_t step;
  const int32_t *ctx_len;  /* [B] */
  const int32_t *tok;      /* input token of row m at tok[m * tok_stride] */
  int32_t tok_stride;      /* 0 means 1 */
  const int32_t *pos;      /* [M] or NULL */
  const int32_t *kv_idx;   /* [M] or NULL; each < 64 */
  const uint64_t *mask;    /* [M] or NULL */
  const int32_t *hid_src;  /* [M] or NULL: row of hid_in feeding row m */
  int32_t max_ctx;         /* an upper bound of ctx_len[b] over the batch, or 0 if
                              unknown; only sizes the attention's key splits */
} spec_rows;

/* Outputs of tree expansion (spec_tree_expand).  Frontier arrays hold the next
 * draft pass's rows (B * top_k rows, in spec_rows form); tree arrays hold the
 * final tree, total+1 nodes per request (node 0 = root). */
typedef struct {
  int32_t *frontier_tok;      /* [B*top_k] */
  int32_t *frontier_pos;      /* [B*top_k] */
  int32_t *frontier_kv_idx;   /* [B*top_k] */
  uint64_t *frontier_mask;    /* [B*top_k] */
  int32_t *frontier_hid_src;  /* [B*top_k] row of the previous pass's output */
  int32_t *tree_tok;          /* [B, total+1] */
  int32_t *tree_parent;       /* [B, total+1], -1 for the root, parent < node */
  int32_t *tree_depth;        /* [B, total+1] */
  int32_t *tree_pos;          /* [B, total+1] ctx_len + depth */
  float *tree_score;          /* [B, total+1] cumulative log-probability */
  uint64_t *tree_mask;        /* [B, total+1] ancestors and self, bit n = node n */
} spec_tree_io;

/* ------------------------------------------------------------------ */
/* Library information and errors.                                     */

const char *spec_status_string(int status);
int spec_version(void);

/* Workspace bytes for spec_fc_fuse / spec_draft_layer / spec_lm_head /
 * spec_lowrank_candidates with at most max_rows rows per call and contexts of
 * at most max_ctx tokens, on the current device.  0 for an invalid descriptor. */
size_t spec_workspace_bytes(const spec_model_desc *desc, int32_t max_rows, int32_t max_ctx);

/* Reads the device error word of a workspace (synchronises ``stream``):
 * SPEC_OK, SPEC_ERR_DEVICE or SPEC_ERR_TIMEOUT in *code_out. */
spec_status spec_get_device_error(const void *ws, int32_t *code_out, spec_stream_t stream);
/* Clears the device error word (asynchronous). */
spec_status spec_clear_device_error(void *ws, spec_stream_t stream);

/* ------------------------------------------------------------------ */
/* Draft step.                                                         */

/* h0 = aux @ fc^T: fuses the three auxiliary target hidden states.
 * [NEURON] "What is EAGLE3?" (FC layer combining the three auxiliary hidden
 * states) and "Eagle3 Draft Model Architecture" (fc: Linear(3H, H); the initial
 * forward mode's combine_hidden_states on [T, 3H]).
 * aux [M, 3H], h0 [M, H], model dtype.  Aux layer choice (e.g. (2, N/2, N-3)
 * or [2, -3, -1]) is the caller's. */
spec_status spec_fc_fuse(const spec_model_desc *desc, const spec_weights *w,
                         const void *aux, void *h0, int32_t M,
                         void *ws, size_t ws_bytes, spec_stream_t stream);

/* One pass of the draft decoder layer over ``rows``.
 * [NEURON] "Eagle3 Draft Model Architecture": embeds = input_layernorm(
 * embed(tok)); hidden = hidden_norm(hid_in); x = cat([embeds, hidden]) (2H);
 * self-attention with QKV sized for 2H input and H output, rotary embedding at
 * pos; out = hid_in + attn; out = mlp(post_attention_layernorm(out)) + out
 * (SwiGLU); returns the pre-norm state (recurrent input of the next pass) and
 * its final norm (input of the LM head).  Attention mask: see spec_rows;
 * sliding window from [EAGLE4] Eagle4Config.sliding_window.
 * K/V of every row are written to the cache (entry ctx_len + kv_idx) before
 * any row attends.  hid_in [*, H] (row hid_src[m] feeds row m),
 * hid_prenorm / hid_normed [M, H]; model dtype.
 * Capacity: ctx_len[b] + 64 must fit in the block table (SPEC_ERR_DEVICE
 * otherwise, detected per row on the device) -- the position cutoff of
 * [NEURON] "Design Choices". */
spec_status spec_draft_layer(const spec_model_desc *desc, const spec_weights *w,
                             const spec_rows *rows, const void *hid_in,
                             void *hid_prenorm, void *hid_normed, const spec_kv *kv,
                             void *ws, size_t ws_bytes, spec_stream_t stream);

/* Full-vocabulary LM head with per-row top-k and log-softmax statistics,
 * without materialising the logits: logits = hn @ lm_head^T; per row the k
 * largest (ties to the smaller id) with log-prob = logit - lse, and
 * lse = log(sum(exp(logits))).
 * [NEURON] "Eagle3 Draft Model Architecture" (LM head) and "Design Choices"
 * (greedy draft sampling: k = 1); top-k per node for trees from [EAGLET]
 * draft_top_k.  With a reduced draft vocabulary (desc.draft_vocab > 0) the
 * softmax and top-k run over the draft_vocab rows of lm_head and the emitted
 * ids are the mapped target ids d2t[row].  hn [M, H]; topk_ids / topk_logprob at [m * ids_ld + j]
 * (ids_ld >= k; 0 means k); lse [M] or NULL; 1 <= k <= 8.
 * logits_or_null: if not NULL, also writes the fp32 logits [M, V]. */
spec_status spec_lm_head(const spec_model_desc *desc, const spec_weights *w,
                         const void *hn, int32_t M, int32_t k,
                         int32_t *topk_ids, int32_t ids_ld, float *topk_logprob,
                         float *lse, float *logits_or_null,
                         void *ws, size_t ws_bytes, spec_stream_t stream);

/* EAGLE-4 rank-r candidate head: s = (hn @ lr_down^T) @ lr_up^T; keep the
 * num_candidates tokens with the largest s (ties to the smaller id), rescore
 * them exactly with lm_head rows, emit the k_out best exact logits.
 * [EAGLE4] module docstring (low-rank head retrieves, serving rescores the
 * retrieved candidates exactly) and Eagle4CandidateHeadConfig.
 * hn [M, H]; cand_ids / cand_logits [M, Kc] (score order) or NULL;
 * out_ids at [m * out_ld + j], 1 <= k_out <= 8 (out_ld 0 means k_out);
 * out_logprob (same layout) or NULL: log-probability of each emitted id under
 * the softmax over the candidates' exact logits (what a top-k draft tree ranks
 * with when it drafts from the candidate head). */
spec_status spec_lowrank_candidates(const spec_model_desc *desc, const spec_weights *w,
                                    const void *hn, int32_t M, int32_t k_out,
                                    int32_t *cand_ids, float *cand_logits,
                                    int32_t *out_ids, float *out_logprob, int32_t out_ld,
                                    void *ws, size_t ws_bytes, spec_stream_t stream);

/* ------------------------------------------------------------------ */
/* Tree expansion.                                                     */

/* Bytes of the tree state (device memory the caller provides). */
size_t spec_tree_state_bytes(int32_t B, int32_t top_k, int32_t draft_depth, int32_t total);

/* One expansion step of a top-k draft tree ranked by cumulative log-prob.
 * [EAGLET] draft_top_k, draft_depth, total_draft_tokens (the draft proposes a
 * tree, the target verifies it in one pass).  Call with depth_idx = 1 after
 * the root pass (topk_* are [B, top_k]; root_tok [B] is read), then with
 * depth_idx = 2 .. draft_depth after each frontier pass (topk_* are
 * [B*top_k, top_k]).  For depth_idx < draft_depth it writes the next
 * frontier rows to io->frontier_*; at depth_idx == draft_depth it selects the
 * total best nodes and writes io->tree_*.  Rules:
 *   depth 1: the root's top_k children, score = log-prob, are the frontier;
 *   depth d >= 2: each frontier node's top_k children, score = parent score +
 *     log-prob (fp32), join the pool; the top_k best form the next frontier;
 *   final: the ``total`` best pool nodes (score, then creation order), numbered
 *     by (depth, score, creation order) after the root.
 * Frontier slot f at depth d uses draft-region entry 1 + (d-1)*top_k + f.
 * Requires total + 1 <= 64, 1 + (draft_depth-1)*top_k <= 64, top_k <= 16,
 * total <= top_k + (draft_depth-1)*top_k^2. */
spec_status spec_tree_expand(int32_t B, int32_t top_k, int32_t depth_idx, int32_t draft_depth,
                             int32_t total, const int32_t *ctx_len, const int32_t *root_tok,
                             const int32_t *topk_ids, const float *topk_logprob,
                             void *tree_state, const spec_tree_io *io, spec_stream_t stream);

/* ------------------------------------------------------------------ */
/* Verification.                                                       */

/* Workspace bytes for the verifiers over B requests of R rows of V logits.
 * Layout: the 256-byte header (error word first), the verifiers' completion
 * counters, chunk records, sampling records, top-k / top-p thresholds.  The
 * workspace must be zero-filled before its first use (the counters start at
 * zero; every call leaves them at zero again).  Header bytes 64..71 hold two
 * optional int32 settings, zero for the defaults: the bound in microseconds on
 * the wait of spec_verify_rejection's sampling CTAs for their request's
 * decision (default 2 s; when it runs out the error word becomes
 * SPEC_ERR_TIMEOUT and that request's emitted token is -1), and a test hook --
 * a value k > 0 keeps request k-1's decision unpublished, so its waits run out.
 * Both verifiers are one kernel launch each (spec_verify_rejection adds one for
 * top-k / top-p thresholds); calls sharing a workspace must not overlap on the
 * GPU. */
size_t spec_verify_workspace_bytes(int32_t B, int32_t R, int32_t V);

/* Greedy verification, one kernel: chunk CTAs reduce the target rows to their
 * argmax; the last CTA of a request to finish (a completion counter, no
 * waiting) makes the request's decisions and moves its K/V.
 * [NEURON] "Rejection Sampling", on-device sampler:
 * t = argmax(target) per row (ties to the smaller id); accept drafts in order
 * until the first mismatch, emit the target token there, or a bonus token when
 * all match; -1 after.  [NEURON] "What is Speculative Decoding?" (bit-exact
 * with target-only greedy decoding).
 *   chain (parent == NULL): target_logits [B, R, V] fp32 with R = K+1,
 *     draft_tok [B, K]; out_tok [B, K+1]; kv_src[b, i] = i for i <= accepted,
 *     -1 after (no K/V moves).
 *   tree (parent != NULL): R = total+1 node rows, draft_tok [B, R] = node
 *     tokens (node 0 = root), parent [B, R] (parent[0] = -1, parent[n] < n).
 *     A node is accepted when its parent is and its token equals the target's
 *     argmax at the parent; the deepest accepted node (smallest index among
 *     equals) gives the path.  out_tok [B, max_depth+1], kv_src [B,
 *     max_depth+1] = node index at each depth of the path, -1 after.  If kv and
 *     desc are not NULL, moves the accepted path's K/V from cache index
 *     ctx_len + node to ctx_len + depth (KV-slot compaction).
 * accept_len [B] = drafts accepted. */
spec_status spec_verify_greedy(int32_t B, int32_t R, int32_t V, const float *target_logits,
                               const int32_t *draft_tok, const int32_t *parent,
                               int32_t max_depth, int32_t *out_tok, int32_t *accept_len,
                               int32_t *kv_src, const spec_model_desc *desc,
                               const spec_kv *kv, const int32_t *ctx_len,
                               void *ws, size_t ws_bytes, spec_stream_t stream);

/* Stochastic verification of a greedy-drafted chain, one kernel: statistics
 * CTAs (max / sum-exp per row chunk), the last of a request's making its
 * accept decisions, then sampling CTAs of the request's one sampled row, which
 * wait (bounded) for that decision.  [NEURON] "Rejection
 * Sampling", CPU sampler (arXiv:2211.17192): p = softmax(target / T); accept
 * draft d at position i when u <= p(d) (draft prob 1); at the first rejection
 * emit argmax_x p(x) / E_x over x != d (Gumbel-max with exponential noise
 * E = -ln u'); if all accepted, a bonus token argmax_x p(x) / E_x at the last
 * row.  temperature[b] <= 0 makes request b greedy.  Uniforms come from
 * Philox4x32-10 (Salmon et al., SC'11) with key = seed and counter
 * (j, i, b, 2*step_offset + purpose): purpose 0 -> acceptance uniform of
 * (b, i) (first word of block 0), purpose 1 -> noise of vocabulary id 4j+l
 * (word l of block j); u = ((x >> 8) + 0.5) * 2^-24.
 * target_logits [B, K+1, V] fp32, draft_tok [B, K], out_tok [B, K+1],
 * accept_len [B], kv_src [B, K+1] (as the greedy chain) or NULL.
 * top_k [B] (0 = off) and top_p [B] (1.0 = off), each NULL for none, filter the
 * target distribution per request before the accept test and both samples
 * ([NEURON] "Rejection Sampling": per-request top-k and top-p): tokens ordered
 * by logit / T (ties to the smaller id), the first top_k kept, then the
 * shortest prefix of those whose renormalised mass reaches top_p. */
spec_status spec_verify_rejection(int32_t B, int32_t K, int32_t V, const float *target_logits,
                                  const int32_t *draft_tok, const float *temperature,
                                  const int32_t *top_k, const float *top_p,
                                  uint64_t seed, uint64_t step_offset, int32_t *out_tok,
                                  int32_t *accept_len, int32_t *kv_src,
                                  void *ws, size_t ws_bytes, spec_stream_t stream);

/* ------------------------------------------------------------------ */
/* Ragged batches.                                                     */

/* SpecDecodeMetadata index builder.  [NEURON] "SpecDecodeMetadata: Index
 * Bookkeeping": for R requests with cumulative scheduled-token counts
 * cu_num_scheduled [R] and draft counts num_draft [R] (each request schedules
 * its last accepted token followed by its drafts):
 *   cu_num_draft [R]            cumulative draft counts;
 *   logits_indices [S + R]      each request's last num_draft+1 scheduled
 *                               positions (S = total drafts);
 *   target_logits_indices [S]   entries of logits_indices that verify drafts;
 *   bonus_logits_indices [R]    the last entry of each request's block;
 *   draft_token_ids [S] or NULL input_ids at the position after each verified
 *                               one (input_ids required then).
 * ws: NULL or a workspace whose error word receives SPEC_ERR_DEVICE when a
 * request schedules fewer than num_draft+1 tokens or a count is negative. */
spec_status spec_decode_metadata(int32_t R, const int32_t *cu_num_scheduled, const int32_t *num_draft,
                                 const int32_t *input_ids, int32_t *cu_num_draft,
                                 int32_t *logits_indices, int32_t *target_logits_indices,
                                 int32_t *bonus_logits_indices, int32_t *draft_token_ids, void *ws,
                                 spec_stream_t stream);

/* Inputs of the batched initial draft pass over the verified tokens ([NEURON]
 * "EagleProposer", propose() prefill phase: the draft processes all target
 * tokens; input ids shifted by one with the new token scattered at the last
 * token position).  Request b verified R tokens input_ids[b, 0..R-1] at
 * positions ctx_len[b] .. ctx_len[b]+R-1 and accepted through row last_idx[b]
 * (0 <= last_idx < R); next_token[b] is the target's new token.  Writes the
 * pass's rows in spec_rows form, all [B*R]:
 *   tok[b*R+j]    = next_token[b] if j == last_idx[b], else input_ids[b, j+1]
 *                   (0 past the end);
 *   pos = ctx_len[b] + j, kv_idx = j, mask = bits 0..j (causal within the
 *   request), and last_row[b] = b*R + last_idx[b] (the row whose LM head gives
 *   the first draft token; gather it with spec_gather_rows), and, if not NULL,
 *   ctx_next[b] = ctx_len[b] + last_idx[b] + 1 (the context of the recurrent
 *   passes that follow).  R <= 64.
 * ws: NULL or a workspace whose error word flags last_idx out of range. */
spec_status spec_prefill_inputs(int32_t B, int32_t R, const int32_t *input_ids, const int32_t *next_token,
                                const int32_t *last_idx, const int32_t *ctx_len, int32_t *tok,
                                int32_t *pos, int32_t *kv_idx, uint64_t *mask, int32_t *last_row,
                                int32_t *ctx_next, void *ws, spec_stream_t stream);

/* dst[r] = src[rows[r]] for r < n; rows of row_bytes bytes (a multiple of 16,
 * 16-byte aligned buffers); src has n_src rows.  An out-of-range index sets the
 * error word of ws (if not NULL) and leaves that row untouched. */
spec_status spec_gather_rows(const void *src, int32_t n_src, int32_t row_bytes, const int32_t *rows,
                             int32_t n, void *dst, void *ws, spec_stream_t stream);

/* Greedy verification without caller-provided scratch.  The paper has no
 * counterpart: this entry point exists for callers that cannot allocate device
 * memory -- a host framework that owns every device buffer and passes only
 * inputs and outputs, a latency-critical loop where cudaMalloc (which
 * synchronises the device) is not allowed, or a plugin without access to an
 * allocator.  Same arguments, results and checks as spec_verify_greedy, minus
 * ws / ws_bytes.  Its scratch is a fixed 256 KiB array of device memory inside
 * the library (held on every GPU that loads the library until the process
 * exits); requests whose scratch (spec_verify_workspace_bytes(B, R, V)) exceeds
 * it return SPEC_ERR_CAPACITY without launching; the scratch a request needs is
 * spec_verify_greedy_static_bytes(B, R, V) (256-byte header, B completion
 * counters, 8 bytes per chunk record: about B*R*ceil(640/(B*R))*8 bytes for
 * large vocabularies) and the array's size is
 * spec_verify_greedy_static_capacity().  The first call on a device looks up
 * the array's device address with that device current and keeps it (it does
 * not survive a cudaDeviceReset of that device); make that first call before
 * any stream capture.  All calls share the one array, so calls that overlap on
 * the GPU (different streams, no ordering) race; calls ordered on one stream
 * are safe.  Each call clears the array's error header and counters;
 * spec_verify_greedy_static_error reads the error word the last call left
 * (device-side index errors, as in the workspace version).  It allocates
 * nothing. */
spec_status spec_verify_greedy_static(int32_t B, int32_t R, int32_t V, const float *target_logits,
                                      const int32_t *draft_tok, const int32_t *parent,
                                      int32_t max_depth, int32_t *out_tok, int32_t *accept_len,
                                      int32_t *kv_src, const spec_model_desc *desc,
                                      const spec_kv *kv, const int32_t *ctx_len, spec_stream_t stream);

/* Size in bytes of spec_verify_greedy_static's fixed scratch array, and the
 * scratch one call over B requests of R rows of V logits needs (the paper has
 * no counterpart; see spec_verify_greedy_static). */
size_t spec_verify_greedy_static_capacity(void);
size_t spec_verify_greedy_static_bytes(int32_t B, int32_t R, int32_t V);

/* The error word spec_verify_greedy_static's last call on the current device
 * left in its fixed scratch array (0 = none, else a spec_status code), read
 * after synchronising ``stream`` (the paper has no counterpart). */
spec_status spec_verify_greedy_static_error(int32_t *code_out, spec_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* EAGLESPEC_H */
