"""Draft step of EAGLE-3 / EAGLE-4, float64.

Sources:
* [NEURON] "Speculative Decoding (EAGLE3) in the vLLM Neuron Framework":
  section "What is EAGLE3?" (FC over three auxiliary hidden states, single
  decoder layer, embedding, LM head); section "Eagle3 Draft Model Architecture"
  (the decoder-layer pseudo-code: input_layernorm on the embeddings, hidden_norm
  on the target hidden state, concatenation [embeds, hidden] of width 2H, QKV
  sized for 2H input, residual add, post_attention_layernorm + MLP + residual,
  final norm, returns (hidden_states, hidden_prenorm)); section "EagleProposer:
  Draft Model Management" (positions + 1 per recurrent step, slot mapping
  ``block_table[pos // block_size] * block_size + pos % block_size``); section
  "Design Choices" (greedy draft sampling).
* [EAGLE4] "nemo_automodel ... eagle4": ``Eagle4Config.sliding_window`` (keys a
  draft query attends to, itself and its chain included); module docstring
  (low-rank candidate head whose retrieved candidates are rescored exactly with
  the full lm_head); ``Eagle4CandidateHeadConfig`` (rank, num_candidates).

Readings where the pages are silent (the plainest choice each time):
* residual of the attention block = the H-wide hidden input of the layer;
* RMSNorm / RoPE / SwiGLU in their Llama forms (see ``numerics``);
* attention scale 1/sqrt(head_dim); q head h uses kv head h // (nq / nkv);
* a row attends to context cache entries [0, ctx) (with a window W > 0: only
  positions > pos - W) plus the entries of the draft region selected by its
  mask (bit i = cache index ctx + i); the row's own entry is written before any
  row of the pass attends;
* storage precision: in bf16 workloads the values the GPU stores in bf16 are
  rounded to bf16 here too (h0, the normalised embedding/hidden halves, q/k/v,
  attention output, post-attention-norm output, MLP activation, hidden_prenorm,
  the normalised output, the low-rank projection z); the residual stream r1/r2
  stays unrounded;
* argmax / top-k decisions are taken on the logits rounded to float32 (the
  kernel's precision), larger value first, ties to the smaller token id.
"""
import numpy as np

from .numerics import to_bf16, rmsnorm, rope, silu, logsumexp, topk_desc


def _r(x, dtype):
    return to_bf16(x) if dtype == "bf16" else np.asarray(x, dtype=np.float64)


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def slot_of(kv, b, cache_idx):
    """Paged slot of logical cache index ``cache_idx`` of request ``b``
    ([NEURON] "EagleProposer", recurrent phase; "KV Cache Sharing")."""
    bs = kv["block_size"]
    cache_idx = np.asarray(cache_idx, dtype=np.int64)
    return kv["block_table"][b, cache_idx // bs].astype(np.int64) * bs + cache_idx % bs


def fc_fuse(desc, W, aux):
    """h0 = fc(cat(aux_low, aux_mid, aux_high)); fc is Linear(3H -> H)
    ([NEURON] "Eagle3 Draft Model Architecture", Eagle3LlamaModel.fc and the
    initial forward mode's combine_hidden_states).

    EAGLE-3.1 ``fc_norm`` ([QUARK] "Background: EAGLE-3 and EAGLE-3.1": extra
    normalisation inside the draft head; Quickstart's eagle_architecture_config
    names the flag).  Reading: an RMSNorm with its own gain ``W["fc_norm"]`` on
    the fused feature, before it enters the decoder layer.
    """
    h0 = _f64(aux) @ _f64(W["fc"]).T
    if getattr(desc, "fc_norm", False):
        h0 = rmsnorm(h0, W["fc_norm"], desc.rms_eps)
    return _r(h0, desc.dtype)


def recurrent_state(desc, prenorm, hn):
    """The hidden state a draft pass hands to the next one: hidden_prenorm
    ([NEURON] "Eagle3 Draft Model Architecture": the recurrent input is the
    pre-norm state); with the EAGLE-3.1 ``norm_output`` flag ([QUARK] "Background:
    EAGLE-3 and EAGLE-3.1", Quickstart) the reading is that the draft's output
    state is the normalised one, so the next pass takes hn."""
    return hn if getattr(desc, "norm_output", False) else prenorm


def expand_rows(rows):
    """Fill the per-row arrays a chain step leaves implicit.

    rows: dict with M, B, R (rows per request), step, ctx_len[B], tok[M] and
    optionally pos[M], kv_idx[M], mask[M] (python ints), hid_src[M].
    Chain defaults for step s: pos = ctx + s, kv_idx = s, mask = bits 0..s.
    """
    M, R, s = rows["M"], rows["R"], rows.get("step", 0)
    req = np.arange(M) // R
    ctx = np.asarray(rows["ctx_len"], dtype=np.int64)[req]
    pos = rows.get("pos")
    pos = ctx + s if pos is None else np.asarray(pos, dtype=np.int64)
    kv_idx = rows.get("kv_idx")
    kv_idx = np.full(M, s, dtype=np.int64) if kv_idx is None else np.asarray(kv_idx, dtype=np.int64)
    mask = rows.get("mask")
    mask = [(1 << (s + 1)) - 1] * M if mask is None else [int(x) for x in mask]
    hid_src = rows.get("hid_src")
    hid_src = np.arange(M) if hid_src is None else np.asarray(hid_src, dtype=np.int64)
    return req, ctx, pos, kv_idx, mask, hid_src


def attention(desc, q, kv, req, ctx, pos, mask):
    """Softmax attention of each row's query heads over its allowed keys, by brute force.

    q: [M, nq, hd] (post-RoPE).  Allowed keys of row m: context cache indices
    j in [lo, ctx) with lo = max(0, pos - W + 1) when W > 0 else 0, plus cache
    index ctx + i for every bit i of mask[m].  Returns [M, nq, hd].
    """
    M = q.shape[0]
    nq, nkv, hd = desc.nq, desc.nkv, desc.hd
    group = nq // nkv
    out = np.zeros((M, nq, hd), dtype=np.float64)
    for m in range(M):
        b = int(req[m])
        lo = max(0, int(pos[m]) - desc.window + 1) if desc.window > 0 else 0
        idx = list(range(lo, int(ctx[m])))
        mk = mask[m]
        i = 0
        while mk:
            if mk & 1:
                idx.append(int(ctx[m]) + i)
            mk >>= 1
            i += 1
        slots = slot_of(kv, b, np.array(idx, dtype=np.int64))
        Kr = _f64(kv["k"][slots])       # [n, nkv, hd]
        Vr = _f64(kv["v"][slots])
        for h in range(nq):
            g = h // group
            s = Kr[:, g, :] @ q[m, h] / np.sqrt(hd)
            p = np.exp(s - s.max())
            p /= p.sum()
            out[m, h] = p @ Vr[:, g, :]
    return out


def draft_layer(desc, W, rows, hid_in, kv):
    """One pass of the single EAGLE-3 draft decoder layer over ``rows``.

    [NEURON] "Eagle3 Draft Model Architecture" (Eagle3LlamaDecoderLayer and
    Eagle3LlamaModel): embeds = input_layernorm(embed(tok)); hidden =
    hidden_norm(target hidden); x = cat([embeds, hidden]) (2H); attention with
    QKV sized for 2H input and output H; out = residual + out;
    out = mlp(post_attention_layernorm(out)) + out; returns the pre-norm state
    (the recurrent input of the next pass) and the final-normed state (to the
    LM head).  K/V of every row are written to the paged cache at cache index
    ctx + kv_idx before attention.  Modifies ``kv`` in place.

    Returns (hidden_prenorm [M, H], hidden_normed [M, H]).
    """
    dt = desc.dtype
    H, nq, nkv, hd = desc.H, desc.nq, desc.nkv, desc.hd
    M = rows["M"]
    req, ctx, pos, kv_idx, mask, hid_src = expand_rows(rows)
    tok = np.asarray(rows["tok"], dtype=np.int64)
    hid = _f64(hid_in)[hid_src]

    e = _r(rmsnorm(_f64(W["embed"])[tok], W["in_norm"], desc.rms_eps), dt)
    g = _r(rmsnorm(hid, W["hidden_norm"], desc.rms_eps), dt)
    x = np.concatenate([e, g], axis=-1)                       # [M, 2H], embeds first

    q = (x @ _f64(W["wq"]).T).reshape(M, nq, hd)
    k = (x @ _f64(W["wk"]).T).reshape(M, nkv, hd)
    v = (x @ _f64(W["wv"]).T).reshape(M, nkv, hd)
    q = _r(rope(q, pos[:, None], desc.rope_theta), dt)
    k = _r(rope(k, pos[:, None], desc.rope_theta), dt)
    v = _r(v, dt)

    for m in range(M):
        s = int(slot_of(kv, int(req[m]), int(ctx[m] + kv_idx[m])))
        kv["k"][s] = k[m]
        kv["v"][s] = v[m]

    a = _r(attention(desc, q, kv, req, ctx, pos, mask).reshape(M, nq * hd), dt)
    r1 = hid + a @ _f64(W["wo"]).T
    n = _r(rmsnorm(r1, W["post_norm"], desc.rms_eps), dt)
    act = _r(silu(n @ _f64(W["wgate"]).T) * (n @ _f64(W["wup"]).T), dt)
    r2 = r1 + act @ _f64(W["wdown"]).T
    prenorm = _r(r2, dt)
    hn = _r(rmsnorm(r2, W["final_norm"], desc.rms_eps), dt)
    return prenorm, hn


def lm_head(desc, W, hn, k):
    """LM head with per-row top-k and log-softmax statistics.

    logits = hn @ lm_head^T ([NEURON] "Eagle3 Draft Model Architecture", LM head;
    greedy draft sampling in "Design Choices" is top-1).  lse = log sum exp of
    the row; log-prob of a token = logit - lse.  Returns (ids [M,k] int64,
    logprob [M,k], lse [M], logits [M,V]).
    """
    logits = _f64(hn) @ _f64(W["lm_head"]).T
    lse = logsumexp(logits, axis=-1)
    ids = topk_desc(logits.astype(np.float32), k)
    lp = np.take_along_axis(logits, ids, axis=-1) - lse[:, None]
    if getattr(desc, "draft_vocab", 0) > 0:
        # reduced draft vocabulary: rows of lm_head are draft entries, emitted ids are
        # the mapped target ids ([QUARK] calibrate_draft_vocab / d2t; [EAGLE4]
        # selected_token_ids); logits stay indexed by draft entry
        ids = np.asarray(W["d2t"], dtype=np.int64)[ids]
    return ids, lp, lse, logits


def lowrank_candidates(desc, W, hn, num_candidates, k_out, with_logprob=False):
    """EAGLE-4 candidate head: low-rank scores retrieve candidates, the full
    lm_head rescores them exactly ([EAGLE4] module docstring and
    Eagle4CandidateHeadConfig: s = (hn @ down^T) @ up^T with down [r, H] and
    up [V, r]; keep the top num_candidates by s; exact logits of those from
    lm_head rows; the draft token is the best exact logit among candidates).

    Returns (cand_ids [M,Kc] in score order, cand_logits [M,Kc] exact,
    out_ids [M,k_out]).
    """
    dt = desc.dtype
    z = _r(_f64(hn) @ _f64(W["lr_down"]).T, dt)               # [M, r]
    s = z @ _f64(W["lr_up"]).T                                  # [M, V]
    cand = topk_desc(s.astype(np.float32), num_candidates)      # [M, Kc]
    Wl = _f64(W["lm_head"])
    M = hn.shape[0]
    exact = np.empty(cand.shape, dtype=np.float64)
    for m in range(M):
        exact[m] = Wl[cand[m]] @ _f64(hn[m])
    out = np.empty((M, k_out), dtype=np.int64)
    out_lp = np.empty((M, k_out), dtype=np.float64)
    for m in range(M):
        order = np.lexsort((cand[m], -exact[m].astype(np.float32)))
        out[m] = cand[m][order[:k_out]]
        # log-probs under the softmax over the candidates (tree drafting from the
        # candidate head ranks children with these)
        out_lp[m] = exact[m][order[:k_out]] - logsumexp(exact[m])
    if with_logprob:
        return cand, exact, out, out_lp
    return cand, exact, out
