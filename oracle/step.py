"""Whole speculative step on the oracle: draft (chain or tree), then verify.

[NEURON] "Speculative Decoding (EAGLE3) in the vLLM Neuron Framework",
section "EagleProposer: Draft Model Management", ``propose()``: an initial pass
on the FC-fused auxiliary hidden states gives the first draft token and a
recurrent state; K-1 recurrent passes follow, each on the previous draft token
and the previous pass's pre-norm state, positions advancing by one, tokens by
greedy argmax.  Tree drafting follows ``oracle.tree``.

Target logits for the synthetic workloads are the draft's own logits plus
Gaussian noise (chain: K+1 draft passes, the last one only for the bonus row;
tree: one extra draft pass over the root and all tree nodes with the tree mask,
every node taking the root's FC feature as hidden input).  That pass also writes
the tree's K/V at cache index ctx + node, which tree verification compacts.
"""
import copy

import numpy as np

from . import draft, tree, verify


def chain_draft(desc, W, aux, root_tok, ctx_len, kv, K, keep_logits=False, trace=None):
    """Returns drafts [B, K] and, with keep_logits, the per-pass logits [B, K, V].
    ``trace``, if a list, receives each pass's normalised output hn [B, H]."""
    B = len(root_tok)
    hid = draft.fc_fuse(desc, W, aux)
    tok = np.asarray(root_tok, dtype=np.int64)
    drafts = np.zeros((B, K), dtype=np.int64)
    logits = [] if keep_logits else None
    for i in range(K):
        rows = {"M": B, "B": B, "R": 1, "step": i, "ctx_len": ctx_len, "tok": tok}
        prenorm, hn = draft.draft_layer(desc, W, rows, hid, kv)
        hid = draft.recurrent_state(desc, prenorm, hn)
        if trace is not None:
            trace.append(hn)
        if desc.rank > 0:
            _, _, ids = draft.lowrank_candidates(desc, W, hn, desc.num_candidates, 1)
            lg = None
            if keep_logits:
                lg = hn @ np.asarray(W["lm_head"], dtype=np.float64).T
        else:
            ids, _, _, lg = draft.lm_head(desc, W, hn, 1)
        drafts[:, i] = ids[:, 0]
        tok = ids[:, 0]
        if keep_logits:
            logits.append(lg)
    if keep_logits:
        return drafts, np.stack(logits, axis=1)
    return drafts


def chain_target(desc, W, aux, root_tok, ctx_len, kv, K, noise):
    """Target logits [B, K+1, V] = draft logits of K+1 chained passes + noise (float32)."""
    kvc = copy.deepcopy(kv)
    _, lg = chain_draft(desc, W, aux, root_tok, ctx_len, kvc, K + 1, keep_logits=True)
    return (lg + noise).astype(np.float32)


def tree_draft(desc, W, aux, root_tok, ctx_len, kv, top_k, depth, total, trace=None):
    """Returns the final tree (see ``tree.tree_finalize``).  ``trace``, if a list,
    receives (rows, hid_in, ids, logprob) per pass."""
    B = len(root_tok)
    h0 = draft.fc_fuse(desc, W, aux)
    rows = {"M": B, "B": B, "R": 1, "step": 0, "ctx_len": ctx_len,
            "tok": np.asarray(root_tok, dtype=np.int64)}
    st = tree.tree_init(B, top_k, depth, total, root_tok, ctx_len)
    hid_in = h0
    for d in range(1, depth + 1):
        prenorm, hn = draft.draft_layer(desc, W, rows, hid_in, kv)
        if desc.rank > 0:
            # EAGLE-4 candidate head drafting a tree: top-k of the rescored candidates,
            # log-probs under the softmax over the candidates
            _, _, ids, lp = draft.lowrank_candidates(desc, W, hn, desc.num_candidates, top_k, with_logprob=True)
        else:
            ids, lp, _, _ = draft.lm_head(desc, W, hn, top_k)
        if trace is not None:
            trace.append((rows, hid_in, ids, lp))
        res = tree.tree_expand(st, d, ids, lp)
        if d < depth:
            rows, hid_in = res, draft.recurrent_state(desc, prenorm, hn)
        else:
            return res


def tree_target(desc, W, aux, ctx_len, kv, final, noise):
    """One draft pass over the root and every tree node with the tree mask (writes
    their K/V at ctx + node) -> target logits [B, N+1, V] = logits + noise."""
    B, N1 = final["tok"].shape
    h0 = draft.fc_fuse(desc, W, aux)
    rows = {"M": B * N1, "B": B, "R": N1, "step": 0, "ctx_len": ctx_len,
            "tok": final["tok"].reshape(-1),
            "pos": final["pos"].reshape(-1),
            "kv_idx": np.tile(np.arange(N1), B),
            "mask": [m for b in range(B) for m in final["mask"][b]],
            "hid_src": np.repeat(np.arange(B), N1)}
    _, hn = draft.draft_layer(desc, W, rows, h0, kv)
    lg = np.asarray(hn, dtype=np.float64) @ np.asarray(W["lm_head"], dtype=np.float64).T
    return (lg.reshape(B, N1, -1) + noise).astype(np.float32)


def chain_step(desc, W, aux, root_tok, ctx_len, kv, K, target, temperature=None,
               seed=0, step_offset=0):
    """Draft K tokens then verify them; returns (drafts, out, accept_len)."""
    drafts = chain_draft(desc, W, aux, root_tok, ctx_len, kv, K)
    if desc.verify == "rejection":
        out, acc, _ = verify.verify_rejection(target, drafts, temperature, seed, step_offset)
    else:
        out, acc, _ = verify.verify_greedy_chain(target, drafts)
    return drafts, out, acc


def prefill_inputs(input_ids, next_token, last_idx, ctx_len):
    """Rows of the batched initial draft pass ([NEURON] "EagleProposer", prefill
    phase: ids shifted by one, the new token scattered at the last accepted row;
    row j of request b at position ctx + j, draft-region entry j, causal mask)."""
    ids = np.asarray(input_ids, dtype=np.int64)
    B, R = ids.shape
    tok = np.zeros((B, R), dtype=np.int64)
    tok[:, :R - 1] = ids[:, 1:]
    for b in range(B):
        tok[b, int(last_idx[b])] = next_token[b]
    ctx = np.asarray(ctx_len, dtype=np.int64)
    pos = (ctx[:, None] + np.arange(R)[None, :]).reshape(-1)
    kv_idx = np.tile(np.arange(R), B)
    mask = [(1 << (j + 1)) - 1 for b in range(B) for j in range(R)]
    last_row = np.arange(B) * R + np.asarray(last_idx, dtype=np.int64)
    return {"M": B * R, "B": B, "R": R, "step": 0, "ctx_len": ctx, "tok": tok.reshape(-1), "pos": pos,
            "kv_idx": kv_idx, "mask": mask}, last_row


def prefill_chain_draft(desc, W, aux_rows, input_ids, next_token, last_idx, ctx_len, kv, K, keep_logits=False):
    """propose() with the prefill phase: FC over every verified token's aux
    states, one draft pass over all of them, the first draft token from each
    request's last accepted row, then K-1 recurrent passes starting after the
    accepted tokens (context ctx + last_idx + 1).  Returns drafts [B, K]."""
    rows, last_row = prefill_inputs(input_ids, next_token, last_idx, ctx_len)
    h0 = draft.fc_fuse(desc, W, aux_rows)
    pre, hn = draft.draft_layer(desc, W, rows, h0, kv)
    ids, _, _, lg = draft.lm_head(desc, W, hn[last_row], 1)
    B = len(next_token)
    drafts = np.zeros((B, K), dtype=np.int64)
    drafts[:, 0] = ids[:, 0]
    logits = [lg]
    hid = draft.recurrent_state(desc, pre, hn)[last_row]
    ctx2 = np.asarray(ctx_len, dtype=np.int64) + np.asarray(last_idx, dtype=np.int64) + 1
    tok = ids[:, 0]
    for i in range(1, K):
        r = {"M": B, "B": B, "R": 1, "step": i - 1, "ctx_len": ctx2, "tok": tok}
        pre_i, hn = draft.draft_layer(desc, W, r, hid, kv)
        hid = draft.recurrent_state(desc, pre_i, hn)
        ids, _, _, lg = draft.lm_head(desc, W, hn, 1)
        drafts[:, i] = ids[:, 0]
        tok = ids[:, 0]
        logits.append(lg)
    if keep_logits:
        return drafts, np.stack(logits, axis=1)
    return drafts
