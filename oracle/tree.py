"""Top-k draft-tree expansion ranked by cumulative log-probability.

Sources: [EAGLET] "Eaglet", section "Approach 1: YAML Recipe" and
"EagletV2Config Reference" (``draft_top_k``, ``draft_depth``,
``total_draft_tokens``; the draft model proposes candidate tokens in a tree and
the target verifies the tree in one forward pass, page introduction).

The pages give only the three parameters.  The reading used (EAGLE-2 style;
the pages fix none of the following):

* the root is the last accepted token (node 0, depth 0, score 0);
* depth 1: the root's top ``k`` tokens become nodes with score = log-prob;
  they form the frontier;
* depth d >= 2: every frontier node contributes its top ``k`` tokens, scored
  parent score + log-prob, all k*k of them join the candidate pool, and the
  best ``k`` of them (score, then creation order) form the next frontier;
* after depth ``draft_depth`` the best ``total_draft_tokens`` nodes of the
  pool (score, then creation order, which is depth-major) are the tree; since
  log-probs are <= 0 a parent always ranks before its children, so the
  selection contains every selected node's ancestors;
* final numbering: node 0 = root, then the selected nodes by (depth, score,
  creation order), so a parent's index is smaller than its children's;
* score arithmetic is float32 (the precision of the log-probs the LM head
  emits and of the kernel), so both sides take identical decisions on
  identical inputs.

Draft-pass bookkeeping for the frontier (a stated reading): frontier slot f
at depth d writes its K/V at draft-region index 1 + (d-1)*k + f, attends to its
ancestors' draft-region entries (bit mask) and itself, sits at position
ctx + d, and takes as hidden input the pre-norm state of the row that produced
it (its parent's row in the previous pass).
"""
import numpy as np


def tree_init(B, top_k, depth, total, root_tok, ctx_len):
    P = top_k + (depth - 1) * top_k * top_k
    if not (1 <= total <= P and total + 1 <= 64 and 1 + (depth - 1) * top_k <= 64):
        raise ValueError("tree does not fit: total=%d pool=%d" % (total, P))
    return {
        "B": B, "k": top_k, "D": depth, "N": total, "P": P,
        "root_tok": np.asarray(root_tok, dtype=np.int64).copy(),
        "ctx_len": np.asarray(ctx_len, dtype=np.int64).copy(),
        "count": np.zeros(B, dtype=np.int64),
        "tok": np.zeros((B, P), dtype=np.int64),
        "parent": np.full((B, P), -1, dtype=np.int64),
        "depth": np.zeros((B, P), dtype=np.int64),
        "score": np.zeros((B, P), dtype=np.float32),
        "mask": [[0] * P for _ in range(B)],
        "frontier": np.zeros((B, top_k), dtype=np.int64),
    }


def _rank(scores, idx):
    """Order of candidates: larger score first, then smaller creation index."""
    return np.lexsort((idx, -np.asarray(scores, dtype=np.float32)))


def tree_expand(st, d, ids, logprob):
    """Consume the top-k of the pass that produced depth-d nodes.

    ids, logprob: [B, k] for d == 1 (root rows) or [B*k, k] for d >= 2
    (frontier rows, request b's rows at b*k .. b*k + k - 1).
    Returns the next pass's rows (dict) for d < D, or the final tree for d == D.
    """
    B, k, D = st["B"], st["k"], st["D"]
    ids = np.asarray(ids, dtype=np.int64)
    lp = np.asarray(logprob, dtype=np.float32)
    for b in range(B):
        c0 = int(st["count"][b])
        new = []
        if d == 1:
            for j in range(k):
                new.append((ids[b, j], -1, np.float32(0.0) + lp[b, j], b))
        else:
            for f in range(k):
                par = int(st["frontier"][b, f])
                row = b * k + f
                for j in range(k):
                    sc = np.float32(st["score"][b, par]) + lp[row, j]
                    new.append((ids[row, j], par, np.float32(sc), row))
        for t, (tk, par, sc, _) in enumerate(new):
            p = c0 + t
            st["tok"][b, p] = tk
            st["parent"][b, p] = par
            st["depth"][b, p] = d
            st["score"][b, p] = sc
        st["count"][b] = c0 + len(new)
        cand = np.arange(c0, c0 + len(new))
        order = _rank(st["score"][b, cand], cand)
        st["frontier"][b] = cand[order[:k]]
        # source rows of the new frontier (row in the pass that produced them)
        st.setdefault("src_row", np.zeros((B, k), dtype=np.int64))
        for f in range(k):
            st["src_row"][b, f] = new[int(order[f])][3]
    if d < D:
        return _frontier_rows(st, d)
    return tree_finalize(st)


def _frontier_rows(st, d):
    B, k = st["B"], st["k"]
    M = B * k
    tok = np.zeros(M, dtype=np.int64)
    pos = np.zeros(M, dtype=np.int64)
    kv_idx = np.zeros(M, dtype=np.int64)
    mask = [0] * M
    hid_src = np.zeros(M, dtype=np.int64)
    for b in range(B):
        for f in range(k):
            node = int(st["frontier"][b, f])
            par = int(st["parent"][b, node])
            pmask = 1 if par < 0 else st["mask"][b][par]
            idx = 1 + (d - 1) * k + f
            st["mask"][b][node] = pmask | (1 << idx)
            m = b * k + f
            tok[m] = st["tok"][b, node]
            pos[m] = st["ctx_len"][b] + d
            kv_idx[m] = idx
            mask[m] = st["mask"][b][node]
            hid_src[m] = st["src_row"][b, f]
    return {"M": M, "B": B, "R": k, "step": 0, "ctx_len": st["ctx_len"].copy(),
            "tok": tok, "pos": pos, "kv_idx": kv_idx, "mask": mask, "hid_src": hid_src}


def tree_finalize(st):
    """Select the tree and number its nodes.  Returns per request arrays of N+1
    entries: tok, parent (-1 for the root), depth, pos, score, mask (python ints)."""
    B, N = st["B"], st["N"]
    out = {k: np.zeros((B, N + 1), dtype=np.int64) for k in ("tok", "parent", "depth", "pos")}
    out["score"] = np.zeros((B, N + 1), dtype=np.float32)
    out["mask"] = [[0] * (N + 1) for _ in range(B)]
    for b in range(B):
        cnt = int(st["count"][b])
        cand = np.arange(cnt)
        sel = cand[_rank(st["score"][b, :cnt], cand)[:N]]
        # depth, then score, then creation
        sel = sel[np.lexsort((sel, -st["score"][b, sel], st["depth"][b, sel]))]
        final = {-1: 0}
        for n, p in enumerate(sel, start=1):
            final[int(p)] = n
        out["tok"][b, 0] = st["root_tok"][b]
        out["parent"][b, 0] = -1
        out["pos"][b, 0] = st["ctx_len"][b]
        out["mask"][b][0] = 1
        for n, p in enumerate(sel, start=1):
            par = int(st["parent"][b, p])
            if par not in final:
                raise AssertionError("selection not closed under ancestors")
            pf = final[par]
            out["tok"][b, n] = st["tok"][b, p]
            out["parent"][b, n] = pf if par >= 0 else 0
            out["depth"][b, n] = st["depth"][b, p]
            out["pos"][b, n] = st["ctx_len"][b] + st["depth"][b, p]
            out["score"][b, n] = st["score"][b, p]
            out["mask"][b][n] = out["mask"][b][out["parent"][b, n]] | (1 << n)
    return out
