"""Verification of drafts against target logits, float64 / exact integers.

[NEURON] "Speculative Decoding (EAGLE3) in the vLLM Neuron Framework":
* section "What is Speculative Decoding?": tokens are accepted in order until
  the first mismatch; the corrected token at the mismatch (or a bonus token when
  all drafts are accepted) is emitted; greedy output is bit-exact with the
  target alone;
* section "Rejection Sampling", on-device sampler: match mask
  ``drafts == argmax(target)``, first mismatch, accept up to and including the
  mismatch position (emitting the target's token there), bonus if all match;
  output ``[batch, max_spec_len + 1]`` with -1 at rejected positions;
* section "Rejection Sampling", CPU sampler (arXiv:2211.17192): accept when
  ``uniform <= target_prob(draft) / draft_prob`` with draft_prob = 1 (greedy
  draft); a rejected position emits a recovered token by the Gumbel-max trick,
  ``argmax(adjusted_prob / exponential_noise)`` with
  ``adjusted_prob = max(target_prob - draft_prob, 0)``, i.e. the target
  distribution with the draft token removed; the bonus token is sampled from
  the target distribution at the last position.

Tree verification ([EAGLET] introduction: the target verifies the whole tree in
one forward pass) reads: node c is accepted when its parent is accepted and its
token equals the target's argmax at the parent; the root is always accepted;
the emitted sequence is the deepest accepted node's root path (ties at equal
depth: smallest node index) followed by the target's argmax at that node.
The accepted path's K/V then moves to contiguous cache indices ctx + depth.

Argmax ties go to the smallest token id.  Temperature <= 0 means greedy for that
request.  Exponential noise E = -ln(u) for u from ``philox``; the sample
argmax_x p(x)/E_x equals argmax_x (logit_x / T - ln(-ln u_x)).
"""
import numpy as np

from . import philox
from .numerics import logsumexp
from .draft import slot_of


def argmax_first(x):
    """Index of the largest entry of each row, smallest index among ties."""
    return np.argmax(np.asarray(x), axis=-1)


def verify_greedy_chain(target, drafts):
    """target [B, K+1, V] float32, drafts [B, K].  Returns out [B, K+1], accept_len [B],
    kv_src [B, K+1] (draft-region index kept at each output position, -1 after)."""
    target = np.asarray(target)
    drafts = np.asarray(drafts, dtype=np.int64)
    B, K1, _ = target.shape
    K = K1 - 1
    t = argmax_first(target)
    out = np.full((B, K + 1), -1, dtype=np.int64)
    kv_src = np.full((B, K + 1), -1, dtype=np.int64)
    acc = np.zeros(B, dtype=np.int64)
    for b in range(B):
        a = 0
        while a < K and drafts[b, a] == t[b, a]:
            a += 1
        out[b, :a] = drafts[b, :a]
        out[b, a] = t[b, a]
        kv_src[b, :a + 1] = np.arange(a + 1)
        acc[b] = a
    return out, acc, kv_src


def verify_greedy_tree(target, tree_tok, tree_parent, max_depth):
    """target [B, N+1, V] (row n = target logits at tree node n), tree_tok /
    tree_parent [B, N+1] (parent[0] = -1, parent[n] < n).  Returns out
    [B, max_depth+1], accept_len [B], kv_src [B, max_depth+1] (node index on the
    accepted path at each depth, -1 after)."""
    target = np.asarray(target)
    tok = np.asarray(tree_tok, dtype=np.int64)
    par = np.asarray(tree_parent, dtype=np.int64)
    B, N1, _ = target.shape
    t = argmax_first(target)
    out = np.full((B, max_depth + 1), -1, dtype=np.int64)
    kv_src = np.full((B, max_depth + 1), -1, dtype=np.int64)
    acc = np.zeros(B, dtype=np.int64)
    for b in range(B):
        accepted = np.zeros(N1, dtype=bool)
        depth = np.zeros(N1, dtype=np.int64)
        accepted[0] = True
        best = 0
        for n in range(1, N1):
            p = par[b, n]
            if not (0 <= p < n):
                raise ValueError("parent index must precede the node")
            depth[n] = depth[p] + 1
            accepted[n] = accepted[p] and tok[b, n] == t[b, p]
            if accepted[n] and depth[n] > depth[best]:
                best = n
        path = []
        n = best
        while n != 0:
            path.append(n)
            n = par[b, n]
        path = path[::-1]
        a = len(path)
        for i, n in enumerate(path):
            out[b, i] = tok[b, n]
            kv_src[b, i + 1] = n
        kv_src[b, 0] = 0
        out[b, a] = t[b, best]
        acc[b] = a
    return out, acc, kv_src


def compact_kv(kv, ctx_len, kv_src, accept_len):
    """Move the accepted draft-region entries to contiguous cache indices: the entry
    at ctx + kv_src[b, d] goes to ctx + d for d = 1 .. accept_len[b]
    (increasing d; no source is overwritten before it is read because
    kv_src[b, d] >= d and the sources increase).  Modifies ``kv`` in place."""
    for b in range(len(accept_len)):
        ctx = int(ctx_len[b])
        for d in range(1, int(accept_len[b]) + 1):
            s = int(slot_of(kv, b, ctx + int(kv_src[b, d])))
            t = int(slot_of(kv, b, ctx + d))
            kv["k"][t] = kv["k"][s]
            kv["v"][t] = kv["v"][s]


def kept_set(l, top_k=0, top_p=1.0):
    """Tokens kept by top-k then top-p filtering of the logits ``l`` (already divided
    by the temperature).  [NEURON] "Rejection Sampling": the CPU sampler supports
    per-request top-k and top-p.  Reading (the page gives only the names): order
    tokens by logit, larger first, ties to the smaller id; top-k keeps the first k;
    top-p then keeps the shortest prefix of those whose renormalised probability
    mass reaches top_p.  Returns (boolean mask, top-p margin), the margin being the
    distance of the deciding cumulative mass from top_p (for near-tie accounting).
    """
    l = np.asarray(l, dtype=np.float64)
    V = l.shape[0]
    order = np.lexsort((np.arange(V), -l))
    n = V
    if top_k and 0 < int(top_k) < V:
        n = int(top_k)
    keep = order[:n]
    margin = np.inf
    if top_p is not None and float(top_p) < 1.0:
        p = np.exp(l[keep] - logsumexp(l[keep]))
        c = np.cumsum(p)
        m = int(np.searchsorted(c, float(top_p))) + 1
        m = min(m, n)
        margin = min(abs(c[m - 1] - top_p), abs(c[m - 2] - top_p) if m >= 2 else np.inf)
        keep = keep[:m]
    mask = np.zeros(V, dtype=bool)
    mask[keep] = True
    return mask, margin


def verify_rejection(target, drafts, temperature, seed, step_offset=0, top_k=None, top_p=None, req_ids=None):
    """Probabilistic verification of a greedy-drafted chain.

    target [B, K+1, V] float32, drafts [B, K], temperature [B]; optional per
    request top_k [B] (0 = off) and top_p [B] (1.0 = off) restrict the target
    distribution (see ``kept_set``) before the accept test, the recovered
    sample and the bonus sample.  ``req_ids`` [B] are the requests' indices in the
    batch (the Philox counter's request word; default 0..B-1), for checking a
    sample of a larger batch.  Returns (out [B, K+1], accept_len [B], info)
    where info holds per (b, i) the acceptance margin u - p(draft), for the
    emitted sampled token the gap between the best and second-best Gumbel keys,
    and the smallest top-p margin met (for near-tie accounting).
    """
    target = np.asarray(target, dtype=np.float64)
    drafts = np.asarray(drafts, dtype=np.int64)
    B, K1, V = target.shape
    K = K1 - 1
    out = np.full((B, K + 1), -1, dtype=np.int64)
    acc = np.zeros(B, dtype=np.int64)
    margins = np.full((B, K), np.inf)
    gaps = np.full(B, np.inf)
    p_margins = np.full(B, np.inf)
    tk = np.zeros(B, dtype=np.int64) if top_k is None else np.asarray(top_k, dtype=np.int64)
    tp = np.ones(B) if top_p is None else np.asarray(top_p, dtype=np.float64)
    rid = np.arange(B) if req_ids is None else np.asarray(req_ids, dtype=np.int64)
    for b in range(B):
        T = float(temperature[b])
        a = 0
        emitted = None
        while a < K:
            row = target[b, a]
            d = int(drafts[b, a])
            if T <= 0.0:
                tgt = int(argmax_first(row.astype(np.float32)))
                if d == tgt:
                    out[b, a] = d
                    a += 1
                    continue
                emitted = tgt
                break
            l = row / T
            kept, pm = kept_set(l, tk[b], tp[b])
            p_margins[b] = min(p_margins[b], pm)
            p_d = np.exp(l[d] - logsumexp(l[kept])) if kept[d] else 0.0
            u = philox.accept_uniform(seed, step_offset, int(rid[b]), a)
            margins[b, a] = u - p_d
            if u <= p_d:
                out[b, a] = d
                a += 1
                continue
            key = l - np.log(-np.log(philox.noise_uniforms(seed, step_offset, int(rid[b]), a, V)))
            key[~kept] = -np.inf
            key[d] = -np.inf
            emitted, gaps[b] = _best(key)
            break
        if emitted is None:
            row = target[b, K]
            if T <= 0.0:
                emitted = int(argmax_first(row.astype(np.float32)))
            else:
                l = row / T
                kept, pm = kept_set(l, tk[b], tp[b])
                p_margins[b] = min(p_margins[b], pm)
                key = l - np.log(-np.log(philox.noise_uniforms(seed, step_offset, int(rid[b]), K, V)))
                key[~kept] = -np.inf
                emitted, gaps[b] = _best(key)
        out[b, a] = emitted
        acc[b] = a
    return out, acc, {"accept_margin": margins, "sample_gap": gaps, "top_p_margin": p_margins}


def _best(key):
    i = int(np.argmax(key))
    rest = np.delete(key, i)
    gap = key[i] - (rest.max() if rest.size else -np.inf)
    return i, gap
