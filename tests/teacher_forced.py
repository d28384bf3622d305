"""Teacher-forced comparison of the GPU's drafting with the oracle (test infrastructure).

A draft decision taken on float logits can go either way at a near-tie, and one
different token changes every later pass.  So instead of comparing two
independent runs, the oracle follows the GPU's own decisions pass by pass:

* every oracle pass runs on the rows the GPU ran (its token ids, positions,
  draft-region entries, masks, hidden-state sources) and on the GPU's own
  hidden inputs (its FC-fused feature for the first pass, its previous pass's
  recurrent state after that -- the same bf16 values), so each pass is
  compared on its own and rounding differences do not accumulate along the
  chain; the pass's hidden states, and the FC-fused feature itself, are
  compared with the GPU's within the bf16 tolerance;
* every head decision is recomputed by the oracle on the GPU's own normalised
  state (the same bf16 values), so the GPU's ids must equal the oracle's except
  where the oracle's two logits lie within 1e-3 * max(1, |logit|) (a decision
  fp32 and fp64 sums may order differently) -- or, for the EAGLE-4 candidate
  head, where an id sits at the low-rank top-Kc boundary within a band derived
  from the bf16 rounding of the rank-r projection (see ``lowrank_score_band``);
  every such exemption is counted;
* tree expansion is fed the GPU's ids and log-probs (identical fp32 inputs),
  so the oracle's frontier rows and final tree must equal the GPU's bit for bit;
* verification runs on the GPU's drafts (or tree) against target logits the
  oracle computes for exactly those drafts.
"""
import copy

import numpy as np
import torch

from oracle import draft as od, numerics as onum, tree as otree

BF16_ATOL, BF16_RTOL = 2e-2, 1e-2
F32_ATOL, F32_RTOL = 1e-5, 1e-4
DECISION_REL = 1e-3      # relative margin below which an fp32-vs-fp64 decision may flip


def _tol(w):
    return (BF16_ATOL, BF16_RTOL) if w.dtype == "bf16" else (F32_ATOL, F32_RTOL)


def recorder():
    """A trace callback for ``ChainStep.draft`` / ``TreeStep.draft`` and its records."""
    recs = {}

    def cb(key, tensors):
        torch.cuda.synchronize()
        out = {}
        for k, v in tensors.items():
            if v.dtype == torch.int64:
                out[k] = v.cpu().numpy().view(np.uint64).copy()
            elif v.dtype == torch.int32:
                out[k] = v.cpu().numpy().copy()
            else:
                out[k] = v.float().cpu().numpy().astype(np.float64)
        recs[key] = out
    return recs, cb


def decision_tie(a, b):
    return abs(a - b) < DECISION_REL * max(1.0, abs(a), abs(b))


def check_hidden(w, got, ref, what, stats=None):
    """Hidden states within the bf16 tolerance, its absolute part taken at the
    row's scale: |gpu - oracle| <= atol * max(1, rms(row)) + rtol * |oracle|.
    The residual stream (hidden_prenorm) grows to an RMS of 3-13 in these
    workloads, and its differences scale with it: besides bf16 storage, the
    attention's second product takes the softmax weights as bf16 operands (a
    relative error up to 2^-9 per weight, against the oracle's exact weights),
    which moves the attention output, and through the output projection the
    whole row, in proportion to the row's magnitude."""
    atol, rtol = _tol(w)
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
    lim = atol * np.maximum(1.0, rms) + rtol * np.abs(ref)
    bad = np.abs(got - ref) > lim
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError("%s: %d of %d elements outside tolerance; first at %s: gpu %.6g oracle %.6g "
                             "(row rms %.4g)" % (what, int(bad.sum()), bad.size, i, got[i], ref[i], rms[i[:-1]][0]))
    if stats is not None:
        stats["max_err_over_rms"] = max(stats.get("max_err_over_rms", 0.0),
                                        float(np.max(np.abs(got - ref) / (rms + 1e-30))))


def check_full_head(w, W, hn, ids, lp, what, stats):
    """GPU top-k ids / log-probs of the full (or reduced-vocabulary) head against
    the oracle's head on the same normalised state ``hn``."""
    k = ids.shape[1]
    ref_ids, _, lse, logits = od.lm_head(w, W, hn, k)
    d2t = np.asarray(W["d2t"], np.int64) if getattr(w, "draft_vocab", 0) > 0 else None
    t2d = {int(t): i for i, t in enumerate(d2t)} if d2t is not None else None
    atol, rtol = _tol(w)
    for m in range(ids.shape[0]):
        for j in range(k):
            g, r = int(ids[m, j]), int(ref_ids[m, j])
            gi, ri = (t2d[g], t2d[r]) if t2d is not None else (g, r)
            if g != r:
                assert decision_tie(logits[m, gi], logits[m, ri]), \
                    "%s row %d rank %d: gpu id %d, oracle id %d, logits %.6g vs %.6g" % (
                        what, m, j, g, r, logits[m, gi], logits[m, ri])
                stats["decision_ties"] += 1
            if lp is not None:
                ref = logits[m, gi] - lse[m]
                assert abs(lp[m, j] - ref) <= atol + rtol * abs(ref), \
                    "%s row %d rank %d: log-prob %.6g vs oracle %.6g" % (what, m, j, lp[m, j], ref)
    return ref_ids


def lowrank_score_band(w, W, hn_row):
    """Low-rank scores s = z @ up^T of one row (oracle, z = bf16(hn @ down^T)) and,
    per token, a bound on how far the GPU's score can be from it: the GPU rounds
    its fp32 sum for z to bf16, so each z_i may sit one bf16 spacing away
    (spacing 2^(e-7) for |z_i| in [2^e, 2^(e+1))), and it sums the r products
    in fp32 (relative error below r * 2^-24 of the absolute sum)."""
    z = od._r(np.asarray(hn_row, np.float64)[None] @ np.asarray(W["lr_down"], np.float64).T, w.dtype)[0]
    up = np.asarray(W["lr_up"], np.float64)
    s = up @ z
    az = np.abs(z)
    spacing = np.where(az > 0, np.exp2(np.floor(np.log2(np.where(az > 0, az, 1.0))) - 7), 0.0)
    if w.dtype != "bf16":
        spacing = np.zeros_like(az)
    absu = np.abs(up)
    band = absu @ spacing + (w.rank * 2.0 ** -24 + 1e-7) * (absu @ az)
    return s, band


def check_candidate_head(w, W, hn, gpu_cand, ids, lp, what, stats):
    """EAGLE-4 candidate head on the GPU's normalised state: the GPU's candidate
    set may differ from the oracle's top-Kc only by ids inside the score band at
    the boundary; its output ids must be the best exact logits of the GPU's own
    candidate set (up to decision ties), and its log-probs the softmax over it."""
    Kc = w.num_candidates
    Wl = np.asarray(W["lm_head"], np.float64)
    atol, rtol = _tol(w)
    for m in range(hn.shape[0]):
        s, band = lowrank_score_band(w, W, hn[m])
        ref_cand = set(np.asarray(onum.topk_desc(s[None].astype(np.float32), Kc)[0]).tolist())
        got = [int(x) for x in gpu_cand[m]]
        assert len(set(got)) == Kc, "%s row %d: duplicate candidates" % (what, m)
        gset = set(got)
        if gset != ref_cand:
            inside = np.zeros(len(s), dtype=bool)
            inside[list(ref_cand)] = True
            lo_in = float(np.min((s - band)[inside]))
            hi_out = float(np.max((s + band)[~inside]))
            for u in gset - ref_cand:     # the GPU took an id the oracle left out
                assert s[u] + band[u] >= lo_in, "%s row %d: candidate %d outside the boundary band" % (what, m, u)
            for v in ref_cand - gset:     # the GPU left out an id the oracle took
                assert s[v] - band[v] <= hi_out, "%s row %d: dropped candidate %d outside the band" % (what, m, v)
            stats["boundary_ties"] += len(gset - ref_cand)
        exact = Wl[got] @ np.asarray(hn[m], np.float64)
        order = sorted(range(Kc), key=lambda i: (-np.float32(exact[i]), got[i]))
        lse = np.logaddexp.reduce(exact)
        for j in range(ids.shape[1]):
            g, r = int(ids[m, j]), got[order[j]]
            if g != r:
                assert g in gset, "%s row %d: output %d is not a candidate" % (what, m, g)
                eg, er = exact[got.index(g)], exact[order[j]]
                assert decision_tie(eg, er), "%s row %d rank %d: gpu id %d vs %d, exact logits %.6g vs %.6g" % (
                    what, m, j, g, r, eg, er)
                stats["decision_ties"] += 1
            if lp is not None:
                ref = exact[got.index(g)] - lse
                assert abs(lp[m, j] - ref) <= atol + rtol * abs(ref), \
                    "%s row %d rank %d: log-prob %.6g vs %.6g" % (what, m, j, lp[m, j], ref)


def gpu_candidates(lib, dm, hn_host, M, k):
    """The GPU candidate head's candidate ids for the recorded normalised states."""
    from eagle_speculative_decoding_step_gb300 import engine
    hn = engine.to_device(np.asarray(hn_host, np.float32), dm.w.dtype, dm.device)
    cand = torch.zeros(M, dm.w.num_candidates, dtype=torch.int32, device=dm.device)
    ids = torch.zeros(M, k, dtype=torch.int32, device=dm.device)
    lib.spec_lowrank_candidates(dm.desc, dm.weights, hn, M, k, ids, cand_ids=cand, ws=dm.ws)
    torch.cuda.synchronize()
    return cand.cpu().numpy(), ids.cpu().numpy()


def new_stats():
    return {"decision_ties": 0, "boundary_ties": 0}


def chain(w, W, aux, root, ctx, kv, recs, drafts, lib=None, dm=None, stats=None, passes=None):
    """Oracle passes of a chain on the GPU's tokens.  Returns the oracle's logits
    of K + 1 passes [B, K+1, V] (the last pass drafts the bonus row) for target
    logits.  ``kv`` is modified (the oracle's K/V writes)."""
    stats = stats if stats is not None else new_stats()
    B, K = drafts.shape
    passes = K + 1 if passes is None else passes
    check_hidden(w, recs[0]["h0"], od.fc_fuse(w, W, aux), "h0 (FC fuse)", stats)
    hid = recs[0]["h0"]
    tok = np.asarray(root, np.int64)
    logits = []
    Wl = np.asarray(W["lm_head"], np.float64)
    for i in range(passes):
        rows = {"M": B, "B": B, "R": 1, "step": i, "ctx_len": ctx, "tok": tok}
        pre, hn = od.draft_layer(w, W, rows, hid, kv)
        if i < K:
            r = recs[i]
            check_hidden(w, r["hn"], hn, "pass %d hidden_normed" % i, stats)
            check_hidden(w, r["pre"], pre, "pass %d hidden_prenorm" % i, stats)
            got = r["ids"].reshape(B, 1)
            if w.rank > 0:
                cand, again = gpu_candidates(lib, dm, r["hn"], B, 1)
                np.testing.assert_array_equal(again, got)        # same state, same kernel: same ids
                check_candidate_head(w, W, r["hn"], cand, got, None, "pass %d" % i, stats)
            else:
                check_full_head(w, W, r["hn"], got, None, "pass %d" % i, stats)
            assert np.array_equal(got[:, 0], drafts[:, i])
        if getattr(w, "draft_vocab", 0) > 0:
            # target logits live on the target vocabulary: scatter the draft entries
            lg = np.full((B, w.V), -30.0)
            lg[:, np.asarray(W["d2t"], np.int64)] = hn @ Wl.T
        else:
            lg = hn @ Wl.T
        logits.append(lg)
        g = recs[min(i, K - 1)]                 # the GPU's recurrent state out of this pass
        hid = g["hn"] if getattr(w, "norm_output", False) else g["pre"]
        if i < K:
            tok = drafts[:, i].astype(np.int64)
    return np.stack(logits, axis=1), stats


def tree(w, W, aux, root, ctx, kv, recs, gpu_tree, lib=None, dm=None, stats=None):
    """Oracle passes of a tree on the GPU's frontier rows, its expansion fed the
    GPU's ids / log-probs; checks every pass and the final tree bit for bit."""
    stats = stats if stats is not None else new_stats()
    B, k, D, N = w.B, w.top_k, w.depth, w.total
    check_hidden(w, recs[1]["h0"], od.fc_fuse(w, W, aux), "h0 (FC fuse)", stats)
    st = otree.tree_init(B, k, D, N, root, ctx)
    rows = {"M": B, "B": B, "R": 1, "step": 0, "ctx_len": ctx, "tok": np.asarray(root, np.int64)}
    hid_in = recs[1]["h0"]
    fin = None
    for d in range(1, D + 1):
        if d >= 2:
            g = recs[("rows", d)]
            for key in ("tok", "pos", "kv_idx", "hid_src"):
                np.testing.assert_array_equal(g[key], rows[key], err_msg="depth %d frontier %s" % (d, key))
            assert [int(x) for x in g["mask"]] == [int(x) for x in rows["mask"]], "depth %d frontier masks" % d
        pre, hn = od.draft_layer(w, W, rows, hid_in, kv)
        r = recs[d]
        M = rows["M"]
        check_hidden(w, r["hn"][:M], hn, "depth %d hidden_normed" % d, stats)
        check_hidden(w, r["pre"][:M], pre, "depth %d hidden_prenorm" % d, stats)
        ids, lp = r["ids"][:M], r["lp"][:M]
        if w.rank > 0:
            cand, again = gpu_candidates(lib, dm, r["hn"][:M], M, k)
            np.testing.assert_array_equal(again, ids)
            check_candidate_head(w, W, r["hn"][:M], cand, ids, lp, "depth %d" % d, stats)
        else:
            check_full_head(w, W, r["hn"][:M], ids, lp, "depth %d" % d, stats)
        res = otree.tree_expand(st, d, ids, lp)
        if d < D:
            # the next pass takes the GPU's recurrent state of this pass's rows
            rows = res
            hid_in = (r["hn"] if getattr(w, "norm_output", False) else r["pre"])[:M]
        else:
            fin = res
    for key, gkey in (("tok", "tok"), ("parent", "par"), ("depth", "dep"), ("pos", "pos")):
        np.testing.assert_array_equal(gpu_tree[gkey], fin[key], err_msg="final tree " + key)
    np.testing.assert_array_equal(gpu_tree["score"], fin["score"], err_msg="final tree scores")
    assert [[int(x) for x in row] for row in gpu_tree["mask"]] == fin["mask"], "final tree masks"
    return fin, stats


def gpu_tree_of(st):
    return {"tok": st.t_tok.cpu().numpy(), "par": st.t_par.cpu().numpy(), "dep": st.t_dep.cpu().numpy(),
            "pos": st.t_pos.cpu().numpy(), "score": st.t_score.cpu().numpy(),
            "mask": st.t_mask.cpu().numpy().view(np.uint64)}


def prefill_chain(w, W, aux_rows, input_ids, next_token, last_idx, ctx, kv, recs, drafts, stats=None):
    """The batched initial pass ([NEURON] "EagleProposer", prefill phase) and the
    recurrent passes after it, on the GPU's own rows, FC feature, states and
    tokens: the index rows bit for bit, every pass's hidden states within the
    tolerance, every draft id against the oracle's head on the GPU's state.
    Returns the oracle's logits of the K passes [B, K, V] (for target logits)."""
    from oracle import step as ostep
    stats = stats if stats is not None else new_stats()
    B, K = drafts.shape
    g = recs["prefill"]
    rows, last_row = ostep.prefill_inputs(input_ids, next_token, last_idx, ctx)
    for key in ("tok", "pos", "kv_idx"):
        np.testing.assert_array_equal(g[key], rows[key], err_msg="prefill rows " + key)
    assert [int(x) for x in g["mask"]] == [int(x) for x in rows["mask"]], "prefill masks"
    np.testing.assert_array_equal(g["last_row"], last_row)
    ctx2 = np.asarray(ctx, np.int64) + np.asarray(last_idx, np.int64) + 1
    np.testing.assert_array_equal(g["ctx_next"], ctx2)
    check_hidden(w, g["h0"], od.fc_fuse(w, W, aux_rows), "prefill h0 (FC fuse)", stats)
    pre, hn = od.draft_layer(w, W, rows, g["h0"], kv)
    check_hidden(w, g["pre"], pre, "prefill hidden_prenorm", stats)
    check_hidden(w, g["hn"], hn, "prefill hidden_normed", stats)
    Wl = np.asarray(W["lm_head"], np.float64)
    hn_last = g["hn"][last_row]
    check_full_head(w, W, hn_last, g["ids"].reshape(B, 1), None, "prefill head", stats)
    logits = [hn[last_row] @ Wl.T]
    state = g["hn"] if getattr(w, "norm_output", False) else g["pre"]
    hid = state[last_row]
    tok = drafts[:, 0].astype(np.int64)
    for i in range(1, K):
        r = {"M": B, "B": B, "R": 1, "step": i - 1, "ctx_len": ctx2, "tok": tok}
        pre_i, hn_i = od.draft_layer(w, W, r, hid, kv)
        gi = recs[i]
        check_hidden(w, gi["pre"], pre_i, "pass %d hidden_prenorm" % i, stats)
        check_hidden(w, gi["hn"], hn_i, "pass %d hidden_normed" % i, stats)
        check_full_head(w, W, gi["hn"], gi["ids"].reshape(B, 1), None, "pass %d" % i, stats)
        logits.append(hn_i @ Wl.T)
        hid = gi["hn"] if getattr(w, "norm_output", False) else gi["pre"]
        tok = drafts[:, i].astype(np.int64)
    return np.stack(logits, axis=1), stats

