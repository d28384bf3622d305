"""GPU parity of the draft step's calls (spec_fc_fuse, spec_draft_layer, spec_lm_head,
spec_lowrank_candidates) against the oracle on the same seeded inputs."""
import copy
from dataclasses import replace

import numpy as np
import pytest
import torch

from eagle_speculative_decoding_step_gb300 import binding as lib
from eagle_speculative_decoding_step_gb300 import configs, synth
from oracle import draft as od, tree as otree
from gpu_helpers import (SMALL_BF16, SMALL_BF16_HD128, assert_close, dev, dev_act, host, ids_match, kv_host,
                         no_device_error, setup)

pytestmark = pytest.mark.gpu

TINY = configs.WORKLOADS["tiny"]
CASES = [TINY, SMALL_BF16, SMALL_BF16_HD128]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_fc_fuse(w):
    W, ctx, kv, dm = setup(w)
    aux = synth.make_aux(w)
    ref = od.fc_fuse(w, W, aux)
    h0 = dm.hidden(w.B)
    lib.spec_fc_fuse(dm.desc, dm.weights, dev_act(aux, w), h0, w.B, dm.ws)
    assert_close(host(h0), ref, w, "h0")
    no_device_error(dm)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("step", [0, 3])
def test_draft_layer_chain_rows(w, step):
    W, ctx, kv, dm = setup(w)
    hid = synth.make_hidden(w, w.B)
    tok = synth.integers(w.seed, 1, 0, w.V, w.B)
    rows = {"M": w.B, "B": w.B, "R": 1, "step": step, "ctx_len": ctx, "tok": tok}
    kv_ref = copy.deepcopy(kv)
    ref_pre, ref_hn = od.draft_layer(w, W, rows, hid, kv_ref)
    pre, hn = dm.hidden(w.B), dm.hidden(w.B)
    r = lib.make_rows(w.B, w.B, 1, dm.ctx_len, dev(tok), step=step)
    lib.spec_draft_layer(dm.desc, dm.weights, r, dev_act(hid, w), pre, hn, dm.kv, dm.ws)
    assert_close(host(pre), ref_pre, w, "hidden_prenorm")
    assert_close(host(hn), ref_hn, w, "hidden_normed")
    got = kv_host(dm)
    assert_close(got["k"], kv_ref["k"], w, "K cache")
    assert_close(got["v"], kv_ref["v"], w, "V cache")
    no_device_error(dm)


@pytest.mark.parametrize("w", [SMALL_BF16, replace(SMALL_BF16_HD128, window=64, ctx=150)], ids=lambda w: w.name)
def test_draft_layer_tree_rows(w):
    """Frontier-style rows: several rows per request, explicit positions, draft-region
    entries, ancestor masks and gathered hidden inputs (sliding window too)."""
    k = 4
    w = replace(w, mode="tree", top_k=k, depth=4, total=12, B=2)
    W, ctx, kv, dm = setup(w, max_rows=w.B * k)
    g = np.random.default_rng(3)
    M = w.B * k
    hid = synth.make_hidden(w, w.B * k)
    tok = g.integers(0, w.V, size=M).astype(np.int32)
    d = 2
    kv_idx = np.array([1 + (d - 1) * k + f for b in range(w.B) for f in range(k)], dtype=np.int32)
    pos = np.array([ctx[b] + d for b in range(w.B) for f in range(k)], dtype=np.int32)
    mask = np.array([1 | (1 << int(g.integers(1, 1 + k))) | (1 << int(kv_idx[m])) for m in range(M)],
                    dtype=np.uint64)
    hid_src = g.integers(0, M, size=M).astype(np.int32)
    rows = {"M": M, "B": w.B, "R": k, "step": 0, "ctx_len": ctx, "tok": tok, "pos": pos, "kv_idx": kv_idx,
            "mask": [int(x) for x in mask], "hid_src": hid_src}
    kv_ref = copy.deepcopy(kv)
    ref_pre, ref_hn = od.draft_layer(w, W, rows, hid, kv_ref)
    pre, hn = dm.hidden(M), dm.hidden(M)
    r = lib.make_rows(M, w.B, k, dm.ctx_len, dev(tok), pos=dev(pos), kv_idx=dev(kv_idx),
                      mask=dev(mask.view(np.int64)), hid_src=dev(hid_src))
    lib.spec_draft_layer(dm.desc, dm.weights, r, dev_act(hid, w), pre, hn, dm.kv, dm.ws)
    assert_close(host(pre), ref_pre, w, "hidden_prenorm")
    assert_close(host(hn), ref_hn, w, "hidden_normed")
    no_device_error(dm)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("k,M", [(1, 3), (8, 8), (1, 64), (8, 1)])
def test_lm_head(w, k, M):
    if w.dtype == "f32" and M > 32:
        pytest.skip("fp32 path serves at most 32 rows")
    W, ctx, kv, dm = setup(w, max_rows=M)
    hn = synth.make_hidden(w, M, sub=5)
    ref_ids, ref_lp, ref_lse, ref_logits = od.lm_head(w, W, hn, k)
    ids = torch.zeros(M, k, dtype=torch.int32, device="cuda")
    lp = torch.zeros(M, k, dtype=torch.float32, device="cuda")
    lse = torch.zeros(M, dtype=torch.float32, device="cuda")
    lib.spec_lm_head(dm.desc, dm.weights, dev_act(hn, w), M, k, ids, lp, lse, ws=dm.ws)
    ids_match(ids.cpu().numpy(), ref_ids, ref_logits)
    assert_close(lse.cpu().numpy(), ref_lse, w, "lse")
    # log-probs of the emitted ids, from the oracle's logits
    got_ids = ids.cpu().numpy()
    want_lp = np.take_along_axis(ref_logits, got_ids, axis=1) - ref_lse[:, None]
    assert_close(lp.cpu().numpy(), want_lp, w, "logprob")
    # debug path: full logits written, same statistics
    logits = torch.zeros(M, w.V, dtype=torch.float32, device="cuda")
    ids2 = torch.zeros_like(ids)
    lp2 = torch.zeros_like(lp)
    lib.spec_lm_head(dm.desc, dm.weights, dev_act(hn, w), M, k, ids2, lp2, None, logits, ws=dm.ws)
    assert_close(logits.cpu().numpy(), ref_logits, w, "logits")
    ids_match(ids2.cpu().numpy(), ref_ids, ref_logits)
    no_device_error(dm)


LOWRANK = replace(SMALL_BF16, name="small_lowrank", rank=64, num_candidates=128, H=512, V=5000)


@pytest.mark.parametrize("M", [1, 5, 64])
def test_lowrank_candidates(M):
    w = LOWRANK
    W, ctx, kv, dm = setup(w, max_rows=M)
    hn = synth.make_hidden(w, M, sub=6)
    cand_ref, exact_ref, out_ref = od.lowrank_candidates(w, W, hn, w.num_candidates, 2)
    cand = torch.zeros(M, w.num_candidates, dtype=torch.int32, device="cuda")
    exact = torch.zeros(M, w.num_candidates, dtype=torch.float32, device="cuda")
    out = torch.zeros(M, 2, dtype=torch.int32, device="cuda")
    lib.spec_lowrank_candidates(dm.desc, dm.weights, dev_act(hn, w), M, 2, out, cand, exact, ws=dm.ws)
    cand, exact, out = cand.cpu().numpy(), exact.cpu().numpy(), out.cpu().numpy()
    # candidate sets: equal up to near-ties at the boundary of the low-rank scores
    z = od._r(np.asarray(hn, np.float64) @ np.asarray(W["lr_down"], np.float64).T, w.dtype)
    s = z @ np.asarray(W["lr_up"], np.float64).T
    for m in range(M):
        a, b = set(cand[m].tolist()), set(cand_ref[m].tolist())
        if a != b:
            kth = np.sort(s[m])[::-1][w.num_candidates - 1]
            for t in a ^ b:
                assert abs(s[m, t] - kth) < 2e-2, "candidate %d far from the boundary" % t
        # exact rescoring of whatever was retrieved
        want = np.asarray(W["lm_head"], np.float64)[cand[m]] @ np.asarray(hn[m], np.float64)
        assert_close(exact[m], want, w, "exact logits")
    full = np.asarray(hn, np.float64) @ np.asarray(W["lm_head"], np.float64).T
    ids_match(out, out_ref, full)
    no_device_error(dm)


DRAFTVOCAB = replace(SMALL_BF16, name="small_d2t", V=6000, draft_vocab=2500, seed=41)


@pytest.mark.parametrize("k,M", [(1, 4), (8, 8)])
def test_lm_head_reduced_draft_vocabulary(k, M):
    """LM head over draft_vocab rows; emitted ids are the mapped target ids (d2t)."""
    w = DRAFTVOCAB
    W, ctx, kv, dm = setup(w, max_rows=M)
    assert W["lm_head"].shape[0] == w.draft_vocab
    hn = synth.make_hidden(w, M, sub=7)
    ref_ids, ref_lp, ref_lse, ref_logits = od.lm_head(w, W, hn, k)
    ids = torch.zeros(M, k, dtype=torch.int32, device="cuda")
    lp = torch.zeros(M, k, dtype=torch.float32, device="cuda")
    lse = torch.zeros(M, dtype=torch.float32, device="cuda")
    lib.spec_lm_head(dm.desc, dm.weights, dev_act(hn, w), M, k, ids, lp, lse, ws=dm.ws)
    got = ids.cpu().numpy()
    # compare in draft-vocabulary indices (t2d of the emitted ids)
    t2d = {int(t): i for i, t in enumerate(W["d2t"])}
    got_d = np.vectorize(t2d.get)(got)
    ref_d = np.vectorize(t2d.get)(ref_ids)
    ids_match(got_d, ref_d, ref_logits)
    assert set(got.reshape(-1).tolist()) <= set(W["d2t"].tolist())
    assert_close(lse.cpu().numpy(), ref_lse, w, "lse")
    no_device_error(dm)
