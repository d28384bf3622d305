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
import teacher_forced as tf
from gpu_helpers import (SMALL_BF16, SMALL_BF16_HD128, assert_close, dev, dev_act, host, ids_match, kv_host,
                         no_device_error, setup)

pytestmark = pytest.mark.gpu

TINY = configs.WORKLOADS["tiny"]
CASES = [TINY, SMALL_BF16, SMALL_BF16_HD128]


@pytest.mark.parametrize("w", CASES + [replace(TINY, name="tiny_fc_norm", fc_norm=True),
                                       replace(SMALL_BF16, name="small_fc_norm", fc_norm=True, B=40)],
                         ids=lambda w: w.name)
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


LONG_WINDOW = replace(configs.WORKLOADS["eagle4_lowrank"], name="long_window", H=512, I=1000, V=3000, rank=0,
                      num_candidates=0, B=16, seed=26)
LONG_RAGGED = replace(configs.WORKLOADS["qwen8b_rejection"], name="long_ragged", H=512, I=1000, V=3000, seed=27)


@pytest.mark.parametrize("w,step", [(LONG_WINDOW, 1), (LONG_RAGGED, 3)], ids=["window1024_ctx8192", "ragged512_2048"])
def test_draft_layer_long_context(w, step):
    """The attention shapes of the large workloads (32 q / 8 kv heads, head dim 128;
    8192-token contexts under a 1024-key sliding window, or ragged 512..2048-token
    contexts over 32 requests) with a narrow hidden size so the oracle stays quick:
    many key tiles per work item, several items per CTA of the persistent grid."""
    W, ctx, kv, dm = setup(w)
    hid = synth.make_hidden(w, w.B)
    tok = synth.integers(w.seed, 1, 0, w.V, w.B)
    rows = {"M": w.B, "B": w.B, "R": 1, "step": step, "ctx_len": ctx, "tok": tok}
    ref_pre, ref_hn = od.draft_layer(w, W, rows, hid, kv)
    pre, hn = dm.hidden(w.B), dm.hidden(w.B)
    r = lib.make_rows(w.B, w.B, 1, dm.ctx_len, dev(tok), step=step, max_ctx=int(ctx.max()))
    lib.spec_draft_layer(dm.desc, dm.weights, r, dev_act(hid, w), pre, hn, dm.kv, dm.ws)
    assert_close(host(pre), ref_pre, w, "hidden_prenorm")
    assert_close(host(hn), ref_hn, w, "hidden_normed")
    no_device_error(dm)


BLOCK_CASES = [
    replace(LONG_RAGGED, name="block8", block_size=8, B=8, seed=31),            # 8-slot runs
    replace(LONG_RAGGED, name="block24", block_size=24, B=8, seed=32),          # runs inside 24-slot blocks
    replace(LONG_RAGGED, name="block12", block_size=12, B=8, seed=33),          # per-row copies
    replace(LONG_WINDOW, name="block64_window", block_size=64, B=4, ctx=3000, seed=34),
    replace(SMALL_BF16, name="block8_hd64", block_size=8, ctx_range=(40, 300), seed=35),
]


@pytest.mark.parametrize("w", BLOCK_CASES, ids=lambda w: w.name)
def test_draft_layer_block_sizes(w):
    """Cache block sizes of 8, 24, 12 and 64 slots: the tensor-copy attention loads
    8- or 16-slot runs of a block (12 takes the per-row copy kernel), with ragged
    contexts or a sliding window, head dims 128 and 64."""
    W, ctx, kv, dm = setup(w)
    hid = synth.make_hidden(w, w.B)
    tok = synth.integers(w.seed, 1, 0, w.V, w.B)
    rows = {"M": w.B, "B": w.B, "R": 1, "step": 2, "ctx_len": ctx, "tok": tok}
    ref_pre, ref_hn = od.draft_layer(w, W, rows, hid, kv)
    pre, hn = dm.hidden(w.B), dm.hidden(w.B)
    r = lib.make_rows(w.B, w.B, 1, dm.ctx_len, dev(tok), step=2, max_ctx=int(ctx.max()))
    lib.spec_draft_layer(dm.desc, dm.weights, r, dev_act(hid, w), pre, hn, dm.kv, dm.ws)
    assert_close(host(pre), ref_pre, w, "hidden_prenorm")
    assert_close(host(hn), ref_hn, w, "hidden_normed")
    no_device_error(dm)


LONG_TREE = replace(configs.WORKLOADS["qwen4b_tree"], name="long_tree", H=512, I=1000, V=3000, B=2, ctx=0,
                    ctx_range=(3000, 4096), seed=28)


@pytest.mark.parametrize("w,k", [(SMALL_BF16, 4), (replace(SMALL_BF16_HD128, window=64, ctx=150), 4),
                                 (replace(SMALL_BF16, name="small_bf16_k8"), 8),
                                 (replace(SMALL_BF16, name="small_bf16_k8_block12", block_size=12), 8),
                                 (replace(SMALL_BF16_HD128, name="hd128_k8", ctx=333), 8),
                                 (replace(SMALL_BF16_HD128, name="hd128_k8_window", window=128, ctx=700), 8),
                                 (replace(SMALL_BF16_HD128, name="hd128_k6", ctx=200), 6),
                                 (LONG_TREE, 8)],
                         ids=["k4", "hd128_window_k4", "k8", "k8_block12", "hd128_k8", "hd128_k8_window", "hd128_k6",
                              "long_tree_32_8_heads"])
def test_draft_layer_tree_rows(w, k):
    """Frontier-style rows: several rows per request, explicit positions, draft-region
    entries, ancestor masks and gathered hidden inputs (sliding window too).  Eight
    rows of four q heads are 32 queries per kv head: items of two m-tiles (six rows:
    24 queries, the second m-tile half empty), with 16- and 12-slot cache blocks,
    head dims 64 and 128, and the tree workload's attention shape (32 / 8 heads,
    contexts of 3000-4096 keys: many tiles per item)."""
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
        # the fp32 path serves at most 32 rows: the call is refused before any launch
        W, ctx, kv, dm = setup(w, max_rows=32)
        hn = torch.zeros(M, w.H, dtype=torch.float32, device="cuda")
        ids = torch.zeros(M, k, dtype=torch.int32, device="cuda")
        lp = torch.zeros(M, k, dtype=torch.float32, device="cuda")
        with pytest.raises(lib.SpecError) as e:
            lib.spec_lm_head(dm.desc, dm.weights, hn, M, k, ids, lp, ws=dm.ws)
        assert e.value.status == -2
        return
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


@pytest.mark.parametrize("w", [LOWRANK, replace(LOWRANK, name="small_lowrank_v5024", V=5024, seed=42)],
                         ids=lambda w: w.name)
@pytest.mark.parametrize("M", [1, 5, 64])
def test_lowrank_candidates(M, w):
    """Candidate head at 1, 5 and 64 rows, vocabularies of 5000 and 5024."""
    W, ctx, kv, dm = setup(w, max_rows=M)
    hn = synth.make_hidden(w, M, sub=6)
    cand_ref, exact_ref, out_ref = od.lowrank_candidates(w, W, hn, w.num_candidates, 2)
    cand = torch.zeros(M, w.num_candidates, dtype=torch.int32, device="cuda")
    exact = torch.zeros(M, w.num_candidates, dtype=torch.float32, device="cuda")
    out = torch.zeros(M, 2, dtype=torch.int32, device="cuda")
    lib.spec_lowrank_candidates(dm.desc, dm.weights, dev_act(hn, w), M, 2, out, cand, exact, ws=dm.ws)
    cand, exact, out = cand.cpu().numpy(), exact.cpu().numpy(), out.cpu().numpy()
    # candidate sets: equal up to ids inside the band the bf16 rounding of z and fp32
    # sums allow at the boundary of the low-rank scores; the outputs are the best
    # exact logits of the GPU's own candidates
    stats = tf.new_stats()
    tf.check_candidate_head(w, W, np.asarray(hn, np.float64), cand, out, None, "lowrank", stats)
    for m in range(M):
        # exact rescoring of whatever was retrieved
        want = np.asarray(W["lm_head"], np.float64)[cand[m]] @ np.asarray(hn[m], np.float64)
        assert_close(exact[m], want, w, "exact logits")
    assert stats["boundary_ties"] <= M
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


@pytest.mark.parametrize("k,M", [(8, 13), (8, 64), (1, 16), (8, 1), (1, 37)])
def test_lm_head_many_tiles_exact_ties(k, M):
    """Several 128-row tiles per CTA, and exact ties planted by duplicating weight rows
    (some duplicates in the same tile, some in other CTAs' ranges): the fused top-k
    equals the top-k of the kernel's own full logits (larger first, equal logits to
    the smaller id) and its lse matches theirs; the ids match the oracle's up to
    near-ties."""
    from eagle_speculative_decoding_step_gb300 import engine
    w = replace(SMALL_BF16, name="small_bf16_v40k", V=40000, seed=23)
    W = synth.make_weights(w)
    hn = synth.make_hidden(w, M, sub=8)
    # plant the rows most likely to be in the top-k several times
    best = np.argsort(-(hn.astype(np.float64) @ W["lm_head"].astype(np.float64).T), axis=1)[:, :3]
    dst = [3, 130, 131, 20000, 39999]
    for i, r in enumerate(best.reshape(-1)[:len(dst)]):
        W["lm_head"][dst[i]] = W["lm_head"][r]
    ctx = synth.context_lengths(w)
    kv = synth.make_kv(w, ctx)
    dm = engine.DeviceModel(w, W, kv, ctx, max_rows=M)
    ids = torch.zeros(M, k, dtype=torch.int32, device="cuda")
    lp = torch.zeros(M, k, dtype=torch.float32, device="cuda")
    lse = torch.zeros(M, dtype=torch.float32, device="cuda")
    lib.spec_lm_head(dm.desc, dm.weights, dev_act(hn, w), M, k, ids, lp, lse, ws=dm.ws)
    logits = torch.zeros(M, w.V, dtype=torch.float32, device="cuda")
    ids2 = torch.zeros_like(ids)
    lp2 = torch.zeros_like(lp)
    lib.spec_lm_head(dm.desc, dm.weights, dev_act(hn, w), M, k, ids2, lp2, None, logits, ws=dm.ws)
    L = logits.cpu().numpy().astype(np.float64)
    got = ids.cpu().numpy()
    for m in range(M):
        order = np.lexsort((np.arange(w.V), -L[m]))[:k]
        np.testing.assert_array_equal(got[m], order, err_msg="row %d" % m)
    want_lse = np.log(np.exp(L - L.max(1, keepdims=True)).sum(1)) + L.max(1)
    np.testing.assert_allclose(lse.cpu().numpy(), want_lse, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(lp.cpu().numpy(), np.take_along_axis(L, got, 1) - want_lse[:, None], rtol=1e-5,
                               atol=1e-5)
    ref_ids, _, ref_lse, ref_logits = od.lm_head(w, W, hn, k)
    ids_match(got, ref_ids, ref_logits)
    assert_close(lse.cpu().numpy(), ref_lse, w, "lse")
    # the planted duplicates did produce exact ties among the emitted ids
    if k == 8:
        assert any(len(set(L[m, got[m]].tolist())) < k for m in range(M))
    no_device_error(dm)


def _lowrank_model(w, up):
    from eagle_speculative_decoding_step_gb300 import engine
    W = synth.make_weights(w)
    W["lr_down"], _ = synth.lowrank_factors(W["lm_head"], w.rank, w.dtype)
    W["lr_up"] = up
    ctx = synth.context_lengths(w)
    kv = synth.make_kv(w, ctx)
    return W, engine.DeviceModel(w, W, kv, ctx, max_rows=8)


def _run_lowrank(w, W, dm, hn, M):
    cand = torch.zeros(M, w.num_candidates, dtype=torch.int32, device="cuda")
    out = torch.zeros(M, 1, dtype=torch.int32, device="cuda")
    lib.spec_lowrank_candidates(dm.desc, dm.weights, dev_act(hn, w), M, 1, out, cand, ws=dm.ws)
    no_device_error(dm)
    return cand.cpu().numpy(), out.cpu().numpy()


def test_lowrank_candidates_tied_groups():
    """Low-rank scores with only 40 distinct values per row (rows of the up factor
    repeat): the Kc-th candidate falls inside a group of equal scores, and the
    candidates taken from it are its smallest ids, in id order."""
    w = replace(LOWRANK, name="small_lowrank_groups", seed=24)
    g = np.random.default_rng(5)
    rows = synth.round_to_bf16(synth.normal((40, w.rank), w.seed, "aux", 0.1, 0.0, 91))
    grp = g.integers(0, 40, size=w.V)
    W, dm = _lowrank_model(w, rows[grp].astype(np.float32))
    M = 6
    hn = synth.make_hidden(w, M, sub=9)
    cand, out = _run_lowrank(w, W, dm, hn, M)
    z = od._r(np.asarray(hn, np.float64) @ np.asarray(W["lr_down"], np.float64).T, w.dtype)
    gv = z @ np.asarray(W["lr_up"], np.float64)[np.unique(grp, return_index=True)[1]].T   # [M, groups present]
    present = np.unique(grp)
    checked = 0
    for m in range(M):
        srt = np.argsort(-gv[m])
        order, vals = present[srt], gv[m][srt]
        want = []
        used = 0
        for gi in order:
            ids = np.nonzero(grp == gi)[0]
            want.extend(ids[:w.num_candidates - len(want)].tolist())
            used += 1
            if len(want) == w.num_candidates:
                break
        # the groups taken (and the next) must be ordered the same in any precision
        if np.min(np.abs(np.diff(vals[:used + 1]))) < 1e-4 * max(1.0, np.abs(vals).max()):
            continue
        np.testing.assert_array_equal(cand[m], want, err_msg="row %d" % m)
        checked += 1
    assert checked >= 3


def test_lowrank_candidates_all_equal_scores():
    """Every low-rank score equal (one repeated up row) and more of them than the
    selection keeps on chip: the candidates are ids 0 .. Kc-1, and the emitted
    token is the best exact logit among them."""
    w = replace(LOWRANK, name="small_lowrank_flat", V=8000, seed=25)
    row = synth.round_to_bf16(synth.normal((1, w.rank), w.seed, "aux", 0.1, 0.0, 92))
    W, dm = _lowrank_model(w, np.repeat(row, w.V, axis=0).astype(np.float32))
    M = 2
    hn = synth.make_hidden(w, M, sub=10)
    cand, out = _run_lowrank(w, W, dm, hn, M)
    for m in range(M):
        np.testing.assert_array_equal(cand[m], np.arange(w.num_candidates))
    exact = np.asarray(hn, np.float64) @ np.asarray(W["lm_head"], np.float64)[:w.num_candidates].T
    ids_match(out[:, 0], np.argmax(exact, axis=1), exact)


def test_lowrank_candidates_full_vocabulary():
    """The candidate head at the EAGLE-4 workload's head shapes (H 4096, V 128256,
    rank 128, 128 candidates, 64 rows; random factors): every candidate set equals
    the oracle's up to near-ties at the boundary of the low-rank scores, and the
    exact rescoring holds for every candidate retrieved."""
    from eagle_speculative_decoding_step_gb300 import engine
    w = replace(configs.WORKLOADS["eagle4_lowrank"], name="lowrank_full_vocab", nq=4, nkv=1, I=256, B=4, ctx=64,
                window=0, seed=28)
    W = synth.make_weights(w)
    W["lr_down"] = synth.round_to_bf16(synth.normal((w.rank, w.H), w.seed, "aux", 0.02, 0.0, 93))
    W["lr_up"] = synth.round_to_bf16(synth.normal((w.V, w.rank), w.seed, "aux", 0.02, 0.0, 94))
    ctx = synth.context_lengths(w)
    dm = engine.DeviceModel(w, W, synth.make_kv(w, ctx), ctx, max_rows=64)
    M = 64
    hn = synth.make_hidden(w, M, sub=11)
    cand = torch.zeros(M, w.num_candidates, dtype=torch.int32, device="cuda")
    exact = torch.zeros(M, w.num_candidates, dtype=torch.float32, device="cuda")
    out = torch.zeros(M, 1, dtype=torch.int32, device="cuda")
    lib.spec_lowrank_candidates(dm.desc, dm.weights, dev_act(hn, w), M, 1, out, cand, exact, ws=dm.ws)
    no_device_error(dm)
    cand, exact = cand.cpu().numpy(), exact.cpu().numpy()
    z = od._r(np.asarray(hn, np.float64) @ np.asarray(W["lr_down"], np.float64).T, w.dtype)
    s = z @ np.asarray(W["lr_up"], np.float64).T
    lm = np.asarray(W["lm_head"], np.float32)
    stats = tf.new_stats()
    tf.check_candidate_head(w, W, np.asarray(hn, np.float64), cand, out.cpu().numpy(), None, "full", stats)
    for m in range(M):
        _, band = tf.lowrank_score_band(w, W, hn[m])
        # candidates come in score order (up to the band)
        sc = s[m, cand[m]]
        assert np.all(np.diff(sc) <= band[cand[m]][:-1] + band[cand[m]][1:])
        want = lm[cand[m]].astype(np.float64) @ np.asarray(hn[m], np.float64)
        assert_close(exact[m], want, w, "exact logits")
