"""Whole speculative step on the GPU (engine.ChainStep / TreeStep through the C-ABI)
against the oracle's step on the same seeded inputs."""
import copy
from dataclasses import replace

import numpy as np
import pytest
import torch

from eagle_speculative_decoding_step_gb300 import configs, engine, synth
from oracle import step as ostep, verify as overify, tree as otree, draft as od
from gpu_helpers import (SMALL_BF16, assert_close, dev, dev_act, host, ids_match, kv_host, no_device_error, setup,
                         tree_mismatch_is_near_tie)

pytestmark = pytest.mark.gpu


def _chain_case(w):
    W, ctx, kv, dm = setup(w)
    aux = synth.make_aux(w)
    root = synth.root_tokens(w)
    noise = synth.noise(w, (w.B, w.K + 1, w.V))
    target = ostep.chain_target(w, W, aux, root, ctx, kv, w.K, noise)
    return W, ctx, kv, dm, aux, root, target


@pytest.mark.parametrize("w", [configs.WORKLOADS["tiny"], SMALL_BF16,
                               replace(SMALL_BF16, name="small_rej", verify="rejection", sigma=1.5, K=4),
                               replace(configs.WORKLOADS["tiny"], name="tiny_eagle31", fc_norm=True, norm_output=True),
                               replace(SMALL_BF16, name="small_eagle31", fc_norm=True, norm_output=True)],
                         ids=lambda w: w.name)
def test_chain_step(w):
    W, ctx, kv, dm, aux, root, target = _chain_case(w)
    temp = np.full(w.B, w.temperature, dtype=np.float32)
    kv_ref = copy.deepcopy(kv)
    drafts_ref, logits_ref = ostep.chain_draft(w, W, aux, root, ctx, copy.deepcopy(kv), w.K, keep_logits=True)
    st = engine.ChainStep(dm, dev_act(aux, w), dev(root), dev(target), temperature=dev(temp), seed=w.philox_seed)
    st.run()
    torch.cuda.synchronize()
    drafts = st.drafts.cpu().numpy()
    # greedy drafting: ids equal to the oracle's up to near-ties; stop comparing after one
    for i in range(w.K):
        if not np.array_equal(drafts[:, i], drafts_ref[:, i]):
            ids_match(drafts[:, i], drafts_ref[:, i], logits_ref[:, i])
            pytest.skip("near-tie in the draft chain at step %d" % i)
    if w.verify == "rejection":
        ref_out, ref_acc, _ = overify.verify_rejection(target, drafts_ref, temp, w.philox_seed, 0)
    else:
        ref_out, ref_acc, _ = overify.verify_greedy_chain(target, drafts_ref)
    np.testing.assert_array_equal(st.out.cpu().numpy(), ref_out)
    np.testing.assert_array_equal(st.acc.cpu().numpy(), ref_acc)
    no_device_error(dm)


@pytest.mark.parametrize("eagle31", [False, True], ids=["eagle3", "eagle31"])
def test_tree_step(eagle31):
    w = replace(SMALL_BF16, name="small_tree", mode="tree", top_k=4, depth=3, total=10, B=2, fc_norm=eagle31,
                norm_output=eagle31)
    W, ctx, kv, dm = setup(w, max_rows=w.B * w.top_k)
    aux = synth.make_aux(w)
    root = synth.root_tokens(w)
    trace = []
    fin = ostep.tree_draft(w, W, aux, root, ctx, copy.deepcopy(kv), w.top_k, w.depth, w.total, trace=trace)
    kv_t = copy.deepcopy(kv)
    noise = synth.noise(w, (w.B, w.total + 1, w.V))
    target = ostep.tree_target(w, W, aux, ctx, kv_t, fin, noise)
    st = engine.TreeStep(dm, dev_act(aux, w), dev(root), dev(target))
    st.draft()
    torch.cuda.synchronize()
    got_tok, got_par = st.t_tok.cpu().numpy(), st.t_par.cpu().numpy()
    if not (np.array_equal(got_tok, fin["tok"]) and np.array_equal(got_par, fin["parent"])):
        assert tree_mismatch_is_near_tie(got_tok, got_par, fin, st.t_score.cpu().numpy()), \
            "tree differs away from any score near-tie"
        pytest.skip("near-tie in tree drafting")
    np.testing.assert_array_equal(st.t_dep.cpu().numpy(), fin["depth"])
    np.testing.assert_allclose(st.t_score.cpu().numpy(), fin["score"], atol=3e-2, rtol=1e-2)
    # verification + compaction on the target-shaped cache
    ref_out, ref_acc, ref_src = overify.verify_greedy_tree(target, fin["tok"], fin["parent"], w.depth)
    dm.tkv["k"].copy_(engine.to_device(kv_t["k"], w.dtype, "cuda"))
    dm.tkv["v"].copy_(engine.to_device(kv_t["v"], w.dtype, "cuda"))
    st.verify()
    np.testing.assert_array_equal(st.out.cpu().numpy(), ref_out)
    np.testing.assert_array_equal(st.acc.cpu().numpy(), ref_acc)
    overify.compact_kv(kv_t, ctx, ref_src, ref_acc)
    got = kv_host(dm)
    np.testing.assert_array_equal(got["k"], kv_t["k"])
    no_device_error(dm)


def test_chain_step_graph_replay():
    """The step captured in a CUDA graph replays to the same outputs."""
    w = SMALL_BF16
    W, ctx, kv, dm, aux, root, target = _chain_case(w)
    st = engine.ChainStep(dm, dev_act(aux, w), dev(root), dev(target))
    st.run()
    torch.cuda.synchronize()
    out0 = st.out.clone()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            st.run()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(st.out, out0)
    no_device_error(dm)


def test_chain_step_reduced_draft_vocabulary():
    w = replace(SMALL_BF16, name="small_d2t_chain", V=6000, draft_vocab=2500, seed=42)
    W, ctx, kv, dm, aux, root, _ = _chain_case_nolm(w)
    drafts_ref, logits_ref = ostep.chain_draft(w, W, aux, root, ctx, copy.deepcopy(kv), w.K, keep_logits=True)
    target = synth.noise(w, (w.B, w.K + 1, w.V))
    st = engine.ChainStep(dm, dev_act(aux, w), dev(root), dev(target))
    st.run()
    torch.cuda.synchronize()
    drafts = st.drafts.cpu().numpy()
    t2d = {int(t): i for i, t in enumerate(W["d2t"])}
    for i in range(w.K):
        if not np.array_equal(drafts[:, i], drafts_ref[:, i]):
            ids_match(np.vectorize(t2d.get)(drafts[:, i]), np.vectorize(t2d.get)(drafts_ref[:, i]), logits_ref[:, i])
            return
    ref_out, ref_acc, _ = overify.verify_greedy_chain(target, drafts_ref)
    np.testing.assert_array_equal(st.out.cpu().numpy(), ref_out)
    no_device_error(dm)


def _chain_case_nolm(w):
    W, ctx, kv, dm = setup(w)
    return W, ctx, kv, dm, synth.make_aux(w), synth.root_tokens(w), None


def test_tree_step_candidate_head():
    """Tree drafting from the EAGLE-4 candidate head: children = top-k of the rescored
    candidates, ranked by log-probs over the candidates."""
    w = replace(SMALL_BF16, name="small_tree_lr", mode="tree", top_k=4, depth=3, total=10, B=2, rank=64,
                num_candidates=128, V=5000, seed=43)
    W, ctx, kv, dm = setup(w, max_rows=w.B * w.top_k)
    aux = synth.make_aux(w)
    root = synth.root_tokens(w)
    fin = ostep.tree_draft(w, W, aux, root, ctx, copy.deepcopy(kv), w.top_k, w.depth, w.total)
    st = engine.TreeStep(dm, dev_act(aux, w), dev(root), None)
    st.draft()
    torch.cuda.synchronize()
    no_device_error(dm)
    tok, par = st.t_tok.cpu().numpy(), st.t_par.cpu().numpy()
    if not (np.array_equal(tok, fin["tok"]) and np.array_equal(par, fin["parent"])):
        assert tree_mismatch_is_near_tie(tok, par, fin, st.t_score.cpu().numpy()), \
            "tree differs away from any score near-tie"
        pytest.skip("near-tie while drafting")
    np.testing.assert_allclose(st.t_score.cpu().numpy(), fin["score"], atol=3e-2, rtol=1e-2)
