"""Whole speculative step on the GPU (engine.ChainStep / TreeStep through the C-ABI)
against the oracle, teacher-forced: the oracle follows the GPU's own draft
decisions pass by pass (``teacher_forced``), so every run compares every pass's
hidden states, every head decision, the tree and the verification outputs --
no run is skipped because of a near-tie."""
import copy
from dataclasses import replace

import numpy as np
import pytest
import torch

from eagle_speculative_decoding_step_gb300 import binding as lib, configs, engine, synth
from oracle import step as ostep, verify as overify
import teacher_forced as tf
from gpu_helpers import SMALL_BF16, dev, dev_act, kv_host, no_device_error, setup

pytestmark = pytest.mark.gpu


def check_rejection(out, acc, ref_out, ref_acc, info, stats):
    """Rejection outputs equal the oracle's, except a request whose accept test
    or Gumbel-max sample sits within float32 reach of its decision (counted)."""
    for b in range(out.shape[0]):
        if np.array_equal(out[b], ref_out[b]) and acc[b] == ref_acc[b]:
            continue
        assert (np.abs(info["accept_margin"][b]) < 1e-5).any() or info["sample_gap"][b] < 1e-4, \
            "request %d: %s / %d vs oracle %s / %d" % (b, out[b], acc[b], ref_out[b], ref_acc[b])
        stats["decision_ties"] += 1


# The step tests draw target logits as the oracle's draft logits + N(0, 0.05): close
# enough to the drafts that requests accept some drafts, so verification is
# exercised past the first position (the workloads' own noise, sigma >= 0.5, lets
# almost nothing through at these vocabulary sizes).
TEST_SIGMA = 0.05


def run_chain_teacher_forced(w, target_noise=True):
    W, ctx, kv, dm = setup(w)
    aux = synth.make_aux(w)
    root = synth.root_tokens(w)
    temp = np.full(w.B, w.temperature, dtype=np.float32)
    tgt = torch.zeros(w.B, w.K + 1, w.V, dtype=torch.float32, device="cuda")
    st = engine.ChainStep(dm, dev_act(aux, w), dev(root), tgt, temperature=dev(temp), seed=w.philox_seed)
    recs, cb = tf.recorder()
    st.draft(trace=cb)
    torch.cuda.synchronize()
    drafts = st.drafts.cpu().numpy()
    lg, stats = tf.chain(w, W, aux, root, ctx, copy.deepcopy(kv), recs, drafts, lib=lib, dm=dm)
    noise = synth.noise(replace(w, sigma=TEST_SIGMA), (w.B, w.K + 1, w.V))
    target = ((lg if target_noise else 0.0) + noise).astype(np.float32)
    st.target.copy_(dev(target))
    st.verify()
    torch.cuda.synchronize()
    out, acc = st.out.cpu().numpy(), st.acc.cpu().numpy()
    if w.verify == "rejection":
        ref_out, ref_acc, info = overify.verify_rejection(target, drafts, temp, w.philox_seed, 0)
        check_rejection(out, acc, ref_out, ref_acc, info, stats)
    else:
        ref_out, ref_acc, _ = overify.verify_greedy_chain(target, drafts)
        np.testing.assert_array_equal(out, ref_out)
        np.testing.assert_array_equal(acc, ref_acc)
    no_device_error(dm)
    print("%s: %s, accept lengths %s" % (w.name, stats, acc.tolist()))
    return stats, acc


@pytest.mark.parametrize("w", [configs.WORKLOADS["tiny"], SMALL_BF16,
                               replace(SMALL_BF16, name="small_rej", verify="rejection", sigma=1.5, K=4),
                               replace(configs.WORKLOADS["tiny"], name="tiny_eagle31", fc_norm=True, norm_output=True),
                               replace(SMALL_BF16, name="small_eagle31", fc_norm=True, norm_output=True),
                               replace(SMALL_BF16, name="small_lowrank_chain", rank=64, num_candidates=128, V=5000,
                                       window=64, ctx=150, seed=44)],
                         ids=lambda w: w.name)
def test_chain_step(w):
    stats, acc = run_chain_teacher_forced(w)
    assert stats["decision_ties"] + stats["boundary_ties"] <= w.B * w.K
    if w.verify == "greedy" and w.rank == 0:
        # some drafts accepted: the accept path ran (the candidate head's drafts need
        # not be the full head's argmax, so its chains may all be rejected)
        assert acc.max() >= 1


def test_chain_step_reduced_draft_vocabulary():
    w = replace(SMALL_BF16, name="small_d2t_chain", V=6000, draft_vocab=2500, seed=42)
    stats, _ = run_chain_teacher_forced(w)
    assert stats["decision_ties"] <= w.B * w.K


def run_tree_teacher_forced(w):
    W, ctx, kv, dm = setup(w, max_rows=w.B * w.top_k)
    aux = synth.make_aux(w)
    root = synth.root_tokens(w)
    st = engine.TreeStep(dm, dev_act(aux, w), dev(root), None)
    recs, cb = tf.recorder()
    st.draft(trace=cb)
    torch.cuda.synchronize()
    no_device_error(dm)
    gt = tf.gpu_tree_of(st)
    fin, stats = tf.tree(w, W, aux, root, ctx, copy.deepcopy(kv), recs, gt, lib=lib, dm=dm)
    # verification + compaction on the GPU's tree (equal to the oracle's teacher-forced
    # one), target logits = the oracle's draft pass over that tree + noise; the GPU's
    # cache gets the K/V of that same pass
    kv_t = copy.deepcopy(kv)
    noise = synth.noise(replace(w, sigma=TEST_SIGMA), (w.B, w.total + 1, w.V))
    target = ostep.tree_target(w, W, aux, ctx, kv_t, fin, noise)
    st.target = dev(target)
    dm.tkv["k"].copy_(engine.to_device(kv_t["k"], w.dtype, "cuda"))
    dm.tkv["v"].copy_(engine.to_device(kv_t["v"], w.dtype, "cuda"))
    st.verify()
    torch.cuda.synchronize()
    ref_out, ref_acc, ref_src = overify.verify_greedy_tree(target, fin["tok"], fin["parent"], w.depth)
    np.testing.assert_array_equal(st.out.cpu().numpy(), ref_out)
    np.testing.assert_array_equal(st.acc.cpu().numpy(), ref_acc)
    np.testing.assert_array_equal(st.kv_src.cpu().numpy(), ref_src)
    overify.compact_kv(kv_t, ctx, ref_src, ref_acc)
    got = kv_host(dm)
    np.testing.assert_array_equal(got["k"], kv_t["k"])
    np.testing.assert_array_equal(got["v"], kv_t["v"])
    no_device_error(dm)
    print("%s: %s, accept lengths %s" % (w.name, stats, ref_acc.tolist()))
    return stats, fin


@pytest.mark.parametrize("eagle31", [False, True], ids=["eagle3", "eagle31"])
def test_tree_step(eagle31):
    w = replace(SMALL_BF16, name="small_tree", mode="tree", top_k=4, depth=3, total=10, B=2, fc_norm=eagle31,
                norm_output=eagle31)
    stats, fin = run_tree_teacher_forced(w)
    assert len(set(fin["parent"][0].tolist())) > 1          # a real tree, not a chain
    assert stats["decision_ties"] <= w.B * w.total


def test_tree_step_candidate_head():
    """Tree drafting from the EAGLE-4 candidate head ([EAGLE4] rescored candidates
    with the [EAGLET] tree parameters): children = top-k of the rescored
    candidates, log-probs over the candidates; compared pass by pass, then the
    tree is verified."""
    w = replace(SMALL_BF16, name="small_tree_lr", mode="tree", top_k=4, depth=3, total=10, B=2, rank=64,
                num_candidates=128, V=5000, seed=43)
    stats, fin = run_tree_teacher_forced(w)
    assert stats["decision_ties"] + stats["boundary_ties"] <= w.B * w.total


def test_chain_step_graph_replay():
    """The step captured in a CUDA graph replays to the same outputs."""
    w = SMALL_BF16
    W, ctx, kv, dm = setup(w)
    aux = synth.make_aux(w)
    root = synth.root_tokens(w)
    target = synth.noise(w, (w.B, w.K + 1, w.V))
    st = engine.ChainStep(dm, dev_act(aux, w), dev(root), dev(target))
    st.run()
    torch.cuda.synchronize()
    out0 = st.out.clone()
    drafts0 = st.drafts.clone()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            st.run()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(st.out, out0)
    assert torch.equal(st.drafts, drafts0)
    no_device_error(dm)
