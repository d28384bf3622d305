"""Parity at the workloads' full sizes, in the launch configuration bench.py times
(whole step captured in a CUDA graph and replayed).  The GPU runs the full
batch; the oracle recomputes a sample of requests one by one (requests are
independent), teacher-forced on the GPU's own decisions (``teacher_forced``):
every pass's hidden states and head decisions of the sampled requests are
compared, then verification on the GPU's drafts against target logits the
oracle computed for exactly those drafts.  The graph replay must reproduce the
eagerly traced drafts bit for bit.
"""
import numpy as np
import pytest
import torch

from eagle_speculative_decoding_step_gb300 import binding as lib, configs, engine, synth
from oracle import step as ostep, verify as overify
import teacher_forced as tf
from gpu_helpers import dev, dev_act
from test_gpu_step import TEST_SIGMA, check_rejection

pytestmark = pytest.mark.gpu


def _f64(W):
    return {k: np.asarray(v, dtype=np.float64) for k, v in W.items()}


def _sub_kv(kv, idx):
    s = dict(kv)
    s["block_table"] = kv["block_table"][idx]
    return s


def _graph(fn):
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fn()
    return g


@pytest.mark.parametrize("name,sample", [("llama8b_chain", [0, 1, 2, 3]), ("qwen8b_rejection", [0, 13, 31]),
                                         ("eagle4_lowrank", [0, 37, 63])])
def test_chain_full_size(name, sample):
    w = configs.WORKLOADS[name]
    W = synth.make_weights(w)
    if w.rank > 0:
        W["lr_down"], W["lr_up"] = synth.lowrank_factors(W["lm_head"], w.rank, w.dtype)
    ctx = synth.context_lengths(w)
    kv = synth.make_kv(w, ctx)
    aux = synth.make_aux(w)
    root = synth.root_tokens(w)
    dm = engine.DeviceModel(w, W, kv, ctx)          # uploads before the oracle touches kv
    W64 = _f64(W)
    del W
    idx = np.array(sample)
    temp = np.full(w.B, w.temperature, dtype=np.float32)
    tgt = torch.zeros(w.B, w.K + 1, w.V, dtype=torch.float32, device="cuda")
    st = engine.ChainStep(dm, dev_act(aux, w), dev(root), tgt, temperature=dev(temp), seed=w.philox_seed)
    recs, cb = tf.recorder()
    st.draft(trace=cb)
    torch.cuda.synchronize()
    assert dm.device_error() == 0
    drafts_all = st.drafts.cpu().numpy().copy()
    sub = {i: {k: v[idx] for k, v in r.items()} for i, r in recs.items()}
    lg, stats = tf.chain(w, W64, aux[idx], root[idx], ctx[idx], _sub_kv(kv, idx), sub, drafts_all[idx], lib=lib,
                         dm=dm)
    # target logits: the oracle's logits for the GPU's drafts + noise on the sampled
    # requests (greedy: small noise, so some drafts are accepted and the accept path
    # runs), the workload's noise elsewhere; then the whole step in the bench's launch form
    noise = synth.noise(w, (w.B, w.K + 1, w.V))
    target = noise.copy()
    small = noise[idx] * (TEST_SIGMA / w.sigma) if w.verify == "greedy" else noise[idx]
    target[idx] = (lg + small).astype(np.float32)
    st.target.copy_(dev(target))
    st.run()
    torch.cuda.synchronize()
    g = _graph(st.run)
    g.replay()
    torch.cuda.synchronize()
    assert dm.device_error() == 0
    np.testing.assert_array_equal(st.drafts.cpu().numpy(), drafts_all)       # replay == traced eager run
    drafts = drafts_all[idx]
    out = st.out.cpu().numpy()[idx]
    acc = st.acc.cpu().numpy()[idx]
    if w.verify == "rejection":
        ref_out, ref_acc, info = overify.verify_rejection(target[idx], drafts, temp[idx], w.philox_seed, 0,
                                                          req_ids=idx)
        check_rejection(out, acc, ref_out, ref_acc, info, stats)
    else:
        ref_out, ref_acc, _ = overify.verify_greedy_chain(target[idx], drafts)
        np.testing.assert_array_equal(out, ref_out)
        np.testing.assert_array_equal(acc, ref_acc)
    print("%s: %s, accept lengths %s" % (name, stats, acc.tolist()))
    assert stats["decision_ties"] + stats["boundary_ties"] <= len(idx) * w.K


def test_tree_full_size():
    w = configs.WORKLOADS["qwen4b_tree"]
    W = synth.make_weights(w)
    ctx = synth.context_lengths(w)
    kv = synth.make_kv(w, ctx)
    aux = synth.make_aux(w)
    root = synth.root_tokens(w)
    dm = engine.DeviceModel(w, W, kv, ctx)
    W64 = _f64(W)
    del W
    st = engine.TreeStep(dm, dev_act(aux, w), dev(root), None)
    recs, cb = tf.recorder()
    st.draft(trace=cb)
    torch.cuda.synchronize()
    assert dm.device_error() == 0
    gt = tf.gpu_tree_of(st)
    fin, stats = tf.tree(w, W64, aux, root, ctx, kv, recs, gt, lib=lib, dm=dm)
    assert len(set(fin["parent"][0].tolist())) > 1
    # the drafting phase replayed as the bench captures it reproduces the same tree
    g = _graph(st.draft)
    g.replay()
    torch.cuda.synchronize()
    assert dm.device_error() == 0
    for key in ("tok", "par", "dep", "pos", "score", "mask"):
        np.testing.assert_array_equal(tf.gpu_tree_of(st)[key], gt[key])
    noise = synth.noise(w, (w.B, w.total + 1, w.V)) * (TEST_SIGMA / w.sigma)
    target = ostep.tree_target(w, W64, aux, ctx, kv, fin, noise)
    st.target = dev(target)
    ref_out, ref_acc, _ = overify.verify_greedy_tree(target, fin["tok"], fin["parent"], w.depth)
    st.verify(compact=False)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(st.out.cpu().numpy(), ref_out)
    np.testing.assert_array_equal(st.acc.cpu().numpy(), ref_acc)
    print("qwen4b_tree: %s, accept length %s" % (stats, ref_acc.tolist()))
