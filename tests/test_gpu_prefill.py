"""GPU parity of the batched initial draft pass over the verified tokens
(spec_prefill_inputs, spec_fc_fuse / spec_draft_layer over B*(1+K) rows,
spec_gather_rows, then the recurrent passes) against the oracle."""
import copy
from dataclasses import replace

import numpy as np
import pytest
import torch

from eagle_speculative_decoding_step_gb300 import binding as lib
from eagle_speculative_decoding_step_gb300 import engine, synth
from oracle import step as ostep, verify as overify
import teacher_forced as tf
from gpu_helpers import SMALL_BF16, assert_close, dev, dev_act, host, ids_match, kv_host, no_device_error

pytestmark = pytest.mark.gpu


def test_prefill_inputs_match_oracle():
    g = np.random.default_rng(1)
    B, R = 7, 6
    ids = g.integers(0, 1000, size=(B, R)).astype(np.int32)
    nxt = g.integers(0, 1000, size=B).astype(np.int32)
    last = g.integers(0, R, size=B).astype(np.int32)
    ctx = g.integers(10, 500, size=B).astype(np.int32)
    rows, last_row = ostep.prefill_inputs(ids, nxt, last, ctx)
    i32 = dict(dtype=torch.int32, device="cuda")
    tok, pos, kvi, lr, cn = (torch.zeros(B * R, **i32), torch.zeros(B * R, **i32), torch.zeros(B * R, **i32),
                             torch.zeros(B, **i32), torch.zeros(B, **i32))
    mask = torch.zeros(B * R, dtype=torch.int64, device="cuda")
    lib.spec_prefill_inputs(B, R, dev(ids), dev(nxt), dev(last), dev(ctx), tok, pos, kvi, mask, lr, cn)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(tok.cpu().numpy(), rows["tok"])
    np.testing.assert_array_equal(pos.cpu().numpy(), rows["pos"])
    np.testing.assert_array_equal(kvi.cpu().numpy(), rows["kv_idx"])
    np.testing.assert_array_equal(mask.cpu().numpy().astype(np.uint64), np.array(rows["mask"], dtype=np.uint64))
    np.testing.assert_array_equal(lr.cpu().numpy(), last_row)
    np.testing.assert_array_equal(cn.cpu().numpy(), ctx + last + 1)


def test_gather_rows():
    src = torch.randn(50, 96, device="cuda").to(torch.bfloat16)
    rows = torch.tensor([3, 0, 49, 7], dtype=torch.int32, device="cuda")
    dst = torch.zeros(4, 96, dtype=torch.bfloat16, device="cuda")
    lib.spec_gather_rows(src, 50, 96 * 2, rows, 4, dst)
    torch.cuda.synchronize()
    assert torch.equal(dst, src[rows.long()])


@pytest.mark.parametrize("B,K", [(3, 4), (60, 4)])        # 15 and 300 rows in the batched pass
def test_prefill_chain_step(B, K):
    """The batched initial pass and the recurrent passes after it, teacher-forced on
    the GPU's own rows, states and drafts (every pass compared, no near-tie
    skipped), then verification against target logits the oracle computed for the
    GPU's drafts."""
    w = replace(SMALL_BF16, name="prefill", B=B, K=K, ctx=70, seed=31)
    R = K + 1
    W = synth.make_weights(w)
    ctx = synth.context_lengths(w)
    kv = synth.make_kv(replace(w, K=2 * K + 1), ctx)          # room for R prefill rows + K-1 recurrent entries
    dm = engine.DeviceModel(w, W, kv, ctx, max_rows=B * R)
    g = np.random.default_rng(B)
    aux = synth.make_aux(w, rows=B * R)
    ids = g.integers(0, w.V, size=(B, R)).astype(np.int32)
    nxt = g.integers(0, w.V, size=B).astype(np.int32)
    last = g.integers(0, R, size=B).astype(np.int32)
    tgt = torch.zeros(B, K + 1, w.V, dtype=torch.float32, device="cuda")
    st = engine.PrefillChainStep(dm, dev_act(aux, w), dev(ids), dev(nxt), dev(last), tgt, K=K)
    recs, cb = tf.recorder()
    st.draft(trace=cb)
    torch.cuda.synchronize()
    no_device_error(dm)
    drafts = st.drafts.cpu().numpy()
    kv_ref = copy.deepcopy(kv)
    lg, stats = tf.prefill_chain(w, W, aux, ids, nxt, last, ctx, kv_ref, recs, drafts)
    # the K/V the batched pass and the recurrent passes wrote (same inputs on both sides)
    got = kv_host(dm)
    assert_close(got["k"], kv_ref["k"], w, "K cache")
    assert_close(got["v"], kv_ref["v"], w, "V cache")
    noise = synth.noise(replace(w, sigma=0.05), (B, K + 1, w.V))
    target = noise.copy()
    target[:, :K] += lg
    st.target.copy_(dev(target.astype(np.float32)))
    st.verify()
    torch.cuda.synchronize()
    ref_out, ref_acc, _ = overify.verify_greedy_chain(target.astype(np.float32), drafts)
    np.testing.assert_array_equal(st.out.cpu().numpy(), ref_out)
    np.testing.assert_array_equal(st.acc.cpu().numpy(), ref_acc)
    assert ref_acc.max() >= 1
    print("prefill B=%d K=%d: %s, accept lengths %s" % (B, K, stats, ref_acc.tolist()[:8]))
    assert stats["decision_ties"] <= B * K
