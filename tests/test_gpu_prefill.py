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
    target = synth.noise(w, (B, K + 1, w.V))
    kv_ref = copy.deepcopy(kv)
    drafts_ref, logits_ref = ostep.prefill_chain_draft(w, W, aux, ids, nxt, last, ctx, kv_ref, K, keep_logits=True)
    st = engine.PrefillChainStep(dm, dev_act(aux, w), dev(ids), dev(nxt), dev(last), dev(target), K=K)
    st.run()
    torch.cuda.synchronize()
    no_device_error(dm)
    drafts = st.drafts.cpu().numpy()
    compared = 0
    for b in range(B):
        ok = True
        for i in range(K):
            if drafts[b, i] != drafts_ref[b, i]:
                ids_match(drafts[b, i:i + 1], drafts_ref[b, i:i + 1], logits_ref[b, i:i + 1])
                ok = False
                break
        compared += ok
    assert compared >= max(1, B - 2)
    # the K/V the batched pass and the recurrent passes wrote
    got = kv_host(dm)
    assert_close(got["k"], kv_ref["k"], w, "K cache")
    assert_close(got["v"], kv_ref["v"], w, "V cache")
    ref_out, ref_acc, _ = overify.verify_greedy_chain(target, drafts)
    np.testing.assert_array_equal(st.out.cpu().numpy(), ref_out)
    np.testing.assert_array_equal(st.acc.cpu().numpy(), ref_acc)
