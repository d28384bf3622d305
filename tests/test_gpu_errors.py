"""Device-side checks: bad indices set the workspace error word and the offending
access is skipped (no trap, the context stays usable)."""
from dataclasses import replace

import numpy as np
import pytest
import torch

from eagle_speculative_decoding_step_gb300 import binding as lib
from eagle_speculative_decoding_step_gb300 import synth
from gpu_helpers import SMALL_BF16, dev, dev_act, setup

pytestmark = pytest.mark.gpu

SPEC_ERR_DEVICE = -6


def test_token_out_of_vocabulary_sets_error_word():
    w = SMALL_BF16
    W, ctx, kv, dm = setup(w)
    lib.spec_clear_device_error(dm.ws)
    assert dm.device_error() == 0
    tok = np.array([1, w.V + 5, 2], dtype=np.int32)
    hid = synth.make_hidden(w, w.B)
    pre, hn = dm.hidden(w.B), dm.hidden(w.B)
    r = lib.make_rows(w.B, w.B, 1, dm.ctx_len, dev(tok), step=0)
    lib.spec_draft_layer(dm.desc, dm.weights, r, dev_act(hid, w), pre, hn, dm.kv, dm.ws)
    torch.cuda.synchronize()
    assert dm.device_error() == SPEC_ERR_DEVICE
    # the context is still usable and the word can be cleared
    lib.spec_clear_device_error(dm.ws)
    tok[1] = 3
    r = lib.make_rows(w.B, w.B, 1, dm.ctx_len, dev(tok), step=0)
    lib.spec_draft_layer(dm.desc, dm.weights, r, dev_act(hid, w), pre, hn, dm.kv, dm.ws)
    torch.cuda.synchronize()
    assert dm.device_error() == 0
    assert torch.isfinite(hn.float()).all()


def test_cache_index_beyond_block_table_sets_error_word():
    w = SMALL_BF16
    W, ctx, kv, dm = setup(w)
    lib.spec_clear_device_error(dm.ws)
    tok = np.array([1, 2, 3], dtype=np.int32)
    # draft-region entry 63 lies past the blocks this request owns
    kv_idx = np.array([0, 63, 0], dtype=np.int32)
    hid = synth.make_hidden(w, w.B)
    pre, hn = dm.hidden(w.B), dm.hidden(w.B)
    r = lib.make_rows(w.B, w.B, 1, dm.ctx_len, dev(tok), step=0, kv_idx=dev(kv_idx))
    lib.spec_draft_layer(dm.desc, dm.weights, r, dev_act(hid, w), pre, hn, dm.kv, dm.ws)
    torch.cuda.synchronize()
    assert dm.device_error() == SPEC_ERR_DEVICE


def test_tree_parent_after_node_sets_error_word():
    B, N, V, D = 1, 4, 4096, 3
    target = torch.zeros(B, N + 1, V, device="cuda")
    tok = torch.zeros(B, N + 1, dtype=torch.int32, device="cuda")
    par = torch.tensor([[-1, 0, 3, 1, 2]], dtype=torch.int32, device="cuda")     # node 2's parent is node 3
    out = torch.zeros(B, D + 1, dtype=torch.int32, device="cuda")
    acc = torch.zeros(B, dtype=torch.int32, device="cuda")
    ws = torch.zeros(lib.spec_verify_workspace_bytes(B, N + 1, V), dtype=torch.uint8, device="cuda")
    lib.spec_verify_greedy(B, N + 1, V, target, tok, out, acc, parent=par, max_depth=D, ws=ws)
    torch.cuda.synchronize()
    assert lib.spec_get_device_error(ws) == SPEC_ERR_DEVICE


SPEC_ERR_TIMEOUT = -7


def _set_verify_knobs(ws, wait_us, withhold):
    """Header bytes 64..71 of a verifier workspace: the bound on a sampling CTA's wait
    (microseconds) and the test hook that keeps request (withhold - 1)'s decision
    unpublished."""
    ws[64:72].copy_(torch.tensor([wait_us, withhold], dtype=torch.int32).view(torch.uint8).cuda())


def test_rejection_wait_runs_out_and_context_stays_usable():
    """A bounded device-side wait that runs out: request 2's decision is never
    published (a flag nothing sets), so its sampling CTAs give up after the 2 ms
    limit, the kernel returns, the error word reads SPEC_ERR_TIMEOUT and that
    request's emitted token is -1; every other request is still right, and the
    next call on the same workspace succeeds."""
    from oracle import verify as overify
    B, K, V = 6, 3, 8192
    target = synth.normal((B, K + 1, V), 5, "noise", 1.5, 0.0, 1)
    drafts = np.argmax(target[:, :K], -1).astype(np.int32)
    drafts[:, 1] = (drafts[:, 1] + 1) % V                    # a likely rejection at position 1
    temp = np.ones(B, dtype=np.float32)
    seed = 99
    ref_out, ref_acc, _ = overify.verify_rejection(target, drafts, temp, seed, 0)
    out = torch.full((B, K + 1), -5, dtype=torch.int32, device="cuda")
    acc = torch.zeros(B, dtype=torch.int32, device="cuda")
    ws = torch.zeros(lib.spec_verify_workspace_bytes(B, K + 1, V), dtype=torch.uint8, device="cuda")
    _set_verify_knobs(ws, 2000, 3)
    lib.spec_verify_rejection(B, K, V, dev(target), dev(drafts), dev(temp), seed, 0, out, acc, ws=ws)
    torch.cuda.synchronize()
    assert lib.spec_get_device_error(ws) == SPEC_ERR_TIMEOUT
    o, a = out.cpu().numpy(), acc.cpu().numpy()
    np.testing.assert_array_equal(a, ref_acc)                # decisions were all made
    assert o[2, a[2]] == -1                                  # the withheld request's sample gave up
    for b in range(B):
        if b != 2:
            np.testing.assert_array_equal(o[b], ref_out[b])
    # the same workspace, knobs and error word cleared: a normal call succeeds
    _set_verify_knobs(ws, 0, 0)
    lib.spec_clear_device_error(ws)
    out.fill_(-5)
    lib.spec_verify_rejection(B, K, V, dev(target), dev(drafts), dev(temp), seed, 0, out, acc, ws=ws)
    torch.cuda.synchronize()
    assert lib.spec_get_device_error(ws) == 0
    np.testing.assert_array_equal(out.cpu().numpy(), ref_out)
    np.testing.assert_array_equal(acc.cpu().numpy(), ref_acc)
