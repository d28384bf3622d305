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
