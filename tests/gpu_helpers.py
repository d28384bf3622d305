"""Shared helpers of the GPU parity tests (test infrastructure)."""
import copy
from dataclasses import replace

import numpy as np
import torch

from eagle_speculative_decoding_step_gb300 import binding as lib
from eagle_speculative_decoding_step_gb300 import configs, engine, synth

# tolerances (stated for bf16 storage by the workload definition; fp32 tighter)
BF16_ATOL, BF16_RTOL = 2e-2, 1e-2
F32_ATOL, F32_RTOL = 1e-5, 1e-4
LOGIT_TIE = 2e-2          # an id may differ from the oracle's only if the oracle logits are this close


def tol(w):
    return (BF16_ATOL, BF16_RTOL) if w.dtype == "bf16" else (F32_ATOL, F32_RTOL)


def assert_close(gpu, ref, w, what=""):
    atol, rtol = tol(w)
    np.testing.assert_allclose(np.asarray(gpu, dtype=np.float64), np.asarray(ref, dtype=np.float64),
                               atol=atol, rtol=rtol, err_msg=what)


def ids_match(gpu_ids, ref_ids, ref_logits, tie=LOGIT_TIE):
    """Token ids equal, except where the oracle's logits of the two ids are within
    `tie` (a near-tie the two precisions may order differently).  Returns the
    number of exempted near-ties."""
    gpu_ids = np.asarray(gpu_ids)
    ref_ids = np.asarray(ref_ids)
    ties = 0
    for idx in zip(*np.nonzero(gpu_ids != ref_ids)):
        row = ref_logits[idx[:-1]] if ref_logits.ndim == gpu_ids.ndim else ref_logits[idx[0]]
        g, r = int(gpu_ids[idx]), int(ref_ids[idx])
        gap = abs(float(row[g]) - float(row[r]))
        assert gap < tie, "id mismatch at %s: gpu %d oracle %d (logit gap %.4g)" % (idx, g, r, gap)
        ties += 1
    return ties


SMALL_BF16 = replace(configs.WORKLOADS["llama8b_chain"], name="small_bf16", H=512, nq=8, nkv=2, hd=64, I=1000,
                     V=3000, B=3, ctx=100, K=3, seed=21)
SMALL_BF16_HD128 = replace(SMALL_BF16, name="small_bf16_hd128", H=384, nq=4, nkv=1, hd=128, I=776, V=2053,
                           seed=22)


def setup(w, max_rows=None):
    W = synth.make_weights(w)
    if w.rank > 0:
        W["lr_down"], W["lr_up"] = synth.lowrank_factors(W["lm_head"], w.rank, w.dtype)
    ctx = synth.context_lengths(w)
    kv = synth.make_kv(w, ctx)
    dm = engine.DeviceModel(w, W, kv, ctx, max_rows=max_rows)
    return W, ctx, kv, dm


def dev(x, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def dev_act(x, w):
    return engine.to_device(np.asarray(x, dtype=np.float32), w.dtype, "cuda")


def host(t):
    return engine.from_device(t)


def kv_host(dm):
    return {"k": host(dm.tkv["k"]), "v": host(dm.tkv["v"]), "block_table": dm.tkv["block_table"].cpu().numpy(),
            "block_size": dm.tkv["block_size"], "max_blocks": dm.tkv["max_blocks"],
            "num_slots": dm.tkv["num_slots"]}


def no_device_error(dm_or_ws):
    ws = dm_or_ws.ws if hasattr(dm_or_ws, "ws") else dm_or_ws
    assert lib.spec_get_device_error(ws) == 0


def tree_mismatch_is_near_tie(got_tok, got_par, fin, got_score=None, tol=2e-2):
    """True if, in every request whose GPU tree differs from the oracle's, the first
    differing node (nodes are numbered depth by depth, best score first, so later
    differences may follow from it) sits next to a node whose oracle score is within
    ``tol``, or where the GPU placed a candidate whose score is within ``tol`` of the
    oracle's node there: two candidates whose ranking the two precisions may swap."""
    got_tok, got_par = np.asarray(got_tok), np.asarray(got_par)
    score = np.asarray(fin["score"], dtype=np.float64)
    diff = (got_tok != fin["tok"]) | (got_par != fin["parent"])
    for b in range(diff.shape[0]):
        if not diff[b].any():
            continue
        n = int(np.argmax(diff[b]))
        near = [abs(score[b, n] - score[b, m]) for m in (n - 1, n + 1) if 1 <= m < score.shape[1]]
        if got_score is not None:
            near.append(abs(float(np.asarray(got_score)[b, n]) - score[b, n]))
        if not near or min(near) >= tol:
            return False
    return True
