"""GPU parity of the verifiers (spec_verify_greedy, spec_verify_rejection) against the oracle."""
import copy
from dataclasses import replace

import numpy as np
import pytest
import torch

from eagle_speculative_decoding_step_gb300 import binding as lib
from eagle_speculative_decoding_step_gb300 import synth
from oracle import verify, draft as odraft
from gpu_helpers import dev, setup, kv_host, SMALL_BF16, no_device_error

pytestmark = pytest.mark.gpu


def _chain_inputs(B, K, V, seed, plant):
    """Random target logits; drafts equal to the target argmax for a planted prefix
    length per request, random afterwards."""
    g = np.random.default_rng(seed)
    target = synth.normal((B, K + 1, V), seed, "noise", 1.0, 0.0, 7)
    t = np.argmax(target, axis=-1)
    drafts = g.integers(0, V, size=(B, K))
    for b in range(B):
        a = plant[b % len(plant)]
        drafts[b, :a] = t[b, :a]
    return target, drafts.astype(np.int32)


@pytest.mark.parametrize("B,K,V", [(1, 1, 7), (3, 5, 5003), (4, 5, 128256), (32, 7, 151936)])
def test_verify_greedy_chain(B, K, V):
    target, drafts = _chain_inputs(B, K, V, seed=B * 31 + K, plant=[0, K, 2, 1, K - 1])
    ref_out, ref_acc, ref_src = verify.verify_greedy_chain(target, drafts)
    out = torch.zeros(B, K + 1, dtype=torch.int32, device="cuda")
    acc = torch.zeros(B, dtype=torch.int32, device="cuda")
    src = torch.zeros(B, K + 1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(lib.spec_verify_workspace_bytes(B, K + 1, V), dtype=torch.uint8, device="cuda")
    lib.spec_verify_greedy(B, K + 1, V, dev(target), dev(drafts), out, acc, src, ws=ws)
    np.testing.assert_array_equal(out.cpu().numpy(), ref_out)
    np.testing.assert_array_equal(acc.cpu().numpy(), ref_acc)
    np.testing.assert_array_equal(src.cpu().numpy(), ref_src)


def test_verify_greedy_chain_ties_and_empty_accept():
    """Rows with exact ties at the maximum (smaller id wins) and all-equal rows."""
    B, K, V = 2, 3, 4096
    target = np.zeros((B, K + 1, V), dtype=np.float32)
    target[0, 0, [17, 900, 4000]] = 5.0          # tie: 17 wins
    target[0, 1, 3] = 1.0
    target[1, :, :] = -1.0                       # all equal: id 0
    drafts = np.array([[17, 3, 9], [0, 0, 1]], dtype=np.int32)
    ref_out, ref_acc, _ = verify.verify_greedy_chain(target, drafts)
    out = torch.zeros(B, K + 1, dtype=torch.int32, device="cuda")
    acc = torch.zeros(B, dtype=torch.int32, device="cuda")
    ws = torch.zeros(lib.spec_verify_workspace_bytes(B, K + 1, V), dtype=torch.uint8, device="cuda")
    lib.spec_verify_greedy(B, K + 1, V, dev(target), dev(drafts), out, acc, ws=ws)
    np.testing.assert_array_equal(out.cpu().numpy(), ref_out)
    np.testing.assert_array_equal(acc.cpu().numpy(), ref_acc)


def _random_tree(N, seed):
    g = np.random.default_rng(seed)
    parent = [-1] + [int(g.integers(0, n)) for n in range(1, N + 1)]
    return np.array(parent, dtype=np.int32)


@pytest.mark.parametrize("B,N,V,D", [(1, 31, 151936, 5), (3, 12, 4099, 8)])
def test_verify_greedy_tree_and_compaction(B, N, V, D):
    w = replace(SMALL_BF16, B=B, mode="tree", top_k=4, depth=D, total=N)
    W, ctx, kv0, dm = setup(w)
    g = np.random.default_rng(5)
    target = synth.normal((B, N + 1, V), 9, "noise", 1.0, 0.0, 3)
    t = np.argmax(target, axis=-1)
    tok = np.zeros((B, N + 1), dtype=np.int32)
    par = np.zeros((B, N + 1), dtype=np.int32)
    for b in range(B):
        p = _random_tree(N, 100 + b)
        depth = np.zeros(N + 1, dtype=int)
        for n in range(1, N + 1):
            depth[n] = depth[p[n]] + 1
        # keep depth <= D by re-parenting deep nodes to the root
        for n in range(1, N + 1):
            if depth[p[n]] + 1 > D:
                p[n] = 0
            depth[n] = depth[p[n]] + 1
        par[b] = p
        tok[b] = g.integers(0, V, size=N + 1)
        # plant matches along one random path so something deep gets accepted
        n = int(g.integers(1, N + 1))
        while n != 0:
            tok[b, n] = t[b, p[n]]
            n = p[n]
    ref_out, ref_acc, ref_src = verify.verify_greedy_tree(target, tok, par, D)
    out = torch.zeros(B, D + 1, dtype=torch.int32, device="cuda")
    acc = torch.zeros(B, dtype=torch.int32, device="cuda")
    src = torch.zeros(B, D + 1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(lib.spec_verify_workspace_bytes(B, N + 1, V), dtype=torch.uint8, device="cuda")
    lib.spec_verify_greedy(B, N + 1, V, dev(target), dev(tok), out, acc, src, parent=dev(par), max_depth=D,
                           desc=dm.desc, kv=dm.kv, ctx_len=dm.ctx_len, ws=ws)
    np.testing.assert_array_equal(out.cpu().numpy(), ref_out)
    np.testing.assert_array_equal(acc.cpu().numpy(), ref_acc)
    np.testing.assert_array_equal(src.cpu().numpy(), ref_src)
    assert ref_acc.max() >= 1
    kv_ref = copy.deepcopy(kv0)
    verify.compact_kv(kv_ref, ctx, ref_src, ref_acc)
    got = kv_host(dm)
    np.testing.assert_array_equal(got["k"], kv_ref["k"])
    np.testing.assert_array_equal(got["v"], kv_ref["v"])
    no_device_error(ws)


@pytest.mark.parametrize("B,K,V,T", [(4, 3, 4096, 1.0), (32, 7, 151936, 1.0), (5, 2, 1001, 0.6)])
def test_verify_rejection(B, K, V, T):
    g = np.random.default_rng(B + K)
    target = synth.normal((B, K + 1, V), 11, "noise", 1.5, 0.0, B)
    # drafts: argmax of the row (likely accepted) or a random token
    drafts = np.where(g.random((B, K)) < 0.7, np.argmax(target[:, :K], -1), g.integers(0, V, (B, K)))
    drafts = drafts.astype(np.int32)
    temp = np.full(B, T, dtype=np.float32)
    temp[1] = 0.0                                   # one greedy request in the batch
    seed, so = 1003, 7
    ref_out, ref_acc, info = verify.verify_rejection(target, drafts, temp, seed, so)
    out = torch.zeros(B, K + 1, dtype=torch.int32, device="cuda")
    acc = torch.zeros(B, dtype=torch.int32, device="cuda")
    ws = torch.zeros(lib.spec_verify_workspace_bytes(B, K + 1, V), dtype=torch.uint8, device="cuda")
    lib.spec_verify_rejection(B, K, V, dev(target), dev(drafts), dev(temp), seed, so, out, acc, ws=ws)
    out, acc = out.cpu().numpy(), acc.cpu().numpy()
    near = 0
    for b in range(B):
        if np.array_equal(out[b], ref_out[b]) and acc[b] == ref_acc[b]:
            continue
        # only a decision within float32 reach of its threshold may differ
        m = np.abs(info["accept_margin"][b])
        assert (m < 1e-5).any() or info["sample_gap"][b] < 1e-4, "request %d differs" % b
        near += 1
    assert near <= max(1, B // 16)
    assert (ref_acc > 0).any() and (ref_acc < K).any()


@pytest.mark.parametrize("B,K,V", [(16, 3, 4096), (8, 7, 151936)])
def test_verify_rejection_top_k_top_p(B, K, V):
    """Per-request top-k / top-p (mixed with greedy and unfiltered requests)."""
    g = np.random.default_rng(B * 7 + K)
    target = synth.normal((B, K + 1, V), 13, "noise", 2.0, 0.0, B)
    drafts = np.where(g.random((B, K)) < 0.8, np.argmax(target[:, :K], -1), g.integers(0, V, (B, K)))
    drafts = drafts.astype(np.int32)
    temp = np.full(B, 1.0, dtype=np.float32)
    temp[1] = 0.0
    temp[2] = 0.7
    top_k = np.array([[0, 5, 40, 1, 0, 200][b % 6] for b in range(B)], dtype=np.int32)
    top_p = np.array([[1.0, 1.0, 0.9, 1.0, 0.5, 0.95][b % 6] for b in range(B)], dtype=np.float32)
    seed, so = 77, 3
    ref_out, ref_acc, info = verify.verify_rejection(target, drafts, temp, seed, so, top_k=top_k,
                                                     top_p=top_p.astype(np.float64))
    out = torch.zeros(B, K + 1, dtype=torch.int32, device="cuda")
    acc = torch.zeros(B, dtype=torch.int32, device="cuda")
    ws = torch.zeros(lib.spec_verify_workspace_bytes(B, K + 1, V), dtype=torch.uint8, device="cuda")
    lib.spec_verify_rejection(B, K, V, dev(target), dev(drafts), dev(temp), seed, so, out, acc, ws=ws,
                              top_k=dev(top_k), top_p=dev(top_p))
    out, acc = out.cpu().numpy(), acc.cpu().numpy()
    near = 0
    for b in range(B):
        if np.array_equal(out[b], ref_out[b]) and acc[b] == ref_acc[b]:
            continue
        m = np.abs(info["accept_margin"][b])
        assert (m < 1e-5).any() or info["sample_gap"][b] < 1e-4 or info["top_p_margin"][b] < 1e-5, \
            "request %d differs: %s vs %s" % (b, out[b], ref_out[b])
        near += 1
    assert near <= max(1, B // 8)
    # filtered requests never emit a token outside their kept set
    for b in range(B):
        if temp[b] <= 0:
            continue
        a = acc[b]
        row = target[b, a].astype(np.float64) / temp[b]
        kept, _ = verify.kept_set(row, top_k[b], float(top_p[b]))
        assert kept[out[b, a]]


def test_verifiers_reuse_their_workspace():
    """Each verifier is one launch whose completion counters return to zero: calls
    in a row on one workspace (alternating greedy and rejection, different batch
    sizes within it) all match the oracle."""
    B, K, V = 9, 4, 20000
    ws = torch.zeros(lib.spec_verify_workspace_bytes(B, K + 1, V), dtype=torch.uint8, device="cuda")
    for call in range(4):
        b = B - call
        target, drafts = _chain_inputs(b, K, V, seed=40 + call, plant=[0, K, 2, 1])
        out = torch.zeros(b, K + 1, dtype=torch.int32, device="cuda")
        acc = torch.zeros(b, dtype=torch.int32, device="cuda")
        if call % 2 == 0:
            ref_out, ref_acc, _ = verify.verify_greedy_chain(target, drafts)
            lib.spec_verify_greedy(b, K + 1, V, dev(target), dev(drafts), out, acc, ws=ws)
        else:
            temp = np.full(b, 0.8, dtype=np.float32)
            ref_out, ref_acc, info = verify.verify_rejection(target, drafts, temp, 5, call)
            lib.spec_verify_rejection(b, K, V, dev(target), dev(drafts), dev(temp), 5, call, out, acc, ws=ws)
        torch.cuda.synchronize()
        got_out, got_acc = out.cpu().numpy(), acc.cpu().numpy()
        for r in range(b):
            if not (np.array_equal(got_out[r], ref_out[r]) and got_acc[r] == ref_acc[r]):
                assert call % 2 == 1 and ((np.abs(info["accept_margin"][r]) < 1e-5).any()
                                          or info["sample_gap"][r] < 1e-4), "call %d request %d" % (call, r)
        assert lib.spec_get_device_error(ws) == 0
