"""spec_verify_greedy_static: greedy verification for callers that cannot allocate
device memory (a host framework that owns every buffer, a serving loop where
cudaMalloc's device synchronisation is not allowed, a plugin without an
allocator).  Its scratch is a fixed array inside the library; the results must
equal spec_verify_greedy's (token ids, accept lengths, K/V bytes: exact) on
consecutive calls, whatever ran before in the process.

This file is collected last on purpose: if it fails, every other test has run.
"""
import numpy as np
import pytest
import torch

from eagle_speculative_decoding_step_gb300 import binding as lib
from eagle_speculative_decoding_step_gb300 import configs, engine, synth

pytestmark = pytest.mark.gpu


def _chain(B, K, V, seed):
    g = np.random.default_rng(seed)
    target = synth.normal((B, K + 1, V), seed, "noise", 1.0, 0.0, 1)
    t = np.argmax(target, axis=-1)
    drafts = g.integers(0, V, size=(B, K))
    for b in range(B):
        a = int(g.integers(0, K + 1))
        drafts[b, :a] = t[b, :a]
    return torch.from_numpy(target).cuda(), torch.from_numpy(drafts.astype(np.int32)).cuda()


def _run_chain(fn_static, B, K, V, target, drafts):
    out = torch.full((B, K + 1), -7, dtype=torch.int32, device="cuda")
    acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    src = torch.full((B, K + 1), -7, dtype=torch.int32, device="cuda")
    if fn_static:
        lib.spec_verify_greedy_static(B, K + 1, V, target, drafts, out, acc, src)
    else:
        ws = torch.zeros(lib.spec_verify_workspace_bytes(B, K + 1, V), dtype=torch.uint8, device="cuda")
        lib.spec_verify_greedy(B, K + 1, V, target, drafts, out, acc, src, ws=ws)
    torch.cuda.synchronize()
    return out.cpu(), acc.cpu(), src.cpu()


def test_static_scratch_chain_matches_workspace_version_twice():
    lib.load()
    for (B, K, V, seed) in [(4, 5, 128256, 1), (3, 7, 5003, 2)]:          # two calls in a row
        target, drafts = _chain(B, K, V, seed)
        want = _run_chain(False, B, K, V, target, drafts)
        got = _run_chain(True, B, K, V, target, drafts)
        for a, b in zip(got, want):
            assert torch.equal(a, b)


def test_static_scratch_tree_with_compaction_matches_workspace_version_twice():
    from dataclasses import replace
    w0 = replace(configs.WORKLOADS["llama8b_chain"], name="noalloc_tree", H=256, nq=4, nkv=2, hd=64, I=256,
                 V=4099, B=2, ctx=40, mode="tree", top_k=4, depth=4, total=12, seed=9)
    for call in range(2):
        w = replace(w0, seed=9 + call)
        W = synth.make_weights(w, with_lm_head=False)
        ctx = synth.context_lengths(w)
        kv = synth.make_kv(w, ctx)
        N, D, B, V = w.total, w.depth, w.B, w.V
        g = np.random.default_rng(20 + call)
        target = synth.normal((B, N + 1, V), w.seed, "noise", 1.0, 0.0, 2)
        t = np.argmax(target, axis=-1)
        par = np.zeros((B, N + 1), dtype=np.int32)
        tok = g.integers(0, V, size=(B, N + 1)).astype(np.int32)
        for b in range(B):
            depth = [0]
            par[b, 0] = -1
            for n in range(1, N + 1):
                p = int(g.integers(0, n))
                while depth[p] + 1 > D:
                    p = int(g.integers(0, n))
                par[b, n] = p
                depth.append(depth[p] + 1)
            n = N
            while n != 0:                        # plant an accepted path
                tok[b, n] = t[b, par[b, n]]
                n = par[b, n]
        results = []
        for static in (False, True):
            dm = engine.DeviceModel(w, W, kv, ctx, max_rows=1)
            out = torch.full((B, D + 1), -7, dtype=torch.int32, device="cuda")
            acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
            src = torch.full((B, D + 1), -7, dtype=torch.int32, device="cuda")
            args = (B, N + 1, V, torch.from_numpy(target).cuda(), torch.from_numpy(tok).cuda(), out, acc, src)
            kw = dict(parent=torch.from_numpy(par).cuda(), max_depth=D, desc=dm.desc, kv=dm.kv, ctx_len=dm.ctx_len)
            if static:
                lib.spec_verify_greedy_static(*args, **kw)
            else:
                ws = torch.zeros(lib.spec_verify_workspace_bytes(B, N + 1, V), dtype=torch.uint8, device="cuda")
                lib.spec_verify_greedy(*args, ws=ws, **kw)
            torch.cuda.synchronize()
            results.append((out.cpu(), acc.cpu(), src.cpu(), dm.tkv["k"].cpu(), dm.tkv["v"].cpu()))
        for a, b in zip(results[1], results[0]):
            assert torch.equal(a, b)
        assert int(results[0][1].max()) >= 1


def _greedy_pair(B, R, V, seed):
    g = np.random.default_rng(seed)
    target = torch.randn(B, R, V, generator=torch.Generator().manual_seed(seed)).cuda()
    t = target.argmax(-1).cpu().numpy()
    drafts = g.integers(0, V, size=(B, R - 1))
    for b in range(B):
        a = int(g.integers(0, R))
        drafts[b, :a] = t[b, :a]
    return target, torch.from_numpy(drafts.astype(np.int32)).cuda()


def test_static_scratch_at_its_capacity_edge():
    """The largest batch whose scratch fits the array runs and matches the workspace
    version; one request more is refused with SPEC_ERR_CAPACITY, and nothing is
    launched (outputs untouched)."""
    cap = lib.spec_verify_greedy_static_capacity()
    R, V = 8, 1024
    B = 1
    while lib.spec_verify_greedy_static_bytes(B + 1, R, V) <= cap:
        B += 1
    assert lib.spec_verify_greedy_static_bytes(B + 1, R, V) > cap
    target, drafts = _greedy_pair(B + 1, R, V, 5)
    want = _run_chain(False, B, R - 1, V, target[:B].contiguous(), drafts[:B].contiguous())
    got = _run_chain(True, B, R - 1, V, target[:B].contiguous(), drafts[:B].contiguous())
    for a, b in zip(got, want):
        assert torch.equal(a, b)
    out = torch.full((B + 1, R), -7, dtype=torch.int32, device="cuda")
    acc = torch.full((B + 1,), -7, dtype=torch.int32, device="cuda")
    with pytest.raises(lib.SpecError) as e:
        lib.spec_verify_greedy_static(B + 1, R, V, target, drafts, out, acc)
    assert e.value.status == -4
    torch.cuda.synchronize()
    assert int(out.min()) == -7 and int(out.max()) == -7 and int(acc.max()) == -7


def test_static_scratch_rejects_oversized_request_without_launch():
    """Real, correctly sized device buffers whose scratch need exceeds the array:
    refused with SPEC_ERR_CAPACITY before any launch."""
    B, R, V = 1000, 40, 16
    assert lib.spec_verify_greedy_static_bytes(B, R, V) > lib.spec_verify_greedy_static_capacity()
    target, drafts = _greedy_pair(B, R, V, 3)
    out = torch.full((B, R), -7, dtype=torch.int32, device="cuda")
    acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    with pytest.raises(lib.SpecError) as e:
        lib.spec_verify_greedy_static(B, R, V, target, drafts, out, acc)
    assert e.value.status == -4
    torch.cuda.synchronize()
    assert int(out.max()) == -7 and int(acc.max()) == -7


def test_static_scratch_error_word_is_readable():
    """A tree whose node 2 names node 3 as its parent (a parent must precede its
    node) sets the array's error word to SPEC_ERR_DEVICE; the next valid call
    clears it."""
    B, N, V = 1, 4, 512
    target = torch.randn(B, N + 1, V, generator=torch.Generator().manual_seed(4)).cuda()
    tok = torch.zeros(B, N + 1, dtype=torch.int32, device="cuda")
    par = torch.tensor([[-1, 0, 3, 0, 1]], dtype=torch.int32, device="cuda")
    out = torch.zeros(B, 4, dtype=torch.int32, device="cuda")
    acc = torch.zeros(B, dtype=torch.int32, device="cuda")
    lib.spec_verify_greedy_static(B, N + 1, V, target, tok, out, acc, parent=par, max_depth=3)
    assert lib.spec_verify_greedy_static_error() == -6
    par_ok = torch.tensor([[-1, 0, 0, 1, 2]], dtype=torch.int32, device="cuda")
    lib.spec_verify_greedy_static(B, N + 1, V, target, tok, out, acc, parent=par_ok, max_depth=3)
    assert lib.spec_verify_greedy_static_error() == 0
