"""Pins of the CPU oracle against facts the source pages and mathematics fix.

None of these compares the oracle with itself: each checks it against a
closed form, a library routine, a published known answer, brute force, a
hand-worked case, or an invariant a plausible mistake would break.
"""
import copy
import json
import os
from dataclasses import replace

import numpy as np
import pytest
import scipy.special
import scipy.stats
import torch

import oracle
from oracle import draft, numerics, philox, step, tree, verify
from eagle_speculative_decoding_step_gb300 import configs, synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

TINY = configs.WORKLOADS["tiny"]
MICRO = replace(TINY, name="micro", H=64, nq=4, nkv=2, hd=16, I=96, V=64, B=2, ctx=20, K=4)


def _setup(w):
    W = synth.make_weights(w)
    ctx = synth.context_lengths(w)
    kv = synth.make_kv(w, ctx)
    return W, ctx, kv


# ---------------------------------------------------------------- Philox
def test_philox_known_answers():
    """Known-answer vectors published with Philox4x32-10 by its authors
    (Salmon et al., SC'11, Random123 distribution)."""
    F = 0xFFFFFFFF
    cases = [
        ((0, 0, 0, 0, 0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
        ((F, F, F, F, F, F), (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
        ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344, 0xA4093822, 0x299F31D0),
         (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
    ]
    for args, want in cases:
        got = tuple(int(x) for x in philox.philox4x32_10(*args))
        assert got == want


def test_philox_uniforms_are_uniform():
    u = philox.noise_uniforms(1234, 0, 3, 2, 200000)
    assert np.all((u > 0) & (u < 1))
    hist, _ = np.histogram(u, bins=50, range=(0, 1))
    assert scipy.stats.chisquare(hist).pvalue > 1e-3
    # successive draws not correlated
    assert abs(np.corrcoef(u[:-1], u[1:])[0, 1]) < 0.01


# ---------------------------------------------------------------- numerics
def test_bf16_rounding_matches_torch():
    x = np.random.default_rng(5).standard_normal(100000) * np.exp(np.random.default_rng(6).uniform(-20, 20, 100000))
    want = torch.tensor(x, dtype=torch.float64).to(torch.bfloat16).to(torch.float64).numpy()
    # torch rounds float64 -> bfloat16 via float32 (double rounding); compare on values
    # exactly representable in float32 so both are single roundings
    x32 = x.astype(np.float32).astype(np.float64)
    want = torch.tensor(x32, dtype=torch.float64).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(numerics.to_bf16(x32), want)


def test_rope_properties():
    rng = np.random.default_rng(0)
    q = rng.standard_normal((5, 64))
    k = rng.standard_normal((5, 64))
    # norm preserved
    np.testing.assert_allclose(np.linalg.norm(numerics.rope(q, np.arange(5) * 37, 1e4), axis=-1),
                               np.linalg.norm(q, axis=-1), rtol=1e-12)
    # dot product depends on the position difference only
    a = numerics.rope(q, 100, 1e4) @ numerics.rope(k, 90, 1e4).T
    b = numerics.rope(q, 2000, 1e4) @ numerics.rope(k, 1990, 1e4).T
    np.testing.assert_allclose(a, b, rtol=1e-9, atol=1e-9)
    # complex-number statement: pairs (i, i + d/2) rotate by pos * theta^(-2i/d)
    pos = 7
    zc = (q[:, :32] + 1j * q[:, 32:]) * np.exp(1j * pos * 1e4 ** (-2 * np.arange(32) / 64))
    got = numerics.rope(q, pos, 1e4)
    np.testing.assert_allclose(got[:, :32], zc.real, atol=1e-12)
    np.testing.assert_allclose(got[:, 32:], zc.imag, atol=1e-12)


def test_rmsnorm_and_lse_against_torch_scipy():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((4, 33))
    g = rng.standard_normal(33)
    want = torch.nn.functional.rms_norm(torch.tensor(x), (33,), torch.tensor(g), eps=1e-6).numpy()
    np.testing.assert_allclose(numerics.rmsnorm(x, g, 1e-6), want, rtol=1e-12)
    y = rng.standard_normal((3, 1000)) * 30
    np.testing.assert_allclose(numerics.logsumexp(y), scipy.special.logsumexp(y, axis=-1), rtol=1e-13)


def test_topk_tie_break():
    v = np.array([[1.0, 3.0, 3.0, 2.0, 3.0]])
    assert numerics.topk_desc(v, 4).tolist() == [[1, 2, 4, 3]]


# ---------------------------------------------------------------- attention
def _attention_case(w, seed):
    W, ctx, kv = _setup(w)
    rng = np.random.default_rng(seed)
    M = w.B
    q = rng.standard_normal((M, w.nq, w.hd))
    req = np.arange(M)
    c = ctx.astype(np.int64)
    pos = c + 2
    mask = [0b101, 0b111][:M] + [1] * (M - 2)
    return q, kv, req, c, pos, mask


def test_attention_matches_torch_sdpa():
    w = replace(MICRO, window=0)
    q, kv, req, c, pos, mask = _attention_case(w, 3)
    got = draft.attention(w, q, kv, req, c, pos, mask)
    for m in range(len(req)):
        n_ctx = int(c[m]) + 8
        idx = np.arange(n_ctx)
        slots = draft.slot_of(kv, m, idx)
        K = torch.tensor(kv["k"][slots], dtype=torch.float64).permute(1, 0, 2)   # [nkv, n, hd]
        V = torch.tensor(kv["v"][slots], dtype=torch.float64).permute(1, 0, 2)
        allowed = np.zeros(n_ctx, dtype=bool)
        allowed[:c[m]] = True
        for i in range(8):
            if mask[m] >> i & 1:
                allowed[c[m] + i] = True
        Q = torch.tensor(q[m], dtype=torch.float64)[:, None, :]                   # [nq, 1, hd]
        Krep = K.repeat_interleave(w.nq // w.nkv, dim=0)
        Vrep = V.repeat_interleave(w.nq // w.nkv, dim=0)
        am = torch.tensor(allowed)[None, None, :].expand(w.nq, 1, n_ctx)
        want = torch.nn.functional.scaled_dot_product_attention(Q, Krep, Vrep, attn_mask=am)
        np.testing.assert_allclose(got[m], want[:, 0, :].numpy(), rtol=1e-10, atol=1e-12)


def test_attention_window_and_causal_reductions():
    w = MICRO
    q, kv, req, c, pos, mask = _attention_case(w, 4)
    full = draft.attention(replace(w, window=0), q, kv, req, c, pos, mask)
    wide = draft.attention(replace(w, window=int(pos.max()) + 64), q, kv, req, c, pos, mask)
    np.testing.assert_allclose(full, wide, rtol=0, atol=0)
    # a window of W keeps exactly W keys ending at the row itself: check with q = 0
    # (uniform weights -> mean of the allowed values)
    W_ = 6
    wq = replace(w, window=W_)
    z = np.zeros_like(q)
    pos1 = c.copy()                         # row at position ctx, mask = itself only
    got = draft.attention(wq, z, kv, req, c, pos1, [1] * len(req))
    for m in range(len(req)):
        keys = list(range(int(pos1[m]) - W_ + 1, int(c[m]))) + [int(c[m])]
        assert len(keys) == W_
        V = kv["v"][draft.slot_of(kv, m, np.array(keys))].astype(np.float64)
        for h in range(w.nq):
            np.testing.assert_allclose(got[m, h], V[:, h // (w.nq // w.nkv)].mean(0), rtol=1e-12)


def test_slot_mapping_formula():
    w = MICRO
    _, ctx, kv = _setup(w)
    bs = kv["block_size"]
    for b in range(w.B):
        for p in [0, 1, bs - 1, bs, int(ctx[b]) + 3]:
            assert draft.slot_of(kv, b, p) == kv["block_table"][b, p // bs] * bs + p % bs


# ---------------------------------------------------------------- draft layer
def test_draft_layer_residual_closed_form():
    """With o_proj and down_proj zero, the layer passes its hidden input through
    (hidden_prenorm == hid) and the normed output is RMSNorm_final(hid)."""
    w = MICRO
    W, ctx, kv = _setup(w)
    W["wo"] = np.zeros_like(W["wo"])
    W["wdown"] = np.zeros_like(W["wdown"])
    hid = synth.make_hidden(w, w.B).astype(np.float64)
    rows = {"M": w.B, "B": w.B, "R": 1, "step": 0, "ctx_len": ctx, "tok": [1, 2]}
    pre, hn = draft.draft_layer(w, W, rows, hid, kv)
    np.testing.assert_allclose(pre, hid, rtol=0, atol=0)
    np.testing.assert_allclose(hn, numerics.rmsnorm(hid, W["final_norm"], w.rms_eps), rtol=1e-12)


def test_draft_layer_uniform_attention_closed_form():
    """With q and k projections zero, every allowed key gets the same weight, so the
    attention output is the mean of the allowed values (context + own row)."""
    w = replace(MICRO, B=1)
    W, ctx, kv = _setup(w)
    W["wq"] = np.zeros_like(W["wq"])
    W["wk"] = np.zeros_like(W["wk"])
    W["wdown"] = np.zeros_like(W["wdown"])
    W["wo"] = np.eye(w.H, w.nq * w.hd)          # o_proj copies the attention output
    hid = np.zeros((1, w.H))
    rows = {"M": 1, "B": 1, "R": 1, "step": 0, "ctx_len": ctx, "tok": [5]}
    kv2 = copy.deepcopy(kv)
    pre, _ = draft.draft_layer(w, W, rows, hid, kv2)
    c = int(ctx[0])
    V = kv2["v"][draft.slot_of(kv2, 0, np.arange(c + 1))].astype(np.float64)   # [c+1, nkv, hd]
    grp = w.nq // w.nkv
    want = np.concatenate([V[:, h // grp].mean(0) for h in range(w.nq)])
    np.testing.assert_allclose(pre[0], want[:w.H], rtol=1e-12, atol=1e-14)
    # the row's own value was written at cache index ctx (= position of step 0)
    e = numerics.rmsnorm(W["embed"][5], W["in_norm"], w.rms_eps)
    g = numerics.rmsnorm(hid, W["hidden_norm"], w.rms_eps)[0]
    x = np.concatenate([e, g])
    # the cache stores the workload's dtype (float32 here)
    np.testing.assert_allclose(V[c].reshape(-1), x @ W["wv"].astype(np.float64).T, rtol=1e-6)


def test_draft_layer_matches_torch_functional():
    """The layer restated with torch.nn.functional primitives, following the
    decoder-layer pseudo-code of the Neuron design page step by step."""
    w = replace(MICRO, dtype="f32")
    W, ctx, kv = _setup(w)
    hid = synth.make_hidden(w, w.B).astype(np.float64)
    tok = [3, 60]
    rows = {"M": w.B, "B": w.B, "R": 1, "step": 1, "ctx_len": ctx, "tok": tok}
    kv_o = copy.deepcopy(kv)
    pre, hn = draft.draft_layer(w, W, rows, hid, kv_o)

    T = {k: torch.tensor(np.asarray(v, dtype=np.float64)) for k, v in W.items()}
    F = torch.nn.functional
    H = w.H
    for m in range(w.B):
        h = torch.tensor(hid[m:m + 1])
        emb = F.embedding(torch.tensor([tok[m]]), T["embed"])
        x = torch.cat([F.rms_norm(emb, (H,), T["in_norm"], eps=w.rms_eps),
                       F.rms_norm(h, (H,), T["hidden_norm"], eps=w.rms_eps)], dim=-1)
        q = F.linear(x, T["wq"]).view(w.nq, w.hd)
        k = F.linear(x, T["wk"]).view(w.nkv, w.hd)
        v = F.linear(x, T["wv"]).view(w.nkv, w.hd)
        p = int(ctx[m]) + 1
        inv = 1.0 / (w.rope_theta ** (torch.arange(0, w.hd, 2, dtype=torch.float64) / w.hd))
        ang = p * inv
        cos = torch.cat([torch.cos(ang), torch.cos(ang)])
        sin = torch.cat([torch.sin(ang), torch.sin(ang)])

        def rot(t):
            return torch.cat([-t[..., w.hd // 2:], t[..., :w.hd // 2]], dim=-1)
        q = q * cos + rot(q) * sin
        k = k * cos + rot(k) * sin
        c = int(ctx[m])
        idx = np.arange(c + 2)                      # context + draft entries 0, 1 (step 1)
        slots = draft.slot_of(kv, m, idx)
        Kc = torch.tensor(kv["k"][slots], dtype=torch.float64)
        Vc = torch.tensor(kv["v"][slots], dtype=torch.float64)
        # entry 0 of the draft region was written by step 0 in a real chain; here it
        # holds the generator's value, entry 1 is this row's own K/V
        Kc[-1] = k.float().double()                 # the cache stores float32
        Vc[-1] = v.float().double()
        grp = w.nq // w.nkv
        att = F.scaled_dot_product_attention(
            q[:, None, :], Kc.permute(1, 0, 2).repeat_interleave(grp, 0),
            Vc.permute(1, 0, 2).repeat_interleave(grp, 0))[:, 0, :].reshape(1, -1)
        out = h + F.linear(att, T["wo"])
        n = F.rms_norm(out, (H,), T["post_norm"], eps=w.rms_eps)
        out = out + F.linear(F.silu(F.linear(n, T["wgate"])) * F.linear(n, T["wup"]), T["wdown"])
        np.testing.assert_allclose(pre[m], out[0].numpy(), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(hn[m], F.rms_norm(out, (H,), T["final_norm"], eps=w.rms_eps)[0].numpy(),
                                   rtol=1e-10, atol=1e-12)


def test_lm_head_statistics():
    w = replace(MICRO, dtype="f32")
    W, _, _ = _setup(w)
    hn = synth.make_hidden(w, 3).astype(np.float64)
    ids, lp, lse, logits = draft.lm_head(w, W, hn, 5)
    np.testing.assert_allclose(lse, scipy.special.logsumexp(hn @ W["lm_head"].astype(np.float64).T, axis=-1),
                               rtol=1e-13)
    assert np.all(lp <= 0)
    np.testing.assert_allclose(np.exp(scipy.special.log_softmax(logits, axis=-1)).sum(-1), 1.0)
    np.testing.assert_array_equal(ids[:, 0], np.argmax(logits, axis=-1))
    assert np.all(np.diff(lp, axis=-1) <= 0)


# ---------------------------------------------------------------- low-rank head
def test_lowrank_full_rank_reproduces_full_head():
    """rank = H: exact factors (numpy SVD) make the low-rank scores equal the full
    logits, so the candidates contain the full head's top-K and the rescored
    argmax is the full head's argmax; num_candidates = V is the full head."""
    w = replace(MICRO, dtype="f32", rank=MICRO.H, num_candidates=8)
    W, _, _ = _setup(w)
    U, S, Vt = np.linalg.svd(W["lm_head"].astype(np.float64), full_matrices=False)
    W["lr_up"] = U * np.sqrt(S)
    W["lr_down"] = np.sqrt(S)[:, None] * Vt
    hn = synth.make_hidden(w, 4).astype(np.float64)
    ids_full, _, _, logits = draft.lm_head(w, W, hn, 8)
    cand, exact, out = draft.lowrank_candidates(w, W, hn, 8, 3)
    for m in range(4):
        assert set(cand[m].tolist()) == set(ids_full[m].tolist())
        np.testing.assert_allclose(exact[m], logits[m, cand[m]], rtol=1e-12)
    np.testing.assert_array_equal(out[:, 0], ids_full[:, 0])
    _, _, out_all = draft.lowrank_candidates(replace(w, num_candidates=w.V), W, hn, w.V, 8)
    np.testing.assert_array_equal(out_all, ids_full)


def test_lowrank_truncated_svd_factors():
    """The generator's factors are the truncated SVD: their product equals the
    best rank-r approximation numpy's SVD gives."""
    rng = np.random.default_rng(2)
    A = (rng.standard_normal((300, 40)) * 0.02).astype(np.float32)
    down, up = synth.lowrank_factors(A, 10, "f32")
    U, S, Vt = np.linalg.svd(A.astype(np.float64), full_matrices=False)
    best = (U[:, :10] * S[:10]) @ Vt[:10]
    np.testing.assert_allclose(up.astype(np.float64) @ down.astype(np.float64), best, atol=2e-6)


# ---------------------------------------------------------------- tree
def _tree_run(w, k, D, N):
    w = replace(w, mode="tree", top_k=k, depth=D, total=N)
    W, ctx, kv = _setup(w)
    aux = synth.make_aux(w)
    root = synth.root_tokens(w)
    trace = []
    fin = step.tree_draft(w, W, aux, root, ctx, kv, k, D, N, trace=trace)
    return fin, trace, (W, ctx, kv, aux, root)


def test_tree_structure_invariants():
    w = replace(MICRO, B=2)
    k, D, N = 4, 4, 12
    fin, trace, _ = _tree_run(w, k, D, N)
    assert len(trace) == D
    for b in range(w.B):
        par = fin["parent"][b]
        assert par[0] == -1 and len(par) == N + 1
        for n in range(1, N + 1):
            assert 0 <= par[n] < n
            assert fin["depth"][b, n] == fin["depth"][b, par[n]] + 1
            assert fin["score"][b, n] <= fin["score"][b, par[n]]
            # mask = own bit | ancestors
            mset = {i for i in range(64) if fin["mask"][b][n] >> i & 1}
            anc = {n}
            p = n
            while p != 0:
                p = par[p]
                anc.add(p)
            assert mset == anc
        # siblings carry distinct tokens
        for n in range(1, N + 1):
            for m in range(n + 1, N + 1):
                if par[n] == par[m]:
                    assert fin["tok"][b, n] != fin["tok"][b, m]
        # BFS order: depth non-decreasing
        assert np.all(np.diff(fin["depth"][b]) >= 0)


def test_tree_selection_brute_force():
    """The final tree is the best N nodes by cumulative log-prob among all
    nodes ever generated (pool), checked by enumerating the pool from the trace."""
    w = replace(MICRO, B=1)
    k, D, N = 3, 3, 7
    fin, trace, _ = _tree_run(w, k, D, N)
    # rebuild the pool scores independently from the per-pass top-k in float32
    pool = []   # (score, token, parent pool id)
    rows_prev = None
    frontier_scores = [np.float32(0.0)]
    frontier_ids = [-1]
    for d, (rows, hid_in, ids, lp) in enumerate(trace, start=1):
        cands = []
        for f in range(len(frontier_ids)):
            for j in range(k):
                sc = np.float32(frontier_scores[f] + np.float32(lp[f, j]))
                cands.append((sc, int(ids[f, j]), frontier_ids[f]))
        base = len(pool)
        pool.extend(cands)
        order = sorted(range(len(cands)), key=lambda i: (-cands[i][0], i))[:k]
        frontier_ids = [base + i for i in order]
        frontier_scores = [cands[i][0] for i in order]
    best = sorted(range(len(pool)), key=lambda i: (-pool[i][0], i))[:N]
    got = sorted(fin["score"][0, 1:].tolist(), reverse=True)
    want = sorted([float(pool[i][0]) for i in best], reverse=True)
    assert got == want
    assert sorted(fin["tok"][0, 1:].tolist()) == sorted(pool[i][1] for i in best)


def test_tree_top1_reduces_to_chain():
    w = replace(MICRO, B=2)
    D = 4
    fin, _, (W, ctx, kv0, aux, root) = _tree_run(w, 1, D, D)
    W2, ctx2, kv2 = _setup(replace(w, mode="tree", top_k=1, depth=D, total=D))
    drafts = step.chain_draft(w, W2, aux, root, ctx2, kv2, D)
    np.testing.assert_array_equal(fin["tok"][:, 1:], drafts)


# ---------------------------------------------------------------- greedy verify
def _onehot_rows(argmax, V):
    r = np.zeros((len(argmax), V), dtype=np.float32)
    r[np.arange(len(argmax)), argmax] = 1.0
    return r


def test_verify_greedy_golden():
    g = json.load(open(os.path.join(GOLDEN, "verify_greedy_cases.json")))
    for c in g["chain"]:
        tgt = _onehot_rows(c["argmax"], g["V"])[None]
        out, acc, kv_src = verify.verify_greedy_chain(tgt, [c["drafts"]])
        assert out[0].tolist() == c["out"], c["name"]
        assert int(acc[0]) == c["accept_len"]
        assert kv_src[0].tolist() == [i if i <= c["accept_len"] else -1 for i in range(len(c["out"]))]
    t = g["chain_tie"]
    for c in t["cases"]:
        out, acc, _ = verify.verify_greedy_chain(np.array(t["rows"], dtype=np.float32)[None], [c["drafts"]])
        assert out[0].tolist() == c["out"] and int(acc[0]) == c["accept_len"]
    tr = g["tree"]
    tgt = _onehot_rows(tr["argmax"], tr["V"])[None]
    out, acc, kv_src = verify.verify_greedy_tree(tgt, [tr["tok"]], [tr["parent"]], tr["max_depth"])
    assert out[0].tolist() == tr["out"]
    assert int(acc[0]) == tr["accept_len"]
    assert kv_src[0].tolist() == tr["kv_src"]


def test_compact_kv_moves_path():
    w = replace(MICRO, B=1)
    _, ctx, kv = _setup(w)
    before = copy.deepcopy(kv)
    kv_src = np.array([[0, 5, 7, -1]])
    verify.compact_kv(kv, ctx, kv_src, [2])
    c = int(ctx[0])
    for d, n in [(1, 5), (2, 7)]:
        np.testing.assert_array_equal(kv["k"][draft.slot_of(kv, 0, c + d)], before["k"][draft.slot_of(kv, 0, c + n)])
        np.testing.assert_array_equal(kv["v"][draft.slot_of(kv, 0, c + d)], before["v"][draft.slot_of(kv, 0, c + n)])
    # the context and the root entry are untouched
    idx = draft.slot_of(kv, 0, np.arange(c + 1))
    np.testing.assert_array_equal(kv["k"][idx], before["k"][idx])


class _TinyTarget:
    """A small causal Llama-like target model (test-only), float64: embedding,
    L decoder layers (RMSNorm, single-head causal attention with RoPE, SwiGLU),
    final norm, LM head.  Auxiliary hidden states are the inputs of layers
    (2, L//2, L-3), the convention of the Neuron page's SupportsEagle3 example."""

    def __init__(self, V, H, L, seed):
        g = np.random.default_rng(seed)
        self.V, self.H, self.L = V, H, L
        self.E = g.standard_normal((V, H))
        self.layers = [dict(q=g.standard_normal((H, H)) / np.sqrt(H), k=g.standard_normal((H, H)) / np.sqrt(H),
                            v=g.standard_normal((H, H)) / np.sqrt(H), o=g.standard_normal((H, H)) / np.sqrt(H),
                            gt=g.standard_normal((2 * H, H)) / np.sqrt(H), up=g.standard_normal((2 * H, H)) / np.sqrt(H),
                            dn=g.standard_normal((H, 2 * H)) / np.sqrt(2 * H)) for _ in range(L)]
        self.head = g.standard_normal((V, H)) * 2.0 / np.sqrt(H)
        self.aux_layers = (2, L // 2, L - 3)

    def forward(self, seq):
        x = self.E[np.asarray(seq)]
        T = len(seq)
        pos = np.arange(T)
        aux = []
        causal = np.tril(np.ones((T, T), dtype=bool))
        for i, p in enumerate(self.layers):
            if i in self.aux_layers:
                aux.append(x)
            n = numerics.rmsnorm(x, 1.0, 1e-6)
            q = numerics.rope(n @ p["q"].T, pos, 1e4)
            k = numerics.rope(n @ p["k"].T, pos, 1e4)
            s = np.where(causal, q @ k.T / np.sqrt(self.H), -np.inf)
            a = np.exp(s - s.max(-1, keepdims=True))
            a /= a.sum(-1, keepdims=True)
            x = x + (a @ (n @ p["v"].T)) @ p["o"].T
            n = numerics.rmsnorm(x, 1.0, 1e-6)
            x = x + (numerics.silu(n @ p["gt"].T) * (n @ p["up"].T)) @ p["dn"].T
        logits = numerics.rmsnorm(x, 1.0, 1e-6) @ self.head.T
        return logits.astype(np.float32), np.concatenate(aux, axis=-1)


def test_closed_loop_greedy_equals_target_only():
    """Greedy speculative decoding emits exactly the target-only greedy sequence
    (the Neuron page: for greedy decoding outputs are bit-exact), for any draft."""
    V, H = 8, 32
    tgt_model = _TinyTarget(V, H, 8, seed=11)
    w = replace(MICRO, name="loop", H=H, nq=2, nkv=1, hd=16, I=48, V=V, B=1, ctx=64, K=3, dtype="f32")
    W, _, _ = _setup(w)
    prompt = [1, 5, 2]
    n_new = 40
    seq = list(prompt)
    for _ in range(n_new):
        lg, _ = tgt_model.forward(seq)
        seq.append(int(np.argmax(lg[-1])))
    want = seq

    ctx_len = np.array([64], dtype=np.int32)
    kv = synth.make_kv(replace(w, ctx=64 + n_new + 8), ctx_len + n_new + 8)
    seq = list(prompt)
    lg, _ = tgt_model.forward(seq)
    x = int(np.argmax(lg[-1]))
    accepted_counts = []
    while len(seq) < len(want) - 1:
        _, aux = tgt_model.forward(seq)
        drafts = step.chain_draft(w, W, aux[-1:], [x], ctx_len, kv, w.K)
        lg, _ = tgt_model.forward(seq + [x] + drafts[0].tolist())
        target = lg[len(seq):][None]                      # rows after x, d1..dK
        out, acc, _ = verify.verify_greedy_chain(target, drafts)
        a = int(acc[0])
        accepted_counts.append(a)
        seq += [x] + drafts[0, :a].tolist()
        x = int(out[0, a])
    seq.append(x)
    n = min(len(seq), len(want))
    assert seq[:n] == want[:n]
    assert max(accepted_counts) >= 1 and min(accepted_counts) == 0


def test_closed_loop_tree_greedy_equals_target_only():
    """Same equivalence with tree drafting and longest-accepted-path verification."""
    V, H = 8, 32
    tgt_model = _TinyTarget(V, H, 8, seed=12)
    w = replace(MICRO, name="loopt", H=H, nq=2, nkv=1, hd=16, I=48, V=V, B=1, ctx=64, dtype="f32",
                mode="tree", top_k=3, depth=3, total=8)
    W, _, _ = _setup(w)
    prompt = [3, 1]
    n_new = 30
    seq = list(prompt)
    for _ in range(n_new):
        lg, _ = tgt_model.forward(seq)
        seq.append(int(np.argmax(lg[-1])))
    want = seq
    ctx_len = np.array([64], dtype=np.int32)
    kv = synth.make_kv(w, ctx_len)
    seq = list(prompt)
    lg, _ = tgt_model.forward(seq)
    x = int(np.argmax(lg[-1]))
    deepest = 0
    while len(seq) < len(want) - 1:
        _, aux = tgt_model.forward(seq)
        fin = step.tree_draft(w, W, aux[-1:], [x], ctx_len, kv, 3, 3, 8)
        # target logits at every tree node: run the target on each node's root path
        N1 = fin["tok"].shape[1]
        rows = []
        for n in range(N1):
            path = []
            p = n
            while p != 0:
                path.append(int(fin["tok"][0, p]))
                p = int(fin["parent"][0, p])
            lg, _ = tgt_model.forward(seq + [x] + path[::-1])
            rows.append(lg[-1])
        out, acc, _ = verify.verify_greedy_tree(np.array(rows)[None], fin["tok"], fin["parent"], 3)
        a = int(acc[0])
        deepest = max(deepest, a)
        seq += [x] + out[0, :a].tolist()
        x = int(out[0, a])
    seq.append(x)
    n = min(len(seq), len(want))
    assert seq[:n] == want[:n]
    assert deepest >= 1


# ---------------------------------------------------------------- rejection sampler
@pytest.mark.parametrize("T", [1.0, 0.7])
def test_rejection_sampler_distribution(T):
    """Brute force on a tiny vocabulary: the first emitted token follows
    softmax(target_0 / T) and, given the first draft was accepted, the second
    follows softmax(target_1 / T) (arXiv:2211.17192, cited by the Neuron page)."""
    V, K, B = 8, 2, 12000
    rng = np.random.default_rng(7)
    rows = rng.standard_normal((K + 1, V)).astype(np.float32) * 1.5
    target = np.broadcast_to(rows, (B, K + 1, V))
    drafts = np.broadcast_to(np.array([int(np.argmax(rows[0])), 3]), (B, K))
    out, acc, _ = verify.verify_rejection(target, drafts, np.full(B, T), seed=99, step_offset=0)
    p0 = scipy.special.softmax(rows[0].astype(np.float64) / T)
    c0 = np.bincount(out[:, 0], minlength=V)
    assert scipy.stats.chisquare(c0, p0 * B).pvalue > 0.01
    sel = acc >= 1
    p1 = scipy.special.softmax(rows[1].astype(np.float64) / T)
    c1 = np.bincount(out[sel, 1], minlength=V)
    assert scipy.stats.chisquare(c1, p1 * sel.sum()).pvalue > 0.01
    # accepted prefix holds the drafts; -1 after the emitted token
    for b in range(50):
        a = acc[b]
        assert out[b, :a].tolist() == drafts[b, :a].tolist()
        assert np.all(out[b, a + 1:] == -1)


def test_rejection_sampler_greedy_rows_and_reject_excludes_draft():
    V, K, B = 6, 3, 400
    rng = np.random.default_rng(8)
    target = rng.standard_normal((B, K + 1, V)).astype(np.float32)
    drafts = rng.integers(0, V, size=(B, K))
    temp = np.where(np.arange(B) % 2 == 0, 0.0, 1.0)
    out, acc, _ = verify.verify_rejection(target, drafts, temp, seed=5)
    g_out, g_acc, _ = verify.verify_greedy_chain(target[::2], drafts[::2])
    np.testing.assert_array_equal(out[::2], g_out)
    np.testing.assert_array_equal(acc[::2], g_acc)
    for b in range(1, B, 2):
        a = acc[b]
        if a < K:
            assert out[b, a] != drafts[b, a]


# ---------------------------------------------------------------- SpecDecodeMetadata
def test_spec_decode_metadata_printed_example():
    """The worked example printed in the Neuron page's SpecDecodeMetadata section."""
    from oracle import metadata
    g = json.load(open(os.path.join(GOLDEN, "spec_decode_metadata.json")))
    got = metadata.spec_decode_metadata(g["cu_num_scheduled_tokens"], g["num_draft_tokens"])
    for k in ("cu_num_draft_tokens", "logits_indices", "target_logits_indices", "bonus_logits_indices"):
        assert got[k].tolist() == g[k], k
    ids = np.arange(1000, 1209)
    got = metadata.spec_decode_metadata(g["cu_num_scheduled_tokens"], g["num_draft_tokens"], ids)
    # drafts follow the verified position: request 0 -> input positions 1, 2, 3
    assert got["draft_token_ids"].tolist() == [1001, 1002, 1003, 1105, 1106, 1208]


@pytest.mark.parametrize("top_k,top_p,T", [(3, 1.0, 1.0), (0, 0.85, 1.0), (4, 0.8, 0.8), (0, 0.3, 1.0)])
def test_rejection_sampler_top_k_top_p_distribution(top_k, top_p, T):
    """With top-k / top-p the emitted tokens follow the filtered, renormalised
    target distribution: brute force on a tiny vocabulary, chi-square over the
    kept tokens, and no token outside the kept set is ever emitted."""
    V, K, B = 8, 2, 12000
    rng = np.random.default_rng(17)
    rows = rng.standard_normal((K + 1, V)).astype(np.float32) * 1.5
    target = np.broadcast_to(rows, (B, K + 1, V))
    drafts = np.broadcast_to(np.array([int(np.argmax(rows[0])), 5]), (B, K))
    out, acc, _ = verify.verify_rejection(target, drafts, np.full(B, T), seed=123, step_offset=0,
                                          top_k=np.full(B, top_k), top_p=np.full(B, top_p))
    for i, sel in ((0, np.ones(B, dtype=bool)), (1, acc >= 1)):
        l = rows[i].astype(np.float64) / T
        kept, _ = verify.kept_set(l, top_k, top_p)
        p = np.where(kept, np.exp(l - l.max()), 0.0)
        p /= p.sum()
        c = np.bincount(out[sel, i], minlength=V)
        assert c[~kept].sum() == 0
        if kept.sum() == 1:
            assert c[kept].sum() == sel.sum()
        else:
            assert scipy.stats.chisquare(c[kept], p[kept] * sel.sum()).pvalue > 0.01


def test_kept_set_closed_forms():
    l = np.array([0.0, 3.0, 1.0, 3.0, 2.0])          # order: 1, 3 (tie -> smaller id), 4, 2, 0
    m, _ = verify.kept_set(l, 2, 1.0)
    assert m.tolist() == [False, True, False, True, False]
    m, _ = verify.kept_set(l, 3, 1.0)
    assert m.tolist() == [False, True, False, True, True]
    p = np.exp(l) / np.exp(l).sum()                   # masses 0.0..: p1 = p3 ~ 0.39, p4 ~ 0.14
    m, _ = verify.kept_set(l, 0, float(p[1] + 1e-9))  # just above one token's mass -> two tokens
    assert m.sum() == 2
    m, _ = verify.kept_set(l, 0, float(p[1] - 1e-9))  # just below -> one token
    assert m.tolist() == [False, True, False, False, False]


# ---------------------------------------------------------------- EAGLE-3.1 options
def test_fc_norm_unit_rms_and_scale_invariance():
    """fc_norm: the fused feature leaves the FC with unit RMS before its gain, so
    h0 / gain has mean square ms / (ms + eps) per row (ms = mean square of the raw
    FC output), and scaling the auxiliary states leaves h0 unchanged up to eps."""
    w = replace(MICRO, name="fcnorm", dtype="f32", fc_norm=True)
    W, _, _ = _setup(w)
    assert "fc_norm" in W and not np.allclose(W["fc_norm"], 1.0)
    aux = synth.make_aux(w).astype(np.float64)
    h0 = draft.fc_fuse(w, W, aux)
    raw = aux @ np.asarray(W["fc"], np.float64).T
    ms = (raw ** 2).mean(-1)
    unit = h0 / np.asarray(W["fc_norm"], np.float64)
    np.testing.assert_allclose((unit ** 2).mean(-1), ms / (ms + w.rms_eps), rtol=1e-12)
    np.testing.assert_allclose(draft.fc_fuse(w, W, 7.0 * aux), h0, rtol=1e-5, atol=1e-7)
    # without the flag: the plain projection
    np.testing.assert_allclose(draft.fc_fuse(replace(w, fc_norm=False), W, aux), raw, rtol=1e-12)


def test_norm_output_recurrence_closed_form():
    """norm_output: with o_proj and down_proj zero the decoder layer passes its
    hidden input through, so the k-th pass's normalised output is RMSNorm_final
    applied k times to h0 (each pass takes the previous normalised output), while
    without the flag every pass sees h0 itself; the first pass is the same either way."""
    w = replace(MICRO, name="normout", dtype="f32", norm_output=True, K=4)
    W, ctx, kv = _setup(w)
    W["wo"] = np.zeros_like(W["wo"])
    W["wdown"] = np.zeros_like(W["wdown"])
    # strongly uneven gains, so that repeated normalisation turns the state
    W["final_norm"] = np.exp(np.random.default_rng(4).normal(0.0, 1.0, w.H)).astype(np.float32)
    aux = synth.make_aux(w).astype(np.float64)
    root = np.array([3, 9])
    lm = np.asarray(W["lm_head"], np.float64)
    g = np.asarray(W["final_norm"], np.float64)
    h = draft.fc_fuse(w, W, aux)
    want_on, want_off = [], []
    x = h
    for _ in range(w.K):
        x = numerics.rmsnorm(x, g, w.rms_eps)
        want_on.append(np.argmax((x @ lm.T).astype(np.float32), -1))
        want_off.append(np.argmax((numerics.rmsnorm(h, g, w.rms_eps) @ lm.T).astype(np.float32), -1))
    got_on = step.chain_draft(w, W, aux, root, ctx, copy.deepcopy(kv), w.K)
    got_off = step.chain_draft(replace(w, norm_output=False), W, aux, root, ctx, copy.deepcopy(kv), w.K)
    np.testing.assert_array_equal(got_on, np.stack(want_on, 1))
    np.testing.assert_array_equal(got_off, np.stack(want_off, 1))
    assert (got_on[:, 0] == got_off[:, 0]).all() and (got_on != got_off).any()


# ---------------------------------------------------------------- batched initial pass (prefill phase)
def test_prefill_inputs_hand_worked_shift_and_scatter():
    """[NEURON] "EagleProposer", ``propose()`` prefill phase: the input ids are
    shifted left by one and the target's new token is scattered at each
    request's last accepted position.  Worked by hand for two requests of four
    verified positions (request 0 accepted everything, request 1 stopped at 1)."""
    ids = np.array([[10, 11, 12, 13], [20, 21, 22, 23]])
    rows, last_row = step.prefill_inputs(ids, next_token=[99, 98], last_idx=[3, 1], ctx_len=[7, 30])
    np.testing.assert_array_equal(rows["tok"], [11, 12, 13, 99, 21, 98, 23, 0])
    np.testing.assert_array_equal(rows["pos"], [7, 8, 9, 10, 30, 31, 32, 33])
    np.testing.assert_array_equal(rows["kv_idx"], [0, 1, 2, 3, 0, 1, 2, 3])
    assert rows["mask"] == [0b1, 0b11, 0b111, 0b1111] * 2          # causal over the draft region
    np.testing.assert_array_equal(last_row, [3, 5])
    assert rows["M"] == 8 and rows["R"] == 4 and rows["B"] == 2


def test_prefill_causal_pass_equals_sequential_single_row_passes():
    """One causal pass over R rows (every row's K/V written, then attention with
    a lower-triangular draft-region mask) equals R single-row passes run one
    after another, pass j writing entry j and attending entries 0..j: same
    hidden states, same K/V bytes."""
    w = replace(MICRO, dtype="f32", B=2, K=4)
    W, ctx, kv = _setup(w)
    R = 4
    rng = np.random.default_rng(5)
    ids = rng.integers(0, w.V, size=(w.B, R))
    rows, _ = step.prefill_inputs(ids, next_token=[3, 4], last_idx=[R - 1, 2], ctx_len=ctx)
    h0 = synth.make_hidden(w, w.B * R).astype(np.float64)
    kv_a = copy.deepcopy(kv)
    pre_a, hn_a = draft.draft_layer(w, W, rows, h0, kv_a)
    kv_b = copy.deepcopy(kv)
    tok = rows["tok"].reshape(w.B, R)
    pre_b = np.zeros_like(pre_a)
    hn_b = np.zeros_like(hn_a)
    for j in range(R):
        r = {"M": w.B, "B": w.B, "R": 1, "step": j, "ctx_len": ctx, "tok": tok[:, j]}
        p, h = draft.draft_layer(w, W, r, h0.reshape(w.B, R, -1)[:, j], kv_b)
        pre_b.reshape(w.B, R, -1)[:, j] = p
        hn_b.reshape(w.B, R, -1)[:, j] = h
    np.testing.assert_allclose(pre_a, pre_b, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(hn_a, hn_b, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(kv_a["k"], kv_b["k"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(kv_a["v"], kv_b["v"], rtol=0, atol=1e-13)


def test_prefill_chain_with_one_verified_token_is_the_chain_drafter():
    """With a single verified position per request (R = 1, last index 0) the
    prefill phase is the chain drafter's first pass on the new token at
    position ctx, and the recurrent passes restart at context ctx + 1: the
    drafts must equal ``chain_draft`` rooted at the new token.  An off-by-one
    in the restart context or the recurrent step index breaks this."""
    w = replace(MICRO, dtype="f32", B=2, K=4)
    W, ctx, kv = _setup(w)
    aux = synth.make_aux(w)
    nxt = np.array([5, 17])
    d_pre, lg_pre = step.prefill_chain_draft(w, W, aux, np.zeros((w.B, 1), dtype=np.int64), nxt, [0, 0], ctx,
                                             copy.deepcopy(kv), w.K, keep_logits=True)
    d_chain, lg_chain = step.chain_draft(w, W, aux, nxt, ctx, copy.deepcopy(kv), w.K, keep_logits=True)
    np.testing.assert_array_equal(d_pre, d_chain)
    np.testing.assert_allclose(lg_pre, lg_chain, rtol=1e-10, atol=1e-12)


def test_prefill_rows_past_the_last_accepted_one_are_ignored():
    """Rows after a request's last accepted position carry rejected drafts; their
    K/V lies where the recurrent passes write before they read, so the drafts
    equal those of a prefill over the accepted rows only."""
    w = replace(MICRO, dtype="f32", B=1, K=3)
    W, ctx, kv = _setup(w)
    R, last = 4, 1
    rng = np.random.default_rng(9)
    ids = rng.integers(0, w.V, size=(1, R))
    aux = synth.make_aux(w, rows=R)
    d_full = step.prefill_chain_draft(w, W, aux, ids, [7], [last], ctx, copy.deepcopy(kv), w.K)
    d_cut = step.prefill_chain_draft(w, W, aux[:last + 1], ids[:, :last + 1], [7], [last], ctx, copy.deepcopy(kv),
                                     w.K)
    np.testing.assert_array_equal(d_full, d_cut)
    # ...while a different token in an accepted row does change them
    ids2 = ids.copy()
    ids2[0, 1] = (ids2[0, 1] + 1) % w.V
    d_other, lg_o = step.prefill_chain_draft(w, W, aux, ids2, [7], [last], ctx, copy.deepcopy(kv), w.K,
                                             keep_logits=True)
    _, lg_f = step.prefill_chain_draft(w, W, aux, ids, [7], [last], ctx, copy.deepcopy(kv), w.K, keep_logits=True)
    assert not np.allclose(lg_o, lg_f)


# ---------------------------------------------------------------- reduced draft vocabulary (d2t)
def test_lm_head_d2t_identity_map_is_the_full_head():
    """A draft vocabulary equal to the target vocabulary with the identity map
    must reproduce the full head exactly."""
    w = replace(MICRO, dtype="f32")
    W, _, _ = _setup(w)
    hn = synth.make_hidden(w, 3).astype(np.float64)
    ids_f, lp_f, lse_f, lg_f = draft.lm_head(w, W, hn, 5)
    Wd = dict(W, d2t=np.arange(w.V, dtype=np.int32))
    ids_d, lp_d, lse_d, lg_d = draft.lm_head(replace(w, draft_vocab=w.V), Wd, hn, 5)
    np.testing.assert_array_equal(ids_d, ids_f)
    np.testing.assert_array_equal(lp_d, lp_f)
    np.testing.assert_array_equal(lse_d, lse_f)


def test_lm_head_d2t_subset_is_the_full_head_restricted():
    """A draft vocabulary S (lm_head rows = the full head's rows at S, d2t = S)
    gives the full head's logits restricted to S: the emitted ids are the
    target ids of the best entries of S, the log-probs normalise over S only."""
    w = replace(MICRO, dtype="f32")
    W, _, _ = _setup(w)
    hn = synth.make_hidden(w, 4).astype(np.float64)
    _, _, _, full = draft.lm_head(w, W, hn, 1)
    S = np.sort(np.random.default_rng(3).choice(w.V, size=23, replace=False)).astype(np.int32)
    Wd = dict(W, lm_head=W["lm_head"][S], d2t=S)
    ids, lp, lse, lg = draft.lm_head(replace(w, draft_vocab=len(S)), Wd, hn, 4)
    for m in range(4):
        sub = full[m, S]
        order = sorted(range(len(S)), key=lambda i: (-np.float32(sub[i]), i))[:4]   # brute force
        np.testing.assert_array_equal(ids[m], S[order])
        z = np.log(np.sum(np.exp(sub - sub.max()))) + sub.max()
        np.testing.assert_allclose(lse[m], z, rtol=1e-13)
        np.testing.assert_allclose(lp[m], sub[order] - z, rtol=1e-12, atol=1e-13)
        assert set(ids[m].tolist()) <= set(S.tolist())


# ---------------------------------------------------------------- candidate log-probs
def test_lowrank_candidate_logprobs_with_every_token_a_candidate():
    """With num_candidates = V every token is a candidate whatever the low-rank
    scores are (rank 4 here, far from exact), so the softmax over the
    candidates is the full softmax: the candidate head's top-k ids and
    log-probs equal the full head's."""
    w = replace(MICRO, dtype="f32", rank=4, num_candidates=MICRO.V)
    W, _, _ = _setup(w)
    W["lr_down"], W["lr_up"] = synth.lowrank_factors(W["lm_head"], 4, "f32")
    hn = synth.make_hidden(w, 3).astype(np.float64)
    ids_f, lp_f, _, _ = draft.lm_head(w, W, hn, 6)
    cand, exact, out, out_lp = draft.lowrank_candidates(w, W, hn, w.V, 6, with_logprob=True)
    np.testing.assert_array_equal(np.sort(cand, axis=1), np.tile(np.arange(w.V), (3, 1)))
    np.testing.assert_array_equal(out, ids_f)
    np.testing.assert_allclose(out_lp, lp_f, rtol=1e-12, atol=1e-13)
    # with fewer candidates the log-probs normalise over the candidates only: they
    # are at least the full log-probs, and exp sums to <= 1 over the kept ones
    _, ex_s, out_s, lp_s = draft.lowrank_candidates(replace(w, num_candidates=10), W, hn, 10, 3,
                                                     with_logprob=True)
    for m in range(3):
        np.testing.assert_allclose(np.exp(ex_s[m] - scipy.special.logsumexp(ex_s[m])).sum(), 1.0)
        full_lp = dict(zip(range(w.V), (hn[m] @ W["lm_head"].astype(np.float64).T
                                        - scipy.special.logsumexp(hn[m] @ W["lm_head"].astype(np.float64).T))))
        for t, l in zip(out_s[m], lp_s[m]):
            assert l >= full_lp[int(t)] - 1e-12
