"""Seeded synthetic inputs for the draft -> tree -> verify step.

This is the one module that both the CPU oracle (through the tests) and the CUDA
library path use.  It draws random numbers and lays them out; it contains none
of the method's arithmetic.  Every array is generated on the host with numpy's
PCG64, chunk by chunk from keys ``(seed, tensor_id, chunk)`` so the result does
not depend on how many threads draw it.

Recipe (shapes follow the workload, values are stand-ins for trained weights
and real activations; no dataset is involved):

* linear weights ~ N(0, 0.02), rounded to bf16 for bf16 workloads;
* RMSNorm gains ~ 1 + N(0, 0.1) (non-unit so a dropped or misplaced gain shows);
* token embedding ~ N(0, 0.02);
* auxiliary target hidden states (3 of them, concatenated) ~ N(0, 1);
* context K/V in the paged cache ~ N(0, 1) (treated as post-RoPE keys); every
  slot of the cache is filled so that reading a key outside the allowed set
  changes results;
* paged cache: ``block_size`` slots per block, blocks handed to requests in a
  random permutation;
* next (root) tokens uniform over the vocabulary;
* target-logit noise ~ N(0, sigma) (the tests add it to draft logits).
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_CHUNK = 1 << 22

# tensor ids for the key of each generated array
_TID = {
    "fc": 1, "embed": 2, "hidden_norm": 3, "in_norm": 4, "post_norm": 5, "final_norm": 6,
    "wq": 7, "wk": 8, "wv": 9, "wo": 10, "wgate": 11, "wup": 12, "wdown": 13, "lm_head": 14,
    "aux": 20, "kv_k": 21, "kv_v": 22, "ctx": 23, "blocks": 24, "root": 25, "noise": 26,
    "hid": 27, "misc": 28, "d2t": 29, "fc_norm": 30,
}


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """float32 array -> float32 array whose values are bf16 (round to nearest even)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).copy()
    u += np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    u &= np.uint32(0xFFFF0000)
    return u.view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """bf16-valued float32 array -> its uint16 bit patterns (exact)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return (u >> np.uint32(16)).astype(np.uint16)


def _normal_into(out: np.ndarray, key: tuple, std: float, mean: float = 0.0):
    flat = out.reshape(-1)
    n = flat.size
    nchunks = (n + _CHUNK - 1) // _CHUNK

    def work(c):
        lo = c * _CHUNK
        hi = min(n, lo + _CHUNK)
        g = np.random.default_rng(list(key) + [c])
        seg = g.standard_normal(hi - lo, dtype=np.float32)
        if std != 1.0:
            seg *= np.float32(std)
        if mean != 0.0:
            seg += np.float32(mean)
        flat[lo:hi] = seg

    if nchunks <= 2:
        for c in range(nchunks):
            work(c)
    else:
        with ThreadPoolExecutor(max_workers=min(nchunks, os.cpu_count() or 4)) as ex:
            list(ex.map(work, range(nchunks)))
    return out


def normal(shape, seed: int, name: str, std: float = 1.0, mean: float = 0.0, sub: int = 0):
    out = np.empty(shape, dtype=np.float32)
    return _normal_into(out, (seed, _TID[name], sub), std, mean)


def _store(x: np.ndarray, dtype: str) -> np.ndarray:
    return round_to_bf16(x) if dtype == "bf16" else x


def make_weights(w, with_lm_head: bool = True) -> dict:
    """Draft-model weights, nn.Linear layout ``[out, in]`` row-major, as float32 arrays
    whose values are exactly representable in the workload's storage dtype."""
    s = w.seed
    H, nq, nkv, hd, I, V = w.H, w.nq, w.nkv, w.hd, w.I, w.V
    W = {}
    W["fc"] = _store(normal((H, 3 * H), s, "fc", 0.02), w.dtype)
    W["embed"] = _store(normal((V, H), s, "embed", 0.02), w.dtype)
    for nm in ("hidden_norm", "in_norm", "post_norm", "final_norm"):
        W[nm] = _store(normal((H,), s, nm, 0.1, 1.0), w.dtype)
    if getattr(w, "fc_norm", False):
        W["fc_norm"] = _store(normal((H,), s, "fc_norm", 0.1, 1.0), w.dtype)
    W["wq"] = _store(normal((nq * hd, 2 * H), s, "wq", 0.02), w.dtype)
    W["wk"] = _store(normal((nkv * hd, 2 * H), s, "wk", 0.02), w.dtype)
    W["wv"] = _store(normal((nkv * hd, 2 * H), s, "wv", 0.02), w.dtype)
    W["wo"] = _store(normal((H, nq * hd), s, "wo", 0.02), w.dtype)
    W["wgate"] = _store(normal((I, H), s, "wgate", 0.02), w.dtype)
    W["wup"] = _store(normal((I, H), s, "wup", 0.02), w.dtype)
    W["wdown"] = _store(normal((H, I), s, "wdown", 0.02), w.dtype)
    if with_lm_head:
        rows = w.draft_vocab if w.draft_vocab > 0 else V
        W["lm_head"] = _store(normal((rows, H), s, "lm_head", 0.02), w.dtype)
        if w.draft_vocab > 0:
            W["d2t"] = draft_vocab_map(w)
    return W


def draft_vocab_map(w) -> np.ndarray:
    """Target token id of each draft-vocabulary entry: a seeded, sorted subset of
    the target vocabulary (stand-in for a calibrated frequent-token list)."""
    g = np.random.default_rng([w.seed, _TID["d2t"]])
    return np.sort(g.choice(w.V, size=w.draft_vocab, replace=False)).astype(np.int32)


def lowrank_factors(lm_head: np.ndarray, rank: int, dtype: str):
    """Rank-r factors of the LM head from its truncated SVD: ``lm_head ~= up @ down``
    with ``down = S^(1/2) V_r^T`` ``[r, H]`` and ``up = U_r S^(1/2)`` ``[V, r]``.

    This is input preparation (the candidate head's initialisation in the
    "nemo_automodel ... eagle4" page, module docstring: factors initialised from
    the truncated SVD of the draft lm_head), not a step of the serving path.  The
    right singular vectors come from the eigendecomposition of ``W^T W``.
    """
    Wt = np.ascontiguousarray(lm_head, dtype=np.float32)
    G = (Wt.T @ Wt).astype(np.float64)
    evals, evecs = np.linalg.eigh(G)
    order = np.argsort(evals)[::-1][:rank]
    sig = np.sqrt(np.maximum(evals[order], 0.0))
    Vr = evecs[:, order]                                   # [H, r]
    US = (Wt.astype(np.float64) @ Vr)                      # U_r S   [V, r]
    root = np.sqrt(np.where(sig > 0, sig, 1.0))
    down = (Vr * root).T                                   # S^(1/2) V_r^T
    up = US / root                                         # U_r S^(1/2)
    return _store(down.astype(np.float32), dtype), _store(up.astype(np.float32), dtype)


def context_lengths(w) -> np.ndarray:
    if w.ctx_range is None:
        return np.full(w.B, w.ctx, dtype=np.int32)
    g = np.random.default_rng([w.seed, _TID["ctx"]])
    lo, hi = w.ctx_range
    return g.integers(lo, hi + 1, size=w.B, dtype=np.int64).astype(np.int32)


def make_kv(w, ctx_len: np.ndarray):
    """Paged K/V cache ``[num_slots, nkv, hd]`` plus block table ``[B, max_blocks]``."""
    bs = w.block_size
    need = (ctx_len.astype(np.int64) + w.draft_region + bs - 1) // bs
    max_blocks = int(need.max())
    total = int(need.sum())
    g = np.random.default_rng([w.seed, _TID["blocks"]])
    perm = g.permutation(total).astype(np.int32)
    table = np.zeros((w.B, max_blocks), dtype=np.int32)
    o = 0
    for b in range(w.B):
        table[b, :need[b]] = perm[o:o + need[b]]
        o += need[b]
    num_slots = total * bs
    K = _store(normal((num_slots, w.nkv, w.hd), w.seed, "kv_k"), w.dtype)
    Vv = _store(normal((num_slots, w.nkv, w.hd), w.seed, "kv_v"), w.dtype)
    return {"k": K, "v": Vv, "block_table": table, "block_size": bs,
            "max_blocks": max_blocks, "num_slots": num_slots}


def make_aux(w, rows: int = None) -> np.ndarray:
    rows = w.B if rows is None else rows
    return _store(normal((rows, 3 * w.H), w.seed, "aux"), w.dtype)


def make_hidden(w, rows: int, sub: int = 0) -> np.ndarray:
    """A stand-in recurrent hidden state ``[rows, H]`` (for single-call tests)."""
    return _store(normal((rows, w.H), w.seed, "hid", 1.0, 0.0, sub), w.dtype)


def root_tokens(w) -> np.ndarray:
    g = np.random.default_rng([w.seed, _TID["root"]])
    return g.integers(0, w.V, size=w.B, dtype=np.int64).astype(np.int32)


def integers(seed: int, sub: int, lo: int, hi: int, size) -> np.ndarray:
    g = np.random.default_rng([seed, _TID["misc"], sub])
    return g.integers(lo, hi, size=size, dtype=np.int64).astype(np.int32)


def uniforms(seed: int, sub: int, size) -> np.ndarray:
    g = np.random.default_rng([seed, _TID["misc"], sub])
    return g.random(size, dtype=np.float64)


def noise(w, shape, sub: int = 0) -> np.ndarray:
    """Target-logit noise ~ N(0, sigma), float32."""
    return normal(shape, w.seed, "noise", w.sigma, 0.0, sub)
