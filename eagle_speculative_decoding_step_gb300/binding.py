"""ctypes binding of libeaglespec (include/eaglespec.h).

Argument marshalling only: every function passes device pointers of torch
tensors, sizes and the current CUDA stream to the C entry point of the same
name and raises ``SpecError`` on a non-zero status.  All computation happens in
the library's CUDA kernels; if the library is not built, loading fails loudly.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# EAGLESPEC_TIMELINE=1 loads the instrumented build (build(timeline=True)): the same
# library with per-block start / end stamps, for timeline.py only
LIB_PATH = os.path.join(_HERE, "libeaglespec_timeline.so" if os.environ.get("EAGLESPEC_TIMELINE") == "1"
                        else "libeaglespec.so")

c_i32 = ctypes.c_int32
c_u64 = ctypes.c_uint64
c_vp = ctypes.c_void_p
c_size = ctypes.c_size_t

DTYPE_F32 = 0
DTYPE_BF16 = 1


class SpecError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        msg = _lib().spec_status_string(status).decode() if _LIB is not None else str(status)
        super().__init__("%s failed: %s (%d)" % (what, msg, status))


class ModelDesc(ctypes.Structure):
    _fields_ = [("hidden", c_i32), ("n_q_heads", c_i32), ("n_kv_heads", c_i32), ("head_dim", c_i32),
                ("intermediate", c_i32), ("vocab", c_i32), ("dtype", c_i32), ("rms_eps", ctypes.c_float),
                ("rope_theta", ctypes.c_float), ("window", c_i32), ("rank", c_i32), ("num_candidates", c_i32),
                ("draft_vocab", c_i32), ("fc_norm", c_i32), ("norm_output", c_i32)]


_WEIGHT_NAMES = ["fc", "embed", "hidden_norm", "in_norm", "post_norm", "final_norm", "wq", "wk", "wv", "wo",
                 "wgate", "wup", "wdown", "lm_head", "lr_down", "lr_up", "d2t", "fc_norm"]


class Weights(ctypes.Structure):
    _fields_ = [(n, c_vp) for n in _WEIGHT_NAMES]


class KV(ctypes.Structure):
    _fields_ = [("k", c_vp), ("v", c_vp), ("block_table", c_vp), ("block_size", c_i32), ("max_blocks", c_i32),
                ("num_slots", c_i32)]


class Rows(ctypes.Structure):
    _fields_ = [("M", c_i32), ("B", c_i32), ("rows_per_req", c_i32), ("step", c_i32), ("ctx_len", c_vp),
                ("tok", c_vp), ("tok_stride", c_i32), ("pos", c_vp), ("kv_idx", c_vp), ("mask", c_vp),
                ("hid_src", c_vp), ("max_ctx", c_i32)]


class TreeIO(ctypes.Structure):
    _fields_ = [(n, c_vp) for n in ["frontier_tok", "frontier_pos", "frontier_kv_idx", "frontier_mask",
                                     "frontier_hid_src", "tree_tok", "tree_parent", "tree_depth", "tree_pos",
                                     "tree_score", "tree_mask"]]


EXPORTS = {
    # name: (restype, argtypes)
    "spec_status_string": (ctypes.c_char_p, [c_i32]),
    "spec_version": (c_i32, []),
    "spec_workspace_bytes": (c_size, [ctypes.POINTER(ModelDesc), c_i32, c_i32]),
    "spec_get_device_error": (c_i32, [c_vp, ctypes.POINTER(c_i32), c_vp]),
    "spec_clear_device_error": (c_i32, [c_vp, c_vp]),
    "spec_fc_fuse": (c_i32, [ctypes.POINTER(ModelDesc), ctypes.POINTER(Weights), c_vp, c_vp, c_i32, c_vp, c_size,
                             c_vp]),
    "spec_draft_layer": (c_i32, [ctypes.POINTER(ModelDesc), ctypes.POINTER(Weights), ctypes.POINTER(Rows), c_vp,
                                 c_vp, c_vp, ctypes.POINTER(KV), c_vp, c_size, c_vp]),
    "spec_lm_head": (c_i32, [ctypes.POINTER(ModelDesc), ctypes.POINTER(Weights), c_vp, c_i32, c_i32, c_vp, c_i32,
                             c_vp, c_vp, c_vp, c_vp, c_size, c_vp]),
    "spec_lowrank_candidates": (c_i32, [ctypes.POINTER(ModelDesc), ctypes.POINTER(Weights), c_vp, c_i32, c_i32,
                                        c_vp, c_vp, c_vp, c_vp, c_i32, c_vp, c_size, c_vp]),
    "spec_tree_state_bytes": (c_size, [c_i32, c_i32, c_i32, c_i32]),
    "spec_tree_expand": (c_i32, [c_i32, c_i32, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp,
                                 ctypes.POINTER(TreeIO), c_vp]),
    "spec_verify_workspace_bytes": (c_size, [c_i32, c_i32, c_i32]),
    "spec_verify_greedy": (c_i32, [c_i32, c_i32, c_i32, c_vp, c_vp, c_vp, c_i32, c_vp, c_vp, c_vp,
                                   ctypes.POINTER(ModelDesc), ctypes.POINTER(KV), c_vp, c_vp, c_size, c_vp]),
    "spec_verify_rejection": (c_i32, [c_i32, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_u64, c_u64, c_vp, c_vp,
                                      c_vp, c_vp, c_size, c_vp]),
    "spec_decode_metadata": (c_i32, [c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp]),
    "spec_prefill_inputs": (c_i32, [c_i32, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp,
                                    c_vp]),
    "spec_gather_rows": (c_i32, [c_vp, c_i32, c_i32, c_vp, c_i32, c_vp, c_vp, c_vp]),
    "spec_verify_greedy_static": (c_i32, [c_i32, c_i32, c_i32, c_vp, c_vp, c_vp, c_i32, c_vp, c_vp, c_vp,
                                          ctypes.POINTER(ModelDesc), ctypes.POINTER(KV), c_vp, c_vp]),
    "spec_verify_greedy_static_capacity": (c_size, []),
    "spec_verify_greedy_static_bytes": (c_size, [c_i32, c_i32, c_i32]),
    "spec_verify_greedy_static_error": (c_i32, [ctypes.POINTER(c_i32), c_vp]),
}

_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("%s is not built (run `python -m eagle_speculative_decoding_step_gb300.build`%s); "
                               "there is no fallback" % (os.path.basename(LIB_PATH),
                                                         " -t" if "timeline" in LIB_PATH else ""))
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in EXPORTS.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _LIB = lib
    return _LIB


def load():
    return _lib()


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _check(st, what):
    if st != 0:
        raise SpecError(st, what)


def make_desc(w) -> ModelDesc:
    """ModelDesc from a workload (configs.Workload)."""
    return ModelDesc(w.H, w.nq, w.nkv, w.hd, w.I, w.V, DTYPE_BF16 if w.dtype == "bf16" else DTYPE_F32,
                     w.rms_eps, w.rope_theta, w.window, w.rank, w.num_candidates, w.draft_vocab,
                     int(getattr(w, "fc_norm", False)), int(getattr(w, "norm_output", False)))


def make_weights(W: dict) -> Weights:
    """Weights struct from a dict of device tensors (names as in the header)."""
    w = Weights(*[_p(W.get(n)) for n in _WEIGHT_NAMES])
    w._keep = dict(W)
    return w


def make_kv(kv: dict) -> KV:
    k = KV(_p(kv["k"]), _p(kv["v"]), _p(kv["block_table"]), int(kv["block_size"]), int(kv["max_blocks"]),
           int(kv["num_slots"]))
    k._keep = (kv["k"], kv["v"], kv["block_table"])
    return k


def make_rows(M, B, R, ctx_len, tok, step=0, tok_stride=1, pos=None, kv_idx=None, mask=None, hid_src=None,
              max_ctx=0) -> Rows:
    r = Rows(M, B, R, step, _p(ctx_len), _p(tok), tok_stride, _p(pos), _p(kv_idx), _p(mask), _p(hid_src),
             int(max_ctx))
    r._keep = (ctx_len, tok, pos, kv_idx, mask, hid_src)      # the struct holds raw pointers
    return r


def make_tree_io(frontier_tok, frontier_pos, frontier_kv_idx, frontier_mask, frontier_hid_src, tree_tok,
                 tree_parent, tree_depth, tree_pos, tree_score, tree_mask) -> TreeIO:
    ts = (frontier_tok, frontier_pos, frontier_kv_idx, frontier_mask, frontier_hid_src, tree_tok, tree_parent,
          tree_depth, tree_pos, tree_score, tree_mask)
    io = TreeIO(*[_p(t) for t in ts])
    io._keep = ts
    return io


# ------------------------------------------------------------------ entry points
def spec_workspace_bytes(desc, max_rows, max_ctx=0):
    return _lib().spec_workspace_bytes(ctypes.byref(desc), max_rows, max_ctx)


def spec_verify_workspace_bytes(B, R, V):
    return _lib().spec_verify_workspace_bytes(B, R, V)


def spec_tree_state_bytes(B, top_k, depth, total):
    return _lib().spec_tree_state_bytes(B, top_k, depth, total)


def spec_get_device_error(ws):
    v = c_i32(0)
    _check(_lib().spec_get_device_error(_p(ws), ctypes.byref(v), _stream()), "spec_get_device_error")
    return v.value


def spec_clear_device_error(ws):
    _check(_lib().spec_clear_device_error(_p(ws), _stream()), "spec_clear_device_error")


def spec_fc_fuse(desc, weights, aux, h0, M, ws):
    _check(_lib().spec_fc_fuse(ctypes.byref(desc), ctypes.byref(weights), _p(aux), _p(h0), M, _p(ws),
                               ws.numel() * ws.element_size(), _stream()), "spec_fc_fuse")


def spec_draft_layer(desc, weights, rows, hid_in, hid_prenorm, hid_normed, kv, ws):
    _check(_lib().spec_draft_layer(ctypes.byref(desc), ctypes.byref(weights), ctypes.byref(rows), _p(hid_in),
                                   _p(hid_prenorm), _p(hid_normed), ctypes.byref(kv), _p(ws),
                                   ws.numel() * ws.element_size(), _stream()), "spec_draft_layer")


def spec_lm_head(desc, weights, hn, M, k, topk_ids, topk_logprob, lse=None, logits=None, ws=None, ids_ld=0):
    _check(_lib().spec_lm_head(ctypes.byref(desc), ctypes.byref(weights), _p(hn), M, k, _p(topk_ids), ids_ld,
                               _p(topk_logprob), _p(lse), _p(logits), _p(ws), ws.numel() * ws.element_size(),
                               _stream()), "spec_lm_head")


def spec_lowrank_candidates(desc, weights, hn, M, k_out, out_ids, cand_ids=None, cand_logits=None, ws=None,
                            out_ld=0, out_logprob=None):
    _check(_lib().spec_lowrank_candidates(ctypes.byref(desc), ctypes.byref(weights), _p(hn), M, k_out,
                                          _p(cand_ids), _p(cand_logits), _p(out_ids), _p(out_logprob), out_ld,
                                          _p(ws), ws.numel() * ws.element_size(), _stream()),
           "spec_lowrank_candidates")


def spec_tree_expand(B, top_k, depth_idx, depth, total, ctx_len, root_tok, topk_ids, topk_logprob, state, io):
    _check(_lib().spec_tree_expand(B, top_k, depth_idx, depth, total, _p(ctx_len), _p(root_tok), _p(topk_ids),
                                   _p(topk_logprob), _p(state), ctypes.byref(io), _stream()), "spec_tree_expand")


def spec_verify_greedy(B, R, V, target_logits, draft_tok, out_tok, accept_len, kv_src=None, parent=None,
                       max_depth=0, desc=None, kv=None, ctx_len=None, ws=None):
    _check(_lib().spec_verify_greedy(B, R, V, _p(target_logits), _p(draft_tok), _p(parent), max_depth, _p(out_tok),
                                     _p(accept_len), _p(kv_src), ctypes.byref(desc) if desc is not None else None,
                                     ctypes.byref(kv) if kv is not None else None, _p(ctx_len), _p(ws),
                                     ws.numel() * ws.element_size(), _stream()), "spec_verify_greedy")


def spec_verify_rejection(B, K, V, target_logits, draft_tok, temperature, seed, step_offset, out_tok, accept_len,
                          kv_src=None, ws=None, top_k=None, top_p=None):
    _check(_lib().spec_verify_rejection(B, K, V, _p(target_logits), _p(draft_tok), _p(temperature), _p(top_k),
                                        _p(top_p), seed, step_offset, _p(out_tok), _p(accept_len), _p(kv_src),
                                        _p(ws), ws.numel() * ws.element_size(), _stream()), "spec_verify_rejection")


def spec_verify_greedy_static(B, R, V, target_logits, draft_tok, out_tok, accept_len, kv_src=None, parent=None,
                              max_depth=0, desc=None, kv=None, ctx_len=None):
    """Greedy verification with the library's fixed scratch array (no workspace)."""
    _check(_lib().spec_verify_greedy_static(B, R, V, _p(target_logits), _p(draft_tok), _p(parent), max_depth,
                                            _p(out_tok), _p(accept_len), _p(kv_src),
                                            ctypes.byref(desc) if desc is not None else None,
                                            ctypes.byref(kv) if kv is not None else None, _p(ctx_len), _stream()),
           "spec_verify_greedy_static")


def spec_verify_greedy_static_capacity():
    return _lib().spec_verify_greedy_static_capacity()


def spec_verify_greedy_static_bytes(B, R, V):
    return _lib().spec_verify_greedy_static_bytes(B, R, V)


def spec_verify_greedy_static_error():
    v = c_i32(0)
    _check(_lib().spec_verify_greedy_static_error(ctypes.byref(v), _stream()), "spec_verify_greedy_static_error")
    return v.value


def spec_decode_metadata(R, cu_num_scheduled, num_draft, cu_num_draft, logits_indices, target_logits_indices,
                         bonus_logits_indices, input_ids=None, draft_token_ids=None, ws=None):
    _check(_lib().spec_decode_metadata(R, _p(cu_num_scheduled), _p(num_draft), _p(input_ids), _p(cu_num_draft),
                                       _p(logits_indices), _p(target_logits_indices), _p(bonus_logits_indices),
                                       _p(draft_token_ids), _p(ws), _stream()), "spec_decode_metadata")


def spec_prefill_inputs(B, R, input_ids, next_token, last_idx, ctx_len, tok, pos, kv_idx, mask, last_row,
                        ctx_next=None, ws=None):
    _check(_lib().spec_prefill_inputs(B, R, _p(input_ids), _p(next_token), _p(last_idx), _p(ctx_len), _p(tok),
                                      _p(pos), _p(kv_idx), _p(mask), _p(last_row), _p(ctx_next), _p(ws),
                                      _stream()),
           "spec_prefill_inputs")


def spec_gather_rows(src, n_src, row_bytes, rows, n, dst, ws=None):
    _check(_lib().spec_gather_rows(_p(src), n_src, row_bytes, _p(rows), n, _p(dst), _p(ws), _stream()),
           "spec_gather_rows")
