"""Device-resident draft model and the whole speculative step, on libeaglespec.

``DeviceModel`` uploads a workload's weights and paged K/V cache to the GPU and
owns the workspaces.  ``ChainStep`` and ``TreeStep`` hold the per-step device
buffers and issue one speculative step as a fixed sequence of library calls on
the current stream (no host synchronisation, so a step can be captured into a
CUDA graph and replayed):

* chain ([NEURON] "Speculative Decoding (EAGLE3) in the vLLM Neuron
  Framework", "EagleProposer" ``propose()``): fc_fuse, then K x (draft_layer,
  LM head or low-rank candidate head), then greedy or rejection verification;
* tree ([EAGLET] draft_top_k / draft_depth / total_draft_tokens): fc_fuse,
  root pass + LM head top-k + tree_expand, (depth-1) x (frontier pass + LM head
  top-k + tree_expand), then greedy tree verification with K/V compaction.

Every computation is a library kernel; torch only allocates device memory and
provides the stream.
"""
import numpy as np
import torch

from . import binding as lib
from . import synth


def to_device(x: np.ndarray, dtype: str, device) -> torch.Tensor:
    """Upload a float32 array holding values of ``dtype`` ("bf16" or "f32")."""
    if dtype == "bf16":
        bits = torch.from_numpy(synth.bf16_bits(x))
        return bits.view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device)


def from_device(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy()


class DeviceModel:
    def __init__(self, w, W: dict, kv: dict, ctx_len: np.ndarray, device="cuda", max_rows=None):
        self.w = w
        self.device = device
        self.desc = lib.make_desc(w)
        self.tW = {k: (torch.from_numpy(np.asarray(v, dtype=np.int32)).to(device) if k == "d2t"
                       else to_device(v, w.dtype, device)) for k, v in W.items()}
        self.weights = lib.make_weights(self.tW)
        self.tkv = {
            "k": to_device(kv["k"], w.dtype, device),
            "v": to_device(kv["v"], w.dtype, device),
            "block_table": torch.from_numpy(kv["block_table"]).to(device),
            "block_size": kv["block_size"], "max_blocks": kv["max_blocks"], "num_slots": kv["num_slots"],
        }
        self.kv = lib.make_kv(self.tkv)
        self.ctx_len = torch.from_numpy(np.asarray(ctx_len, dtype=np.int32)).to(device)
        self.max_rows = max_rows or max(w.rows_max, w.B)
        nb = lib.spec_workspace_bytes(self.desc, self.max_rows, w.max_ctx)
        self.ws = torch.zeros(nb, dtype=torch.uint8, device=device)
        self.tdtype = torch.bfloat16 if w.dtype == "bf16" else torch.float32

    def hidden(self, rows):
        return torch.zeros(rows, self.w.H, dtype=self.tdtype, device=self.device)

    def device_error(self):
        return lib.spec_get_device_error(self.ws)


class ChainStep:
    """Buffers and call sequence of one chain speculative step."""

    def __init__(self, dm: DeviceModel, aux: torch.Tensor, root_tok: torch.Tensor, target: torch.Tensor,
                 temperature=None, seed=0, step_offset=0, top_k=None, top_p=None):
        w = dm.w
        self.dm = dm
        B, K, V = w.B, w.K, w.V
        self.B, self.K, self.V = B, K, V
        dev = dm.device
        self.aux = aux
        self.root = root_tok
        self.target = target
        self.h0 = dm.hidden(B)
        self.pre = [dm.hidden(B), dm.hidden(B)]
        self.hn = dm.hidden(B)
        self.hns = [self.hn, dm.hidden(B)] if w.norm_output else [self.hn]
        self.drafts = torch.zeros(B, K, dtype=torch.int32, device=dev)
        self.lp = torch.zeros(B, K, dtype=torch.float32, device=dev)
        self.out = torch.zeros(B, K + 1, dtype=torch.int32, device=dev)
        self.acc = torch.zeros(B, dtype=torch.int32, device=dev)
        self.kv_src = torch.zeros(B, K + 1, dtype=torch.int32, device=dev)
        self.temperature = temperature if temperature is not None else torch.full((B,), w.temperature,
                                                                                     device=dev)
        self.seed, self.step_offset = seed, step_offset
        self.top_k, self.top_p = top_k, top_p
        self.vws = torch.zeros(lib.spec_verify_workspace_bytes(B, K + 1, V), dtype=torch.uint8, device=dev)

    def draft(self, trace=None):
        """Issue the drafting calls.  ``trace(i, tensors)``, if given, is called on
        the host after pass i is issued (tensors: that pass's hn, pre-norm state
        and draft ids, and the FC-fused feature h0); it must synchronise before
        reading them."""
        dm, w, B, K = self.dm, self.dm.w, self.B, self.K
        lib.spec_fc_fuse(dm.desc, dm.weights, self.aux, self.h0, B, dm.ws)
        hid = self.h0
        for i in range(K):
            if i == 0:
                rows = lib.make_rows(B, B, 1, dm.ctx_len, self.root, step=0, max_ctx=w.max_ctx)
            else:
                rows = lib.make_rows(B, B, 1, dm.ctx_len, self.drafts.data_ptr() + 4 * (i - 1), step=i,
                                     tok_stride=K, max_ctx=w.max_ctx)
            out = self.pre[i % 2]
            # EAGLE-3.1 norm_output: the next pass takes the normalised state (two buffers)
            hn = self.hns[i % 2] if w.norm_output else self.hn
            lib.spec_draft_layer(dm.desc, dm.weights, rows, hid, out, hn, dm.kv, dm.ws)
            ids = self.drafts.data_ptr() + 4 * i
            if w.rank > 0:
                lib.spec_lowrank_candidates(dm.desc, dm.weights, hn, B, 1, ids, ws=dm.ws, out_ld=K)
            else:
                lib.spec_lm_head(dm.desc, dm.weights, hn, B, 1, ids, self.lp.data_ptr() + 4 * i, ws=dm.ws,
                                 ids_ld=K)
            if trace is not None:
                trace(i, {"hn": hn, "pre": out, "ids": self.drafts[:, i], "h0": self.h0})
            hid = hn if w.norm_output else out

    def verify(self):
        w = self.dm.w
        if w.verify == "rejection":
            lib.spec_verify_rejection(self.B, self.K, self.V, self.target, self.drafts, self.temperature, self.seed,
                                      self.step_offset, self.out, self.acc, self.kv_src, ws=self.vws,
                                      top_k=self.top_k, top_p=self.top_p)
        else:
            lib.spec_verify_greedy(self.B, self.K + 1, self.V, self.target, self.drafts, self.out, self.acc,
                                   self.kv_src, ws=self.vws)

    def run(self):
        self.draft()
        self.verify()


class TreeStep:
    """Buffers and call sequence of one tree speculative step."""

    def __init__(self, dm: DeviceModel, aux: torch.Tensor, root_tok: torch.Tensor, target: torch.Tensor = None):
        w = dm.w
        self.dm = dm
        B, k, D, N, V = w.B, w.top_k, w.depth, w.total, w.V
        self.B, self.k, self.D, self.N, self.V = B, k, D, N, V
        dev = dm.device
        self.aux, self.root, self.target = aux, root_tok, target
        self.h0 = dm.hidden(B)
        self.pre = [dm.hidden(B * k), dm.hidden(B * k)]
        self.hn = dm.hidden(B * k)
        self.hns = [self.hn, dm.hidden(B * k)]
        self.ids = torch.zeros(B * k, k, dtype=torch.int32, device=dev)
        self.lp = torch.zeros(B * k, k, dtype=torch.float32, device=dev)
        i32 = dict(dtype=torch.int32, device=dev)
        self.f_tok = torch.zeros(B * k, **i32)
        self.f_pos = torch.zeros(B * k, **i32)
        self.f_kv = torch.zeros(B * k, **i32)
        self.f_mask = torch.zeros(B * k, dtype=torch.int64, device=dev)
        self.f_src = torch.zeros(B * k, **i32)
        self.t_tok = torch.zeros(B, N + 1, **i32)
        self.t_par = torch.zeros(B, N + 1, **i32)
        self.t_dep = torch.zeros(B, N + 1, **i32)
        self.t_pos = torch.zeros(B, N + 1, **i32)
        self.t_score = torch.zeros(B, N + 1, dtype=torch.float32, device=dev)
        self.t_mask = torch.zeros(B, N + 1, dtype=torch.int64, device=dev)
        self.io = lib.make_tree_io(self.f_tok, self.f_pos, self.f_kv, self.f_mask, self.f_src, self.t_tok, self.t_par,
                                   self.t_dep, self.t_pos, self.t_score, self.t_mask)
        self.state = torch.zeros(lib.spec_tree_state_bytes(B, k, D, N), dtype=torch.uint8, device=dev)
        self.out = torch.zeros(B, D + 1, **i32)
        self.acc = torch.zeros(B, **i32)
        self.kv_src = torch.zeros(B, D + 1, **i32)
        self.vws = torch.zeros(lib.spec_verify_workspace_bytes(B, N + 1, V), dtype=torch.uint8, device=dev)

    def draft(self, trace=None):
        """Issue the drafting calls.  ``trace(d, tensors)``, if given, is called on
        the host after depth d's pass and head are issued (tensors: the pass's hn,
        pre-norm state, top-k ids and log-probs, and at depth 1 the FC-fused
        feature h0); it must synchronise before reading them.  The frontier rows of pass d + 1 are the ``f_*`` buffers once
        the following expansion has run."""
        dm, B, k, D, N = self.dm, self.B, self.k, self.D, self.N
        lib.spec_fc_fuse(dm.desc, dm.weights, self.aux, self.h0, B, dm.ws)
        rows = lib.make_rows(B, B, 1, dm.ctx_len, self.root, step=0, max_ctx=dm.w.max_ctx)
        no = dm.w.norm_output          # EAGLE-3.1: children take the parent's normalised state
        lib.spec_draft_layer(dm.desc, dm.weights, rows, self.h0, self.pre[0], self.hns[0], dm.kv, dm.ws)
        self._head(B, self.hns[0])
        if trace is not None:
            trace(1, {"hn": self.hns[0][:B], "pre": self.pre[0][:B], "ids": self.ids[:B], "lp": self.lp[:B],
                      "h0": self.h0})
        lib.spec_tree_expand(B, k, 1, D, N, dm.ctx_len, self.root, self.ids, self.lp, self.state, self.io)
        for d in range(2, D + 1):
            if trace is not None:
                trace(("rows", d), {"tok": self.f_tok, "pos": self.f_pos, "kv_idx": self.f_kv, "mask": self.f_mask,
                                    "hid_src": self.f_src})
            rows = lib.make_rows(B * k, B, k, dm.ctx_len, self.f_tok, pos=self.f_pos, kv_idx=self.f_kv,
                                 mask=self.f_mask, hid_src=self.f_src, max_ctx=dm.w.max_ctx)
            src, dst = self.pre[d % 2], self.pre[(d + 1) % 2]
            hsrc, hdst = self.hns[d % 2], self.hns[(d + 1) % 2]
            lib.spec_draft_layer(dm.desc, dm.weights, rows, hsrc if no else src, dst, hdst, dm.kv, dm.ws)
            self._head(B * k, hdst)
            if trace is not None:
                trace(d, {"hn": hdst, "pre": dst, "ids": self.ids, "lp": self.lp})
            lib.spec_tree_expand(B, k, d, D, N, dm.ctx_len, self.root, self.ids, self.lp, self.state, self.io)

    def _head(self, M, hn):
        """top-k ids and log-probs per row: full LM head, or the EAGLE-4 candidate head
        (log-probs over its rescored candidates)."""
        dm, k = self.dm, self.k
        if dm.w.rank > 0:
            lib.spec_lowrank_candidates(dm.desc, dm.weights, hn, M, k, self.ids, ws=dm.ws, out_logprob=self.lp)
        else:
            lib.spec_lm_head(dm.desc, dm.weights, hn, M, k, self.ids, self.lp, ws=dm.ws)

    def verify(self, compact=True):
        dm = self.dm
        lib.spec_verify_greedy(self.B, self.N + 1, self.V, self.target, self.t_tok, self.out, self.acc, self.kv_src,
                               parent=self.t_par, max_depth=self.D, desc=dm.desc if compact else None,
                               kv=dm.kv if compact else None, ctx_len=dm.ctx_len, ws=self.vws)

    def run(self):
        self.draft()
        self.verify()


class PrefillChainStep:
    """Chain step whose first draft pass runs over all R = 1 + K verified tokens of
    every request ([NEURON] "EagleProposer", propose() prefill phase): index
    kernel (shifted ids, positions, causal masks), FC fuse over the B*R aux
    rows, one draft pass over B*R rows, gather of each request's last accepted
    row, LM head, then K-1 recurrent passes after the accepted tokens, then
    verification against target logits [B, K+1, V]."""

    def __init__(self, dm: DeviceModel, aux_rows, input_ids, next_token, last_idx, target, K=None):
        w = dm.w
        self.dm = dm
        B = w.B
        R = input_ids.shape[1]
        K = K or w.K
        self.B, self.R, self.K, self.V = B, R, K, w.V
        dev = dm.device
        i32 = dict(dtype=torch.int32, device=dev)
        self.aux, self.ids_in, self.next_tok, self.last_idx, self.target = aux_rows, input_ids, next_token, last_idx, target
        M = B * R
        self.tok = torch.zeros(M, **i32)
        self.pos = torch.zeros(M, **i32)
        self.kv_idx = torch.zeros(M, **i32)
        self.mask = torch.zeros(M, dtype=torch.int64, device=dev)
        self.last_row = torch.zeros(B, **i32)
        self.ctx_next = torch.zeros(B, **i32)
        self.h0 = dm.hidden(M)
        self.pre_all = dm.hidden(M)
        self.hn_all = dm.hidden(M)
        self.pre = [dm.hidden(B), dm.hidden(B)]
        self.hn = dm.hidden(B)
        self.hns = [self.hn, dm.hidden(B)]
        self.drafts = torch.zeros(B, K, **i32)
        self.lp = torch.zeros(B, K, dtype=torch.float32, device=dev)
        self.out = torch.zeros(B, K + 1, **i32)
        self.acc = torch.zeros(B, **i32)
        self.kv_src = torch.zeros(B, K + 1, **i32)
        self.vws = torch.zeros(lib.spec_verify_workspace_bytes(B, K + 1, w.V), dtype=torch.uint8, device=dev)

    def draft(self, trace=None):
        """Issue the drafting calls.  ``trace(key, tensors)``, if given, is called on
        the host after the batched pass and its head ("prefill": the pass's rows,
        FC feature, pre-norm and normalised states, the gathered last rows and the
        first draft ids) and after recurrent pass i (i: hn, pre-norm state, ids);
        it must synchronise before reading them."""
        dm, w, B, R, K = self.dm, self.dm.w, self.B, self.R, self.K
        M = B * R
        es = 2 if w.dtype == "bf16" else 4
        lib.spec_prefill_inputs(B, R, self.ids_in, self.next_tok, self.last_idx, dm.ctx_len, self.tok, self.pos,
                                self.kv_idx, self.mask, self.last_row, self.ctx_next, ws=dm.ws)
        lib.spec_fc_fuse(dm.desc, dm.weights, self.aux, self.h0, M, dm.ws)
        rows = lib.make_rows(M, B, R, dm.ctx_len, self.tok, pos=self.pos, kv_idx=self.kv_idx, mask=self.mask,
                             max_ctx=w.max_ctx)
        lib.spec_draft_layer(dm.desc, dm.weights, rows, self.h0, self.pre_all, self.hn_all, dm.kv, dm.ws)
        lib.spec_gather_rows(self.hn_all, M, w.H * es, self.last_row, B, self.hn, ws=dm.ws)
        lib.spec_gather_rows(self.pre_all, M, w.H * es, self.last_row, B, self.pre[1], ws=dm.ws)
        lib.spec_lm_head(dm.desc, dm.weights, self.hn, B, 1, self.drafts, self.lp, ws=dm.ws, ids_ld=K)
        if trace is not None:
            trace("prefill", {"tok": self.tok, "pos": self.pos, "kv_idx": self.kv_idx, "mask": self.mask,
                              "last_row": self.last_row, "ctx_next": self.ctx_next, "h0": self.h0,
                              "pre": self.pre_all, "hn": self.hn_all, "ids": self.drafts[:, 0]})
        # EAGLE-3.1 norm_output: the recurrent passes take the normalised state
        hid = self.hn if w.norm_output else self.pre[1]
        for i in range(1, K):
            rows = lib.make_rows(B, B, 1, self.ctx_next, self.drafts.data_ptr() + 4 * (i - 1), step=i - 1,
                                 tok_stride=K, max_ctx=w.max_ctx + R)
            out = self.pre[(i + 1) % 2]
            hn = self.hns[i % 2]
            lib.spec_draft_layer(dm.desc, dm.weights, rows, hid, out, hn, dm.kv, dm.ws)
            lib.spec_lm_head(dm.desc, dm.weights, hn, B, 1, self.drafts.data_ptr() + 4 * i,
                             self.lp.data_ptr() + 4 * i, ws=dm.ws, ids_ld=K)
            if trace is not None:
                trace(i, {"hn": hn, "pre": out, "ids": self.drafts[:, i]})
            hid = hn if w.norm_output else out

    def verify(self):
        lib.spec_verify_greedy(self.B, self.K + 1, self.V, self.target, self.drafts, self.out, self.acc, self.kv_src,
                               ws=self.vws)

    def run(self):
        self.draft()
        self.verify()
