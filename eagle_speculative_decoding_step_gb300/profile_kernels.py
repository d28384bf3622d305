"""Runs one library call at a workload's sizes a few times (for ncu captures and
per-kernel timing).

    python -m eagle_speculative_decoding_step_gb300.profile_kernels --call lm_head --config llama8b_chain

Calls: lm_head (fused top-k / lse LM head), draft_layer (one recurrent draft
pass), fc_fuse, verify (greedy chain verification), lowrank (EAGLE-4 candidate
head).  Only the tensors the call needs are allocated (random values; the
timings do not depend on them).  Prints per-call CUDA-event time and the
call's algorithmic bytes and GB/s.
"""
import argparse
import json
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))

from eagle_speculative_decoding_step_gb300 import binding as lib  # noqa: E402
from eagle_speculative_decoding_step_gb300 import configs  # noqa: E402


def rand(shape, dtype, scale=0.02, gen=None):
    return (torch.randn(*shape, generator=gen, device="cuda", dtype=torch.float32) * scale).to(dtype)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--call", default="lm_head", choices=["lm_head", "draft_layer", "fc_fuse", "verify", "lowrank"])
    ap.add_argument("--config", default="llama8b_chain")
    ap.add_argument("--rows", type=int, default=0, help="rows per call (default: the workload's draft rows)")
    ap.add_argument("--iters", type=int, default=5)
    ap.add_argument("--ctx", type=int, default=0, help="context length override (draft_layer)")
    args = ap.parse_args()
    w = configs.WORKLOADS[args.config]
    if args.ctx > 0:
        from dataclasses import replace
        w = replace(w, ctx=args.ctx, ctx_range=None)
    lib.load()
    torch.manual_seed(0)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    es = 2 if w.dtype == "bf16" else 4
    M = args.rows or w.rows_max
    d = lib.make_desc(w)
    H, V = w.H, w.V
    W = {}
    ws = torch.zeros(lib.spec_workspace_bytes(d, M, w.max_ctx), dtype=torch.uint8, device="cuda")
    nbytes = 0
    if args.call == "lm_head":
        W["lm_head"] = rand((V, H), dt)
        hn = rand((M, H), dt, 1.0)
        k = 1 if w.mode == "chain" else w.top_k
        ids = torch.zeros(M, k, dtype=torch.int32, device="cuda")
        lp = torch.zeros(M, k, device="cuda")
        wt = lib.make_weights(W)
        fn = lambda: lib.spec_lm_head(d, wt, hn, M, k, ids, lp, ws=ws)  # noqa: E731
        nbytes = V * H * es + M * H * es
    elif args.call == "lowrank":
        W["lm_head"] = rand((V, H), dt)
        W["lr_down"] = rand((w.rank, H), dt)
        W["lr_up"] = rand((V, w.rank), dt)
        hn = rand((M, H), dt, 1.0)
        out = torch.zeros(M, 1, dtype=torch.int32, device="cuda")
        wt = lib.make_weights(W)
        fn = lambda: lib.spec_lowrank_candidates(d, wt, hn, M, 1, out, ws=ws)  # noqa: E731
        nbytes = (w.rank * H + V * w.rank) * es + M * w.num_candidates * H * es
    elif args.call == "fc_fuse":
        W["fc"] = rand((H, 3 * H), dt)
        aux = rand((M, 3 * H), dt, 1.0)
        h0 = torch.zeros(M, H, dtype=dt, device="cuda")
        wt = lib.make_weights(W)
        fn = lambda: lib.spec_fc_fuse(d, wt, aux, h0, M, ws)  # noqa: E731
        nbytes = 3 * H * H * es
    elif args.call == "draft_layer":
        nq, nkv, hd, I = w.nq, w.nkv, w.hd, w.I
        for n, shp in [("embed", (V, H)), ("wq", (nq * hd, 2 * H)), ("wk", (nkv * hd, 2 * H)),
                       ("wv", (nkv * hd, 2 * H)), ("wo", (H, nq * hd)), ("wgate", (I, H)), ("wup", (I, H)),
                       ("wdown", (H, I))]:
            W[n] = rand(shp, dt)
        for n in ("hidden_norm", "in_norm", "post_norm", "final_norm"):
            W[n] = torch.ones(H, dtype=dt, device="cuda")
        B = w.B
        R = M // B
        ctxmax = w.max_ctx
        bs = w.block_size
        nblk = (ctxmax + 64 + bs - 1) // bs
        slots = B * nblk * bs
        kvd = {"k": rand((slots, nkv, hd), dt, 1.0), "v": rand((slots, nkv, hd), dt, 1.0),
               "block_table": torch.arange(B * nblk, dtype=torch.int32, device="cuda").reshape(B, nblk),
               "block_size": bs, "max_blocks": nblk, "num_slots": slots}
        kv = lib.make_kv(kvd)
        ctx = torch.full((B,), ctxmax, dtype=torch.int32, device="cuda")
        tok = torch.randint(0, V, (M,), dtype=torch.int32, device="cuda")
        hid = rand((M, H), dt, 1.0)
        pre, hn = torch.zeros_like(hid), torch.zeros_like(hid)
        if R == 1:
            rows = lib.make_rows(M, B, 1, ctx, tok, step=2, max_ctx=ctxmax)
        else:
            pos = ctx.repeat_interleave(R) + 2
            kvi = torch.arange(R, dtype=torch.int32, device="cuda").repeat(B) + 9
            mask = (torch.ones(M, dtype=torch.int64, device="cuda") | (1 << kvi.long()))
            rows = lib.make_rows(M, B, R, ctx, tok, pos=pos.int(), kv_idx=kvi, mask=mask, max_ctx=ctxmax)
        wt = lib.make_weights(W)
        fn = lambda: lib.spec_draft_layer(d, wt, rows, hid, pre, hn, kv, ws)  # noqa: E731
        keys = min(ctxmax, w.window) if w.window > 0 else ctxmax
        nbytes = (2 * H * (nq + 2 * nkv) * hd + nq * hd * H + 3 * H * I) * es + B * (keys + 3) * 2 * nkv * hd * es
    else:
        B, R = w.B, w.verify_rows
        target = torch.randn(B, R, V, device="cuda")
        drafts = torch.randint(0, V, (B, R - 1), dtype=torch.int32, device="cuda")
        out = torch.zeros(B, R, dtype=torch.int32, device="cuda")
        acc = torch.zeros(B, dtype=torch.int32, device="cuda")
        vws = torch.zeros(lib.spec_verify_workspace_bytes(B, R, V), dtype=torch.uint8, device="cuda")
        fn = lambda: lib.spec_verify_greedy(B, R, V, target, drafts, out, acc, ws=vws)  # noqa: E731
        nbytes = B * R * V * 4
    fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(args.iters):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    ms = float(np.median(times))
    print(json.dumps({"call": args.call, "config": w.name, "rows": M, "ms": ms, "bytes": nbytes,
                      "GBps": nbytes / (ms * 1e-3) / 1e9}))


if __name__ == "__main__":
    main()
