"""Benchmark of one EAGLE speculative step on libeaglespec (GB300).

A step is the whole hot path over one batch: FC fuse of the auxiliary hidden
states, the draft passes (draft layer + LM head or candidate head, plus tree
expansion for a tree), verification of the drafts against target logits.

Headline workload (the largest of the five by bytes per step): the
Qwen3-8B-shaped serving batch (H 4096, 32/8 heads, MLP 12288, vocab 151936,
bf16, batch 32, contexts uniform in [512, 2048], chain of 7, temperature-1
rejection sampling), 13.0 GB of algorithmic HBM traffic per step.  The line
also carries the other three large workloads (Llama-3.1-8B-shaped chain,
Qwen3-4B-shaped tree, EAGLE-4 low-rank candidate head at batch 64) as
sub-records, and the tensor-core-bound batched initial pass (384 rows) of the
EAGLE-4 workload.  Synthetic random-init weights and inputs of those shapes.

Prints one JSON line.  ``--impl reference`` times the CPU oracle instead (real
steps on a bounded sample of the requests).  Under torchrun every rank runs its
own replica (requests are independent: weak scaling, no data-path collective).
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from eagle_speculative_decoding_step_gb300 import configs, synth  # noqa: E402

METRIC = "spec steps/s"
HEADLINE = "qwen8b_rejection"
SUB_WORKLOADS = ["llama8b_chain", "qwen4b_tree", "eagle4_lowrank"]
CSRC = os.path.join(ROOT, "eagle_speculative_decoding_step_gb300", "csrc")
TRAFFIC_MD = os.path.join(ROOT, "profiles", "traffic_dominant_calls.md")
# kernel sources whose change invalidates a recorded DRAM-traffic capture
CALL_SOURCES = {
    "lm_head": ["lmhead.cu", "tc_kernel.cuh", "tc_core.cuh", "common.cuh"],
    "draft_layer": ["api.cu", "layer.cu", "tc_gemm.cu", "tc_kernel.cuh", "tc_core.cuh", "common.cuh", "plan.cuh"],
}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return (d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0),
                d.get("bf16_tflops_sustained", d.get("bf16_tflops", 1700.0)), "measured")
    return 6800.0, 1900.0, 1700.0, "fallback"


def source_hash(call):
    h = hashlib.sha256()
    for f in CALL_SOURCES[call]:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


def recorded_traffic(workload, call):
    """DRAM bytes (read + write) per launch of a dominant call, from the committed
    ncu capture table, or None when there is none or the kernels changed since."""
    if not os.path.exists(TRAFFIC_MD):
        return None
    want = source_hash(call)
    for line in open(TRAFFIC_MD):
        f = [x.strip() for x in line.strip().strip("|").split("|")]
        if len(f) >= 4 and f[0] == workload and f[1] == call and re.fullmatch(r"[0-9a-f]{12}", f[3] or ""):
            try:
                return float(f[2]) if f[3] == want else None
            except ValueError:
                return None
    return None


def max_over_ranks(ms, dist, device="cpu"):
    """The slowest rank's time (barrier-bracketed timing of independent replicas).
    Works for nccl (device tensors) and gloo (host tensors)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(ms)
    import torch
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_steps_per_s(world, ms_step):
    """Whole-job steps/s: every rank ran its own replica for the same number of
    steps, bounded by the slowest rank."""
    return world * 1000.0 / ms_step


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def layer_bytes(w):
    es = 2 if w.dtype == "bf16" else 4
    H, nq, nkv, hd, I = w.H, w.nq, w.nkv, w.hd, w.I
    return (2 * H * (nq + 2 * nkv) * hd + nq * hd * H + 3 * H * I) * es


def head_bytes(w):
    es = 2 if w.dtype == "bf16" else 4
    if w.rank == 0:
        return (w.draft_vocab or w.V) * w.H * es
    return (w.H * w.rank + w.V * w.rank) * es + w.B * w.num_candidates * w.H * es


def step_bytes(w):
    """Algorithmic HBM bytes of one step (every weight read once per draft pass, the
    allowed context K/V once per pass and request, target logits once) and the
    LM head's bytes per launch."""
    es = 2 if w.dtype == "bf16" else 4
    ctx = synth.context_lengths(w).astype(np.int64)
    keys = np.minimum(ctx, w.window) if w.window > 0 else ctx        # allowed context keys per request
    kv_per_pass = int((keys + w.draft_region).sum()) * 2 * w.nkv * w.hd * es
    passes = w.K if w.mode == "chain" else w.depth
    verify = w.B * w.verify_rows * w.V * 4
    total = 3 * w.H * w.H * es + passes * (layer_bytes(w) + head_bytes(w) + kv_per_pass) + verify
    rows = w.B if w.mode == "chain" else w.B * w.top_k
    lm_launch = (w.draft_vocab or w.V) * w.H * es + rows * w.H * es
    return total, lm_launch


def config_of(w):
    """The workload as both arms report it."""
    total_bytes, _ = step_bytes(w)
    return {"workload": w.name, "H": w.H, "heads": [w.nq, w.nkv], "head_dim": w.hd, "I": w.I, "V": w.V,
            "batch": w.B, "ctx": list(w.ctx_range) if w.ctx_range else w.ctx, "mode": w.mode,
            "K": w.K if w.mode == "chain" else None,
            "tree": [w.top_k, w.depth, w.total] if w.mode == "tree" else None,
            "window": w.window, "rank": w.rank, "num_candidates": w.num_candidates, "verify": w.verify,
            "l2": "inputs larger than L2 (%.2f GB of weights, K/V and logits streamed per step)" % (total_bytes / 1e9)}


def launches_per_step(w):
    layer = 11                                   # prologue, 4 GEMMs, 4 epilogues, attention + combine
    head = 6 if w.rank > 0 else 2                # fused LM head + merge, or the candidate head's 6
    verify = 1                                   # one verifier kernel (greedy or rejection, no top-k / top-p)
    if w.mode == "chain":
        return 2 + w.K * (layer + head) + verify
    return 2 + w.depth * (layer + head + 1) + verify  # + tree expansion per depth


def build_chain_step(w, dm, aux_d, root_d, device):
    """Chain step whose target logits are the draft's own logits over K+1 chained
    passes plus N(0, sigma) noise (built once, untimed, with the library's
    full-logits LM head)."""
    import torch
    from eagle_speculative_decoding_step_gb300 import binding as lib, engine
    B, K, V = w.B, w.K, w.V
    target = torch.empty(B, K + 1, V, dtype=torch.float32, device=device)
    h0 = dm.hidden(B)
    pre = [dm.hidden(B), dm.hidden(B)]
    hn = dm.hidden(B)
    ids = torch.zeros(B, K + 1, dtype=torch.int32, device=device)
    lp = torch.zeros(B, K + 1, dtype=torch.float32, device=device)
    logits = torch.empty(B, V, dtype=torch.float32, device=device)
    scratch_ids = torch.zeros(B, 1, dtype=torch.int32, device=device)
    scratch_lp = torch.zeros(B, 1, dtype=torch.float32, device=device)
    lib.spec_fc_fuse(dm.desc, dm.weights, aux_d, h0, B, dm.ws)
    hid = h0
    for i in range(K + 1):
        tok = root_d if i == 0 else ids.data_ptr() + 4 * (i - 1)
        rows = lib.make_rows(B, B, 1, dm.ctx_len, tok, step=i, tok_stride=1 if i == 0 else K + 1,
                             max_ctx=w.max_ctx)
        lib.spec_draft_layer(dm.desc, dm.weights, rows, hid, pre[i % 2], hn, dm.kv, dm.ws)
        if w.rank > 0:
            lib.spec_lowrank_candidates(dm.desc, dm.weights, hn, B, 1, ids.data_ptr() + 4 * i, ws=dm.ws,
                                        out_ld=K + 1)
            lib.spec_lm_head(dm.desc, dm.weights, hn, B, 1, scratch_ids, scratch_lp, None, logits, ws=dm.ws)
        else:
            lib.spec_lm_head(dm.desc, dm.weights, hn, B, 1, ids.data_ptr() + 4 * i, lp.data_ptr() + 4 * i, None,
                             logits, ws=dm.ws, ids_ld=K + 1)
        target[:, i].copy_(logits)
        hid = pre[i % 2]
    target.add_(torch.from_numpy(synth.noise(w, (B, K + 1, V))).to(device))
    torch.cuda.synchronize()
    temp = torch.full((B,), w.temperature, dtype=torch.float32, device=device)
    return engine.ChainStep(dm, aux_d, root_d, target, temperature=temp, seed=w.philox_seed)


def build_tree_step(w, dm, aux_d, root_d, device):
    """Tree step whose target logits are one draft pass over the root and all tree
    nodes (tree mask, root FC feature as every node's hidden input) plus noise."""
    import torch
    from eagle_speculative_decoding_step_gb300 import binding as lib, engine
    B, N, V = w.B, w.total, w.V
    st = engine.TreeStep(dm, aux_d, root_d, None)
    st.draft()
    M = B * (N + 1)
    big = engine.DeviceModel.__new__(engine.DeviceModel)
    big.__dict__.update(dm.__dict__)
    nb = lib.spec_workspace_bytes(dm.desc, M, w.max_ctx)
    big.ws = torch.zeros(nb, dtype=torch.uint8, device=device)
    kv_idx = torch.arange(N + 1, dtype=torch.int32, device=device).repeat(B)
    hid_src = torch.arange(B, dtype=torch.int32, device=device).repeat_interleave(N + 1)
    rows = lib.make_rows(M, B, N + 1, dm.ctx_len, st.t_tok.reshape(-1), pos=st.t_pos.reshape(-1), kv_idx=kv_idx,
                         mask=st.t_mask.reshape(-1), hid_src=hid_src, max_ctx=w.max_ctx)
    pre, hn = big.hidden(M), big.hidden(M)
    lib.spec_draft_layer(dm.desc, dm.weights, rows, st.h0, pre, hn, dm.kv, big.ws)
    target = torch.empty(B, N + 1, V, dtype=torch.float32, device=device)
    for b in range(B):
        lib.spec_lm_head(dm.desc, dm.weights, hn[b * (N + 1):(b + 1) * (N + 1)], N + 1, 1,
                         torch.zeros(N + 1, 1, dtype=torch.int32, device=device),
                         torch.zeros(N + 1, 1, device=device), None, target[b], ws=big.ws)
    target.add_(torch.from_numpy(synth.noise(w, (B, N + 1, V))).to(device))
    torch.cuda.synchronize()
    del big
    st.target = target
    return st


def time_on_stream(stream, fn, n, warm=3):
    """Average CUDA-event time (ms) of ``fn`` over n calls on ``stream``."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(warm):
            fn()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(n):
            fn()
        a1.record(stream)
    torch.cuda.synchronize()
    return a0.elapsed_time(a1) / n


def dominant_call(w, st, dm, stream, device, hbm):
    """The step's dominant library call timed alone (CUDA events on its stream): the
    fused LM head for a full-vocabulary head, else the draft layer (weights + the
    allowed K/V dominate once the candidate head replaces the full head)."""
    import torch
    from eagle_speculative_decoding_step_gb300 import binding as lib
    es = 2 if w.dtype == "bf16" else 4
    if w.rank == 0:
        rows = w.B if w.mode == "chain" else w.B * w.top_k
        k = 1 if w.mode == "chain" else w.top_k
        ids = torch.zeros(rows, k, dtype=torch.int32, device=device)
        lp = torch.zeros(rows, k, dtype=torch.float32, device=device)
        ms = time_on_stream(stream, lambda: lib.spec_lm_head(dm.desc, dm.weights, st.hn, rows, k, ids, lp, ws=dm.ws), 20)
        _, nbytes = step_bytes(w)
        call, kernel = "lm_head", "tc_kernel<SchedRows, EpiStats> + lm_merge_kernel (LM head, fused top-k/lse)"
    else:
        # the last chain pass (step K-1) on its own inputs: writes the same K/V again
        K, B = w.K, w.B
        rows = lib.make_rows(B, B, 1, dm.ctx_len, st.drafts.data_ptr() + 4 * (K - 2), step=K - 1, tok_stride=K,
                             max_ctx=w.max_ctx)
        hid = st.pre[(K - 2) % 2]
        pre, hn = dm.hidden(B), dm.hidden(B)
        ms = time_on_stream(stream, lambda: lib.spec_draft_layer(dm.desc, dm.weights, rows, hid, pre, hn, dm.kv,
                                                                 dm.ws), 20)
        keys = w.window if w.window > 0 else w.max_ctx + K
        nbytes = layer_bytes(w) + B * keys * 2 * w.nkv * w.hd * es
        call, kernel = "draft_layer", "spec_draft_layer (4 tcgen05 GEMMs, attention, epilogues)"
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"kernel": kernel, "call": call, "bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
            "frac": gbs / hbm, "traffic": recorded_traffic(w.name, call), "algorithmic_bytes": nbytes,
            "ms_per_launch": ms}


def run_workload(args, w, dist, device, world):
    """Build, warm up, capture and time one workload's step; then the dominant call
    alone and the end-to-end loop through host buffers."""
    import torch
    from eagle_speculative_decoding_step_gb300 import binding as lib, engine
    t0 = time.time()
    W = synth.make_weights(w)
    if w.rank > 0:
        W["lr_down"], W["lr_up"] = synth.lowrank_factors(W["lm_head"], w.rank, w.dtype)
    ctx = synth.context_lengths(w)
    kv = synth.make_kv(w, ctx)
    aux = synth.make_aux(w)
    root = synth.root_tokens(w)
    dm = engine.DeviceModel(w, W, kv, ctx, device=device)
    del W, kv
    gen_s = time.time() - t0
    aux_d = engine.to_device(aux, w.dtype, device)
    root_d = torch.from_numpy(root).to(device)
    B = w.B
    st = build_tree_step(w, dm, aux_d, root_d, device) if w.mode == "tree" else \
        build_chain_step(w, dm, aux_d, root_d, device)
    target = st.target
    for _ in range(max(1, args.warmup)):
        st.run()
    torch.cuda.synchronize()
    assert dm.device_error() == 0, "device error after warm-up"
    stream = torch.cuda.Stream(device=device)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            st.run()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clocks = sampler.stop()
    ms = max_over_ranks(e0.elapsed_time(e1), dist, device)
    ms_step = ms / args.steps
    acc = st.acc.cpu().numpy()
    verified = float((acc + 1).sum())
    proposed = B * (w.K if w.mode == "chain" else w.total)

    hbm, tf_burst, tf_sust, kind = _peaks()
    dom = dominant_call(w, st, dm, stream, device, hbm)
    dom["peak_kind"] = kind + " (burst copy)"

    # end to end through the public API with host buffers: every step copies its inputs
    # H2D from pinned memory and reads its result back.  Two sets of device input
    # buffers (aux features, root tokens, target logits) alternate between steps, each
    # with its own pair of graphs (drafting, verification): step s's copies go on a copy
    # stream as soon as step s-2 (the last user of that set) is verified, so they run
    # while step s-1 computes; on the copy stream the drafting inputs come first, then
    # the target logits, which only verification reads.
    aux_h = aux_d.cpu().pin_memory()
    root_h = root_d.cpu().pin_memory()
    tgt_h = target.cpu().pin_memory()
    out_h = torch.empty(tuple(st.out.shape), dtype=torch.int32).pin_memory()
    acc_h = torch.empty(B, dtype=torch.int32).pin_memory()
    sets = [(aux_d, root_d, target), (torch.empty_like(aux_d), torch.empty_like(root_d), torch.empty_like(target))]
    graphs = []
    with torch.cuda.stream(stream):
        for a_d, r_d, t_d in sets:
            st.aux, st.root, st.target = a_d, r_d, t_d
            g_draft, g_verify = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_draft, stream=stream):
                st.draft()
            with torch.cuda.graph(g_verify, stream=stream):
                st.verify()
            graphs.append((g_draft, g_verify))
    st.aux, st.root, st.target = sets[0]
    torch.cuda.synchronize()
    copy_stream = torch.cuda.Stream(device=device)
    in_ready = [torch.cuda.Event(), torch.cuda.Event()]
    t_ready = [torch.cuda.Event(), torch.cuda.Event()]
    v_done = [torch.cuda.Event(), torch.cuda.Event()]
    n_e2e = max(4, args.steps // 2)
    with torch.cuda.stream(stream):
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        v_done[0].record(stream)
        v_done[1].record(stream)
        for s_i in range(n_e2e):
            k = s_i % 2
            a_d, r_d, t_d = sets[k]
            copy_stream.wait_event(v_done[k])
            with torch.cuda.stream(copy_stream):
                a_d.copy_(aux_h, non_blocking=True)
                r_d.copy_(root_h, non_blocking=True)
                in_ready[k].record(copy_stream)
                t_d.copy_(tgt_h, non_blocking=True)
                t_ready[k].record(copy_stream)
            stream.wait_event(in_ready[k])
            graphs[k][0].replay()
            stream.wait_event(t_ready[k])
            graphs[k][1].replay()
            out_h.copy_(st.out, non_blocking=True)
            acc_h.copy_(st.acc, non_blocking=True)
            v_done[k].record(stream)
        b1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(b0.elapsed_time(b1) / n_e2e, dist, device)
    h2d = aux_h.numel() * aux_h.element_size() + root_h.numel() * 4 + tgt_h.numel() * 4
    d2h = out_h.numel() * 4 + acc_h.numel() * 4
    assert dm.device_error() == 0, "device error in the timed region"
    total_bytes, _ = step_bytes(w)
    t_roof = total_bytes / (hbm * 1e9) * 1e3
    res = {
        "value": aggregate_steps_per_s(world, ms_step), "ms_per_step": ms_step,
        "draft_tokens_per_s": world * proposed * 1000.0 / ms_step,
        "verified_tokens_per_s": world * verified * 1000.0 / ms_step,
        "step_roofline": {"bytes": total_bytes, "t_roof_ms": t_roof, "frac": t_roof / ms_step,
                          "peak": hbm, "peak_kind": kind + " (burst copy)"},
        "roofline": dom,
        "e2e": {"value": world * 1000.0 / e2e_ms, "unit": "steps/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "overlap": "two input buffer sets: a step's inputs and target logits are copied on a side "
                           "stream while the previous step computes"},
        "gpu_launches": launches_per_step(w) * args.steps,
        "clocks": clocks, "setup_s": gen_s, "config": config_of(w),
    }
    del st, graph, g_draft, g_verify, dm, target
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def run_prefill_tensor(args, device):
    """The batched initial pass of the EAGLE-4 workload ([NEURON] "EagleProposer"
    prefill phase, "Warmup with Speculation Enabled": batch x (1 + K) tokens):
    64 requests x 6 verified tokens = 384 rows through FC fuse and the draft layer
    -- the tensor-core-bound GEMM regime (384 flop per weight byte, above the
    bf16 ridge).  Each call timed alone with CUDA events; TFLOP/s against the
    measured bf16 peak."""
    import torch
    from dataclasses import replace
    from eagle_speculative_decoding_step_gb300 import binding as lib, engine
    w0 = configs.WORKLOADS["eagle4_lowrank"]
    R = w0.K + 1
    w = replace(w0, K=2 * w0.K + 1)        # cache room for R prefill rows + K-1 recurrent entries
    B, H, M = w.B, w.H, w.B * R
    W = synth.make_weights(w)
    W["lr_down"], W["lr_up"] = synth.lowrank_factors(W["lm_head"], w.rank, w.dtype)
    ctx = synth.context_lengths(w)
    kv = synth.make_kv(w, ctx)
    dm = engine.DeviceModel(w, W, kv, ctx, device=device, max_rows=M)
    del W, kv
    g = np.random.default_rng(7)
    aux = engine.to_device(synth.make_aux(w, rows=M), w.dtype, device)
    ids = torch.from_numpy(g.integers(0, w.V, size=(B, R)).astype(np.int32)).to(device)
    nxt = torch.from_numpy(g.integers(0, w.V, size=B).astype(np.int32)).to(device)
    last = torch.from_numpy(g.integers(0, R, size=B).astype(np.int32)).to(device)
    target = torch.zeros(B, w0.K + 1, w.V, device=device)
    st = engine.PrefillChainStep(dm, aux, ids, nxt, last, target, K=w0.K)
    st.run()
    torch.cuda.synchronize()
    assert dm.device_error() == 0
    stream = torch.cuda.Stream(device=device)
    rows = lib.make_rows(M, B, R, dm.ctx_len, st.tok, pos=st.pos, kv_idx=st.kv_idx, mask=st.mask,
                         max_ctx=w.max_ctx)
    ms_fc = time_on_stream(stream, lambda: lib.spec_fc_fuse(dm.desc, dm.weights, aux, st.h0, M, dm.ws), 20)
    ms_layer = time_on_stream(stream, lambda: lib.spec_draft_layer(dm.desc, dm.weights, rows, st.h0, st.pre_all,
                                                                   st.hn_all, dm.kv, dm.ws), 20)
    ms_step = time_on_stream(stream, st.run, 10)
    hbm, tf_burst, tf_sust, kind = _peaks()
    es = 2
    fc_flops = 2.0 * M * 3 * H * H
    layer_flops = 2.0 * M * layer_bytes(w) / es
    attn_flops = 2.0 * 2 * M * w.nq * w.hd * (w.window + R)
    res = {"workload": "eagle4_lowrank batched initial pass: %d requests x %d verified tokens = %d rows" % (B, R, M),
           "fc_fuse": {"ms": ms_fc, "tflops": fc_flops / (ms_fc * 1e-3) / 1e12},
           "draft_layer": {"ms": ms_layer, "tflops": (layer_flops + attn_flops) / (ms_layer * 1e-3) / 1e12,
                           "gemm_flops": layer_flops, "attention_flops": attn_flops},
           "prefill_step_ms": ms_step, "peak_tflops_burst": tf_burst, "peak_tflops_sustained": tf_sust,
           "peak_kind": kind}
    for k in ("fc_fuse", "draft_layer"):
        res[k]["frac_burst"] = res[k]["tflops"] / tf_burst
        res[k]["frac_sustained"] = res[k]["tflops"] / tf_sust
    del st, dm
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------- the oracle on the host cores
def sample_requests(w):
    """Requests the oracle runs per timed step (requests are independent; the fp64
    passes over one request already stream every weight once)."""
    return min(w.B, 4)


class OracleStep:
    """Real oracle speculative steps (fp64 numpy, as it stands) on a bounded sample
    of the workload's requests: FC fuse, every draft pass (chain or tree), and
    verification (greedy chain / tree with K/V compaction, or rejection) against
    target logits built once outside the timing.  A step over n of B requests
    counts as n/B of a workload step."""

    def __init__(self, w, n_req=None):
        from oracle import step as ostep
        self.ostep, self.w = ostep, w
        t0 = time.time()
        n = sample_requests(w) if n_req is None else n_req
        self.idx = np.arange(n)
        W = synth.make_weights(w)
        if w.rank > 0:
            W["lr_down"], W["lr_up"] = synth.lowrank_factors(W["lm_head"], w.rank, w.dtype)
        self.W = {k: np.asarray(v, dtype=np.float64) for k, v in W.items()}
        del W
        ctx = synth.context_lengths(w)
        kv = synth.make_kv(w, ctx)
        self.ctx = ctx[self.idx]
        self.kv = dict(kv, block_table=kv["block_table"][self.idx])
        self.aux = synth.make_aux(w)[self.idx]
        self.root = synth.root_tokens(w)[self.idx]
        self.temp = np.full(n, w.temperature, dtype=np.float32)
        if w.mode == "tree":
            fin = ostep.tree_draft(w, self.W, self.aux, self.root, self.ctx, self.kv, w.top_k, w.depth, w.total)
            noise = synth.noise(w, (w.B, w.total + 1, w.V))[self.idx]
            self.target = ostep.tree_target(w, self.W, self.aux, self.ctx, self.kv, fin, noise)
        else:
            noise = synth.noise(w, (w.B, w.K + 1, w.V))[self.idx]
            self.target = ostep.chain_target(w, self.W, self.aux, self.root, self.ctx, self.kv, w.K, noise)
        self.setup_s = time.time() - t0

    @property
    def fraction(self):
        return len(self.idx) / self.w.B

    def step_seconds(self):
        from oracle import verify as ov
        w, os_ = self.w, self.ostep
        t1 = time.time()
        if w.mode == "tree":
            fin = os_.tree_draft(w, self.W, self.aux, self.root, self.ctx, self.kv, w.top_k, w.depth, w.total)
            out, acc, src = ov.verify_greedy_tree(self.target, fin["tok"], fin["parent"], w.depth)
            ov.compact_kv(self.kv, self.ctx, src, acc)
        else:
            os_.chain_step(w, self.W, self.aux, self.root, self.ctx, self.kv, w.K, self.target, self.temp,
                           w.philox_seed, 0)
        return time.time() - t1

    def describe(self):
        return ("real oracle steps on %d of the %d requests (FC fuse, %s, %s verification on target logits of "
                "the oracle's own drafts + noise); each counts as %d/%d of a workload step; fp64 numpy; input "
                "generation, float64 conversion and target logits (%.1fs) excluded"
                % (len(self.idx), self.w.B, "%d draft passes" % self.w.K if self.w.mode == "chain" else
                   "tree drafting %d/%d/%d" % (self.w.top_k, self.w.depth, self.w.total), self.w.verify,
                   len(self.idx), self.w.B, self.setup_s))


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(v, "").isdigit():
            return int(os.environ[v])
    return os.cpu_count()


def oracle_probe(name, reps):
    """Median of ``reps`` oracle steps of a workload (run in a child process, so the
    BLAS thread count can be fixed before numpy loads)."""
    w = configs.WORKLOADS[name]
    o = OracleStep(w)
    ts = [o.step_seconds() for _ in range(reps)]
    return {"workload": name, "value": o.fraction / statistics.median(ts), "unit": "steps/s",
            "cores": blas_threads(), "runs": reps, "seconds": ts, "sample": o.describe()}


def single_thread_probe(name, reps=3):
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-probe", name, "--steps", str(reps)],
                       capture_output=True, text=True, env=env, timeout=600)
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    if r.returncode != 0 or not lines:
        return {"workload": name, "error": (r.stderr or r.stdout)[-300:]}
    return json.loads(lines[-1])


def cpu_baseline(w, reps=3):
    """The oracle on the host cores: median of ``reps`` real steps on the request
    sample of the workload, all BLAS threads; plus single-thread figures of the
    two smallest workloads."""
    o = OracleStep(w)
    ts = [o.step_seconds() for _ in range(reps)]
    res = {"value": o.fraction / statistics.median(ts), "unit": "steps/s", "cores": blas_threads(), "kind": "oracle",
           "sample": o.describe(), "runs": reps, "seconds": ts}
    del o
    res["single_thread"] = [single_thread_probe(n) for n in ("tiny", "llama8b_chain")]
    return res


def run_reference(args, w):
    """The reference arm: the oracle, as it stands, timed on the host cores."""
    t0 = time.time()
    o = OracleStep(w)
    for _ in range(args.warmup):
        o.step_seconds()
    ts = [o.step_seconds() for _ in range(args.steps)]
    ms = 1000.0 * statistics.median(ts)
    v = o.fraction * 1000.0 / ms
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "steps/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w),
            "timing": "wall clock per oracle step on %d of %d requests (median of the timed steps); value = "
                      "%d/%d x steps per second" % (len(o.idx), w.B, len(o.idx), w.B),
            "cpu_baseline": {"value": v, "unit": "steps/s", "cores": blas_threads(), "kind": "oracle",
                             "sample": o.describe()},
            "e2e": {"value": v, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": time.time() - t0}


def summary(r):
    keep = ("value", "ms_per_step", "draft_tokens_per_s", "verified_tokens_per_s", "step_roofline", "roofline",
            "e2e", "gpu_launches", "clocks", "config")
    return {k: r[k] for k in keep}


def run_timeline(args, w):
    """The workload's step, captured as in the bench, replayed three times with the
    instrumented library's per-block log attached; writes the last step's per-kernel
    table and launch sequence (markdown) to args.timeline."""
    os.environ["EAGLESPEC_TIMELINE"] = "1"
    from eagle_speculative_decoding_step_gb300 import build
    build.build(timeline=True)
    import torch
    from eagle_speculative_decoding_step_gb300 import binding as lib, engine, timeline
    device = "cuda:0"
    L = lib.load()
    W = synth.make_weights(w)
    if w.rank > 0:
        W["lr_down"], W["lr_up"] = synth.lowrank_factors(W["lm_head"], w.rank, w.dtype)
    ctx = synth.context_lengths(w)
    kv = synth.make_kv(w, ctx)
    aux = synth.make_aux(w)
    root = synth.root_tokens(w)
    dm = engine.DeviceModel(w, W, kv, ctx, device=device)
    del W, kv
    aux_d = engine.to_device(aux, w.dtype, device)
    root_d = torch.from_numpy(root).to(device)
    st = build_tree_step(w, dm, aux_d, root_d, device) if w.mode == "tree" else \
        build_chain_step(w, dm, aux_d, root_d, device)
    for _ in range(max(1, args.warmup)):
        st.run()
    stream = torch.cuda.Stream(device=device)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            st.run()
        for _ in range(args.warmup):
            graph.replay()
    torch.cuda.synchronize()
    log = torch.zeros(timeline.LOG_WORDS, dtype=torch.int64, device=device)
    timeline.attach(L, log.data_ptr())
    with torch.cuda.stream(stream):
        for _ in range(3):
            graph.replay()
    torch.cuda.synchronize()
    timeline.attach(L, 0)
    assert dm.device_error() == 0, "device error"
    step = timeline.last_step(timeline.launches(log.cpu().numpy()))
    with open(args.timeline, "w") as f:
        f.write("# Timeline: %s, one graph-replayed step (instrumented build)\n\n" % w.name)
        f.write(timeline.markdown(step) + "\n\nLaunch sequence (us from the step's first launch: start, end, "
                "duration, tail, kernel, blocks):\n\n```\n" + timeline.sequence(step) + "\n```\n")
    print(timeline.markdown(step))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=HEADLINE)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sub", action="store_true", help="headline workload only")
    ap.add_argument("--oracle-probe", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--timeline", default=None, metavar="FILE",
                    help="instead of the bench line: per-kernel timeline of the workload's graph-replayed step "
                         "from the instrumented library (markdown to FILE)")
    args = ap.parse_args()
    if args.oracle_probe:
        print(json.dumps(oracle_probe(args.oracle_probe, max(1, args.steps))))
        return
    w = configs.WORKLOADS[args.config]
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        # the reference arm is the CPU oracle (no other implementation of this path exists)
        if rank != 0:
            return
        print(json.dumps(run_reference(args, w)))
        return

    if args.timeline:
        run_timeline(args, w)
        return
    import torch
    from eagle_speculative_decoding_step_gb300 import binding as lib
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = "cuda:%d" % local
    lib.load()
    r = run_workload(args, w, dist, device, world)
    res = {"metric": METRIC, "value": r["value"], "unit": "steps/s", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": r["ms_per_step"], "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": w.dtype,
           "data": "synthetic (seeded random-init weights, N(0,1) aux states and context K/V)",
           "config": r["config"], "timing": "one CUDA graph per step, CUDA events on the replay stream"}
    for k in ("draft_tokens_per_s", "verified_tokens_per_s", "step_roofline", "roofline", "e2e", "gpu_launches",
              "clocks", "setup_s"):
        res[k] = r[k]
    if not args.no_sub and args.config == HEADLINE:
        res["workloads"] = {}
        for name in SUB_WORKLOADS:
            res["workloads"][name] = summary(run_workload(args, configs.WORKLOADS[name], dist, device, world))
        res["tensor_bound"] = run_prefill_tensor(args, device)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(w)
        print(json.dumps(res))


if __name__ == "__main__":
    main()
