"""Benchmark of one EAGLE speculative step on libeaglespec (GB300).

A step is the whole hot path over one batch: FC fuse of the auxiliary hidden
states, K draft passes (draft layer + LM head), verification of the drafts
against target logits.  Default workload: the Llama-3.1-8B-shaped EAGLE-3 chain
(H 4096, 32/8 heads, MLP 14336, vocab 128256, bf16, batch 4, context 256,
K 5, greedy verification) with synthetic random-init weights and inputs.

Prints one JSON line.  `--impl reference` times the CPU oracle instead on a
bounded sample of the same workload.  Under torchrun every rank runs its own
replica (requests are independent: weak scaling, no data-path collective).
"""
import argparse
import json
import os
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


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


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


def step_bytes(w):
    """Algorithmic HBM bytes of one step (every weight read once per draft pass, the
    allowed context K/V once per pass and request, target logits once) and the
    dominant kernel's (LM head) bytes per launch."""
    es = 2 if w.dtype == "bf16" else 4
    H, nq, nkv, hd, I, V = w.H, w.nq, w.nkv, w.hd, w.I, w.V
    layer = (2 * H * (nq + 2 * nkv) * hd + nq * hd * H + 3 * H * I) * es
    fc = 3 * H * H * es
    head = V * H * es if w.rank == 0 else (H * w.rank + V * w.rank) * es + w.B * w.num_candidates * H * es
    keys = min(w.max_ctx, w.window) if w.window > 0 else w.max_ctx
    kv_per_pass = w.B * (keys + w.draft_region) * 2 * nkv * hd * es
    passes = w.K if w.mode == "chain" else w.depth
    verify = w.B * w.verify_rows * V * 4
    total = fc + passes * (layer + head + kv_per_pass) + verify
    rows = w.B if w.mode == "chain" else w.B * w.top_k
    lm_launch = V * H * es + rows * H * es
    return total, lm_launch


# DRAM traffic per launch of the dominant kernel (dram__bytes_read.sum +
# dram__bytes_write.sum from one ncu capture of the current kernel at this
# workload's LM-head shape); workloads without a capture report null.
LM_TRAFFIC = {"llama8b_chain": 1.086754e9 + 3.369472e6}


def config_of(w):
    """The workload as both arms report it."""
    total_bytes, _ = step_bytes(w)
    return {"workload": w.name, "H": w.H, "heads": [w.nq, w.nkv], "head_dim": w.hd, "I": w.I, "V": w.V,
            "batch": w.B, "ctx": list(w.ctx_range) if w.ctx_range else w.ctx, "mode": w.mode,
            "K": w.K if w.mode == "chain" else None,
            "tree": [w.top_k, w.depth, w.total] if w.mode == "tree" else None,
            "window": w.window, "rank": w.rank, "verify": w.verify,
            "l2": "inputs larger than L2 (weights %.2f GB streamed per step)" % (total_bytes / 1e9)}


def launches_per_step(w):
    layer = 11                                   # prologue, 4 GEMMs, 4 epilogues, attention + combine
    head = 6 if w.rank > 0 else 2                # fused LM head + merge, or the candidate head's 6
    verify = 4 if w.verify == "rejection" else 2  # row statistics, decisions, sampled row, emit / argmax + finalize
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
    st.target = target
    return st


def run_gpu(args, w):
    import torch
    from eagle_speculative_decoding_step_gb300 import binding as lib, engine

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = "cuda:%d" % local
    lib.load()

    t0 = time.time()
    W = synth.make_weights(w)
    if w.rank > 0:
        W["lr_down"], W["lr_up"] = synth.lowrank_factors(W["lm_head"], w.rank, w.dtype)
    ctx = synth.context_lengths(w)
    kv = synth.make_kv(w, ctx)
    aux = synth.make_aux(w)
    root = synth.root_tokens(w)
    dm = engine.DeviceModel(w, W, kv, ctx, device=device)
    del W
    gen_s = time.time() - t0

    aux_d = engine.to_device(aux, w.dtype, device)
    root_d = torch.from_numpy(root).to(device)
    B, V = w.B, w.V
    if w.mode == "tree":
        st = build_tree_step(w, dm, aux_d, root_d, device)
    else:
        st = build_chain_step(w, dm, aux_d, root_d, device)
    target = st.target
    # warm-up (also builds tensor maps / sets kernel attributes), then capture one step
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

    sampler = ClockSampler(local)
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
    lm_rows = B if w.mode == "chain" else B * w.top_k
    lm_k = 1 if w.mode == "chain" else w.top_k

    # dominant kernel (LM head GEMM with fused top-k / lse epilogue), timed alone
    lm_ids = torch.zeros(lm_rows, lm_k, dtype=torch.int32, device=device)
    lm_lp = torch.zeros(lm_rows, lm_k, dtype=torch.float32, device=device)
    n_lm = 20
    with torch.cuda.stream(stream):
        for _ in range(3):
            lib.spec_lm_head(dm.desc, dm.weights, st.hn, lm_rows, lm_k, lm_ids, lm_lp, ws=dm.ws)
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(n_lm):
            lib.spec_lm_head(dm.desc, dm.weights, st.hn, lm_rows, lm_k, lm_ids, lm_lp, ws=dm.ws)
        a1.record(stream)
    torch.cuda.synchronize()
    lm_ms = a0.elapsed_time(a1) / n_lm

    # end to end through the public API with host buffers: every step copies its inputs
    # H2D from pinned memory and reads its result back.  The target logits are read only
    # by verification, so their copy runs on a second stream while the step drafts (it
    # waits for the previous step's verification, which read the same buffer); the
    # drafting and verification phases replay as two graphs with the copy's event between.
    aux_h = aux_d.cpu().pin_memory()
    root_h = root_d.cpu().pin_memory()
    tgt_h = target.cpu().pin_memory()
    out_h = torch.empty(tuple(st.out.shape), dtype=torch.int32).pin_memory()
    acc_h = torch.empty(B, dtype=torch.int32).pin_memory()
    g_draft, g_verify = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g_draft, stream=stream):
            st.draft()
        with torch.cuda.graph(g_verify, stream=stream):
            st.verify()
    torch.cuda.synchronize()
    copy_stream = torch.cuda.Stream(device=device)
    t_ready, v_done = torch.cuda.Event(), torch.cuda.Event()
    n_e2e = max(3, args.steps // 2)
    with torch.cuda.stream(stream):
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        v_done.record(stream)
        for _ in range(n_e2e):
            # the step's small input copies first, then the target logits on the side stream
            aux_d.copy_(aux_h, non_blocking=True)
            root_d.copy_(root_h, non_blocking=True)
            copy_stream.wait_event(v_done)
            with torch.cuda.stream(copy_stream):
                target.copy_(tgt_h, non_blocking=True)
                t_ready.record(copy_stream)
            g_draft.replay()
            stream.wait_event(t_ready)
            g_verify.replay()
            out_h.copy_(st.out, non_blocking=True)
            acc_h.copy_(st.acc, non_blocking=True)
            v_done.record(stream)
        b1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = b0.elapsed_time(b1) / n_e2e
    h2d = aux_h.numel() * aux_h.element_size() + root_h.numel() * 4 + tgt_h.numel() * 4
    d2h = out_h.numel() * 4 + acc_h.numel() * 4
    assert dm.device_error() == 0, "device error in the timed region"

    hbm, tf, kind = _peaks()
    total_bytes, lm_bytes = step_bytes(w)
    lm_gbs = lm_bytes / (lm_ms * 1e-3) / 1e9
    res = {
        "metric": METRIC, "value": aggregate_steps_per_s(world, ms_step), "unit": "steps/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded random-init weights, N(0,1) aux states and context K/V)",
        "config": config_of(w), "timing": "one CUDA graph per step, CUDA events on the replay stream",
        "draft_tokens_per_s": world * proposed * 1000.0 / ms_step,
        "verified_tokens_per_s": world * verified * 1000.0 / ms_step,
        "step_roofline": {"bytes": total_bytes, "t_roof_ms": total_bytes / (hbm * 1e9) * 1e3,
                          "frac": (total_bytes / (hbm * 1e9) * 1e3) / ms_step},
        "roofline": {"kernel": "tc_kernel<SchedRows, EpiStats> (LM head, fused top-k/lse)", "bound": "hbm",
                     "achieved": lm_gbs, "peak": hbm, "unit": "GB/s", "frac": lm_gbs / hbm,
                     "traffic": LM_TRAFFIC.get(w.name),
                     "peak_kind": kind + " (burst copy)", "ms_per_launch": lm_ms},
        "e2e": {"value": world * 1000.0 / e2e_ms, "unit": "steps/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "overlap": "target logits copied on a side stream while drafting"},
        "gpu_launches": launches_per_step(w) * args.steps,
        "clocks": clocks,
        "setup_s": gen_s,
    }
    return res, rank


class OracleSample:
    """The oracle (fp64 numpy, as it stands) on a bounded sample of the workload:
    one draft pass (FC fuse + draft layer + LM head) over the whole batch plus one
    greedy verification; a step is extrapolated as K such passes + the verify.
    Inputs are generated and converted to float64 once, outside the timing."""

    def __init__(self, w):
        from oracle import draft as od, verify as ov
        self.od, self.ov, self.w = od, ov, w
        t0 = time.time()
        W = synth.make_weights(w)
        if w.rank > 0:
            W["lr_down"], W["lr_up"] = synth.lowrank_factors(W["lm_head"], w.rank, w.dtype)
        self.W = {k: np.asarray(v, dtype=np.float64) for k, v in W.items()}
        del W
        self.ctx = synth.context_lengths(w)
        self.kv = synth.make_kv(w, self.ctx)
        self.aux = synth.make_aux(w)
        self.root = synth.root_tokens(w)
        self.setup_s = time.time() - t0

    def step_seconds(self):
        od, ov, w = self.od, self.ov, self.w
        t1 = time.time()
        h0 = od.fc_fuse(w, self.W, self.aux)
        rows = {"M": w.B, "B": w.B, "R": 1, "step": 0, "ctx_len": self.ctx, "tok": self.root}
        pre, hn = od.draft_layer(w, self.W, rows, h0, self.kv)
        if w.rank > 0:
            _, _, ids = od.lowrank_candidates(w, self.W, hn, w.num_candidates, 1)
            logits = hn @ self.W["lm_head"].T
        else:
            ids, _, _, logits = od.lm_head(w, self.W, hn, 1)
        t_pass = time.time() - t1
        target = np.repeat(logits[:, None, :], w.K + 1, axis=1).astype(np.float32)
        t2 = time.time()
        ov.verify_greedy_chain(target, np.repeat(ids, w.K, axis=1))
        t_ver = time.time() - t2
        return w.K * t_pass + t_ver

    def describe(self):
        return ("one draft pass (FC fuse + draft layer + LM head) over the full batch of %d, timed, x K=%d, "
                "plus one greedy verification of [B, K+1, V] logits; fp64 numpy; input generation and "
                "float64 conversion (%.1fs) excluded" % (self.w.B, self.w.K, self.setup_s))


def cpu_baseline(w, samples=1):
    o = OracleSample(w)
    ts = [o.step_seconds() for _ in range(samples)]
    v = 1.0 / statistics.median(ts)
    return {"value": v, "unit": "steps/s", "cores": os.cpu_count(), "kind": "oracle", "sample": o.describe()}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="llama8b_chain")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    w = configs.WORKLOADS[args.config]
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        # the reference arm is the CPU oracle (no other implementation of this path exists)
        if rank != 0:
            return
        t0 = time.time()
        o = OracleSample(w)
        for _ in range(args.warmup):
            o.step_seconds()
        ts = [o.step_seconds() for _ in range(args.steps)]
        ms = 1000.0 * statistics.median(ts)
        v = 1000.0 / ms
        print(json.dumps({"impl": "reference", "metric": METRIC, "value": v, "unit": "steps/s", "n_gpus": 1,
                          "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
                          "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                          "config": config_of(w),
                          "cpu_baseline": {"value": v, "unit": "steps/s", "cores": os.cpu_count(),
                                           "kind": "oracle", "sample": o.describe()},
                          "e2e": {"value": v, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
                          "wall_s": time.time() - t0}))
        return
    res, rank = run_gpu(args, w)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(w)
        print(json.dumps(res))


if __name__ == "__main__":
    main()
